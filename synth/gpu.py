"""Device-side filling of seeded synthetic layers (binding of libmoe_synth.so).

Writes the same bytes as ``synth.gen_matrix`` (checked by tests/test_synth_gpu.py)
straight into device memory, so full-size layer stacks never pass through the
host. Input generation only: nothing here computes the layer.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

from . import (DOWN, GATE, IQ3_XXS, UP, LayerConfig, expert_formats, gen_logits, gen_x_bf16, iq3_grid, layer_seed,
               padded_stride, row_bytes, weight_key, BLOCK_ELEMS)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_synth.so")


class SynthMatrix(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("row_stride_bytes", ctypes.c_int64), ("format", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("cols", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("key", ctypes.c_uint64)]


_lib = None


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        _lib = ctypes.CDLL(LIB_PATH)
        _lib.moe_synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p]
        _lib.moe_synth_fill.restype = ctypes.c_int
    return _lib


def fill(mats: List[Tuple[torch.Tensor, int, int, int, int, int]], stream=None) -> None:
    """mats: (uint8 CUDA tensor, fmt, rows, cols, stride, key) per matrix."""
    L = load()
    s = stream if stream is not None else torch.cuda.current_stream()
    for c0 in range(0, len(mats), 60000):
        chunk = mats[c0:c0 + 60000]
        arr = (SynthMatrix * len(chunk))()
        max_rows, max_nb = 0, 0
        for i, (t, fmt, rows, cols, stride, key) in enumerate(chunk):
            assert t.is_cuda and t.dtype == torch.uint8 and t.numel() >= rows * stride
            arr[i] = SynthMatrix(t.data_ptr(), stride, fmt, rows, cols, 0, key)
            max_rows = max(max_rows, rows)
            max_nb = max(max_nb, cols // BLOCK_ELEMS[fmt])
        host = torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8)
        dev = host.to(device="cuda", non_blocking=False)
        rc = L.moe_synth_fill(ctypes.c_void_p(dev.data_ptr()), len(chunk), max_rows, max_nb,
                              ctypes.c_void_p(s.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"moe_synth_fill failed ({rc})")
        s.synchronize()       # keep `dev` alive until the kernel has read it


@dataclass
class DeviceLayer:
    cfg: LayerConfig
    seed: int
    fmts: List[Tuple[int, int]]
    storage: torch.Tensor                   # all of the layer's weight bytes
    experts: List[Dict[str, tuple]]         # name -> (fmt, rows, cols, stride, uint8 view)
    x_bf16: torch.Tensor                    # bf16 [T, H] on the device
    logits: torch.Tensor                    # fp32 [T, E] on the device
    x_host: np.ndarray                      # uint16 bf16 bits [T, H]
    logits_host: np.ndarray                 # fp32 [T, E]
    weight_bytes_unpadded: int
    grid: Optional[torch.Tensor] = None     # IQ3_XXS grid (int32 [256] on the device), if the layer has IQ3_XXS

    def expert_bytes(self, e: int) -> int:
        gu, dn = self.fmts[e]
        H, I = self.cfg.hidden, self.cfg.inter
        return 2 * I * row_bytes(gu, H) + H * row_bytes(dn, I)


def make_device_layer(cfg: LayerConfig, layer: int = 0, tokens: Optional[int] = None,
                      fill_weights: bool = True) -> DeviceLayer:
    seed = layer_seed(cfg, layer)
    T = cfg.tokens if tokens is None else tokens
    fmts = expert_formats(cfg, seed)
    H, I = cfg.hidden, cfg.inter
    spec = []        # (offset, fmt, rows, cols, stride, key, expert, name)
    off = 0
    for e in range(cfg.n_entries):
        gu, dn = fmts[e]
        for name, mat, fmt, rows, cols in (("gate", GATE, gu, I, H), ("up", UP, gu, I, H), ("down", DOWN, dn, H, I)):
            stride = padded_stride(fmt, cols)
            spec.append((off, fmt, rows, cols, stride, weight_key(seed, e, mat), e, name))
            off += (rows * stride + 255) // 256 * 256
    storage = torch.empty(off, dtype=torch.uint8, device="cuda")
    experts: List[Dict[str, tuple]] = [dict() for _ in range(cfg.n_entries)]
    mats = []
    for (o, fmt, rows, cols, stride, key, e, name) in spec:
        view = storage[o:o + rows * stride]
        experts[e][name] = (fmt, rows, cols, stride, view)
        mats.append((view, fmt, rows, cols, stride, key))
    if fill_weights:
        fill(mats)
    x_host = gen_x_bf16(seed, T, H)
    logits_host = gen_logits(seed, T, cfg.n_experts, cfg.zipf_bias)
    x = torch.from_numpy(x_host.view(np.int16).copy()).to("cuda").view(torch.bfloat16)
    lg = torch.from_numpy(logits_host.copy()).to("cuda")
    unpadded = sum(2 * I * row_bytes(gu, H) + H * row_bytes(dn, I) for gu, dn in fmts)
    grid = None
    if any(IQ3_XXS in f for f in fmts):
        grid = torch.from_numpy(iq3_grid().view(np.int32).copy()).to("cuda")
    return DeviceLayer(cfg, seed, fmts, storage, experts, x, lg, x_host, logits_host, unpadded, grid)
