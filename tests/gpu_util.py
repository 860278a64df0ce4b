"""Helpers of the GPU tests: build the library, move seeded layers to the
device, compare with the oracle. Imported by test modules only."""
from __future__ import annotations

import contextlib
import os

import numpy as np
import torch

import synth

# Parity bar for the FFN output: relative L2 error <= 1e-3 and max abs error
# <= 1e-2 * RMS of the oracle output (RMS and norms over the whole [T, H]).
REL_L2_TOL = 1e-3
MAX_ABS_RMS_TOL = 1e-2
# Router weights: |w_gpu - w_oracle| <= 4e-6 * w_oracle (+ 1e-12 for zero weights).
W_REL_TOL = 4e-6


def ensure_built():
    import __graft_entry__
    __graft_entry__.build()


def host_layer_to_device(L: synth.SynthLayer):
    """SynthLayer (host bytes) -> (experts for WeightTable, x bf16, logits) on the device."""
    experts = []
    for ex in L.experts:
        d = {}
        for name in ("gate", "up", "down"):
            m = ex[name]
            d[name] = (m.fmt, m.rows, m.cols, m.stride, torch.from_numpy(m.data.copy()).to("cuda"))
        experts.append(d)
    x = torch.from_numpy(L.x_bf16.view(np.int16).copy()).to("cuda").view(torch.bfloat16)
    logits = torch.from_numpy(L.logits.copy()).to("cuda")
    return experts, x, logits


def parity_errors(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = gpu - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    mx = np.abs(diff).max() if diff.size else 0.0
    return rel, mx, rms


def assert_parity(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    rel, mx, rms = parity_errors(gpu, ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    if rms == 0:
        assert mx == 0, f"{what}: expected all zeros, max abs {mx}"
        return
    assert rel <= REL_L2_TOL, f"{what}: rel-L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAX_ABS_RMS_TOL * rms, f"{what}: max abs {mx:.3e} > {MAX_ABS_RMS_TOL} * rms {rms:.3e}"


# ------------------------------------------------------------------ full-size oracle
_ORACLE_CACHE = {}


@contextlib.contextmanager
def oracle_pool():
    """A spawned process pool for the oracle's per-expert jobs (spawned, so it
    is safe after CUDA work in this process), one BLAS thread per worker."""
    import multiprocessing as mp
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        pool = mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield pool
    finally:
        pool.close()
        pool.join()


def oracle_full_layer(cfg: synth.LayerConfig, DL, tokens=None) -> np.ndarray:
    """The oracle's output of a device-filled layer (synth.gpu.DeviceLayer) for
    `tokens` (default: all), expert by expert over a process pool; cached per
    (config, seed, tokens) for the session."""
    from oracle import ffn as offn
    key = (cfg.name, DL.seed, DL.x_host.shape[0], None if tokens is None else tuple(tokens))
    if key not in _ORACLE_CACHE:
        lazy = synth.LazyExperts(cfg, DL.seed, DL.fmts)
        with oracle_pool() as pool:
            _ORACLE_CACHE[key] = offn.moe_ffn_by_expert(lazy, DL.x_host, DL.logits_host, cfg.k, tokens=tokens,
                                                        gate_formats=lazy.gate_formats(), map_fn=pool.map,
                                                        n_shared=cfg.n_shared)
    return _ORACLE_CACHE[key]
