"""ctypes binding of libmoe_route.so (C ABI: include/moe_route.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. If the
shared library is missing this module raises; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_route.so")

Q8_0, Q4_K, Q6_K, MXFP4, IQ4_NL, IQ4_XS, IQ3_XXS, T5_G128 = 1, 2, 3, 4, 5, 6, 7, 8
BLOCK_ELEMS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, MXFP4: 32, IQ4_NL: 32, IQ4_XS: 256, IQ3_XXS: 256, T5_G128: 128}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, MXFP4: 17, IQ4_NL: 18, IQ4_XS: 136, IQ3_XXS: 98, T5_G128: 28}

MOE_OK = 0
MOE_TABLE_PREPARED = 0x4D4F4554
PATH_AUTO, PATH_GEMV, PATH_TENSOR, PATH_FUSED = 0, 1, 2, 3
GEMV_TILED, GEMV_STREAMING = 0, 1
FLAG_NONFINITE_LOGIT, FLAG_BAD_ID, FLAG_DUPLICATE_ID, FLAG_WAIT_TIMEOUT = 1, 2, 4, 8

EXPORTED = [
    "moe_strerror", "moe_last_cuda_error", "moe_table_device_bytes", "moe_table_prepare",
    "moe_route_topk", "moe_bucket", "moe_ffn_workspace_size", "moe_ffn_workspace_init",
    "moe_ffn_forward", "moe_ffn_read_status", "moe_ffn_workspace_views", "moe_ffn_forward_noalloc",
    "moe_ffn_path", "moe_ffn_gemv_kernels", "moe_ffn_workspace_size_for_path", "moe_sum_partials",
    "moe_set_wait_timeout_ns",
]
NOALLOC_SCRATCH_BYTES = 4 << 20


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        super().__init__(f"{fn} failed: {code} ({detail})")
        self.code = code


class Matrix(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("rows", ctypes.c_int32), ("cols", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("row_stride_bytes", ctypes.c_int64), ("data", ctypes.c_void_p)]


class Expert(ctypes.Structure):
    _fields_ = [("gate", Matrix), ("up", Matrix), ("down", Matrix)]


class WeightTableC(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("experts", ctypes.POINTER(Expert)),
                ("device_table", ctypes.c_void_p), ("formats_present", ctypes.c_uint32),
                ("prepared", ctypes.c_uint32), ("gateup_formats", ctypes.c_uint32),
                ("down_formats", ctypes.c_uint32), ("max_gateup_stride", ctypes.c_int64),
                ("max_down_stride", ctypes.c_int64), ("uniform_layout", ctypes.c_int32),
                ("tc_maps", ctypes.c_int32), ("uniform_base", Expert),
                ("uniform_step", ctypes.c_int64 * 3), ("iq3_grid", ctypes.c_void_p), ("n_cold", ctypes.c_int32),
                ("reserved2", ctypes.c_int32), ("cold_bytes_max", ctypes.c_int64)]


class Options(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("renormalize", ctypes.c_int32),
                ("format_mask", ctypes.c_uint32), ("expert_lo", ctypes.c_int32),
                ("expert_hi", ctypes.c_int32), ("path", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("timing_events", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
    L.moe_strerror.argtypes, L.moe_strerror.restype = [ctypes.c_int], ctypes.c_char_p
    L.moe_last_cuda_error.argtypes, L.moe_last_cuda_error.restype = [], ctypes.c_int
    L.moe_table_device_bytes.argtypes, L.moe_table_device_bytes.restype = [i32], sz
    L.moe_table_prepare.argtypes = [ctypes.POINTER(WeightTableC), vp, sz, vp]
    L.moe_route_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp]
    L.moe_bucket.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    L.moe_ffn_workspace_size.argtypes = [ctypes.POINTER(WeightTableC), i32, i32]
    L.moe_ffn_workspace_size.restype = sz
    L.moe_ffn_workspace_size_for_path.argtypes = [ctypes.POINTER(WeightTableC), i32, i32, i32]
    L.moe_ffn_workspace_size_for_path.restype = sz
    L.moe_ffn_workspace_init.argtypes = [vp, sz, vp]
    L.moe_ffn_forward.argtypes = [ctypes.POINTER(WeightTableC), vp, vp, i32, i32, ctypes.POINTER(Options),
                                  vp, vp, sz, vp]
    L.moe_ffn_read_status.argtypes = [vp, ctypes.POINTER(u32), vp]
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.moe_ffn_workspace_views.argtypes = [ctypes.POINTER(WeightTableC), i32, i32, vp, pp, pp, pp, pp, pp, pp]
    L.moe_ffn_path.argtypes = [ctypes.POINTER(WeightTableC), i32, i32, ctypes.POINTER(Options)]
    L.moe_ffn_path.restype = ctypes.c_int
    L.moe_ffn_gemv_kernels.argtypes = [ctypes.POINTER(WeightTableC), i32, i32]
    L.moe_ffn_gemv_kernels.restype = ctypes.c_int
    L.moe_ffn_forward_noalloc.argtypes = [ctypes.POINTER(WeightTableC), vp, vp, i32, i32, ctypes.POINTER(Options),
                                          vp, vp]
    L.moe_sum_partials.argtypes = [vp, i32, ctypes.c_int64, vp, vp]
    L.moe_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    for name in ("moe_table_prepare", "moe_route_topk", "moe_bucket", "moe_ffn_workspace_init",
                 "moe_ffn_forward", "moe_ffn_read_status", "moe_ffn_workspace_views", "moe_ffn_forward_noalloc",
                 "moe_sum_partials", "moe_set_wait_timeout_ns"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(fn: str, rc: int) -> None:
    if rc != MOE_OK:
        L = load()
        raise MoeError(fn, rc, L.moe_strerror(rc).decode() + f"; cuda error {L.moe_last_cuda_error()}")


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev(t: torch.Tensor, name: str, dtype=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# ----------------------------------------------------------------------------
class WeightTable:
    """A prepared per-expert format-tagged weight table.

    ``experts`` is a sequence of dicts with keys "gate", "up", "down"; each value
    is a tuple (format, rows, cols, row_stride_bytes, uint8 CUDA tensor). The
    tensors are kept alive by this object."""

    def __init__(self, experts: Sequence[dict], hidden: int, inter: int, stream=None,
                 grid: Optional[torch.Tensor] = None, n_shared: int = 0):
        """experts: per expert {"gate"|"up"|"down": (fmt, rows, cols, stride, uint8 CUDA tensor)},
        the routed experts followed by the ``n_shared`` shared experts (run on
        every token with weight 1); grid: the IQ3_XXS grid (256 x 32-bit CUDA
        tensor), needed when a matrix is IQ3_XXS."""
        L = load()
        E = len(experts)
        if not 0 <= n_shared < E:
            raise ValueError(f"bad shared-expert count {n_shared} for {E} experts")
        self.n_entries, self.n_shared = E, n_shared
        self.n_experts, self.hidden, self.inter = E - n_shared, hidden, inter
        self._keep: List[torch.Tensor] = []
        arr = (Expert * E)()
        for e, ex in enumerate(experts):
            for name in ("gate", "up", "down"):
                fmt, rows, cols, stride, data = ex[name]
                if data.is_cuda:
                    _dev(data, f"expert {e} {name}", torch.uint8)
                elif not (data.is_pinned() and data.dtype == torch.uint8 and data.is_contiguous()):
                    raise ValueError(f"expert {e} {name}: a CUDA tensor, or a pinned host tensor (cold tier)")
                self._keep.append(data)
                setattr(arr[e], name, Matrix(fmt, rows, cols, 0, stride, data.data_ptr()))
        self._arr = arr
        self.c = WeightTableC(E - n_shared, hidden, inter, n_shared, ctypes.cast(arr, ctypes.POINTER(Expert)))
        if grid is not None:
            if grid.numel() != 256 or grid.element_size() != 4:
                raise ValueError("grid must hold 256 32-bit entries")
            _dev(grid, "grid")
            self._keep.append(grid)
            self.c.iq3_grid = grid.data_ptr()
        nbytes = L.moe_table_device_bytes(E)
        if nbytes == 0:
            raise ValueError(f"bad expert count {E}")
        self.device_buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        _check("moe_table_prepare", L.moe_table_prepare(ctypes.byref(self.c), _ptr(self.device_buf), nbytes,
                                                        _stream(stream)))
        self.gate_formats = [ex["gate"][0] for ex in experts]

    @property
    def formats_present(self) -> int:
        return self.c.formats_present


class Workspace:
    """Device workspace of moe_ffn_forward for (table, T, k), zero-initialised."""

    def __init__(self, table: WeightTable, T: int, k: int, stream=None, path: int = 0):
        """path: size for that MOE_PATH_* (0 = the one AUTO picks)."""
        L = load()
        self.table, self.T, self.k = table, T, k
        self.nbytes = L.moe_ffn_workspace_size_for_path(ctypes.byref(table.c), T, k, path)
        if self.nbytes == 0:
            raise ValueError("bad workspace arguments")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device="cuda")
        _check("moe_ffn_workspace_init", L.moe_ffn_workspace_init(_ptr(self.buf), self.nbytes, _stream(stream)))

    def routing(self) -> dict:
        """Views (CUDA tensors) of the routing results of the last forward:
        ids [T, k+S], weights [T, k+S], offsets [E+S+1], active [E+S+1],
        pairs, pos [T*(k+S)] (S shared experts: slots k.. of every token)."""
        L = load()
        ptrs = [ctypes.c_void_p() for _ in range(6)]
        _check("moe_ffn_workspace_views", L.moe_ffn_workspace_views(
            ctypes.byref(self.table.c), self.T, self.k, _ptr(self.buf), *[ctypes.byref(p) for p in ptrs]))
        base = self.buf.data_ptr()
        T, k, E = self.T, self.k + self.table.n_shared, self.table.n_entries

        def view(p, n, dtype):
            off = p.value - base
            return self.buf[off:off + 4 * n].view(dtype)
        return {"ids": view(ptrs[0], T * k, torch.int32).view(T, k),
                "weights": view(ptrs[1], T * k, torch.float32).view(T, k),
                "offsets": view(ptrs[2], E + 1, torch.int32), "active": view(ptrs[3], E + 1, torch.int32),
                "pairs": view(ptrs[4], T * k, torch.int32), "pos": view(ptrs[5], T * k, torch.int32)}

    def read_status(self, stream=None) -> int:
        L = load()
        v = ctypes.c_uint32(0)
        _check("moe_ffn_read_status", L.moe_ffn_read_status(_ptr(self.buf), ctypes.byref(v), _stream(stream)))
        return v.value


def route_topk(logits: torch.Tensor, k: int, renormalize: bool = True, status: Optional[torch.Tensor] = None,
               ids: Optional[torch.Tensor] = None, weights: Optional[torch.Tensor] = None, stream=None):
    """logits fp32 [T, E] (CUDA) -> (ids int32 [T, k], weights fp32 [T, k])."""
    _dev(logits, "logits", torch.float32)
    T, E = logits.shape
    ids = ids if ids is not None else torch.empty((T, k), dtype=torch.int32, device=logits.device)
    weights = weights if weights is not None else torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check("moe_route_topk", load().moe_route_topk(_ptr(logits), T, E, k, int(renormalize), _ptr(ids),
                                                    _ptr(weights), _ptr(status), _stream(stream)))
    return ids, weights


def bucket(ids: torch.Tensor, n_experts: int, expert_lo: int = 0, expert_hi: Optional[int] = None,
           status: Optional[torch.Tensor] = None, stream=None):
    """ids int32 [T, k] (CUDA) -> (offsets [E+1], pairs [T*k], pos [T*k], active [E+1])."""
    _dev(ids, "ids", torch.int32)
    T, k = ids.shape
    E = n_experts
    hi = E if expert_hi is None else expert_hi
    dev = ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pairs = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    pos = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    active = torch.empty(E + 1, dtype=torch.int32, device=dev)
    _check("moe_bucket", load().moe_bucket(_ptr(ids), T, k, E, expert_lo, hi, _ptr(offsets), _ptr(pairs),
                                            _ptr(pos), _ptr(active), _ptr(status), _stream(stream)))
    return offsets, pairs[: T * k], pos[: T * k], active


def ffn_path(table: "WeightTable", T: int, k: int, options: Optional[Options] = None) -> int:
    """The path moe_ffn_forward takes (PATH_GEMV / PATH_TENSOR / PATH_FUSED), -1 if none."""
    opt = ctypes.byref(options) if options is not None else None
    return load().moe_ffn_path(ctypes.byref(table.c), T, k, opt)


def gemv_kernels(table: "WeightTable", T: int, k: int) -> int:
    """GEMV_STREAMING or GEMV_TILED: the kernels the grouped GEMV path runs; -1 if invalid."""
    return load().moe_ffn_gemv_kernels(ctypes.byref(table.c), T, k)


def make_options(renormalize: bool = True, format_mask: int = 0xFFFFFFFF, expert_lo: int = 0,
                 expert_hi: Optional[int] = None, n_experts: int = 0, path: int = PATH_AUTO,
                 timing_events: Optional[Sequence["torch.cuda.Event"]] = None) -> Options:
    """Options of ffn_forward. ``n_experts``: the table length (WeightTable.n_entries,
    routed + shared), the default expert_hi. ``timing_events``: 3 torch.cuda.Event
    (enable_timing) recorded before the gate/up kernel, between gate/up and down,
    after down."""
    hi = n_experts if expert_hi is None else expert_hi
    o = Options(ctypes.sizeof(Options), int(renormalize), format_mask & 0xFFFFFFFF, expert_lo, hi, path, 0, None)
    if timing_events is not None:
        if len(timing_events) != 3:
            raise ValueError("timing_events needs 3 events")
        for ev in timing_events:
            if ev.cuda_event == 0:        # torch creates the CUDA event on first record
                ev.record(torch.cuda.current_stream())
        torch.cuda.current_stream().synchronize()
        arr = (ctypes.c_void_p * 3)(*[ev.cuda_event for ev in timing_events])
        o._events_keep = (arr, list(timing_events))
        o.timing_events = ctypes.cast(arr, ctypes.c_void_p)
    return o


def ffn_forward(table: WeightTable, x_bf16: torch.Tensor, logits: torch.Tensor, k: int,
                out: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None,
                options: Optional[Options] = None, stream=None) -> torch.Tensor:
    """The whole layer. x bf16 [T, H], logits fp32 [T, E] (CUDA) -> out fp32 [T, H]."""
    if x_bf16.dtype == torch.bfloat16:
        x_bits = x_bf16.view(torch.int16)
    else:
        x_bits = x_bf16
    _dev(x_bits, "x", torch.int16)
    _dev(logits, "logits", torch.float32)
    T, H = x_bits.shape
    if H != table.hidden or logits.shape != (T, table.n_experts):
        raise ValueError("x / logits shape does not match the table")
    out = out if out is not None else torch.empty((T, H), dtype=torch.float32, device=x_bits.device)
    _dev(out, "out", torch.float32)
    if ws is None:
        # sized for the requested path; for a path that cannot run this layer,
        # for AUTO's, so that the forward itself reports the refusal
        path = options.path if options is not None else 0
        if path and load().moe_ffn_workspace_size_for_path(ctypes.byref(table.c), T, k, path) == 0:
            path = 0
        ws = Workspace(table, T, k, stream, path=path)
    opt = ctypes.byref(options) if options is not None else None
    _check("moe_ffn_forward", load().moe_ffn_forward(ctypes.byref(table.c), _ptr(x_bits), _ptr(logits), T, k,
                                                      opt, _ptr(out), _ptr(ws.buf), ws.nbytes, _stream(stream)))
    return out


def ffn_forward_noalloc(table: WeightTable, x_bf16: torch.Tensor, logits: torch.Tensor, k: int,
                        out: Optional[torch.Tensor] = None, options: Optional[Options] = None,
                        stream=None) -> torch.Tensor:
    """The whole layer without a workspace argument (moe_ffn_forward_noalloc):
    the library keeps the scratch in its own fixed 4 MiB device array, for
    callers that cannot allocate device memory. Calls share that array, so
    calls that overlap on the GPU race; keep them on one stream. Sizes whose
    workspace would exceed 4 MiB raise MoeError (code 8)."""
    x_bits = x_bf16.view(torch.int16) if x_bf16.dtype == torch.bfloat16 else x_bf16
    _dev(x_bits, "x", torch.int16)
    _dev(logits, "logits", torch.float32)
    T, H = x_bits.shape
    if H != table.hidden or logits.shape != (T, table.n_experts):
        raise ValueError("x / logits shape does not match the table")
    out = out if out is not None else torch.empty((T, H), dtype=torch.float32, device=x_bits.device)
    _dev(out, "out", torch.float32)
    opt = ctypes.byref(options) if options is not None else None
    _check("moe_ffn_forward_noalloc", load().moe_ffn_forward_noalloc(
        ctypes.byref(table.c), _ptr(x_bits), _ptr(logits), T, k, opt, _ptr(out), _stream(stream)))
    return out


def noalloc_read_status(stream=None) -> int:
    """Read and clear the device status flags (FLAG_*) that calls of
    ffn_forward_noalloc accumulated in the library's array on the current
    device (moe_ffn_read_status with a NULL workspace). Synchronises."""
    v = ctypes.c_uint32(0)
    _check("moe_ffn_read_status", load().moe_ffn_read_status(None, ctypes.byref(v), _stream(stream)))
    return v.value


def sum_partials(parts: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """parts fp32 [n, ...] (CUDA, contiguous) -> out fp32 [...] = sum over n in
    ascending order, one fp32 add at a time (moe_sum_partials)."""
    _dev(parts, "parts", torch.float32)
    n = parts.shape[0]
    out = out if out is not None else torch.empty(parts.shape[1:], dtype=torch.float32, device=parts.device)
    _dev(out, "out", torch.float32)
    _check("moe_sum_partials", load().moe_sum_partials(_ptr(parts), n, parts[0].numel(), _ptr(out),
                                                        _stream(stream)))
    return out


def set_wait_timeout_ns(ns: int = 0) -> None:
    """Bound (ns) on the kernels' device-side waits (0: the default, 2 s);
    see moe_set_wait_timeout_ns."""
    _check("moe_set_wait_timeout_ns", load().moe_set_wait_timeout_ns(int(ns)))
