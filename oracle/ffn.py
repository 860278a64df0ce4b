"""The routed MoE FFN layer, fp64. Test infrastructure.

Sources: "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南"
(section 瓶颈分析: each token runs the FFN of the k experts its router picked;
section 优化策略三: decode fuses the gate and up mat-muls with the activation;
section 优化策略二: per-expert formats, three tiers in one layer) and "一张 RTX
3090 跑 Llama 70B：三层流式缓存 + NVMe 直连" (section 4.4: SwiGLU activation).

Readings taken where the pages are silent:

* Expert e: g = W_gate[e] x, u = W_up[e] x (W_gate, W_up are [I, H]),
  h = silu(g) * u with silu(z) = z / (1 + exp(-z)), y = W_down[e] h (W_down is
  [H, I]). The activation is applied to the gate branch.
* The router weight scales the expert's down-projection output, and
  out[t] = sum over slots j = 0..k-1, in ascending j, of w[t, j] * y_{t,j}.
* x is the exact bf16 value; every weight is the exact decoded value; all
  arithmetic is fp64.
* Shared experts ("多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出
  120 t/s", memory layout: the model keeps shared experts beside the routed
  ones, stored there in Q8_0) run on every token with weight 1 and are added
  after the routed experts: with S shared experts as entries E .. E+S-1 of the
  expert list, slot k + s of every token holds expert E + s, weight 1, and the
  ascending-slot sum runs over all k + S slots. The expert-range and format
  filters apply to them like to any expert.

Experts are given as a list of mappings with keys "gate", "up", "down"; each
value has attributes fmt, rows, cols, stride and data (uint8 bytes).
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from . import formats, router, bucket as bucket_mod


def bf16_bits_to_f64(xb: np.ndarray) -> np.ndarray:
    u = np.asarray(xb, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def dense(m) -> np.ndarray:
    """A matrix (attributes fmt, rows, cols, stride, data; IQ3_XXS matrices also
    carry their grid) -> fp64 [rows, cols]."""
    return formats.dequant_matrix(m.fmt, m.rows, m.cols, m.stride, m.data, getattr(m, "grid", None))


class DenseCache:
    """Decodes each expert's matrices at most once."""

    def __init__(self, experts):
        self.experts = experts
        self._d: Dict[int, tuple] = {}

    def __call__(self, e: int):
        if e not in self._d:
            ex = self.experts[e]
            self._d[e] = (dense(ex["gate"]), dense(ex["up"]), dense(ex["down"]))
        return self._d[e]


def expert_forward(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, x: np.ndarray):
    """x fp64 [n, H] -> (g, u, h [n, I], y [n, H])."""
    g = x @ Wg.T
    u = x @ Wu.T
    h = silu(g) * u
    y = h @ Wd.T
    return g, u, h, y


def token_slots(logits: np.ndarray, k: int, renormalize: bool, n_shared: int):
    """Every token's slots: (ids [T, k + S], weights [T, k + S]): the router's
    k experts, then the S shared experts E .. E+S-1 with weight 1."""
    ids, w, _ = router.route_topk(logits, k, renormalize)
    if n_shared == 0:
        return ids, w
    T, E = logits.shape
    sid = np.broadcast_to(np.arange(E, E + n_shared, dtype=ids.dtype), (T, n_shared))
    return np.concatenate([ids, sid], axis=1), np.concatenate([w, np.ones((T, n_shared), w.dtype)], axis=1)


def _check_entries(experts, logits, n_shared):
    if not 0 <= n_shared or len(experts) != logits.shape[1] + n_shared:
        raise ValueError("the expert list must hold the E routed experts, then the n_shared shared ones")


def moe_ffn(experts, x_bf16: np.ndarray, logits: np.ndarray, k: int, renormalize: bool = True,
            expert_lo: int = 0, expert_hi: Optional[int] = None, format_mask: int = 0xFFFFFFFF,
            tokens: Optional[Sequence[int]] = None, cache: Optional[DenseCache] = None,
            gate_formats: Optional[Sequence[int]] = None, n_shared: int = 0):
    """Layer output fp64 [len(tokens) or T, H].

    Routing (router.route_topk) and bucketing (bucket.bucket) run on all T
    tokens; ``tokens`` only restricts which output rows are evaluated.
    ``experts`` may be any indexable of length E + n_shared (e.g. a lazy
    generator): the E routed experts, then the shared ones; only the experts
    that are routed to are read. ``gate_formats`` (format tag of each expert's
    gate matrix) is needed by the format filter; by default it is read from
    every expert."""
    x = bf16_bits_to_f64(x_bf16)
    T, H = x.shape
    _check_entries(experts, logits, n_shared)
    E = len(experts)
    ids, w = token_slots(logits, k, renormalize, n_shared)
    k = k + n_shared
    if gate_formats is None:
        gate_formats = [experts[e]["gate"].fmt for e in range(E)]
    _, _, pos, _, _ = bucket_mod.bucket(ids, E, expert_lo, expert_hi, format_mask, gate_formats)
    cache = cache or DenseCache(experts)
    tok = list(range(T)) if tokens is None else [int(t) for t in tokens]
    out = np.zeros((len(tok), H), dtype=np.float64)
    for row, t in enumerate(tok):
        for j in range(k):                      # ascending slot order
            if pos[t * k + j] < 0:
                continue
            Wg, Wu, Wd = cache(int(ids[t, j]))
            _, _, _, y = expert_forward(Wg, Wu, Wd, x[t:t + 1])
            out[row] += w[t, j] * y[0]
    return out


def _expert_job(job):
    """(experts, e, xr [n, H] fp64) -> y [n, H]: expert e on the rows xr."""
    experts, e, xr = job
    ex = experts[e]
    Wg, Wu, Wd = dense(ex["gate"]), dense(ex["up"]), dense(ex["down"])
    release = getattr(experts, "release", None)
    if release is not None:
        release(e)
    return expert_forward(Wg, Wu, Wd, xr)[3]


def moe_ffn_by_expert(experts, x_bf16: np.ndarray, logits: np.ndarray, k: int, renormalize: bool = True,
                      expert_lo: int = 0, expert_hi: Optional[int] = None, format_mask: int = 0xFFFFFFFF,
                      tokens: Optional[Sequence[int]] = None,
                      gate_formats: Optional[Sequence[int]] = None, map_fn=map, n_shared: int = 0):
    """The same layer output as ``moe_ffn``, evaluated one expert at a time:
    every routed pair of the wanted tokens is grouped by its expert, each
    expert's matrices are decoded once, applied to all of its rows, and
    dropped, so memory stays at one expert's dense matrices (per worker)
    whatever the layer size. The combine is the same ascending-slot sum.
    ``map_fn`` maps the per-expert jobs (``map``, or a process pool's map; the
    jobs carry ``experts`` and must then be picklable)."""
    x = bf16_bits_to_f64(x_bf16)
    T, H = x.shape
    _check_entries(experts, logits, n_shared)
    E = len(experts)
    ids, w = token_slots(logits, k, renormalize, n_shared)
    k = k + n_shared
    if gate_formats is None:
        gate_formats = [experts[e]["gate"].fmt for e in range(E)]
    _, _, pos, _, _ = bucket_mod.bucket(ids, E, expert_lo, expert_hi, format_mask, gate_formats)
    tok = list(range(T)) if tokens is None else [int(t) for t in tokens]
    by_expert: Dict[int, list] = {}
    for t in sorted(set(tok)):
        for j in range(k):
            if pos[t * k + j] >= 0:
                by_expert.setdefault(int(ids[t, j]), []).append((t, j))
    order = sorted(by_expert)
    jobs = [(experts, e, x[[t for t, _ in by_expert[e]]]) for e in order]
    y = {}
    for e, ye in zip(order, map_fn(_expert_job, jobs)):
        for (t, j), row in zip(by_expert[e], ye):
            y[(t, j)] = row
    out = np.zeros((len(tok), H), dtype=np.float64)
    for row, t in enumerate(tok):
        for j in range(k):                      # ascending slot order
            if (t, j) in y:
                out[row] += w[t, j] * y[(t, j)]
    return out


def moe_ffn_bruteforce(experts, x_bf16: np.ndarray, logits: np.ndarray, k: int,
                       renormalize: bool = True, n_shared: int = 0) -> np.ndarray:
    """Independent second evaluation for small layers: every expert on every
    token (dense fp64 matrices), then a dense [T, E + S] routing-weight matrix
    selects and weights the results (the shared experts' columns are all
    ones). Shares only the decoders and the router with ``moe_ffn``; no
    bucketing, no per-pair loop, no slot list."""
    x = bf16_bits_to_f64(x_bf16)
    T, H = x.shape
    _check_entries(experts, logits, n_shared)
    E = len(experts)
    ids, w, _ = router.route_topk(logits, k, renormalize)
    R = np.zeros((T, E), dtype=np.float64)
    R[:, E - n_shared:] = 1.0
    for t in range(T):
        for j in range(k):
            R[t, ids[t, j]] += w[t, j]
    Y = np.empty((E, T, H), dtype=np.float64)
    for e in range(E):
        Wg, Wu, Wd = dense(experts[e]["gate"]), dense(experts[e]["up"]), dense(experts[e]["down"])
        Y[e] = (silu(x @ Wg.T) * (x @ Wu.T)) @ Wd.T
    return np.einsum("te,eth->th", R, Y)
