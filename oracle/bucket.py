"""Token -> expert bucketing. Integer; test infrastructure.

Source: "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南",
section 优化策略三 (the tiered mul_mat_id keeps only ids inside
[min_expert_id, max_expert_id) and skips the rest) and section 关键 Bug 修复与调试
踩坑记录 (bug 1: redirecting skipped ids to expert 0 duplicated it within a token
and broke the expert grouping; bug 3: the -1 skip id must never be promoted to
an unsigned index).

A pair is (token t, slot j), numbered p = t*k + j. Readings taken:

* ids == -1 means "no expert" and is skipped silently.
* Any other id outside [0, E) is an error: flagged, and the pair skipped.
* A pair is kept only if expert_lo <= id < expert_hi and bit (1 << fmt) of
  format_mask is set, where fmt is the format tag of the expert's gate matrix
  (its tier). Dropped pairs contribute nothing.
* Within an expert, pairs are listed in ascending p; experts in ascending id.
* An id repeated within one token (impossible from the router) is flagged; the
  pairs are still bucketed as ordinary pairs.

Outputs: offsets [E+1] (exclusive prefix sum of per-expert counts), pairs
[n_kept] (pair numbers in bucket order), pos [T*k] (bucket position of each
pair, -1 if dropped), active (expert ids with a non-zero count, ascending).
"""
from __future__ import annotations

import numpy as np

FLAG_BAD_ID = 2
FLAG_DUPLICATE_ID = 4


def bucket(ids: np.ndarray, n_experts: int, expert_lo: int = 0, expert_hi: int = None,
           format_mask: int = 0xFFFFFFFF, gate_formats=None):
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    E = n_experts
    if expert_hi is None:
        expert_hi = E
    flags = 0
    flat = ids.reshape(-1)
    keep = np.zeros(flat.shape[0], dtype=bool)
    for p, e in enumerate(flat):
        if e == -1:
            continue
        if e < 0 or e >= E:
            flags |= FLAG_BAD_ID
            continue
        if not (expert_lo <= e < expert_hi):
            continue
        if gate_formats is not None and not ((format_mask >> int(gate_formats[e])) & 1):
            continue
        keep[p] = True
    for t in range(T):
        row = [int(e) for e in ids[t] if 0 <= e < E]
        if len(set(row)) != len(row):
            flags |= FLAG_DUPLICATE_ID
    counts = np.zeros(E, dtype=np.int64)
    for p in np.nonzero(keep)[0]:
        counts[flat[p]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    pairs = np.empty(int(offsets[-1]), dtype=np.int64)
    pos = np.full(flat.shape[0], -1, dtype=np.int64)
    for p in range(flat.shape[0]):          # ascending p -> stable within expert
        if keep[p]:
            e = flat[p]
            pairs[fill[e]] = p
            pos[p] = fill[e]
            fill[e] += 1
    active = np.nonzero(counts)[0]
    return (offsets.astype(np.int32), pairs.astype(np.int32), pos.astype(np.int32),
            active.astype(np.int32), flags)
