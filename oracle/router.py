"""Router: softmax over the experts, then top-k. fp64. Test infrastructure.

Source: "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南",
section 瓶颈分析 (a light router picks, per token, the 10 best-matching of the
layer's 512 experts). The page gives no equations; readings taken:

* Selection key: the raw fp32 logit, largest first; equal logits go to the
  lower expert index. Softmax is monotone, so this is the top-k of the
  probabilities, and comparing logits keeps the choice exact.
* Non-finite logits (NaN, +-inf) rank below every finite logit (ties among them
  by index again) and have probability 0; a row without a finite logit gets
  weight 0 in every slot. Such rows are flagged.
* Weights: the softmax over all E experts in fp64, then (default) the k
  selected probabilities renormalised to sum to 1; ``renormalize=False`` keeps
  the plain selected probabilities.
* Slot order: descending logit (slot 0 is the best expert).
"""
from __future__ import annotations

import numpy as np


def softmax_row(logits_row: np.ndarray) -> np.ndarray:
    """fp64 softmax over the finite entries; non-finite entries get 0."""
    v = np.asarray(logits_row, dtype=np.float64)
    finite = np.isfinite(v)
    p = np.zeros_like(v)
    if not finite.any():
        return p
    m = v[finite].max()
    ex = np.exp(v[finite] - m)
    p[finite] = ex / ex.sum()
    return p


def topk_order(logits_row: np.ndarray) -> np.ndarray:
    """Expert indices ordered by (logit descending, index ascending), with
    non-finite logits last (by index)."""
    v = np.asarray(logits_row, dtype=np.float64)
    key = np.where(np.isfinite(v), v, -np.inf)
    # lexsort: last key is primary -> primary = -key, secondary = index
    return np.lexsort((np.arange(v.shape[0]), -key))


def route_topk(logits: np.ndarray, k: int, renormalize: bool = True):
    """logits fp32 [T, E] -> (ids int32 [T, k], weights fp64 [T, k], flags).

    ``flags`` is a bool [T] marking rows that held a non-finite logit."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError(f"need 1 <= k <= E, got k={k}, E={E}")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    flags = np.zeros(T, dtype=bool)
    for t in range(T):
        row = logits[t]
        flags[t] = not np.isfinite(row).all()
        sel = topk_order(row)[:k]
        p = softmax_row(row)
        ps = p[sel]
        if renormalize:
            s = ps.sum()
            ps = ps / s if s > 0 else np.zeros_like(ps)
        ids[t] = sel
        w[t] = ps
    return ids, w, flags
