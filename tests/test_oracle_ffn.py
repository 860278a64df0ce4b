"""Pins of the oracle FFN layer (CPU only).

* Closed form: Q8_0 experts whose matrices are a permutation matrix, the
  identity and twice the identity give out = w0*silu(Px)*x + w1*silu(x)*2x.
  This fixes the matrix orientation, the branch that takes the activation, and
  how the router weights enter.
* Brute force: every expert on every token through dense matrices, then
  selection by a dense routing matrix, equals the per-pair evaluation.
* Mixed tiers: the full mixed-format layer equals the sum of format-masked
  runs (one tier at a time), and an expert-range split sums back to the whole.
* Permutation: permuting the expert table together with the logit columns
  leaves the output unchanged.
* All-zero scales give a zero output.
"""
import numpy as np
import pytest

import synth
from oracle import ffn, formats
from synth import MatrixBytes


def q8_0_matrix(Q: np.ndarray, d: float = 1.0) -> MatrixBytes:
    """Integer matrix [rows, cols] (|q| <= 127) -> Q8_0 bytes with scale d."""
    rows, cols = Q.shape
    nb = cols // 32
    stride = synth.padded_stride(synth.Q8_0, cols)
    data = np.zeros((rows, stride), np.uint8)
    dbytes = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    for r in range(rows):
        for b in range(nb):
            data[r, 34 * b: 34 * b + 2] = dbytes
            data[r, 34 * b + 2: 34 * b + 34] = Q[r, 32 * b: 32 * b + 32].astype(np.int8).view(np.uint8)
    return MatrixBytes(synth.Q8_0, rows, cols, stride, data.reshape(-1))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    return synth.f32_to_bf16_bits(x.astype(np.float32))


def small_layer(tiers="mixed", E=12, k=3, H=256, I=64, T=5, seed=77, bias=True):
    cfg = synth.LayerConfig("t", E, k, H, I, T, tiers, bias, seed)
    return synth.make_layer(cfg, 0)


def test_closed_form_identity_experts():
    n = 32
    P = np.roll(np.eye(n, dtype=np.int64), 5, axis=1)          # (Px)_i = x_{i+5 mod n}
    Id = np.eye(n, dtype=np.int64)
    experts = [
        {"gate": q8_0_matrix(P), "up": q8_0_matrix(Id), "down": q8_0_matrix(Id)},
        {"gate": q8_0_matrix(Id), "up": q8_0_matrix(2 * Id), "down": q8_0_matrix(Id)},
    ]
    rng = np.random.default_rng(30)
    x = rng.standard_normal((3, n))
    xb = bf16_bits(x)
    xq = ffn.bf16_bits_to_f64(xb)
    logits = np.array([[1.0, 0.25], [-0.5, 0.75], [0.0, 0.0]], np.float32)
    out = ffn.moe_ffn(experts, xb, logits, k=2)
    l = logits.astype(np.float64)
    for t in range(3):
        w0 = np.exp(l[t, 0]) / np.exp(l[t]).sum()
        y0 = ffn.silu(xq[t] @ P.T) * xq[t]
        y1 = ffn.silu(xq[t]) * 2 * xq[t]
        np.testing.assert_allclose(out[t], w0 * y0 + (1 - w0) * y1, rtol=1e-13, atol=1e-15)
    # k = 1 keeps only the best expert with weight 1
    out1 = ffn.moe_ffn(experts, xb[:2], logits[:2], k=1)
    np.testing.assert_allclose(out1[0], ffn.silu(xq[0] @ P.T) * xq[0], rtol=1e-14)
    np.testing.assert_allclose(out1[1], ffn.silu(xq[1]) * 2 * xq[1], rtol=1e-14)


def test_silu_values():
    z = np.array([0.0, 1.0, -1.0, 40.0, -800.0])
    s = ffn.silu(z)
    assert s[0] == 0.0
    np.testing.assert_allclose(s[1], 1 / (1 + np.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(s[2], -1 / (1 + np.e), rtol=1e-15)
    np.testing.assert_allclose(s[3], 40.0, rtol=1e-15)
    assert s[4] == 0.0


def test_tiny_config_matches_brute_force():
    L = synth.make_layer(synth.CONFIGS["tiny"], 0)
    out = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k)
    bf = ffn.moe_ffn_bruteforce(L.experts, L.x_bf16, L.logits, L.cfg.k)
    np.testing.assert_allclose(out, bf, rtol=1e-12, atol=1e-12 * np.abs(bf).max())
    assert np.abs(out).max() > 0


@pytest.mark.parametrize("renorm", [True, False])
def test_mixed_layer_matches_brute_force(renorm):
    L = small_layer()
    out = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, renormalize=renorm)
    bf = ffn.moe_ffn_bruteforce(L.experts, L.x_bf16, L.logits, L.cfg.k, renormalize=renorm)
    np.testing.assert_allclose(out, bf, rtol=1e-12, atol=1e-12 * np.abs(bf).max())


def test_tier_decomposition():
    L = small_layer(E=16, k=4, T=6)
    fm = {ex["gate"].fmt for ex in L.experts}
    assert len(fm) == 3
    full = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k)
    parts = sum(ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, format_mask=1 << f) for f in fm)
    np.testing.assert_allclose(parts, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())
    lo = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, expert_lo=0, expert_hi=7)
    hi = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, expert_lo=7, expert_hi=16)
    np.testing.assert_allclose(lo + hi, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())


def test_permutation_invariance():
    L = small_layer(E=10, k=3, T=4, seed=5)
    full = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k)
    perm = np.random.default_rng(31).permutation(10)       # new slot s holds old expert perm[s]
    experts2 = [L.experts[int(p)] for p in perm]
    logits2 = L.logits[:, perm]
    out2 = ffn.moe_ffn(experts2, L.x_bf16, logits2, L.cfg.k)
    np.testing.assert_allclose(out2, full, rtol=1e-12, atol=1e-13 * np.abs(full).max())


def test_zero_scales_give_zero():
    L = synth.make_layer(synth.CONFIGS["tiny"], 0)
    experts = []
    for ex in L.experts:
        e2 = {}
        for name, m in ex.items():
            data = m.data.copy().reshape(m.rows, m.stride)
            for b in range(m.cols // 32):
                data[:, 34 * b: 34 * b + 2] = 0
            e2[name] = MatrixBytes(m.fmt, m.rows, m.cols, m.stride, data.reshape(-1))
        experts.append(e2)
    out = ffn.moe_ffn(experts, L.x_bf16, L.logits, L.cfg.k)
    assert np.all(out == 0)


def test_token_subset_rows():
    L = small_layer(T=7)
    full = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k)
    sub = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, tokens=[6, 2])
    np.testing.assert_array_equal(sub, full[[6, 2]])


def test_planted_transpose_fails_closed_form():
    """A transposed gate (P^T instead of P) must break the closed form."""
    n = 32
    P = np.roll(np.eye(n, dtype=np.int64), 5, axis=1)
    Id = np.eye(n, dtype=np.int64)
    experts = [{"gate": q8_0_matrix(P), "up": q8_0_matrix(Id), "down": q8_0_matrix(Id)}]
    x = np.random.default_rng(32).standard_normal((1, n))
    xq = ffn.bf16_bits_to_f64(bf16_bits(x))
    right = ffn.silu(xq[0] @ P.T) * xq[0]
    wrong = ffn.silu(xq[0] @ P) * xq[0]
    out = ffn.moe_ffn(experts, bf16_bits(x), np.zeros((1, 1), np.float32), k=1)[0]
    np.testing.assert_allclose(out, right, rtol=1e-14)
    assert np.abs(out - wrong).max() > 1e-3


# --------------------------------------------------------------- bf16 activations
# bf16 bit patterns with their values written out by hand: sign, 8 exponent
# bits (bias 127), 7 fraction bits.
BF16_LITERALS = [
    (0x3F80, 1.0),                          # 0 01111111 0000000
    (0xC040, -3.0),                         # 1 10000000 1000000 = -1.5 * 2
    (0x4049, 3.140625),                     # 0 10000000 1001001 = 2 * (1 + 73/128)
    (0x3E80, 0.25),                         # 0 01111101 0000000
    (0x0001, 2.0 ** -133),                  # smallest subnormal: 2^-126 * 2^-7
    (0x0080, 2.0 ** -126),                  # smallest normal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),   # largest finite
    (0x8000, -0.0),
    (0x7F80, float("inf")),
    (0xFF80, float("-inf")),
]


def test_bf16_bits_literal_values():
    bits = np.array([b for b, _ in BF16_LITERALS], np.uint16)
    got = ffn.bf16_bits_to_f64(bits)
    for (b, v), g in zip(BF16_LITERALS, got):
        assert g == v, (hex(b), g, v)
        assert np.signbit(g) == np.signbit(v), hex(b)
    nan = ffn.bf16_bits_to_f64(np.array([0x7FC0], np.uint16))[0]
    assert np.isnan(nan)
    # shape is kept: a [T, H] matrix of bits decodes element by element
    m = ffn.bf16_bits_to_f64(bits[:4].reshape(2, 2))
    assert m.shape == (2, 2) and m[1, 0] == 3.140625


def test_bf16_planted_shift_fails():
    """A decoder shifting by 15 instead of 16 must miss the literal values."""
    def wrong(xb):
        u = np.asarray(xb, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
        return u.view(np.float32).astype(np.float64)
    bits = np.array([b for b, _ in BF16_LITERALS[:7]], np.uint16)
    vals = np.array([v for _, v in BF16_LITERALS[:7]])
    assert np.any(wrong(bits) != vals)
    assert np.all(ffn.bf16_bits_to_f64(bits) == vals)


# --------------------------------------------------------------- one-hot activations
def _golden_block(name):
    import os
    from tests.test_oracle_formats import load_golden
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    return load_golden(here)


def _scaled_rows(fmt, block, n_rows, scale_offsets):
    """n_rows copies of a one-block row whose fp16 scales at scale_offsets are
    multiplied by 2^(r % 4) (exact: the exponent field goes up by r % 4), so
    row r's weights are the block's weights times 2^(r % 4)."""
    stride = synth.padded_stride(fmt, 256)
    data = np.zeros((n_rows, stride), np.uint8)
    for r in range(n_rows):
        b = block.copy()
        for off in scale_offsets:
            h = int(b[off]) | (int(b[off + 1]) << 8)
            h += (r % 4) << 10
            b[off], b[off + 1] = h & 0xFF, h >> 8
        data[r, :b.shape[0]] = b
    return MatrixBytes(fmt, n_rows, 256, stride, data.reshape(-1))


@pytest.mark.parametrize("name,scale_offsets", [("q4_k_block.txt", (0, 2)), ("q6_k_block.txt", (208,))])
def test_one_hot_x_gives_weight_column(name, scale_offsets):
    """x = e_i (a one-hot bf16 row) through a layer of one expert: the gate
    output is column i of W_gate, whose entries are the golden block's
    hand-computed weight i times 2^(r % 4); with up = gate and a down matrix
    that copies h_r to out_r (r < 32), out_r = silu(c_r) * c_r."""
    fmt, block, expected = _golden_block(name)
    I, H = 32, 256
    G = _scaled_rows(fmt, block, I, scale_offsets)
    D = np.zeros((H, I), np.int64)
    D[np.arange(I), np.arange(I)] = 1
    experts = [{"gate": G, "up": G, "down": q8_0_matrix(D)}]
    for i, w_i in expected:
        c = np.array([w_i * 2.0 ** (r % 4) for r in range(I)])
        x = np.zeros((1, H), np.uint16)
        x[0, i] = 0x3F80                                   # bf16 1.0
        g, u, h, y = ffn.expert_forward(ffn.dense(G), ffn.dense(G), ffn.dense(experts[0]["down"]),
                                        ffn.bf16_bits_to_f64(x))
        np.testing.assert_array_equal(g[0], c)
        out = ffn.moe_ffn(experts, x, np.zeros((1, 1), np.float32), k=1)[0]
        with np.errstate(over="ignore"):                   # exp(-c) = inf for c << 0: silu -> -0
            expect = c * c / (1.0 + np.exp(-c))
        np.testing.assert_allclose(out[:I], expect, rtol=1e-14, atol=0)
        assert np.all(out[I:] == 0)


# --------------------------------------------------------------- expert-by-expert evaluation
@pytest.mark.parametrize("kw", [{}, {"renormalize": False}, {"tokens": [4, 0, 2]},
                                {"expert_lo": 3, "expert_hi": 11}, {"format_mask": 1 << synth.Q4_K}])
def test_by_expert_matches_per_pair(kw):
    L = small_layer(E=16, k=4, T=6, seed=9)
    gf = [ex["gate"].fmt for ex in L.experts]
    a = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, gate_formats=gf, **kw)
    b = ffn.moe_ffn_by_expert(L.experts, L.x_bf16, L.logits, L.cfg.k, gate_formats=gf, **kw)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12 * max(np.abs(a).max(), 1e-300))


def test_by_expert_lazy_experts_and_pool():
    """Lazily generated experts (released after use), mapped over a spawned
    process pool, give the per-pair result."""
    import multiprocessing as mp
    cfg = synth.LayerConfig("t", 12, 3, 256, 64, 5, "mixed", True, 41)
    L = synth.make_layer(cfg, 0, with_weights=False)
    lazy = synth.LazyExperts(cfg, L.seed, L.fmts)
    ref = ffn.moe_ffn(synth.make_layer(cfg, 0).experts, L.x_bf16, L.logits, cfg.k)
    got = ffn.moe_ffn_by_expert(lazy, L.x_bf16, L.logits, cfg.k, gate_formats=lazy.gate_formats())
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert not lazy._cache                                # every expert was released
    with mp.get_context("spawn").Pool(2) as pool:
        got2 = ffn.moe_ffn_by_expert(lazy, L.x_bf16, L.logits, cfg.k, gate_formats=lazy.gate_formats(),
                                     map_fn=pool.map)
    np.testing.assert_array_equal(got2, got)


# --------------------------------------------------------------- shared experts
def _shared_closed_form_layer():
    """The closed-form pair of routed experts plus one shared expert with
    gate = I, up = I, down = 3 I: y_shared = 3 silu(x) x on every token."""
    n = 32
    P = np.roll(np.eye(n, dtype=np.int64), 5, axis=1)
    Id = np.eye(n, dtype=np.int64)
    experts = [
        {"gate": q8_0_matrix(P), "up": q8_0_matrix(Id), "down": q8_0_matrix(Id)},
        {"gate": q8_0_matrix(Id), "up": q8_0_matrix(2 * Id), "down": q8_0_matrix(Id)},
        {"gate": q8_0_matrix(Id), "up": q8_0_matrix(Id), "down": q8_0_matrix(3 * Id)},
    ]
    rng = np.random.default_rng(32)
    xb = bf16_bits(rng.standard_normal((3, n)))
    logits = np.array([[1.0, 0.25], [-0.5, 0.75], [0.0, 0.0]], np.float32)
    return experts, xb, logits, P


def _shared_expected(xb, logits, P):
    xq = ffn.bf16_bits_to_f64(xb)
    l = logits.astype(np.float64)
    routed, shared = np.empty_like(xq), np.empty_like(xq)
    for t in range(xq.shape[0]):
        w0 = np.exp(l[t, 0]) / np.exp(l[t]).sum()
        routed[t] = w0 * ffn.silu(xq[t] @ P.T) * xq[t] + (1 - w0) * ffn.silu(xq[t]) * 2 * xq[t]
        shared[t] = 3 * ffn.silu(xq[t]) * xq[t]
    return routed, shared


@pytest.mark.parametrize("evaluate", ["per_pair", "by_expert", "bruteforce"])
def test_shared_expert_closed_form(evaluate):
    """A shared expert is added with weight 1 to the routed experts' weighted
    sum, whatever the router's weights (renormalised or not)."""
    experts, xb, logits, P = _shared_closed_form_layer()
    routed, shared = _shared_expected(xb, logits, P)
    fn = {"per_pair": ffn.moe_ffn, "by_expert": ffn.moe_ffn_by_expert,
          "bruteforce": ffn.moe_ffn_bruteforce}[evaluate]
    out = fn(experts, xb, logits, 2, n_shared=1)
    np.testing.assert_allclose(out, routed + shared, rtol=1e-13, atol=1e-15)


def test_shared_expert_filters():
    """The expert range and the format filter treat the shared expert (entry
    E) like any other: [0, E) gives the routed part, [E, E + 1) the shared
    part alone."""
    experts, xb, logits, P = _shared_closed_form_layer()
    routed, shared = _shared_expected(xb, logits, P)
    r = ffn.moe_ffn(experts, xb, logits, 2, n_shared=1, expert_lo=0, expert_hi=2)
    s = ffn.moe_ffn(experts, xb, logits, 2, n_shared=1, expert_lo=2, expert_hi=3)
    np.testing.assert_allclose(r, routed, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(s, shared, rtol=1e-13, atol=1e-15)
    none = ffn.moe_ffn(experts, xb, logits, 2, n_shared=1, format_mask=1 << synth.Q4_K)
    assert np.all(none == 0)


def test_shared_expert_slots():
    """Slots k .. k+S-1 of every token hold the shared experts E .. E+S-1,
    weight 1, after the router's k slots."""
    logits = np.array([[0.5, -1.0, 2.0, 0.0], [1.0, 1.0, 1.0, 1.0]], np.float32)
    ids, w = ffn.token_slots(logits, 2, True, 2)
    np.testing.assert_array_equal(ids, [[2, 0, 4, 5], [0, 1, 4, 5]])
    assert np.all(w[:, 2:] == 1.0)
    np.testing.assert_allclose(w[:, :2].sum(axis=1), 1.0, rtol=1e-15)
    with pytest.raises(ValueError):
        ffn.moe_ffn([None] * 4, np.zeros((2, 32), np.uint16), logits, 2, n_shared=1)


def test_shared_planted_renormalised_weight_fails():
    """Planted mistake: a shared expert that joins the router's softmax (its
    weight renormalised together with the routed ones) fails the closed form."""
    experts, xb, logits, P = _shared_closed_form_layer()
    routed, shared = _shared_expected(xb, logits, P)
    ids, w = ffn.token_slots(logits, 2, True, 1)
    w_bad = w / w.sum(axis=1, keepdims=True)
    xq = ffn.bf16_bits_to_f64(xb)
    dense = [tuple(ffn.dense(ex[m]) for m in ("gate", "up", "down")) for ex in experts]
    out = np.zeros_like(xq)
    for t in range(xq.shape[0]):
        for j in range(3):
            out[t] += w_bad[t, j] * ffn.expert_forward(*dense[ids[t, j]], xq[t:t + 1])[3][0]
    assert not np.allclose(out, routed + shared, rtol=1e-6)


def test_shared_layer_matches_brute_force():
    cfg = synth.LayerConfig("t", 12, 3, 256, 64, 5, "mixed", True, 44, 1)
    L = synth.make_layer(cfg, 0)
    assert len(L.experts) == 13 and L.fmts[-1] == (synth.Q8_0, synth.Q8_0)
    out = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=1)
    bf = ffn.moe_ffn_bruteforce(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=1)
    np.testing.assert_allclose(out, bf, rtol=1e-12, atol=1e-12 * np.abs(bf).max())
    routed = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=1, expert_hi=12)
    plain = ffn.moe_ffn(L.experts[:12], L.x_bf16, L.logits, cfg.k)
    np.testing.assert_array_equal(routed, plain)
