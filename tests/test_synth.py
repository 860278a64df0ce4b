"""The seeded input generator (CPU part): SplitMix64 against its published
reference outputs, field distributions, and the routing statistics the layer
configurations ask for (Zipf-shaped router bias: the top 25% of experts take
about 52% of the selections and the top 80% about 95%)."""
import numpy as np

import synth
from oracle import formats, router


def test_splitmix64_reference_sequence():
    # SplitMix64 seeded with 0: the first outputs of the reference generator
    # (Vigna's splitmix64.c) are 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F.
    r = synth.draws(0, np.arange(3))
    assert [int(v) for v in r] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_differ_and_are_deterministic():
    a = synth.draws(synth.stream_key(5, 1), np.arange(100))
    b = synth.draws(synth.stream_key(5, 2), np.arange(100))
    c = synth.draws(synth.stream_key(5, 1), np.arange(100))
    assert not np.array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_block_field_ranges():
    key = synth.stream_key(1, 99)
    n = 4000
    q8 = synth.gen_blocks(synth.Q8_0, key, np.arange(n))
    d = q8[:, 0:2].copy().view("<f2").astype(np.float64)[:, 0]
    assert d.min() >= 0.00199 and d.max() <= 0.02001
    q = q8[:, 2:].view(np.int8)
    assert q.min() == -127 and q.max() == 127
    mx = synth.gen_blocks(synth.MXFP4, key, np.arange(n))
    assert set(np.unique(mx[:, 0]).tolist()) == {124, 125, 126}
    q6 = synth.gen_blocks(synth.Q6_K, key, np.arange(n))
    s6 = q6[:, 192:208].view(np.int8)
    assert s6.min() == -127 and s6.max() == 127
    q4 = synth.gen_blocks(synth.Q4_K, key, np.arange(n))
    sc, m = formats.q4_k_scale_min(q4[:, 4:16])
    assert sc.min() == 0 and sc.max() == 63 and m.min() == 0 and m.max() == 63
    t5 = synth.gen_blocks(synth.T5_G128, key, np.arange(n))
    s = t5[:, 0:2].copy().view("<f2").astype(np.float64)[:, 0]
    assert s.min() >= 0.2499 and s.max() <= 1.0001
    assert t5[:, 2:27].min() == 0 and t5[:, 2:27].max() == 242        # five base-3 digits
    assert t5[:, 27].min() == 0 and t5[:, 27].max() == 26             # three digits, two unused
    w = formats.DECODERS[synth.T5_G128](t5) / s[:, None]
    assert set(np.unique(w).tolist()) == {-1.0, 0.0, 1.0}
    assert abs((w == 0).mean() - 1 / 3) < 0.01


def test_weight_rms_comparable_across_formats():
    key = synth.stream_key(2, 7)
    for fmt in (synth.Q8_0, synth.Q4_K, synth.Q6_K, synth.MXFP4, synth.T5_G128):
        blk = synth.gen_blocks(fmt, key, np.arange(256))
        w = formats.DECODERS[fmt](blk)
        rms = np.sqrt((w ** 2).mean())
        assert 0.3 < rms < 2.0, (fmt, rms)


def test_matrix_padding_is_zero():
    m = synth.gen_matrix(synth.Q8_0, 5, 640, synth.stream_key(3, 3))
    assert m.stride == 688
    rows = m.data.reshape(5, 688)
    assert np.all(rows[:, 680:] == 0)


def test_tier_bounds_and_formats():
    assert synth.tier_bounds(512) == (128, 410)
    cfg = synth.CONFIGS["mtp6"]
    fm = synth.expert_formats(cfg, 4000)
    counts = {}
    for f in fm:
        counts[f] = counts.get(f, 0) + 1
    assert counts == {(synth.Q6_K, synth.Q8_0): 128, (synth.Q4_K, synth.Q8_0): 282,
                      (synth.MXFP4, synth.MXFP4): 102}
    perm = synth.permutation(4000, 512)
    assert fm[int(perm[0])] == (synth.Q6_K, synth.Q8_0)
    assert fm[int(perm[511])] == (synth.MXFP4, synth.MXFP4)


def test_zipf_routing_shares():
    E, T = 512, 1500
    tot = np.zeros(E)
    for layer in range(2):
        seed = 3000 + layer
        ids, _, _ = router.route_topk(synth.gen_logits(seed, T, E, True), 10)
        perm = synth.permutation(seed, E)
        rank = np.empty(E, np.int64)
        rank[perm] = np.arange(E)
        np.add.at(tot, rank[ids.reshape(-1)], 1)
    c = np.cumsum(tot) / tot.sum()
    assert 0.49 < c[127] < 0.55
    assert 0.92 < c[409] < 0.97


def test_bf16_rounding():
    x = np.array([1.0, 1.00390625, 1.005859375, -3.0e-3, 65504.0], np.float32)
    b = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(b)
    assert back[0] == 1.0
    assert back[1] == 1.0            # halfway 1 + 2^-8 rounds to even (1.0)
    assert back[2] == 1.0078125      # above halfway rounds up
    assert abs(back[3] - x[3]) <= abs(x[3]) * 2 ** -8
