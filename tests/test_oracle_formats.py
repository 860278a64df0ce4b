"""Pins of the oracle's block decoders (CPU only).

* Hand-built single blocks with hand-computed weights (tests/golden/*_block.txt).
* Round trips: codes and scales chosen at random, packed into bytes by an
  encoder written here from the layout description (the inverse direction of
  the decoders), decoded, and compared with the value formula evaluated
  directly on the chosen codes.
* Planted mistakes: each decoder with one plausible bug (dropped term, swapped
  nibbles, wrong scale index, wrong sign bit) must fail the pins above.
"""
import glob
import os

import numpy as np
import pytest

from oracle import formats

FMT = {"Q8_0": formats.Q8_0, "Q4_K": formats.Q4_K, "Q6_K": formats.Q6_K, "MXFP4": formats.MXFP4,
       "IQ4_NL": formats.IQ4_NL, "IQ4_XS": formats.IQ4_XS, "IQ3_XXS": formats.IQ3_XXS, "T5_G128": formats.T5_G128}


def load_golden(path, with_grid=False):
    fmt, data, exp, grid = None, None, [], None
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            if p[0] == "format":
                fmt = FMT[p[1]]
            elif p[0] == "bytes":
                data = np.array([int(x, 16) for x in p[1:]], dtype=np.uint8)
            elif p[0] == "grid":
                grid = np.array([int(x, 16) for x in p[1:]], dtype=np.int64)
            elif p[0] == "w":
                exp.append((int(p[1]), float(p[2])))
    return (fmt, data, exp, grid) if with_grid else (fmt, data, exp)


def golden_files(golden_dir):
    files = sorted(glob.glob(os.path.join(golden_dir, "*_block.txt")))
    assert len(files) >= 9
    return files


def check_golden(decoders, golden_dir):
    for path in golden_files(golden_dir):
        fmt, data, exp, grid = load_golden(path, with_grid=True)
        assert data.shape[0] == formats.BLOCK_BYTES[fmt]
        w = decoders[fmt](data[None, :], grid)[0] if fmt == formats.IQ3_XXS else decoders[fmt](data[None, :])[0]
        for i, v in exp:
            if w[i] != v:
                return False, (os.path.basename(path), i, w[i], v)
    return True, None


def test_golden_blocks(golden_dir):
    ok, bad = check_golden(formats.DECODERS, golden_dir)
    assert ok, bad


def test_q8_0_unit_scale_gives_codes():
    rng = np.random.default_rng(1)
    q = rng.integers(-127, 128, size=(5, 32)).astype(np.int8)
    blk = np.zeros((5, 34), dtype=np.uint8)
    blk[:, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    blk[:, 2:] = q.view(np.uint8)
    np.testing.assert_array_equal(formats.dequant_q8_0(blk), q.astype(np.float64))


def test_mxfp4_scale_doubles(golden_dir):
    _, b127, _ = load_golden(os.path.join(golden_dir, "mxfp4_e127_block.txt"))
    _, b128, _ = load_golden(os.path.join(golden_dir, "mxfp4_e128_block.txt"))
    w127 = formats.dequant_mxfp4(b127[None])[0]
    w128 = formats.dequant_mxfp4(b128[None])[0]
    np.testing.assert_array_equal(w128, 2 * w127)
    assert sorted(set(np.abs(w127).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_mxfp4_rejects_nan_scale():
    blk = np.zeros((1, 17), dtype=np.uint8)
    blk[0, 0] = 255
    with pytest.raises(ValueError):
        formats.dequant_mxfp4(blk)


# ---------------------------------------------------------------- encoders
def enc_q4_k(d, dmin, sc, m, q):
    """sc, m: int [8] (0..63); q: int [256] (0..15)."""
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    s = np.zeros(12, dtype=np.int64)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    b[4:16] = s
    for g in range(4):
        for i in range(32):
            b[16 + 32 * g + i] = q[64 * g + i] | (q[64 * g + 32 + i] << 4)
    return b


def val_q4_k(d, dmin, sc, m, q):
    d, dmin = float(np.float16(d)), float(np.float16(dmin))
    sub = np.arange(256) // 32
    return d * sc[sub] * q - dmin * m[sub]


def enc_q6_k(d, scales, q):
    """scales int [16] (-128..127); q int [256] (0..63)."""
    b = np.zeros(210, dtype=np.uint8)
    ql = np.zeros(128, dtype=np.int64)
    qh = np.zeros(64, dtype=np.int64)
    for n in range(256):
        h, r, i = n // 128, (n % 128) // 32, n % 32
        lo, hi = q[n] & 15, q[n] >> 4
        ql_idx = 64 * h + (32 if r in (1, 3) else 0) + i
        ql[ql_idx] |= lo << (4 if r >= 2 else 0)
        qh[32 * h + i] |= hi << (2 * r)
    b[0:128] = ql
    b[128:192] = qh
    b[192:208] = np.asarray(scales, dtype=np.int8).view(np.uint8)
    b[208:210] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    return b


def val_q6_k(d, scales, q):
    d = float(np.float16(d))
    return d * np.asarray(scales, dtype=np.float64)[np.arange(256) // 16] * (q - 32)


def enc_mxfp4(e, codes):
    b = np.zeros(17, dtype=np.uint8)
    b[0] = e
    b[1:17] = codes[:16] | (codes[16:] << 4)
    return b


def val_mxfp4(e, codes):
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    sign = np.where(codes >= 8, -1.0, 1.0)
    return 2.0 ** (e - 127) * sign * mag[codes & 7]


IQ4_VALUES = np.array([-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113], dtype=np.float64)


def enc_iq4_nl(d, codes):
    b = np.zeros(18, dtype=np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:18] = codes[:16] | (codes[16:] << 4)
    return b


def enc_iq4_xs(d, ls, codes):
    """ls int [8] (0..63); codes int [256] (0..15)."""
    b = np.zeros(136, dtype=np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    sh = 0
    for j in range(8):
        sh |= (int(ls[j]) >> 4) << (2 * j)
        b[4 + j // 2] |= (int(ls[j]) & 15) << (4 * (j % 2))
    b[2], b[3] = sh & 255, sh >> 8
    for j in range(8):
        for i in range(16):
            b[8 + 16 * j + i] = codes[32 * j + i] | (codes[32 * j + 16 + i] << 4)
    return b


def enc_iq3_xxs(d, q, signs7, scales4):
    """q int [64] grid indices; signs7 int [8, 4] (0..127); scales4 int [8] (0..15)."""
    b = np.zeros(98, dtype=np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:66] = q
    for j in range(8):
        a = int(scales4[j]) << 28
        for l in range(4):
            a |= int(signs7[j, l]) << (7 * l)
        b[66 + 4 * j: 70 + 4 * j] = np.frombuffer(np.uint32(a).tobytes(), np.uint8)
    return b


def val_iq3_xxs(d, q, signs7, scales4, grid):
    d = float(np.float16(d))
    out = np.zeros(256)
    for j in range(8):
        sc = d * (0.5 + scales4[j]) / 2
        for l in range(4):
            s = int(signs7[j, l])
            sbits = s | ((bin(s).count("1") & 1) << 7)
            for t in range(8):
                entry = int(grid[q[8 * j + 2 * l + t // 4]])
                mag = (entry >> (8 * (t % 4))) & 255
                out[32 * j + 8 * l + t] = sc * mag * (-1.0 if (sbits >> t) & 1 else 1.0)
    return out


def test_iq4_roundtrips():
    rng = np.random.default_rng(6)
    for _ in range(20):
        codes = rng.integers(0, 16, 32)
        d = rng.uniform(1e-3, 1.0)
        np.testing.assert_array_equal(formats.dequant_iq4_nl(enc_iq4_nl(d, codes)[None])[0],
                                      float(np.float16(d)) * IQ4_VALUES[codes])
        ls = rng.integers(0, 64, 8)
        codes = rng.integers(0, 16, 256)
        w = formats.dequant_iq4_xs(enc_iq4_xs(d, ls, codes)[None])[0]
        np.testing.assert_array_equal(w, float(np.float16(d)) * (ls[np.arange(256) // 32] - 32) * IQ4_VALUES[codes])


def test_iq3_xxs_roundtrip():
    rng = np.random.default_rng(7)
    for _ in range(10):
        grid = rng.integers(0, 2 ** 32, 256, dtype=np.int64)
        q = rng.integers(0, 256, 64)
        signs7 = rng.integers(0, 128, (8, 4))
        scales4 = rng.integers(0, 16, 8)
        d = rng.uniform(1e-3, 1.0)
        w = formats.dequant_iq3_xxs(enc_iq3_xxs(d, q, signs7, scales4)[None], grid)[0]
        np.testing.assert_array_equal(w, val_iq3_xxs(d, q, signs7, scales4, grid))
    # the eighth sign is implied: every group has an even number of negative weights
    grid = np.full(256, 0x01010101, dtype=np.int64)
    blk = enc_iq3_xxs(1.0, rng.integers(0, 256, 64), rng.integers(0, 128, (8, 4)), np.zeros(8, np.int64))
    w = formats.dequant_iq3_xxs(blk[None], grid)[0].reshape(32, 8)
    assert np.all((w < 0).sum(axis=1) % 2 == 0)


def enc_t5(scale, trits):
    """trits int [128] in {-1, 0, 1} -> 28 bytes (scale, then five base-3 digits per byte)."""
    b = np.zeros(28, dtype=np.uint8)
    b[0:2] = np.frombuffer(np.float16(scale).tobytes(), np.uint8)
    d = np.concatenate([np.asarray(trits) + 1, np.ones(2, np.int64)])
    for j in range(26):
        b[2 + j] = sum(int(d[5 * j + i]) * 3 ** i for i in range(5))
    return b


def test_t5_g128_roundtrip():
    rng = np.random.default_rng(8)
    for _ in range(20):
        trits = rng.integers(-1, 2, 128)
        s = rng.uniform(0.1, 2.0)
        np.testing.assert_array_equal(formats.dequant_t5_g128(enc_t5(s, trits)[None])[0],
                                      float(np.float16(s)) * trits)
    # every byte value decodes to digits 0..2 (values above 242 included)
    blk = np.zeros((1, 28), np.uint8)
    blk[0, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    blk[0, 2:] = 255
    assert set(np.unique(formats.dequant_t5_g128(blk))) <= {-1.0, 0.0, 1.0}


def _t5_msd_first(blk):
    # digits most significant first
    s = formats._f16(blk[..., 0:2])
    v = blk[..., 2:28].astype(np.int64)
    digits = np.stack([(v // 3 ** (4 - i)) % 3 for i in range(5)], axis=-1).reshape(blk.shape[:-1] + (130,))
    return s[..., None] * (digits[..., :128] - 1).astype(np.float64)


def _t5_no_offset(blk):
    # the digit itself instead of digit - 1
    return formats.dequant_t5_g128(blk) + formats._f16(blk[..., 0:2])[..., None]


def test_iq3_xxs_needs_its_grid():
    with pytest.raises(ValueError):
        formats.decode_blocks(formats.IQ3_XXS, np.zeros((1, 98), np.uint8))


def test_q4_k_roundtrip():
    rng = np.random.default_rng(2)
    for _ in range(20):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        d, dmin = rng.uniform(1e-3, 1.0), rng.uniform(1e-3, 1.0)
        blk = enc_q4_k(d, dmin, sc, m, q)
        np.testing.assert_array_equal(formats.dequant_q4_k(blk[None])[0], val_q4_k(d, dmin, sc, m, q))


def test_q6_k_roundtrip():
    rng = np.random.default_rng(3)
    for _ in range(20):
        scales = rng.integers(-128, 128, 16)
        q = rng.integers(0, 64, 256)
        d = rng.uniform(1e-3, 1.0)
        blk = enc_q6_k(d, scales, q)
        np.testing.assert_array_equal(formats.dequant_q6_k(blk[None])[0], val_q6_k(d, scales, q))


def test_mxfp4_roundtrip():
    rng = np.random.default_rng(4)
    for _ in range(20):
        e = int(rng.integers(100, 150))
        codes = rng.integers(0, 16, 32)
        np.testing.assert_array_equal(formats.dequant_mxfp4(enc_mxfp4(e, codes)[None])[0],
                                      val_mxfp4(e, codes))


def test_matrix_rows_and_padding():
    """A matrix with a padded stride decodes row by row like single blocks."""
    rng = np.random.default_rng(5)
    rows, cols, stride = 3, 64, 80          # Q8_0: 2 blocks = 68 bytes per row
    data = rng.integers(0, 256, rows * stride).astype(np.uint8)
    for r in range(rows):
        data[r * stride: r * stride + 2] = np.frombuffer(np.float16(0.25).tobytes(), np.uint8)
        data[r * stride + 34: r * stride + 36] = np.frombuffer(np.float16(-2.0).tobytes(), np.uint8)
    W = formats.dequant_matrix(formats.Q8_0, rows, cols, stride, data)
    for r in range(rows):
        q0 = data[r * stride + 2: r * stride + 34].view(np.int8)
        q1 = data[r * stride + 36: r * stride + 68].view(np.int8)
        np.testing.assert_array_equal(W[r, :32], 0.25 * q0)
        np.testing.assert_array_equal(W[r, 32:], -2.0 * q1)
    np.testing.assert_array_equal(formats.dequant_rows(formats.Q8_0, cols, stride, data, [2, 0]), W[[2, 0]])


# ---------------------------------------------------------------- planted mistakes
def _q4_k_no_min(blk):
    out = formats.dequant_q4_k(blk)
    d = formats._f16(blk[..., 2:4])
    _, m = formats.q4_k_scale_min(blk[..., 4:16])
    sub = np.arange(256) // 32
    return out + d[..., None] * m[..., sub]          # drops the "- dmin*m" term


def _q4_k_swapped_nibbles(blk):
    out = formats.dequant_q4_k(blk)
    r = out.reshape(out.shape[:-1] + (4, 2, 32))
    return r[..., ::-1, :].reshape(out.shape)


def _q6_k_scale_per_32(blk):
    q = formats.q6_k_codes(blk)
    scales = np.ascontiguousarray(blk[..., 192:208]).view(np.int8).astype(np.float64)
    d = formats._f16(blk[..., 208:210])
    idx = np.minimum(np.arange(256) // 32 * 2, 15)   # wrong scale index
    return d[..., None] * scales[..., idx] * (q - 32)


def _mxfp4_unsigned(blk):
    return np.abs(formats.dequant_mxfp4(blk))


def _q8_0_wrong_offset(blk):
    d = formats._f16(blk[..., 0:2])
    q = np.ascontiguousarray(blk[..., 2:34]).view(np.uint8).astype(np.float64)   # unsigned read
    return d[..., None] * q


def _iq4_nl_linear(blk):
    # a linear 4-bit code (q - 8) * 16 instead of the codebook
    d = formats._f16(blk[..., 0:2])
    qs = blk[..., 2:18].astype(np.int64)
    codes = np.concatenate([qs & 15, qs >> 4], axis=-1)
    return d[..., None] * (codes - 8) * 16.0


def _iq4_xs_unsigned_scale(blk):
    # the sub-block scale d * ls instead of d * (ls - 32)
    d = formats._f16(blk[..., 0:2])
    ls = formats.iq4_xs_scales(blk)
    qs = blk[..., 8:136].astype(np.int64)
    out = np.empty(blk.shape[:-1] + (256,))
    for b in range(8):
        byte = qs[..., 16 * b: 16 * b + 16]
        scale = (d * ls[..., b])[..., None]
        out[..., 32 * b: 32 * b + 16] = scale * formats.IQ4_CODEBOOK[byte & 15]
        out[..., 32 * b + 16: 32 * b + 32] = scale * formats.IQ4_CODEBOOK[byte >> 4]
    return out


def _iq3_xxs_no_parity(blk, grid):
    # the eighth sign of each group taken as positive instead of from the parity
    w = formats.dequant_iq3_xxs(blk, grid).copy()
    g = w.reshape(w.shape[:-1] + (32, 8))
    g[..., 7] = np.abs(g[..., 7])
    return g.reshape(w.shape)


def _iq3_xxs_scale_half(blk, grid):
    # scale d * (0.5 + s) without the final halving
    return 2 * formats.dequant_iq3_xxs(blk, grid)


@pytest.mark.parametrize("fmt,bad", [
    (formats.T5_G128, _t5_msd_first),
    (formats.T5_G128, _t5_no_offset),
    (formats.IQ4_NL, _iq4_nl_linear),
    (formats.IQ4_XS, _iq4_xs_unsigned_scale),
    (formats.IQ3_XXS, _iq3_xxs_no_parity),
    (formats.IQ3_XXS, _iq3_xxs_scale_half),
    (formats.Q4_K, _q4_k_no_min),
    (formats.Q4_K, _q4_k_swapped_nibbles),
    (formats.Q6_K, _q6_k_scale_per_32),
    (formats.MXFP4, _mxfp4_unsigned),
    (formats.Q8_0, _q8_0_wrong_offset),
])
def test_planted_mistakes_fail_the_pins(golden_dir, fmt, bad):
    decoders = dict(formats.DECODERS)
    decoders[fmt] = bad
    ok, _ = check_golden(decoders, golden_dir)
    assert not ok
