"""Block-format decoders, fp64. Test infrastructure (see ``oracle/__init__``).

The pages name the formats (Q8_0, Q4_K, Q6_K, MXFP4 in the tiers of "三张 RTX
3090 … 优化指南", section 优化策略二, whose middle and tail tiers are IQ4_XS
gate/up with IQ4_NL down and IQ3_XXS gate/up with MXFP4 down;
Q8_0/Q4_K/Q6_K in the GGUF list of "一张 RTX 3090 跑 Llama 70B", section 一) but
print no byte layout. Reading taken: the public GGUF block layouts for
Q8_0/Q4_K/Q6_K/IQ4_NL/IQ4_XS/IQ3_XXS and the OCP Microscaling (MX) v1.0
element/scale encoding for MXFP4, little-endian, fp16 = IEEE binary16
(subnormals included); the ternary t5_g128 format of "RTX 4080 SUPER 原生
Windows 跑 27B" (section 九.2) is described there only by its packing (five
base-3 weights per byte, one fp16 scale per 128 weights), and the layout below
is the plainest one that fits it (scale first, digits least significant
first). Each decoder below states its layout. IQ3_XXS maps
8-bit indices through a 256-entry grid of four magnitudes; the grid is an
input of the decoder (its values are not reproduced here).

A matrix is ``rows`` rows of ``cols`` weights; blocks run along the columns; row
r starts at byte ``r * stride``.
"""
from __future__ import annotations

import numpy as np

Q8_0, Q4_K, Q6_K, MXFP4, IQ4_NL, IQ4_XS, IQ3_XXS, T5_G128 = 1, 2, 3, 4, 5, 6, 7, 8
BLOCK_ELEMS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, MXFP4: 32, IQ4_NL: 32, IQ4_XS: 256, IQ3_XXS: 256, T5_G128: 128}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, MXFP4: 17, IQ4_NL: 18, IQ4_XS: 136, IQ3_XXS: 98, T5_G128: 28}

# The non-linear 4-bit codebook of IQ4_NL and IQ4_XS: value of code 0..15.
IQ4_CODEBOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113],
                        dtype=np.float64)

# E2M1 magnitudes for codes 0..7 (sign is bit 3): OCP MX v1.0, FP4 E2M1 table.
E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _f16(b: np.ndarray) -> np.ndarray:
    """uint8 [..., 2] little-endian binary16 -> fp64 [...]."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    return b.view("<f2")[..., 0].astype(np.float64)


def dequant_q8_0(blk: np.ndarray) -> np.ndarray:
    """Q8_0, 34 bytes per 32 weights: fp16 d at [0:2], int8 q[32] at [2:34];
    w_i = d * q_i."""
    d = _f16(blk[..., 0:2])
    q = np.ascontiguousarray(blk[..., 2:34]).view(np.int8).astype(np.float64)
    return d[..., None] * q


def q4_k_scale_min(s: np.ndarray):
    """The eight 6-bit (scale, min) pairs of a Q4_K block from its 12 scale
    bytes s[0..11]: for j < 4, sc_j = s[j] & 63 and m_j = s[j+4] & 63; for
    j >= 4 the low four bits come from s[j+4] (scale: low nibble, min: high
    nibble) and the top two bits from bits 6-7 of s[j-4] (scale) and s[j]
    (min)."""
    s = s.astype(np.int64)
    sc = np.empty(s.shape[:-1] + (8,), dtype=np.int64)
    m = np.empty_like(sc)
    for j in range(8):
        if j < 4:
            sc[..., j] = s[..., j] & 63
            m[..., j] = s[..., j + 4] & 63
        else:
            sc[..., j] = (s[..., j + 4] & 15) | ((s[..., j - 4] >> 6) << 4)
            m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    return sc, m


def dequant_q4_k(blk: np.ndarray) -> np.ndarray:
    """Q4_K, 144 bytes per 256 weights: fp16 d [0:2], fp16 dmin [2:4], 12 scale
    bytes [4:16], 128 code bytes qs [16:144]. Weights 64g .. 64g+63 (g = 0..3)
    use qs[32g .. 32g+31]: weight 64g+i (i < 32) is the low nibble of qs[32g+i]
    and belongs to sub-block 2g; weight 64g+32+i is the high nibble and belongs
    to sub-block 2g+1. w = d * sc_b * q - dmin * m_b."""
    d = _f16(blk[..., 0:2])
    dmin = _f16(blk[..., 2:4])
    sc, m = q4_k_scale_min(blk[..., 4:16])
    qs = blk[..., 16:144].astype(np.int64)
    out = np.empty(blk.shape[:-1] + (256,), dtype=np.float64)
    for g in range(4):
        byte = qs[..., 32 * g: 32 * g + 32]
        for half, q in ((0, byte & 15), (1, byte >> 4)):
            b = 2 * g + half
            scale = (d * sc[..., b])[..., None]
            offset = (dmin * m[..., b])[..., None]
            out[..., 64 * g + 32 * half: 64 * g + 32 * half + 32] = scale * q - offset
    return out


def q6_k_codes(blk: np.ndarray) -> np.ndarray:
    """The 256 unsigned 6-bit codes of a Q6_K block (ql [0:128], qh [128:192]).
    Half h in {0, 1} covers weights 128h .. 128h+127 and uses ql[64h ..],
    qh[32h ..]. For i < 32 with Q = qh[32h+i]:
      weight 128h+i    = low nibble of ql[64h+i]     | bits 0-1 of Q << 4
      weight 128h+32+i = low nibble of ql[64h+32+i]  | bits 2-3 of Q << 4
      weight 128h+64+i = high nibble of ql[64h+i]    | bits 4-5 of Q << 4
      weight 128h+96+i = high nibble of ql[64h+32+i] | bits 6-7 of Q << 4"""
    ql = blk[..., 0:128].astype(np.int64)
    qh = blk[..., 128:192].astype(np.int64)
    q = np.empty(blk.shape[:-1] + (256,), dtype=np.int64)
    for h in range(2):
        Q = qh[..., 32 * h: 32 * h + 32]
        lo_a = ql[..., 64 * h: 64 * h + 32]
        lo_b = ql[..., 64 * h + 32: 64 * h + 64]
        base = 128 * h
        q[..., base + 0: base + 32] = (lo_a & 15) | ((Q & 3) << 4)
        q[..., base + 32: base + 64] = (lo_b & 15) | (((Q >> 2) & 3) << 4)
        q[..., base + 64: base + 96] = (lo_a >> 4) | (((Q >> 4) & 3) << 4)
        q[..., base + 96: base + 128] = (lo_b >> 4) | (((Q >> 6) & 3) << 4)
    return q


def dequant_q6_k(blk: np.ndarray) -> np.ndarray:
    """Q6_K, 210 bytes per 256 weights: ql [0:128], qh [128:192], 16 int8
    scales [192:208], fp16 d [208:210]. Weight 128h+32r+i (r = 0..3, i < 32)
    uses scale number 8h + 2r + (i >= 16), i.e. one scale per 16 weights.
    w = d * scale * (q - 32)."""
    q = q6_k_codes(blk)
    scales = np.ascontiguousarray(blk[..., 192:208]).view(np.int8).astype(np.float64)
    d = _f16(blk[..., 208:210])
    n = np.arange(256)
    h, rem = n // 128, n % 128
    r, i = rem // 32, rem % 32
    scale_idx = 8 * h + 2 * r + (i >= 16)
    return d[..., None] * scales[..., scale_idx] * (q - 32).astype(np.float64)


def dequant_mxfp4(blk: np.ndarray) -> np.ndarray:
    """MXFP4, 17 bytes per 32 weights: E8M0 scale byte e at [0], 16 code bytes
    at [1:17]; weight i < 16 is the low nibble of byte 1+i, weight 16+i its high
    nibble. An E2M1 nibble has the sign in bit 3 and magnitude index in bits
    0-2. w = 2**(e - 127) * E2M1(code). e = 255 (NaN in E8M0) is rejected."""
    e = blk[..., 0].astype(np.int64)
    if np.any(e == 255):
        raise ValueError("MXFP4 block with E8M0 scale 0xFF (NaN)")
    qs = blk[..., 1:17].astype(np.int64)
    codes = np.concatenate([qs & 15, qs >> 4], axis=-1)
    mag = E2M1_MAGNITUDE[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    return np.ldexp(1.0, e - 127)[..., None] * val


def dequant_iq4_nl(blk: np.ndarray) -> np.ndarray:
    """IQ4_NL, 18 bytes per 32 weights: fp16 d at [0:2], 16 code bytes at
    [2:18]; weight i < 16 is the low nibble of byte 2+i, weight 16+i its high
    nibble. w = d * IQ4_CODEBOOK[code]."""
    d = _f16(blk[..., 0:2])
    qs = blk[..., 2:18].astype(np.int64)
    codes = np.concatenate([qs & 15, qs >> 4], axis=-1)
    return d[..., None] * IQ4_CODEBOOK[codes]


def iq4_xs_scales(blk: np.ndarray) -> np.ndarray:
    """The eight 6-bit sub-block scales ls_0..ls_7 of an IQ4_XS block: the
    low four bits of ls_b are nibble (b % 2) of byte 4 + b // 2 (low nibble
    first), the high two bits are bits 2b, 2b+1 of the uint16 at [2:4]."""
    sh = blk[..., 2].astype(np.int64) | (blk[..., 3].astype(np.int64) << 8)
    sl = blk[..., 4:8].astype(np.int64)
    ls = np.empty(blk.shape[:-1] + (8,), dtype=np.int64)
    for b in range(8):
        ls[..., b] = ((sl[..., b // 2] >> (4 * (b % 2))) & 15) | (((sh >> (2 * b)) & 3) << 4)
    return ls


def dequant_iq4_xs(blk: np.ndarray) -> np.ndarray:
    """IQ4_XS, 136 bytes per 256 weights: fp16 d [0:2], uint16 high scale
    bits [2:4], 4 bytes of low scale nibbles [4:8], 128 code bytes [8:136].
    Sub-block b (weights 32b .. 32b+31) has scale d * (ls_b - 32) and code
    bytes [8+16b, 8+16b+16): weight 32b+i (i < 16) is the low nibble of its
    byte i, weight 32b+16+i the high nibble. w = d * (ls_b - 32) *
    IQ4_CODEBOOK[code]."""
    d = _f16(blk[..., 0:2])
    ls = iq4_xs_scales(blk)
    qs = blk[..., 8:136].astype(np.int64)
    out = np.empty(blk.shape[:-1] + (256,), dtype=np.float64)
    for b in range(8):
        byte = qs[..., 16 * b: 16 * b + 16]
        scale = (d * (ls[..., b] - 32))[..., None]
        out[..., 32 * b: 32 * b + 16] = scale * IQ4_CODEBOOK[byte & 15]
        out[..., 32 * b + 16: 32 * b + 32] = scale * IQ4_CODEBOOK[byte >> 4]
    return out


def iq3_sign_byte(idx7: np.ndarray) -> np.ndarray:
    """The eight signs of an IQ3_XXS group from its 7-bit index: bits 0..6
    are the index, bit 7 makes the number of set bits even (so the eighth
    sign is implied by the other seven). Bit j set: weight j is negative."""
    idx7 = np.asarray(idx7, dtype=np.int64) & 127
    pop = np.zeros_like(idx7)
    for j in range(7):
        pop += (idx7 >> j) & 1
    return idx7 | ((pop & 1) << 7)


def dequant_iq3_xxs(blk: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """IQ3_XXS, 98 bytes per 256 weights: fp16 d [0:2], 64 grid-index bytes
    [2:66], 8 little-endian uint32 words [66:98], one per sub-block of 32.
    Word a of sub-block b: bits 28..31 give its scale d * (0.5 + (a >> 28)) /
    2; bits 7l .. 7l+6 (l = 0..3) give the sign index of its group l of 8
    weights. Group l uses grid entries grid[q[8b+2l]] (weights 0..3 of the
    group) and grid[q[8b+2l+1]] (weights 4..7); byte j of an entry (uint32,
    little-endian) is the magnitude of its weight j. w = scale * magnitude *
    (-1 if the weight's sign bit is set)."""
    grid = np.asarray(grid, dtype=np.int64).reshape(256)
    d = _f16(blk[..., 0:2])
    q = blk[..., 2:66].astype(np.int64)
    words = np.ascontiguousarray(blk[..., 66:98]).view("<u4").astype(np.int64)
    out = np.empty(blk.shape[:-1] + (256,), dtype=np.float64)
    for b in range(8):
        a = words[..., b]
        scale = d * (0.5 + (a >> 28)) * 0.5
        for l in range(4):
            signs = iq3_sign_byte(a >> (7 * l))
            for half in range(2):
                entry = grid[q[..., 8 * b + 2 * l + half]]
                for j in range(4):
                    mag = ((entry >> (8 * j)) & 255).astype(np.float64)
                    neg = (signs >> (4 * half + j)) & 1
                    out[..., 32 * b + 8 * l + 4 * half + j] = scale * np.where(neg == 1, -mag, mag)
    return out


def dequant_t5_g128(blk: np.ndarray) -> np.ndarray:
    """Ternary t5_g128 ("RTX 4080 SUPER 原生 Windows 跑 27B", section 九.2: ternary
    codes packed base-3, five weights per byte, and one fp16 scale per 128
    weights, 1.75 bits per weight), 28 bytes per 128 weights: fp16 scale s at
    [0:2], 26 code bytes at [2:28]. Weight 5b + i (i < 5) is base-3 digit i
    of byte 2 + b, least significant first (digit i = floor(v / 3^i) mod 3);
    the last byte's digits 3 and 4 are unused. w = s * (digit - 1)."""
    s = _f16(blk[..., 0:2])
    v = blk[..., 2:28].astype(np.int64)
    digits = np.stack([(v // 3 ** i) % 3 for i in range(5)], axis=-1).reshape(blk.shape[:-1] + (130,))
    return s[..., None] * (digits[..., :128] - 1).astype(np.float64)


DECODERS = {Q8_0: dequant_q8_0, Q4_K: dequant_q4_k, Q6_K: dequant_q6_k, MXFP4: dequant_mxfp4,
            IQ4_NL: dequant_iq4_nl, IQ4_XS: dequant_iq4_xs, IQ3_XXS: dequant_iq3_xxs, T5_G128: dequant_t5_g128}


def decode_blocks(fmt: int, blocks: np.ndarray, grid=None) -> np.ndarray:
    """Blocks [..., block bytes] -> weights [..., block weights]; IQ3_XXS needs
    its grid (256 uint32)."""
    if fmt == IQ3_XXS:
        if grid is None:
            raise ValueError("IQ3_XXS needs its grid")
        return dequant_iq3_xxs(blocks, grid)
    return DECODERS[fmt](blocks)


def dequant_matrix(fmt: int, rows: int, cols: int, stride: int, data: np.ndarray, grid=None) -> np.ndarray:
    """Whole matrix -> fp64 [rows, cols]."""
    be, bb = BLOCK_ELEMS[fmt], BLOCK_BYTES[fmt]
    if cols % be:
        raise ValueError(f"cols={cols} is not a multiple of the block size {be}")
    nb = cols // be
    if stride < nb * bb:
        raise ValueError("row stride shorter than a row")
    raw = np.asarray(data, dtype=np.uint8).reshape(-1)[: rows * stride]
    blocks = raw.reshape(rows, stride)[:, : nb * bb].reshape(rows, nb, bb)
    return decode_blocks(fmt, blocks, grid).reshape(rows, cols)


def dequant_rows(fmt: int, cols: int, stride: int, data: np.ndarray, rows_idx, grid=None) -> np.ndarray:
    """Selected rows only -> fp64 [len(rows_idx), cols]."""
    be, bb = BLOCK_ELEMS[fmt], BLOCK_BYTES[fmt]
    nb = cols // be
    raw = np.asarray(data, dtype=np.uint8).reshape(-1)
    rows_idx = np.asarray(rows_idx, dtype=np.int64)
    sel = raw.reshape(-1, stride)[rows_idx][:, : nb * bb].reshape(len(rows_idx), nb, bb)
    return decode_blocks(fmt, sel, grid).reshape(len(rows_idx), cols)
