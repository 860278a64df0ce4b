"""Writes the hand-built single-block fixtures ``*_block.txt`` in this folder.

Each block's bytes follow a stated construction rule; the expected weights are
HAND-COMPUTED from the block layout (worked out on paper, typed in below as
literals, with the working in the comments) and are not produced by any
decoder. The format names come from "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80
Token 每秒的高效推理优化指南", section 优化策略二 (Q6_K / Q8_0 top tier, MXFP4 tail
tier) and the GGUF format list of "一张 RTX 3090 跑 Llama 70B：三层流式缓存 + NVMe
直连", section 一 (Q8_0, Q4_K, Q6_K); the pages print no byte layout, so the
layouts are the public GGUF block layouts (Q8_0, Q4_K, Q6_K) and the OCP MX v1.0
FP4 E2M1 / E8M0 encoding (MXFP4).

Run:  python tests/golden/make_golden_blocks.py
"""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def q8_0_block():
    # d = 1.0 (binary16 0x3C00, little-endian bytes 00 3C); q_i = i - 16.
    b = [0x00, 0x3C] + [(i - 16) & 0xFF for i in range(32)]
    # w_i = 1.0 * (i - 16)
    expected = [(i, float(i - 16)) for i in range(32)]
    rule = "d = 1.0 (0x3C00); q_i = i - 16 (int8); w_i = q_i exactly"
    return b, expected, rule


def q8_0_half_block():
    # d = 0.5 (0x3800); q = 127 at i = 0, -127 at i = 1, else (i % 7) - 3.
    q = [127, -127] + [(i % 7) - 3 for i in range(2, 32)]
    b = [0x00, 0x38] + [v & 0xFF for v in q]
    expected = [
        (0, 63.5),    # 0.5 * 127
        (1, -63.5),   # 0.5 * -127
        (2, -0.5),    # (2 % 7) - 3 = -1
        (5, 1.0),     # (5 % 7) - 3 = 2
        (9, -0.5),    # (9 % 7) - 3 = -1
        (31, 0.0),    # (31 % 7) - 3 = 0
    ]
    rule = "d = 0.5 (0x3800); q_0 = 127, q_1 = -127, q_i = (i % 7) - 3 for i >= 2"
    return b, expected, rule


def q4_k_block():
    # d = 0.25 (0x3400), dmin = 0.125 (0x3000).
    # (sc_j) = 17, 22, 35, 48, 63, 16, 29, 40 ; (m_j) = 18, 21, 33, 50, 61, 19, 27, 44
    # all >= 16, so the 2-bit high parts of j >= 4 are exercised. Packing:
    #   s[0..3] = sc_j | (sc_{j+4} >> 4) << 6 = 0xD1 0x56 0x63 0xB0
    #   s[4..7] = m_j  | (m_{j+4}  >> 4) << 6 = 0xD2 0x55 0x61 0xB2
    #   s[8..11] = (sc_{j+4} & 15) | (m_{j+4} & 15) << 4 = 0xDF 0x30 0xBD 0xC8
    scales = [0xD1, 0x56, 0x63, 0xB0, 0xD2, 0x55, 0x61, 0xB2, 0xDF, 0x30, 0xBD, 0xC8]
    # qs[32g + i] = ((i + g) % 16) | (((15 - i) % 16) << 4)
    qs = [((i + g) % 16) | (((15 - i) % 16) << 4) for g in range(4) for i in range(32)]
    b = [0x00, 0x34, 0x00, 0x30] + scales + qs
    expected = [
        (0, -2.25),      # g0 lo i0: q=0, sb0: 0 - 0.125*18
        (1, 2.0),        # q=1: 0.25*17*1 - 2.25
        (33, 74.375),    # g0 hi i1: q=14, sb1: 0.25*22*14 - 0.125*21 = 77 - 2.625
        (69, 48.375),    # g1 lo i5: q=6, sb2: 0.25*35*6 - 0.125*33 = 52.5 - 4.125
        (140, 212.875),  # g2 lo i12: q=14, sb4: 0.25*63*14 - 0.125*61 = 220.5 - 7.625
        (168, 25.625),   # g2 hi i8: q=7, sb5: 0.25*16*7 - 0.125*19 = 28 - 2.375
        (200, 76.375),   # g3 lo i8: q=11, sb6: 0.25*29*11 - 0.125*27 = 79.75 - 3.375
        (230, 84.5),     # g3 hi i6: q=9, sb7: 0.25*40*9 - 0.125*44 = 90 - 5.5
        (255, -5.5),     # g3 hi i31: q=0, sb7: -0.125*44
    ]
    rule = ("d = 0.25, dmin = 0.125; (sc) = 17 22 35 48 63 16 29 40; (m) = 18 21 33 50 61 19 27 44; "
            "qs[32g+i] = ((i+g)%16) | (((15-i)%16) << 4)")
    return b, expected, rule


def q6_k_block():
    # ql[i] = i (i < 128); qh[i] = (37 i) & 255 (i < 64);
    # scales = 1 -1 2 -2 127 -128 3 4 5 6 7 8 -9 -10 11 12 ; d = 0.5 (0x3800, last)
    ql = list(range(128))
    qh = [(37 * i) & 255 for i in range(64)]
    sc = [1, -1, 2, -2, 127, -128, 3, 4, 5, 6, 7, 8, -9, -10, 11, 12]
    b = ql + qh + [s & 0xFF for s in sc] + [0x00, 0x38]
    expected = [
        (0, -16.0),     # h0 r0 i0: ql0=0, qh0=0 -> q=0; scale0=1: 0.5*1*(0-32)
        (15, 15.5),     # h0 r0 i15: ql15&15=15, qh15=43 (bits0-1 = 3) -> q=63; 0.5*1*31
        (37, 5.0),      # h0 r1 i5: ql37&15=5, qh5=185 (bits2-3 = 2) -> q=37; scale2=2: 0.5*2*5
        (65, 0.0),      # h0 r2 i1: ql1>>4=0, qh1=37 (bits4-5 = 2) -> q=32; scale4=127: 0
        (90, 1984.0),   # h0 r2 i26: ql26>>4=1, qh26=194 (bits4-5 = 0) -> q=1; scale5=-128: 0.5*-128*-31
        (127, -26.0),   # h0 r3 i31: ql63>>4=3, qh31=123 (bits6-7 = 1) -> q=19; scale7=4: 0.5*4*-13
        (128, -80.0),   # h1 r0 i0: ql64&15=0, qh32=160 (bits0-1 = 0) -> q=0; scale8=5: 0.5*5*-32
        (180, -48.0),   # h1 r1 i20: ql116&15=4, qh52=132 (bits2-3 = 1) -> q=20; scale11=8: 0.5*8*-12
        (200, 126.0),   # h1 r2 i8: ql72>>4=4, qh40=200 (bits4-5 = 0) -> q=4; scale12=-9: 0.5*-9*-28
        (255, -150.0),  # h1 r3 i31: ql127>>4=7, qh63=27 (bits6-7 = 0) -> q=7; scale15=12: 0.5*12*-25
    ]
    rule = ("ql[i] = i; qh[i] = (37*i) & 255; scales = 1 -1 2 -2 127 -128 3 4 5 6 7 8 -9 -10 11 12; "
            "d = 0.5")
    return b, expected, rule


def mxfp4_block(e):
    # qs[i] = i | ((15 - i) << 4): weight i has code i, weight 16+i has code 15-i.
    qs = [i | ((15 - i) << 4) for i in range(16)]
    b = [e] + qs
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    s = 2.0 ** (e - 127)
    expected = [(i, s * table[i]) for i in range(16)] + [(16 + i, s * table[15 - i]) for i in range(16)]
    rule = f"e = {e} (scale 2^{e - 127}); weight i has E2M1 code i, weight 16+i code 15-i"
    return b, expected, rule


# The IQ4 codebook as the format defines it (value of code 0..15), typed in.
IQ4 = [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113]


def iq4_nl_block():
    # d = 0.5 (0x3800); qs[i] = i | ((15 - i) << 4): weight i has code i,
    # weight 16+i has code 15-i. w = 0.5 * IQ4[code].
    b = [0x00, 0x38] + [i | ((15 - i) << 4) for i in range(16)]
    expected = [
        (0, -63.5),    # code 0: 0.5 * -127
        (7, -5.0),     # code 7: 0.5 * -10
        (8, 0.5),      # code 8: 0.5 * 1
        (15, 56.5),    # code 15: 0.5 * 113
        (16, 56.5),    # high nibble of qs[0] = 15
        (20, 19.0),    # high nibble of qs[4] = 11: 0.5 * 38
        (31, -63.5),   # high nibble of qs[15] = 0
    ]
    rule = "d = 0.5; qs[i] = i | ((15 - i) << 4): weight i has code i, weight 16+i code 15-i"
    return b, expected, rule


def iq4_xs_block():
    # d = 0.25 (0x3400). Sub-block scales ls = 32 33 31 40 0 63 16 48, i.e.
    # ls - 32 = 0 1 -1 8 -32 31 -16 16.
    #   scales_l (low nibbles, sub-block 2k in the low half of byte k):
    #     [0x10, 0x8F, 0xF0, 0x00]   (32&15=0, 33&15=1 | 31&15=15, 40&15=8 | 0, 63&15=15 | 16&15=0, 48&15=0)
    #   scales_h (bits 2b..2b+1 = ls_b >> 4): 2 2 1 2 0 3 1 3
    #     = 2 + 2*4 + 1*16 + 2*64 + 0*256 + 3*1024 + 1*4096 + 3*16384 = 56474 = 0xDC9A -> bytes 9A DC
    # qs[16b + j] = j | (((j + b) & 15) << 4): weight 32b+j has code j,
    # weight 32b+16+j has code (j + b) & 15.
    qs = [j | (((j + b) & 15) << 4) for b in range(8) for j in range(16)]
    b = [0x00, 0x34, 0x9A, 0xDC, 0x10, 0x8F, 0xF0, 0x00] + qs
    expected = [
        (0, 0.0),        # b0: ls - 32 = 0
        (32, -31.75),    # b1 j0: 0.25 * 1 * IQ4[0] = -127/4
        (48, -26.0),     # b1 high j0: code 1: 0.25 * 1 * -104
        (69, 8.75),      # b2 j5: 0.25 * -1 * IQ4[5] = -0.25 * -35
        (111, 226.0),    # b3 j15: 0.25 * 8 * 113
        (114, -70.0),    # b3 high j2: code 5: 2 * -35
        (137, -104.0),   # b4 j9: 0.25 * -32 * 13
        (186, 875.75),   # b5 high j10: code 15: 0.25 * 31 * 113
        (195, 260.0),    # b6 j3: 0.25 * -16 * -65
        (255, -88.0),    # b7 high j15: code (15 + 7) & 15 = 6: 0.25 * 16 * -22
    ]
    rule = ("d = 0.25; ls = 32 33 31 40 0 63 16 48; qs[16b+j] = j | (((j + b) & 15) << 4)")
    return b, expected, rule


def iq3_grid():
    # A test grid (the format's own grid is an input of the decoder): byte 0 of
    # entry i is 4 + 8 * (i & 7), byte 1 is 4 + 8 * ((i >> 3) & 7), byte 2 is
    # 4 + 8 * ((i >> 6) & 3), byte 3 is 62.
    return [(4 + 8 * (i & 7)) | ((4 + 8 * ((i >> 3) & 7)) << 8) | ((4 + 8 * ((i >> 6) & 3)) << 16) | (62 << 24)
            for i in range(256)]


def iq3_xxs_block():
    # d = 1.0 (0x3C00). Grid indices q[k] = (37 k + 5) & 255. Sub-block b's
    # word: sign indices s_l = (5 (4b + l)) & 127 in bits 7l.., scale 2b in
    # bits 28..31, so its scale is (0.5 + 2b) / 2 = 0.25 + b.
    q = [(37 * k + 5) & 255 for k in range(64)]
    words = []
    for blk in range(8):
        a = (2 * blk) << 28
        for l in range(4):
            a |= ((5 * (4 * blk + l)) & 127) << (7 * l)
        words += [a & 255, (a >> 8) & 255, (a >> 16) & 255, (a >> 24) & 255]
    b = [0x00, 0x3C] + q + words
    expected = [
        # b0 (scale 0.25), group 0: sign index 0 -> all positive; q0 = 5, q1 = 42
        (0, 11.0),     # grid[5] byte 0 = 4 + 8*5 = 44
        (1, 1.0),      # grid[5] byte 1 = 4
        (3, 15.5),     # byte 3 = 62
        (4, 5.0),      # grid[42] byte 0 = 4 + 8*2 = 20
        (5, 11.0),     # grid[42] byte 1 = 4 + 8*5 = 44
        # b0 group 1: sign index 5 = 0b101 (two bits, even): weights 0 and 2 negative; q2 = 79
        (8, -15.0),    # grid[79] byte 0 = 4 + 8*7 = 60
        (9, 3.0),      # byte 1 = 4 + 8*1 = 12
        (10, -3.0),    # byte 2 = 4 + 8*1 = 12, negative
        (11, 15.5),
        # b0 group 3: sign index 15 (four bits, even): weights 0-3 negative; q7 = 8 (weights 4-7)
        (28, 1.0),     # grid[8] byte 0 = 4
        (29, 3.0),     # grid[8] byte 1 = 12
        # b1 (scale 1.25), group 0: sign index 20 = 0b10100: weights 2 and 4 negative; q8 = 45, q9 = 82
        (32, 55.0),    # grid[45] byte 0 = 44
        (34, -5.0),    # grid[45] byte 2 = 4, negative
        (36, -25.0),   # grid[82] byte 0 = 20, negative
        (37, 25.0),    # grid[82] byte 1 = 20
        (38, 15.0),    # grid[82] byte 2 = 12
        (39, 77.5),    # byte 3 = 62
        # b1 group 1: sign index 25 = 0b11001 (three bits, odd): bit 7 set; weights 0, 3, 4, 7
        # negative; q10 = 119, q11 = 156
        (40, -75.0),   # grid[119] byte 0 = 60, negative
        (41, 65.0),    # grid[119] byte 1 = 4 + 8*6 = 52
        (43, -77.5),   # byte 3 = 62, negative
        (44, -45.0),   # grid[156] byte 0 = 4 + 8*4 = 36, negative
        (45, 35.0),    # grid[156] byte 1 = 4 + 8*3 = 28
        (47, -77.5),   # byte 3 = 62, negative (the implied eighth sign)
        # b7 (scale 7.25), group 0: sign index 140 & 127 = 12 = 0b1100: weights 2, 3 negative; q56 = 29
        (224, 319.0),  # grid[29] byte 0 = 44
        (226, -29.0),  # byte 2 = 4
        (227, -449.5),  # byte 3 = 62
    ]
    rule = ("d = 1.0; q[k] = (37k + 5) & 255; sub-block b: sign indices (5(4b + l)) & 127, scale 2b; "
            "grid entry i bytes 4+8(i&7), 4+8((i>>3)&7), 4+8((i>>6)&3), 62")
    return b, expected, rule


def t5_g128_block():
    # s = 0.5 (0x3800). Byte b (b < 26) holds weights 5b..5b+4 with base-3
    # digits (b + i) % 3 for i = 0..4, least significant first; w = 0.5 * (digit - 1).
    #   byte 0: digits 0 1 2 0 1 -> 0 + 3 + 18 + 0 + 81  = 102 (0x66)
    #   byte 1: digits 1 2 0 1 2 -> 1 + 6 + 0 + 27 + 162 = 196 (0xC4)
    #   byte 2: digits 2 0 1 2 0 -> 2 + 0 + 9 + 54 + 0   = 65  (0x41)
    # and the pattern repeats every three bytes.
    codes = [[102, 196, 65][b % 3] for b in range(26)]
    b = [0x00, 0x38] + codes
    expected = [
        (0, -0.5),     # byte 0 digit 0 = 0
        (1, 0.0),      # byte 0 digit 1 = 1
        (2, 0.5),      # byte 0 digit 2 = 2
        (4, 0.0),      # byte 0 digit 4 = 1
        (5, 0.0),      # byte 1 digit 0 = 1
        (9, 0.5),      # byte 1 digit 4 = 2
        (64, 0.0),     # byte 12 (like byte 0) digit 4 = 1
        (100, 0.5),    # byte 20 (like byte 2) digit 0 = 2
        (126, 0.5),    # byte 25 (like byte 1) digit 1 = 2
        (127, -0.5),   # byte 25 digit 2 = 0
    ]
    rule = "s = 0.5; byte b holds digits (b + i) % 3 for i = 0..4, least significant first"
    return b, expected, rule


def write(name, fmt, block, expected, rule, grid=None):
    path = os.path.join(HERE, name)
    with open(path, "w") as f:
        f.write(f"# Hand-built {fmt} block. Construction: {rule}\n")
        f.write("# Expected weights hand-computed from the block layout (see make_golden_blocks.py).\n")
        f.write("# Layout reading: GGUF block layouts (Q8_0/Q4_K/Q6_K/IQ4_NL/IQ4_XS/IQ3_XXS), OCP MX v1.0\n")
        f.write("# (MXFP4) and the base-3 packing of 'RTX 4080 SUPER 原生 Windows 跑 27B', 九.2 (T5_G128);\n")
        f.write("# format names from '三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南',\n")
        f.write("# 优化策略二.\n")
        f.write(f"format {fmt}\n")
        f.write("bytes " + " ".join(f"{x:02x}" for x in block) + "\n")
        if grid is not None:
            f.write("grid " + " ".join(f"{x:08x}" for x in grid) + "\n")
        for i, v in expected:
            f.write(f"w {i} {v!r}\n")


if __name__ == "__main__":
    write("q8_0_block.txt", "Q8_0", *q8_0_block())
    write("q8_0_half_block.txt", "Q8_0", *q8_0_half_block())
    write("q4_k_block.txt", "Q4_K", *q4_k_block())
    write("q6_k_block.txt", "Q6_K", *q6_k_block())
    write("mxfp4_e127_block.txt", "MXFP4", *mxfp4_block(127))
    write("mxfp4_e128_block.txt", "MXFP4", *mxfp4_block(128))
    write("iq4_nl_block.txt", "IQ4_NL", *iq4_nl_block())
    write("iq4_xs_block.txt", "IQ4_XS", *iq4_xs_block())
    write("iq3_xxs_block.txt", "IQ3_XXS", *iq3_xxs_block(), grid=iq3_grid())
    write("t5_g128_block.txt", "T5_G128", *t5_g128_block())
