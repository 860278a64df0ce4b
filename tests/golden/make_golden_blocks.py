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


def write(name, fmt, block, expected, rule):
    path = os.path.join(HERE, name)
    with open(path, "w") as f:
        f.write(f"# Hand-built {fmt} block. Construction: {rule}\n")
        f.write("# Expected weights hand-computed from the block layout (see make_golden_blocks.py).\n")
        f.write("# Layout reading: GGUF block layouts (Q8_0/Q4_K/Q6_K), OCP MX v1.0 (MXFP4); format names from\n")
        f.write("# '三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南', 优化策略二.\n")
        f.write(f"format {fmt}\n")
        f.write("bytes " + " ".join(f"{x:02x}" for x in block) + "\n")
        for i, v in expected:
            f.write(f"w {i} {v!r}\n")


if __name__ == "__main__":
    write("q8_0_block.txt", "Q8_0", *q8_0_block())
    write("q8_0_half_block.txt", "Q8_0", *q8_0_half_block())
    write("q4_k_block.txt", "Q4_K", *q4_k_block())
    write("q6_k_block.txt", "Q6_K", *q6_k_block())
    write("mxfp4_e127_block.txt", "MXFP4", *mxfp4_block(127))
    write("mxfp4_e128_block.txt", "MXFP4", *mxfp4_block(128))
