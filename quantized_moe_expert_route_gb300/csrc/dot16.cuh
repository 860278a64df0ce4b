// Integer dot products of block-quantized weight rows with int16 activations,
// shared by the fused decode kernel and the streaming decode kernels.
//
// Activations: one row of x becomes int16 with a per-row power-of-two scale.
// For a 64-column group g of the row (columns 64 g .. 64 g + 63) a lane holds
// 32 words xq: xq[4m], xq[4m+1] are columns 4m .. 4m+3 of the group's first
// 32 (part A) and xq[4m+2], xq[4m+3] columns 4m .. 4m+3 of its second 32
// (part B), two int16 per word (lower column in the low half). Weight codes
// enter dp2a as bytes against these pairs, so every product and every sum
// inside a scale group is an exact int32; scales are applied in fp32 once per
// group.
//
// The formats follow the GGUF block layouts (Q8_0, Q4_K, Q6_K) and the OCP
// Microscaling v1.0 encoding for MXFP4 that the layer's tiers use ("三张 RTX
// 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南", section 优化策略二).
#pragma once

#include "moe_internal.cuh"

namespace moe {

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v & 0xffff))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v >> 16))); }

// Power-of-two scale for fp16: returns sigma with max * 2^sigma in [2^14, 2^15)
// (0 for max == 0), clamped so that 2^sigma and 2^-sigma are normal floats.
__device__ __forceinline__ int pow2_shift(float maxabs) {
    if (!(maxabs > 0.0f)) return 0;
    const int e = (int)((__float_as_uint(maxabs) >> 23) & 0xff);
    int s = 141 - e;
    return s < -126 ? -126 : (s > 126 ? 126 : s);
}
__device__ __forceinline__ float exp2i(int s) { return __uint_as_float((uint32_t)(127 + s) << 23); }

// Sums of 2 per-lane values over the warp: value 0 ends in lanes 0..15, value 1 in 16..31.
__device__ __forceinline__ float warp_reduce2(const float v[2]) {
    const bool b16 = threadIdx.x & 16;
    float y = (b16 ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, b16 ? v[0] : v[1], 16);
    y += __shfl_xor_sync(0xffffffffu, y, 8);
    y += __shfl_xor_sync(0xffffffffu, y, 4);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    return y;
}

// Scales and mins of Q4_K sub-blocks 2g and 2g+1 from the 12 scale bytes
// (three little-endian words), without branches: bytes j' = 2 (g & 1) and
// j' + 1 of each word; for g >= 2 the low four bits come from s[8..11] and
// the top two from bits 6-7 of s[0..3] (scales) and s[4..7] (mins).
__device__ __forceinline__ void q4k_pair_scales(int g, uint32_t s03, uint32_t s47, uint32_t s811, float &sc0,
                                                float &sc1, float &m0, float &m1) {
    const int sh = (g & 1) * 16;
    const uint32_t a = (s03 >> sh) & 0xFFFFu, m = (s47 >> sh) & 0xFFFFu, h = (s811 >> sh) & 0xFFFFu;
    const uint32_t sc_lo = a & 0x3F3Fu, mn_lo = m & 0x3F3Fu;
    const uint32_t sc_hi = (h & 0x0F0Fu) | ((a >> 2) & 0x3030u);
    const uint32_t mn_hi = ((h >> 4) & 0x0F0Fu) | ((m >> 2) & 0x3030u);
    const uint32_t scp = g < 2 ? sc_lo : sc_hi, mnp = g < 2 ? mn_lo : mn_hi;
    sc0 = (float)(scp & 0xFFu);
    sc1 = (float)(scp >> 8);
    m0 = (float)(mnp & 0xFFu);
    m1 = (float)(mnp >> 8);
}

__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
    return c;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
    return c;
}

// Four bytes at any byte address p of shared memory, from the two words that
// cover them (the word after the first is always read).
__device__ __forceinline__ uint32_t ld_u32_any(const uint8_t *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
    return __funnelshift_r(w[0], w[1], 8 * (uint32_t)(a & 3));
}
__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

// One lane's share of a Q4_K row dot product: the 64 weights of pair g of
// super-block blk (sub-blocks 2g, 2g+1) against xq, with XA, XB the sums of
// the activations of parts A and B. Q4_K: 144 bytes per 256 weights = fp16 d,
// fp16 dmin, 12 bytes of 6-bit (scale, min) pairs, 128 bytes of 4-bit codes;
// sub-blocks 2g and 2g+1 are the low and high nibbles of codes 32g .. 32g+31;
// w = d sc q - dmin m.
__device__ __forceinline__ float q4k_dot64(const uint8_t *blk, int g, const uint32_t xq[32], float XA, float XB) {
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const uint4 c0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * g);
    const uint4 c1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * g);
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    int sA0 = 0, sA1 = 0, sB0 = 0, sB1 = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t lo = cw[m] & 0x0F0F0F0Fu, hi = (cw[m] >> 4) & 0x0F0F0F0Fu;
        sA0 = dp2a_lo(xq[4 * m + 0], lo, sA0);
        sA1 = dp2a_hi(xq[4 * m + 1], lo, sA1);
        sB0 = dp2a_lo(xq[4 * m + 2], hi, sB0);
        sB1 = dp2a_hi(xq[4 * m + 3], hi, sB1);
    }
    float sc0, sc1, m0, m1;
    q4k_pair_scales(g, hdr.y, hdr.z, hdr.w, sc0, sc1, m0, m1);
    const float d = half_lo(hdr.x), dmin = half_hi(hdr.x);
    return d * (sc0 * (float)(sA0 + sA1) + sc1 * (float)(sB0 + sB1)) - dmin * (m0 * XA + m1 * XB);
}

// Q8_0 (34 bytes per 32 weights: fp16 d, 32 int8 codes; w = d q): group g is
// blocks 2g (part A) and 2g+1 (part B) of the row, 68 bytes from byte 68 g,
// which is 4-byte aligned. Block 2g's codes start 2 bytes into a word,
// block 2g+1's on a word.
__device__ __forceinline__ float q8_0_dot64(const uint8_t *row, int g, const uint32_t xq[32]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row + 68 * g);
    uint32_t W[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) W[i] = w[i];
    int sA = 0, sB = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t ca = __funnelshift_r(W[m], W[m + 1], 16);
        const uint32_t cb = W[9 + m];
        sA = dp2a_lo(xq[4 * m + 0], ca, sA);
        sA = dp2a_hi(xq[4 * m + 1], ca, sA);
        sB = dp2a_lo(xq[4 * m + 2], cb, sB);
        sB = dp2a_hi(xq[4 * m + 3], cb, sB);
    }
    return half_lo(W[0]) * (float)sA + half_hi(W[8]) * (float)sB;
}

// Q6_K (210 bytes per 256 weights: ql[128], qh[64], 16 int8 scales, fp16 d;
// w = d sc (q - 32), one scale per 16 weights). Group g is quarter j = g & 3
// of super-block g >> 2, weights 128 h + 64 o + [0, 64) with h = j >> 1,
// o = j & 1: part A is run r = 2o (nibble o of ql[64h + i], bits 4o, 4o+1 of
// qh[32h + i]), part B run r = 2o + 1 (nibble o of ql[64h + 32 + i], bits
// 4o+2, 4o+3 of qh[32h + i]); their scales are 8h + 4o + {0, 1} (A) and
// + {2, 3} (B). The codes enter dp2a unsigned; X16 holds the exact sums of
// the activations per 16 (A lo, A hi, B lo, B hi) for the -32 offset.
// A super-block starts 2 bytes into a word when g >> 2 is odd.
__device__ __forceinline__ float q6k_dot64(const uint8_t *row, int g, const uint32_t xq[32], int4 X16) {
    const int h = (g >> 1) & 1, o = g & 1;
    const uint8_t *sb = row + 210 * (g >> 2);
    const uint8_t *ql = sb + 64 * h, *qh = sb + 128 + 32 * h;
    const uint32_t ns = 4 * o;
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t la = ld_u32_any(ql + 4 * m), lb = ld_u32_any(ql + 32 + 4 * m), hb = ld_u32_any(qh + 4 * m);
        const uint32_t ca = ((la >> ns) & 0x0F0F0F0Fu) | (((hb >> ns) & 0x03030303u) << 4);
        const uint32_t cb = ((lb >> ns) & 0x0F0F0F0Fu) | (((hb >> (ns + 2)) & 0x03030303u) << 4);
        if (m < 4) {
            s0 = dp2a_lo(xq[4 * m + 0], ca, s0);
            s0 = dp2a_hi(xq[4 * m + 1], ca, s0);
            s2 = dp2a_lo(xq[4 * m + 2], cb, s2);
            s2 = dp2a_hi(xq[4 * m + 3], cb, s2);
        } else {
            s1 = dp2a_lo(xq[4 * m + 0], ca, s1);
            s1 = dp2a_hi(xq[4 * m + 1], ca, s1);
            s3 = dp2a_lo(xq[4 * m + 2], cb, s3);
            s3 = dp2a_hi(xq[4 * m + 3], cb, s3);
        }
    }
    const uint8_t *scp = sb + 192 + 8 * h + 4 * o;
    const uint32_t sa = ld_u16(scp), sbw = ld_u16(scp + 2);
    const float d = __half2float(__ushort_as_half((uint16_t)ld_u16(sb + 208)));
    const float f0 = (float)(int8_t)(sa & 0xff), f1 = (float)(int8_t)(sa >> 8);
    const float f2 = (float)(int8_t)(sbw & 0xff), f3 = (float)(int8_t)(sbw >> 8);
    // (s - 32 X) = sum (q - 32) x, below 2^24 in magnitude: exact in fp32
    return d * (f0 * (float)(s0 - 32 * X16.x) + f1 * (float)(s1 - 32 * X16.y) + f2 * (float)(s2 - 32 * X16.z) +
                f3 * (float)(s3 - 32 * X16.w));
}

// Four E2M1 codes (the low nibble of each byte of c) as four int8 values equal
// to twice the E2M1 value (0, 1, 2, 3, 4, 6, 8, 12 and their negatives; bit 3
// of a code is its sign), through byte permutations of two 8-entry tables.
__device__ __forceinline__ uint32_t e2m1x2_bytes(uint32_t c) {
    uint32_t s = (c | (c >> 4)) & 0x00FF00FFu;
    s = (s | (s >> 8)) & 0xFFFFu;   // code k in bits [4k, 4k + 4)
    const uint32_t idx = s & 0x7777u;
    const uint32_t pos = __byte_perm(0x03020100u, 0x0C080604u, idx);
    const uint32_t neg = __byte_perm(0xFDFEFF00u, 0xF4F8FAFCu, idx);
    return __byte_perm(pos, neg, 0x3210u | ((s & 0x8888u) >> 1));
}

// MXFP4 (17 bytes per 32 weights: E8M0 scale e, then 16 code bytes; weight
// i < 16 is the low nibble of code byte i, weight 16 + i its high nibble;
// w = 2^(e - 127) E2M1(code)): group g is blocks 2g (part A) and 2g + 1
// (part B), 34 bytes from byte 34 g. Part A's columns 4m .. 4m+3 are xq[4m],
// xq[4m+1], so code word i's low nibbles meet xq[4i..4i+1] and its high
// nibbles xq[4(i+4)..]; part B likewise on xq[4m+2], xq[4m+3].
__device__ __forceinline__ float mxfp4_dot64(const uint8_t *row, int g, const uint32_t xq[32]) {
    const uint8_t *b = row + 34 * g;
    int sA = 0, sB = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t wa = ld_u32_any(b + 1 + 4 * i), wb = ld_u32_any(b + 18 + 4 * i);
        const uint32_t al = e2m1x2_bytes(wa & 0x0F0F0F0Fu), ah = e2m1x2_bytes((wa >> 4) & 0x0F0F0F0Fu);
        const uint32_t bl = e2m1x2_bytes(wb & 0x0F0F0F0Fu), bh = e2m1x2_bytes((wb >> 4) & 0x0F0F0F0Fu);
        sA = dp2a_lo(xq[4 * i + 0], al, sA);
        sA = dp2a_hi(xq[4 * i + 1], al, sA);
        sA = dp2a_lo(xq[4 * (i + 4) + 0], ah, sA);
        sA = dp2a_hi(xq[4 * (i + 4) + 1], ah, sA);
        sB = dp2a_lo(xq[4 * i + 2], bl, sB);
        sB = dp2a_hi(xq[4 * i + 3], bl, sB);
        sB = dp2a_lo(xq[4 * (i + 4) + 2], bh, sB);
        sB = dp2a_hi(xq[4 * (i + 4) + 3], bh, sB);
    }
    return e8m0_half_scale(b[0]) * (float)sA + e8m0_half_scale(b[17]) * (float)sB;
}

}  // namespace moe
