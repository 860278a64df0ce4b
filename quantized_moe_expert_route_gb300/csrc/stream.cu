// Streaming grouped GEMV for decode batches of up to 16 token rows, any mix of
// the gate/up formats (Q8_0, Q4_K, Q6_K, MXFP4, IQ4_NL, IQ4_XS, IQ3_XXS) and
// Q8_0, MXFP4 or IQ4_NL down, and of up to 32 rows when every gate/up matrix
// is Q8_0 or Q4_K. Layers with IQ formats run a variant of the two kernels
// that carries their decoders.
//
// The grouped multi-session decode of "多卡 CUDA 张量并行：DwarfStar 如何在 8 张
// L40S 上跑出 120 t/s" (section 120 t/s 的秘密) reads each selected expert's
// weights once for all the rows that picked it; the tiered mul_mat_id of "三张
// RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南" (section
// 优化策略三) serves each expert in its own format. Here two persistent kernels
// (one CTA per SM, 16 warps) stream the weights:
//
//   gate/up: the active experts' gate/up rows, in chunks of 1, 2 or 4 row
//     pairs, are split over the CTAs by cost (rows times the expert's tokens,
//     plus the streaming), not by length. Warp w < 15 consumes the CTA's
//     chunks w, w + 15, ... from a ring of shared-memory slots that TMA bulk
//     copies fill; lanes 0-7 of warp 15 refill each slot with the chunk NS
//     ahead as soon as the slot's chunk is consumed, so no CTA-wide barrier
//     stands in the loop and no consumer waits on a copy it issued. A warp
//     holds its slot while it computes, so the chunk size is chosen to leave
//     slots in flight (HBM latency x bandwidth per SM) beyond those being
//     computed. For every row pair and every token of the chunk's expert the
//     warp forms both dot products (lane = 64-column group, int16
//     activations, dp2a on the codes) and writes h = silu(W_gate x) (W_up x)
//     in fp32.
//   down: the active experts' down rows are split the same way in chunks of
//     4 rows (8 lanes per row); each CTA first stages the h rows of the
//     pairs of its experts as int16 with a power-of-two scale per 32-block,
//     then writes y = W_down h in fp32 per pair; the combine kernel adds the
//     k rows of a token in slot order.
//
// The down kernel is launched with programmatic dependent launch: it reads
// its experts and issues its first weight copies while the gate/up kernel
// finishes, and waits for it only before reading h.
#include <algorithm>
#include <climits>

#include "moe_internal.cuh"
#include "dot16.cuh"

namespace moe {

namespace {

constexpr int SG_THREADS = 512;
constexpr int SG_WARPS = SG_THREADS / 32;
constexpr int SG_CONS = SG_WARPS - 1;   // consumer warps; lane 0 of the last warp refills the ring
constexpr int SG_MAX_SLOTS = 64;
// Row limits, from per-layer times of the 512-expert layer against the
// tensor-core path: with Q4_K gate/up the streaming kernels take 159, 179 and
// 273 us at 20, 24 and 32 rows against 226, 249 and 292 us; with the mixed
// tiers (Q6_K and MXFP4 dots cost 2.3-2.5 times Q4_K's per token) they break
// even at 16 rows (213 against 212 us) and lose beyond (249 against 240 us at
// 20 rows).
constexpr int SG_MAX_T = 32;        // Q8_0 / Q4_K gate/up
constexpr int SG_MAX_T_MIXED = 16;  // with Q6_K or MXFP4 gate/up
constexpr int SG_DN_ROWS = 4;   // down rows per chunk: 8 lanes per row
constexpr int SG_HQW = 20;      // words per staged 32-block of h: 16 int16 pairs, 2^-sigma, padding to 16 bytes

struct SgExp {
    DevMatrix a, b;   // gate, up (gate/up kernel) or down, unused (down kernel)
    int e, q0, n, pad;
};

struct SgArgs {
    const DevExpert *table;
    const int32_t *offsets, *pairs, *active;
    const uint16_t *x;   // bf16 [T, H]
    float *h;            // fp32 [kept pairs, I], bucket order
    float *y;            // fp32 [kept pairs, H], bucket order
    uint32_t *status;
    const uint32_t *grid;   // the IQ3_XXS grid (256 entries), or null
    int T, k, H, I, E;
    int cr, ns, stage, nexp;   // gate/up: row pairs per chunk, ring slots, slot bytes, experts per CTA (bound)
    int nsb, stageb, nq;       // down: ring slots, slot bytes, staged pairs per CTA (bound)
};

__device__ __forceinline__ void sg_flag(uint32_t *status, uint32_t f) {
    if (status) atomicOr(status, f);
}

// A slot's chunks j, j + ns, j + 2 ns, ... complete its mbarrier's phases
// 0, 1, 2, ...; a parity wait is only meaningful once the slot's previous
// phase has completed (a wait on the parity of a phase two ahead of the
// current one returns at once). Chunk j is issued only after chunk j - ns was
// consumed, so a consumer first waits (bounded) until the slot's issue record
// shows chunk j, then on the parity.
__device__ __forceinline__ bool sg_wait_chunk(uint64_t *full, const int *last, int s, int j, int ns) {
    const volatile int *l = last + s;
    if (*l != j) {
        const unsigned long long t0 = now_ns(), bound = *(volatile unsigned long long *)&g_wait_ns;
        for (uint32_t i = 0; *l != j; ++i) {
            if (i >= WAIT_LIMIT || now_ns() - t0 > bound) return false;
            __nanosleep(32);
        }
    }
    return mbar_wait_timed(&full[s], (uint32_t)(j / ns) & 1u);
}

// The ring's producer (warp 15): lane l < SG_PL issues the chunks
// j = ns + l, ns + l + SG_PL, ... in order, each into slot j % ns once that
// slot's previous chunk has been consumed (used[s] names the last chunk
// consumed from slot s). With ns a multiple of SG_PL every slot is served by
// one lane, and the lanes' copies go out together. False if a wait gave up.
constexpr int SG_PL = 8;
template <class Issue>
__device__ bool sg_produce(int ns, int n, const int *used, Issue issue) {
    const int lane = threadIdx.x & 31;
    int next = ns + lane;
    uint32_t idle = 0;
    const unsigned long long bound = *(volatile unsigned long long *)&g_wait_ns;
    unsigned long long t_idle = 0;
    for (;;) {
        const bool want = lane < SG_PL && next < n;
        if (!__any_sync(0xffffffffu, want)) return true;
        const bool ready = want && *reinterpret_cast<const volatile int *>(used + next % ns) == next - ns;
        if (ready) {
            issue(next);
            next += SG_PL;
        }
        if (__any_sync(0xffffffffu, ready)) {
            idle = 0;
        } else {
            const unsigned long long t = now_ns();
            if (idle == 0) t_idle = t;
            if (++idle >= WAIT_LIMIT || t - t_idle > bound) return false;
            __nanosleep(64);
        }
    }
}

// Waits (bounded, thread 0) for the last copy issued into every slot, so that
// no copy lands in the shared memory of an exited CTA.
__device__ void sg_drain(uint64_t *full, const int *last, int ns) {
    for (int s = 0; s < ns; ++s)
        if (last[s] >= 0) mbar_wait(&full[s], (uint32_t)(last[s] / ns) & 1u);
}

// ---- the IQ formats ("三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理
// 优化指南", 优化策略二: IQ4_XS gate/up with IQ4_NL down for the middle tier, IQ3_XXS
// gate/up for the tail). Codebook values and signed grid magnitudes enter dp2a
// as bytes, so the sums per scale group stay exact int32 as for the other
// formats.

// prmt.b32 in its default mode: a selector nibble with bit 3 set gives the
// selected byte's sign bit in all eight bits (__byte_perm ignores that bit).
__device__ __forceinline__ uint32_t sg_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// The codes of bytes 0..3 of w (low nibbles, or high nibbles with hi) as a
// 16-bit selector, code i in nibble i.
__device__ __forceinline__ uint32_t sg_nibble_sel(uint32_t w, bool hi) {
    const uint32_t v = hi ? (w >> 4) : w;
    const uint32_t x = (v & 0x000F000Fu) | ((v >> 4) & 0x00F000F0u);
    return __byte_perm(x, 0u, 0x0020u);
}
// The IQ4 codebook entries (signed bytes) of four codes (nibbles 0..3 of
// sel16): -127 -104 -83 -65 -49 -35 -22 -10 1 13 25 38 53 69 89 113, by a byte
// permute of each half of the book and a byte select from bit 3 of each code.
__device__ __forceinline__ uint32_t sg_iq4_bytes(uint32_t sel16) {
    const uint32_t s7 = sel16 & 0x7777u;
    const uint32_t lo = __byte_perm(0xBFAD9881u, 0xF6EADDCFu, s7);
    const uint32_t hi = __byte_perm(0x26190D01u, 0x71594535u, s7);
    const uint32_t m = sg_prmt(0u, 0x80808080u, ((sel16 >> 1) & 0x4444u) | 0x8888u);
    return (hi & m) | (lo & ~m);
}
// 32 IQ4 codes (words w[0..3]: weight i < 16 the low nibble of byte i, 16 + i
// the high nibble) against the activation pairs xq[o + 4m], xq[o + 4m + 1]
// of columns 4m .. 4m + 3 (o = 0: part A, 2: part B).
__device__ __forceinline__ int sg_iq4_sum32(const uint32_t (&w)[4], const uint32_t xq[32], int o) {
    int s = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = sg_iq4_bytes(sg_nibble_sel(w[k], false)), hi = sg_iq4_bytes(sg_nibble_sel(w[k], true));
        s = dp2a_lo(xq[4 * k + o], lo, s);
        s = dp2a_hi(xq[4 * k + o + 1], lo, s);
        s = dp2a_lo(xq[4 * (k + 4) + o], hi, s);
        s = dp2a_hi(xq[4 * (k + 4) + o + 1], hi, s);
    }
    return s;
}
// IQ4_XS (136 bytes per 256 weights: fp16 d, uint16 high scale bits, 4 bytes
// of low scale nibbles, 128 code bytes): group g is sub-blocks 2j, 2j + 1
// (j = g & 3) of super-block g >> 2, which starts on 8 bytes; scale
// d (ls - 32) with ls the 6-bit field of the sub-block.
__device__ __forceinline__ float iq4xs_dot64(const uint8_t *row, int g, const uint32_t xq[32]) {
    const uint8_t *sb = row + 136 * (g >> 2);
    const int j = g & 3;
    const uint2 hdr = *reinterpret_cast<const uint2 *>(sb);
    uint32_t wa[4], wb[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint2 a = *reinterpret_cast<const uint2 *>(sb + 8 + 32 * j + 8 * k);
        const uint2 b = *reinterpret_cast<const uint2 *>(sb + 24 + 32 * j + 8 * k);
        wa[2 * k] = a.x;
        wa[2 * k + 1] = a.y;
        wb[2 * k] = b.x;
        wb[2 * k + 1] = b.y;
    }
    const int sA = sg_iq4_sum32(wa, xq, 0), sB = sg_iq4_sum32(wb, xq, 2);
    const uint32_t sh = hdr.x >> 16;
    const int ja = 2 * j, jb = 2 * j + 1;
    const int lsA = (int)((hdr.y >> (8 * (ja >> 1) + 4 * (ja & 1))) & 15u) | (int)(((sh >> (2 * ja)) & 3u) << 4);
    const int lsB = (int)((hdr.y >> (8 * (jb >> 1) + 4 * (jb & 1))) & 15u) | (int)(((sh >> (2 * jb)) & 3u) << 4);
    return half_lo(hdr.x) * ((float)(lsA - 32) * (float)sA + (float)(lsB - 32) * (float)sB);
}
// IQ4_NL (18 bytes per 32 weights: fp16 d, 16 code bytes): group g is blocks
// 2g (part A) and 2g + 1 (part B), 36 bytes from byte 36 g (4-byte aligned).
__device__ __forceinline__ float iq4nl_dot64(const uint8_t *row, int g, const uint32_t xq[32]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row + 36 * g);
    uint32_t W[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) W[i] = w[i];
    // block A: d in the low half of W[0], codes from byte 2; block B: d in
    // the high half of W[4], codes from byte 20 (W[5..8])
    uint32_t wa[4], wb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        wa[k] = __funnelshift_r(W[k], W[k + 1], 16);
        wb[k] = W[5 + k];
    }
    return half_lo(W[0]) * (float)sg_iq4_sum32(wa, xq, 0) + half_hi(W[4]) * (float)sg_iq4_sum32(wb, xq, 2);
}
// IQ3_XXS (98 bytes per 256 weights: fp16 d, 64 grid-index bytes, 8 words of
// scale and signs): group g is sub-blocks 2j, 2j + 1 (j = g & 3) of
// super-block g >> 2 (2-byte aligned). Group l of 8 weights of sub-block b
// takes magnitudes from grid entries q[8b + 2l] (weights 0..3) and
// q[8b + 2l + 1] (4..7) and signs from its 7-bit index in word b with the
// parity as the eighth; scale d (0.5 + (word >> 28)) / 2. The magnitudes go to
// dp2a as unsigned bytes, and the ones with a sign bit again masked: sum =
// all - 2 negatives.
__device__ __forceinline__ int dp2a_lo_u8(uint32_t a, uint32_t b, int c) {
    asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
    return c;
}
__device__ __forceinline__ int dp2a_hi_u8(uint32_t a, uint32_t b, int c) {
    asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(c) : "r"(a), "r"(b));
    return c;
}
__device__ __forceinline__ int sg_iq3_sum32(const uint32_t q0, const uint32_t q1, uint32_t a, const uint32_t *grid,
                                            const uint32_t xq[32], int o) {
    int sp = 0, sn = 0;
#pragma unroll
    for (int l = 0; l < 4; ++l) {
        const uint32_t s7 = (a >> (7 * l)) & 127u;
        const uint32_t sb = s7 | ((__popc(s7) & 1u) << 7);
        const uint32_t qw = l < 2 ? q0 : q1;
        const uint32_t e0 = __ldg(grid + ((qw >> (16 * (l & 1))) & 0xffu));
        const uint32_t e1 = __ldg(grid + ((qw >> (16 * (l & 1) + 8)) & 0xffu));
        // bit i of a 4-bit sign field -> bit 7 of byte i, then each byte's bit 7 replicated
        const uint32_t m0 = sg_prmt((sb & 15u) * 0x10204080u, 0u, 0xBA98u);
        const uint32_t m1 = sg_prmt((sb >> 4) * 0x10204080u, 0u, 0xBA98u);
        sp = dp2a_lo_u8(xq[8 * l + o], e0, sp);
        sp = dp2a_hi_u8(xq[8 * l + o + 1], e0, sp);
        sp = dp2a_lo_u8(xq[8 * l + 4 + o], e1, sp);
        sp = dp2a_hi_u8(xq[8 * l + 4 + o + 1], e1, sp);
        sn = dp2a_lo_u8(xq[8 * l + o], e0 & m0, sn);
        sn = dp2a_hi_u8(xq[8 * l + o + 1], e0 & m0, sn);
        sn = dp2a_lo_u8(xq[8 * l + 4 + o], e1 & m1, sn);
        sn = dp2a_hi_u8(xq[8 * l + 4 + o + 1], e1 & m1, sn);
    }
    return sp - 2 * sn;
}
__device__ __forceinline__ float iq3xxs_dot64(const uint8_t *row, int g, const uint32_t xq[32], const uint32_t *grid) {
    const uint8_t *sb = row + 98 * (g >> 2);
    const int j = g & 3;
    const uint32_t qa0 = ld_u32_any(sb + 2 + 16 * j), qa1 = ld_u32_any(sb + 6 + 16 * j);
    const uint32_t qb0 = ld_u32_any(sb + 10 + 16 * j), qb1 = ld_u32_any(sb + 14 + 16 * j);
    const uint32_t aA = ld_u32_any(sb + 66 + 8 * j), aB = ld_u32_any(sb + 70 + 8 * j);
    const float d = __half2float(__ushort_as_half((uint16_t)ld_u16(sb)));
    const int sA = sg_iq3_sum32(qa0, qa1, aA, grid, xq, 0), sB = sg_iq3_sum32(qb0, qb1, aB, grid, xq, 2);
    return d * ((0.5f + (float)(aA >> 28)) * 0.5f * (float)sA + (0.5f + (float)(aB >> 28)) * 0.5f * (float)sB);
}

// One 64-column group of CR rows of gate and of up against one token.
template <int FMT, int CR>
__device__ __forceinline__ void sg_rows(const uint8_t *g0, int gs, const uint8_t *u0, int us, int G64,
                                        const uint32_t xv[32], int4 X16, float ag[CR], float au[CR],
                                        const uint32_t *grid) {
    const float XA = (float)(X16.x + X16.y), XB = (float)(X16.z + X16.w);
#pragma unroll
    for (int r = 0; r < CR; ++r) {
        const uint8_t *gr = g0 + r * gs, *ur = u0 + r * us;
        if constexpr (FMT == MOE_Q4_K) {
            ag[r] += q4k_dot64(gr + 144 * (G64 >> 2), G64 & 3, xv, XA, XB);
            au[r] += q4k_dot64(ur + 144 * (G64 >> 2), G64 & 3, xv, XA, XB);
        } else if constexpr (FMT == MOE_Q8_0) {
            ag[r] += q8_0_dot64(gr, G64, xv);
            au[r] += q8_0_dot64(ur, G64, xv);
        } else if constexpr (FMT == MOE_Q6_K) {
            ag[r] += q6k_dot64(gr, G64, xv, X16);
            au[r] += q6k_dot64(ur, G64, xv, X16);
        } else if constexpr (FMT == MOE_MXFP4) {
            ag[r] += mxfp4_dot64(gr, G64, xv);
            au[r] += mxfp4_dot64(ur, G64, xv);
        } else if constexpr (FMT == MOE_IQ4_XS) {
            ag[r] += iq4xs_dot64(gr, G64, xv);
            au[r] += iq4xs_dot64(ur, G64, xv);
        } else if constexpr (FMT == MOE_IQ4_NL) {
            ag[r] += iq4nl_dot64(gr, G64, xv);
            au[r] += iq4nl_dot64(ur, G64, xv);
        } else {
            ag[r] += iq3xxs_dot64(gr, G64, xv, grid);
            au[r] += iq3xxs_dot64(ur, G64, xv, grid);
        }
    }
}

// One chunk of the gate/up kernel: CR row pairs of one expert, every token of
// the expert. The slot holds the CR gate rows, then the CR up rows.
template <int FMT, int CR>
__device__ void sg_gateup_chunk(const SgArgs &A, const SgExp &X, const int *tok, const uint8_t *st, int r0,
                                const uint4 *xs4, const int4 *x16, const float *xsc) {
    const int lane = threadIdx.x & 31, H64 = A.H / 64;
    const int gs = (int)X.a.stride, us = (int)X.b.stride;
    const uint8_t *u0 = st + CR * gs;
    for (int qi = 0; qi < X.n; ++qi) {
        // an expert has at most T pairs unless a token repeats it
        const int t = qi < A.T ? tok[qi] : A.pairs[X.q0 + qi] / A.k;
        float ag[CR], au[CR];
#pragma unroll
        for (int r = 0; r < CR; ++r) ag[r] = au[r] = 0.0f;
        for (int G64 = lane; G64 < H64; G64 += 32) {
            uint32_t xv[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 q = xs4[((size_t)t * 8 + v) * H64 + G64];
                xv[4 * v + 0] = q.x;
                xv[4 * v + 1] = q.y;
                xv[4 * v + 2] = q.z;
                xv[4 * v + 3] = q.w;
            }
            sg_rows<FMT, CR>(st, gs, u0, us, G64, xv, x16[(size_t)t * H64 + G64], ag, au, A.grid);
        }
        const float s = xsc[t];
#pragma unroll
        for (int r = 0; r < CR; ++r) {
            const float v2[2] = {ag[r], au[r]};
            const float tot = warp_reduce2(v2) * s;   // gate in lanes 0..15, up in 16..31
            const float upv = __shfl_down_sync(0xffffffffu, tot, 16);
            if (lane == 0) A.h[(size_t)(X.q0 + qi) * A.I + r0 + r] = silu_f32(tot) * upv;
        }
    }
}

template <int CR, bool IQ>
__device__ __forceinline__ void sg_gateup_dispatch(const SgArgs &A, const SgExp &X, const int *tok, const uint8_t *st,
                                                   int r0, const uint4 *xs4, const int4 *x16, const float *xsc) {
    switch (X.a.fmt) {
        case MOE_Q4_K: sg_gateup_chunk<MOE_Q4_K, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
        case MOE_Q8_0: sg_gateup_chunk<MOE_Q8_0, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
        case MOE_Q6_K: sg_gateup_chunk<MOE_Q6_K, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
        case MOE_MXFP4: sg_gateup_chunk<MOE_MXFP4, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
        default:
            if constexpr (IQ) {
                switch (X.a.fmt) {
                    case MOE_IQ4_XS: sg_gateup_chunk<MOE_IQ4_XS, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
                    case MOE_IQ4_NL: sg_gateup_chunk<MOE_IQ4_NL, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
                    case MOE_IQ3_XXS: sg_gateup_chunk<MOE_IQ3_XXS, CR>(A, X, tok, st, r0, xs4, x16, xsc); break;
                    default: break;
                }
            }
            break;
    }
}

// Shared memory of the gate/up kernel after the ring (ring first, so that the
// 4-byte reads that run up to 7 bytes past a row stay inside the allocation).
struct SgLayoutA {
    size_t xs, x16, xsc, xsg, full, last, used, ex, tok, cost, total;
};
__host__ __device__ inline SgLayoutA sg_layout_a(int T, int H, int E, int ns, int stage, int nexp) {
    SgLayoutA L;
    size_t o = align_up((size_t)ns * stage + 16, 128);
    L.xs = o;
    o += (size_t)T * H * 2;
    L.x16 = o;
    o += (size_t)T * (H / 64) * 16;
    L.xsc = o;
    o = align_up(o + (size_t)T * 4, 16);
    L.xsg = o;
    o = align_up(o + (size_t)T * 4, 16);
    L.full = o;
    o += (size_t)SG_MAX_SLOTS * 8;
    L.last = o;
    o += (size_t)SG_MAX_SLOTS * 4;
    L.used = o;
    o += (size_t)SG_MAX_SLOTS * 4;
    L.ex = align_up(o, 16);
    o = L.ex + (size_t)nexp * sizeof(SgExp);
    L.tok = o;
    o += (size_t)nexp * T * 4;
    L.cost = align_up(o, 16);
    o = L.cost + (size_t)(E + 1) * 4;
    L.total = align_up(o, 128);
    return L;
}

struct SgLayoutB {
    size_t hq, full, last, used, ex, cost, total;
};
__host__ __device__ inline SgLayoutB sg_layout_b(int I, int E, int nsb, int stageb, int nq, int nexp) {
    SgLayoutB L;
    size_t o = align_up((size_t)nsb * stageb + 16, 128);
    L.hq = o;
    o += (size_t)nq * (I / 32) * SG_HQW * 4;
    L.full = align_up(o, 8);
    o = L.full + (size_t)SG_MAX_SLOTS * 8;
    L.last = o;
    o += (size_t)SG_MAX_SLOTS * 4;
    L.used = o;
    o += (size_t)SG_MAX_SLOTS * 4;
    L.ex = align_up(o, 16);
    o = L.ex + (size_t)nexp * sizeof(SgExp);
    L.cost = align_up(o, 16);
    o = L.cost + (size_t)(E + 1) * 4;
    L.total = align_up(o, 128);
    return L;
}

// The CTA's share of the chunk list [n_act experts x cpe chunks]: [c0, c1),
// its experts a0 .. a0 + na - 1 (indices into the active list). The list is
// split by cost, not by length: a chunk of expert a costs n_a + 1, its rows
// times the expert's n_a pairs of dot products plus one for streaming the
// rows, so the CTAs holding the rows of experts that many tokens picked get
// fewer of them. S: shared scratch of n_act + 1 ints (the prefix costs).
// Cost of one chunk of an expert in format f with n tokens: streaming its
// rows plus n dot products per row, in ns per gate/up row pair or per 4-row
// down chunk. Least-squares fits of the per-CTA times of 28 layers (4 to 16
// rows; Q4_K, Q8_0 and mixed tiers; globaltimer stamps in an instrumented
// copy) against each CTA's chunks by format, plus a constant per CTA, gave
// the down costs and the gate/up ratios: the Q6_K and MXFP4 dots cost 3.3
// and 3.8 times the Q4_K one per token, the Q8_0 one 0.65 times. The gate/up
// costs keep the Q4_K-only fit (45 + 65 n) and scale the other formats by
// those ratios: the joint fit's own Q4_K row (53 + 42 n) moved the cuts of
// the 16-row Q4_K layer and cost it 2.7%. The shares are cut by this cost:
// a split by tokens + 1 left the CTAs of the 6-row mixed-tier layer
// finishing between 32 and 65 us.
__device__ __forceinline__ int sg_chunk_cost(bool gateup, int f, int n) {
    if (gateup) {
        switch (f) {
            case MOE_Q8_0: return 91 + 42 * n;
            case MOE_Q6_K: return 41 + 217 * n;
            case MOE_MXFP4: return 42 + 245 * n;
            case MOE_IQ4_XS:   // codebook lookups like MXFP4's; IQ3_XXS two dots per grid entry
            case MOE_IQ4_NL: return 42 + 245 * n;
            case MOE_IQ3_XXS: return 41 + 217 * n;
            default: return 45 + 65 * n;   // Q4_K
        }
    }
    return f == MOE_Q8_0 ? 22 + 54 * n : 18 + 94 * n;   // Q8_0, or MXFP4 / IQ4_NL down, 4 rows
}
// Bounds that follow from the costs a + b n (n >= 1 per active expert, so a +
// b n <= (a + b) n): a gate/up chunk costs at least SG_GU_CMIN_CHUNK and a
// chunk row of the whole list at most SG_GU_CMAX_PAIR per pair; a down chunk
// at least SG_DN_CMIN_CHUNK, a row of the list at most SG_DN_CMAX_PAIR per
// pair, one more pair of an expert at least SG_DN_CMIN_TOKEN.
constexpr int SG_GU_CMIN_CHUNK = 110, SG_GU_CMAX_PAIR = 287;
constexpr int SG_DN_CMIN_CHUNK = 76, SG_DN_CMAX_PAIR = 112, SG_DN_CMIN_TOKEN = 54;
static_assert(SG_DN_CMAX_PAIR * SG_GU_CMIN_CHUNK <= SG_GU_CMAX_PAIR * SG_DN_CMIN_CHUNK,
              "the gate/up bound on experts per share covers the down kernel's");

__device__ void sg_range(const SgArgs &A, bool gateup, int n_act, int cpe, int *S, int &c0, int &nloc, int &a0,
                         int &na) {
    const int tid = threadIdx.x, lane = tid & 31;
    for (int a = tid; a < n_act; a += SG_THREADS) {
        const int e = A.active[1 + a];
        const int f = gateup ? A.table[e].gate.fmt : A.table[e].down.fmt;
        S[a] = cpe * sg_chunk_cost(gateup, f, A.offsets[e + 1] - A.offsets[e]);
    }
    __syncthreads();
    if (tid < 32) {   // exclusive prefix sums in place, S[n_act] = total
        const int per = (n_act + 31) / 32, b = min(n_act, lane * per), e = min(n_act, b + per);
        int sum = 0;
        for (int a = b; a < e; ++a) sum += S[a];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int a = b; a < e; ++a) {
            const int w = S[a];
            S[a] = run;
            run += w;
        }
        if (lane == 31) S[n_act] = incl;
    }
    __syncthreads();
    // the first chunk that starts at or after cost t
    auto chunk_at = [&](long long t) -> int {
        int lo = 0, hi = n_act;   // largest a with S[a] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (S[mid] <= t) lo = mid; else hi = mid - 1;
        }
        if (lo >= n_act) return n_act * cpe;
        const int w = (S[lo + 1] - S[lo]) / cpe;
        const long long k = (t - S[lo] + w - 1) / w;
        return lo * cpe + (k < cpe ? (int)k : cpe);
    };
    const long long tot = S[n_act];
    const int G = gridDim.x, c = blockIdx.x;
    c0 = chunk_at(tot * c / G);
    const int c1 = chunk_at(tot * (c + 1) / G);
    nloc = c1 - c0;
    a0 = nloc > 0 ? c0 / cpe : 0;
    na = nloc > 0 ? (c1 - 1) / cpe - a0 + 1 : 0;
}

// IQ: the variant that also decodes the IQ formats (layers without them keep
// the smaller code: with it the 16-row Q4_K layer measured 137.2 us against
// 135.0 us).
template <bool IQ>
__global__ void __launch_bounds__(SG_THREADS, 1) sg_gateup_kernel(SgArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = A.T, H = A.H, H64 = H / 64;
    const SgLayoutA L = sg_layout_a(T, H, A.E, A.ns, A.stage, A.nexp);
    uint8_t *ring = smem;
    uint4 *xs4 = reinterpret_cast<uint4 *>(smem + L.xs);   // [T][8][H/64]
    int4 *x16 = reinterpret_cast<int4 *>(smem + L.x16);    // [T][H/64] activation sums per 16
    float *xsc = reinterpret_cast<float *>(smem + L.xsc);  // [T] 2^-sigma
    int *xsg = reinterpret_cast<int *>(smem + L.xsg);      // [T] sigma
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    int *last = reinterpret_cast<int *>(smem + L.last);    // last chunk issued into each slot
    int *used = reinterpret_cast<int *>(smem + L.used);    // last chunk consumed from each slot
    SgExp *ex = reinterpret_cast<SgExp *>(smem + L.ex);
    int *tok = reinterpret_cast<int *>(smem + L.tok);      // [nexp][T] tokens of each expert's pairs

    // the routing comes from the previous kernels in the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_act = A.active[0], cpe = A.I / A.cr;
    int c0, nloc, a0, na;
    sg_range(A, true, n_act, cpe, reinterpret_cast<int *>(smem + L.cost), c0, nloc, a0, na);
    if (na > A.nexp) {   // beyond the planned bound (cannot happen): skip, flagged
        if (tid == 0) sg_flag(A.status, MOE_FLAG_WAIT_TIMEOUT);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < A.ns; ++s) {
            mbar_init(&full[s], 1);
            last[s] = -1;
            used[s] = -1;
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane < na) {
        const int e = A.active[1 + a0 + lane];
        SgExp X;
        X.a = A.table[e].gate;
        X.b = A.table[e].up;
        X.e = e;
        X.q0 = A.offsets[e];
        X.n = A.offsets[e + 1] - X.q0;
        X.pad = 0;
        ex[lane] = X;
    }
    __syncthreads();
    auto issue = [&](int j) {   // local chunk j into slot j % ns (one thread)
        const int gc = c0 + j, la = gc / cpe - a0, r0 = (gc - (gc / cpe) * cpe) * A.cr, s = j % A.ns;
        const SgExp &X = ex[la];
        const uint32_t bg = (uint32_t)(A.cr * X.a.stride), bu = (uint32_t)(A.cr * X.b.stride);
        uint8_t *dst = ring + (size_t)s * A.stage;
        mbar_expect_tx(&full[s], bg + bu);
        bulk_g2s(dst, X.a.data + (size_t)r0 * X.a.stride, bg, &full[s]);
        bulk_g2s(dst + bg, X.b.data + (size_t)r0 * X.b.stride, bu, &full[s]);
        *reinterpret_cast<volatile int *>(&last[s]) = j;
    };
    if (lane == 0)
        for (int j = warp; j < min(A.ns, nloc); j += SG_WARPS) issue(j);
    for (int i = tid; i < na * T; i += SG_THREADS) {
        const int la = i / T, qi = i - la * T;
        tok[i] = qi < ex[la].n ? A.pairs[ex[la].q0 + qi] / A.k : 0;
    }
    // activations: per-token power-of-two scale (max |x| in [2^14, 2^15))
    for (int t = warp; t < T; t += SG_WARPS) {
        const uint4 *src = reinterpret_cast<const uint4 *>(A.x + (size_t)t * H);
        float m = 0.0f;
        for (int i = lane; i < H / 8; i += 32) {
            const uint4 q = src[i];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) {
            const int sg = pow2_shift(m);
            xsg[t] = sg;
            xsc[t] = exp2i(-sg);
        }
    }
    __syncthreads();
    // int16 activations in the dot layout: four lanes per 64-column group, lane
    // q takes columns 8q .. 8q+7 of part A and of part B (uint4 words 2q, 2q+1)
    {
        const int ntask = 4 * T * H64;
        for (int base = warp * 32; base < ntask; base += SG_THREADS) {
            const int task = base + lane;
            const bool ok = task < ntask;
            const int g = ok ? task >> 2 : 0, q = task & 3;
            const int t = g / H64, G64 = g - t * H64;
            const float up = exp2i(xsg[t]);
            const uint4 *src = reinterpret_cast<const uint4 *>(A.x + (size_t)t * H) + 8 * G64;
            const uint4 qa = src[q], qb = src[4 + q];
            const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
            int ia[8], ib[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ia[2 * i] = max(-32767, min(32767, __float2int_rn(__uint_as_float(wa[i] << 16) * up)));
                ia[2 * i + 1] = max(-32767, min(32767, __float2int_rn(__uint_as_float(wa[i] & 0xffff0000u) * up)));
                ib[2 * i] = max(-32767, min(32767, __float2int_rn(__uint_as_float(wb[i] << 16) * up)));
                ib[2 * i + 1] = max(-32767, min(32767, __float2int_rn(__uint_as_float(wb[i] & 0xffff0000u) * up)));
            }
            int sa = 0, sb = 0;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int i = 4 * h2;
                const uint32_t w0 = ((uint32_t)ia[i] & 0xffffu) | ((uint32_t)ia[i + 1] << 16);
                const uint32_t w1 = ((uint32_t)ia[i + 2] & 0xffffu) | ((uint32_t)ia[i + 3] << 16);
                const uint32_t w2 = ((uint32_t)ib[i] & 0xffffu) | ((uint32_t)ib[i + 1] << 16);
                const uint32_t w3 = ((uint32_t)ib[i + 2] & 0xffffu) | ((uint32_t)ib[i + 3] << 16);
                if (ok) xs4[((size_t)t * 8 + 2 * q + h2) * H64 + G64] = make_uint4(w0, w1, w2, w3);
                sa += ia[i] + ia[i + 1] + ia[i + 2] + ia[i + 3];
                sb += ib[i] + ib[i + 1] + ib[i + 2] + ib[i + 3];
            }
            // lanes q = 0, 1 cover columns 0..15 of each part, q = 2, 3 columns 16..31
            sa += __shfl_xor_sync(0xffffffffu, sa, 1);
            sb += __shfl_xor_sync(0xffffffffu, sb, 1);
            const int sa_hi = __shfl_down_sync(0xffffffffu, sa, 2), sb_hi = __shfl_down_sync(0xffffffffu, sb, 2);
            if (ok && q == 0) x16[(size_t)t * H64 + G64] = make_int4(sa, sa_hi, sb, sb_hi);
        }
    }
    __syncthreads();
    // the down kernel may begin its launch (it waits for this grid before reading h)
    asm volatile("griddepcontrol.launch_dependents;");

    bool ok = true;
    if (warp < SG_CONS) {
        for (int j = warp; j < nloc; j += SG_CONS) {
            const int s = j % A.ns;
            const int gc = c0 + j, la = gc / cpe - a0, r0 = (gc - (gc / cpe) * cpe) * A.cr;
            if (!sg_wait_chunk(full, last, s, j, A.ns)) {
                ok = false;
                break;
            }
            const uint8_t *st = ring + (size_t)s * A.stage;
            const SgExp &X = ex[la];
            const int *tk = tok + la * T;
            if (A.cr == 4) sg_gateup_dispatch<4, IQ>(A, X, tk, st, r0, xs4, x16, xsc);
            else if (A.cr == 2) sg_gateup_dispatch<2, IQ>(A, X, tk, st, r0, xs4, x16, xsc);
            else sg_gateup_dispatch<1, IQ>(A, X, tk, st, r0, xs4, x16, xsc);
            __syncwarp();
            if (lane == 0) *reinterpret_cast<volatile int *>(&used[s]) = j;
        }
    } else {
        ok = sg_produce(A.ns, nloc, used, issue);
    }
    if (!ok && lane == 0) sg_flag(A.status, MOE_FLAG_WAIT_TIMEOUT);
    __syncwarp();
    __syncthreads();
    if (tid == 0) sg_drain(full, last, A.ns);
}

// Down: one 32-block b of a row against staged h (16 int16 pairs, 2^-sigma).
template <int FMT>
__device__ __forceinline__ float sg_down_block(const uint8_t *wrow, int b, const uint32_t *hb) {
    uint32_t hv[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 q = reinterpret_cast<const uint4 *>(hb)[v];
        hv[4 * v] = q.x;
        hv[4 * v + 1] = q.y;
        hv[4 * v + 2] = q.z;
        hv[4 * v + 3] = q.w;
    }
    const float hs = __uint_as_float(hb[16]);
    int s = 0;
    if constexpr (FMT == MOE_Q8_0) {
        // 34 bytes per block: fp16 d, then 32 int8 codes from byte 2
        const uint8_t *blk = wrow + 34 * b;
        const uintptr_t a = reinterpret_cast<uintptr_t>(blk + 2);
        const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
        const uint32_t sh = 8 * (uint32_t)(a & 3);
        uint32_t W[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) W[i] = w[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t c = __funnelshift_r(W[i], W[i + 1], sh);
            s = dp2a_lo(hv[2 * i], c, s);
            s = dp2a_hi(hv[2 * i + 1], c, s);
        }
        return __half2float(__ushort_as_half((uint16_t)ld_u16(blk))) * hs * (float)s;
    } else if constexpr (FMT == MOE_MXFP4) {
        // MXFP4, 17 bytes per block: E8M0 e, then 16 code bytes
        const uint8_t *blk = wrow + 17 * b;
        const uintptr_t a = reinterpret_cast<uintptr_t>(blk + 1);
        const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
        const uint32_t sh = 8 * (uint32_t)(a & 3);
        uint32_t W[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) W[i] = w[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t c = __funnelshift_r(W[i], W[i + 1], sh);
            const uint32_t lo = e2m1x2_bytes(c & 0x0F0F0F0Fu), hi = e2m1x2_bytes((c >> 4) & 0x0F0F0F0Fu);
            s = dp2a_lo(hv[2 * i], lo, s);
            s = dp2a_hi(hv[2 * i + 1], lo, s);
            s = dp2a_lo(hv[8 + 2 * i], hi, s);
            s = dp2a_hi(hv[8 + 2 * i + 1], hi, s);
        }
        return e8m0_half_scale(blk[0]) * hs * (float)s;
    } else {
        // IQ4_NL, 18 bytes per 32 weights: fp16 d, then 16 code bytes
        const uint8_t *blk = wrow + 18 * b;
        const uintptr_t a = reinterpret_cast<uintptr_t>(blk + 2);
        const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
        const uint32_t sh = 8 * (uint32_t)(a & 3);
        uint32_t W[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) W[i] = w[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t c = __funnelshift_r(W[i], W[i + 1], sh);
            const uint32_t lo = sg_iq4_bytes(sg_nibble_sel(c, false)), hi = sg_iq4_bytes(sg_nibble_sel(c, true));
            s = dp2a_lo(hv[2 * i], lo, s);
            s = dp2a_hi(hv[2 * i + 1], lo, s);
            s = dp2a_lo(hv[8 + 2 * i], hi, s);
            s = dp2a_hi(hv[8 + 2 * i + 1], hi, s);
        }
        return __half2float(__ushort_as_half((uint16_t)ld_u16(blk))) * hs * (float)s;
    }
}

// A Q8_0 block of a row that starts on 16 bytes, with the parity of b known:
// block b starts at byte 34 b, so an even block starts on a word (its scale
// in the low half of the word, its codes 2 bytes in) and an odd block 2 bytes
// into one (its scale in the high half, its codes on a word). Each code pair
// is then one half of a word at a fixed place, which dp2a.lo or dp2a.hi reads
// as it is: no funnel shifts. The same integer sum and the same fp32 product
// as sg_down_block.
template <bool ODD>
__device__ __forceinline__ float sg_down_q8_0_fixed(const uint8_t *wrow, int b, const uint32_t *hb) {
    uint32_t hv[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 q = reinterpret_cast<const uint4 *>(hb)[v];
        hv[4 * v] = q.x;
        hv[4 * v + 1] = q.y;
        hv[4 * v + 2] = q.z;
        hv[4 * v + 3] = q.w;
    }
    const float hs = __uint_as_float(hb[16]);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(wrow + 34 * b - (ODD ? 2 : 0));
    uint32_t W[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) W[i] = w[i];
    int s = 0;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        // code pair m: bytes 2 + 2m (even block) or 4 + 2m (odd) of the words
        const int word = ODD ? 1 + (m >> 1) : (m + 1) >> 1;
        const bool hi = ODD ? (m & 1) != 0 : ((m + 1) & 1) != 0;
        s = hi ? dp2a_hi(hv[m], W[word], s) : dp2a_lo(hv[m], W[word], s);
    }
    return (ODD ? half_hi(W[0]) : half_lo(W[0])) * hs * (float)s;
}

// Where block b of a staged h row sits: in each whole group of 16 blocks the
// even blocks come first, then the odd ones, so the eight lanes of a row that
// read blocks 2i (or 2i + 1) of a group read consecutive staged blocks (80
// bytes apart: no bank conflicts); blocks after the last whole group stay.
__device__ __forceinline__ int sg_hslot(int b, int U) {
    return b < (U & ~15) ? (b & ~15) + ((b & 1) << 3) + ((b & 15) >> 1) : b;
}

template <int FMT>
__device__ void sg_down_chunk(const SgArgs &A, const SgExp &X, const uint8_t *st, int r0, const uint32_t *hq,
                              int qbase) {
    const int lane = threadIdx.x & 31, row = lane >> 3, qd = lane & 7, U = A.I / 32;
    const uint8_t *wrow = st + (size_t)row * X.a.stride;
    for (int qi = 0; qi < X.n; ++qi) {
        const int q = X.q0 + qi;
        const uint32_t *hrow = hq + (size_t)(q - qbase) * U * SG_HQW;
        float acc = 0.0f;
        // blocks in groups of 16: lane qd takes 2 qd and 2 qd + 1, so for
        // Q8_0 the warp runs one block parity at a time (sg_down_q8_0_fixed),
        // and the staged h of both lie 80 bytes apart across the lanes
        // (sg_hslot); the blocks after the last whole group as before
        const int full = U / 16;
        for (int o = 0; o < full; ++o) {
            const int b = 16 * o + 2 * qd;
            const uint32_t *h0 = hrow + (16 * o + qd) * SG_HQW, *h1 = hrow + (16 * o + 8 + qd) * SG_HQW;
            if constexpr (FMT == MOE_Q8_0) {
                acc += sg_down_q8_0_fixed<false>(wrow, b, h0);
                acc += sg_down_q8_0_fixed<true>(wrow, b + 1, h1);
            } else {
                acc += sg_down_block<FMT>(wrow, b, h0);
                acc += sg_down_block<FMT>(wrow, b + 1, h1);
            }
        }
        for (int b = 16 * full + qd; b < U; b += 8) acc += sg_down_block<FMT>(wrow, b, hrow + b * SG_HQW);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (qd == 0) A.y[(size_t)q * A.H + r0 + row] = acc;
    }
}

template <bool IQ>
__global__ void __launch_bounds__(SG_THREADS, 1) sg_down_kernel(SgArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int U = A.I / 32;
    const SgLayoutB L = sg_layout_b(A.I, A.E, A.nsb, A.stageb, A.nq, A.nexp);
    uint8_t *ring = smem;
    uint32_t *hq = reinterpret_cast<uint32_t *>(smem + L.hq);   // [staged pairs][U][SG_HQW]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    int *last = reinterpret_cast<int *>(smem + L.last);
    int *used = reinterpret_cast<int *>(smem + L.used);
    SgExp *ex = reinterpret_cast<SgExp *>(smem + L.ex);

    // The routing was complete before the gate/up kernel began (it waited for
    // it), and this kernel starts after that kernel's trigger: the experts and
    // the first weight copies need no wait.
    const int n_act = A.active[0], cpe = A.H / SG_DN_ROWS;
    int c0, nloc, a0, na;
    sg_range(A, false, n_act, cpe, reinterpret_cast<int *>(smem + L.cost), c0, nloc, a0, na);
    if (na > A.nexp) {
        if (tid == 0) sg_flag(A.status, MOE_FLAG_WAIT_TIMEOUT);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < A.nsb; ++s) {
            mbar_init(&full[s], 1);
            last[s] = -1;
            used[s] = -1;
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane < na) {
        const int e = A.active[1 + a0 + lane];
        SgExp X;
        X.a = A.table[e].down;
        X.b = X.a;
        X.e = e;
        X.q0 = A.offsets[e];
        X.n = A.offsets[e + 1] - X.q0;
        X.pad = 0;
        ex[lane] = X;
    }
    __syncthreads();
    auto issue = [&](int j) {
        const int gc = c0 + j, la = gc / cpe - a0, r0 = (gc - (gc / cpe) * cpe) * SG_DN_ROWS, s = j % A.nsb;
        const SgExp &X = ex[la];
        const uint32_t bd = (uint32_t)(SG_DN_ROWS * X.a.stride);
        mbar_expect_tx(&full[s], bd);
        bulk_g2s(ring + (size_t)s * A.stageb, X.a.data + (size_t)r0 * X.a.stride, bd, &full[s]);
        *reinterpret_cast<volatile int *>(&last[s]) = j;
    };
    if (lane == 0)
        for (int j = warp; j < min(A.nsb, nloc); j += SG_WARPS) issue(j);

    // h of the gate/up kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int qbase = na > 0 ? ex[0].q0 : 0;
    const int nql = na > 0 ? ex[na - 1].q0 + ex[na - 1].n - qbase : 0;   // the experts' pairs are contiguous
    bool ok = nql <= A.nq;
    if (ok) {
        // eight threads per 32-block: four values each, a shared maximum, then
        // 16 int16 pairs and 2^-sigma with max |h| 2^sigma in [2^13, 2^14)
        const int ntask = nql * U * 8;
        for (int base = warp * 32; base < ntask; base += SG_THREADS) {
            const int task = base + lane;
            const bool in = task < ntask;
            const int blk = in ? task >> 3 : 0, part = task & 7;
            const int qq = blk / U, b = blk - qq * U;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (in) v = __ldcg(reinterpret_cast<const float4 *>(A.h + (size_t)(qbase + qq) * A.I + 32 * b) + part);
            float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            if (!in) continue;
            uint32_t *dst = hq + ((size_t)qq * U + sg_hslot(b, U)) * SG_HQW;
            const int be = (int)((__float_as_uint(m) >> 23) & 0xffu);
            if (be == 255) {   // inf or nan in the block: it propagates
                *reinterpret_cast<uint2 *>(dst + 2 * part) = make_uint2(0u, 0u);
                if (part == 0) dst[16] = 0x7fc00000u;
                continue;
            }
            const int sg = m > 0.0f ? max(-100, min(100, 140 - be)) : 0;
            const float up = __uint_as_float((uint32_t)(127 + sg) << 23);
            const int q0 = __float2int_rn(v.x * up), q1 = __float2int_rn(v.y * up);
            const int q2 = __float2int_rn(v.z * up), q3 = __float2int_rn(v.w * up);
            *reinterpret_cast<uint2 *>(dst + 2 * part) =
                make_uint2(((uint32_t)q0 & 0xffffu) | ((uint32_t)q1 << 16), ((uint32_t)q2 & 0xffffu) | ((uint32_t)q3 << 16));
            if (part == 0) dst[16] = (uint32_t)(127 - sg) << 23;
        }
    }
    __syncthreads();
    if (ok && warp < SG_CONS) {
        for (int j = warp; j < nloc; j += SG_CONS) {
            const int s = j % A.nsb;
            const int gc = c0 + j, la = gc / cpe - a0, r0 = (gc - (gc / cpe) * cpe) * SG_DN_ROWS;
            if (!sg_wait_chunk(full, last, s, j, A.nsb)) {
                ok = false;
                break;
            }
            const SgExp &X = ex[la];
            const uint8_t *st = ring + (size_t)s * A.stageb;
            if (X.a.fmt == MOE_Q8_0) sg_down_chunk<MOE_Q8_0>(A, X, st, r0, hq, qbase);
            else if (!IQ || X.a.fmt == MOE_MXFP4) sg_down_chunk<MOE_MXFP4>(A, X, st, r0, hq, qbase);
            else if constexpr (IQ) sg_down_chunk<MOE_IQ4_NL>(A, X, st, r0, hq, qbase);
            __syncwarp();
            if (lane == 0) *reinterpret_cast<volatile int *>(&used[s]) = j;
        }
    } else if (ok) {
        ok = sg_produce(A.nsb, nloc, used, issue);
    }
    if (!ok && lane == 0) sg_flag(A.status, MOE_FLAG_WAIT_TIMEOUT);
    __syncwarp();
    __syncthreads();
    if (tid == 0) sg_drain(full, last, A.nsb);
}

int optin_smem() {
    static int cached[64] = {};
    const int dev = current_device();
    if (dev < 64 && cached[dev]) return cached[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev] = v;
    return v;
}

}  // namespace

SgPlan stream_plan(int T, int k, int E, int H, int I, uint32_t gu_formats, uint32_t down_formats, int64_t gu_stride,
                   int64_t dn_stride) {
    SgPlan p{};
    p.ok = false;
    const int G = sm_count(), optin = optin_smem();
    if (G <= 0 || optin <= 0) return p;
    if (T < 1 || T > SG_MAX_T || H % 64 != 0 || I % 32 != 0 || H % SG_DN_ROWS != 0) return p;
    if (T > SG_MAX_T_MIXED && (gu_formats & ~((1u << MOE_Q8_0) | (1u << MOE_Q4_K))) != 0) return p;
    if ((down_formats & ~((1u << MOE_Q8_0) | (1u << MOE_MXFP4) | (1u << MOE_IQ4_NL))) != 0) return p;
    if ((gu_formats & ~((1u << MOE_Q8_0) | (1u << MOE_Q4_K) | (1u << MOE_Q6_K) | (1u << MOE_MXFP4) |
                        (1u << MOE_IQ4_XS) | (1u << MOE_IQ4_NL) | (1u << MOE_IQ3_XXS))) != 0)
        return p;
    if (gu_stride <= 0 || dn_stride <= 0 || gu_stride % 16 != 0 || dn_stride % 16 != 0) return p;
    const int P = T * k, nmax = std::min(P, E);
    p.iq = ((gu_formats | down_formats) &
            ((1u << MOE_IQ4_XS) | (1u << MOE_IQ4_NL) | (1u << MOE_IQ3_XXS))) != 0;
    // the prefix costs of sg_range are ints: chunks per expert (at most I or
    // H / 4) times the list's cost per chunk row
    if ((long long)I * SG_GU_CMAX_PAIR * P > INT_MAX || (long long)(H / SG_DN_ROWS) * SG_DN_CMAX_PAIR * P > INT_MAX)
        return p;
    // experts one CTA's share can touch (sg_chunk_cost): an expert costs at
    // least SG_GU_CMIN_CHUNK per chunk, the whole list at most SG_GU_CMAX_PAIR
    // * P per chunk row, so a share holds at most SG_GU_CMAX_PAIR * P /
    // (SG_GU_CMIN_CHUNK * G) whole experts plus the two it starts and ends in
    // (fewer in the down kernel's shares)
    p.nexp = (int)(((long long)SG_GU_CMAX_PAIR * P + (long long)SG_GU_CMIN_CHUNK * G - 1) /
                   ((long long)SG_GU_CMIN_CHUNK * G)) + 2;
    // gate/up: each of the 15 consumer warps holds one slot while it
    // computes, so the slots beyond 15 are the copies in flight: the largest
    // chunk (4, 2 or 1 row pairs) that gives at least 24 slots (the 6-row
    // mixed-tier layer: 121 us with 2-pair chunks in 24 slots, 123 us with
    // 1-pair chunks in 56)
    const size_t fixed_a = sg_layout_a(T, H, E, 0, 0, p.nexp).total;
    if ((size_t)optin <= fixed_a + 16) return p;
    const size_t budget_a = (size_t)optin - fixed_a - 16;
    {
        const int min_ns = 24;
        for (int cr : {4, 2, 1}) {
            if (I % cr != 0) continue;
            const size_t stage = (size_t)2 * cr * gu_stride;
            const size_t ns = std::min<size_t>(SG_MAX_SLOTS, budget_a / stage) / SG_PL * SG_PL;
            if (ns >= (size_t)min_ns) {
                p.cr = cr;
                p.stage = (int)stage;
                p.ns = (int)ns;
                break;
            }
        }
    }
    if (p.cr == 0) return p;
    p.smem_a = sg_layout_a(T, H, E, p.ns, p.stage, p.nexp).total;
    // down: 4 rows per chunk, at least 24 slots
    // pairs of the experts of one down share: the whole experts' pairs cost at
    // least SG_DN_CMIN_TOKEN each, so there are at most SG_DN_CMAX_PAIR * P /
    // (SG_DN_CMIN_TOKEN * G) of them, plus the two partial experts' T each
    p.nq = std::min(P, (int)(((long long)SG_DN_CMAX_PAIR * P + (long long)SG_DN_CMIN_TOKEN * G - 1) /
                             ((long long)SG_DN_CMIN_TOKEN * G)) + 2 * T);
    p.stageb = (int)(SG_DN_ROWS * dn_stride);
    const size_t fixed_b = sg_layout_b(I, E, 0, 0, p.nq, p.nexp).total;
    if ((size_t)optin <= fixed_b + 16) return p;
    p.nsb = (int)(std::min<size_t>(SG_MAX_SLOTS, ((size_t)optin - fixed_b - 16) / p.stageb) / SG_PL * SG_PL);
    if (p.nsb < 24) return p;
    p.smem_b = sg_layout_b(I, E, p.nsb, p.stageb, p.nq, p.nexp).total;
    p.ok = p.smem_a <= (size_t)optin && p.smem_b <= (size_t)optin;
    return p;
}

cudaError_t launch_stream_path(const DevExpert *table, const SgPlan &p, int T, int k, int E, int H, int I,
                               const int32_t *offsets, const int32_t *pairs, const int32_t *active, const uint16_t *x,
                               float *h, float *y, uint32_t *status, const uint32_t *grid, cudaEvent_t const *events,
                               cudaStream_t s) {
    static bool attr_done[64] = {};
    const int dev = current_device();
    if (dev >= 64 || !attr_done[dev]) {
        cudaError_t err = allow_max_dynamic_smem(reinterpret_cast<const void *>(sg_gateup_kernel<false>));
        if (err == cudaSuccess) err = allow_max_dynamic_smem(reinterpret_cast<const void *>(sg_down_kernel<false>));
        if (err == cudaSuccess) err = allow_max_dynamic_smem(reinterpret_cast<const void *>(sg_gateup_kernel<true>));
        if (err == cudaSuccess) err = allow_max_dynamic_smem(reinterpret_cast<const void *>(sg_down_kernel<true>));
        if (err != cudaSuccess) return err;
        if (dev < 64) attr_done[dev] = true;
    }
    SgArgs A{};
    A.table = table;
    A.offsets = offsets;
    A.pairs = pairs;
    A.active = active;
    A.x = x;
    A.h = h;
    A.y = y;
    A.status = status;
    A.grid = grid;
    A.T = T;
    A.k = k;
    A.H = H;
    A.I = I;
    A.E = E;
    A.cr = p.cr;
    A.ns = p.ns;
    A.stage = p.stage;
    A.nexp = p.nexp;
    A.nsb = p.nsb;
    A.stageb = p.stageb;
    A.nq = p.nq;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(sm_count());
    cfg.blockDim = dim3(SG_THREADS);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (events && (err = record_event(events[0], s)) != cudaSuccess) return err;
    cfg.dynamicSmemBytes = p.smem_a;
    err = p.iq ? cudaLaunchKernelEx(&cfg, sg_gateup_kernel<true>, A) : cudaLaunchKernelEx(&cfg, sg_gateup_kernel<false>, A);
    if (err != cudaSuccess) return err;
    // with timing events the down kernel's early start (its prologue under
    // the gate/up kernel's tail) is given up for a clean split
    if (events && (err = record_event(events[1], s)) != cudaSuccess) return err;
    cfg.dynamicSmemBytes = p.smem_b;
    err = p.iq ? cudaLaunchKernelEx(&cfg, sg_down_kernel<true>, A) : cudaLaunchKernelEx(&cfg, sg_down_kernel<false>, A);
    if (err != cudaSuccess) return err;
    if (events && (err = record_event(events[2], s)) != cudaSuccess) return err;
    return cudaSuccess;
}

// This file's copy of the wait bound (moe_set_wait_timeout_ns).
cudaError_t set_wait_ns_stream(unsigned long long ns) { return set_tu_wait_ns(ns); }

}  // namespace moe
