// Grouped GEMV path (decode rows): gate/up with the fused SwiGLU, down
// projection, and the slot-ordered combine.
//
// Each CTA takes one (active expert, tile of rows) work unit, so an expert's
// quantized rows are streamed from HBM once per layer no matter how many of
// the batch's tokens picked it: the grouped multi-session decode of "多卡 CUDA
// 张量并行：DwarfStar 如何在 8 张 L40S 上跑出 120 t/s" (section 120 t/s 的秘密), and the
// per-expert-format dispatch of the tiered mul_mat_id in "三张 RTX 3090 显卡实现
// Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南" (section 优化策略三), here done by
// a per-CTA switch on the expert's format tag inside one launch. The gate and
// up rows of a tile are used together, so the activation is fused (section
// 关键 Bug 修复与调试踩坑记录, item 4; "一张 RTX 3090 跑 Llama 70B", section 4.4).
//
// A tile's bytes are staged into shared memory by the TMA engine (one 1-D
// cp.async.bulk per matrix, completion on an mbarrier), then decoded from
// shared memory. Weights are dequantized exactly in fp32 registers and
// multiplied with fp32 activations, fp32 accumulation.
//
// Every format is handled as 32-weight units: w_i = s_i * c_i - m with small
// integer codes c_i (exact in fp32), s_i = s_lo for i < 16 and s_hi for i >= 16.
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {

namespace {

constexpr int GV_THREADS = 256;
constexpr int GV_SLICES = 8;                        // threads sharing one row-dot
constexpr int GV_ROWDOTS = GV_THREADS / GV_SLICES;  // 32 row-dots per CTA pass
constexpr int GU_ROWS = GV_ROWDOTS / 2;             // gate/up: 16 rows of each
constexpr int DN_ROWS = GV_ROWDOTS;                 // down: 32 rows
constexpr int GV_NT = 4;                            // tokens per pass

struct Unit {
    float c[32];
    float s_lo, s_hi, m;
};

__device__ __forceinline__ uint16_t ld16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

template <int FMT>
__device__ __forceinline__ void decode_unit(const uint8_t *row, int u, Unit &U);

// Q8_0: 34 B = fp16 d | int8 q[32]; w = d * q.
template <>
__device__ __forceinline__ void decode_unit<MOE_Q8_0>(const uint8_t *row, int u, Unit &U) {
    const uint8_t *b = row + 34 * u;
    float d = half_bits_to_f32(ld16(b));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint16_t two = ld16(b + 2 + 2 * i);
        U.c[2 * i] = (float)(int8_t)(two & 0xff);
        U.c[2 * i + 1] = (float)(int8_t)(two >> 8);
    }
    U.s_lo = U.s_hi = d;
    U.m = 0.0f;
}

// Q4_K: 144 B per 256 = fp16 d | fp16 dmin | 12 B packed (scale, min) | 128 B
// codes. Unit u is sub-block j = u % 8 of super-block u / 8: codes are the low
// (j even) or high (j odd) nibbles of qs[32 (j/2) .. +31]; w = d sc_j q - dmin m_j.
template <>
__device__ __forceinline__ void decode_unit<MOE_Q4_K>(const uint8_t *row, int u, Unit &U) {
    const int sb = u >> 3, j = u & 7;
    const uint8_t *b = row + 144 * sb;
    const uint32_t dd = *reinterpret_cast<const uint32_t *>(b);
    const float d = half_bits_to_f32(dd & 0xffff), dmin = half_bits_to_f32(dd >> 16);
    const uint8_t *s = b + 4;
    int sc, mn;
    if (j < 4) {
        sc = s[j] & 63;
        mn = s[j + 4] & 63;
    } else {
        sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
    const uint4 *qs = reinterpret_cast<const uint4 *>(b + 16 + 32 * (j >> 1));
    const int sh = (j & 1) * 4;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        uint4 q = qs[v];
        uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int by = 0; by < 4; ++by) U.c[16 * v + 4 * a + by] = (float)((w[a] >> (8 * by + sh)) & 15u);
    }
    U.s_lo = U.s_hi = d * (float)sc;
    U.m = dmin * (float)mn;
}

// Q6_K: 210 B per 256 = ql[128] | qh[64] | int8 scale[16] | fp16 d. Unit
// u % 8 = 4h + r covers weights 128h + 32r .. +31: low nibble of
// ql[64h (+32 if r odd) + i] for r < 2, high nibble for r >= 2, plus bits
// 2r, 2r+1 of qh[32h + i] as bits 4-5; scales 8h + 2r (i < 16) and 8h + 2r + 1.
template <>
__device__ __forceinline__ void decode_unit<MOE_Q6_K>(const uint8_t *row, int u, Unit &U) {
    const int sb = u >> 3, uu = u & 7, h = uu >> 2, r = uu & 3;
    const uint8_t *b = row + 210 * sb;
    const uint8_t *ql = b + 64 * h + ((r & 1) ? 32 : 0);
    const uint8_t *qh = b + 128 + 32 * h;
    const int lsh = (r >= 2) ? 4 : 0, hsh = 2 * r;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint16_t l2 = ld16(ql + 2 * i), h2 = ld16(qh + 2 * i);
        int q0 = ((l2 >> lsh) & 15) | (((h2 >> hsh) & 3) << 4);
        int q1 = ((l2 >> (8 + lsh)) & 15) | (((h2 >> (8 + hsh)) & 3) << 4);
        U.c[2 * i] = (float)(q0 - 32);
        U.c[2 * i + 1] = (float)(q1 - 32);
    }
    const float d = half_bits_to_f32(ld16(b + 208));
    const int8_t *sc = reinterpret_cast<const int8_t *>(b + 192 + 8 * h + 2 * r);
    U.s_lo = d * (float)sc[0];
    U.s_hi = d * (float)sc[1];
    U.m = 0.0f;
}

// MXFP4: 17 B = E8M0 e | 16 B codes; weight i < 16 low nibble of byte 1 + i,
// 16 + i high nibble. Codes are taken as twice the E2M1 value (integers) and
// the scale as 2^(e - 128).
__device__ __forceinline__ float e2m1_x2(uint32_t c) {
    const float mag = (float)((0xC8643210u >> (4 * (c & 7))) & 15u);  // 0 1 2 3 4 6 8 12
    return (c & 8) ? -mag : mag;
}

template <>
__device__ __forceinline__ void decode_unit<MOE_MXFP4>(const uint8_t *row, int u, Unit &U) {
    const uint8_t *b = row + 17 * u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t q = b[1 + i];
        U.c[i] = e2m1_x2(q & 15);
        U.c[16 + i] = e2m1_x2(q >> 4);
    }
    U.s_lo = U.s_hi = e8m0_half_scale(b[0]);
    U.m = 0.0f;
}

// The non-linear codebook of IQ4_NL / IQ4_XS: value of code 0..15 as a signed
// byte, four codes per word (code 4w + i in byte i of word w):
//   -127 -104 -83 -65 | -49 -35 -22 -10 | 1 13 25 38 | 53 69 89 113.
__device__ __forceinline__ int iq4_value(uint32_t c) {
    const uint32_t w0 = (c & 8) ? 0x26190D01u : 0xBFAD9881u;
    const uint32_t w1 = (c & 8) ? 0x71594535u : 0xF6EADDCFu;
    uint32_t b;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b) : "r"(w0), "r"(w1), "r"(c & 7u));
    return (int)(int8_t)(b & 0xffu);
}

// IQ4_NL: 18 B = fp16 d | 16 B codes; weight i < 16 low nibble of byte 2 + i,
// 16 + i its high nibble; w = d * codebook[code].
template <>
__device__ __forceinline__ void decode_unit<MOE_IQ4_NL>(const uint8_t *row, int u, Unit &U) {
    const uint8_t *b = row + 18 * u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t q = b[2 + i];
        U.c[i] = (float)iq4_value(q & 15);
        U.c[16 + i] = (float)iq4_value(q >> 4);
    }
    U.s_lo = U.s_hi = half_bits_to_f32(ld16(b));
    U.m = 0.0f;
}

// IQ4_XS: 136 B per 256 = fp16 d | uint16 high scale bits | 4 B low scale
// nibbles | 128 B codes. Unit u is sub-block j = u % 8: scale
// d * (ls_j - 32), ls_j = nibble (j % 2) of byte 4 + j / 2 | bits 2j.. of the
// uint16 << 4; codes 16 j .. +15 low nibbles then high nibbles.
template <>
__device__ __forceinline__ void decode_unit<MOE_IQ4_XS>(const uint8_t *row, int u, Unit &U) {
    const int sb = u >> 3, j = u & 7;
    const uint8_t *b = row + 136 * sb;
    const uint32_t sh = ld16(b + 2);
    const int ls = ((b[4 + (j >> 1)] >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4);
    const uint8_t *qs = b + 8 + 16 * j;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t q = qs[i];
        U.c[i] = (float)iq4_value(q & 15);
        U.c[16 + i] = (float)iq4_value(q >> 4);
    }
    U.s_lo = U.s_hi = half_bits_to_f32(ld16(b)) * (float)(ls - 32);
    U.m = 0.0f;
}

// IQ3_XXS: 98 B per 256 = fp16 d | 64 grid-index bytes | 8 words. Unit u is
// sub-block j = u % 8, word a = word j: scale d * (0.5 + (a >> 28)) / 2;
// group l (weights 8l .. 8l+7) takes magnitudes from grid[q[8j + 2l]] (4) and
// grid[q[8j + 2l + 1]] (4), signs from the 7-bit index (a >> 7l) & 127 plus
// the parity bit for the eighth.
__device__ __forceinline__ void decode_iq3_unit(const uint8_t *row, int u, const uint32_t *grid, Unit &U) {
    const int sb = u >> 3, j = u & 7;
    const uint8_t *b = row + 98 * sb;
    const uint32_t a = (uint32_t)ld16(b + 66 + 4 * j) | ((uint32_t)ld16(b + 68 + 4 * j) << 16);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
        const uint32_t s7 = (a >> (7 * l)) & 127u;
        const uint32_t signs = s7 | ((__popc(s7) & 1u) << 7);
        const uint32_t g0 = __ldg(grid + b[2 + 8 * j + 2 * l]), g1 = __ldg(grid + b[3 + 8 * j + 2 * l]);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float mag = (float)(((t < 4 ? g0 : g1) >> (8 * (t & 3))) & 255u);
            U.c[8 * l + t] = ((signs >> t) & 1u) ? -mag : mag;
        }
    }
    U.s_lo = U.s_hi = half_bits_to_f32(ld16(b)) * (0.5f + (float)(a >> 28)) * 0.5f;
    U.m = 0.0f;
}

// T5_G128: 28 B per 128 = fp16 s | 26 code bytes; weight 5c + i is base-3
// digit i (least significant first) of code byte c; w = s * (digit - 1). Unit
// u is quarter j = u % 4 of block u / 4: weights 32j .. 32j + 31, which start
// at digit (32j) % 5 of code byte (32j) / 5 and span at most 8 code bytes.
// floor(v / 3) = (v * 171) >> 9 for every byte value v.
template <>
__device__ __forceinline__ void decode_unit<MOE_T5_G128>(const uint8_t *row, int u, Unit &U) {
    const uint8_t *b = row + 28 * (u >> 2);
    const int j = u & 3, first = (32 * j) / 5, off = (32 * j) % 5;   // {0, 6, 12, 19}, {0, 2, 4, 1}
    int dig[40];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        int v = b[2 + min(first + c, 25)];   // the clamped bytes are never selected below
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const int q = (v * 171) >> 9;
            dig[5 * c + i] = v - 3 * q;
            v = q;
        }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int d = off == 0 ? dig[i] : off == 1 ? dig[i + 1] : off == 2 ? dig[i + 2] : dig[i + 4];
        U.c[i] = (float)(d - 1);
    }
    U.s_lo = U.s_hi = half_bits_to_f32(ld16(b));
    U.m = 0.0f;
}

// acc += dot(w, x) for one 32-weight unit; x in shared memory (fp32).
__device__ __forceinline__ float unit_dot(const Unit &U, const float *x) {
    float lo = 0.0f, hi = 0.0f, sx = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) lo = fmaf(U.c[i], x[i], lo);
#pragma unroll
    for (int i = 16; i < 32; ++i) hi = fmaf(U.c[i], x[i], hi);
    if (U.m != 0.0f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) sx += x[i];
    }
    return U.s_lo * lo + U.s_hi * hi - U.m * sx;
}

// Row-dot of GV_SLICES threads: thread `slice` takes units slice, slice + 8, ...
template <int FMT>
__device__ __forceinline__ void row_dot(const uint8_t *row, int units, int slice, const float *xs, int xstride,
                                        int nt, float acc[GV_NT], const uint32_t *grid) {
#pragma unroll
    for (int t = 0; t < GV_NT; ++t) acc[t] = 0.0f;
    for (int u = slice; u < units; u += GV_SLICES) {
        Unit U;
        if constexpr (FMT == MOE_IQ3_XXS)
            decode_iq3_unit(row, u, grid, U);
        else
            decode_unit<FMT>(row, u, U);
#pragma unroll
        for (int t = 0; t < GV_NT; ++t)
            if (t < nt) acc[t] += unit_dot(U, xs + t * xstride + 32 * u);
    }
#pragma unroll
    for (int t = 0; t < GV_NT; ++t) {
        acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 1);
        acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 2);
        acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 4);
    }
}

// All threads wait (bounded) for the tile's bulk copies; the outcome is made
// uniform across the CTA. On a timeout the tile is skipped, the flag is set and
// thread 0 waits once more (bounded) so no copy is left landing in a CTA that
// has exited.
__device__ __forceinline__ bool tile_ready(uint64_t *bar, uint32_t *status) {
    const bool ok = mbar_wait_timed(bar, 0);
    if (__syncthreads_and(ok)) return true;
    if (threadIdx.x == 0) {
        atomicOr(status, (uint32_t)MOE_FLAG_WAIT_TIMEOUT);
        mbar_wait(bar, 0);
    }
    return false;
}

struct GvArgs {
    const DevExpert *table;
    int H, I, k;
    const int32_t *offsets, *pairs, *active;
    const uint16_t *x;   // bf16 [T, H]
    float *h;            // fp32 [pairs, I] in bucket order
    float *y;            // fp32 [pairs, H] in bucket order
    uint32_t *status;
    int64_t wstride;     // smem bytes reserved per weight row (max stride)
    const uint32_t *grid;   // IQ3_XXS grid (256 words) or null
};

template <int FMT>
__device__ void gateup_tile(const GvArgs &A, const DevMatrix &G, const DevMatrix &Uw, int e, int r0, int nrows,
                            unsigned char *smem, uint64_t *bar) {
    const int tid = threadIdx.x;
    uint8_t *wg = smem;
    uint8_t *wu = smem + GU_ROWS * A.wstride;
    float *xs = reinterpret_cast<float *>(smem + 2 * GU_ROWS * A.wstride);
    float *gu = xs + GV_NT * A.H;  // [2][GU_ROWS][GV_NT]

    if (tid == 0) {
        const uint32_t bytes_g = (uint32_t)(nrows * G.stride), bytes_u = (uint32_t)(nrows * Uw.stride);
        mbar_expect_tx(bar, bytes_g + bytes_u);
        bulk_g2s(wg, G.data + (size_t)r0 * G.stride, bytes_g, bar);
        bulk_g2s(wu, Uw.data + (size_t)r0 * Uw.stride, bytes_u, bar);
    }
    const int q0 = A.offsets[e], n = A.offsets[e + 1] - q0;
    const int rd = tid / GV_SLICES, slice = tid % GV_SLICES;
    const int mat = rd / GU_ROWS, row = rd % GU_ROWS;
    const int units = A.H / 32;
    bool waited = false;

    for (int t0 = 0; t0 < n; t0 += GV_NT) {
        const int nt = min(GV_NT, n - t0);
        for (int i = tid; i < nt * A.H; i += GV_THREADS) {
            int t = i / A.H, c = i - t * A.H;
            int tok = A.pairs[q0 + t0 + t] / A.k;
            xs[t * A.H + c] = bf16_to_f32(A.x[(size_t)tok * A.H + c]);
        }
        if (!waited) {
            if (!tile_ready(bar, A.status)) return;
            waited = true;
        }
        __syncthreads();
        float acc[GV_NT];
        {
            // every lane takes part in the shuffles; rows past the tile's end
            // recompute the last row and discard it
            const int rr = row < nrows ? row : nrows - 1;
            const uint8_t *rp = (mat ? wu + rr * Uw.stride : wg + rr * G.stride);
            row_dot<FMT>(rp, units, slice, xs, A.H, nt, acc, A.grid);
            if (slice == 0 && row < nrows)
#pragma unroll
                for (int t = 0; t < GV_NT; ++t) gu[(mat * GU_ROWS + row) * GV_NT + t] = acc[t];
        }
        __syncthreads();
        for (int i = tid; i < nrows * nt; i += GV_THREADS) {
            int r = i / nt, t = i - r * nt;
            float g = gu[r * GV_NT + t], u = gu[(GU_ROWS + r) * GV_NT + t];
            A.h[(size_t)(q0 + t0 + t) * A.I + r0 + r] = silu_f32(g) * u;
        }
        __syncthreads();
    }
    if (!waited) tile_ready(bar, A.status);
}

__global__ void __launch_bounds__(GV_THREADS) gateup_gemv_kernel(GvArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    const int a = blockIdx.y;
    if (a >= A.active[0]) return;
    const int e = A.active[1 + a];
    const int r0 = blockIdx.x * GU_ROWS;
    if (r0 >= A.I) return;
    const int nrows = min(GU_ROWS, A.I - r0);
    const DevMatrix G = A.table[e].gate, Uw = A.table[e].up;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    switch (G.fmt) {
        case MOE_Q8_0: gateup_tile<MOE_Q8_0>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_Q4_K: gateup_tile<MOE_Q4_K>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_Q6_K: gateup_tile<MOE_Q6_K>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_MXFP4: gateup_tile<MOE_MXFP4>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_IQ4_NL: gateup_tile<MOE_IQ4_NL>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_IQ4_XS: gateup_tile<MOE_IQ4_XS>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_IQ3_XXS: gateup_tile<MOE_IQ3_XXS>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        case MOE_T5_G128: gateup_tile<MOE_T5_G128>(A, G, Uw, e, r0, nrows, smem, &bar); break;
        default: break;
    }
}

template <int FMT>
__device__ void down_tile(const GvArgs &A, const DevMatrix &D, int e, int r0, int nrows, unsigned char *smem,
                          uint64_t *bar) {
    const int tid = threadIdx.x;
    uint8_t *wd = smem;
    float *hs = reinterpret_cast<float *>(smem + DN_ROWS * A.wstride);
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)(nrows * D.stride);
        mbar_expect_tx(bar, bytes);
        bulk_g2s(wd, D.data + (size_t)r0 * D.stride, bytes, bar);
    }
    const int q0 = A.offsets[e], n = A.offsets[e + 1] - q0;
    const int row = tid / GV_SLICES, slice = tid % GV_SLICES;
    const int units = A.I / 32;
    bool waited = false;
    for (int t0 = 0; t0 < n; t0 += GV_NT) {
        const int nt = min(GV_NT, n - t0);
        for (int i = tid; i < nt * A.I; i += GV_THREADS) hs[i] = A.h[(size_t)(q0 + t0) * A.I + i];
        if (!waited) {
            if (!tile_ready(bar, A.status)) return;
            waited = true;
        }
        __syncthreads();
        float acc[GV_NT];
        {
            const int rr = row < nrows ? row : nrows - 1;
            row_dot<FMT>(wd + rr * D.stride, units, slice, hs, A.I, nt, acc, A.grid);
            if (slice == 0 && row < nrows)
                for (int t = 0; t < nt; ++t) A.y[(size_t)(q0 + t0 + t) * A.H + r0 + row] = acc[t];
        }
        __syncthreads();
    }
    if (!waited) tile_ready(bar, A.status);
}

__global__ void __launch_bounds__(GV_THREADS) down_gemv_kernel(GvArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    const int a = blockIdx.y;
    if (a >= A.active[0]) return;
    const int e = A.active[1 + a];
    const int r0 = blockIdx.x * DN_ROWS;
    if (r0 >= A.H) return;
    const int nrows = min(DN_ROWS, A.H - r0);
    const DevMatrix D = A.table[e].down;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    switch (D.fmt) {
        case MOE_Q8_0: down_tile<MOE_Q8_0>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_Q4_K: down_tile<MOE_Q4_K>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_Q6_K: down_tile<MOE_Q6_K>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_MXFP4: down_tile<MOE_MXFP4>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_IQ4_NL: down_tile<MOE_IQ4_NL>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_IQ4_XS: down_tile<MOE_IQ4_XS>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_IQ3_XXS: down_tile<MOE_IQ3_XXS>(A, D, e, r0, nrows, smem, &bar); break;
        case MOE_T5_G128: down_tile<MOE_T5_G128>(A, D, e, r0, nrows, smem, &bar); break;
        default: break;
    }
}

// out[t] = sum_j w[t, j] * y[pos[t, j]] in ascending j (0 if no pair is kept).
// With SCALED, row q of y is multiplied first by yscale[q], a power of two,
// which is exact: the tensor path leaves that scale to this kernel.
template <bool SCALED>
__global__ void combine_kernel(int T, int k, int H, const int32_t *__restrict__ pos, const float *__restrict__ wts,
                               const float *__restrict__ y, const float *__restrict__ yscale, float *__restrict__ out) {
    pdl_trigger();
    pdl_wait();   // y comes from the down kernel
    const int t = blockIdx.y;
    const int i4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (i4 * 4 >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        int q = pos[t * k + j];
        if (q < 0) continue;
        float w = wts[t * k + j];
        float4 v = reinterpret_cast<const float4 *>(y + (size_t)q * H)[i4];
        if (SCALED) {
            const float sq = yscale[q];
            v.x *= sq;
            v.y *= sq;
            v.z *= sq;
            v.w *= sq;
        }
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    reinterpret_cast<float4 *>(out + (size_t)t * H)[i4] = acc;
}

}  // namespace

// Records a profiling event; inside a stream capture it becomes an external
// event-record node of the graph.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(s, &cs);
    if (err != cudaSuccess) return err;
    return cudaEventRecordWithFlags(ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0);
}

// Lets `fn` use all of the opt-in shared memory that its static shared
// memory leaves free.
cudaError_t allow_max_dynamic_smem(const void *fn) {
    int dev = 0, optin = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (err == cudaSuccess) err = cudaFuncGetAttributes(&fa, fn);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    return err;
}

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

cudaError_t launch_combine(int T, int k, int H, const int32_t *pos, const float *wts, const float *y, float *out,
                           cudaStream_t s, const float *yscale) {
    if (T <= 0) return cudaSuccess;
    dim3 g((H / 4 + 127) / 128, T);
    if (yscale) return launch_pdl(combine_kernel<true>, g, dim3(128), 0, s, T, k, H, pos, wts, y, yscale, out);
    return launch_pdl(combine_kernel<false>, g, dim3(128), 0, s, T, k, H, pos, wts, y, (const float *)nullptr, out);
}

size_t gateup_smem_bytes(int H, int64_t wstride) {
    return (size_t)(2 * GU_ROWS * wstride) + (size_t)GV_NT * H * 4 + 2 * GU_ROWS * GV_NT * 4;
}
size_t down_smem_bytes(int I, int64_t wstride) { return (size_t)(DN_ROWS * wstride) + (size_t)GV_NT * I * 4; }

cudaError_t launch_gemv_path(const DevExpert *table, int T, int k, int E, int H, int I, int64_t gu_stride,
                             int64_t dn_stride, uint32_t gu_formats, uint32_t down_formats, const uint32_t *grid,
                             const int32_t *offsets, const int32_t *pairs, const int32_t *active, const int32_t *pos,
                             const float *wts, const uint16_t *x, float *h, float *y, float *out, uint32_t *status,
                             cudaEvent_t const *events, cudaStream_t s) {
    // decode batches of up to 16 rows (32 with Q8_0 / Q4_K gate/up): the streaming kernels (stream.cu)
    if (T > 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const SgPlan p = stream_plan(T, k, E, H, I, gu_formats, down_formats, gu_stride, dn_stride);
        if (p.ok) {
            cudaError_t err =
                launch_stream_path(table, p, T, k, E, H, I, offsets, pairs, active, x, h, y, status, grid, events, s);
            if (err != cudaSuccess) return err;
            return launch_combine(T, k, H, pos, wts, y, out, s);
        }
    }
    static bool attr_done[64] = {};
    int dev = current_device();
    if (dev >= 64 || !attr_done[dev]) {
        cudaError_t err = allow_max_dynamic_smem(reinterpret_cast<const void *>(gateup_gemv_kernel));
        if (err == cudaSuccess) err = allow_max_dynamic_smem(reinterpret_cast<const void *>(down_gemv_kernel));
        if (err != cudaSuccess) return err;
        if (dev < 64) attr_done[dev] = true;
    }
    const int max_active = T * k < E ? T * k : E;
    if (T > 0 && max_active > 0) {
        GvArgs A{table, H, I, k, offsets, pairs, active, x, h, y, status, gu_stride, grid};
        cudaError_t err;
        if (events && (err = record_event(events[0], s)) != cudaSuccess) return err;
        dim3 g1((I + GU_ROWS - 1) / GU_ROWS, max_active);
        gateup_gemv_kernel<<<g1, GV_THREADS, gateup_smem_bytes(H, gu_stride), s>>>(A);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        if (events && (err = record_event(events[1], s)) != cudaSuccess) return err;
        A.wstride = dn_stride;
        dim3 g2((H + DN_ROWS - 1) / DN_ROWS, max_active);
        down_gemv_kernel<<<g2, GV_THREADS, down_smem_bytes(I, dn_stride), s>>>(A);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        if (events && (err = record_event(events[2], s)) != cudaSuccess) return err;
    }
    if (T > 0) {
        dim3 g3((H / 4 + 127) / 128, T);
        combine_kernel<false><<<g3, 128, 0, s>>>(T, k, H, pos, wts, y, nullptr, out);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

// This file's copy of the wait bound (moe_set_wait_timeout_ns).
cudaError_t set_wait_ns_gemv(unsigned long long ns) { return set_tu_wait_ns(ns); }

}  // namespace moe
