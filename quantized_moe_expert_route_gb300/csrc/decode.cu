// Fused decode path: the whole routed-expert FFN of a few token rows in one
// persistent, cooperative kernel (one CTA per SM).
//
// The pages' decode kernels are prior art here: the grouped multi-session
// decode of "多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出 120 t/s" (section
// 120 t/s 的秘密: one launch serves the decode rows of all sessions over a
// Q4_K routed-expert layout), the gate/up + activation fusion of "三张 RTX 3090
// 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南" (section 关键 Bug 修复与调试
// 踩坑记录, item 4) and the single-token GEMV of "一张 RTX 3090 跑 Llama 70B" (section
// 4.4). On GB300 a decode layer is a few microseconds of HBM streaming and
// every dependent global-memory round trip costs about a microsecond, so the
// design removes kernel boundaries and round trips:
//
//   1. Every CTA computes the softmax top-k and the per-expert bucketing of
//      the token rows itself: each warp sorts a 32-logit slice (bitonic, in
//      registers), then candidates are ranked by counting. The routed
//      experts' descriptors are requested right after selection.
//   2. The routed experts' gate/up rows are split evenly across the CTAs.
//      Lane s of warp 0 streams the CTA's gate/up rows, then its down rows,
//      through ring slot s of 16 shared-memory stages of up to 12 KB with TMA
//      bulk copies: the first fill as soon as the chunk table exists (for one
//      token nearly the whole share is then in flight), each refill when the
//      16 warps have finished a round of chunks. The warps decode the stages
//      and write h = silu(W_gate x) * (W_up x) (fp32) to global memory.
//   3. A bounded grid barrier (cooperative launch: all CTAs co-resident)
//      separates gate/up from down; then each CTA reads every pair's h.
//   4. Each CTA owns a slice of output rows for every routed expert, so the
//      router-weighted combine runs in-CTA in ascending slot order.
//
// Arithmetic: activations become int16 with a per-row power-of-two scale (x)
// or a per-32-block one (h); the quantised codes enter dp2a (int16 x int8 ->
// int32) undecoded (Q8_0) or unpacked to bytes (Q4_K), so each block's sum is
// an exact integer, scaled once per block in fp32. The Q4_K minimum term uses
// the exact per-sub-block activation sums. This path handles Q4_K gate/up with
// Q8_0 down; other layers take the tensor-core or grouped GEMV path.
#include <algorithm>
#include <type_traits>

#include "moe_internal.cuh"
#include "dot16.cuh"

namespace moe {

namespace {

constexpr int DC_CW = 16;                        // warps (all consume; warp 0 also issues the copies)
constexpr int DC_WARPS = DC_CW;
constexpr int DC_THREADS = DC_WARPS * 32;        // 4 warps per SM sub-partition: up to 128 registers
constexpr int DC_STAGE_MAX = 12 * 1024;          // ring stage bytes (smaller when shared memory is tight)
constexpr int DC_NSTAGE = 16;                    // ring slots; slot s is served by lane s of warp 0
constexpr int DC_MAX_PAIRS = 64;                 // T * k
constexpr int DC_ROWS_A = 4;                     // max gate/up row pairs per chunk
constexpr int DC_SURV = 64;                      // top-k survivors ranked from the short list

constexpr int DC_HQW = 20;                       // words per staged h block: 16 int16 pairs, the scale, pad

struct DcLayout {
    size_t ring, xs, xsum, xsc, xmax, hq, ybuf, rowk, smax, surv, scnt, tau, ss, selk, ids, wts, keep, act, aoff,
        plist,
        dpair, chunks, full, misc, total;
    int rb, ns;
};

__host__ __device__ inline DcLayout dc_layout(int T, int k, int E, int H, int I, int G, int stage, int chunk_cap) {
    DcLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t r = o;
        o = align_up(o + bytes, 128);
        return r;
    };
    const int P = T * k;
    L.rb = (H + G - 1) / G;
    L.ns = (E + 31) / 32;
    L.ring = take((size_t)DC_NSTAGE * stage);
    L.xs = take((size_t)T * H * 2);
    L.xsum = take((size_t)T * (H / 64) * 2 * 4);
    L.xsc = take((size_t)T * 4);
    L.xmax = take((size_t)T * 4);
    // h of every pair, staged after gate/up as int16 with one power-of-two
    // scale per 32-column block; the down outputs per K part (8 blocks)
    L.hq = take((size_t)P * (I / 32) * DC_HQW * 4);
    L.ybuf = take((size_t)((I / 32 + 7) / 8) * P * L.rb * 4);
    L.rowk = take((size_t)T * L.ns * 32 * 4);
    L.smax = take((size_t)T * L.ns * 8);
    L.surv = take((size_t)T * DC_SURV * 8);
    L.scnt = take((size_t)T * 4);
    L.tau = take((size_t)T * 8);
    L.ss = take((size_t)T * L.ns * 4);
    L.selk = take((size_t)P * 4);
    L.ids = take((size_t)P * 4);
    L.wts = take((size_t)P * 4);
    L.keep = take((size_t)P);
    L.act = take((size_t)P * 4);
    L.aoff = take((size_t)(P + 1) * 4);
    L.plist = take((size_t)P * 4);
    L.dpair = take((size_t)P * sizeof(DevExpert));
    L.chunks = take((size_t)chunk_cap * 16);
    L.full = take((size_t)DC_NSTAGE * 8);
    L.misc = take(128);
    L.total = o;
    return L;
}

struct DcArgs {
    const DevExpert *table;
    int E, H, I, T, k, renorm, lo, hi;
    uint32_t fmt_mask;
    const float *logits;
    const uint16_t *x;
    float *out;
    float *h;                       // [T*k][I] fp32, pair p = t*k + j
    int32_t *ids_out, *offsets_out, *active_out, *pairs_out, *pos_out;
    float *wts_out;
    unsigned char *sync;            // workspace state: the launch counter at offset 8
    uint32_t *status;
    int stage;                      // bytes per ring slot
    int rows_a, rows_b;             // gate/up row pairs per chunk, down rows per chunk
    int chunk_cap;                  // capacity of the shared-memory chunk table
    int uniform;                    // experts at a constant step: descriptor = u + e * ustep
    DevExpert u;
    long long ustep[3];
};

// Named barriers are written as inline PTX. bar.sync is .aligned (all
// threads of a warp execute it together), and nothing makes the compiler
// reconverge a warp before inline assembly, so a warp whose lanes may have
// diverged (one lane polling, a few lanes issuing copies) is reconverged
// with __syncwarp() first.
__device__ __forceinline__ void consumer_sync() {
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(DC_CW * 32) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Ascending bitonic sort of one int key per lane within each group of W lanes.
template <int W>
__device__ __forceinline__ int warp_sort_asc(int key) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= W; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int other = __shfl_xor_sync(0xffffffffu, key, stride);
            const bool asc = (lane & size) == 0 || size == W;
            const bool lower = (lane & stride) == 0;
            key = (lower == asc) ? min(key, other) : max(key, other);
        }
    }
    return key;
}

// cp.async of 8 bytes global -> shared (L1-allocating); completion via cp_async_wait_all.
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}




// One lane's down-projection partial over up to 8 consecutive Q8_0 blocks
// (one 272-byte period of a row: 8 x 34 bytes = 17 x 16 bytes, so that it
// starts and ends 16-byte aligned) against staged int16 h. Block b's scale is
// half-word 17 b of the period and its code pairs are half-words 17 b + 1 ...
// 17 b + 16: the codes enter dp2a undecoded, taking the low or high half of
// each word as the half-word's parity says (all offsets are compile-time
// constants). hb: DC_HQW words per block, 16 int16 pairs then the fp32
// scale 2^-sigma. Returns sum_b d_b * 2^-sigma_b * sum_i q_bi h_bi.
__device__ __forceinline__ uint32_t u4_word(const uint4 &v, int c) {
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}
__device__ __forceinline__ float q8_0_period_dot(const uint8_t *wrow, const uint32_t *hb, int nb) {
    const uint4 *src = reinterpret_cast<const uint4 *>(wrow);
    uint4 Q[17];
    float acc = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        if (b >= nb) break;
        const int khi = ((17 * b + 16) >> 1) >> 2;
        const int kfirst = b == 0 ? 0 : (((17 * (b - 1) + 16) >> 1) >> 2) + 1;
#pragma unroll
        for (int kk = kfirst; kk <= khi; ++kk) Q[kk] = src[kk];
        const uint4 *h4 = reinterpret_cast<const uint4 *>(hb + b * DC_HQW);
        uint32_t hv[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 q = h4[v];
            hv[4 * v] = q.x;
            hv[4 * v + 1] = q.y;
            hv[4 * v + 2] = q.z;
            hv[4 * v + 3] = q.w;
        }
        const float hinv = __uint_as_float(hb[b * DC_HQW + 16]);
        const int wd = (17 * b) >> 1;
        const uint32_t dw = u4_word(Q[wd >> 2], wd & 3);
        const float d = half_bits_to_f32((uint16_t)((b & 1) ? (dw >> 16) : (dw & 0xffffu)));
        int s0 = 0, s1 = 0;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int hw = 17 * b + 1 + m, w = hw >> 1;
            const uint32_t word = u4_word(Q[w >> 2], w & 3);
            int &sm = (m & 1) ? s1 : s0;
            sm = (hw & 1) ? dp2a_hi(hv[m], word, sm) : dp2a_lo(hv[m], word, sm);
        }
        acc = fmaf((float)(s0 + s1), d * hinv, acc);
    }
    return acc;
}

// Before an aborting CTA exits (after a CTA barrier, so no copy is issued
// any more): wait (bounded) for the bulk copy last issued into each ring
// slot, so that none still writes its shared memory.
__device__ __forceinline__ void drain_copies(uint64_t *full, int *misc) {
    if (threadIdx.x != 0) return;
    for (int s = 0; s < DC_NSTAGE; ++s) {
        const int ci = *reinterpret_cast<volatile int *>(&misc[16 + s]);
        if (ci >= 0) mbar_wait(&full[s], (uint32_t)(ci / DC_NSTAGE) & 1u);
    }
}

__device__ __forceinline__ void set_abort(int *misc, uint32_t *status) {
    atomicOr(status, (uint32_t)MOE_FLAG_WAIT_TIMEOUT);
    *reinterpret_cast<volatile int *>(&misc[1]) = 1;
}

// ---------------------------------------------------------------- once-per-launch steps
// (out of line: one copy each keeps the kernel's code small)

__device__ __noinline__ int dc_bucket_sorted(int P, const uint8_t *keep, const int *ids, int *plist, int *act,
                                             int *aoff, int *misc) {
    const int lane = threadIdx.x & 31;
    constexpr int SENT = 0x7fffffff;
    int key[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int p = lane + 32 * r;
        key[r] = (p < P && keep[p]) ? ((ids[p] << 8) | p) : SENT;
    }
    if (P <= 16) {
        key[0] = warp_sort_asc<16>(key[0]);
        if (lane >= 16) key[0] = SENT;
    } else if (P <= 32) {
        key[0] = warp_sort_asc<32>(key[0]);
    } else {
#pragma unroll 1
        for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll 1
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                if (stride == 32) {
                    const int lo = min(key[0], key[1]), hi = max(key[0], key[1]);   // size == 64: ascending
                    key[0] = lo;
                    key[1] = hi;
                } else {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int i = lane + 32 * r;
                        const int other = __shfl_xor_sync(0xffffffffu, key[r], stride);
                        const bool asc = (i & size) == 0;
                        const bool lower = (lane & stride) == 0;
                        key[r] = (lower == asc) ? min(key[r], other) : max(key[r], other);
                    }
                }
            }
        }
    }
    // element i = lane + 32 r holds key[r]; starts of expert runs
    const int prev0 = __shfl_up_sync(0xffffffffu, key[0], 1);
    const int prev1 = __shfl_up_sync(0xffffffffu, key[1], 1);
    const int last0 = __shfl_sync(0xffffffffu, key[0], 31);
    const int pk[2] = {lane == 0 ? -1 : prev0, lane == 0 ? last0 : prev1};
    bool start[2], valid[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        valid[r] = key[r] != SENT;
        start[r] = valid[r] && (pk[r] < 0 || (pk[r] >> 8) != (key[r] >> 8));
    }
    const unsigned s0 = __ballot_sync(0xffffffffu, start[0]), s1 = __ballot_sync(0xffffffffu, start[1]);
    const unsigned v0 = __ballot_sync(0xffffffffu, valid[0]), v1 = __ballot_sync(0xffffffffu, valid[1]);
    const int n_kept = __popc(v0) + __popc(v1), n_act = __popc(s0) + __popc(s1);
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = lane + 32 * r;
        if (valid[r]) plist[i] = key[r] & 0xff;
        if (start[r]) {
            const int a = r == 0 ? __popc(s0 & below) : __popc(s0) + __popc(s1 & below);
            act[a] = key[r] >> 8;
            aoff[a] = i;
        }
    }
    if (lane == 0) {
        aoff[n_act] = n_kept;
        misc[0] = n_act;
        misc[6] = n_kept;
    }

    return n_act;
}

__device__ __noinline__ void dc_route_weights(int t, int k, int NS, int renorm, const float *selk, const float2 *smax,
                                              const float *sls, float *wts) {
    const int lane = threadIdx.x & 31;
    const float m = selk[t * k];                     // the row's largest logit (or -inf)
    const bool any_finite = m > -INFINITY;
    const float kj = lane < k ? selk[t * k + lane] : -INFINITY;
    const float ex = (lane < k && any_finite && kj > -INFINITY) ? expf(kj - m) : 0.0f;
    float denom;
    if (renorm) {
        denom = warp_sum(ex);
    } else {
        float s = 0.0f;
        for (int w = lane; w < NS; w += 32) {
            const float mw = smax[t * NS + w].x;
            if (any_finite && mw > -INFINITY) s += sls[t * NS + w] * expf(mw - m);
        }
        denom = warp_sum(s);
    }
    if (lane < k) {
        const int p = t * k + lane;
        wts[p] = denom > 0.0f ? ex / denom : 0.0f;
    }
}

__device__ __noinline__ void dc_build_chunks(int n_act, int I, int H, int c, int G, int rows_a, int rows_b,
                                             int chunk_cap, int4 *chunk, int *misc) {
    const int lane = threadIdx.x & 31;
    // the chunk table: gate/up chunks of at most rows_a row pairs, never
    // crossing an expert, over this CTA's share [a_begin, a_end) of the
    // (active expert, row) space; then, per active expert, the CTA's down
    // rows in chunks of rows_b. Lane j first sizes the j-th expert
    // segment of the share; then each lane fills chunk entries.
    const int NA = n_act * I;
    const int a_begin = (int)((unsigned)NA * c / G), a_end = (int)((unsigned)NA * (c + 1) / G);
    const int b0 = (int)((unsigned)H * c / G), b1 = (int)((unsigned)H * (c + 1) / G);
    const int nrows_b = b1 - b0;
    const int a_first = a_begin / I, a_last = a_end > a_begin ? (a_end - 1) / I : a_first - 1;
    int total = 0;
    for (int seg0 = a_first; seg0 <= a_last; seg0 += 32) {
        const int a = seg0 + lane;
        int len = 0, rs = 0;
        if (a <= a_last) {
            rs = max(a_begin, a * I);
            len = min(a_end, (a + 1) * I) - rs;
        }
        const int nch = (len + rows_a - 1) / rows_a;
        int inc = nch;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        const int first = total + inc - nch;          // this segment's first chunk
        const int nseg = min(32, a_last - seg0 + 1);
        const int segtot = __shfl_sync(0xffffffffu, inc, 31);
        for (int n0 = 0; n0 < segtot; n0 += 32) {
            const int n = total + n0 + lane;
            int j = 0;
            for (int q = 1; q < nseg; ++q)
                if (__shfl_sync(0xffffffffu, first, q) <= n) j = q;
            const int fj = __shfl_sync(0xffffffffu, first, j);
            const int rsj = __shfl_sync(0xffffffffu, rs, j), lenj = __shfl_sync(0xffffffffu, len, j);
            if (n0 + lane < segtot && n < chunk_cap) {
                const int aj = seg0 + j;
                const int r = rsj + (n - fj) * rows_a;
                chunk[n] = make_int4(aj, r - aj * I, min(rows_a, rsj + lenj - r), 0);
            }
        }
        total += segtot;
    }
    const int nb = (nrows_b + rows_b - 1) / rows_b;
    for (int i = lane; i < n_act * nb; i += 32) {
        const int a = i / nb, j = i - a * nb;
        if (total + i < chunk_cap) chunk[total + i] = make_int4(a, j * rows_b, min(rows_b, nrows_b - j * rows_b), 1);
    }
    if (lane == 0) {
        misc[4] = min(total, chunk_cap);
        misc[5] = min(total + n_act * nb, chunk_cap);
    }
}

__device__ __noinline__ void dc_issue_chunk(int ci, int nchunks_a, int b0, uint8_t *ring, int stage,
                                            const int4 *chunk, const DevExpert *dpair, const int *plist,
                                            const int *aoff, uint64_t *full, int *misc) {
    const int s = ci % DC_NSTAGE;
    uint8_t *dst = ring + (size_t)s * stage;
    const int4 ch = chunk[ci];
    const DevExpert &X = dpair[plist[aoff[ch.x]]];
    if (ci < nchunks_a) {
        const uint32_t bg = (uint32_t)(ch.z * X.gate.stride), bu = (uint32_t)(ch.z * X.up.stride);
        mbar_expect_tx(&full[s], bg + bu);
        bulk_g2s(dst, X.gate.data + (size_t)ch.y * X.gate.stride, bg, &full[s]);
        bulk_g2s(dst + bg, X.up.data + (size_t)ch.y * X.up.stride, bu, &full[s]);
    } else {
        const uint32_t bd = (uint32_t)(ch.z * X.down.stride);
        mbar_expect_tx(&full[s], bd);
        bulk_g2s(dst, X.down.data + (size_t)(b0 + ch.y) * X.down.stride, bd, &full[s]);
    }
    *reinterpret_cast<volatile int *>(&misc[16 + s]) = ci;
}

// ---------------------------------------------------------------- the kernel
// ONE: one token with H <= 2048 (the activations fit a lane's registers);
// compiled separately so that this kernel's code holds only its own path.
template <bool ONE>
__global__ void __launch_bounds__(DC_THREADS, 1) decode_fused_kernel(DcArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int G = gridDim.x, c = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = ONE ? 1 : A.T, k = A.k, E = A.E, H = A.H, I = A.I, P = T * k;
    const DcLayout L = dc_layout(T, k, E, H, I, G, A.stage, A.chunk_cap);
    const int NS = L.ns, NSE = 32 * L.ns, H64 = H / 64, U = I / 32;

    uint8_t *ring = smem + L.ring;
    // the raw activation rows occupy the ring's last slots during the prologue
    const int nraw = (T * H * 2 + A.stage - 1) / A.stage;
    uint8_t *xraw = ring + (size_t)DC_NSTAGE * A.stage - (size_t)T * H * 2;
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem + L.xs);     // per token: [8][H/64] uint4 (half2 words)
    float *xsum = reinterpret_cast<float *>(smem + L.xsum);       // [T][H/64][2]
    float *xsc = reinterpret_cast<float *>(smem + L.xsc);
    unsigned *xmax = reinterpret_cast<unsigned *>(smem + L.xmax);
    float *ybuf = reinterpret_cast<float *>(smem + L.ybuf);       // [K parts][P][rb] partial down outputs
    uint32_t *hq = reinterpret_cast<uint32_t *>(smem + L.hq);     // [P][I/32][DC_HQW] h as int16 + scale
    float *rowk = reinterpret_cast<float *>(smem + L.rowk);       // [T][NS*32] logits (-inf if not finite)
    float2 *smax = reinterpret_cast<float2 *>(smem + L.smax);     // [T][NS] slice best (key, index bits)
    float2 *surv = reinterpret_cast<float2 *>(smem + L.surv);     // [T][DC_SURV] survivors (key, index bits)
    int *scnt = reinterpret_cast<int *>(smem + L.scnt);           // [T] survivor counts
    float2 *tau = reinterpret_cast<float2 *>(smem + L.tau);       // [T] the k-th best slice best
    float *sls = reinterpret_cast<float *>(smem + L.ss);          // [T][NS] slice sum exp(l - max)
    float *selk = reinterpret_cast<float *>(smem + L.selk);       // [P] selected logits
    int *ids = reinterpret_cast<int *>(smem + L.ids);
    float *wts = reinterpret_cast<float *>(smem + L.wts);
    uint8_t *keep = smem + L.keep;
    int *act = reinterpret_cast<int *>(smem + L.act);             // active experts, ascending
    int *aoff = reinterpret_cast<int *>(smem + L.aoff);           // [n_act + 1] starts in plist
    int *plist = reinterpret_cast<int *>(smem + L.plist);         // kept pairs by (expert, pair)
    DevExpert *dpair = reinterpret_cast<DevExpert *>(smem + L.dpair);   // descriptor of each pair's expert
    int4 *chunk = reinterpret_cast<int4 *>(smem + L.chunks);   // (a, first row, rows): gate/up, then down
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    // [0] n_act [1] abort [2] flags [4] nchunks_a [5] nchunks [6] n_kept [7] chunks issued
    // before the ring's raw-activation slots are free [16 + s] the last chunk issued into
    // ring slot s (-1: none)
    int *misc = reinterpret_cast<int *>(smem + L.misc);
    unsigned long long *barrier_ctr = reinterpret_cast<unsigned long long *>(A.sync + 8);

    // The layer's inputs may come from the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (tid == 0) {
        for (int s = 0; s < DC_NSTAGE; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        for (int i = 0; i < 16; ++i) misc[i] = 0;
        for (int i = 16; i < 16 + DC_NSTAGE; ++i) misc[i] = -1;
    }
    for (int t = tid; t < T; t += DC_THREADS) {
        xmax[t] = 0u;
        scnt[t] = 0;
    }
    __syncthreads();
    // the grid barrier's count before this launch's arrivals: each CTA
    // arrives once, after its prologue, so fewer than G of this launch's
    // arrivals can precede this read (a launch starts after the previous one
    // completes) and count / G is the launch's generation. Loaded beside the
    // logit and activation loads, so that the latencies overlap.
    // Read (and later used) by the thread that arrives at the barrier only.
    unsigned long long gen_count = 0;
    if (tid == 32 * (DC_CW - 1)) gen_count = ld_relaxed_u64(barrier_ctr);

    // ---- 1. activation maxima (16-byte loads of 8 bf16; the raw rows are kept
    // in the ring's last slots, which are filled last) and, per warp,
    // the best logit of one 32-logit slice of one token row (under the
    // selection order: larger logit, then lower expert index). Each warp's
    // first logit load is issued before the activation loads so the two
    // latencies overlap.
    float lv0 = -INFINITY;
    if (warp < T * NS) {
        const int t = warp / NS, e = 32 * (warp - t * NS) + lane;
        if (e < E) lv0 = A.logits[(size_t)t * E + e];
    }
    for (int i = tid; i < T * (H / 8); i += DC_THREADS) {
        const int t = i / (H / 8);
        const uint4 q = reinterpret_cast<const uint4 *>(A.x)[i];
        reinterpret_cast<uint4 *>(xraw)[i] = q;
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
        atomicMax(&xmax[t], __float_as_uint(m));
    }
    for (int task = warp; task < T * NS; task += DC_WARPS) {
        const int t = task / NS, w = task - t * NS;
        const int e = 32 * w + lane;
        const float v = task == warp ? lv0 : (e < E ? A.logits[(size_t)t * E + e] : -INFINITY);
        const bool fin = isfinite(v);
        const float key = fin ? v : -INFINITY;
        if (__any_sync(0xffffffffu, e < E && !fin) && lane == 0)
            atomicOr(reinterpret_cast<unsigned *>(&misc[2]), (unsigned)MOE_FLAG_NONFINITE_LOGIT);
        rowk[t * NSE + e] = key;
        float bk = key;
        int bi = e < E ? e : 0x7fffffff;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (topk_beats(ok, oi, bk, bi)) {
                bk = ok;
                bi = oi;
            }
        }
        if (!A.renorm) {   // the slice's sum of exp(l - max) for the full-softmax denominator
            const float s = warp_sum((bk > -INFINITY && key > -INFINITY) ? expf(key - bk) : 0.0f);
            if (lane == 0) sls[t * NS + w] = s;
        }
        if (lane == 0) smax[t * NS + w] = make_float2(bk, __int_as_float(bi));
    }
    __syncthreads();

    // ---- 2. top-k. The k-th best slice best tau (per row) is a lower bound
    // of the row's k-th best logit: only logits that tau does not beat can be
    // selected, usually a few more than k. (a) warp t < T finds tau of row t
    // by counting, (b) every warp lists the survivors of its slices, (c) warp
    // t ranks the survivors of row t by counting (ranks are unique: the
    // order is total) and keeps ranks < k. Rows with more survivors than the
    // list holds are ranked over the whole row.
    if (warp < T) {
        const int t = warp;
        bool found = false;
        for (int l = lane; l < NS; l += 32) {
            const float2 me = smax[t * NS + l];
            int rank = 0;
#pragma unroll 4
            for (int j = 0; j < NS; ++j) {
                const float2 o = smax[t * NS + j];
                rank += topk_beats(o.x, __float_as_int(o.y), me.x, __float_as_int(me.y)) ? 1 : 0;
            }
            if (rank == k - 1) {
                tau[t] = me;
                found = true;
            }
        }
        if (!__any_sync(0xffffffffu, found) && lane == 0)   // fewer than k slices: every logit survives
            tau[t] = make_float2(-INFINITY, __int_as_float(0x7fffffff));
    }
    __syncthreads();
    for (int task = warp; task < T * NS; task += DC_WARPS) {
        const int t = task / NS, e = 32 * (task - t * NS) + lane;
        const float key = rowk[t * NSE + e];
        const float2 tt = tau[t];
        const bool sv = e < E && !topk_beats(tt.x, __float_as_int(tt.y), key, e);
        const unsigned b = __ballot_sync(0xffffffffu, sv);
        int base = 0;
        if (lane == 0 && b) base = atomicAdd(&scnt[t], __popc(b));
        base = __shfl_sync(0xffffffffu, base, 0) + __popc(b & ((1u << lane) - 1u));
        if (sv && base < DC_SURV) surv[t * DC_SURV + base] = make_float2(key, __int_as_float(e));
    }
    __syncthreads();

    // (c), then the kept flags and the (asynchronous) fetch of the selected
    // experts' descriptors; the router weights are needed only by the
    // combine. Warps >= T meanwhile convert the activations.
    // warp 0: sorts the (expert, pair) keys of the kept pairs (at most 64: two
    // per lane; one per lane, in 16 or 32 lanes, for up to 32 pairs), which
    // yields the active experts in ascending order and each expert's pairs in
    // ascending pair order; returns the number of active experts
    auto bucket_sorted = [&]() -> int { return dc_bucket_sorted(P, keep, ids, plist, act, aoff, misc); };
    auto route_weights = [&](int t) { dc_route_weights(t, k, NS, A.renorm, selk, smax, sls, wts); };
    // the chunk table (warp 0): see below
    auto build_chunks = [&](int n_act) { dc_build_chunks(n_act, I, H, c, G, A.rows_a, A.rows_b, A.chunk_cap, chunk, misc); };
    // one thread (lane ci % 16 of warp 0) issues the bulk copies of chunk ci
    // into ring slot ci % 16
    auto issue_chunk = [&](int ci, int nchunks_a, int b0) {
        dc_issue_chunk(ci, nchunks_a, b0, ring, A.stage, chunk, dpair, plist, aoff, full, misc);
    };

    if (warp < T) {
        const int t = warp;
        const int M = scnt[t];
        if (M <= DC_SURV) {
            for (int m = lane; m < M; m += 32) {
                const float2 me = surv[t * DC_SURV + m];
                const int mi = __float_as_int(me.y);
                int rank = 0;
#pragma unroll 4
                for (int o = 0; o < M; ++o) {
                    const float2 ot = surv[t * DC_SURV + o];
                    rank += topk_beats(ot.x, __float_as_int(ot.y), me.x, mi) ? 1 : 0;
                }
                if (rank < k) {
                    ids[t * k + rank] = mi;
                    selk[t * k + rank] = me.x;
                }
            }
        } else {
            const float2 tt = tau[t];
            for (int e = lane; e < E; e += 32) {
                const float key = rowk[t * NSE + e];
                if (topk_beats(tt.x, __float_as_int(tt.y), key, e)) continue;
                int rank = 0;
                for (int o = 0; o < E; ++o) rank += topk_beats(rowk[t * NSE + o], o, key, e) ? 1 : 0;
                if (rank < k) {
                    ids[t * k + rank] = e;
                    selk[t * k + rank] = key;
                }
            }
        }
        __syncwarp();
        if (lane < k) {
            const int p = t * k + lane;
            const int e = ids[p];
            bool kp = e >= A.lo && e < A.hi;
            if (kp && A.fmt_mask != 0xffffffffu) kp = (A.fmt_mask >> A.table[e].gate.fmt) & 1u;
            keep[p] = kp ? 1 : 0;
        }
        if (A.uniform) {
            // experts laid out at a constant step: no descriptor load
            if (lane < k) {
                const int p = t * k + lane;
                const long long e = ids[p];
                DevExpert d = A.u;
                d.gate.data += e * A.ustep[0];
                d.up.data += e * A.ustep[1];
                d.down.data += e * A.ustep[2];
                dpair[p] = d;
            }
        } else {
            constexpr int DW = (int)(sizeof(DevExpert) / 8);
            for (int i = lane; i < k * DW; i += 32) {
                const int p = t * k + i / DW, w = i % DW;
                cp_async8(reinterpret_cast<uint64_t *>(dpair + p) + w,
                          reinterpret_cast<const uint64_t *>(A.table + ids[p]) + w);
            }
            cp_async_commit();
        }
        if constexpr (!ONE) {
            route_weights(t);
            cp_async_wait_all();   // descriptors: warp 0 issues copies after the next barrier
        }
    } else {
        // activations -> int16 (per-token power-of-two scale: max |x| in
        // [2^14, 2^15)), in the order the Q4_K dot pairs codes with, stored
        // [v][group] for conflict-free reads. Four lanes per 64-column group:
        // lane q takes columns 8q..8q+7 and 32+8q..32+8q+7 (output words 2q
        // and 2q+1); the group's two exact activation sums are combined over
        // the four lanes.
        const int ntask = 4 * T * H64;
        for (int base = (warp - T) * 32; base < ntask; base += (DC_WARPS - T) * 32) {
            const int task = base + lane;
            const bool ok = task < ntask;
            const int g = ok ? task >> 2 : 0, q = task & 3;
            const int t = g / H64, G64 = g - t * H64;
            const int sg = pow2_shift(__uint_as_float(xmax[t]));
            const float up = exp2i(sg);
            const uint4 *src = reinterpret_cast<const uint4 *>(xraw) + (size_t)t * (H / 8) + 8 * G64;
            float xa[8], xb[8];
            {
                const uint4 qa = src[q], qb = src[4 + q];
                const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xa[2 * i] = __uint_as_float(wa[i] << 16) * up;
                    xa[2 * i + 1] = __uint_as_float(wa[i] & 0xffff0000u) * up;
                    xb[2 * i] = __uint_as_float(wb[i] << 16) * up;
                    xb[2 * i + 1] = __uint_as_float(wb[i] & 0xffff0000u) * up;
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)t * H / 2);
            int ia[8], ib[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ia[i] = max(-32767, min(32767, __float2int_rn(xa[i])));
                ib[i] = max(-32767, min(32767, __float2int_rn(xb[i])));
            }
            int sa = 0, sb = 0;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int i = 4 * h2;
                const uint32_t w0 = ((uint32_t)ia[i] & 0xffffu) | ((uint32_t)ia[i + 1] << 16);
                const uint32_t w1 = ((uint32_t)ia[i + 2] & 0xffffu) | ((uint32_t)ia[i + 3] << 16);
                const uint32_t w2 = ((uint32_t)ib[i] & 0xffffu) | ((uint32_t)ib[i + 1] << 16);
                const uint32_t w3 = ((uint32_t)ib[i + 2] & 0xffffu) | ((uint32_t)ib[i + 3] << 16);
                if (ok) dst[(2 * q + h2) * H64 + G64] = make_uint4(w0, w1, w2, w3);
                sa += ia[i] + ia[i + 1] + ia[i + 2] + ia[i + 3];
                sb += ib[i] + ib[i + 1] + ib[i + 2] + ib[i + 3];
            }
            sa += __shfl_xor_sync(0xffffffffu, sa, 1);
            sb += __shfl_xor_sync(0xffffffffu, sb, 1);
            sa += __shfl_xor_sync(0xffffffffu, sa, 2);
            sb += __shfl_xor_sync(0xffffffffu, sb, 2);
            if (ok && q == 0) {
                xsum[((size_t)t * H64 + G64) * 2 + 0] = (float)sa;
                xsum[((size_t)t * H64 + G64) * 2 + 1] = (float)sb;
                if (G64 == 0) xsc[t] = exp2i(-sg);
            }
        }
    }

    // ---- 3. bucketing, then the chunk table, both by warp 0.
    // One token: its selected experts are distinct, so the active experts are
    // taken in rank order, one pair each, without a sort (the published
    // routing is sorted at the end); warp 0 then issues the copies of the
    // ring slots that the raw activations do not occupy, and computes the
    // router weights while they are in flight.
    if (ONE && warp == 0) {
        cp_async_wait_all();
        __syncwarp();
        const bool kp = lane < k && keep[lane];
        const unsigned b = __ballot_sync(0xffffffffu, kp);
        const int n_act = __popc(b);
        if (kp) {
            const int a = __popc(b & ((1u << lane) - 1u));
            act[a] = ids[lane];
            aoff[a] = a;
            plist[a] = lane;
        }
        if (lane == 0) {
            aoff[n_act] = n_act;
            misc[0] = n_act;
            misc[6] = n_act;
        }
        __syncwarp();
        // the chunk table (the same chunks as in the general case below), each
        // lane computing its entries directly; the first ring fill is issued
        // as the entries are made (lane j: chunk j, ring slot j)
        {
            const int NA = n_act * I;
            const int a_begin = (int)((unsigned)NA * c / G), a_end = (int)((unsigned)NA * (c + 1) / G);
            const int b0 = (int)((unsigned)H * c / G), nrows_b = (int)((unsigned)H * (c + 1) / G) - b0;
            const int a_first = a_begin / I, a_last = a_end > a_begin ? (a_end - 1) / I : a_first - 1;
            const int ra = A.rows_a, rlog = 31 - __clz(ra);
            int total_a = 0;
            for (int a = a_first; a <= a_last; ++a) {
                const int rs = max(a_begin, a * I), len = min(a_end, (a + 1) * I) - rs;
                total_a += (len + ra - 1) >> rlog;
            }
            const int nb = (nrows_b + A.rows_b - 1) / A.rows_b;
            const int na = min(total_a, A.chunk_cap), nc = min(total_a + n_act * nb, A.chunk_cap);
            const int n0 = min(nc, DC_NSTAGE - nraw);
            for (int j = lane; j < nc; j += 32) {
                int4 d;
                if (j < total_a) {
                    int jj = j, a = a_first;
                    for (;; ++a) {
                        const int rs = max(a_begin, a * I), len = min(a_end, (a + 1) * I) - rs;
                        const int nch = (len + ra - 1) >> rlog;
                        if (jj < nch) {
                            d = make_int4(a, rs - a * I + (jj << rlog), min(ra, len - (jj << rlog)), 0);
                            break;
                        }
                        jj -= nch;
                    }
                } else {
                    const int jd = j - total_a, a = jd / nb, jb = jd - a * nb;
                    d = make_int4(a, jb * A.rows_b, min(A.rows_b, nrows_b - jb * A.rows_b), 1);
                }
                chunk[j] = d;
                if (j < n0) {
                    uint64_t *bar = &full[j];
                    uint8_t *dst = ring + (size_t)j * A.stage;
                    const DevExpert &X = dpair[plist[aoff[d.x]]];
                    if (j < na) {
                        const uint32_t bg = (uint32_t)(d.z * X.gate.stride), bu = (uint32_t)(d.z * X.up.stride);
                        mbar_expect_tx(bar, bg + bu);
                        bulk_g2s(dst, X.gate.data + (size_t)d.y * X.gate.stride, bg, bar);
                        bulk_g2s(dst + bg, X.up.data + (size_t)d.y * X.up.stride, bu, bar);
                    } else {
                        const uint32_t bd = (uint32_t)(d.z * X.down.stride);
                        mbar_expect_tx(bar, bd);
                        bulk_g2s(dst, X.down.data + (size_t)(b0 + d.y) * X.down.stride, bd, bar);
                    }
                    misc[16 + j] = j;
                }
            }
            if (lane == 0) {
                misc[4] = na;
                misc[5] = nc;
                misc[7] = n0;
            }
        }
        route_weights(0);
    }
    __syncthreads();
    // Several tokens: the sorted bucketing, then the chunk table.
    if (!ONE && warp == 0) {
        const int n_act = bucket_sorted();
        build_chunks(n_act);
        __syncwarp();
        const int n0 = min(misc[5], DC_NSTAGE - nraw);
        if (lane < n0) issue_chunk(lane, misc[4], (int)((unsigned)H * c / G));
        if (lane == 0) misc[7] = n0;
    }
    cp_async_wait_all();
    __syncthreads();
    const int nchunks_a = misc[4], nchunks = misc[5];
    const int b0 = (int)((unsigned)H * c / G), b1 = (int)((unsigned)H * (c + 1) / G);
    const int nrows_b = b1 - b0;
    // the next kernel in the stream may begin its launch; it waits for this
    // grid's completion before reading anything this grid writes
    asm volatile("griddepcontrol.launch_dependents;");

    // the ring slots that held the raw activations are free now
    if (warp == 0) {
        const int n_early = misc[7];
        if (lane >= n_early && lane < min(nchunks, DC_NSTAGE)) issue_chunk(lane, nchunks_a, b0);
    }

    // ---------------- the warps consume in rounds of up to 16 chunks (the
    // ring): a round's work items are spread over all 16 warps; a barrier ends
    // the round, and then lane s of warp 0 refills the slots the round used
    // (chunk ci + 16 after chunk ci), so no wait is ever more than one phase
    // ahead.
    // T = 1: every gate/up row meets the same activations; keep them in registers
    uint32_t xv1[32];
    float XA1 = 0.0f, XB1 = 0.0f;
    if (ONE && lane < H64) {
        const uint4 *xv4 = reinterpret_cast<const uint4 *>(xs);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const uint4 q = xv4[v * H64 + lane];
            xv1[4 * v + 0] = q.x;
            xv1[4 * v + 1] = q.y;
            xv1[4 * v + 2] = q.z;
            xv1[4 * v + 3] = q.w;
        }
        XA1 = xsum[lane * 2 + 0];
        XB1 = xsum[lane * 2 + 1];
    }
    // the gate/up rounds, compiled once with the activations hoisted into
    // registers (one token) and once general, so that the loop that runs is
    // compact in the instruction cache
    const int ra_log = 31 - __clz(A.rows_a);   // rows_a is a power of two
    auto phase_a = [&](auto hoist) {
        constexpr bool HOIST = decltype(hoist)::value;
        for (int cr = 0; cr < nchunks_a; cr += DC_NSTAGE) {
            const int cend = min(cr + DC_NSTAGE, nchunks_a);
            for (int f = cr * A.rows_a + warp; f < cend * A.rows_a; f += DC_CW) {
                const int ci = f >> ra_log, row = f & (A.rows_a - 1);
                const int4 ch = chunk[ci];
                const int n = ch.z, r0 = ch.y;
                if (row >= n) continue;
                const int s = ci % DC_NSTAGE;
                if (*reinterpret_cast<volatile int *>(&misc[1]) ||
                    !mbar_wait_timed(&full[s], (uint32_t)(ci / DC_NSTAGE) & 1u)) {
                    if (lane == 0) set_abort(misc, A.status);
                    break;
                }
                const int q0 = aoff[ch.x], ne = aoff[ch.x + 1] - q0;
                const DevExpert &X = dpair[plist[q0]];
                const uint8_t *stage = ring + (size_t)s * A.stage;
                const uint8_t *grow = stage + row * (int)X.gate.stride;
                const uint8_t *urow = stage + n * (int)X.gate.stride + row * (int)X.up.stride;
                for (int qi = 0; qi < ne; ++qi) {
                    const int p = plist[q0 + qi], t = HOIST ? 0 : p / k;
                    float part[2] = {0.0f, 0.0f};
                    if constexpr (HOIST) {
                        if (lane < H64) {
                            part[0] = q4k_dot64(grow + 144 * (lane >> 2), lane & 3, xv1, XA1, XB1);
                            part[1] = q4k_dot64(urow + 144 * (lane >> 2), lane & 3, xv1, XA1, XB1);
                        }
                    } else {
                        const uint4 *xv4 = reinterpret_cast<const uint4 *>(xs + (size_t)t * H / 2);
                        for (int G64 = lane; G64 < H64; G64 += 32) {
                            uint32_t xv[32];
    #pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const uint4 q = xv4[v * H64 + G64];
                                xv[4 * v + 0] = q.x;
                                xv[4 * v + 1] = q.y;
                                xv[4 * v + 2] = q.z;
                                xv[4 * v + 3] = q.w;
                            }
                            const float XA = xsum[((size_t)t * H64 + G64) * 2 + 0];
                            const float XB = xsum[((size_t)t * H64 + G64) * 2 + 1];
                            part[0] += q4k_dot64(grow + 144 * (G64 >> 2), G64 & 3, xv, XA, XB);
                            part[1] += q4k_dot64(urow + 144 * (G64 >> 2), G64 & 3, xv, XA, XB);
                        }
                    }
                    // gate total in lanes 0..15, up total in lanes 16..31
                    const float tot = warp_reduce2(part) * xsc[t];
                    const float upv = __shfl_down_sync(0xffffffffu, tot, 16);
                    if (lane == 0) A.h[(size_t)p * I + r0 + row] = silu_f32(tot) * upv;
                }
            }
            consumer_sync();
            // the last round's refills wait until warp 15 has arrived at the
            // grid barrier (below)
            if (warp == 0 && cr + DC_NSTAGE < nchunks_a && lane < cend - cr && cr + lane + DC_NSTAGE < nchunks &&
                !*reinterpret_cast<volatile int *>(&misc[1]))
                issue_chunk(cr + lane + DC_NSTAGE, nchunks_a, b0);
        }
    };
    phase_a(std::integral_constant<bool, ONE>{});

    // ---- grid barrier: every CTA's h is complete and visible. Warp 15
    // arrives (a release add: the CTA barrier orders the other warps' h
    // stores before it) and polls (bounded). Its fence waits for memory
    // operations still in flight, bulk copies included (it took about 1,700
    // cycles with the last refills just issued, 1,100 without), so warp 0
    // issues the last gate/up round's refills only after the arrival, on
    // named barrier 3 (warps 0 and 15).
    consumer_sync();
    if (warp == 0) {
        __syncwarp();
        asm volatile("bar.sync 3, 64;" ::: "memory");
        if (nchunks_a > 0) {
            const int cr = ((nchunks_a - 1) / DC_NSTAGE) * DC_NSTAGE;
            const int cend = min(cr + DC_NSTAGE, nchunks_a);
            if (lane < cend - cr && cr + lane + DC_NSTAGE < nchunks && !*reinterpret_cast<volatile int *>(&misc[1]))
                issue_chunk(cr + lane + DC_NSTAGE, nchunks_a, b0);
        }
    }
    if (c == 0 && warp < DC_CW - 1) {
        // CTA 0's warps 0..14 publish the routing while warp 15 waits at the
        // barrier. For one token the bucketing was used in rank order; the
        // published one is sorted here (into scratch, the rank-order arrays
        // are still in use).
        constexpr int SENT = 0x7fffffff;
        constexpr int PUB = 32 * (DC_CW - 1);
        int *sexp = reinterpret_cast<int *>(surv);   // sorted active experts (prologue scratch)
        if constexpr (ONE) {
            if (warp == 0) {
                int key = (lane < P && keep[lane]) ? ((ids[lane] << 8) | lane) : SENT;
                key = P <= 16 ? warp_sort_asc<16>(key) : warp_sort_asc<32>(key);
                if (P <= 16 && lane >= 16) key = SENT;
                const bool valid = key != SENT;
                const int nk = __popc(__ballot_sync(0xffffffffu, valid));
                if (valid) {
                    A.pairs_out[lane] = key & 0xff;
                    A.pos_out[key & 0xff] = lane;
                    A.active_out[1 + lane] = key >> 8;
                    sexp[lane] = key >> 8;
                }
                if (lane == 0) {
                    A.active_out[0] = nk;
                    misc[11] = nk;
                }
            }
            __syncwarp();
            asm volatile("bar.sync 2, %0;" ::"n"(PUB) : "memory");
            const int nk = misc[11];
#pragma unroll 1
            for (int e = tid; e <= E; e += PUB) {   // pairs of experts below e (one pair per expert)
                int cnt = 0;
#pragma unroll 1
                for (int i = 0; i < nk; ++i) cnt += sexp[i] < e ? 1 : 0;
                A.offsets_out[e] = cnt;
            }
        } else {
            const int n_act = misc[0], n_kept = misc[6];
            for (int e = tid; e <= E; e += PUB) {
                int lo = 0, hi = n_act;          // first active expert >= e
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (act[mid] < e) lo = mid + 1; else hi = mid;
                }
                A.offsets_out[e] = aoff[lo];
            }
            for (int a = tid; a < n_act; a += PUB) A.active_out[1 + a] = act[a];
            if (tid == 0) A.active_out[0] = n_act;
            for (int q = tid; q < n_kept; q += PUB) {
                A.pairs_out[q] = plist[q];
                A.pos_out[plist[q]] = q;
            }
        }
#pragma unroll 1
        for (int p = tid; p < P; p += PUB) {
            A.ids_out[p] = ids[p];
            A.wts_out[p] = wts[p];
            if (!keep[p]) A.pos_out[p] = -1;
        }
        if (tid == 0 && misc[2]) atomicOr(A.status, (uint32_t)misc[2]);
    }
    if (warp == DC_CW - 1) {
        if (lane == 0) red_release_add_u64(barrier_ctr, 1ull);
        __syncwarp();
        asm volatile("bar.arrive 3, 64;" ::: "memory");   // the whole warp: warp 0 may refill now
    }
    if (tid == 32 * (DC_CW - 1)) {
        // G arrivals past this launch's generation
        const unsigned long long target = (gen_count / (unsigned long long)G + 1ull) * (unsigned long long)G;
        const unsigned long long t_start = globaltimer_ns(), bound = *(volatile unsigned long long *)&g_wait_ns;
        while (ld_acquire_u64(barrier_ctr) < target) {
            if (globaltimer_ns() - t_start > bound) {
                set_abort(misc, A.status);
                break;
            }
        }
    }
    consumer_sync();
    if (*reinterpret_cast<volatile int *>(&misc[1])) {
        drain_copies(full, misc);
        return;
    }
    // ---- h of every pair -> shared memory as int16 with a power-of-two scale
    // per 32-column block (max |h| * 2^sigma in [2^13, 2^14)): eight
    // consecutive threads load one block with coalesced 16-byte loads from L2
    // (four in flight per thread), share its maximum and write 16 int16
    // pairs and 2^-sigma.
    if (nrows_b > 0) {
        const int n4 = I / 4, tot4 = P * n4;
        constexpr int NB = 4;
        for (int f0 = tid; f0 - tid < tot4; f0 += NB * DC_THREADS) {
            float4 v[NB];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int f = f0 + u * DC_THREADS;
                const int p = f / n4;
                v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (f < tot4 && keep[p]) v[u] = __ldcg(reinterpret_cast<const float4 *>(A.h + (size_t)p * I) + (f - p * n4));
            }
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int f = f0 + u * DC_THREADS;
                float m = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                if (f >= tot4) continue;
                const int p = f / n4, i4 = f - p * n4;
                uint32_t *dst = hq + ((size_t)p * U + (i4 >> 3)) * DC_HQW;
                const int be = (int)((__float_as_uint(m) >> 23) & 0xffu);   // m in [2^(be-127), 2^(be-126))
                if (be == 255) {   // inf or nan in the block: it propagates
                    *reinterpret_cast<uint2 *>(dst + 2 * (i4 & 7)) = make_uint2(0u, 0u);
                    if ((i4 & 7) == 0) dst[16] = 0x7fc00000u;
                    continue;
                }
                const int sg = m > 0.0f ? max(-100, min(100, 140 - be)) : 0;
                const float up = __uint_as_float((uint32_t)(127 + sg) << 23);
                const int q0 = __float2int_rn(v[u].x * up), q1 = __float2int_rn(v[u].y * up);
                const int q2 = __float2int_rn(v[u].z * up), q3 = __float2int_rn(v[u].w * up);
                *reinterpret_cast<uint2 *>(dst + 2 * (i4 & 7)) =
                    make_uint2(((uint32_t)q0 & 0xffffu) | ((uint32_t)q1 << 16), ((uint32_t)q2 & 0xffffu) | ((uint32_t)q3 << 16));
                if ((i4 & 7) == 0) dst[16] = (uint32_t)(127 - sg) << 23;   // 2^-sigma
            }
        }
    }
    consumer_sync();
    if (*reinterpret_cast<volatile int *>(&misc[1])) {
        drain_copies(full, misc);
        return;
    }
    if (nrows_b > 0) {
        // ---- down: this CTA's output rows [b0, b1) of every routed expert.
        // A unit is (down chunk, group of 16 rows, K part of 8 blocks); each
        // half-warp takes one, lane r its row r, over every pair of the
        // chunk's expert. The row's 8 blocks are one aligned 272-byte period
        // read with 16-byte loads (rows of a half-warp fall in distinct
        // banks); h is read by broadcast. The partial per K part lands in
        // ybuf and the combine adds the parts in order.
        const int KP = (U + 7) >> 3, NGR = (A.rows_b + 15) >> 4, upc = NGR * KP;
        const int r = lane & 15, hw = lane >> 4;
        for (int cr = nchunks_a; cr < nchunks; cr += DC_NSTAGE) {
            const int cend = min(cr + DC_NSTAGE, nchunks);
            const int nunits = (cend - cr) * upc;
            for (int uid = 2 * warp + hw; uid < nunits; uid += 2 * DC_CW) {
                const int ci = cr + uid / upc, rem = uid - (ci - cr) * upc;
                const int rg = rem / KP, kp = rem - rg * KP;
                const int4 ch = chunk[ci];
                const int nr = ch.z, row = 16 * rg + r;
                if (16 * rg >= nr) continue;
                const int s = ci % DC_NSTAGE;
                if (*reinterpret_cast<volatile int *>(&misc[1]) ||
                    !mbar_wait_timed(&full[s], (uint32_t)(ci / DC_NSTAGE) & 1u)) {
                    set_abort(misc, A.status);
                    break;
                }
                if (row >= nr) continue;
                const int q0 = aoff[ch.x], ne = aoff[ch.x + 1] - q0;
                const DevMatrix &D = dpair[plist[q0]].down;
                const uint8_t *wrow = ring + (size_t)s * A.stage + (size_t)row * D.stride + 272 * kp;
                const int nb = min(8, U - 8 * kp);
                for (int qi = 0; qi < ne; ++qi) {
                    const int p = plist[q0 + qi];
                    const float y = q8_0_period_dot(wrow, hq + ((size_t)p * U + 8 * kp) * DC_HQW, nb);
                    ybuf[(kp * P + p) * L.rb + ch.y + row] = y;
                }
            }
            consumer_sync();
            if (warp == 0 && lane < cend - cr && cr + lane + DC_NSTAGE < nchunks &&
                !*reinterpret_cast<volatile int *>(&misc[1]))
                issue_chunk(cr + lane + DC_NSTAGE, nchunks_a, b0);
        }
    }
    consumer_sync();
    if (*reinterpret_cast<volatile int *>(&misc[1])) {
        drain_copies(full, misc);
        return;
    }

    // ---- the down outputs: K parts added in order (one thread per output),
    // then the combine in ascending slot order
    const int KP = (U + 7) >> 3;
    if (KP > 1) {
        for (int i = tid; i < P * nrows_b; i += DC_THREADS) {
            const int p = i / nrows_b, rr = i - p * nrows_b;
            float y = ybuf[p * L.rb + rr];
            for (int kp = 1; kp < KP; ++kp) y += ybuf[(kp * P + p) * L.rb + rr];
            ybuf[p * L.rb + rr] = y;
        }
        consumer_sync();
    }
    for (int i = tid; i < T * nrows_b; i += DC_THREADS) {
        const int t = i / nrows_b, rr = i - t * nrows_b;
        float acc = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int p = t * k + j;
            if (keep[p]) acc = fmaf(wts[p], ybuf[p * L.rb + rr], acc);
        }
        A.out[(size_t)t * H + b0 + rr] = acc;
    }
}

int g_sm_count[64] = {};
bool g_attr_done[64] = {};

}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 64 && g_sm_count[dev]) return g_sm_count[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) g_sm_count[dev] = n;
    return n;
}

struct DcPlan {
    int stage, rows_a, rows_b, chunk_cap;
    size_t smem;
};

// Ring slot size, rows per chunk and shared-memory bytes of the fused decode
// kernel for a layer shape; smem = 0 if the shape does not fit.
DcPlan decode_fused_plan(int T, int k, int E, int H, int I, int G, int64_t gu_stride, int64_t dn_stride) {
    DcPlan pl{0, 0, 0, 0, 0};
    const size_t limit = 227 * 1024 - 1024;   // opt-in limit less the kernel's static shared memory
    const int64_t rowpair = 2 * gu_stride;
    const int rb = (H + G - 1) / G;
    for (int stage = DC_STAGE_MAX; stage >= 2048; stage -= 512) {
        int rows_a = (int)std::min<int64_t>(DC_ROWS_A, stage / rowpair);
        while (rows_a & (rows_a - 1)) --rows_a;   // a power of two: items split by shifts
        const int rows_b = (int)std::min<int64_t>(rb, stage / dn_stride);
        if (rows_a < 1 || rows_b < 1) return pl;
        const int P = T * k;
        const int share = P * I / G + 1;
        const int cap = share / rows_a + P + 2 + P * ((rb + rows_b - 1) / rows_b);
        const DcLayout L = dc_layout(T, k, E, H, I, G, stage, cap);
        // the raw activation rows are staged in the ring during the prologue
        if ((size_t)T * H * 2 > (size_t)DC_NSTAGE * stage) continue;
        if (L.total <= limit) {
            pl.stage = stage;
            pl.rows_a = rows_a;
            pl.rows_b = rows_b;
            pl.chunk_cap = cap;
            pl.smem = L.total;
            return pl;
        }
    }
    return pl;
}

// Whether the fused decode kernel handles this layer shape.
bool decode_fused_eligible(int T, int k, int E, int H, int I, uint32_t gateup_formats, uint32_t down_formats,
                           int64_t gu_stride, int64_t dn_stride) {
    if (T < 1 || T > DC_WARPS - 1 || T * k > DC_MAX_PAIRS || E > MOE_MAX_EXPERTS || E > 2 * DC_THREADS) return false;
    if (gateup_formats != (1u << MOE_Q4_K) || down_formats != (1u << MOE_Q8_0)) return false;
    if (H % 64 != 0 || I % 32 != 0 || I / 32 > 32) return false;
    const int G = sm_count();
    if (G <= 0) return false;
    return decode_fused_plan(T, k, E, H, I, G, gu_stride, dn_stride).smem != 0;
}

cudaError_t launch_decode_fused(const DevExpert *table, const moe_weight_table *W, int T, int k, int E, int H, int I,
                                int64_t gu_stride, int64_t dn_stride, int renorm, int lo, int hi, uint32_t fmt_mask, const float *logits,
                                const uint16_t *x, float *out, float *h, int32_t *ids, float *wts, int32_t *offsets,
                                int32_t *active, int32_t *pairs, int32_t *pos, unsigned char *sync, uint32_t *status,
                                cudaStream_t s) {
    const int G = sm_count();
    const DcPlan pl = decode_fused_plan(T, k, E, H, I, G, gu_stride, dn_stride);
    const size_t smem = pl.smem;
    if (G <= 0 || smem == 0) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || !g_attr_done[dev]) {
        int optin = 0;
        err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (err != cudaSuccess) return err;
        for (int one = 0; one < 2; ++one) {
            const void *fn = one ? reinterpret_cast<const void *>(&decode_fused_kernel<true>)
                                 : reinterpret_cast<const void *>(&decode_fused_kernel<false>);
            cudaFuncAttributes fa;
            err = cudaFuncGetAttributes(&fa, fn);
            if (err != cudaSuccess) return err;
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
            if (err != cudaSuccess) return err;
        }
        if (dev < 64) g_attr_done[dev] = true;
    }
    DcArgs A;
    A.table = table;
    A.E = E;
    A.H = H;
    A.I = I;
    A.T = T;
    A.k = k;
    A.renorm = renorm;
    A.lo = lo;
    A.hi = hi;
    A.fmt_mask = fmt_mask;
    A.logits = logits;
    A.x = x;
    A.out = out;
    A.h = h;
    A.ids_out = ids;
    A.wts_out = wts;
    A.offsets_out = offsets;
    A.active_out = active;
    A.pairs_out = pairs;
    A.pos_out = pos;
    A.sync = sync;
    A.status = status;
    A.stage = pl.stage;
    A.rows_a = pl.rows_a;
    A.rows_b = pl.rows_b;
    A.chunk_cap = pl.chunk_cap;
    A.uniform = W->uniform_layout;
    {
        const moe_matrix *src[3] = {&W->uniform_base.gate, &W->uniform_base.up, &W->uniform_base.down};
        DevMatrix *dst[3] = {&A.u.gate, &A.u.up, &A.u.down};
        for (int i = 0; i < 3; ++i) {
            dst[i]->data = static_cast<const uint8_t *>(src[i]->data);
            dst[i]->stride = src[i]->row_stride_bytes;
            dst[i]->fmt = src[i]->format;
            dst[i]->rows = src[i]->rows;
            A.ustep[i] = W->uniform_step[i];
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(DC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (T == 1 && H / 64 <= 32) return cudaLaunchKernelEx(&cfg, decode_fused_kernel<true>, A);
    return cudaLaunchKernelEx(&cfg, decode_fused_kernel<false>, A);
}

// This file's copy of the wait bound (moe_set_wait_timeout_ns).
cudaError_t set_wait_ns_decode(unsigned long long ns) { return set_tu_wait_ns(ns); }

}  // namespace moe
