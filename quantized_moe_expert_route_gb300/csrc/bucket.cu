// Token -> expert bucketing: per-expert counts, exclusive prefix sum, stable
// scatter of pair numbers, active-expert list. One CTA; integer only.
//
// "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南", section
// 优化策略三 (ids outside the kept range [min, max) are skipped, not redirected)
// and section 关键 Bug 修复与调试踩坑记录 (bug 1: redirecting skipped ids to expert 0
// duplicated it within a token and broke the grouping; bug 3: -1 must stay a
// signed skip id). Here ids stay int32 throughout, -1 is dropped before any
// indexing, and every other out-of-range id is flagged and dropped.
//
// Stability (pairs ascending within an expert) comes from processing the pairs
// in chunks of 1024 in order: within a warp, __match_any_sync ranks the lanes
// that share an expert; per expert, an exclusive scan over the 32 warps of the
// chunk orders the warps; a running per-expert count orders the chunks.
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {

namespace {

constexpr int BK_THREADS = 1024;
constexpr int BK_WARPS = BK_THREADS / 32;

__device__ __forceinline__ bool keep_pair(int e, int E, int lo, int hi, uint32_t fmt_mask, const DevExpert *table,
                                          uint32_t &flags) {
    if (e == -1) return false;
    if (e < 0 || e >= E) {
        flags |= MOE_FLAG_BAD_ID;
        return false;
    }
    if (e < lo || e >= hi) return false;
    if (table && !((fmt_mask >> table[e].gate.fmt) & 1u)) return false;
    return true;
}

// Block-wide exclusive scan of one int per thread; returns the total too.
__device__ int block_excl_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_tot[lane] = wi - w;  // exclusive warp offsets
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    int r = warp_tot[warp] + incl - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(BK_THREADS, 1)
bucket_kernel(const int32_t *__restrict__ ids, int T, int k, int E, int lo, int hi, uint32_t fmt_mask,
              const DevExpert *__restrict__ table, int32_t *__restrict__ offsets, int32_t *__restrict__ pairs,
              int32_t *__restrict__ pos, int32_t *__restrict__ active, uint32_t *__restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_trigger();
    pdl_wait();   // the ids come from the router kernel
    int *count = reinterpret_cast<int *>(smem);        // [E]
    int *base = count + E;                              // [E] bucket start
    int *run = base + E;                                // [E] pairs placed so far
    int *ctot = run + E;                                // [E] pairs in this chunk
    uint16_t *wcnt = reinterpret_cast<uint16_t *>(ctot + E);  // [32][E]
    __shared__ int warp_tot[33];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = T * k;
    uint32_t flags = 0;

    for (int e = tid; e < E; e += BK_THREADS) {
        count[e] = 0;
        run[e] = 0;
    }
    for (int i = tid; i < BK_WARPS * E; i += BK_THREADS) wcnt[i] = 0;
    __syncthreads();

    for (int p = tid; p < P; p += BK_THREADS) {
        int e = ids[p];
        if (keep_pair(e, E, lo, hi, fmt_mask, table, flags)) atomicAdd(&count[e], 1);
    }
    for (int t = tid; t < T; t += BK_THREADS) {
        const int32_t *r = ids + (size_t)t * k;
        for (int a = 0; a < k; ++a) {
            int ea = r[a];
            if (ea < 0 || ea >= E) continue;
            for (int b = a + 1; b < k; ++b)
                if (r[b] == ea) flags |= MOE_FLAG_DUPLICATE_ID;
        }
    }
    __syncthreads();

    // offsets and active list (E <= 1024 = one expert per thread)
    int c = tid < E ? count[tid] : 0;
    int total, nact;
    int excl = block_excl_scan(c, warp_tot, total);
    int aexcl = block_excl_scan(c > 0 ? 1 : 0, warp_tot, nact);
    if (tid < E) {
        offsets[tid] = excl;
        base[tid] = excl;
        if (c > 0) active[1 + aexcl] = tid;
    }
    if (tid == 0) {
        offsets[E] = total;
        active[0] = nact;
    }
    __syncthreads();

    // stable scatter, chunk by chunk
    for (int c0 = 0; c0 < P; c0 += BK_THREADS) {
        int p = c0 + tid;
        uint32_t dummy = 0;
        int e = p < P ? ids[p] : -1;
        bool kp = p < P && keep_pair(e, E, lo, hi, fmt_mask, table, dummy);
        int key = kp ? e : -1;
        uint32_t peers = __match_any_sync(0xffffffffu, key);
        int rank = __popc(peers & ((1u << lane) - 1u));
        if (kp && rank == 0) wcnt[warp * E + e] = (uint16_t)__popc(peers);
        __syncthreads();
        for (int x = tid; x < E; x += BK_THREADS) {
            int acc = 0;
            for (int w = 0; w < BK_WARPS; ++w) {
                int v = wcnt[w * E + x];
                wcnt[w * E + x] = (uint16_t)acc;
                acc += v;
            }
            ctot[x] = acc;
        }
        __syncthreads();
        if (kp) {
            int q = base[e] + run[e] + wcnt[warp * E + e] + rank;
            pairs[q] = p;
            pos[p] = q;
        } else if (p < P) {
            pos[p] = -1;
        }
        __syncthreads();
        for (int x = tid; x < E; x += BK_THREADS) {
            run[x] += ctot[x];
            for (int w = 0; w < BK_WARPS; ++w) wcnt[w * E + x] = 0;
        }
        __syncthreads();
    }

    flags = __reduce_or_sync(0xffffffffu, flags);
    if (flags && lane == 0 && status) atomicOr(status, flags);
}

// ---- many pairs: three short kernels over 512-pair ranges (one CTA each)
constexpr int BM_THREADS = BUCKET_RANGE;
constexpr int BM_WARPS = BM_THREADS / 32;

// 1. per-range expert histograms -> cnt[c][e]; duplicate-id flags per token
__global__ void __launch_bounds__(BM_THREADS) bucket_count_kernel(const int32_t *__restrict__ ids, int T, int k, int E,
                                                                 int lo, int hi, uint32_t fmt_mask,
                                                                 const DevExpert *__restrict__ table,
                                                                 int32_t *__restrict__ cnt, uint32_t *__restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_trigger();
    pdl_wait();
    int *hist = reinterpret_cast<int *>(smem);   // [E]
    const int tid = threadIdx.x, P = T * k;
    for (int e = tid; e < E; e += BM_THREADS) hist[e] = 0;
    __syncthreads();
    uint32_t flags = 0;
    const int p = blockIdx.x * BM_THREADS + tid;
    if (p < P) {
        const int e = ids[p];
        if (keep_pair(e, E, lo, hi, fmt_mask, table, flags)) atomicAdd(&hist[e], 1);
        // duplicates: compare with the later slots of the same token
        const int t = p / k, j = p - t * k;
        if (e >= 0 && e < E)
            for (int b = j + 1; b < k; ++b)
                if (ids[(size_t)t * k + b] == e) flags |= MOE_FLAG_DUPLICATE_ID;
    }
    __syncthreads();
    for (int e = tid; e < E; e += BM_THREADS) cnt[(size_t)blockIdx.x * E + e] = hist[e];
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (flags && (tid & 31) == 0 && status) atomicOr(status, flags);
}

// 2. one CTA: per expert, exclusive scan over the ranges (cnt becomes each
// range's first bucket position), offsets, active list
__global__ void __launch_bounds__(BK_THREADS, 1) bucket_scan_kernel(int G, int E, int32_t *__restrict__ cnt,
                                                                    int32_t *__restrict__ offsets,
                                                                    int32_t *__restrict__ active) {
    __shared__ int warp_tot[33];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    constexpr int BATCH = 16;   // independent loads in flight per thread (one range's load at a time took ~15 us)
    int c = 0;
    if (tid < E) {
        for (int r0 = 0; r0 < G; r0 += BATCH) {
            int v[BATCH];
#pragma unroll
            for (int j = 0; j < BATCH; ++j) v[j] = r0 + j < G ? cnt[(size_t)(r0 + j) * E + tid] : 0;
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                if (r0 + j < G) cnt[(size_t)(r0 + j) * E + tid] = c;
                c += v[j];
            }
        }
    }
    int total, nact;
    const int excl = block_excl_scan(c, warp_tot, total);
    const int aexcl = block_excl_scan(c > 0 ? 1 : 0, warp_tot, nact);
    if (tid < E) {
        offsets[tid] = excl;
        if (c > 0) active[1 + aexcl] = tid;
        for (int r0 = 0; r0 < G; r0 += BATCH) {
            int v[BATCH];
#pragma unroll
            for (int j = 0; j < BATCH; ++j) v[j] = r0 + j < G ? cnt[(size_t)(r0 + j) * E + tid] : 0;
#pragma unroll
            for (int j = 0; j < BATCH; ++j)
                if (r0 + j < G) cnt[(size_t)(r0 + j) * E + tid] = v[j] + excl;
        }
    }
    if (tid == 0) {
        offsets[E] = total;
        active[0] = nact;
    }
}

// 3. per range: stable scatter (warps in order, lanes in order within a warp)
__global__ void __launch_bounds__(BM_THREADS) bucket_scatter_kernel(const int32_t *__restrict__ ids, int P, int E,
                                                                   int lo, int hi, uint32_t fmt_mask,
                                                                   const DevExpert *__restrict__ table,
                                                                   const int32_t *__restrict__ cnt,
                                                                   int32_t *__restrict__ pairs,
                                                                   int32_t *__restrict__ pos) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_trigger();
    pdl_wait();
    uint16_t *wcnt = reinterpret_cast<uint16_t *>(smem);   // [BM_WARPS][E]: exclusive per-warp offsets
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < BM_WARPS * E; i += BM_THREADS) wcnt[i] = 0;
    __syncthreads();
    const int p = blockIdx.x * BM_THREADS + tid;
    uint32_t dummy = 0;
    const int e = p < P ? ids[p] : -1;
    const bool kp = p < P && keep_pair(e, E, lo, hi, fmt_mask, table, dummy);
    const int key = kp ? e : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (kp && rank == 0) wcnt[warp * E + e] = (uint16_t)__popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += BM_THREADS) {
        int acc = 0;
        for (int w = 0; w < BM_WARPS; ++w) {
            const int v = wcnt[w * E + x];
            wcnt[w * E + x] = (uint16_t)acc;
            acc += v;
        }
    }
    __syncthreads();
    if (kp) {
        const int q = cnt[(size_t)blockIdx.x * E + e] + wcnt[warp * E + e] + rank;
        pairs[q] = p;
        pos[p] = q;
    } else if (p < P) {
        pos[p] = -1;
    }
}

}  // namespace

size_t bucket_smem_bytes(int E) { return (size_t)E * 4 * 4 + (size_t)BK_WARPS * E * 2; }


cudaError_t launch_bucket(const int32_t *ids, int T, int k, int E, int lo, int hi, uint32_t fmt_mask,
                          const DevExpert *table, int32_t *offsets, int32_t *pairs, int32_t *pos, int32_t *active,
                          uint32_t *status, int32_t *scratch, cudaStream_t s) {
    size_t smem = bucket_smem_bytes(E);
    static bool attr_set[64] = {};  // the attribute is per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !attr_set[dev]) {
        cudaError_t err =
            cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
        if (err != cudaSuccess) return err;
        if (dev < 64) attr_set[dev] = true;
    }
    const int P = T * k;
    if (P > BUCKET_MANY && scratch) {
        const int G = (P + BM_THREADS - 1) / BM_THREADS;
        cudaError_t err = launch_pdl(bucket_count_kernel, dim3(G), dim3(BM_THREADS), (size_t)E * 4, s, ids, T, k, E,
                                     lo, hi, fmt_mask, table, scratch, status);
        if (err != cudaSuccess) return err;
        err = launch_pdl(bucket_scan_kernel, dim3(1), dim3(BK_THREADS), 0, s, G, E, scratch, offsets, active);
        if (err != cudaSuccess) return err;
        return launch_pdl(bucket_scatter_kernel, dim3(G), dim3(BM_THREADS), (size_t)BM_WARPS * E * 2, s, ids, P, E, lo,
                          hi, fmt_mask, table, (const int32_t *)scratch, pairs, pos);
    }
    return launch_pdl(bucket_kernel, dim3(1), dim3(BK_THREADS), smem, s, ids, T, k, E, lo, hi, fmt_mask, table, offsets,
                      pairs, pos, active, status);
}

}  // namespace moe
