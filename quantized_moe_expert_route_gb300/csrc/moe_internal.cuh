// Internal definitions shared by the library's kernels (not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "moe_route.h"

namespace moe {

// Device copy of one matrix descriptor (24 bytes).
struct DevMatrix {
    const uint8_t *data;
    int64_t stride;
    int32_t fmt;
    int32_t rows;
};

struct DevExpert {
    DevMatrix gate, up, down;
};

// Bytes at the start of a workspace that hold its device state: the status
// word (offset 0) and the fused kernel's grid-barrier counter (offset 8).
constexpr size_t SYNC_BYTES = 1024;

// Bucketing of more than BUCKET_MANY pairs runs over ranges of BUCKET_RANGE
// pairs and needs per-range expert histograms in the workspace.
constexpr int BUCKET_MANY = 2048;
constexpr int BUCKET_RANGE = 512;
inline size_t bucket_scratch_bytes(int T, int k, int E) {
    const size_t P = (size_t)T * k;
    return P > (size_t)BUCKET_MANY ? ((P + BUCKET_RANGE - 1) / BUCKET_RANGE) * (size_t)E * 4 : 0;
}

// Workspace layout of moe_ffn_forward; offsets in bytes from the workspace base.
struct WsLayout {
    size_t status, ids, wts, offsets, active, pairs, pos, h, y, bscratch, total;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(int T, int k, int E, int H, int I) {
    WsLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
    size_t P = (size_t)T * k;
    L.status = take(SYNC_BYTES);
    L.ids = take(P * 4);
    L.wts = take(P * 4);
    L.offsets = take((size_t)(E + 1) * 4);
    L.active = take((size_t)(E + 1) * 4);
    L.pairs = take(P * 4);
    L.pos = take(P * 4);
    L.h = take(P * (size_t)I * 4);
    L.y = take(P * (size_t)H * 4);
    L.bscratch = take(bucket_scratch_bytes(T, k, E));
    L.total = o;
    return L;
}

// Extra workspace of the tensor-core path, after the common layout (only
// sized in when that path can run; offsets from the workspace base):
// activations in bucket order as fp16 [P][H] with inverse row scales, |h|
// maxima, h as fp16 [P][I] with inverse row scales, and the chunk table.
struct TcLayout {
    size_t xg, xinv, hmax, h16, hinv, chunks, n_chunks, unit_next, total;
};

inline size_t tc_max_chunks(int T, int k, int E) {
    const size_t P = (size_t)T * k;
    return P / 128 + (P < (size_t)E ? P : (size_t)E) + 1;
}

inline TcLayout tc_ws_layout(int T, int k, int E, int H, int I) {
    const WsLayout L = ws_layout(T, k, E, H, I);
    TcLayout C;
    size_t o = L.total;
    auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
    const size_t P = (size_t)T * k;
    C.xg = take(P * H * 2);
    C.xinv = take(P * 4);
    C.hmax = take(P * 4);
    C.h16 = take(P * I * 2);
    C.hinv = take(P * 4);
    C.chunks = take(tc_max_chunks(T, k, E) * 16);
    C.n_chunks = take(4);
    C.unit_next = take(8);   // the two GEMMs' unit counters
    C.total = o;
    return C;
}

// The cold-expert tier (cold.cu): workspace regions after the path's own
// (remapped descriptor table, copy segments, staging of the routed cold
// experts' bytes), present when the weight table has cold experts.
struct ColdSeg {
    const uint8_t *src;
    uint8_t *dst;
    uint64_t bytes;
};
struct ColdLayout {
    size_t remap, segs, n_segs, staging, total;
};
inline ColdLayout cold_ws_layout(size_t after, int T, int k, int E, int n_cold, int64_t cold_bytes_max) {
    ColdLayout C;
    size_t o = after;
    auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
    const size_t P = (size_t)T * k, nc = P < (size_t)n_cold ? P : (size_t)n_cold;
    C.remap = take((size_t)E * sizeof(DevExpert));
    C.segs = take(3 * nc * sizeof(ColdSeg));
    C.n_segs = take(4);
    C.staging = take(nc * (size_t)cold_bytes_max);
    C.total = o;
    return C;
}
cudaError_t launch_cold_staging(const DevExpert *table, const uint8_t *cold, int E, const int32_t *active,
                                char *ws_base, const ColdLayout &C, cudaStream_t s);

constexpr int BLOCK_ELEMS[9] = {0, 32, 256, 256, 32, 32, 256, 256, 128};
constexpr int BLOCK_BYTES[9] = {0, 34, 144, 210, 17, 18, 136, 98, 28};

// Bounded waits: a wait that exceeds this many polls sets MOE_FLAG_WAIT_TIMEOUT.
constexpr uint32_t WAIT_LIMIT = 1u << 26;

// The time bound (ns) of the kernels' waits for data or for other threads
// (ring slots, barriers); the waits for a CTA's own copies in flight before
// it exits (drains) keep the poll bound above. Default 2 s: a whole layer
// takes well under a millisecond. Each translation unit has its own copy
// (no relocatable device code); moe_set_wait_timeout_ns sets all of them.
constexpr unsigned long long DEFAULT_WAIT_NS = 2000000000ull;
static __device__ unsigned long long g_wait_ns = DEFAULT_WAIT_NS;
static inline cudaError_t set_tu_wait_ns(unsigned long long ns) {
    return cudaMemcpyToSymbol(g_wait_ns, &ns, sizeof(ns));
}

// Host helpers shared by the launchers (gemv.cu, decode.cu).
cudaError_t record_event(cudaEvent_t ev, cudaStream_t s);   // event (graph node when capturing)
cudaError_t allow_max_dynamic_smem(const void *fn);         // opt in to all free shared memory
int current_device();
int sm_count();
// out[t] = sum over slots j ascending of w[t,j] * y[pos[t,j]]; y in bucket order,
// each row q first multiplied by yscale[q] (a power of two) when yscale is given
cudaError_t launch_combine(int T, int k, int H, const int32_t *pos, const float *wts, const float *y, float *out,
                           cudaStream_t s, const float *yscale = nullptr);

// Streaming grouped GEMV for decode batches (stream.cu): the launch plan
// (ok == false if the kernels cannot run the layer) and the launcher of its
// gate/up and down kernels (the combine is launched separately).
struct SgPlan {
    bool ok;
    bool iq;   // the variant of the kernels that decodes the IQ formats
    int cr, ns, stage, nexp, nsb, stageb, nq;
    size_t smem_a, smem_b;
};
SgPlan stream_plan(int T, int k, int E, int H, int I, uint32_t gu_formats, uint32_t down_formats, int64_t gu_stride,
                   int64_t dn_stride);
cudaError_t launch_stream_path(const DevExpert *table, const SgPlan &p, int T, int k, int E, int H, int I,
                               const int32_t *offsets, const int32_t *pairs, const int32_t *active, const uint16_t *x,
                               float *h, float *y, uint32_t *status, const uint32_t *grid, cudaEvent_t const *events,
                               cudaStream_t s);

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Returns true once the phase with the given parity has completed; false after
// WAIT_LIMIT polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    uint32_t addr = smem_addr(bar);
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Returns true once the phase with the given parity has completed; false
// after g_wait_ns (or WAIT_LIMIT polls). For waits on data or on other
// threads; drains use mbar_wait.
static __device__ __noinline__ bool mbar_wait_timed_slow(uint32_t addr, uint32_t parity) {
    const unsigned long long t0 = now_ns(), bound = *(volatile unsigned long long *)&g_wait_ns;
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if (now_ns() - t0 > bound) return false;
    }
    return false;
}
__device__ __forceinline__ bool mbar_wait_timed(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_addr(bar);
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    return done || mbar_wait_timed_slow(addr, parity);
}

// 1-D bulk copy global -> shared (TMA engine). dst, src 16-byte aligned,
// bytes a multiple of 16. Completion is signalled on `bar` as tx bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ float half_bits_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// 2^(e-128) for an E8M0 byte e, exact (subnormal for e < 2).
__device__ __forceinline__ float e8m0_half_scale(uint32_t e) {
    return e >= 2 ? __uint_as_float((e - 1) << 23) : __uint_as_float(0x00200000u << e);
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// (key, idx) a ranks before (key, idx) b: larger key, or equal key and lower index.
__device__ __forceinline__ bool topk_beats(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Softmax top-k of one row of E logits by one warp (E <= 32 * V, k <= 32).
// Selection compares the raw fp32 logits (largest first, equal logits to the
// lower expert index); non-finite logits rank last with probability 0. Lane
// j < k receives slot j's expert id and weight: its softmax probability,
// divided by the sum over the k selected ones when renorm != 0. Returns true
// (in every lane) if the row holds a non-finite logit.
template <int V>
__device__ __forceinline__ bool warp_topk(const float *__restrict__ lr, int E, int k, int renorm, int &sel_idx,
                                          float &weight) {
    const int lane = threadIdx.x & 31;
    float key[V];
    bool nonfinite = false;
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int e = lane + 32 * i;
        const float v = e < E ? lr[e] : -INFINITY;
        const bool fin = isfinite(v);
        if (e < E && !fin) nonfinite = true;
        key[i] = fin ? v : -INFINITY;
        m = fmaxf(m, key[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const bool any_finite = m > -INFINITY;
    nonfinite = __any_sync(0xffffffffu, nonfinite);

    uint32_t taken = 0;
    float sel_key = -INFINITY;
    sel_idx = 0;
    for (int j = 0; j < k; ++j) {
        float bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !(taken & (1u << i)) && topk_beats(key[i], e, bk, bi)) {
                bk = key[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (topk_beats(ok, oi, bk, bi)) {
                bk = ok;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            sel_key = bk;
            sel_idx = bi;
        }
    }
    const float ex = (lane < k && any_finite && sel_key > -INFINITY) ? expf(sel_key - m) : 0.0f;
    float denom;
    if (renorm) {
        denom = ex;
#pragma unroll
        for (int o = 16; o; o >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, o);
    } else {
        float s = 0.0f;
        if (any_finite) {
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (key[i] > -INFINITY) s += expf(key[i] - m);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        denom = s;
    }
    weight = denom > 0.0f ? ex / denom : 0.0f;
    return nonfinite;
}

}  // namespace moe
