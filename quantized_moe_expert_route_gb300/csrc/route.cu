// Router: softmax over E logits and top-k, one warp per token row.
//
// "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南", section
// 瓶颈分析: a light router picks, per token, the k best-matching experts of the
// layer. Selection compares the raw fp32 logits (softmax is monotone), largest
// first, equal logits resolved to the lower expert index, non-finite logits
// last; the weights are the selected softmax probabilities, optionally
// renormalised to sum to one.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int ROUTE_WARPS = 8;

// (key, idx) a beats (key, idx) b: larger key, or equal key and lower index.
__device__ __forceinline__ bool beats(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

template <int V>  // logits per lane: E <= 32 * V
__global__ void __launch_bounds__(ROUTE_WARPS * 32)
route_topk_kernel(const float *__restrict__ logits, int T, int E, int k, int renorm, int32_t *__restrict__ ids,
                  float *__restrict__ wts, uint32_t *__restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * ROUTE_WARPS + (threadIdx.x >> 5);
    if (row >= T) return;
    const float *lr = logits + (size_t)row * E;

    float key[V];
    bool nonfinite = false;
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        int e = lane + 32 * i;
        float v = e < E ? lr[e] : -INFINITY;
        bool fin = isfinite(v);
        if (e < E && !fin) nonfinite = true;
        key[i] = fin ? v : -INFINITY;
        m = fmaxf(m, key[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const bool any_finite = m > -INFINITY;
    nonfinite = __any_sync(0xffffffffu, nonfinite);

    // top-k by repeated warp arg-max over the untaken entries
    uint32_t taken = 0;
    float sel_key = -INFINITY;
    int sel_idx = 0;
    for (int j = 0; j < k; ++j) {
        float bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            int e = lane + 32 * i;
            if (e < E && !(taken & (1u << i)) && beats(key[i], e, bk, bi)) {
                bk = key[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (beats(ok, oi, bk, bi)) {
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

    // weights
    float ex = (lane < k && any_finite && sel_key > -INFINITY) ? expf(sel_key - m) : 0.0f;
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
    if (lane < k) {
        ids[(size_t)row * k + lane] = sel_idx;
        wts[(size_t)row * k + lane] = denom > 0.0f ? ex / denom : 0.0f;
    }
    if (nonfinite && lane == 0 && status) atomicOr(status, (uint32_t)MOE_FLAG_NONFINITE_LOGIT);
}

template <int V>
cudaError_t launch_v(const float *logits, int T, int E, int k, int renorm, int32_t *ids, float *wts, uint32_t *status,
                     cudaStream_t s) {
    dim3 grid((T + ROUTE_WARPS - 1) / ROUTE_WARPS);
    route_topk_kernel<V><<<grid, ROUTE_WARPS * 32, 0, s>>>(logits, T, E, k, renorm, ids, wts, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route_topk(const float *logits, int T, int E, int k, int renorm, int32_t *ids, float *wts,
                              uint32_t *status, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    int v = (E + 31) / 32;
    if (v <= 1) return launch_v<1>(logits, T, E, k, renorm, ids, wts, status, s);
    if (v <= 2) return launch_v<2>(logits, T, E, k, renorm, ids, wts, status, s);
    if (v <= 4) return launch_v<4>(logits, T, E, k, renorm, ids, wts, status, s);
    if (v <= 8) return launch_v<8>(logits, T, E, k, renorm, ids, wts, status, s);
    if (v <= 16) return launch_v<16>(logits, T, E, k, renorm, ids, wts, status, s);
    return launch_v<32>(logits, T, E, k, renorm, ids, wts, status, s);
}

}  // namespace moe
