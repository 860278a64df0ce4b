// Router: softmax over E logits and top-k, one warp per token row.
//
// "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南", section
// 瓶颈分析: a light router picks, per token, the k best-matching experts of the
// layer. Selection compares the raw fp32 logits (softmax is monotone), largest
// first, equal logits resolved to the lower expert index, non-finite logits
// last; the weights are the selected softmax probabilities, optionally
// renormalised to sum to one.
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {

namespace {

constexpr int ROUTE_WARPS = 8;

template <int V>  // logits per lane: E <= 32 * V
__global__ void __launch_bounds__(ROUTE_WARPS * 32)
route_topk_kernel(const float *__restrict__ logits, int T, int E, int k, int renorm, int32_t *__restrict__ ids,
                  float *__restrict__ wts, uint32_t *__restrict__ status, int stride, int n_shared) {
    // the logits may come from the previous kernel in the stream
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * ROUTE_WARPS + (threadIdx.x >> 5);
    if (row >= T) return;
    int sel;
    float w;
    const bool nonfinite = warp_topk<V>(logits + (size_t)row * E, E, k, renorm, sel, w);
    if (lane < k) {
        ids[(size_t)row * stride + lane] = sel;
        wts[(size_t)row * stride + lane] = w;
    } else if (lane < k + n_shared) {
        // the shared experts (ids E, E + 1, ...) in the slots after the routed ones, weight 1
        ids[(size_t)row * stride + lane] = E + (lane - k);
        wts[(size_t)row * stride + lane] = 1.0f;
    }
    if (nonfinite && lane == 0 && status) atomicOr(status, (uint32_t)MOE_FLAG_NONFINITE_LOGIT);
}

template <int V>
cudaError_t launch_v(const float *logits, int T, int E, int k, int renorm, int32_t *ids, float *wts, uint32_t *status,
                     int stride, int n_shared, cudaStream_t s) {
    dim3 grid((T + ROUTE_WARPS - 1) / ROUTE_WARPS);
    return launch_pdl(route_topk_kernel<V>, grid, dim3(ROUTE_WARPS * 32), 0, s, logits, T, E, k, renorm, ids, wts,
                      status, stride, n_shared);
}

}  // namespace

// Rows of `stride` = k + n_shared slots: the k routed experts, then the
// n_shared shared experts (ids E, E + 1, ...) with weight 1 (k + n_shared <= 32).
cudaError_t launch_route_topk(const float *logits, int T, int E, int k, int renorm, int32_t *ids, float *wts,
                              uint32_t *status, cudaStream_t s, int n_shared) {
    if (T == 0) return cudaSuccess;
    const int st = k + n_shared;
    int v = (E + 31) / 32;
    if (v <= 1) return launch_v<1>(logits, T, E, k, renorm, ids, wts, status, st, n_shared, s);
    if (v <= 2) return launch_v<2>(logits, T, E, k, renorm, ids, wts, status, st, n_shared, s);
    if (v <= 4) return launch_v<4>(logits, T, E, k, renorm, ids, wts, status, st, n_shared, s);
    if (v <= 8) return launch_v<8>(logits, T, E, k, renorm, ids, wts, status, st, n_shared, s);
    if (v <= 16) return launch_v<16>(logits, T, E, k, renorm, ids, wts, status, st, n_shared, s);
    return launch_v<32>(logits, T, E, k, renorm, ids, wts, status, st, n_shared, s);
}

}  // namespace moe
