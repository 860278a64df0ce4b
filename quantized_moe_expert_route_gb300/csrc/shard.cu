// Expert sharding across GPUs: the fixed-order sum of the per-rank partial
// layer outputs.
//
// "多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出 120 t/s", section "8 张卡是怎么
// 配对的": within a pair of GPUs the routed experts are split 50/50 and the
// router is replicated, so each GPU evaluates the layer over its own experts
// (moe_ffn_forward with an expert range) and the partial outputs are summed.
// The sum here takes the parts in ascending rank order, one fp32 add at a
// time, so every rank obtains the same bits whatever the transport delivered
// first.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int SP_THREADS = 256;

__global__ void __launch_bounds__(SP_THREADS) sum_partials4_kernel(const float4 *__restrict__ parts, int n_parts,
                                                                  int64_t count4, float4 *__restrict__ out) {
    for (int64_t i = blockIdx.x * (int64_t)SP_THREADS + threadIdx.x; i < count4; i += (int64_t)gridDim.x * SP_THREADS) {
        float4 acc = parts[i];
        for (int p = 1; p < n_parts; ++p) {
            const float4 v = parts[(int64_t)p * count4 + i];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        out[i] = acc;
    }
}

__global__ void __launch_bounds__(SP_THREADS) sum_partials_kernel(const float *__restrict__ parts, int n_parts,
                                                                 int64_t count, float *__restrict__ out) {
    for (int64_t i = blockIdx.x * (int64_t)SP_THREADS + threadIdx.x; i < count; i += (int64_t)gridDim.x * SP_THREADS) {
        float acc = parts[i];
        for (int p = 1; p < n_parts; ++p) acc += parts[(int64_t)p * count + i];
        out[i] = acc;
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_sum_partials(const float *parts, int32_t n_parts, int64_t count, float *out, moe_stream_t stream) {
    if (n_parts <= 0 || count < 0) return MOE_ERR_INVALID_ARG;
    if (count == 0) return MOE_OK;
    if (!parts || !out) return MOE_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return MOE_ERR_CUDA;
    const bool vec = count % 4 == 0 && (reinterpret_cast<uintptr_t>(parts) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    const int64_t n = vec ? count / 4 : count;
    const int64_t blocks = std::min<int64_t>((n + SP_THREADS - 1) / SP_THREADS, (int64_t)sms * 8);
    if (vec)
        sum_partials4_kernel<<<(unsigned)blocks, SP_THREADS, 0, stream>>>(reinterpret_cast<const float4 *>(parts),
                                                                          n_parts, n, reinterpret_cast<float4 *>(out));
    else
        sum_partials_kernel<<<(unsigned)blocks, SP_THREADS, 0, stream>>>(parts, n_parts, n, out);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
