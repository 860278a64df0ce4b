// The cold-expert tier: experts whose weights stay in host memory (on GB300,
// the Grace CPU's LPDDR, which the GPU reads coherently over NVLink-C2C).
//
// "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南", section
// 优化策略一 (专家使用频率排序, 热/冷分离): the experts are ranked by how often the
// router picks them, the hot ones are kept in GPU memory and the coldest in
// host RAM. There the CPU computes the cold experts; here the GPU does: once
// a layer's routing is known, the routed cold experts' bytes are pulled over
// the chip-to-chip link into a staging area of the workspace by a copy kernel
// on every SM (plain 16-byte loads from host memory), and the layer's kernels
// then read a copy of the descriptor table whose routed cold entries point at
// the staged bytes. Unrouted cold experts cost nothing.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int CP_THREADS = 256;

__device__ __forceinline__ uint64_t matrix_bytes(const DevMatrix &m) { return align_up((uint64_t)m.rows * m.stride, 256); }

// One CTA: the remapped table (a copy of all E descriptors with every routed
// cold expert's matrices redirected into `staging`, in active-list order) and
// the copy segments {src, dst, bytes}, three per routed cold expert.
__global__ void __launch_bounds__(CP_THREADS) cold_plan_kernel(const DevExpert *__restrict__ table,
                                                              const uint8_t *__restrict__ cold, int E,
                                                              const int32_t *__restrict__ active, DevExpert *remap,
                                                              ColdSeg *segs, int32_t *n_segs, uint8_t *staging) {
    __shared__ uint64_t scan[CP_THREADS];
    __shared__ int cnt[CP_THREADS];
    for (int e = threadIdx.x; e < E; e += CP_THREADS) remap[e] = table[e];
    __syncthreads();
    const int n_act = active[0];
    uint64_t base = 0;
    int nseg = 0;
    for (int c0 = 0; c0 < n_act; c0 += CP_THREADS) {
        const int i = c0 + threadIdx.x;
        const int e = i < n_act ? active[1 + i] : -1;
        const bool is_cold = e >= 0 && cold[e];
        uint64_t bytes = 0;
        if (is_cold) bytes = matrix_bytes(table[e].gate) + matrix_bytes(table[e].up) + matrix_bytes(table[e].down);
        scan[threadIdx.x] = bytes;
        cnt[threadIdx.x] = is_cold ? 1 : 0;
        __syncthreads();
        for (int o = 1; o < CP_THREADS; o <<= 1) {
            const uint64_t v = threadIdx.x >= o ? scan[threadIdx.x - o] : 0;
            const int c = threadIdx.x >= o ? cnt[threadIdx.x - o] : 0;
            __syncthreads();
            scan[threadIdx.x] += v;
            cnt[threadIdx.x] += c;
            __syncthreads();
        }
        if (is_cold) {
            uint64_t off = base + scan[threadIdx.x] - bytes;
            const int s = 3 * (nseg + cnt[threadIdx.x] - 1);
            const DevMatrix *src[3] = {&table[e].gate, &table[e].up, &table[e].down};
            DevMatrix *dst[3] = {&remap[e].gate, &remap[e].up, &remap[e].down};
            for (int m = 0; m < 3; ++m) {
                const uint64_t mb = (uint64_t)src[m]->rows * src[m]->stride;
                segs[s + m] = ColdSeg{src[m]->data, staging + off, mb};
                dst[m]->data = staging + off;
                off += matrix_bytes(*src[m]);
            }
        }
        base += scan[CP_THREADS - 1];
        nseg += cnt[CP_THREADS - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) *n_segs = 3 * nseg;
}

// Every SM: the segments' bytes from host memory into the staging area, 16
// bytes per load (the rows and strides are multiples of 16 bytes).
__global__ void __launch_bounds__(CP_THREADS) cold_copy_kernel(const ColdSeg *__restrict__ segs,
                                                              const int32_t *__restrict__ n_segs) {
    const int n = *n_segs;
    const size_t tid = (size_t)blockIdx.x * CP_THREADS + threadIdx.x, nth = (size_t)gridDim.x * CP_THREADS;
    for (int s = 0; s < n; ++s) {
        const ColdSeg g = segs[s];
        const uint4 *src = reinterpret_cast<const uint4 *>(g.src);
        uint4 *dst = reinterpret_cast<uint4 *>(g.dst);
        const size_t n16 = g.bytes / 16;
        for (size_t i = tid; i < n16; i += nth) dst[i] = src[i];
    }
}

}  // namespace

cudaError_t launch_cold_staging(const DevExpert *table, const uint8_t *cold, int E, const int32_t *active,
                                char *ws_base, const ColdLayout &C, cudaStream_t s) {
    DevExpert *remap = reinterpret_cast<DevExpert *>(ws_base + C.remap);
    ColdSeg *segs = reinterpret_cast<ColdSeg *>(ws_base + C.segs);
    int32_t *n_segs = reinterpret_cast<int32_t *>(ws_base + C.n_segs);
    cold_plan_kernel<<<1, CP_THREADS, 0, s>>>(table, cold, E, active, remap, segs, n_segs,
                                               reinterpret_cast<uint8_t *>(ws_base + C.staging));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int G = sm_count();
    if (G <= 0) return cudaErrorInvalidConfiguration;
    cold_copy_kernel<<<4 * G, CP_THREADS, 0, s>>>(segs, n_segs);
    return cudaGetLastError();
}

}  // namespace moe
