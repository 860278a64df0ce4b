// moe_ffn_forward_noalloc: the whole layer without a caller-supplied
// workspace, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a host framework
// whose own memory planner owns all device memory and forbids raw
// allocations, latency-critical loops where cudaMalloc/cudaFree would
// implicitly synchronise the device, and small C clients that only receive
// input and output pointers from another runtime and have no allocator to size
// a workspace with. This entry point keeps the layer's scratch (routing
// arrays, the SwiGLU intermediate and the per-pair down outputs) in a
// file-scope device array of fixed size instead. The source pages have no
// counterpart of this entry point; it is a property of this library only.
#include "moe_internal.cuh"

namespace {

// The scratch: every GPU that loads this library holds these bytes until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void *g_scratch_ptr[MAX_DEVICES] = {};

// Device address of the scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return (int)err;
    if (dev < 0 || dev >= MAX_DEVICES) return (int)cudaErrorInvalidDevice;
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return (int)err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return 0;
}

}  // namespace

extern "C" int moe_ffn_forward_noalloc(const moe_weight_table *W, const uint16_t *x, const float *logits,
                                       int32_t T, int32_t k, const moe_options *opt, float *out,
                                       moe_stream_t stream) {
    if (!W) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_ffn_workspace_size(W, T, k);
    if (need == 0) return MOE_ERR_INVALID_ARG;
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != 0) return MOE_ERR_CUDA;
    // The array starts zeroed (a static device array). Each call clears the
    // status word (offset 0); the fused kernel's grid-barrier counter (offset
    // 8) only grows, its generation is count / gridDim. Every other region is
    // written before it is read.
    if (cudaMemsetAsync(scratch, 0, 8, stream) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_ffn_forward(W, x, logits, T, k, opt, out, scratch, MOE_NOALLOC_SCRATCH_BYTES, stream);
}
