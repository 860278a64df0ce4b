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
#include <atomic>

#include "moe_internal.cuh"

namespace {

// The scratch: every GPU that loads this library holds these bytes until the
// process exits. A static device array starts zeroed.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::atomic<void *> g_scratch_ptr[MAX_DEVICES];

}  // namespace

namespace moe {

// Device address of the scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current (threads that race on the first lookup
// store the same value).
int noalloc_scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return (int)err;
    if (dev < 0 || dev >= MAX_DEVICES) return (int)cudaErrorInvalidDevice;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return (int)err;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return 0;
}

}  // namespace moe

extern "C" int moe_ffn_forward_noalloc(const moe_weight_table *W, const uint16_t *x, const float *logits,
                                       int32_t T, int32_t k, const moe_options *opt, float *out,
                                       moe_stream_t stream) {
    if (!W) return MOE_ERR_INVALID_ARG;
    if (opt && opt->struct_size != sizeof(moe_options)) return MOE_ERR_INVALID_ARG;
    // sized for the path the forward will take (a requested tensor path needs
    // more than AUTO's); 0 means invalid arguments or a path that cannot run
    // the layer, which moe_ffn_forward rejects before enqueuing anything
    const size_t need = moe_ffn_workspace_size_for_path(W, T, k, opt ? opt->path : MOE_PATH_AUTO);
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (moe::noalloc_scratch_address(&scratch) != 0) return MOE_ERR_CUDA;
    // Offset 0 holds the device status flags (sticky until read with
    // moe_ffn_read_status(NULL, ...)); offset 8 the fused kernel's grid-barrier
    // counter, which only grows (its generation is count / gridDim, the same
    // grid on every launch). Every other region is written before it is read.
    return moe_ffn_forward(W, x, logits, T, k, opt, out, scratch, MOE_NOALLOC_SCRATCH_BYTES, stream);
}
