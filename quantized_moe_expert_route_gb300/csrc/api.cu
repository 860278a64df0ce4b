// C ABI of the library: argument validation, workspace layout, launches.
// Every step of the layer runs in this library's kernels; nothing here
// computes on the host beyond checking arguments.
#include <cstring>
#include <vector>

#include "moe_internal.cuh"

namespace moe {
cudaError_t launch_route_topk(const float *logits, int T, int E, int k, int renorm, int32_t *ids, float *wts,
                              uint32_t *status, cudaStream_t s, int n_shared = 0);
cudaError_t launch_bucket(const int32_t *ids, int T, int k, int E, int lo, int hi, uint32_t fmt_mask,
                          const DevExpert *table, int32_t *offsets, int32_t *pairs, int32_t *pos, int32_t *active,
                          uint32_t *status, int32_t *scratch, cudaStream_t s);
size_t bucket_smem_bytes(int E);
size_t gateup_smem_bytes(int H, int64_t wstride);
size_t down_smem_bytes(int I, int64_t wstride);
cudaError_t launch_gemv_path(const DevExpert *table, int T, int k, int E, int H, int I, int64_t gu_stride,
                             int64_t dn_stride, uint32_t gu_formats, uint32_t down_formats, const uint32_t *grid,
                             const int32_t *offsets, const int32_t *pairs, const int32_t *active, const int32_t *pos,
                             const float *wts, const uint16_t *x, float *h, float *y, float *out, uint32_t *status,
                             cudaEvent_t const *events, cudaStream_t s);
bool decode_fused_eligible(int T, int k, int E, int H, int I, uint32_t gateup_formats, uint32_t down_formats,
                           int64_t gu_stride, int64_t dn_stride);
cudaError_t launch_decode_fused(const DevExpert *table, const moe_weight_table *W, int T, int k, int E, int H, int I,
                                int64_t gu_stride, int64_t dn_stride, int renorm, int lo, int hi, uint32_t fmt_mask, const float *logits,
                                const uint16_t *x, float *out, float *h, int32_t *ids, float *wts, int32_t *offsets,
                                int32_t *active, int32_t *pairs, int32_t *pos, unsigned char *sync, uint32_t *status,
                                cudaStream_t s);
bool tc_path_eligible(int H, int I);
size_t tc_weight_map_bytes(int E);
bool tc_encode_weight_maps(const moe_weight_table *W, void *out);
cudaError_t launch_tc_path(const DevExpert *table, const void *wmaps, uint32_t gu_formats, uint32_t dn_formats,
                           const uint32_t *grid, int T, int k, int E,
                           int H, int I, const int32_t *offsets, const int32_t *active, const int32_t *pos,
                           const float *wts, const uint16_t *x, float *h32, float *y, char *ws_base,
                           const TcLayout &C, float *out, uint32_t *status, cudaEvent_t const *events,
                           cudaStream_t s);
int noalloc_scratch_address(void **out);
cudaError_t set_wait_ns_stream(unsigned long long ns);
cudaError_t set_wait_ns_gemv(unsigned long long ns);
cudaError_t set_wait_ns_decode(unsigned long long ns);
cudaError_t set_wait_ns_tc(unsigned long long ns);
}  // namespace moe

using namespace moe;

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return MOE_ERR_CUDA;
}

constexpr size_t SMEM_LIMIT = 227 * 1024 - 1024;   // opt-in limit less the kernels' static shared memory
constexpr int MAX_T = 65535;

cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(s, &cs);
    if (err != cudaSuccess) return err;
    return cudaEventRecordWithFlags(ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0);
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Offset of the tensor path's weight maps in the prepared device table, and
// of the per-expert cold flags after them.
size_t map_offset(int E) { return align_up((size_t)E * sizeof(DevExpert), 128); }
size_t cold_offset(int E) { return align_up(map_offset(E) + tc_weight_map_bytes(E), 256); }

// Where a matrix's bytes live: 1 device memory, 0 host memory the GPU can read
// (pinned or registered; the cold tier), -1 neither. *dptr: the device-side
// address.
int locate(const void *p, const void **dptr) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *dptr = p;
        return 1;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer) {
        *dptr = a.devicePointer;
        return 0;
    }
    return -1;
}

int check_matrix(const moe_matrix &m, int rows, int cols) {
    if (m.format < MOE_Q8_0 || m.format > MOE_T5_G128) return MOE_ERR_BAD_FORMAT;
    if (m.rows != rows || m.cols != cols) return MOE_ERR_BAD_SHAPE;
    const int be = BLOCK_ELEMS[m.format], bb = BLOCK_BYTES[m.format];
    if (cols % be != 0) return MOE_ERR_BAD_SHAPE;
    const int64_t row_bytes = (int64_t)(cols / be) * bb;
    if (m.row_stride_bytes < row_bytes || m.row_stride_bytes % 16 != 0) return MOE_ERR_BAD_SHAPE;
    if (!m.data || !aligned(m.data, 16)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Resolve the path of a forward; -1 if the requested path cannot run it.
// Shared experts ride along as entries E .. E + n_shared - 1 of the table and
// as slots k .. k + n_shared - 1 of every token (weight 1): the kernels after
// the router see k + n_shared slots over E + n_shared experts.
int n_all(const moe_weight_table *W) { return W->n_experts + W->n_shared; }
int k_all(const moe_weight_table *W, int k) { return k + W->n_shared; }

int resolve_path(const moe_weight_table *W, int T, int k, int requested) {
    // a table with cold (host-resident) experts runs on the grouped GEMV
    // kernels, which read the routed cold experts from their staged copy; the
    // fused kernel routes in-kernel and has no shared-expert slots
    const bool hot_only = W->n_cold == 0;
    const int kk = k_all(W, k), EE = n_all(W);
    const bool fused_ok = hot_only && W->n_shared == 0 &&
                          decode_fused_eligible(T, k, W->n_experts, W->hidden, W->inter, W->gateup_formats,
                                                W->down_formats, W->max_gateup_stride, W->max_down_stride);
    const bool tc_ok = hot_only && W->tc_maps == 1 && tc_path_eligible(W->hidden, W->inter);
    const bool stream_ok = stream_plan(T, kk, EE, W->hidden, W->inter, W->gateup_formats, W->down_formats,
                                       W->max_gateup_stride, W->max_down_stride).ok;
    switch (requested) {
        case MOE_PATH_AUTO:
            // measured on GB300 per layer: the fused kernel where it applies;
            // else the streaming GEMV kernels for decode batches (16-row
            // decode 144 us vs 225 us on the tensor path, 6-row mixed tiers
            // 123 vs 151); else the tensor path (2048-row prefill 1.2 ms vs
            // 74 ms with the tiled GEMV kernels); else GEMV
            return fused_ok ? MOE_PATH_FUSED : stream_ok ? MOE_PATH_GEMV : tc_ok ? MOE_PATH_TENSOR : MOE_PATH_GEMV;
        case MOE_PATH_GEMV: return MOE_PATH_GEMV;
        case MOE_PATH_TENSOR: return tc_ok ? MOE_PATH_TENSOR : -1;
        case MOE_PATH_FUSED: return fused_ok ? MOE_PATH_FUSED : -1;
        default: return -1;
    }
}

// Workspace bytes of a forward on `path` (the tensor path adds its regions).
size_t path_ws_bytes(const moe_weight_table *W, int T, int k, int path) {
    const int kk = k_all(W, k), EE = n_all(W);
    if (path == MOE_PATH_TENSOR) return tc_ws_layout(T, kk, EE, W->hidden, W->inter).total;
    const size_t base = ws_layout(T, kk, EE, W->hidden, W->inter).total;
    if (W->prepared == MOE_TABLE_PREPARED && W->n_cold > 0)
        return cold_ws_layout(base, T, kk, EE, W->n_cold, W->cold_bytes_max).total;
    return base;
}

// Options with defaults filled in; false if they are invalid.
bool effective_options(const moe_weight_table *W, const moe_options *opt, moe_options &o) {
    o = moe_options{sizeof(moe_options), 1, 0xffffffffu, 0, n_all(W), MOE_PATH_AUTO, 0, nullptr};
    if (!opt) return true;
    if (opt->struct_size != sizeof(moe_options)) return false;
    o = *opt;
    if (o.expert_lo < 0 || o.expert_hi > n_all(W) || o.expert_lo > o.expert_hi) return false;
    if (o.path < MOE_PATH_AUTO || o.path > MOE_PATH_FUSED) return false;
    return true;
}

}  // namespace

extern "C" {

const char *moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_BAD_SHAPE: return "bad shape";
        case MOE_ERR_BAD_FORMAT: return "bad format";
        case MOE_ERR_BAD_ID: return "bad expert id";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_NOT_PREPARED: return "weight table not prepared";
        case MOE_ERR_UNSUPPORTED: return "unsupported size";
        default: return "unknown status";
    }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

size_t moe_table_device_bytes(int32_t n_experts) {
    if (n_experts <= 0 || n_experts > MOE_MAX_EXPERTS) return 0;
    return align_up(cold_offset(n_experts) + (size_t)n_experts, 256);
}

int moe_table_prepare(moe_weight_table *W, void *device_buf, size_t device_bytes, moe_stream_t stream) {
    if (!W || !W->experts || !device_buf) return MOE_ERR_INVALID_ARG;
    W->prepared = 0;
    if (W->n_shared < 0 || W->n_shared > MOE_MAX_SHARED || W->n_experts <= 0) return MOE_ERR_INVALID_ARG;
    const int E = W->n_experts + W->n_shared, H = W->hidden, I = W->inter;   // every table entry
    if (E <= 0 || E > MOE_MAX_EXPERTS || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (H > MOE_MAX_HIDDEN || I > MOE_MAX_INTER) return MOE_ERR_UNSUPPORTED;
    if (device_bytes < moe_table_device_bytes(E) || !aligned(device_buf, 16)) return MOE_ERR_INVALID_ARG;
    std::vector<DevExpert> dev(E);
    std::vector<uint8_t> cold(E, 0);
    uint32_t present = 0, gu_present = 0, dn_present = 0;
    int64_t gu_max = 0, dn_max = 0, cold_max = 0;
    int n_cold = 0;
    for (int e = 0; e < E; ++e) {
        const moe_expert &x = W->experts[e];
        int rc;
        if ((rc = check_matrix(x.gate, I, H)) != MOE_OK) return rc;
        if ((rc = check_matrix(x.up, I, H)) != MOE_OK) return rc;
        if ((rc = check_matrix(x.down, H, I)) != MOE_OK) return rc;
        if (x.gate.format != x.up.format) return MOE_ERR_BAD_FORMAT;
        present |= 1u << x.gate.format;
        present |= 1u << x.down.format;
        gu_present |= 1u << x.gate.format;
        dn_present |= 1u << x.down.format;
        gu_max = std::max<int64_t>(gu_max, std::max(x.gate.row_stride_bytes, x.up.row_stride_bytes));
        dn_max = std::max<int64_t>(dn_max, x.down.row_stride_bytes);
        const moe_matrix *src[3] = {&x.gate, &x.up, &x.down};
        DevMatrix *dst[3] = {&dev[e].gate, &dev[e].up, &dev[e].down};
        int where[3];
        for (int i = 0; i < 3; ++i) {
            const void *dp = nullptr;
            where[i] = locate(src[i]->data, &dp);
            if (where[i] < 0) return MOE_ERR_INVALID_ARG;
            dst[i]->data = static_cast<const uint8_t *>(dp);
            dst[i]->stride = src[i]->row_stride_bytes;
            dst[i]->fmt = src[i]->format;
            dst[i]->rows = src[i]->rows;
        }
        // a cold expert keeps all three matrices in host memory
        if (where[0] != where[1] || where[0] != where[2]) return MOE_ERR_INVALID_ARG;
        if (where[0] == 0) {
            cold[e] = 1;
            ++n_cold;
            int64_t b = 0;
            for (int i = 0; i < 3; ++i) b += (int64_t)align_up((size_t)src[i]->rows * src[i]->row_stride_bytes, 256);
            cold_max = std::max(cold_max, b);
        }
    }
    if (gateup_smem_bytes(H, gu_max) > SMEM_LIMIT || down_smem_bytes(I, dn_max) > SMEM_LIMIT)
        return MOE_ERR_UNSUPPORTED;
    // IQ3_XXS weights are read through the caller's 256-entry grid
    if ((present & (1u << MOE_IQ3_XXS)) && (!W->iq3_grid || !aligned(W->iq3_grid, 16))) return MOE_ERR_INVALID_ARG;
    cudaError_t err = cudaMemcpyAsync(device_buf, dev.data(), (size_t)E * sizeof(DevExpert), cudaMemcpyHostToDevice,
                                      stream);
    if (err != cudaSuccess) return cuda_fail(err);
    err = cudaMemcpyAsync(static_cast<char *>(device_buf) + cold_offset(E), cold.data(), (size_t)E,
                          cudaMemcpyHostToDevice, stream);
    if (err != cudaSuccess) return cuda_fail(err);
    // the tensor path's TMA descriptors of every weight matrix
    std::vector<unsigned char> maps;
    W->tc_maps = 0;
    if (tc_path_eligible(H, I)) {
        maps.resize(tc_weight_map_bytes(E));
        if (tc_encode_weight_maps(W, maps.data())) {
            err = cudaMemcpyAsync(static_cast<char *>(device_buf) + map_offset(E), maps.data(), maps.size(),
                                  cudaMemcpyHostToDevice, stream);
            if (err != cudaSuccess) return cuda_fail(err);
            W->tc_maps = 1;
        }
    }
    err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err);
    // uniform layout: experts at a constant step with identical formats and strides
    int uniform = 1;
    int64_t step[3] = {0, 0, 0};
    if (E > 1) {
        const moe_matrix *m0[3] = {&W->experts[0].gate, &W->experts[0].up, &W->experts[0].down};
        const moe_matrix *m1[3] = {&W->experts[1].gate, &W->experts[1].up, &W->experts[1].down};
        for (int i = 0; i < 3; ++i)
            step[i] = (int64_t)((const char *)m1[i]->data - (const char *)m0[i]->data);
        for (int e = 0; e < E && uniform; ++e) {
            const moe_matrix *me[3] = {&W->experts[e].gate, &W->experts[e].up, &W->experts[e].down};
            for (int i = 0; i < 3; ++i) {
                if (me[i]->format != m0[i]->format || me[i]->row_stride_bytes != m0[i]->row_stride_bytes ||
                    (const char *)me[i]->data != (const char *)m0[i]->data + step[i] * e)
                    uniform = 0;
            }
        }
    }
    W->uniform_layout = uniform;
    W->uniform_base = W->experts[0];
    for (int i = 0; i < 3; ++i) W->uniform_step[i] = step[i];
    W->device_table = device_buf;
    W->formats_present = present;
    W->gateup_formats = gu_present;
    W->down_formats = dn_present;
    W->max_gateup_stride = gu_max;
    W->max_down_stride = dn_max;
    W->n_cold = n_cold;
    W->cold_bytes_max = cold_max;
    W->prepared = MOE_TABLE_PREPARED;
    return MOE_OK;
}

int moe_route_topk(const float *logits, int32_t T, int32_t E, int32_t k, int32_t renormalize, int32_t *ids,
                   float *weights, uint32_t *status, moe_stream_t stream) {
    if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS || k > MOE_MAX_K) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!logits || !ids || !weights)) return MOE_ERR_INVALID_ARG;
    cudaError_t err = launch_route_topk(logits, T, E, k, renormalize, ids, weights, status, stream);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

int moe_bucket(const int32_t *ids, int32_t T, int32_t k, int32_t E, int32_t expert_lo, int32_t expert_hi,
               int32_t *offsets, int32_t *pairs, int32_t *pos, int32_t *active, uint32_t *status,
               moe_stream_t stream) {
    if (T < 0 || k <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS || k > MOE_MAX_K || (int64_t)T * k > (1 << 24)) return MOE_ERR_UNSUPPORTED;
    if (!offsets || !active || (T > 0 && (!ids || !pairs || !pos))) return MOE_ERR_INVALID_ARG;
    cudaError_t err = launch_bucket(ids, T, k, E, expert_lo, expert_hi, 0xffffffffu, nullptr, offsets, pairs, pos,
                                    active, status, nullptr, stream);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

size_t moe_ffn_workspace_size(const moe_weight_table *W, int32_t T, int32_t k) {
    return moe_ffn_workspace_size_for_path(W, T, k, MOE_PATH_AUTO);
}

size_t moe_ffn_workspace_size_for_path(const moe_weight_table *W, int32_t T, int32_t k, int32_t path) {
    if (!W || T < 0 || k <= 0 || k > W->n_experts || W->n_experts <= 0) return 0;
    if (path < MOE_PATH_AUTO || path > MOE_PATH_FUSED) return 0;
    const int p = W->prepared == MOE_TABLE_PREPARED ? resolve_path(W, T > 0 ? T : 1, k, path)
                                                    : (path == MOE_PATH_AUTO ? MOE_PATH_GEMV : path);
    if (p < 0) return 0;
    return path_ws_bytes(W, T, k, p);
}

int moe_ffn_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ws || ws_bytes < SYNC_BYTES) return MOE_ERR_INVALID_ARG;
    cudaError_t err = cudaMemsetAsync(ws, 0, ws_bytes, stream);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

int moe_ffn_forward(const moe_weight_table *W, const uint16_t *x, const float *logits, int32_t T, int32_t k,
                    const moe_options *opt, float *out, void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!W) return MOE_ERR_INVALID_ARG;
    if (W->prepared != MOE_TABLE_PREPARED || !W->device_table) return MOE_ERR_NOT_PREPARED;
    const int ER = W->n_experts, H = W->hidden, I = W->inter;
    if (T < 0 || k <= 0 || k > ER) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_K || k + W->n_shared > MOE_MAX_K || T > MAX_T) return MOE_ERR_UNSUPPORTED;
    // after the router: k + n_shared slots per token over E + n_shared experts
    const int E = n_all(W), kr = k;
    k = k_all(W, k);
    if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !logits || !out)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!aligned(out, 16))) return MOE_ERR_INVALID_ARG;
    moe_options o;
    if (!effective_options(W, opt, o)) return MOE_ERR_INVALID_ARG;
    int path = resolve_path(W, T > 0 ? T : 1, kr, o.path);
    // the fused and tensor paths read activation rows with 16-byte loads
    if ((path == MOE_PATH_FUSED || path == MOE_PATH_TENSOR) && T > 0 && !aligned(x, 16))
        path = o.path == MOE_PATH_AUTO ? MOE_PATH_GEMV : -1;
    if (path < 0) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(T, k, E, H, I);
    if (ws_bytes < path_ws_bytes(W, T, kr, path)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (T == 0) return MOE_OK;

    char *base = static_cast<char *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(base + L.status);
    int32_t *ids = reinterpret_cast<int32_t *>(base + L.ids);
    float *wts = reinterpret_cast<float *>(base + L.wts);
    int32_t *offsets = reinterpret_cast<int32_t *>(base + L.offsets);
    int32_t *active = reinterpret_cast<int32_t *>(base + L.active);
    int32_t *pairs = reinterpret_cast<int32_t *>(base + L.pairs);
    int32_t *pos = reinterpret_cast<int32_t *>(base + L.pos);
    float *h = reinterpret_cast<float *>(base + L.h);
    float *y = reinterpret_cast<float *>(base + L.y);
    const DevExpert *table = static_cast<const DevExpert *>(W->device_table);

    cudaEvent_t const *events = reinterpret_cast<cudaEvent_t const *>(o.timing_events);
    cudaError_t err;
    if (path == MOE_PATH_FUSED) {
        if (events && (err = record_timing_event(events[0], stream)) != cudaSuccess) return cuda_fail(err);
        err = launch_decode_fused(table, W, T, kr, ER, H, I, W->max_gateup_stride, W->max_down_stride, o.renormalize,
                                  o.expert_lo, o.expert_hi, o.format_mask, logits,
                                  x, out, h, ids, wts, offsets, active, pairs, pos,
                                  reinterpret_cast<unsigned char *>(base + L.status), status, stream);
        if (err != cudaSuccess) return cuda_fail(err);
        if (events) {
            if ((err = record_timing_event(events[1], stream)) != cudaSuccess) return cuda_fail(err);
            if ((err = record_timing_event(events[2], stream)) != cudaSuccess) return cuda_fail(err);
        }
        return MOE_OK;
    }
    err = launch_route_topk(logits, T, ER, kr, o.renormalize, ids, wts, status, stream, W->n_shared);
    if (err != cudaSuccess) return cuda_fail(err);
    err = launch_bucket(ids, T, k, E, o.expert_lo, o.expert_hi, o.format_mask, table, offsets, pairs, pos, active,
                        status, reinterpret_cast<int32_t *>(base + L.bscratch), stream);
    if (err != cudaSuccess) return cuda_fail(err);
    if (path == MOE_PATH_TENSOR)
        err = launch_tc_path(table, static_cast<const char *>(W->device_table) + map_offset(E), W->gateup_formats,
                             W->down_formats, static_cast<const uint32_t *>(W->iq3_grid), T, k, E, H, I, offsets,
                             active, pos, wts, x,
                             h, y, base, tc_ws_layout(T, k, E, H, I), out, status, events, stream);
    else {
        if (W->n_cold > 0) {
            // the routed cold experts' bytes into the workspace, read through a remapped table
            const ColdLayout CL = cold_ws_layout(L.total, T, k, E, W->n_cold, W->cold_bytes_max);
            err = launch_cold_staging(table, static_cast<const uint8_t *>(W->device_table) + cold_offset(E), E,
                                      active, base, CL, stream);
            if (err != cudaSuccess) return cuda_fail(err);
            table = reinterpret_cast<const DevExpert *>(base + CL.remap);
        }
        err = launch_gemv_path(table, T, k, E, H, I, W->max_gateup_stride, W->max_down_stride, W->gateup_formats,
                               W->down_formats, static_cast<const uint32_t *>(W->iq3_grid), offsets, pairs, active,
                               pos, wts, x, h, y, out, status, events, stream);
    }
    if (err != cudaSuccess) return cuda_fail(err);
    return MOE_OK;
}

int moe_ffn_gemv_kernels(const moe_weight_table *W, int32_t T, int32_t k) {
    if (!W || W->prepared != MOE_TABLE_PREPARED || T < 0 || k <= 0 || k > W->n_experts) return -1;
    return stream_plan(T > 0 ? T : 1, k_all(W, k), n_all(W), W->hidden, W->inter, W->gateup_formats, W->down_formats,
                       W->max_gateup_stride,
                       W->max_down_stride).ok
               ? MOE_GEMV_STREAMING
               : MOE_GEMV_TILED;
}

int moe_ffn_path(const moe_weight_table *W, int32_t T, int32_t k, const moe_options *opt) {
    if (!W || W->prepared != MOE_TABLE_PREPARED || T < 0 || k <= 0 || k > W->n_experts) return -1;
    moe_options o;
    if (!effective_options(W, opt, o)) return -1;
    return resolve_path(W, T > 0 ? T : 1, k, o.path);
}

int moe_ffn_workspace_views(const moe_weight_table *W, int32_t T, int32_t k, void *ws, int32_t **ids,
                            float **weights, int32_t **offsets, int32_t **active, int32_t **pairs,
                            int32_t **pos) {
    if (!W || !ws || T < 0 || k <= 0 || W->n_experts <= 0 || k > W->n_experts) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, k_all(W, k), n_all(W), W->hidden, W->inter);
    char *b = static_cast<char *>(ws);
    if (ids) *ids = reinterpret_cast<int32_t *>(b + L.ids);
    if (weights) *weights = reinterpret_cast<float *>(b + L.wts);
    if (offsets) *offsets = reinterpret_cast<int32_t *>(b + L.offsets);
    if (active) *active = reinterpret_cast<int32_t *>(b + L.active);
    if (pairs) *pairs = reinterpret_cast<int32_t *>(b + L.pairs);
    if (pos) *pos = reinterpret_cast<int32_t *>(b + L.pos);
    return MOE_OK;
}

int moe_ffn_read_status(void *ws, uint32_t *status_out, moe_stream_t stream) {
    if (!status_out) return MOE_ERR_INVALID_ARG;
    if (!ws && noalloc_scratch_address(&ws) != 0) return MOE_ERR_CUDA;   // the noalloc entry point's array
    cudaError_t err = cudaMemcpyAsync(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
    if (err != cudaSuccess) return cuda_fail(err);
    err = cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream);
    if (err != cudaSuccess) return cuda_fail(err);
    err = cudaStreamSynchronize(stream);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

int moe_set_wait_timeout_ns(uint64_t ns) {
    const unsigned long long v = ns ? (unsigned long long)ns : DEFAULT_WAIT_NS;
    cudaError_t err;
    if ((err = set_wait_ns_stream(v)) != cudaSuccess || (err = set_wait_ns_gemv(v)) != cudaSuccess ||
        (err = set_wait_ns_decode(v)) != cudaSuccess || (err = set_wait_ns_tc(v)) != cudaSuccess)
        return cuda_fail(err);
    return MOE_OK;
}

}  // extern "C"
