/*
 * moe_route.h -- C ABI of the GB300 (sm_103a) routed mixture-of-experts FFN
 * layer over block-quantized expert weights.
 *
 * The layer (per token t, with x_t in bf16 and router logits in fp32):
 *
 *     ids[t, 0..k-1], w[t, 0..k-1] = top-k of softmax(logits[t])
 *     out[t] = sum_{j = 0..k-1} w[t, j] * W_down[e] ( silu(W_gate[e] x_t) * (W_up[e] x_t) ),
 *     e = ids[t, j],  silu(z) = z / (1 + exp(-z)),  sum in ascending slot j.
 *
 * Source: "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南":
 * section 瓶颈分析 (a light router picks 10 of a layer's 512 experts per token),
 * section 优化策略二 (per-expert precision tiers: Q6_K gate/up with Q8_0 down,
 * a middle tier, MXFP4 for the tail; down has K = 640, so only 32-weight
 * block formats fit it), section 优化策略三 (one mul_mat_id drives experts of
 * several formats in one layer; an expert-id range filter [min, max) skips
 * the others) and section 关键 Bug 修复与调试踩坑记录 (-1 is a "skip" id that must
 * stay signed; gate/up/activation are fused in decode). The grouped
 * multi-session decode (one launch serves the decode rows of 16 sessions) is
 * from "多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出 120 t/s", section
 * "120 t/s 的秘密：微批次分组解码".
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must be device memory of the current CUDA
 *     device; "host" pointers are ordinary host memory.
 *   - The caller owns every buffer. The library allocates no device memory.
 *   - Work is enqueued asynchronously on `stream` (NULL = the legacy default
 *     stream); no entry point synchronises the host except
 *     moe_table_prepare and moe_ffn_read_status, which say so.
 *   - Every entry point returns an moe_status code; no C++ exception crosses
 *     the ABI. Argument errors are detected on the host before anything is
 *     enqueued. Errors the GPU finds in the data (bad ids, non-finite logits)
 *     are OR-ed into a device status word; see moe_device_flags.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

/* Return codes. */
typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null pointer, bad count, misaligned pointer */
    MOE_ERR_BAD_SHAPE = 2,           /* dims disagree, cols not a multiple of the block, bad stride */
    MOE_ERR_BAD_FORMAT = 3,          /* unknown format tag, gate/up formats differ */
    MOE_ERR_BAD_ID = 4,              /* reserved for host-checked ids */
    MOE_ERR_WORKSPACE_TOO_SMALL = 5, /* ws_bytes below the size query */
    MOE_ERR_CUDA = 6,                /* a CUDA call failed; see moe_last_cuda_error */
    MOE_ERR_NOT_PREPARED = 7,        /* weight table was not (successfully) prepared */
    MOE_ERR_UNSUPPORTED = 8          /* valid, but beyond this build's limits (MOE_MAX_*) */
} moe_status;

/* Device status flags (OR-ed, sticky until read). */
typedef enum {
    MOE_FLAG_NONFINITE_LOGIT = 1,    /* a logit was NaN or +-inf (ranked last, weight 0) */
    MOE_FLAG_BAD_ID = 2,             /* an id outside [-1, E) (the pair was skipped) */
    MOE_FLAG_DUPLICATE_ID = 4,       /* an expert repeated within one token (still computed) */
    MOE_FLAG_WAIT_TIMEOUT = 8        /* a bounded device wait gave up (the tile was skipped) */
} moe_device_flags;

/* Weight block formats (little-endian; fp16 = IEEE binary16).
 *  Q8_0    : 34 B / 32 weights : fp16 d, int8 q[32];                 w = d*q
 *  Q4_K    : 144 B / 256       : fp16 d, fp16 dmin, 12 B packed 6-bit
 *                                (scale, min) x 8, 128 B 4-bit codes; w = d*sc*q - dmin*m
 *  Q6_K    : 210 B / 256       : 128 B low nibbles, 64 B high 2-bit pairs,
 *                                int8 scale x 16, fp16 d (last);      w = d*scale*(q - 32)
 *  MXFP4   : 17 B / 32         : E8M0 scale e, 16 B E2M1 codes;       w = 2^(e-127) * E2M1
 *  IQ4_NL  : 18 B / 32         : fp16 d, 16 B 4-bit codes (low nibbles = weights 0..15);
 *                                w = d * NL[code], NL = -127 -104 -83 -65 -49 -35 -22 -10
 *                                1 13 25 38 53 69 89 113
 *  IQ4_XS  : 136 B / 256       : fp16 d, uint16 high scale bits, 4 B low scale
 *                                nibbles, 128 B codes; sub-block b of 32:
 *                                w = d * (ls_b - 32) * NL[code]
 *  IQ3_XXS : 98 B / 256        : fp16 d, 64 B grid indices, 8 x uint32 (4-bit
 *                                scale s, four 7-bit sign indices) per
 *                                sub-block of 32; w = d * (0.5 + s) / 2 *
 *                                magnitude from the grid * sign (the eighth
 *                                sign of a group of 8 is its parity)
 * These are the public GGUF layouts (Q8_0, Q4_K, Q6_K, IQ4_NL, IQ4_XS, IQ3_XXS)
 * and the OCP MX v1.0 encoding (MXFP4); the pages name the formats (the tiers
 * of "三张 RTX 3090 …", section 优化策略二: Q6_K/Q8_0, IQ4_XS/IQ4_NL,
 * IQ3_XXS/MXFP4) but print no layout. IQ3_XXS needs the 256-entry grid of
 * four magnitude bytes per entry that its model file was made with, passed in
 * moe_weight_table.iq3_grid. IQ formats run on the tensor-core path and on
 * both kinds of grouped GEMV kernels (the streaming ones decode batches of up
 * to 16 rows).
 *   MOE_T5_G128 ternary, 128 weights / 28 B: fp16 s, then 26 code bytes;
 *                                weight 5b + i is base-3 digit i (least
 *                                significant first) of code byte b (the last
 *                                byte's digits 3 and 4 unused); w = s * (digit - 1)
 * The ternary packing is the one "RTX 4080 SUPER 原生 Windows 跑 27B", section
 * 九.2 gives (five weights per byte, one fp16 scale per 128 weights, 1.75 bits
 * per weight); the digit order within a byte and the scale's place in front
 * of the codes are this library's reading. It runs on the tensor-core and the
 * tiled grouped GEMV paths. */
typedef enum {
    MOE_Q8_0 = 1, MOE_Q4_K = 2, MOE_Q6_K = 3, MOE_MXFP4 = 4,
    MOE_IQ4_NL = 5, MOE_IQ4_XS = 6, MOE_IQ3_XXS = 7, MOE_T5_G128 = 8
} moe_format;

/* Limits of this build. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_K 32           /* k + n_shared <= MOE_MAX_K */
#define MOE_MAX_SHARED 4
#define MOE_MAX_HIDDEN 8192
#define MOE_MAX_INTER 8192

/* One quantized matrix: `rows` rows of `cols` weights, blocks along the
 * columns (the reduction axis). Row r starts at data + r * row_stride_bytes.
 * row_stride_bytes >= (cols / block_elems) * block_bytes and a multiple of 16;
 * data is a 16-byte aligned pointer to rows * row_stride_bytes bytes, in
 * device memory, or, for the experts of the cold tier, in pinned or registered
 * host memory that the GPU can read (on GB300 the Grace CPU's memory, read
 * over NVLink-C2C; "三张 RTX 3090 …", section 优化策略一 keeps the coldest experts
 * in host RAM). An expert's three matrices are all in device memory or all in
 * host memory. A layer with cold experts runs on the grouped GEMV path: after
 * routing, the routed cold experts' bytes are copied by the GPU into the
 * workspace (sized by moe_ffn_workspace_size) and read from there. */
typedef struct {
    int32_t format;            /* moe_format */
    int32_t rows;
    int32_t cols;
    int32_t reserved;          /* 0 */
    int64_t row_stride_bytes;
    const void *data;          /* device */
} moe_matrix;

/* One expert: gate and up are [inter rows x hidden cols] in the same format;
 * down is [hidden rows x inter cols]. */
typedef struct {
    moe_matrix gate, up, down;
} moe_expert;

#define MOE_TABLE_PREPARED 0x4d4f4554u

/* The per-expert format-tagged weight table of one layer. The caller fills
 * n_experts, hidden, inter, n_shared and experts; moe_table_prepare fills the
 * rest.
 *
 * Shared experts ("多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出
 * 120 t/s", memory layout: the router and the shared experts sit beside the
 * routed experts; the model there stores them in Q8_0) run for every token
 * with weight 1, added to the routed experts' weighted sum. They are table
 * entries E .. E + n_shared - 1 and take the token slots k .. k + n_shared - 1
 * after the routed ones, so they go through the same bucketing, grouped
 * kernels and ordered combine; moe_options.expert_lo/hi range over all
 * E + n_shared entries. */
typedef struct {
    int32_t n_experts;         /* E: routed experts, 1..MOE_MAX_EXPERTS */
    int32_t hidden;            /* H */
    int32_t inter;             /* I */
    int32_t n_shared;          /* S: shared experts, 0..MOE_MAX_SHARED; E + S <= MOE_MAX_EXPERTS */
    const moe_expert *experts; /* host array [E + S]; read by moe_table_prepare only */
    /* ---- written by moe_table_prepare ---- */
    void *device_table;        /* device copy of the descriptors */
    uint32_t formats_present;  /* bit (1 << format) for every format in use */
    uint32_t prepared;         /* MOE_TABLE_PREPARED after a successful prepare */
    uint32_t gateup_formats;   /* bit (1 << format) for every gate/up format in use */
    uint32_t down_formats;     /* bit (1 << format) for every down format in use */
    int64_t max_gateup_stride; /* largest gate/up row stride, bytes */
    int64_t max_down_stride;   /* largest down row stride, bytes */
    /* Set when every expert has the formats and strides of expert 0 and its
     * gate/up/down data sit at expert 0's plus e * uniform_step[0/1/2] bytes
     * (experts stored as one strided tensor): kernels then compute the
     * descriptors instead of reading them. */
    int32_t uniform_layout;
    int32_t tc_maps;           /* 1 when the tensor path's per-matrix TMA descriptors were built */
    moe_expert uniform_base;
    int64_t uniform_step[3];
    /* ---- filled by the caller ---- */
    const void *iq3_grid;      /* device uint32 [256], 16-byte aligned: the IQ3_XXS grid
                                  (required if any matrix is IQ3_XXS, else may be NULL) */
    /* ---- written by moe_table_prepare ---- */
    int32_t n_cold;            /* experts whose weights are in host memory (the cold tier) */
    int32_t reserved2;
    int64_t cold_bytes_max;    /* largest cold expert, bytes (256-aligned matrices) */
} moe_weight_table;

/* Paths for moe_options.path. */
#define MOE_PATH_AUTO 0        /* FUSED where it applies, else GEMV where its streaming kernels
                                  apply (moe_ffn_gemv_kernels), else TENSOR where it applies,
                                  else GEMV (see moe_ffn_path) */
#define MOE_PATH_GEMV 1        /* grouped GEMV kernels (route, bucket, gate/up, down, combine); any layer */
#define MOE_PATH_TENSOR 2      /* tcgen05 grouped GEMMs with TMEM-resident dequantised weights
                                  (prefill chunks):
                                  H % 128 == 0, I % 64 == 0, any format mix. Each weight is
                                  represented in fp16, so it must lie within fp16 range
                                  (|w| <= 65504; quantized LLM weights are O(1)). */
#define MOE_PATH_FUSED 3       /* one persistent cooperative kernel per layer for decode rows:
                                  T * k <= 64, Q4_K gate/up and Q8_0 down, H % 64 == 0,
                                  I % 32 == 0, I <= 1024, no shared experts, no cold tier */

/* Options of moe_ffn_forward (NULL = defaults). */
typedef struct {
    uint32_t struct_size;      /* sizeof(moe_options); checked */
    int32_t renormalize;       /* 1 (default): the k selected weights sum to 1; 0: plain softmax values */
    uint32_t format_mask;      /* keep an expert only if bit (1 << its gate format) is set; default all */
    int32_t expert_lo;         /* keep experts in [expert_lo, expert_hi); default [0, E + n_shared) */
    int32_t expert_hi;
    int32_t path;              /* MOE_PATH_* */
    int32_t reserved;          /* 0 */
    /* Profiling hook: NULL, or a host array of 3 cudaEvent_t recorded on the
     * stream around the expert mat-mul kernels: before the gate/up kernel,
     * between it and the down kernel, and after the down kernel. On the fused
     * path, where one kernel does both, events 1 and 2 are both recorded after
     * it; on the tensor path the h conversion falls between events 1 and 2. During stream capture they become external event-record nodes. */
    void *const *timing_events;
} moe_options;

/* Human-readable name of a moe_status code (static string). */
const char *moe_strerror(int code);

/* The last CUDA error seen by this thread (cudaError_t value, 0 if none). */
int moe_last_cuda_error(void);

/* Bytes of device memory moe_table_prepare needs for `n_experts` table
 * entries (routed plus shared experts): the 72-byte descriptors, a cold-tier
 * flag byte and 3 x 128-byte TMA tensor maps per entry for the tensor path. */
size_t moe_table_device_bytes(int32_t n_experts);

/* Validate W (shapes, formats, strides, alignment) and copy its descriptors
 * into `device_buf` (caller-owned device memory of at least
 * moe_table_device_bytes(W->n_experts + W->n_shared) bytes). Synchronises `stream`.
 * On success sets W->device_table = device_buf, W->prepared and the summary
 * fields. The weight data itself is not read or copied; its device pointers
 * must stay valid while forwards that use W run. Re-prepare after changing
 * W->experts. Errors: INVALID_ARG, BAD_SHAPE, BAD_FORMAT, UNSUPPORTED, CUDA. */
int moe_table_prepare(moe_weight_table *W, void *device_buf, size_t device_bytes, moe_stream_t stream);

/* Router (step 1). logits: device fp32 [T, E] row-major. For every row, the k
 * experts with the largest logits (equal logits: lower expert index first;
 * non-finite logits rank last) go to ids (device int32 [T, k], slot order =
 * rank) and their softmax probabilities (fp32; divided by their sum when
 * renormalize != 0) to weights (device fp32 [T, k]). Non-finite logits set
 * MOE_FLAG_NONFINITE_LOGIT in *status (device uint32, may be NULL) and get
 * weight 0. 1 <= k <= min(E, MOE_MAX_K), E <= MOE_MAX_EXPERTS, T >= 0. */
int moe_route_topk(const float *logits, int32_t T, int32_t E, int32_t k, int32_t renormalize,
                   int32_t *ids, float *weights, uint32_t *status, moe_stream_t stream);

/* Bucketing (step 2). ids: device int32 [T, k]. Pair p = t*k + j is kept if
 * expert_lo <= ids[p] < expert_hi; -1 is skipped silently, other ids outside
 * [0, E) set MOE_FLAG_BAD_ID and are skipped, and an expert repeated within
 * one token sets MOE_FLAG_DUPLICATE_ID (its pairs are still bucketed).
 * Outputs (device int32): offsets [E + 1] = exclusive prefix sum of the kept
 * per-expert counts; pairs [T*k] = kept pair numbers grouped by expert
 * (ascending expert, ascending p within an expert; entries past offsets[E]
 * are unspecified); pos [T*k] = bucket position of each pair or -1;
 * active [E + 1] = {n_active, active expert ids ascending...}.
 * status: device uint32 or NULL. E <= MOE_MAX_EXPERTS. */
int moe_bucket(const int32_t *ids, int32_t T, int32_t k, int32_t E, int32_t expert_lo, int32_t expert_hi,
               int32_t *offsets, int32_t *pairs, int32_t *pos, int32_t *active, uint32_t *status,
               moe_stream_t stream);

/* Workspace bytes moe_ffn_forward needs for a prepared W, T tokens and top-k
 * on the path MOE_PATH_AUTO picks (0 if the arguments are invalid). */
size_t moe_ffn_workspace_size(const moe_weight_table *W, int32_t T, int32_t k);

/* The same for an explicitly requested path (MOE_PATH_*); 0 if the arguments
 * are invalid or the path cannot run this layer. The tensor path needs
 * about P * (2H + 2I + 12) + 16 * (P/128 + min(P, E)) bytes more than the
 * others (P = T * k): its fp16 activation and h copies in bucket order, row
 * scales and chunk table. */
size_t moe_ffn_workspace_size_for_path(const moe_weight_table *W, int32_t T, int32_t k, int32_t path);

/* The path moe_ffn_forward takes for these arguments (MOE_PATH_GEMV,
 * MOE_PATH_TENSOR or MOE_PATH_FUSED; resolves MOE_PATH_AUTO), or -1 if the
 * requested path cannot run this layer. Host-only. */
int moe_ffn_path(const moe_weight_table *W, int32_t T, int32_t k, const moe_options *opt);

/* Which kernels the grouped GEMV path (MOE_PATH_GEMV) runs for these
 * arguments: MOE_GEMV_STREAMING (persistent gate/up and down kernels that
 * stream the routed experts' rows through a shared-memory ring; decode
 * batches of 1..16 rows, or 1..32 rows when every gate/up matrix is Q8_0 or
 * Q4_K; gate/up in Q8_0, Q4_K, Q6_K, MXFP4, IQ4_NL, IQ4_XS or IQ3_XXS and down
 * in Q8_0, MXFP4 or IQ4_NL; shared memory permitting, and an activation
 * pointer aligned to 16 bytes at the forward) or MOE_GEMV_TILED (one CTA per expert
 * tile; any other layer). -1 if the arguments are invalid. Host-only. */
#define MOE_GEMV_TILED 0
#define MOE_GEMV_STREAMING 1
int moe_ffn_gemv_kernels(const moe_weight_table *W, int32_t T, int32_t k);

/* Zero a workspace (all ws_bytes, among them the status word and the fused
 * kernel's grid-barrier counter) once, before its first forward.
 * ws: device, at least moe_ffn_workspace_size bytes. */
int moe_ffn_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* The whole layer (steps 1-6): router, bucketing, grouped gate/up with the
 * fused SwiGLU, grouped down projection and the slot-ordered combine; with
 * n_shared > 0 the shared experts ride in the same kernels as slots k.. of
 * every token (weight 1) and are added after the routed experts.
 * x: device bf16 bits [T, H]; logits: device fp32 [T, E]; out: device fp32
 * [T, H] (fully overwritten; tokens whose pairs are all dropped get 0).
 * ws: device workspace of ws_bytes >= moe_ffn_workspace_size(W, T, k), 256-byte
 * aligned, initialised once with moe_ffn_workspace_init. opt: NULL or options
 * (format_mask / expert range drop the other experts' contributions).
 * Forwards that share a workspace must be ordered on one stream.
 * Errors: INVALID_ARG, NOT_PREPARED, WORKSPACE_TOO_SMALL, UNSUPPORTED, CUDA. */
int moe_ffn_forward(const moe_weight_table *W, const uint16_t *x, const float *logits, int32_t T,
                    int32_t k, const moe_options *opt, float *out, void *ws, size_t ws_bytes,
                    moe_stream_t stream);

/* Device pointers (into ws) of the routing results the last forward with this
 * workspace left: ids [T*K], weights [T*K], offsets [N+1], active [N+1],
 * pairs [T*K] and pos [T*K] (K = k + n_shared slots per token, the shared
 * experts in the last n_shared with weight 1; N = E + n_shared), with the
 * meaning given at moe_route_topk and moe_bucket. Output pointers may be
 * NULL. Host-only; no CUDA call. */
int moe_ffn_workspace_views(const moe_weight_table *W, int32_t T, int32_t k, void *ws, int32_t **ids,
                            float **weights, int32_t **offsets, int32_t **active, int32_t **pairs,
                            int32_t **pos);

/* Read and clear the device status flags of a workspace (moe_device_flags).
 * ws = NULL reads those of moe_ffn_forward_noalloc's scratch array on the
 * current device. Synchronises `stream`. *status_out is a host pointer. */
int moe_ffn_read_status(void *ws, uint32_t *status_out, moe_stream_t stream);

/* Bound (ns) on every device-side wait of the layer's kernels for data or for
 * other threads (ring slots, mbarriers, the fused kernel's grid barrier) on
 * the current device; 0 restores the default of 2 s (a layer takes well
 * under a millisecond). A wait that exceeds it gives up: the kernel sets
 * MOE_FLAG_WAIT_TIMEOUT in the status word, skips the rest of its work, waits
 * (with a separate, long poll bound) for its own bulk copies and MMAs still in
 * flight, releases its tensor memory and returns, so the context stays usable;
 * that call's output is then incomplete. Meant for tests of this path and for
 * callers that want an earlier deadline. A blocking copy to the device (it
 * synchronises with the legacy default stream); not during stream capture.
 * This follows no passage of the pages: it is the library's failure
 * detection. Errors: CUDA. */
int moe_set_wait_timeout_ns(uint64_t ns);

/* Expert sharding across GPUs ("多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出
 * 120 t/s", section "8 张卡是怎么配对的": the routed experts are split 50/50
 * across a pair of GPUs and the router is replicated). Each rank runs
 * moe_ffn_forward over the same x and logits with its expert range
 * (moe_options.expert_lo/expert_hi) and gets a partial out[T, H]; after the
 * partials of all ranks are gathered, this sums them:
 *     out[i] = ((parts[0][i] + parts[1][i]) + parts[2][i]) + ...
 * one fp32 add at a time in ascending part (rank) order, so every rank gets
 * bit-identical results. parts: device fp32 [n_parts][count] (contiguous);
 * out: device fp32 [count] (may alias parts[0]). n_parts >= 1, count >= 0.
 * Errors: INVALID_ARG, CUDA. */
int moe_sum_partials(const float *parts, int32_t n_parts, int64_t count, float *out, moe_stream_t stream);

/* Size of the device scratch array that moe_ffn_forward_noalloc uses. */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* The whole layer, like moe_ffn_forward, for callers that cannot allocate
 * device memory: a host framework whose memory planner owns all device memory,
 * a latency-critical loop where cudaMalloc/cudaFree would synchronise the
 * device, or a C client that only receives input and output pointers. The
 * layer's scratch lives in a fixed device array of MOE_NOALLOC_SCRATCH_BYTES
 * (4 MiB) inside this library, held by every GPU that loads the library until
 * the process exits; no workspace argument, and no allocation of any kind.
 * The source pages have no counterpart of this entry point.
 *   - Sizes: accepted when the workspace of the path the call takes
 *     (moe_ffn_workspace_size_for_path with opt->path, AUTO by default) fits in
 *     4 MiB: e.g. up to 25 tokens at E = 512, k = 10, H = 2048, I = 640, where
 *     AUTO sends one token to the fused kernel and up to 16 rows (25 with
 *     Q8_0 / Q4_K gate/up) to the streaming GEMV kernels, and the tensor path
 *     (requested, or AUTO's choice for other formats above 16 rows) up to about 20
 *     tokens; larger sizes return MOE_ERR_UNSUPPORTED before anything is
 *     enqueued.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents:
 *     calls whose work overlaps on the GPU (different streams, or several host
 *     threads) race and corrupt each other's results; order them on one
 *     stream. Device status flags accumulate in the array until read with
 *     moe_ffn_read_status(NULL, ...).
 * Other arguments, errors and ownership as for moe_ffn_forward. */
int moe_ffn_forward_noalloc(const moe_weight_table *W, const uint16_t *x, const float *logits, int32_t T,
                            int32_t k, const moe_options *opt, float *out, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
