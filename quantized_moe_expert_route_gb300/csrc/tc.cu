// Tensor-core grouped path: the gate/up and down projections of every active
// expert as grouped GEMMs on the 5th-generation tensor cores, for prefill
// chunks (hundreds to thousands of rows per layer).
//
// "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理优化指南",
// 优化策略二/三: one grouped mat-mul over the routed experts of a layer, whose
// weights come in per-expert tiers of block formats (Q6_K/Q8_0, 4-bit,
// MXFP4), with explicit skipping of unrouted (-1) ids. "一张 RTX 3090 跑 Llama
// 70B", 4.4: SwiGLU fused with the FC so g and u never reach memory.
//
// Layer = route -> bucket -> tc_prep (fp16 activations in bucket order, chunk
// table) -> tc_gemm<gate/up> (SwiGLU epilogue, fp32 h) -> tc_hprep (fp16 h
// with a per-row power-of-two scale) -> tc_gemm<down> (fp32 y in bucket order)
// -> combine (ascending slot).
//
// tc_gemm is a persistent kernel, one CTA per SM, that works through units of
// (chunk of <= 128 bucket rows of one expert, 128 weight rows). Per unit it
// computes D[128 weight rows, n act rows] = W_e[rows, :] . act[chunk, :]^T with
// tcgen05.mma (M = 128, N = n rounded up to 16, K = 16 per instruction):
//   - A (weights) lives in TMEM. A TMA producer warp streams each weight row's
//     quantized blocks (256 K at a time) into a shared-memory ring with 1-D
//     bulk copies; 16 dequantising warps turn them into exact-then-rounded
//     fp16 and write them to TMEM with tcgen05.st, 64 K per stage.
//   - B (activations, fp16, K-major) is TMA-tiled from the bucket-ordered
//     activation matrix with 128-byte swizzle, 16 rows per box.
//   - D accumulates in fp32 in TMEM (two buffers, so the epilogue of one unit
//     overlaps the next unit's MMAs); 4 epilogue warps read it with tcgen05.ld.
// Gate/up units hold 64 gate rows (TMEM lanes 0-63) and the same 64 up rows
// (lanes 64-127), so SwiGLU needs only the CTA's own accumulator.
#include <cuda.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int TC_M = 128;                    // weight rows per unit = TMEM lanes
constexpr int TC_NCHUNK = 128;               // activation rows per chunk (MMA N <= 128)
constexpr int TC_KA = 64;                    // K per A step: one 128-byte row of fp16
constexpr int TC_KR = 256;                   // K per raw (quantized) stage
constexpr int TC_ASTAGES = 8;                // A stages in TMEM, 32 columns each: 2 events of 4
constexpr int TC_AEV = 4;                    // A steps per event (one raw stage)
constexpr int TC_EVSLOTS = TC_ASTAGES / TC_AEV;
constexpr int TC_BSTAGES = 3;                // B stages in shared memory
constexpr int TC_BSTAGE_BYTES = 2 * TC_NCHUNK * 128;   // 32 KB: up to 4 A steps of <= 64 rows
constexpr int TC_BOX_ROWS = 16;              // rows per activation TMA box
constexpr int TC_DG = TC_KR / TC_KA;         // dequantising warpgroups
constexpr int TC_PPG = (TC_KR / TC_KA) / TC_DG;   // 64-K pieces per group per raw stage
constexpr int TC_DQ0 = 4;                    // warps 0-3 epilogue, 4..19 dequant
constexpr int TC_PROD = TC_DQ0 + 4 * TC_DG;  // 20: weight producer (TMA)
constexpr int TC_MMA = TC_PROD + 1;          // 21: MMA issuer
constexpr int TC_BPROD = TC_MMA + 1;         // 22: activation producer (TMA)
constexpr int TC_WARPS = TC_BPROD + 1;
constexpr int TC_THREADS = TC_WARPS * 32;    // 736
constexpr int TC_TMEM_COLS = 512;
constexpr int TC_ACOL0 = 2 * TC_NCHUNK;      // A stages after the two accumulators
constexpr int TC_RS_MAX = 8;
constexpr int TC_UBUF_FLOATS = 16 * 128;     // epilogue exchange: 16 columns x 128 lanes
constexpr int TC_NBARS = 2 * TC_RS_MAX + TC_EVSLOTS + 2 * TC_BSTAGES + 4 + 1;
constexpr uint32_t TC_NEG1152 = 0xE480E480u;  // fp16 pair (-1152, -1152)
constexpr uint32_t TC_NEG1056 = 0xE420E420u;  // fp16 pair (-1056, -1056)
constexpr uint32_t TC_MAGIC = 0x64006400u;    // fp16 pair (1024, 1024)

// Raw stage geometry per format (index = moe_format): a stage holds, for each
// weight row, the blocks of 256 K as TMA boxes of RAW_W bytes (widened to
// 16-byte boundaries); Q8_0's 272 bytes take two boxes, 128 bytes apart;
// T5_G128's 56 bytes start 0 or 8 bytes into a 64-byte box.
__host__ __device__ constexpr int raw_w(int f) {
    return f == MOE_Q6_K ? 240 : f == MOE_IQ3_XXS ? 112 : f == MOE_T5_G128 ? 64 : 144;
}
__host__ __device__ constexpr int raw_nbox(int f) { return f == MOE_Q8_0 ? 2 : 1; }
__host__ __device__ constexpr int blk_elems(int f) {
    return f == MOE_Q4_K || f == MOE_Q6_K || f == MOE_IQ4_XS || f == MOE_IQ3_XXS ? 256
         : f == MOE_T5_G128 ? 128 : 32;
}
__host__ __device__ constexpr int blk_bytes(int f) {
    return f == MOE_Q8_0 ? 34 : f == MOE_Q4_K ? 144 : f == MOE_Q6_K ? 210 : f == MOE_MXFP4 ? 17
         : f == MOE_IQ4_NL ? 18 : f == MOE_IQ4_XS ? 136 : f == MOE_IQ3_XXS ? 98 : 28;
}
// Kernel variants by the decoders they carry: the four standard formats; with
// the IQ formats (and the IQ3_XXS grid in shared memory); with the IQ formats
// and T5_G128. Each layer takes the smallest variant that decodes it.
constexpr int TC_XV_STD = 0, TC_XV_IQ = 1, TC_XV_T5 = 2;
constexpr uint32_t TC_IQ_FORMATS = (1u << MOE_IQ4_NL) | (1u << MOE_IQ4_XS) | (1u << MOE_IQ3_XXS);
constexpr int TC_GRID_BYTES = 1024;          // the IQ3_XXS grid in shared memory (IQ variants)
constexpr int TC_UQ = 16;                    // unit queue entries (per CTA, shared memory)
constexpr int TC_UQ_BYTES = TC_UQ * 16 + 32; // entries of 16 bytes, the two counters, alignment

static_assert(TC_ACOL0 + TC_ASTAGES * 32 <= TC_TMEM_COLS, "TMEM budget");
static_assert(TC_DG * TC_PPG == TC_KR / TC_KA, "groups x pieces cover a raw stage");
static_assert(TC_AEV == TC_KR / TC_KA, "an event is one raw stage");

struct TcArgs {
    const DevExpert *table;
    const CUtensorMap *wmaps;  // per expert: gate, up, down weight maps (bytes [rows][stride])
    const int4 *chunks;        // {expert, first bucket row, rows, 0}
    const int32_t *n_chunks;
    int K;                     // reduction length: H (gate/up) or I (down)
    int S;                     // units per chunk: I/64 (gate/up) or H/128 (down)
    int H, I;
    int slot_bytes;            // raw stage bytes
    int RS;                    // raw stages in the ring
    const float *ascale;       // per bucket row: 2^-sigma of its fp16 activation row
    float *h32;                // gate/up: h [rows][I] fp32, bucket order
    uint32_t *hmax;            // gate/up: max |h| bits per bucket row
    float *y;                  // down: y [rows][H] fp32, bucket order
    uint32_t *status;
    const uint32_t *grid;      // IQ3_XXS grid (256 words) or null
    int32_t *unit_next;        // next unit to hand out (zeroed by tc_prep_kernel)
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));  // (a & mask) | bits
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t half2_bits(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}
__device__ __forceinline__ uint32_t splat_half(__half h) { return half2_bits(h, h); }
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// N little-endian words starting at any byte address of shared memory.
template <int N>
__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t (&w)[N]) {
    const uint32_t base = addr & ~3u, sh = (addr & 3u) * 8u;
    uint32_t v[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) v[i] = lds32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

__device__ __forceinline__ void mbar_arrive_cta(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Each poll may suspend the thread up to this long (ns); it resumes as soon
// as the phase completes, so waiting warps do not spin on the issue slots.
constexpr uint32_t TC_SUSPEND_NS = 20000;

__device__ __forceinline__ bool try_wait_parity(uint32_t addr, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    return done != 0;
}

// The polling loop of a bounded parity wait (g_wait_ns, or WAIT_LIMIT
// polls) that also gives up once another role has aborted; `suspend` polls
// with a suspend-time hint. Out of line: every role's waits share one copy of
// the code, which keeps the kernel small enough for the instruction caches.
__device__ __noinline__ bool tc_wait_slow(uint32_t addr, uint32_t parity, volatile int *abort_flag, bool suspend) {
    const uint64_t t0 = global_ns(), bound = *(volatile unsigned long long *)&g_wait_ns;
    const uint32_t check = suspend ? 0u : 1023u;
    const uint32_t hint = bound < TC_SUSPEND_NS ? (uint32_t)bound : TC_SUSPEND_NS;
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        uint32_t done;
        if (suspend)
            asm volatile(
                "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                : "=r"(done)
                : "r"(addr), "r"(parity), "r"(hint)
                : "memory");
        else
            done = try_wait_parity(addr, parity);
        if (done) return true;
        if ((i & check) == check) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > bound) return false;
        }
    }
    return false;
}
// Bounded parity wait for roles that may wait long (producers, dequantisers,
// epilogue): polls with a suspend hint.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    const uint32_t addr = smem_addr(bar);
    return try_wait_parity(addr, parity) || tc_wait_slow(addr, parity, abort_flag, true);
}
// The same without a suspend hint, for the MMA issuer: its waits are short and
// on the critical path.
__device__ __forceinline__ bool tc_spin(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    const uint32_t addr = smem_addr(bar);
    return try_wait_parity(addr, parity) || tc_wait_slow(addr, parity, abort_flag, false);
}

__device__ __forceinline__ void tc_fail(volatile int *abort_flag, uint32_t *status) {
    if (!*abort_flag) {
        *abort_flag = 1;
        atomicOr(status, (uint32_t)MOE_FLAG_WAIT_TIMEOUT);
    }
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] . B[smem]^T, kind::f16 (fp16 A and B, fp32 D), cta_group::1.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same, accumulating, with the B descriptor given as its two 32-bit
// words: the issuing thread adds a tile's offset to the low word alone (the
// start-address field, which no offset inside shared memory carries out of).
// One add per MMA instead of a 64-bit add: 772 -> 762 us per 2048-token layer.
__device__ __forceinline__ void mma_f16_ts_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                               uint32_t idesc) {
    asm volatile(
        "{ .reg .b64 bd; mov.b64 bd, {%2, %3}; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, 1; }" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc)
        : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart; the tile starts 1024-aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                      // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                      // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                      // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: fp32 D, fp16 A and B, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_f16(int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(TC_M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// silu(z) = z / (1 + e^-z) with the hardware exponential and reciprocal
// (relative error ~1e-6, far inside the layer's 1e-3 bound).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// v[j] (j < 8) of every lane -> lanes 0..7 return the max over the warp of
// v[lane]; v is clobbered.
__device__ __forceinline__ float warp_colmax8(float (&v)[8]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; ++j) {
            const float send = up ? v[j] : v[j + o];
            const float keep = up ? v[j + o] : v[j];
            v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
    float m = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 8));
    return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
}


// ------------------------------------------------------------------ dequantisation
// Each function turns one weight row's 64 consecutive K elements (piece g of
// a raw stage) into 32 fp16 pairs in K order (low half = lower K), the TMEM
// layout of the MMA's A operand. Integer codes become exact fp16 values
// through the 1024 + q exponent trick; the block scales are applied in fp16
// FMAs, so each weight is rounded once or twice to fp16 (11-bit significand).

// Q4_K 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes.
__device__ __forceinline__ void q4k_scale_min(int j, uint32_t s03, uint32_t s47, uint32_t s811, int &sc, int &m) {
    const int sh = 8 * (j & 3);
    const int a = (s03 >> sh) & 0xff, b = (s47 >> sh) & 0xff, c = (s811 >> sh) & 0xff;
    if (j < 4) {
        sc = a & 63;
        m = b & 63;
    } else {
        sc = (c & 15) | ((a >> 6) << 4);
        m = (c >> 4) | ((b >> 6) << 4);
    }
}

// Q4_K super-block at `blk` (16-aligned); piece g = elements 64g..64g+63:
// low nibbles of qs[32g..32g+31] (sub-block 2g), then their high nibbles
// (sub-block 2g+1). w = d*sc*q - dmin*m.
__device__ __forceinline__ void dq_q4k(uint32_t blk, int g, uint32_t (&r)[32]) {
    uint32_t h0, s03, s47, s811;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(h0), "=r"(s03), "=r"(s47), "=r"(s811) : "r"(blk));
    int sc0, m0, sc1, m1;
    q4k_scale_min(2 * g, s03, s47, s811, sc0, m0);
    q4k_scale_min(2 * g + 1, s03, s47, s811, sc1, m1);
    const uint32_t D2 = (h0 & 0xffffu) * 0x10001u;
    const float dmin = __half2float(__ushort_as_half((uint16_t)(h0 >> 16)));
    // (1024 + q) * sc - 1024 * sc = sc * q exactly (<= 945); likewise for the
    // high nibble read as 1024 + 16 q with sc / 16
    const uint32_t SC0 = splat_half(__int2half_rn(sc0)), NS0 = splat_half(__int2half_rn(-1024 * sc0));
    const uint32_t SC1 = splat_half(__float2half_rn(0.0625f * (float)sc1)), NS1 = splat_half(__int2half_rn(-64 * sc1));
    const uint32_t MT0 = splat_half(__float2half_rn(-dmin * (float)m0));
    const uint32_t MT1 = splat_half(__float2half_rn(-dmin * (float)m1));
    uint32_t w[8];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(blk + 16 + 32 * g));
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "r"(blk + 32 + 32 * g));
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t t0 = prmt(w[m], 0u, 0x4140u), t1 = prmt(w[m], 0u, 0x4342u);
        r[2 * m] = hfma2(hfma2(lop_and_or(t0, 0x000F000Fu, TC_MAGIC), SC0, NS0), D2, MT0);
        r[2 * m + 1] = hfma2(hfma2(lop_and_or(t1, 0x000F000Fu, TC_MAGIC), SC0, NS0), D2, MT0);
        r[16 + 2 * m] = hfma2(hfma2(lop_and_or(t0, 0x00F000F0u, TC_MAGIC), SC1, NS1), D2, MT1);
        r[17 + 2 * m] = hfma2(hfma2(lop_and_or(t1, 0x00F000F0u, TC_MAGIC), SC1, NS1), D2, MT1);
    }
}

// Q8_0: a piece is two consecutive blocks (68 bytes, 4-aligned at p). w = d*q.
__device__ __forceinline__ void dq_q8_0(uint32_t p, uint32_t (&r)[32]) {
    uint32_t v[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) v[i] = lds32(p + 4 * i);
    const uint32_t D0 = (v[0] & 0xffffu) * 0x10001u, D1 = (v[8] >> 16) * 0x10001u;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        // bytes as 1152 + q (q + 128 in the low byte of 0x64xx), less 1152
        const uint32_t c0 = __funnelshift_r(v[m], v[m + 1], 16) ^ 0x80808080u;
        const uint32_t c1 = v[9 + m] ^ 0x80808080u;
        r[2 * m] = hmul2(hadd2(prmt(c0, 0x64646464u, 0x5140u), TC_NEG1152), D0);
        r[2 * m + 1] = hmul2(hadd2(prmt(c0, 0x64646464u, 0x7362u), TC_NEG1152), D0);
        r[16 + 2 * m] = hmul2(hadd2(prmt(c1, 0x64646464u, 0x5140u), TC_NEG1152), D1);
        r[17 + 2 * m] = hmul2(hadd2(prmt(c1, 0x64646464u, 0x7362u), TC_NEG1152), D1);
    }
}

// Q6_K super-block at `blk` (2-aligned); piece g covers quarters r0 = 2(g&1)
// and r0+1 of half g>>1. w = d*scale*(q - 32).
__device__ __forceinline__ void dq_q6k(uint32_t blk, int g, uint32_t (&r)[32]) {
    const int hh = g >> 1, r0 = 2 * (g & 1);
    uint32_t L0[8], L1[8], Q[8], SC[1], DW[1];
    lds_words<8>(blk + 64 * hh, L0);
    lds_words<8>(blk + 64 * hh + 32, L1);
    lds_words<8>(blk + 128 + 32 * hh, Q);
    lds_words<1>(blk + 192 + 8 * hh + 2 * r0, SC);
    lds_words<1>(blk + 208, DW);
    const uint32_t D2 = (DW[0] & 0xffffu) * 0x10001u;
    uint32_t S[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) S[i] = splat_half(__int2half_rn((int)(int8_t)(SC[0] >> (8 * i))));
    const int ns = 4 * (g & 1);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t q0 = ((L0[m] >> ns) & 0x0F0F0F0Fu) | (((Q[m] >> (2 * r0)) & 0x03030303u) << 4);
        const uint32_t q1 = ((L1[m] >> ns) & 0x0F0F0F0Fu) | (((Q[m] >> (2 * r0 + 2)) & 0x03030303u) << 4);
        const uint32_t sa = m < 4 ? S[0] : S[1], sb = m < 4 ? S[2] : S[3];
        r[2 * m] = hmul2(hmul2(hadd2(prmt(q0, 0x64646464u, 0x5140u), TC_NEG1056), sa), D2);
        r[2 * m + 1] = hmul2(hmul2(hadd2(prmt(q0, 0x64646464u, 0x7362u), TC_NEG1056), sa), D2);
        r[16 + 2 * m] = hmul2(hmul2(hadd2(prmt(q1, 0x64646464u, 0x5140u), TC_NEG1056), sb), D2);
        r[17 + 2 * m] = hmul2(hmul2(hadd2(prmt(q1, 0x64646464u, 0x7362u), TC_NEG1056), sb), D2);
    }
}

// E2M1 nibble pair (bits 0-3 of each 16-bit half) as fp16 of value * 2^-14.
__device__ __forceinline__ uint32_t e2m1_pair_bits(uint32_t x) {
    return ((x & 0x00070007u) << 9) | ((x & 0x00080008u) << 12);
}
// The two fp16 factors SA, SB with (v * 2^-14) * SA * SB = v * 2^(e-127) for an
// E2M1 value v, such that the first product is exact and only the second
// rounds (one rounding in all): e in [99, 128] takes SA = 2^(e-113), SB = 1;
// larger e takes SA = 2^15 and the rest in SB (results beyond fp16 range
// overflow, as any weight outside it would); e < 99 gives |w| < 2^-26, which
// rounds to 0; e = 255 (NaN in E8M0) gives NaN. Selects, no branches: the
// lanes of a warp hold different rows' scales.
__device__ __forceinline__ void mxfp4_scales(uint32_t e, uint32_t &SA, uint32_t &SB) {
    const int k = (int)e - 113;
    const int ka = min(max(k, -14), 15), kb = min(max(k - 15, 0), 15);
    SA = ((uint32_t)(ka + 15) << 10) * 0x10001u;
    SB = ((uint32_t)(kb + 15) << 10) * 0x10001u;
    SA = k < -14 ? 0u : SA;
    SA = e == 255u ? 0x7e007e00u : SA;
}
// MXFP4: piece g = blocks 2g and 2g+1 of the stage (17 bytes each) at byte
// 34g of `blk`; element i < 16 of a block is the low nibble of qs[i], element
// 16 + i the high nibble. w = 2^(e-127) * E2M1.
__device__ __forceinline__ void dq_mxfp4(uint32_t blk, int g, uint32_t (&r)[32]) {
    uint32_t w[9];
    lds_words<9>(blk + 34 * g, w);
    uint32_t qs[2][4], e[2];
    e[0] = w[0] & 0xffu;
    e[1] = (w[4] >> 8) & 0xffu;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        qs[0][k] = __funnelshift_r(w[k], w[k + 1], 8);
        qs[1][k] = __funnelshift_r(w[4 + k], w[5 + k], 16);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        uint32_t SA, SB;
        mxfp4_scales(e[b], SA, SB);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const uint32_t t = prmt(qs[b][(jj & 7) >> 1], 0u, (jj & 1) ? 0x4342u : 0x4140u);
            const uint32_t x = (jj >= 8 ? (t >> 4) : t) & 0x000F000Fu;
            r[16 * b + jj] = hmul2(hmul2(e2m1_pair_bits(x), SA), SB);
        }
    }
}

// ---- the IQ formats (IQ variant of the kernel)
// Signed bytes of four IQ4 codes (nibbles 0..3 of sel16) from the non-linear
// codebook -127 -104 -83 -65 -49 -35 -22 -10 1 13 25 38 53 69 89 113 (four
// codes per word, code 4w + i in byte i): a byte permute in each half of the
// book, then a byte mask from bit 3 of each code (prmt sign-replicate).
__device__ __forceinline__ uint32_t iq4_lookup4(uint32_t sel16) {
    const uint32_t s7 = sel16 & 0x7777u;
    const uint32_t lo = prmt(0xBFAD9881u, 0xF6EADDCFu, s7);
    const uint32_t hi = prmt(0x26190D01u, 0x71594535u, s7);
    const uint32_t m = prmt(0u, 0x80808080u, ((sel16 >> 1) & 0x4444u) | 0x8888u);
    return (hi & m) | (lo & ~m);
}
// Codes of bytes 0..3 of w, low nibbles (hi = false) or high nibbles, as a
// 16-bit selector with code i in nibble i.
__device__ __forceinline__ uint32_t nibble_sel(uint32_t w, bool hi) {
    const uint32_t v = hi ? (w >> 4) : w;
    const uint32_t x = (v & 0x000F000Fu) | ((v >> 4) & 0x00F000F0u);
    return prmt(x, 0u, 0x0020u);
}
// Four signed bytes -> two fp16 pairs (exact), times D (one rounding).
__device__ __forceinline__ void i8x4_to_half(uint32_t c, uint32_t D, uint32_t &p0, uint32_t &p1) {
    c ^= 0x80808080u;
    p0 = hmul2(hadd2(prmt(c, 0x64646464u, 0x5140u), TC_NEG1152), D);
    p1 = hmul2(hadd2(prmt(c, 0x64646464u, 0x7362u), TC_NEG1152), D);
}
// 32 IQ4 codes (16 code bytes w[0..3]: weights 0..15 low nibbles, 16..31
// high nibbles) times scale pair D -> 16 fp16 pairs in K order at r[o..o+15].
__device__ __forceinline__ void iq4_32(const uint32_t (&w)[4], uint32_t D, uint32_t (&r)[32], int o) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        i8x4_to_half(iq4_lookup4(nibble_sel(w[k], false)), D, r[o + 2 * k], r[o + 2 * k + 1]);
        i8x4_to_half(iq4_lookup4(nibble_sel(w[k], true)), D, r[o + 8 + 2 * k], r[o + 8 + 2 * k + 1]);
    }
}
// IQ4_NL: piece g = blocks 2g, 2g+1 of the stage (18 bytes each: fp16 d,
// 16 code bytes). w = d * codebook[code].
__device__ __forceinline__ void dq_iq4nl(uint32_t blk, int g, uint32_t (&r)[32]) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const uint32_t p = blk + 36 * g + 18 * b;
        uint32_t dw[1], w[4];
        lds_words<1>(p, dw);
        lds_words<4>(p + 2, w);
        iq4_32(w, (dw[0] & 0xffffu) * 0x10001u, r, 16 * b);
    }
}
// IQ4_XS: super-block at `blk` (8-byte aligned); piece g = sub-blocks 2g,
// 2g+1: code bytes [8 + 32g, +32), scales d * (ls - 32) with ls from the
// 6-bit fields (low nibble in byte 4 + j/2, high bits j of the uint16 at 2).
__device__ __forceinline__ void dq_iq4xs(uint32_t blk, int g, uint32_t (&r)[32]) {
    uint32_t h[2], w[8];
    lds_words<2>(blk, h);
    lds_words<8>(blk + 8 + 32 * g, w);
    const float d = __half2float(__ushort_as_half((uint16_t)(h[0] & 0xffffu)));
    const uint32_t sh = h[0] >> 16;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * g + jj;
        const int ls = (int)((h[1] >> (8 * (j >> 1) + 4 * (j & 1))) & 15u) | (int)(((sh >> (2 * j)) & 3u) << 4);
        const uint32_t D = splat_half(__float2half_rn(d * (float)(ls - 32)));
        const uint32_t ww[4] = {w[4 * jj], w[4 * jj + 1], w[4 * jj + 2], w[4 * jj + 3]};
        iq4_32(ww, D, r, 16 * jj);
    }
}
// IQ3_XXS: super-block at `blk` (2-byte aligned); piece g = sub-blocks 2g,
// 2g+1: grid indices [2 + 16g, +16), words [66 + 8g, +8); scale
// d * (0.5 + (a >> 28)) / 2; group l of 8 weights takes its magnitudes from
// two grid entries (grid_s, shared memory) and its signs from the 7-bit
// index (a >> 7l) & 127 with the parity as the eighth.
__device__ __forceinline__ void dq_iq3xxs(uint32_t blk, int g, const uint32_t *grid_s, uint32_t (&r)[32]) {
    uint32_t dw[1], q[4], a[2];
    lds_words<1>(blk, dw);
    lds_words<4>(blk + 2 + 16 * g, q);
    lds_words<2>(blk + 66 + 8 * g, a);
    const float d = __half2float(__ushort_as_half((uint16_t)(dw[0] & 0xffffu)));
    constexpr uint32_t NEG1024 = 0xE400E400u;   // fp16 pair (-1024, -1024)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const uint32_t S = splat_half(__float2half_rn(d * (0.5f + (float)(a[jj] >> 28)) * 0.5f));
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            const uint32_t s7 = (a[jj] >> (7 * l)) & 127u;
            const uint32_t sb = s7 | ((__popc(s7) & 1u) << 7);
            const uint32_t qw = q[2 * jj + (l >> 1)];
            const uint32_t e0 = grid_s[(qw >> (16 * (l & 1))) & 0xffu];
            const uint32_t e1 = grid_s[(qw >> (16 * (l & 1) + 8)) & 0xffu];
#pragma unroll
            for (int t = 0; t < 8; t += 2) {
                const uint32_t e = t < 4 ? e0 : e1;
                const uint32_t m = hadd2(prmt(e, 0x64646464u, (t & 2) ? 0x7362u : 0x5140u), NEG1024);
                const uint32_t sg = ((sb << (15 - t)) & 0x8000u) | ((sb << (30 - t)) & 0x80000000u);
                r[16 * jj + 4 * l + (t >> 1)] = hmul2(m, S ^ sg);
            }
        }
    }
}

// ---- T5_G128 (T5 variant)
// Half HALF of a 128-weight block: weights 64 HALF .. + 63, i.e. code digits
// from 64 HALF on, which begin at digit 4 HALF of code byte 12 HALF. Each code
// byte is split into its five base-3 digits (floor(v / 3) = (v * 171) >> 9 for
// every byte value); digit d of weight t goes into half t % 2 of pair t / 2 as
// the fp16 1024 + d, and (1024 + d) - 1025 = d - 1 and (d - 1) * s are exact.
template <int HALF>
__device__ __forceinline__ void t5_half(uint32_t codes, uint32_t S, uint32_t (&r)[32]) {
    constexpr uint32_t NEG1025 = 0xE401E401u;   // fp16 pair (-1025, -1025)
    uint32_t w[4];
    lds_words<4>(codes + 12 * HALF, w);           // code bytes 12 HALF .. + 15
#pragma unroll
    for (int m = 0; m < 32; ++m) r[m] = TC_MAGIC;
#pragma unroll
    for (int c = 0; c < 14; ++c) {
        uint32_t v = (w[c >> 2] >> (8 * (c & 3))) & 0xffu;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const int t = 5 * c + i - 4 * HALF;   // the piece's weight
            const uint32_t q = (v * 171u) >> 9;
            if (t >= 0 && t < 64) r[t >> 1] |= (v - 3u * q) << (16 * (t & 1));
            v = q;
        }
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) r[m] = hmul2(hadd2(r[m], NEG1025), S);
}
// Piece g = half g % 2 of block g / 2 of the stage (28 bytes each: fp16 s, 26
// code bytes); w = s * (digit - 1).
__device__ __forceinline__ void dq_t5(uint32_t blk, int g, uint32_t (&r)[32]) {
    const uint32_t b = blk + 28 * (g >> 1);
    uint32_t dw[1];
    lds_words<1>(b, dw);
    const uint32_t S = (dw[0] & 0xffffu) * 0x10001u;
    if (g & 1)
        t5_half<1>(b + 2, S, r);
    else
        t5_half<0>(b + 2, S, r);
}

// Raw stage rs of a weight row: the byte offset (within the row) of the first
// block of K range [256 rs, ...), the 16-byte-aligned x of its TMA box and the
// lead of the block inside the box.
__host__ __device__ __forceinline__ void raw_x(int fmt, int rs, int &x0, int &lead) {
    const int s = (rs * TC_KR / blk_elems(fmt)) * blk_bytes(fmt);
    x0 = s & ~15;
    lead = s - x0;
}

// ------------------------------------------------------------------ the grouped GEMM
size_t tc_smem_bytes(int slot_bytes, int RS, bool iq = false) {
    return 1024 + (size_t)TC_BSTAGES * TC_BSTAGE_BYTES + (size_t)RS * slot_bytes + TC_UBUF_FLOATS * 4 +
           TC_NBARS * 8 + 64 + TC_UQ_BYTES + (iq ? TC_GRID_BYTES : 0);
}

struct __align__(16) Unit {
    int e, row0, n, s;   // e < 0: no more units
};

// Units are handed out dynamically: the weight producer takes the next unit
// index from a global counter and publishes the unit in a per-CTA queue in
// shared memory; every other role takes the CTA's units from the queue in the
// same order. (Handing out units round-robin by index left the CTAs finishing
// up to 6% apart.) Four epilogue warps acknowledge each entry, which bounds
// how far the producer runs ahead. The IQ variant publishes the static
// round-robin order through the same queue.
struct UnitQueue {
    Unit *q;             // [TC_UQ]
    uint32_t *n_pub;     // entries published
    uint32_t *n_ack;     // epilogue acknowledgements (4 per entry)
};
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p);
__device__ __noinline__ bool uq_spin_slow(const uint32_t *p, uint32_t target, volatile int *abort_flag);
template <bool INL>
__device__ __forceinline__ bool uq_spin_body(const uint32_t *p, uint32_t target, volatile int *abort_flag);
// Entry k of the queue (bounded wait until it is published).
__device__ __forceinline__ bool uq_get(const UnitQueue &Q, uint32_t k, volatile int *abort_flag, Unit &out) {
    if ((int32_t)(ld_acquire_u32(Q.n_pub) - (k + 1)) < 0 && !uq_spin_slow(Q.n_pub, k + 1, abort_flag)) return false;
    out = Q.q[k % TC_UQ];
    return true;
}

// Unit u: its chunk and slice.
__device__ __forceinline__ Unit load_unit(const TcArgs &A, int u) {
    const int4 ch = A.chunks[u / A.S];
    Unit x{ch.x, ch.y, ch.z, u % A.S};
    return x;
}

// The CTA's k-th unit (e = -1 once all are handed out) and its weight format:
// the next one from the global counter (DYN), or unit blockIdx.x + k * grid.
template <bool GATEUP, bool DYN>
__device__ __forceinline__ Unit grab_unit(const TcArgs &A, int n_units, uint32_t k, int &fmt) {
    const int u = DYN ? atomicAdd(A.unit_next, 1) : (int)(blockIdx.x + k * gridDim.x);
    fmt = 0;
    if (u >= n_units) {
        Unit x{-1, 0, 0, 0};
        return x;
    }
    const Unit x = load_unit(A, u);
    fmt = GATEUP ? A.table[x.e].gate.fmt : A.table[x.e].down.fmt;
    return x;
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = tc_wait(bar, parity, abort_flag);
    return __shfl_sync(0xffffffffu, ok, 0);
}
// Entry k of the unit queue for a whole warp: lane 0 waits, every lane reads.
template <bool INL = false>
__device__ __forceinline__ bool warp_uq_get(const UnitQueue &Q, uint32_t k, volatile int *abort_flag, Unit &out) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = (int32_t)(ld_acquire_u32(Q.n_pub) - (k + 1)) >= 0 ||
             (INL ? uq_spin_body<true>(Q.n_pub, k + 1, abort_flag) : uq_spin_slow(Q.n_pub, k + 1, abort_flag));
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
        (void)ld_acquire_u32(Q.n_pub);   // every lane acquires the published entries
        out = Q.q[k % TC_UQ];
    }
    return ok;
}

// AND of `pred` over the 128 epilogue threads (warps 0-3), with a barrier.
__device__ __forceinline__ bool epi_all(bool pred) {
    uint32_t r;
    __syncwarp();   // the barrier is .aligned: reconverge the warp first
    asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, 1, 128, p; selp.u32 %0, 1, 0, q; }"
                 : "=r"(r)
                 : "r"((uint32_t)pred)
                 : "memory");
    return r != 0;
}
__device__ __forceinline__ void epi_sync() {
    __syncwarp();   // the barrier is .aligned: reconverge the warp first
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// A steps per B stage for a unit of n rows (Npad = n rounded up to 16): 4 if
// four Npad-row tiles fit a stage, else 2. Either divides an event.
__device__ __forceinline__ int b_steps_per_stage(int n) {
    const int npad = (n + 15) & ~15;
    return npad <= 64 ? 4 : 2;
}

__device__ __forceinline__ uint32_t ld_acquire_shared(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) { return ld_acquire_shared(p); }
// Spin until the counter reaches `target` (wrapping compare), with a sleep
// between polls; bounded like the other waits. One out-of-line copy for most
// roles; the epilogue inlines it (as a call it made the epilogue spill
// registers around it).
template <bool INL>
__device__ __forceinline__ bool uq_spin_body(const uint32_t *p, uint32_t target, volatile int *abort_flag) {
    const uint64_t t0 = global_ns(), bound = *(volatile unsigned long long *)&g_wait_ns;
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if ((int32_t)(ld_acquire_shared(p) - target) >= 0) return true;
        if ((i & 15u) == 15u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > bound) return false;
        }
        __nanosleep(64);
    }
    return false;
}
__device__ __noinline__ bool uq_spin_slow(const uint32_t *p, uint32_t target, volatile int *abort_flag) {
    return uq_spin_body<false>(p, target, abort_flag);
}
__device__ __forceinline__ void red_release_shared(uint32_t *p, uint32_t v) {
    asm volatile("red.release.cta.shared.add.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __noinline__ bool counter_spin_slow(const uint32_t *p, uint32_t target, volatile int *abort_flag) {
    const uint64_t t0 = global_ns(), bound = *(volatile unsigned long long *)&g_wait_ns;
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if ((int32_t)(ld_acquire_shared(p) - target) >= 0) return true;
        if ((i & 1023u) == 1023u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > bound) return false;
        }
    }
    return false;
}
__device__ __forceinline__ bool counter_spin(const uint32_t *p, uint32_t target, volatile int *abort_flag) {
    return (int32_t)(ld_acquire_shared(p) - target) >= 0 || counter_spin_slow(p, target, abort_flag);
}

template <bool GATEUP, int XV>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap bmap, const TcArgs A) {
    extern __shared__ __align__(16) uint8_t tc_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *bring = sm;
    uint8_t *raw = bring + TC_BSTAGES * TC_BSTAGE_BYTES;
    float *ubuf = reinterpret_cast<float *>(raw + (size_t)A.RS * A.slot_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ubuf + TC_UBUF_FLOATS);
    uint64_t *raw_full = bars, *raw_empty = bars + TC_RS_MAX;
    uint64_t *a_empty = bars + 2 * TC_RS_MAX;   // per event slot, committed by the MMA thread
    uint64_t *b_full = a_empty + TC_EVSLOTS, *b_empty = b_full + TC_BSTAGES;
    uint64_t *acc_full = b_empty + TC_BSTAGES, *acc_empty = acc_full + 2, *fin = acc_empty + 2;
    uint32_t *raw_info = reinterpret_cast<uint32_t *>(bars + TC_NBARS);  // [TC_RS_MAX]: fmt | lead << 8
    uint32_t *a_ready = raw_info + TC_RS_MAX;   // [TC_EVSLOTS]: dequant warps done, 16 per use
    uint32_t *tmem_slot = a_ready + TC_EVSLOTS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // after the 64-byte misc area: the unit queue (16-byte aligned), then the
    // IQ3_XXS grid (IQ variants)
    uint8_t *qbase = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(reinterpret_cast<uint8_t *>(bars + TC_NBARS) + 64) + 15) & ~(uintptr_t)15);
    const UnitQueue Q{reinterpret_cast<Unit *>(qbase), reinterpret_cast<uint32_t *>(qbase + TC_UQ * 16),
                      reinterpret_cast<uint32_t *>(qbase + TC_UQ * 16) + 1};
    uint32_t *grid_s = reinterpret_cast<uint32_t *>(qbase + TC_UQ * 16 + 16);
    if (XV != TC_XV_STD && A.grid)
        for (int i = threadIdx.x; i < 256; i += TC_THREADS) grid_s[i] = A.grid[i];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int R = GATEUP ? 64 : 128;          // weight rows per matrix box
    constexpr int NMAT = GATEUP ? 2 : 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < A.RS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 4 * TC_DG);
        }
        for (int i = 0; i < TC_EVSLOTS; ++i) {
            mbar_init(&a_empty[i], 1);
            a_ready[i] = 0;
        }
        for (int i = 0; i < TC_BSTAGES; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(fin, 1);
        *abort_flag = 0;
        *Q.n_pub = 0;
        *Q.n_ack = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_units = *A.n_chunks * A.S;
    const int nR = (A.K + TC_KR - 1) / TC_KR, nA = A.K / TC_KA;

    if (warp == TC_PROD) {
        // ---- weight producer: takes the CTA's units from the global counter and
        // publishes them; per raw stage one 2-D TMA box per matrix (two for Q8_0).
        // It runs ahead of the consumers by the raw ring, which hides the
        // chunk-table loads of each new unit.
        if (lane == 0) {
            uint32_t rg = 0;
            bool ok = true;
            for (uint32_t k = 0; ok; ++k) {
                int fmt;
                // dynamic order (measured per 2048-token layer: 793 -> 775 us,
                // and 902 -> 878 us for the ternary 512-token layer); the IQ
                // variant keeps the static order, with which its layer measured
                // 918 us against 945 us dynamic
                const Unit cu = grab_unit<GATEUP, (XV != TC_XV_IQ)>(A, n_units, k, fmt);
                // entry k reuses the slot of entry k - TC_UQ: wait until the four
                // epilogue warps have taken that one
                if (k >= TC_UQ) {
                    const uint32_t need = 4u * (k - TC_UQ + 1);
                    if ((int32_t)(ld_acquire_shared(Q.n_ack) - need) < 0 && !uq_spin_slow(Q.n_ack, need, abort_flag)) {
                        ok = false;
                        break;
                    }
                }
                Q.q[k % TC_UQ] = cu;
                red_release_shared(Q.n_pub, 1u);
                if (cu.e < 0) break;
                const int W = raw_w(fmt), nbox = raw_nbox(fmt);
                const uint32_t bytes = (uint32_t)(NMAT * nbox * R * W);
                const CUtensorMap *m0 = A.wmaps + 3 * cu.e + (GATEUP ? 0 : 2);
                for (int rs = 0; rs < nR; ++rs) {
                    const uint32_t slot = rg % A.RS, use = rg / A.RS;
                    if (use > 0 && !tc_wait(&raw_empty[slot], (use - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    int x0, lead;
                    raw_x(fmt, rs, x0, lead);
                    raw_info[slot] = (uint32_t)fmt | ((uint32_t)lead << 8);
                    mbar_expect_tx(&raw_full[slot], bytes);
                    uint8_t *dst = raw + (size_t)slot * A.slot_bytes;
                    for (int m = 0; m < NMAT; ++m)
                        for (int b = 0; b < nbox; ++b)
                            tma_load_2d(dst + (m * nbox + b) * R * W, m0 + m, x0 + 128 * b, R * cu.s,
                                        &raw_full[slot]);
                    ++rg;
                }
            }
            if (!ok) {
                tc_fail(abort_flag, A.status);
                for (uint32_t j = rg > (uint32_t)A.RS ? rg - A.RS : 0; j < rg; ++j)
                    mbar_wait(&raw_full[j % A.RS], (j / A.RS) & 1);
            }
        }
    } else if (warp == TC_BPROD) {
        // ---- activation producer: q A steps of the unit's rows per B stage. Lane 0
        // waits for the stage to be free and sets its byte count; then the warp's
        // lanes issue the stage's boxes, one each (a single thread issuing a
        // stage's dozen boxes back to back left the MMA issuer waiting on B).
        uint32_t bg = 0;
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            Unit cu;
            if (!warp_uq_get(Q, k, abort_flag, cu)) {
                ok = false;
                break;
            }
            if (cu.e < 0) break;
            const int nb = (cu.n + TC_BOX_ROWS - 1) / TC_BOX_ROWS, q = b_steps_per_stage(cu.n);
            const int sub_bytes = nb * TC_BOX_ROWS * 128;
            for (int a0 = 0; a0 < nA; a0 += q) {
                const uint32_t bs = bg % TC_BSTAGES, buse = bg / TC_BSTAGES;
                if (buse > 0 && !warp_wait(&b_empty[bs], (buse - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int qa = min(q, nA - a0);
                if (lane == 0) mbar_expect_tx(&b_full[bs], (uint32_t)(qa * sub_bytes));
                __syncwarp();
                for (int t = lane; t < qa * nb; t += 32) {
                    const int j = t / nb, i = t - j * nb;
                    tma_load_2d(bring + bs * TC_BSTAGE_BYTES + j * sub_bytes + i * TC_BOX_ROWS * 128, &bmap,
                                (a0 + j) * TC_KA, cu.row0 + i * TC_BOX_ROWS, &b_full[bs]);
                }
                ++bg;
            }
        }
        if (!ok && lane == 0) {
            tc_fail(abort_flag, A.status);
            for (uint32_t j = bg > (uint32_t)TC_BSTAGES ? bg - TC_BSTAGES : 0; j < bg; ++j)
                mbar_wait(&b_full[j % TC_BSTAGES], (j / TC_BSTAGES) & 1);
        }
    } else if (warp == TC_MMA) {
        // ---- MMA issuer: one thread; per event (raw stage) one wait on the dequantisers'
        // counter, then per B stage (one of 4 A steps, or two of 2 when the chunk has more
        // than 64 rows) one wait and its MMAs back to back, then one commit
        if (lane == 0) {
            uint32_t ev = 0, bg = 0, uc = 0;
            bool ok = true, issued = false;
            for (uint32_t k = 0; ok; ++k) {
                Unit cu;
                if (!uq_get(Q, k, abort_flag, cu)) {
                    ok = false;
                    break;
                }
                if (cu.e < 0) break;
                const int N = (cu.n + 15) & ~15, q = b_steps_per_stage(cu.n);
                const uint32_t idesc = idesc_f16(N);
                const uint32_t sub_step = (uint32_t)(N * 128) >> 4;   // descriptor units per B tile
                const uint32_t d = uc & 1, use = uc >> 1;
                if (use > 0 && !tc_wait(&acc_empty[d], (use - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tmem_fence_after();
                const uint32_t dcol = tmem + d * TC_NCHUNK;
                for (int rs = 0; rs < nR; ++rs) {
                    const int na = min(TC_AEV, nA - TC_AEV * rs);
                    const uint32_t slot = ev & (TC_EVSLOTS - 1);
                    if (!counter_spin(&a_ready[slot], 4u * TC_DG * ((ev >> 1) + 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tmem_fence_after();
                    const uint32_t acol0 = tmem + TC_ACOL0 + slot * (TC_AEV * 32);
                    // the raw stage's B stages: one of 4 A steps (q = 4) or two of 2
                    for (int h0 = 0; h0 < na; h0 += q) {
                        const uint32_t bs = bg % TC_BSTAGES;
                        if (!tc_spin(&b_full[bs], (bg / TC_BSTAGES) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tmem_fence_after();
                        const uint64_t bd = smem_desc_sw128(smem_addr(bring + bs * TC_BSTAGE_BYTES));
                        const int nh = min(q, na - h0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (i < nh) {
                                const uint32_t acol = acol0 + 32 * (h0 + i);
                                const uint32_t blo = (uint32_t)bd + (uint32_t)(i * sub_step), bhi = (uint32_t)(bd >> 32);
                                if ((rs | h0 | i) != 0)
                                    mma_f16_ts_acc(dcol, acol, blo, bhi, idesc);
                                else
                                    mma_f16_ts(dcol, acol, bd, idesc, 0);   // the unit's first: overwrite D
                                mma_f16_ts_acc(dcol, acol + 8, blo + 2, bhi, idesc);
                                mma_f16_ts_acc(dcol, acol + 16, blo + 4, bhi, idesc);
                                mma_f16_ts_acc(dcol, acol + 24, blo + 6, bhi, idesc);
                            }
                        }
                        issued = true;   // before any later wait can give up: TMEM is freed only after these complete
                        mma_commit(&b_empty[bs]);
                        ++bg;
                    }
                    if (!ok) break;
                    mma_commit(&a_empty[slot]);
                    ++ev;
                }
                if (!ok) break;
                mma_commit(&acc_full[d]);
                ++uc;
            }
            if (!ok) tc_fail(abort_flag, A.status);
            if (issued) {
                // every MMA has completed before TMEM is released
                mma_commit(fin);
                mbar_wait(fin, 0);
            }
        }
    } else if (warp >= TC_DQ0) {
        // ---- dequantisers: group g writes piece g (64 K) of every raw stage to TMEM
        const int g = (warp - TC_DQ0) >> 2, qd = warp & 3, l = 32 * qd + lane;
        const int mat = GATEUP ? (l >> 6) : 0, row = GATEUP ? (l & 63) : l;
        uint32_t rg = 0;   // raw stages = events seen
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            Unit cu;
            if (!warp_uq_get(Q, k, abort_flag, cu)) {
                ok = false;
                break;
            }
            if (cu.e < 0) break;
            for (int rs = 0; rs < nR; ++rs) {
                const uint32_t slot = rg % A.RS, es = rg & (TC_EVSLOTS - 1), euse = rg >> 1;
                if (!warp_wait(&raw_full[slot], (rg / A.RS) & 1, abort_flag) ||
                    (euse > 0 && !warp_wait(&a_empty[es], (euse - 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int pp = 0; pp < TC_PPG; ++pp) {
                const int gp = g + TC_DG * pp;   // the piece this warp decodes
                const int a = TC_AEV * rs + gp;
                if (a < nA) {
                    tmem_fence_after();
                    const uint32_t info = raw_info[slot];
                    const int fmt = info & 0xff, lead = info >> 8;
                    const int W = raw_w(fmt), nbox = raw_nbox(fmt);
                    const uint32_t tile = smem_addr(raw + (size_t)slot * A.slot_bytes) + (uint32_t)(mat * nbox * R * W);
                    const uint32_t base = tile + (uint32_t)(row * W + lead);
                    uint32_t r[32];
                    if (fmt == MOE_Q4_K)
                        dq_q4k(base, gp, r);
                    else if (fmt == MOE_Q8_0)
                        dq_q8_0(gp < 2 ? base + 68 * gp : base + (uint32_t)(R * W) + 68 * gp - 128, r);
                    else if (fmt == MOE_Q6_K)
                        dq_q6k(base, gp, r);
                    else if (XV == TC_XV_STD || fmt == MOE_MXFP4)
                        dq_mxfp4(base, gp, r);
                    else if (fmt == MOE_IQ4_NL)
                        dq_iq4nl(base, gp, r);
                    else if (fmt == MOE_IQ4_XS)
                        dq_iq4xs(base, gp, r);
                    else if (XV == TC_XV_IQ || fmt == MOE_IQ3_XXS)
                        dq_iq3xxs(base, gp, grid_s, r);
                    else
                        dq_t5(base, gp, r);
                    tmem_st32(tmem + ((uint32_t)(32 * qd) << 16) + TC_ACOL0 + es * (TC_AEV * 32) + gp * 32, r);
                }
                }
                tmem_wait_st();
                tmem_fence_before();
                __syncwarp();
                if (lane == 0) {
                    red_release_shared(&a_ready[es], 1u);
                    mbar_arrive_cta(&raw_empty[slot]);
                }
                ++rg;
            }
        }
        if (!ok && lane == 0) tc_fail(abort_flag, A.status);
    } else {
        // ---- epilogue: warps 0-3 read TMEM lanes 32w..32w+31
        const int l = 32 * warp + lane;
        uint32_t uc = 0;
        for (uint32_t k = 0;; ++k) {
            Unit cu;
            bool ok = warp_uq_get<true>(Q, k, abort_flag, cu);
            if (ok) {
                __syncwarp();   // every lane has read entry k
                if (lane == 0) red_release_shared(Q.n_ack, 1u);
            }
            const bool more = ok && cu.e >= 0;
            const int n = cu.n, row0 = cu.row0, s = cu.s;
            const uint32_t d = uc & 1;
            if (more) ok = warp_wait(&acc_full[d], (uc >> 1) & 1, abort_flag);
            // the gate/up epilogue's warps meet at barriers: they leave together
            if (GATEUP) ok = epi_all(ok);
            if (!ok) {
                if (lane == 0) tc_fail(abort_flag, A.status);
                break;
            }
            if (!more) break;   // the end of the queue (the same entry for every warp)
            tmem_fence_after();
            if (GATEUP) {
                // 16 columns at a time: every lane's g or u to shared memory, then
                // thread l computes h for row l & 63 and 8 of the columns
                const int r = l & 63, ch = l >> 6;
                for (int cb = 0; cb < n; cb += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + d * TC_NCHUNK + cb, v);
                    const int jn = min(16, n - cb);
                    const float scl = lane < jn ? A.ascale[row0 + cb + lane] : 0.0f;
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) ubuf[j * 128 + l] = __uint_as_float(v[j]);
                    epi_sync();
                    float hv[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = 8 * ch + jj;
                        const float sc = __shfl_sync(0xffffffffu, scl, j);
                        hv[jj] = silu_fast(ubuf[j * 128 + r] * sc) * (ubuf[j * 128 + 64 + r] * sc);
                    }
                    float *hrow = A.h32 + (size_t)(row0 + cb + 8 * ch) * A.I + 64 * s + r;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        if (8 * ch + jj < jn) hrow[(size_t)jj * A.I] = hv[jj];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) hv[jj] = fabsf(hv[jj]);
                    const float m = warp_colmax8(hv);
                    if (lane < 8 && 8 * ch + lane < jn) atomicMax(&A.hmax[row0 + cb + 8 * ch + lane], __float_as_uint(m));
                    epi_sync();
                }
            } else {
                // D as it is: the combine applies the h row's power-of-two
                // scale (exact, so the output is bit for bit the same), and
                // the epilogue only moves the accumulator (2048-token layer:
                // 762 -> 754 us)
                for (int cb = 0; cb < n; cb += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + d * TC_NCHUNK + cb, v);
                    const int jn = min(32, n - cb);
                    tmem_wait_ld();
                    float *yrow = A.y + (size_t)(row0 + cb) * A.H + TC_M * s + l;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn) yrow[(size_t)j * A.H] = __uint_as_float(v[j]);
                }
            }
            tmem_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cta(&acc_empty[d]);
            ++uc;
        }
    }

    tmem_fence_before();
    __syncthreads();
    if (warp == 0) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------------ preparation kernels
constexpr int PREP_THREADS = 256;

// sigma with maxabs * 2^sigma in [2^14, 2^15): fp16 keeps 11 significant bits
// of every value within 2^-10 of the row's largest and cannot overflow.
__device__ __forceinline__ int row_shift(float maxabs) {
    if (!(maxabs > 0.0f) || !isfinite(maxabs)) return 0;
    int e;
    frexpf(maxabs, &e);  // maxabs = f * 2^e, f in [0.5, 1)
    return max(-120, min(120, 15 - e));
}
__device__ __forceinline__ float pow2f(int s) { return ldexpf(1.0f, s); }

__device__ __forceinline__ float block_max(float v, float *red) {
    v = warp_max_f(v);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[w] = v;
    __syncthreads();
    if (w == 0) {
        v = lane < PREP_THREADS / 32 ? red[lane] : 0.0f;
        v = warp_max_f(v);
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

// Blocks 0..T-1: token t's bf16 row -> fp16 scaled by 2^sigma_t, copied to the
// bucket row of each of its kept pairs (so every expert's rows are contiguous
// for the B tiles); that row's inverse scale; its |h| maximum cleared.
// Block T: the chunk table, <= 128 bucket rows of one expert per chunk, in
// ascending expert order; and the two GEMMs' unit counters, zeroed.
__global__ void __launch_bounds__(PREP_THREADS) tc_prep_kernel(const uint16_t *__restrict__ x, int T, int k, int H,
                                                               int E, const int32_t *__restrict__ pos,
                                                               const int32_t *__restrict__ offsets,
                                                               const int32_t *__restrict__ active, __half *xg,
                                                               float *xinv, uint32_t *hmax, int4 *chunks,
                                                               int32_t *n_chunks, int32_t *unit_next) {
    __shared__ float red[PREP_THREADS / 32];
    __shared__ int scan[PREP_THREADS];
    if ((int)blockIdx.x < T) {
        const int t = blockIdx.x;
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        const int n8 = H / 8;
        float m = 0.0f;
        for (int i = threadIdx.x; i < n8; i += PREP_THREADS) {
            const uint4 v = xr[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
        }
        m = block_max(m, red);
        const int sg = row_shift(m);
        const float sc = pow2f(sg), inv = pow2f(-sg);
        for (int j = 0; j < k; ++j) {
            const int q = pos[(size_t)t * k + j];
            if (q < 0) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(xg + (size_t)q * H);
            for (int i = threadIdx.x; i < n8; i += PREP_THREADS) {
                const uint4 v = xr[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const __half2 h2 = __floats2half2_rn(__uint_as_float(w[jj] << 16) * sc,
                                                         __uint_as_float(w[jj] & 0xffff0000u) * sc);
                    o[jj] = *reinterpret_cast<const uint32_t *>(&h2);
                }
                dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            if (threadIdx.x == 0) {
                xinv[q] = inv;
                hmax[q] = 0u;
            }
        }
        return;
    }
    // chunk table
    const int n_act = active[0];
    int total = 0;
    for (int base = 0; base < n_act; base += PREP_THREADS) {
        const int i = base + threadIdx.x;
        int e = 0, cnt = 0, nch = 0;
        if (i < n_act) {
            e = active[1 + i];
            cnt = offsets[e + 1] - offsets[e];
            nch = (cnt + TC_NCHUNK - 1) / TC_NCHUNK;
        }
        scan[threadIdx.x] = nch;
        __syncthreads();
        for (int o = 1; o < PREP_THREADS; o <<= 1) {
            const int v = threadIdx.x >= o ? scan[threadIdx.x - o] : 0;
            __syncthreads();
            scan[threadIdx.x] += v;
            __syncthreads();
        }
        const int first = total + scan[threadIdx.x] - nch;
        for (int c = 0; c < nch; ++c)
            chunks[first + c] = make_int4(e, offsets[e] + c * TC_NCHUNK, min(TC_NCHUNK, cnt - c * TC_NCHUNK), 0);
        total += scan[PREP_THREADS - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *n_chunks = total;
        unit_next[0] = 0;
        unit_next[1] = 0;
    }
}

// One warp per bucket row: h (fp32) -> fp16 scaled by 2^sigma from the row's
// |h| maximum, and the inverse scale.
__global__ void __launch_bounds__(PREP_THREADS) tc_hprep_kernel(const float *__restrict__ h32,
                                                                const uint32_t *__restrict__ hmax,
                                                                const int32_t *__restrict__ offsets, int E, int I,
                                                                __half *h16, float *hinv) {
    const int q = blockIdx.x * (PREP_THREADS / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (q >= offsets[E]) return;
    const int sg = row_shift(__uint_as_float(hmax[q]));
    const float sc = pow2f(sg);
    const float4 *src = reinterpret_cast<const float4 *>(h32 + (size_t)q * I);
    uint2 *dst = reinterpret_cast<uint2 *>(h16 + (size_t)q * I);
    for (int i = lane; i < I / 4; i += 32) {
        const float4 v = src[i];
        const __half2 a = __floats2half2_rn(v.x * sc, v.y * sc), b = __floats2half2_rn(v.z * sc, v.w * sc);
        dst[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
    }
    if (lane == 0) hinv[q] = pow2f(-sg);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// fp16 matrix [rows][cols] row-major: boxes of 64 columns (128 bytes) x 16
// rows, 128-byte swizzle, zero fill outside.
bool encode_act_map(CUtensorMap *map, const void *base, int rows, int cols) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {TC_KA, TC_BOX_ROWS};
    const cuuint32_t es[2] = {1, 1};
    return f(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of one raw stage for the formats in `fmask`: per weight matrix of the
// unit, its box(es) of R rows x raw_w bytes.
int raw_slot_bytes(uint32_t fmask, bool gateup) {
    const int R = gateup ? 64 : 128, nmat = gateup ? 2 : 1;
    int sb = 0;
    for (int f = MOE_Q8_0; f <= MOE_T5_G128; ++f)
        if (fmask & (1u << f)) sb = std::max(sb, nmat * raw_nbox(f) * R * raw_w(f));
    return sb;
}

int g_tc_smem_optin[64] = {};

int smem_optin() {
    const int dev = current_device();
    if (dev < 64 && g_tc_smem_optin[dev]) return g_tc_smem_optin[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    const void *kernels[6] = {(const void *)tc_gemm_kernel<true, TC_XV_STD>, (const void *)tc_gemm_kernel<false, TC_XV_STD>,
                              (const void *)tc_gemm_kernel<true, TC_XV_IQ>, (const void *)tc_gemm_kernel<false, TC_XV_IQ>,
                              (const void *)tc_gemm_kernel<true, TC_XV_T5>, (const void *)tc_gemm_kernel<false, TC_XV_T5>};
    for (const void *kf : kernels)
        if (cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, v) != cudaSuccess) return 0;
    if (dev < 64) g_tc_smem_optin[dev] = v;
    return v;
}

// Raw ring depth that fits next to the fixed shared memory; 0 if < 2.
int raw_stages(int slot_bytes, bool iq) {
    const int optin = smem_optin();
    if (optin <= 0 || slot_bytes <= 0) return 0;
    const long room = (long)optin - (long)tc_smem_bytes(slot_bytes, 0, iq);
    long rs = room / slot_bytes;
    if (rs > TC_RS_MAX) rs = TC_RS_MAX;
    return rs >= 2 ? (int)rs : 0;
}

}  // namespace

bool tc_path_eligible(int H, int I) { return H >= TC_M && H % TC_M == 0 && I >= 64 && I % 64 == 0; }

size_t tc_weight_map_bytes(int E) { return (size_t)E * 3 * sizeof(CUtensorMap); }

// The tensor path's weight tensor maps, 3 per expert (gate, up, down) into
// `out` (host memory, tc_weight_map_bytes(E) bytes): the matrix's bytes as a
// 2-D uint8 tensor [rows][row stride], boxes of raw_w(format) bytes x 64 rows
// (gate/up) or 128 rows (down). False if the driver refuses one.
bool tc_encode_weight_maps(const moe_weight_table *W, void *out) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    CUtensorMap *maps = static_cast<CUtensorMap *>(out);
    for (int e = 0; e < W->n_experts + W->n_shared; ++e) {
        const moe_matrix *m[3] = {&W->experts[e].gate, &W->experts[e].up, &W->experts[e].down};
        for (int i = 0; i < 3; ++i) {
            const cuuint64_t dims[2] = {(cuuint64_t)m[i]->row_stride_bytes, (cuuint64_t)m[i]->rows};
            const cuuint64_t strides[1] = {(cuuint64_t)m[i]->row_stride_bytes};
            const cuuint32_t box[2] = {(cuuint32_t)raw_w(m[i]->format), (cuuint32_t)(i < 2 ? 64 : 128)};
            const cuuint32_t es[2] = {1, 1};
            if (f(&maps[3 * e + i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(m[i]->data), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
        }
    }
    return true;
}

cudaError_t launch_tc_path(const DevExpert *table, const void *wmaps, uint32_t gu_formats, uint32_t dn_formats,
                           const uint32_t *grid, int T, int k, int E,
                           int H, int I, const int32_t *offsets, const int32_t *active, const int32_t *pos,
                           const float *wts, const uint16_t *x, float *h32, float *y, char *ws_base,
                           const TcLayout &C, float *out, uint32_t *status, cudaEvent_t const *events,
                           cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int P = T * k;
    const int sb1 = raw_slot_bytes(gu_formats, true), sb2 = raw_slot_bytes(dn_formats, false);
    // layers with IQ or T5_G128 formats take a kernel variant with their
    // decoders (and the IQ3_XXS grid in shared memory); the others keep the
    // smaller code
    const uint32_t fm = gu_formats | dn_formats;
    const int xv = (fm & (1u << MOE_T5_G128)) ? TC_XV_T5 : (fm & TC_IQ_FORMATS) ? TC_XV_IQ : TC_XV_STD;
    const bool iq = xv != TC_XV_STD;
    if ((fm & (1u << MOE_IQ3_XXS)) && !grid) return cudaErrorInvalidValue;
    const int rs1 = raw_stages(sb1, iq), rs2 = raw_stages(sb2, iq);
    const CUtensorMap *maps = static_cast<const CUtensorMap *>(wmaps);
    const int G = sm_count();
    if (!rs1 || !rs2 || G <= 0) return cudaErrorInvalidConfiguration;
    __half *xg = reinterpret_cast<__half *>(ws_base + C.xg);
    __half *h16 = reinterpret_cast<__half *>(ws_base + C.h16);
    float *xinv = reinterpret_cast<float *>(ws_base + C.xinv);
    float *hinv = reinterpret_cast<float *>(ws_base + C.hinv);
    uint32_t *hmax = reinterpret_cast<uint32_t *>(ws_base + C.hmax);
    int4 *chunks = reinterpret_cast<int4 *>(ws_base + C.chunks);
    int32_t *n_chunks = reinterpret_cast<int32_t *>(ws_base + C.n_chunks);
    int32_t *unit_next = reinterpret_cast<int32_t *>(ws_base + C.unit_next);
    CUtensorMap xmap, hmap;
    if (!encode_act_map(&xmap, xg, P, H) || !encode_act_map(&hmap, h16, P, I)) return cudaErrorInvalidValue;

    cudaError_t err;
    tc_prep_kernel<<<T + 1, PREP_THREADS, 0, s>>>(x, T, k, H, E, pos, offsets, active, xg, xinv, hmax, chunks,
                                                   n_chunks, unit_next);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (events && (err = record_event(events[0], s)) != cudaSuccess) return err;

    TcArgs a1{table, maps, chunks, n_chunks, H, I / 64, H, I, sb1, rs1, xinv, h32, hmax, nullptr, status, grid,
              unit_next};
    const size_t smem1 = tc_smem_bytes(sb1, rs1, iq);
    if (xv == TC_XV_T5)
        tc_gemm_kernel<true, TC_XV_T5><<<G, TC_THREADS, smem1, s>>>(xmap, a1);
    else if (xv == TC_XV_IQ)
        tc_gemm_kernel<true, TC_XV_IQ><<<G, TC_THREADS, smem1, s>>>(xmap, a1);
    else
        tc_gemm_kernel<true, TC_XV_STD><<<G, TC_THREADS, smem1, s>>>(xmap, a1);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (events && (err = record_event(events[1], s)) != cudaSuccess) return err;

    tc_hprep_kernel<<<(P + PREP_THREADS / 32 - 1) / (PREP_THREADS / 32), PREP_THREADS, 0, s>>>(h32, hmax, offsets, E,
                                                                                             I, h16, hinv);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    TcArgs a2{table, maps, chunks, n_chunks, I, H / TC_M, H, I, sb2, rs2, hinv, nullptr, nullptr, y, status, grid,
              unit_next + 1};
    const size_t smem2 = tc_smem_bytes(sb2, rs2, iq);
    if (xv == TC_XV_T5)
        tc_gemm_kernel<false, TC_XV_T5><<<G, TC_THREADS, smem2, s>>>(hmap, a2);
    else if (xv == TC_XV_IQ)
        tc_gemm_kernel<false, TC_XV_IQ><<<G, TC_THREADS, smem2, s>>>(hmap, a2);
    else
        tc_gemm_kernel<false, TC_XV_STD><<<G, TC_THREADS, smem2, s>>>(hmap, a2);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (events && (err = record_event(events[2], s)) != cudaSuccess) return err;
    return launch_combine(T, k, H, pos, wts, y, out, s, hinv);
}

// This file's copy of the wait bound (moe_set_wait_timeout_ns).
cudaError_t set_wait_ns_tc(unsigned long long ns) { return set_tu_wait_ns(ns); }

}  // namespace moe
