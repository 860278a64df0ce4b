// GPU filler for the seeded synthetic weights: the same recipe as the numpy
// generator in synth/__init__.py (SplitMix64 draws at the field offsets of
// each block format). Input generation for tests and benchmarks only.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_synth.h"

namespace {

constexpr uint64_t GAMMA = 0x9E3779B97F4A7C15ull;
constexpr int DRAWS_PER_BLOCK = 32;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

// f16(lo + span * u24(r)): one fp32 multiply and one fp32 add, each rounded to
// nearest even, then fp16 rounding to nearest even. The constants are the
// fp32 roundings of the double literals, as numpy's float32(x) makes them.
__device__ __forceinline__ uint16_t f16_uniform(uint64_t r, float lo, float span) {
    const float u = (float)(r >> 40) * 5.9604644775390625e-08f;  // 2^-24, exact
    const float v = __fadd_rn(lo, __fmul_rn(span, u));
    unsigned short h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
    return h;
}

// fp16 fields sit at even offsets of 16-byte aligned rows: one 16-bit store.
__device__ __forceinline__ void put16(uint8_t *p, uint16_t v) { *reinterpret_cast<uint16_t *>(p) = v; }

__device__ __forceinline__ int ubelow16(uint64_t chunk, uint64_t n) { return (int)((chunk * n) >> 16); }

__device__ __forceinline__ uint8_t byte_of(uint64_t r, int i) { return (uint8_t)(r >> (8 * i)); }

__global__ void synth_fill_kernel(const moe_synth_matrix *__restrict__ descs) {
    const moe_synth_matrix M = descs[blockIdx.y];
    const int be = (M.format == 2 || M.format == 3 || M.format == 6 || M.format == 7) ? 256
                 : M.format == 8 ? 128 : 32;
    const int bb = M.format == 1 ? 34 : M.format == 2 ? 144 : M.format == 3 ? 210 : M.format == 4 ? 17
                 : M.format == 5 ? 18 : M.format == 6 ? 136 : M.format == 7 ? 98 : 28;
    const int nb = M.cols / be;
    const int64_t nblocks = (int64_t)M.rows * nb;
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const int row = (int)(b / nb), j = (int)(b - (int64_t)row * nb);
    uint8_t *out = static_cast<uint8_t *>(M.data) + (int64_t)row * M.row_stride_bytes + (int64_t)j * bb;
    const uint64_t base = (uint64_t)b * DRAWS_PER_BLOCK;
    const uint64_t key = M.key;

    if (M.format == 1) {  // Q8_0
        put16(out, f16_uniform(draw(key, base + 0), (float)0.002, (float)0.018));
        for (int g = 0; g < 8; ++g) {
            uint64_t r = draw(key, base + 1 + g);
            for (int c = 0; c < 4; ++c) out[2 + 4 * g + c] = (uint8_t)(ubelow16((r >> (16 * c)) & 0xFFFF, 255) - 127);
        }
    } else if (M.format == 2) {  // Q4_K
        put16(out, f16_uniform(draw(key, base + 0), (float)0.0005, (float)0.0045));
        put16(out + 2, f16_uniform(draw(key, base + 1), (float)0.0005, (float)0.0045));
        for (int g = 0; g < 18; ++g) {
            uint64_t r = draw(key, base + 2 + g);
            for (int c = 0; c < 8; ++c) {
                int i = 8 * g + c;
                if (i < 140) out[4 + i] = byte_of(r, c);
            }
        }
    } else if (M.format == 3) {  // Q6_K
        for (int g = 0; g < 24; ++g) {
            uint64_t r = draw(key, base + g);
            for (int c = 0; c < 8; ++c) out[8 * g + c] = byte_of(r, c);
        }
        for (int g = 0; g < 4; ++g) {
            uint64_t r = draw(key, base + 24 + g);
            for (int c = 0; c < 4; ++c)
                out[192 + 4 * g + c] = (uint8_t)(ubelow16((r >> (16 * c)) & 0xFFFF, 255) - 127);
        }
        put16(out + 208, f16_uniform(draw(key, base + 28), (float)1e-4, (float)9e-4));
    } else if (M.format == 4) {  // MXFP4
        uint64_t r0 = draw(key, base + 0);
        out[0] = (uint8_t)(124 + (((r0 & 0xFFFFFFFFull) * 3ull) >> 32));
        for (int g = 0; g < 2; ++g) {
            uint64_t r = draw(key, base + 1 + g);
            for (int c = 0; c < 8; ++c) out[1 + 8 * g + c] = byte_of(r, c);
        }
    } else if (M.format == 5) {  // IQ4_NL (fp16 d at an even offset of the 16-aligned row: 18 j is even)
        put16(out, f16_uniform(draw(key, base + 0), (float)0.002, (float)0.018));
        for (int g = 0; g < 2; ++g) {
            uint64_t r = draw(key, base + 1 + g);
            for (int c = 0; c < 8; ++c) out[2 + 8 * g + c] = byte_of(r, c);
        }
    } else if (M.format == 6) {  // IQ4_XS
        put16(out, f16_uniform(draw(key, base + 0), (float)2e-4, (float)1e-3));
        const uint64_t r1 = draw(key, base + 1);
        for (int c = 0; c < 6; ++c) out[2 + c] = byte_of(r1, c);
        for (int g = 0; g < 16; ++g) {
            uint64_t r = draw(key, base + 2 + g);
            for (int c = 0; c < 8; ++c) out[8 + 8 * g + c] = byte_of(r, c);
        }
    } else if (M.format == 7) {  // IQ3_XXS
        put16(out, f16_uniform(draw(key, base + 0), (float)0.001, (float)0.009));
        for (int g = 0; g < 12; ++g) {
            uint64_t r = draw(key, base + 1 + g);
            for (int c = 0; c < 8; ++c) out[2 + 8 * g + c] = byte_of(r, c);
        }
    } else {  // T5_G128 (fp16 s at an even offset: 28 j is even)
        put16(out, f16_uniform(draw(key, base + 0), (float)0.25, (float)0.75));
        for (int g = 0; g < 7; ++g) {
            uint64_t r = draw(key, base + 1 + g);
            for (int c = 0; c < 4; ++c) {
                const int i = 4 * g + c;
                const uint64_t ch = (r >> (16 * c)) & 0xFFFF;
                if (i < 25) out[2 + i] = (uint8_t)ubelow16(ch, 243);
                else if (i == 25) out[2 + i] = (uint8_t)ubelow16(ch, 27);
            }
        }
    }
    if (j == nb - 1) {  // zero the row padding
        uint8_t *row_end = static_cast<uint8_t *>(M.data) + (int64_t)row * M.row_stride_bytes + (int64_t)nb * bb;
        for (int64_t i = 0; i < M.row_stride_bytes - (int64_t)nb * bb; ++i) row_end[i] = 0;
    }
}

}  // namespace

extern "C" int moe_synth_fill(const moe_synth_matrix *descs, int32_t n, int32_t max_rows,
                              int32_t max_blocks_per_row, moe_stream_t stream) {
    if (n < 0 || n > 65535 || max_rows < 0 || max_blocks_per_row < 0) return 1;
    if (n == 0 || max_rows == 0 || max_blocks_per_row == 0) return 0;
    if (!descs) return 1;
    const int64_t nblocks = (int64_t)max_rows * max_blocks_per_row;
    const int threads = 256;
    const int64_t gx = (nblocks + threads - 1) / threads;
    if (gx > 0x7fffffff) return 1;
    synth_fill_kernel<<<dim3((unsigned)gx, (unsigned)n), threads, 0, (cudaStream_t)stream>>>(descs);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
}
