/*
 * moe_synth.h -- GPU filler for seeded synthetic block-quantized weights.
 *
 * Benchmark and test input generation only; not part of the layer. It writes
 * the same bytes as the numpy generator in synth/__init__.py (SplitMix64 draws
 * placed at the field offsets of each block format; see that module for the
 * recipe), so that full-size layers (tens of GB) can be made on the device
 * and any expert can be regenerated on the host for a parity check.
 */
#ifndef MOE_SYNTH_H
#define MOE_SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t;

/* One matrix to fill: `rows` rows of `cols` weights in block format `format`
 * (1 Q8_0, 2 Q4_K, 3 Q6_K, 4 MXFP4, 5 IQ4_NL, 6 IQ4_XS, 7 IQ3_XXS), row stride `row_stride_bytes`, drawn from
 * the SplitMix64 sequence with key `key`. Padding bytes are written as 0. */
typedef struct {
    void *data;               /* device, rows * row_stride_bytes bytes */
    int64_t row_stride_bytes;
    int32_t format;
    int32_t rows;
    int32_t cols;
    int32_t reserved;
    uint64_t key;
} moe_synth_matrix;

/* Fill `n` matrices. `descs` is a DEVICE array of n descriptors. Returns 0 on
 * success, 1 on a bad argument, 6 on a CUDA error. Asynchronous on stream. */
int moe_synth_fill(const moe_synth_matrix *descs, int32_t n, int32_t max_rows, int32_t max_blocks_per_row,
                   moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_SYNTH_H */
