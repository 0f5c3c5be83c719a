/*
 * Decode stand-in for the interference measurement of kvx.
 *
 * The pages measure the copy kernel's cost as the tail slowdown of a decode
 * that runs beside it on the same GPU (PegaFlow issue #408, "Kernel transfer
 * backend causes decode TPOT tail spikes under concurrent KV transfers",
 * §Results and follow-up §1). Without a model, an HBM-bound bf16 GEMV that
 * streams several GB per step stands in for one decode step: like a decode
 * at batch 1, it is bound by reading the weights from HBM.
 *
 * y[r] = sum_c W[r * cols + c] * x[c] for r < rows, with W (row-major) and x
 * in bf16, products and sums in fp32, y in fp32. Not part of the copy path.
 */
#ifndef KVX_STANDIN_H
#define KVX_STANDIN_H

#include <stddef.h>
#include <stdint.h>

#include "kvx.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Enqueue the GEMV on `stream` (a cudaStream_t). W: rows x cols bf16 device
 * array, 16-byte aligned; x: cols bf16 device array; y: rows fp32 device
 * array. cols must be a multiple of 256 and at most 4096; rows >= 1.
 * `ctas` = grid size of 256-thread CTAs (0 = about 8 rows per warp). Returns
 * KVX_ERR_INVALID_ARG / KVX_ERR_ALIGN for bad arguments (nothing enqueued) and
 * KVX_ERR_CUDA if the launch fails. */
kvx_status kvx_standin_gemv_bf16(uint64_t W, uint64_t x, uint64_t y, uint64_t rows, uint32_t cols,
                                 int ctas, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVX_STANDIN_H */
