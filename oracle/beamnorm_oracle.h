/*
 * beamnorm_oracle.h -- C interface of the CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * Host pointers throughout.  BF16 tensors are uint16_t bit patterns, row-major:
 *   partials   [R, T, H]        expert_out [R, T*k, H]
 *   perm, w    [R, T, k]        shared     [R, T, H] (NULL means zeros)
 *   residual   [T, H]           gamma_post, gamma_pre [H] (FP32)
 * rows selects which token rows to compute (NULL with nrows == T means all);
 * every output is compact: row i of an output belongs to token rows[i].
 *   residual_out, out [nrows, H]   sum_out [nrows, H] FP32 (NULL = skip)
 *   ss_out [nrows, 2] FP32 = (post-norm, pre-norm) sums of squares (NULL = skip)
 *   z_out  [R, nrows, H] BF16 per-shard finalize results (NULL = skip)
 * If out or residual_out is NULL only the reduction (and z) is computed.
 */
#ifndef BEAMNORM_ORACLE_H
#define BEAMNORM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_OK = 0, ORACLE_ERR_ARGS = -1, ORACLE_ERR_PERM = -2 };

/* flags */
enum {
    ORACLE_SINGLE_NORM = 1,                /* AllReduce + residual + RMSNorm (no post-norm) */
    ORACLE_PRENORM_FROM_BF16_RESIDUAL = 2  /* sensitivity switch, not a served variant */
};

uint16_t oracle_bf16_from_f32(float f);
float oracle_f32_from_bf16(uint16_t b);

int oracle_reduce_norm(const uint16_t *partials, int R, int T, int H,
                       const uint16_t *residual, const float *gamma_post,
                       const float *gamma_pre, float eps, int flags,
                       const int32_t *rows, int nrows,
                       uint16_t *residual_out, uint16_t *out,
                       float *sum_out, float *ss_out);

int oracle_finalize_reduce_norm(const uint16_t *expert_out, const int32_t *perm,
                                const float *w, const uint16_t *shared,
                                int R, int T, int k, int H,
                                const uint16_t *residual, const float *gamma_post,
                                const float *gamma_pre, float eps, int flags,
                                const int32_t *rows, int nrows,
                                uint16_t *residual_out, uint16_t *out,
                                float *sum_out, float *ss_out, uint16_t *z_out);

int oracle_norm(const float *sum, int T, int H, const uint16_t *residual,
                const float *gamma_post, const float *gamma_pre, float eps, int flags,
                const int32_t *rows, int nrows,
                uint16_t *residual_out, uint16_t *out, float *ss_out);

#ifdef __cplusplus
}
#endif

#endif
