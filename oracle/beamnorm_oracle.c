/*
 * beamnorm_oracle.c -- the CPU oracle for libbeamnorm.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * definition of what the GPU path computes.  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark may load it.  It shares no code,
 * header, table or helper with the CUDA library, and the library never calls it.
 *
 * What it computes (sources):
 *   - "Fuse Beam's TP all-reduce with its sandwich norms" (vLLM pull request
 *     62366), section "Claims", first bullet: an all-reduce whose epilogue is an
 *     FP32 norm-residual-norm, with an optional MoE top-k finalize applied
 *     *before* the reduction that keeps each rank's local BF16 rounding.
 *   - same page, section "Details", "Build" bullet: the FP32 epilogue math is
 *     not contracted into FMAs.  This file must be built with
 *     -ffp-contract=off and without -ffast-math (the build script does so).
 *   - sglang pull request 34134 ("cute-dsl" MNNVL all-reduce fusion backend),
 *     description and "Motivation": the two fused patterns, "AllReduce +
 *     residual + RMSNorm" and "MoE finalize + shared-expert add + AllReduce +
 *     residual + RMSNorm", whose output feeds the next layer's input RMSNorm.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - rank order: s = p_0, then s = s + p_r for r = 1..R-1 (not 0 + p_0);
 *   - RMSNorm(x) = (x * (1 / sqrt(mean(x^2) + eps))) * gamma, plain gamma,
 *     eps inside the square root, mean as an FP32 divide by H;
 *   - the sum of squares is accumulated in double and rounded to FP32 once;
 *   - the pre-norm reads the FP32 h = residual + y, not its BF16 rounding;
 *   - finalize: acc = w_0*x_0, acc = acc + w_j*x_j for j ascending, then
 *     acc = acc + shared, then one round to BF16; perm is a gather index.
 *
 * BF16 values travel as uint16_t bit patterns.  Outputs for a selected set of
 * token rows are written compactly (row i of an output is token rows[i]).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "beamnorm_oracle.h"

/* ---- BF16 <-> FP32, written from the definition of the formats ---------- */

/* BF16 is the upper half of an IEEE binary32; widening is exact. */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest BF16, ties to even.  The 16 dropped bits
 * are compared with one half of the kept unit in the last place; a carry out
 * of the mantissa correctly moves to the next binade (or to infinity).  Any
 * NaN becomes a quiet NaN with the same sign. */
static uint16_t f32_to_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

uint16_t oracle_bf16_from_f32(float f) { return f32_to_bf16_rn(f); }
float oracle_f32_from_bf16(uint16_t b) { return bf16_to_f32(b); }

/* ---- one RMSNorm factor ------------------------------------------------- */

/* Sum of squares of a row, accumulated in double (each square of an FP32
 * value is exact in double) and rounded to FP32 once. */
static float sum_of_squares(const float *x, int H)
{
    double acc = 0.0;
    for (int h = 0; h < H; ++h)
        acc += (double)x[h] * (double)x[h];
    return (float)acc;
}

/* 1 / sqrt(mean + eps) as two correctly rounded FP32 operations. */
static float rms_factor(float ss, int H, float eps)
{
    float mean = ss / (float)H;
    return 1.0f / sqrtf(mean + eps);
}

/* ---- the norm-residual-norm epilogue of one token row -------------------
 * s       : FP32 reduced sum of the row (H values)
 * res_in  : BF16 residual row
 * Writes the BF16 updated residual, the BF16 output of the next layer's
 * input RMSNorm, and the two sums of squares.  hbuf is H floats of work
 * space.  With ORACLE_SINGLE_NORM there is no post-norm: h = residual + s
 * (the plain "AllReduce + residual + RMSNorm" pattern). */
static void epilogue_row(const float *s, const uint16_t *res_in,
                         const float *gamma_post, const float *gamma_pre,
                         float eps, int H, int flags,
                         uint16_t *res_out, uint16_t *out, float *ss_out,
                         float *hbuf)
{
    float ss1 = 0.0f;
    if (flags & ORACLE_SINGLE_NORM) {
        for (int h = 0; h < H; ++h) {
            hbuf[h] = bf16_to_f32(res_in[h]) + s[h];
            res_out[h] = f32_to_bf16_rn(hbuf[h]);
        }
    } else {
        /* post-RMSNorm of the reduced sum, then the residual add */
        ss1 = sum_of_squares(s, H);
        float r1 = rms_factor(ss1, H, eps);
        for (int h = 0; h < H; ++h) {
            float y = (s[h] * r1) * gamma_post[h];
            hbuf[h] = bf16_to_f32(res_in[h]) + y;
            res_out[h] = f32_to_bf16_rn(hbuf[h]);
        }
    }
    /* Sensitivity switch only: let the pre-norm read the BF16 residual. */
    if (flags & ORACLE_PRENORM_FROM_BF16_RESIDUAL)
        for (int h = 0; h < H; ++h)
            hbuf[h] = bf16_to_f32(res_out[h]);
    /* the next layer's input RMSNorm */
    float ss2 = sum_of_squares(hbuf, H);
    float r2 = rms_factor(ss2, H, eps);
    for (int h = 0; h < H; ++h)
        out[h] = f32_to_bf16_rn((hbuf[h] * r2) * gamma_pre[h]);
    if (ss_out) {
        ss_out[0] = ss1;
        ss_out[1] = ss2;
    }
}

static int token_of(const int32_t *rows, int i) { return rows ? rows[i] : i; }

static int check_rows(const int32_t *rows, int nrows, int T)
{
    if (nrows < 0) return 0;
    if (!rows) return nrows == T;
    for (int i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= T) return 0;
    return 1;
}

/* ---- reduce_norm -------------------------------------------------------- */

int oracle_reduce_norm(const uint16_t *partials, int R, int T, int H,
                       const uint16_t *residual, const float *gamma_post,
                       const float *gamma_pre, float eps, int flags,
                       const int32_t *rows, int nrows,
                       uint16_t *residual_out, uint16_t *out,
                       float *sum_out, float *ss_out)
{
    if (R < 1 || T < 0 || H < 1 || !check_rows(rows, nrows, T)) return ORACLE_ERR_ARGS;
    float *s = (float *)malloc(sizeof(float) * (size_t)H);
    float *hbuf = (float *)malloc(sizeof(float) * (size_t)H);
    if (!s || !hbuf) { free(s); free(hbuf); return ORACLE_ERR_ARGS; }

    for (int i = 0; i < nrows; ++i) {
        int t = token_of(rows, i);
        /* rank-ordered FP32 reduction: s = p_0, then s = s + p_r */
        for (int r = 0; r < R; ++r) {
            const uint16_t *p = partials + ((size_t)r * T + t) * H;
            for (int h = 0; h < H; ++h) {
                float v = bf16_to_f32(p[h]);
                s[h] = (r == 0) ? v : s[h] + v;
            }
        }
        if (sum_out) memcpy(sum_out + (size_t)i * H, s, sizeof(float) * (size_t)H);
        if (out && residual_out)
            epilogue_row(s, residual + (size_t)t * H, gamma_post, gamma_pre, eps, H,
                         flags, residual_out + (size_t)i * H, out + (size_t)i * H,
                         ss_out ? ss_out + 2 * (size_t)i : NULL, hbuf);
    }
    free(s);
    free(hbuf);
    return ORACLE_OK;
}

/* ---- the MoE top-k finalize of one shard and one token ------------------
 * z[h] = bf16_rn( (w_0 x_0[h] + w_1 x_1[h] + ... + w_{k-1} x_{k-1}[h]) + shared[h] )
 * where x_j is row perm[j] of this shard's expert outputs. */
static int finalize_one(const uint16_t *xr /* [T*k, H] of shard r */,
                        const int32_t *perm /* k */, const float *w /* k */,
                        const uint16_t *shared_row /* H or NULL */,
                        int T, int k, int H, uint16_t *z)
{
    for (int j = 0; j < k; ++j)
        if (perm[j] < 0 || (int64_t)perm[j] >= (int64_t)T * k) return ORACLE_ERR_PERM;
    for (int h = 0; h < H; ++h) {
        float acc = w[0] * bf16_to_f32(xr[(size_t)perm[0] * H + h]);
        for (int j = 1; j < k; ++j)
            acc = acc + w[j] * bf16_to_f32(xr[(size_t)perm[j] * H + h]);
        if (shared_row) acc = acc + bf16_to_f32(shared_row[h]);
        z[h] = f32_to_bf16_rn(acc);
    }
    return ORACLE_OK;
}

int oracle_finalize_reduce_norm(const uint16_t *expert_out, const int32_t *perm,
                                const float *w, const uint16_t *shared,
                                int R, int T, int k, int H,
                                const uint16_t *residual, const float *gamma_post,
                                const float *gamma_pre, float eps, int flags,
                                const int32_t *rows, int nrows,
                                uint16_t *residual_out, uint16_t *out,
                                float *sum_out, float *ss_out, uint16_t *z_out)
{
    if (R < 1 || T < 0 || k < 1 || H < 1 || !check_rows(rows, nrows, T)) return ORACLE_ERR_ARGS;
    float *s = (float *)malloc(sizeof(float) * (size_t)H);
    float *hbuf = (float *)malloc(sizeof(float) * (size_t)H);
    uint16_t *z = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)H);
    if (!s || !hbuf || !z) { free(s); free(hbuf); free(z); return ORACLE_ERR_ARGS; }
    int status = ORACLE_OK;

    for (int i = 0; i < nrows && status == ORACLE_OK; ++i) {
        int t = token_of(rows, i);
        for (int r = 0; r < R && status == ORACLE_OK; ++r) {
            /* per-shard finalize, rounded to BF16 locally (before the reduction) */
            const uint16_t *xr = expert_out + (size_t)r * T * k * H;
            const int32_t *pr = perm + ((size_t)r * T + t) * k;
            const float *wr = w + ((size_t)r * T + t) * k;
            const uint16_t *sh = shared ? shared + ((size_t)r * T + t) * H : NULL;
            status = finalize_one(xr, pr, wr, sh, T, k, H, z);
            if (status != ORACLE_OK) break;
            if (z_out) memcpy(z_out + ((size_t)r * nrows + i) * H, z, sizeof(uint16_t) * (size_t)H);
            /* rank-ordered FP32 reduction of the BF16 finalize results */
            for (int h = 0; h < H; ++h) {
                float v = bf16_to_f32(z[h]);
                s[h] = (r == 0) ? v : s[h] + v;
            }
        }
        if (status != ORACLE_OK) break;
        if (sum_out) memcpy(sum_out + (size_t)i * H, s, sizeof(float) * (size_t)H);
        if (out && residual_out)
            epilogue_row(s, residual + (size_t)t * H, gamma_post, gamma_pre, eps, H,
                         flags, residual_out + (size_t)i * H, out + (size_t)i * H,
                         ss_out ? ss_out + 2 * (size_t)i : NULL, hbuf);
    }
    free(s);
    free(hbuf);
    free(z);
    return status;
}

/* ---- the epilogue alone, given the FP32 sum (the unfused split's second half) */

int oracle_norm(const float *sum, int T, int H, const uint16_t *residual,
                const float *gamma_post, const float *gamma_pre, float eps, int flags,
                const int32_t *rows, int nrows,
                uint16_t *residual_out, uint16_t *out, float *ss_out)
{
    if (T < 0 || H < 1 || !check_rows(rows, nrows, T)) return ORACLE_ERR_ARGS;
    float *hbuf = (float *)malloc(sizeof(float) * (size_t)H);
    if (!hbuf) return ORACLE_ERR_ARGS;
    for (int i = 0; i < nrows; ++i) {
        int t = token_of(rows, i);
        epilogue_row(sum + (size_t)t * H, residual + (size_t)t * H, gamma_post, gamma_pre,
                     eps, H, flags, residual_out + (size_t)i * H, out + (size_t)i * H,
                     ss_out ? ss_out + 2 * (size_t)i : NULL, hbuf);
    }
    free(hbuf);
    return ORACLE_OK;
}
