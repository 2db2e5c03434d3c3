/*
 * beamnorm.h -- C ABI of libbeamnorm: the arithmetic epilogue of a fused
 * tensor-parallel all-reduce in an LLM decoder layer, on one GB300 GPU.
 *
 * The operation (sources):
 *   "Fuse Beam's TP all-reduce with its sandwich norms" (vLLM pull request
 *   62366), section "Claims", first bullet: an all-reduce followed by an FP32
 *   norm-residual-norm epilogue, with an optional MoE top-k finalize before
 *   the reduction that keeps each rank's local BF16 rounding; section
 *   "Details", "Build" bullet: the FP32 epilogue is not contracted into FMAs;
 *   the workspace declines (returns nothing) for shapes it does not serve.
 *   sglang pull request 34134 (cute-dsl MNNVL all-reduce fusion backend),
 *   description: two fused patterns, the plain one (all-reduce, residual add,
 *   RMSNorm) and the MoE one (finalize and shared-expert add folded in ahead
 *   of the all-reduce, residual add and RMSNorm); a deferred finalize that
 *   meets a path which does not fuse is written out on its own; a decline
 *   must never drop the reduction that is still owed.
 *
 * Here the R tensor-parallel shards are all resident on the calling GPU; the
 * reduction is over a data dimension and nothing is communicated.
 *
 * Arithmetic, per token row t (all FP32 operations single IEEE operations,
 * round to nearest even, no FMA contraction, no flush to zero):
 *   finalize (finalize entries only), for each shard r:
 *       acc = w[r,t,0] * x_0;  acc = acc + w[r,t,j] * x_j  for j = 1..k-1
 *       (x_j = BF16 row perm[r,t,j] of expert_out[r], widened exactly)
 *       acc = acc + shared[r,t]            (when shared is not NULL)
 *       z[r,t] = bf16(acc)                 (local BF16 rounding per shard)
 *   rank-ordered reduction:  s = p_0;  s = s + p_r  for r = 1..R-1
 *       (p_r = partials[r,t] or z[r,t], widened exactly)
 *   post-RMSNorm:  ss1 = sum_h s^2;  r1 = 1 / sqrt(ss1 / H + eps);
 *                  y = (s * r1) * gamma_post
 *   residual add:  h = residual[t] + y;  residual[t] = bf16(h)      (in place)
 *   pre-RMSNorm:   ss2 = sum_h h^2;  r2 = 1 / sqrt(ss2 / H + eps);
 *                  out[t] = bf16((h * r2) * gamma_pre)
 * The sums of squares are compensated: each square's rounding error and each
 * addition's are carried in a second FP32 accumulator, and the pair is rounded
 * once.  That is as accurate as a sum carried in twice the precision: beyond
 * the final rounding it is off the exact sum by at most about (n * 2^-24)^2
 * relative and typically by about sqrt(n) * 2^-48, so it is the FP32 rounding
 * of the exact sum unless that lies within such a distance of a rounding
 * boundary.  So results practically never depend on how a row is split
 * across threads.  Where squares fall below the FP32 normal range a
 * product's error is itself rounded and one pass is off by up to H * 2^-150;
 * for eps < 2^-50 a row whose sum is below 2^-80 is therefore summed again
 * with its values scaled by a power of two, which restores the exact sum
 * rounded once.  For larger eps that pass cannot change an output, since
 * fl(ss / H) + eps rounds to eps, so it is skipped there (bn_tuning.tiny_pass
 * overrides).  A sum beyond the FP32 range is +inf, as the exact sum rounded.
 *
 * Conventions for every entry point:
 *   - BF16 tensors are passed as uint16_t bit patterns.  All tensors are dense,
 *     row-major, contiguous.  Every pointer is a device pointer on the current
 *     CUDA device, except where stated.
 *   - BF16 and FP32 tensor pointers must be 16-byte aligned; perm and w must be
 *     4-byte aligned.  H must be a multiple of 8 (16-byte rows).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.  The caller owns
 *     every buffer; the library allocates nothing.
 *   - On any status other than BN_OK nothing was enqueued, except BN_ERR_CUDA
 *     from a failed launch.  bn_last_error() describes the failure.
 *   - Arguments are validated on the host before any CUDA call: a NULL
 *     required pointer, R or k outside [1, 16], T < 0, H <= 0, H % 8 != 0, a
 *     misaligned pointer, eps negative or not finite, or an output range that
 *     overlaps an input range gives BN_ERR_INVALID.  A valid shape that is not
 *     served gives BN_ERR_UNSUPPORTED with nothing enqueued -- the decline: the
 *     fused entry points serve H <= 32768, the unfused pieces (the caller's
 *     fallback) H <= 131072, and every entry with a finalize needs
 *     T * k < 2^31.  bn_supports() and bn_supports_op() predict it.  T == 0 returns BN_OK after the shape checks, enqueues
 *     nothing and does not examine the pointers (empty tensors may be NULL).
 *   - dbg (nullable) asks for intermediate values, for testing:
 *       dbg->sum [T,H] FP32 reduced sum s, dbg->ss [T,2] FP32 (ss1, ss2),
 *       dbg->z [R,T,H] BF16 per-shard finalize results (finalize entries).
 *     Any member may be NULL.  With dbg == NULL nothing extra is written.
 */
#ifndef BEAMNORM_H
#define BEAMNORM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BN_API __attribute__((visibility("default")))
#else
#define BN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BN_OK = 0,
    BN_ERR_INVALID = 1,      /* bad argument; nothing enqueued */
    BN_ERR_UNSUPPORTED = 2,  /* valid shape that is declined; nothing enqueued */
    BN_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    BN_ERR_DEVICE = 4        /* bn_check_device_error found a device-side error bit */
} bn_status;

/* Device-side error bits (see bn_check_device_error). */
#define BN_DEVERR_PERM_RANGE 1u  /* a perm value outside [0, T*k): clamped to 0, never trapped */
#define BN_DEVERR_TIMEOUT 2u     /* a pipeline wait gave up after its time limit */

typedef struct {
    float *sum;    /* [T, H] FP32, or NULL */
    float *ss;     /* [T, 2] FP32 (post-norm, pre-norm sum of squares), or NULL */
    uint16_t *z;   /* [R, T, H] BF16 per-shard finalize results, or NULL */
} bn_debug;

/* ---- fused entry points ------------------------------------------------ */

/* Sandwich epilogue after a tensor-parallel all-reduce.
 *   partials   [R, T, H] BF16   one partial output per shard (rank r = row block r)
 *   residual   [T, H]    BF16   read, then overwritten with bf16(h)
 *   gamma_post [H]       FP32   post-RMSNorm weight (applied to the reduced sum)
 *   gamma_pre  [H]       FP32   next layer's input-RMSNorm weight
 *   out        [T, H]    BF16   written; must not overlap any input
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Claims". */
BN_API bn_status bn_reduce_norm(const uint16_t *partials, int R, int T, int H,
                         uint16_t *residual, const float *gamma_post,
                         const float *gamma_pre, float eps, uint16_t *out,
                         const bn_debug *dbg, void *stream);

/* MoE top-k finalize per shard, then the sandwich epilogue.
 *   expert_out [R, T*k, H] BF16  permuted expert-output rows of each shard
 *   perm       [R, T, k]   int32 gather index: slot j of token t reads row
 *                                perm[r,t,j] of expert_out[r]; values outside
 *                                [0, T*k) set BN_DEVERR_PERM_RANGE and read row 0
 *   w          [R, T, k]   FP32  top-k weights of each shard
 *   shared     [R, T, H]   BF16  shared-expert output of each shard, or NULL (zeros)
 *   residual, gamma_post, gamma_pre, out: as bn_reduce_norm
 * Sources: "Fuse Beam's TP all-reduce with its sandwich norms", "Claims";
 * sglang pull request 34134, description. */
BN_API bn_status bn_finalize_reduce_norm(const uint16_t *expert_out, const int32_t *perm,
                                  const float *w, const uint16_t *shared,
                                  int R, int T, int k, int H,
                                  uint16_t *residual, const float *gamma_post,
                                  const float *gamma_pre, float eps, uint16_t *out,
                                  const bn_debug *dbg, void *stream);

/* The plain single-norm pattern (all-reduce, residual add, RMSNorm): no post-norm,
 * h = residual + s, then the RMSNorm with weight gamma.  dbg->ss[:,0] is 0.
 * Source: sglang pull request 34134, description (first fused pattern). */
BN_API bn_status bn_reduce_residual_norm(const uint16_t *partials, int R, int T, int H,
                                  uint16_t *residual, const float *gamma, float eps,
                                  uint16_t *out, const bn_debug *dbg, void *stream);

/* The MoE single-norm pattern: per-shard finalize with the shared-expert add,
 * then all-reduce, residual add and RMSNorm (no post-norm).
 * Source: sglang pull request 34134, description (second fused pattern). */
BN_API bn_status bn_finalize_reduce_residual_norm(const uint16_t *expert_out, const int32_t *perm,
                                           const float *w, const uint16_t *shared,
                                           int R, int T, int k, int H,
                                           uint16_t *residual, const float *gamma, float eps,
                                           uint16_t *out, const bn_debug *dbg, void *stream);

/* ---- finalize with a caller-provided workspace (few token rows) --------- */

/* Bytes of workspace with which bn_finalize_reduce_norm_ws and
 * bn_finalize_reduce_residual_norm_ws spread each token row over many CTAs,
 * or 0 when that path does not serve the shape (it serves 1 <= T <= 8 and
 * H <= 8192, where one CTA or one cluster per token row leaves most SMs
 * idle).  Pure host logic.  Layout: the counters (T words, padded to 256
 * bytes), then the per-shard BF16 finalize results [T, R, H].
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Details"
 * (the fused op runs on a workspace sized for the shapes it serves). */
BN_API size_t bn_finalize_workspace_bytes(int R, int T, int k, int H);

/* bn_finalize_reduce_norm with a workspace.
 *   workspace        device memory, 16-byte aligned, owned by the caller; it
 *                    must be zero-filled before its first use, and every
 *                    call leaves its counters at zero again.  One workspace
 *                    serves one call at a time: calls that may run
 *                    concurrently (different streams) need their own.
 *   workspace_bytes  its size.  With at least bn_finalize_workspace_bytes()
 *                    bytes (and that size non-zero) the row's finalize is
 *                    split over many CTAs and its epilogue run by the CTA
 *                    that finishes the row last; otherwise the workspace is
 *                    not touched and the call is bn_finalize_reduce_norm.
 * The results are those of bn_finalize_reduce_norm: the same per-shard BF16
 * rounding, rank-ordered FP32 sum and norms.  The workspace must not overlap
 * any other buffer of the call (BN_ERR_INVALID).
 * Sources: "Fuse Beam's TP all-reduce with its sandwich norms", "Claims" and
 * "Details" (the fused op's workspace); sglang pull request 34134,
 * description. */
BN_API bn_status bn_finalize_reduce_norm_ws(const uint16_t *expert_out, const int32_t *perm,
                                     const float *w, const uint16_t *shared,
                                     int R, int T, int k, int H,
                                     uint16_t *residual, const float *gamma_post,
                                     const float *gamma_pre, float eps, uint16_t *out,
                                     const bn_debug *dbg, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* bn_finalize_reduce_residual_norm with a workspace, as above.
 * Source: sglang pull request 34134, description (second fused pattern). */
BN_API bn_status bn_finalize_reduce_residual_norm_ws(const uint16_t *expert_out,
                                              const int32_t *perm, const float *w,
                                              const uint16_t *shared, int R, int T, int k,
                                              int H, uint16_t *residual, const float *gamma,
                                              float eps, uint16_t *out, const bn_debug *dbg,
                                              void *workspace, size_t workspace_bytes,
                                              void *stream);

/* ---- the same finalize for callers that cannot allocate -------------------- */

/* bn_finalize_reduce_norm_ws without a caller workspace: the library uses its
 * own scratch, a static device array of 2 MiB (2097152 bytes).
 *
 * Who needs it: a caller that is handed only the op's input and output
 * tensors and may not allocate device memory itself -- for example a serving
 * engine whose memory pool has already reserved nearly all of HBM and owns
 * every allocation, a plugin hook of an inference runtime that passes in and
 * out pointers and no workspace slot, or a latency-critical path where
 * cudaMalloc's implicit device synchronisation is not acceptable.
 *
 * Arguments, results and errors are those of bn_finalize_reduce_norm_ws.  The
 * call allocates nothing (no cudaMalloc or cudaFree) and serves the shapes the
 * many-CTA finalize serves (1 <= T <= 8, H <= 8192) whose workspace fits the
 * scratch (bn_finalize_workspace_bytes(R, T, k, H) <= 2 MiB); any other valid
 * shape gives BN_ERR_UNSUPPORTED with nothing enqueued (bn_last_error says
 * why; bn_finalize_reduce_norm needs no scratch at all).
 *
 * The scratch:
 *   - is reserved on a device by the first call there, which also looks up its
 *     address once with that device current; make that first call before any
 *     stream capture.  It then stays reserved on that device until the process
 *     exits.
 *   - is shared by every call of this entry point in the process and keeps the
 *     last call's contents; each call clears the row counters it needs on
 *     `stream` before its kernel.  Calls whose work may overlap on the GPU
 *     (different streams without ordering between them) race on the scratch
 *     and give wrong results: order them, or give them bn_finalize_reduce_norm_ws
 *     with a workspace each.
 * Source: none -- the pages describe no such entry point; it has no
 * counterpart there. */
BN_API bn_status bn_finalize_reduce_norm_noalloc(const uint16_t *expert_out,
                                                 const int32_t *perm, const float *w,
                                                 const uint16_t *shared, int R, int T, int k,
                                                 int H, uint16_t *residual,
                                                 const float *gamma_post, const float *gamma_pre,
                                                 float eps, uint16_t *out, const bn_debug *dbg,
                                                 void *stream);

/* ---- unfused pieces (the decline / fallback path and its measurement) --- */

/* Rank-ordered FP32 sum only: sum_out [T, H] FP32 = s.  Rows up to H = 131072.
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Claims" (the
 * all-reduce the epilogue follows); sglang pull request 34134, description
 * (the unfused path a declined call falls back to). */
BN_API bn_status bn_reduce_only(const uint16_t *partials, int R, int T, int H,
                         float *sum_out, void *stream);

/* Per-shard finalize rounded to BF16, then the rank-ordered FP32 sum only.
 * Rows up to H = 131072.
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Claims" (the
 * finalize before the reduction keeps each shard's BF16 rounding). */
BN_API bn_status bn_finalize_reduce_only(const uint16_t *expert_out, const int32_t *perm,
                                  const float *w, const uint16_t *shared,
                                  int R, int T, int k, int H, float *sum_out,
                                  void *stream);

/* The sandwich epilogue given the FP32 sum [T, H] (post-norm, residual add,
 * pre-norm).  Together with bn_reduce_only / bn_finalize_reduce_only it gives
 * the same bits as the fused entry points.  Rows up to H = 131072.
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Claims" (the
 * FP32 norm-residual-norm epilogue). */
BN_API bn_status bn_norm_only(const float *sum, int T, int H, uint16_t *residual,
                       const float *gamma_post, const float *gamma_pre, float eps,
                       uint16_t *out, const bn_debug *dbg, void *stream);

/* The single-norm epilogue given the FP32 sum [T, H]: h = residual + sum,
 * residual = bf16(h) in place, out = bf16((h * r) * gamma) with
 * r = 1 / sqrt(sum(h^2) / H + eps).  Together with bn_reduce_only /
 * bn_finalize_reduce_only it gives the bits of bn_reduce_residual_norm /
 * bn_finalize_reduce_residual_norm.  dbg->ss[:,0] is 0.
 * Source: sglang pull request 34134, description (the plain all-reduce,
 * residual add and RMSNorm pattern; the fallback when fusion declines). */
BN_API bn_status bn_residual_norm_only(const float *sum, int T, int H, uint16_t *residual,
                                       const float *gamma, float eps, uint16_t *out,
                                       const bn_debug *dbg, void *stream);

/* The deferred finalize materialised on its own: z_out [R, T, H] BF16 =
 * bf16(sum_j w*x_j + shared) per shard, with no reduction.
 * Source: sglang pull request 34134, description (the deferred finalize written
 * out on its own when the fused path declines). */
BN_API bn_status bn_finalize_only(const uint16_t *expert_out, const int32_t *perm,
                           const float *w, const uint16_t *shared,
                           int R, int T, int k, int H, uint16_t *z_out, void *stream);

/* ---- queries and errors ------------------------------------------------ */

/* 1 if the fused entry points serve this shape (k = 0 for the reduce-only
 * entries), 0 if the caller must fall back.  Pure host logic.
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Details"
 * (the fused op declines shapes it does not serve). */
BN_API int bn_supports(int R, int T, int k, int H);

/* Synchronises `stream`, reads the device-side error bits of the current
 * device into *bits (nullable), clears them, and returns BN_ERR_DEVICE if any
 * bit was set, BN_ERR_CUDA if the synchronisation failed, else BN_OK.
 * Source: sglang pull request 34134, NextN follow-up (a path that cannot do
 * its work fails loudly rather than silently). */
BN_API bn_status bn_check_device_error(void *stream, unsigned *bits);

/* Message describing the last failure on the calling thread ("" if none).
 * Source: no passage: library utility. */
BN_API const char *bn_last_error(void);

/* Name of a status code.
 * Source: no passage: library utility. */
BN_API const char *bn_status_string(bn_status status);

/* Library version, major * 10000 + minor * 100 + patch.
 * Source: no passage: library utility. */
BN_API int bn_version(void);

/* Does nothing, and may be called at any time.  The library allocates no
 * memory it would have to release: its device state (the error word, the
 * static scratch of bn_finalize_reduce_norm_noalloc) is static device memory,
 * released with the CUDA context; the host state is static too.  Provided so
 * that a caller can pair it with the first call.
 * Source: no passage: library utility. */
BN_API void bn_shutdown(void);

/* Launch-shape overrides for measurement sweeps (process-wide).  Every field
 * 0 means automatic.  Results do not depend on these settings, only speed
 * (tiny_pass aside, which can change the debug sums of squares of rows of
 * tiny values and nothing else). */
typedef struct {
    int cluster_size;  /* CTAs per token row, at most 16 (a shard split takes
                          one that divides R) */
    int stages;        /* pipeline depth in stages, at most 64 */
    int threads;       /* consumer threads per CTA: a multiple of 32, at most 512 */
    int ctas_per_sm;   /* CTAs sharing one SM, at most 8 (capped by registers) */
    int wait_mode;     /* 1: suspending try_wait, 2: polling test_wait */
    int group;         /* row copies per pipeline stage, at most 64; the finalize
                          modes only (the other modes carry one copy a stage) */
    int split;         /* 1 split rows by columns, 2 finalize rows by shard,
                          3 one cluster per row with one (shard, chunk) task per
                          thread (the fused entry points) */
    int dependent_launch; /* 1: plain stream order, 2: programmatic dependent
                             launch (the launch and the kernel's setup overlap
                             the previous kernel in the stream) */
    int wait_limit_polls; /* for tests of the failure path: the copy-pipeline
                             waits give up after this many polls (the default
                             is 2^26 polls or 2^29 SM cycles).  A call whose
                             wait gives up sets BN_DEVERR_TIMEOUT, stores
                             nothing more, still drains its copies and returns;
                             its outputs are then unspecified (each within its
                             own buffer).  Not applied to the many-CTA
                             finalize, which never waits. */
    int tiny_pass;        /* the second pass over a row whose sum of squares is
                             below 2^-80 (its squares near or below FP32's
                             subnormal range, where the one-pass compensated
                             sum is off by up to H * 2^-150): 1 never, 2
                             always.  Automatic: for eps < 2^-50 only, the
                             one range of eps where the pass can change an
                             output; elsewhere it would change only the debug
                             sums of squares. */
} bn_tuning;

/* Set the overrides; NULL restores automatic choices.  BN_ERR_INVALID on an
 * out-of-range field (nothing changes then).
 * Source: no passage: library utility (measurement sweeps and tests). */
BN_API bn_status bn_set_tuning(const bn_tuning *tuning);

/* The operations of the entry points above, for bn_query_launch. */
typedef enum {
    BN_OP_REDUCE_NORM = 0,
    BN_OP_FINALIZE_REDUCE_NORM = 1,
    BN_OP_REDUCE_RESIDUAL_NORM = 2,
    BN_OP_FINALIZE_REDUCE_RESIDUAL_NORM = 3,
    BN_OP_REDUCE_ONLY = 4,
    BN_OP_FINALIZE_REDUCE_ONLY = 5,
    BN_OP_NORM_ONLY = 6,
    BN_OP_FINALIZE_ONLY = 7,
    BN_OP_RESIDUAL_NORM_ONLY = 8
} bn_op;

/* The launch shape one call would use on the current device. */
typedef struct {
    int split;                /* 1: a cluster splits each row by shard; 2: a cluster
                                 splits each row by column slices with one
                                 (shard, chunk) finalize task per thread, and
                                 chunks_per_thread is then the tasks per thread */
    int cluster_size;         /* CTAs per token row */
    int threads;              /* threads per CTA: consumer threads + one producer warp */
    int chunks_per_thread;    /* 16-byte chunks of the CTA's slice per consumer thread */
    int grid;                 /* CTAs launched (persistent; rows are grid-strided) */
    int resident_ctas;        /* CTAs of this shape the device holds at once */
    int stages;               /* pipeline stages in the shared-memory ring */
    int stage_bytes;
    int group;                /* row copies per stage */
    int smem_bytes;           /* dynamic shared memory per CTA */
} bn_launch_info;

/* Fill *info with the launch shape that `op` would use for this shape on the
 * current device, under the current tuning overrides, for eps >= 2^-50 (the
 * kernels of smaller eps, see bn_tuning.tiny_pass, may take another shape);
 * nothing is enqueued.
 * k is ignored by the operations without a finalize; has_shared says whether
 * the finalize call would pass a shared-expert row.  Shape errors and
 * declines are reported as by the entry point itself; T == 0 gives BN_OK and
 * an all-zero *info (no launch).  Needs a CUDA device (occupancy queries).
 * Source: no passage: library utility (measurement sweeps and tests). */
BN_API bn_status bn_query_launch(bn_op op, int R, int T, int k, int H, int has_shared,
                                 bn_launch_info *info);

/* 1 if entry point `op` serves this shape, 0 if it would decline (or the
 * arguments are invalid).  k is ignored without a finalize; R is ignored by
 * the epilogue pieces.  The unfused pieces serve rows the fused entry points
 * decline (H up to 131072), which is what a caller falls back to.  Pure host
 * logic.
 * Source: "Fuse Beam's TP all-reduce with its sandwich norms", "Details"
 * (the workspace declines shapes it does not serve); sglang pull request
 * 34134, description (a decline must not drop the reduction still owed). */
BN_API int bn_supports_op(bn_op op, int R, int T, int k, int H);

#ifdef __cplusplus
}
#endif

#endif /* BEAMNORM_H */
