// bn_wide.h -- the finalize at small T with each token row spread over many
// CTAs (internal to libbeamnorm; not installed).
//
// Few token rows leave most SMs idle when one CTA or one cluster owns a row:
// a C4 row (R=8, k=10, H=8192) is 1.4 MB of gathered copies, and 8 to 16 SMs
// pull it at a few tens of GB/s each.  Here every CTA of a row takes up to
// kWideThreads (shard, 16-byte chunk) tasks of that row's finalize with plain
// 16-byte loads, writes the BF16 results z into a caller-provided workspace,
// and counts itself done on the row's counter; the CTA that completes the
// count runs the row's whole epilogue (rank-ordered sum, post-RMSNorm,
// residual add, pre-RMSNorm) from the workspace, which is still in L2.  No CTA
// waits for another: the last one to finish does the rest.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "bn_internal.h"

namespace bn {

constexpr int kWideThreads = 512;  // threads per CTA: tasks per CTA and epilogue threads
constexpr int kWideMaxCpt = 2;     // epilogue chunks per thread: H <= 8 * 512 * 2 = 8192

struct WideArgs {
    Args a;             // operands, sizes, eps, debug outputs, error word (stages unused)
    uint16_t *zws;      // workspace z rows, [T][R][H] BF16
    unsigned *count;    // workspace counters of finished CTAs, [T]; zero between calls
    int tasks;          // finalize tasks per CTA: kWideThreads, or a half or a quarter of it
    int parts;          // CTAs per token row: ceil(R * H/8 / tasks)
};

// Dynamic shared memory of the kernel: the epilogue's gammas (FP32 [H] each).
inline size_t wide_smem_bytes(bool postnorm, int H) { return (postnorm ? 2u : 1u) * (size_t)H * 4u; }

// Workspace bytes: the counters (padded to 256 bytes), then the z rows.
inline size_t wide_counter_bytes(int T) { return ((size_t)T * 4u + 255u) & ~(size_t)255u; }
inline size_t wide_workspace_bytes(int R, int T, int H)
{
    return wide_counter_bytes(T) + (size_t)T * (size_t)R * (size_t)H * 2u;
}

// Enqueue the kernel: grid T * parts CTAs of kWideThreads threads.  postnorm
// selects the sandwich (post-RMSNorm before the residual add) or the single
// pre-RMSNorm; cpt is the epilogue's chunks per thread (1 or 2, kWideMaxCpt).
cudaError_t launch_wide(const WideArgs &w, bool postnorm, int cpt, bool pdl, cudaStream_t st);

// Size of the library-owned scratch behind bn_finalize_reduce_norm_noalloc
// (a static device array, bn_noalloc.cu): 2 MiB, enough for the workspace of
// every shape the many-CTA finalize serves with R <= 15 (R = 16, T = 8,
// H = 8192 needs 256 bytes more and is declined).
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;

// Device address of that scratch on the current device.  The first call on a
// device looks it up (cudaGetSymbolAddress, with that device current); later
// calls return the cached address.  Allocates nothing.
cudaError_t noalloc_scratch(void **ptr);

}  // namespace bn
