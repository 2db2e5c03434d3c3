// bn_cluster.h -- the finalize at small T with each token row spread over a
// thread-block cluster (internal to libbeamnorm; not installed).
//
// One cluster of cs CTAs per token row; CTA q owns the column slice
// [q*nch/cs, (q+1)*nch/cs) of 16-byte chunks.  Each of its threads takes one
// (shard, chunk) task of that slice -- up to TPT tasks -- and gathers the k
// expert chunks and the shared-expert chunk with plain 16-byte loads, all in
// flight at once (for the reduce entry points a task loads the shard's
// partial chunk).  The BF16 finalize results stay in the CTA's shared memory,
// where the slice's threads sum them in rank order and run the epilogue; the
// two row-wide sums of squares cross the cluster as one asynchronous remote
// store per CTA pair, counted on the receiver's barrier.  Nothing goes through
// global memory but the inputs and the outputs.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "bn_internal.h"

namespace bn {

constexpr int kClusterThreads = 512;   // threads per CTA: finalize tasks, then the slice's epilogue
constexpr int kClusterMaxTpt = 2;      // finalize tasks per thread

struct ClusterArgs {
    Args a;        // operands, sizes, eps, debug outputs, error word (pipeline fields unused)
    int tasks;     // R * largest slice: the finalize tasks of one CTA
};

// Expert slots a finalize task unrolls so that all its k gathers are in
// flight: the smallest of 4, 8, 10 and 16 that holds k; 0 for the reduce entry
// points.  A kernel unrolled for 16 slots was 11 to 28 % more code than one
// for 10, and at a few rows, where the kernel's code runs about once per call,
// the smaller kernels were 4 to 10 % faster on GB300 (C4 T=1 5.29 -> 5.07 us,
// R=4 k=8 T=1 4.02 -> 3.63).  (The many-CTA finalize with a workspace, its
// time set by the hand-off of each row between CTAs through global memory,
// showed no consistent gain and keeps 16.)
inline int cluster_slots(bool fin, int k)
{
    return !fin ? 0 : k <= 4 ? 4 : k <= 8 ? 8 : k <= 10 ? 10 : kMaxK;
}

// Dynamic shared memory: the slice's finalize results, [R][slice] 16-byte chunks.
inline size_t cluster_smem_bytes(int R, int slice) { return (size_t)R * (size_t)slice * 16u; }

// Enqueue one cluster of cs CTAs per token row (grid T * cs).  fin selects the
// finalize tasks (expert rows, c.a.k of them a task) or the partial rows of the
// reduce entry points; postnorm the sandwich or the single pre-RMSNorm; tpt is
// 1 or 2.
cudaError_t launch_cluster_fin(const ClusterArgs &c, bool fin, bool postnorm, int tpt, int cs,
                               bool pdl, cudaStream_t st);

// Clusters of this shape the device holds at once (0 if none), for the planner;
// tiny selects the kernel with the second pass over rows of tiny values
// (Args::tiny), which launch_cluster_fin takes from c.a.tiny.
int cluster_fin_resident(bool fin, int k, bool postnorm, int tpt, bool tiny, int cs, size_t smem,
                         cudaError_t *err);

}  // namespace bn
