// bn_internal.h -- shared between the C-ABI translation unit and the kernel
// translation units of libbeamnorm (not installed, not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace bn {

// Mode bits of the main kernel template.  Each served entry point is one mode.
enum : int {
    F_FIN = 1,        // sources are gathered expert rows, finalized per shard
    F_SUM_IN = 2,     // the source is one FP32 reduced-sum row (epilogue only)
    F_POSTNORM = 4,   // post-RMSNorm of the reduced sum before the residual add
    F_RESNORM = 8,    // residual add, residual write-back, pre-RMSNorm -> out
    F_SUM_OUT = 16,   // write the FP32 reduced sum (first half of the split)
    F_Z_OUT = 32,     // write the per-shard BF16 finalize results only
};

constexpr int kModeReduceNorm = F_POSTNORM | F_RESNORM;
constexpr int kModeFinReduceNorm = F_FIN | F_POSTNORM | F_RESNORM;
constexpr int kModeReduceResNorm = F_RESNORM;
constexpr int kModeFinReduceResNorm = F_FIN | F_RESNORM;
constexpr int kModeReduceOnly = F_SUM_OUT;
constexpr int kModeFinReduceOnly = F_FIN | F_SUM_OUT;
constexpr int kModeNormOnly = F_SUM_IN | F_POSTNORM | F_RESNORM;
constexpr int kModeFinOnly = F_FIN | F_Z_OUT;
constexpr int kModeResNormOnly = F_SUM_IN | F_RESNORM;

constexpr int kMaxR = 16;
constexpr int kMaxK = 16;
constexpr int kMaxMeta = 256;        // R * k slots staged per token row
constexpr int kMaxH = 32768;         // fused entry points (whole-row epilogue in one launch)
constexpr int kMaxPieceH = 131072;   // unfused pieces (the fallback when a fused call declines)
constexpr int kMaxConsumers = 512;   // consumer threads per CTA
constexpr int kMaxCpt = 4;           // 16-byte chunks per consumer thread: 1, 2 or 4
constexpr int kMaxCptFin = 2;        // the same for the finalize modes: 1 or 2
constexpr int kMaxStages = 64;
constexpr int kMaxCluster = 16;

// Kernel arguments (passed by value).
struct Args {
    const uint16_t *src;      // partials [R,T,H] or expert_out [R,T*k,H]
    const float *sum_in;      // [T,H] FP32 (F_SUM_IN)
    const int32_t *perm;      // [R,T,k]
    const float *w;           // [R,T,k]
    const uint16_t *shared;   // [R,T,H] or null
    uint16_t *residual;       // [T,H] read, then written
    const float *gamma_post;  // [H]
    const float *gamma_pre;   // [H]
    uint16_t *out;            // [T,H]
    float *sum_out;           // [T,H] (F_SUM_OUT, or debug)
    float *ss_out;            // [T,2] debug
    uint16_t *z_out;          // [R,T,H] (F_Z_OUT, or debug)
    unsigned *err;            // device error word
    int R, T, H, k;
    int nchunks;              // H / 8 sixteen-byte chunks per row
    int stages;               // pipeline depth
    int stage_bytes;          // bytes of one stage = group * item_bytes
    int group;                // row copies (items) per stage
    int item_bytes;           // stride of one item in a stage (multiple of 128)
    int gamma_bytes;          // shared-memory bytes of the per-thread gamma slots
    int gamma_stride;         // 16-byte slots per gamma half: the largest column slice in chunks
    int zbuf_bytes;           // shard split: shared-memory bytes of one full z row
    int spin_wait;            // 1: poll barriers with test_wait; 0: try_wait
    int wait_polls;           // polls after which a pipeline wait gives up (0: the default)
    int tiny;                 // 1: the kernel with the second pass over rows of tiny values
    float eps;
};

// A row whose sum of squares is below 2^-80 has squares in or near FP32's
// subnormal range, where the compensated sum is inexact (an error below
// H * 2^-150); the kernels built with a second, rescaled pass over such rows
// (TINY) restore the exactly accumulated sum rounded once.  The pass can
// change an output only when eps < 2^-50: for any larger eps the RMS factor's
// sum fl(fl(ss / H) + eps) is eps itself for both sums (ss / H < 2^-79, below
// half the FP32 spacing at eps, which is at least eps * 2^-24 >= 2^-74).  The
// planner takes the TINY kernels for eps < 2^-50 (or NaN) only; elsewhere
// the pass would change nothing but the debug sums of squares.
constexpr float kTinyPassEps = 0x1p-50f;

// Launch shape chosen on the host.
struct Launch {
    int split;       // 1: the CTAs of a cluster split a row by shard (finalize modes)
    int cluster;     // CTAs per token row (thread-block cluster size)
    int consumers;   // consumer threads per CTA (multiple of 32)
    int cpt;         // 16-byte chunks per consumer thread: 1, 2 or 4
    int grid;        // CTAs (a multiple of cluster)
    size_t smem;     // dynamic shared memory bytes
    int pdl;         // 1: programmatic dependent launch (setup overlaps the previous kernel)
    int full;        // 1: every slice is exactly cpt * consumers chunks (unchecked kernel)
    int tiny;        // 1: the kernel with the second pass over rows of tiny values (Args::tiny)
};

// Dynamic shared-memory layout, identical on host and device.
struct SmemLayout {
    uint32_t stages_off, gamma_off, zbuf_off, bars_off, red_off, xslot_off, meta_off, total;
    __host__ __device__ static SmemLayout make(int stages, int stage_bytes, int gamma_bytes,
                                               int zbuf_bytes, bool fin) {
        SmemLayout L;
        L.stages_off = 0;
        L.gamma_off = (uint32_t)stages * (uint32_t)stage_bytes;           // 128-aligned
        L.zbuf_off = L.gamma_off + (((uint32_t)gamma_bytes + 127u) & ~127u);
        L.bars_off = L.zbuf_off + (((uint32_t)zbuf_bytes + 127u) & ~127u);
        // full, empty, meta x2 x2, exchange x2, z ready
        uint32_t nbars = 2u * (uint32_t)stages + 7u;
        L.red_off = L.bars_off + ((nbars * 8u + 15u) & ~15u);
        L.xslot_off = L.red_off + 2u * 32u * 8u;                          // float2 [2][32]
        L.meta_off = L.xslot_off + 2u * (uint32_t)kMaxCluster * 8u;       // float2 [2][16]
        // gather indices and weights (finalize modes only): int32 + float [2][256]
        L.total = L.meta_off + (fin ? 2u * (uint32_t)kMaxMeta * 8u : 0u);
        return L;
    }
};

// Shared-memory bytes of the gamma slots: 32 bytes per chunk per gamma.
__host__ __device__ inline int gamma_slot_bytes(int mode, int slice_chunks)
{
    if (!(mode & F_RESNORM)) return 0;
    const int ngamma = (mode & F_POSTNORM) ? 2 : 1;
    return ngamma * 32 * slice_chunks;
}

// Per-mode host entry points, defined in the kernel translation units:
//   launch_<mode>     enqueue the kernel with the given launch shape;
//   occupancy_<mode>  resident clusters on the whole current device for that
//                     shape (0 if it cannot be resident); sets the kernel's
//                     shared-memory and cluster attributes for the device first.
#define BN_DECLARE_MODE(name)                                                   \
    cudaError_t launch_##name(const Args &, const Launch &, cudaStream_t);      \
    int occupancy_##name(const Launch &, cudaError_t *);
BN_DECLARE_MODE(reduce_norm)
BN_DECLARE_MODE(fin_reduce_norm)
BN_DECLARE_MODE(reduce_resnorm)
BN_DECLARE_MODE(fin_reduce_resnorm)
BN_DECLARE_MODE(reduce_only)
BN_DECLARE_MODE(fin_reduce_only)
BN_DECLARE_MODE(norm_only)
BN_DECLARE_MODE(fin_only)
BN_DECLARE_MODE(resnorm_only)
#undef BN_DECLARE_MODE

}  // namespace bn
