// bn_abi.cu -- the C ABI of libbeamnorm: host-side validation, the choice of
// launch shape, launches, and the device error word.
//
// Every entry point validates its arguments on the host before any CUDA call
// and either enqueues exactly one kernel on the caller's stream or enqueues
// nothing (bn_finalize_reduce_norm_noalloc first clears its scratch counters
// with one memset on the same stream).  Declining a valid shape (BN_ERR_UNSUPPORTED) never does part of
// the work: the caller falls back to an unfused path and owes the whole
// reduction (sglang pull request 34134, description: a decline must not skip
// the owed all-reduce).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/beamnorm.h"
#include "bn_cluster.h"
#include "bn_internal.h"
#include "bn_wide.h"

// The device error word: one per device that loads the library.  Kernels
// receive its address; they set bits with atomicOr and never trap.
__device__ unsigned g_bn_device_error;

namespace bn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kVersion = 10200;  // 1.2.0

thread_local char g_msg[512] = "";

bn_status fail(bn_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

bn_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(BN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---- tuning overrides (process-wide) -------------------------------------------

std::atomic<int> g_tune_cluster{0}, g_tune_stages{0}, g_tune_threads{0}, g_tune_ctas{0},
    g_tune_wait{0}, g_tune_group{0}, g_tune_split{0}, g_tune_pdl{0}, g_tune_polls{0},
    g_tune_tiny{0};

// 1 if a call of this mode runs the kernel with the second pass over rows of
// tiny values: modes with the norms, eps below kTinyPassEps (or NaN), unless
// the tuning says otherwise.
int tiny_for(int mode, float eps)
{
    if (!(mode & F_RESNORM)) return 0;
    const int t = g_tune_tiny.load();
    if (t != 0) return t == 2 ? 1 : 0;
    return eps >= kTinyPassEps ? 0 : 1;
}

// ---- per-device state ------------------------------------------------------------

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;      // dynamic + static shared memory one CTA may use
    int smem_per_sm = 0;     // shared memory of one SM
    int smem_reserved = 0;   // shared memory the system reserves per CTA
    unsigned *err = nullptr;  // address of g_bn_device_error on this device
};

std::once_flag g_dev_once[kMaxDevices];
DeviceInfo g_dev[kMaxDevices];
cudaError_t g_dev_status[kMaxDevices];

bn_status device_info(const DeviceInfo **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(BN_ERR_CUDA, "device ordinal %d out of range", dev);
    std::call_once(g_dev_once[dev], [dev]() {
        DeviceInfo &d = g_dev[dev];
        cudaError_t st = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (st == cudaSuccess)
            st = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (st == cudaSuccess)
            st = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (st == cudaSuccess)
            st = cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (st == cudaSuccess)
            st = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_bn_device_error);
        g_dev_status[dev] = st;
    });
    if (g_dev_status[dev] != cudaSuccess) return cuda_fail(g_dev_status[dev], "device setup");
    *out = &g_dev[dev];
    return BN_OK;
}

// ---- validation helpers ----------------------------------------------------------

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    const void *p;
    size_t bytes;
    const char *name;
};

bool overlaps(const Range &x, const Range &y)
{
    if (!x.p || !y.p || x.bytes == 0 || y.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(x.p), a1 = a0 + x.bytes;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(y.p), b1 = b0 + y.bytes;
    return a0 < b1 && b0 < a1;
}

// Each written range must not overlap any other range in the list (the
// residual is read and written through one pointer, which is intended).
bn_status check_overlaps(const Range *writes, int nw, const Range *reads, int nr)
{
    for (int i = 0; i < nw; ++i) {
        for (int j = 0; j < nr; ++j)
            if (overlaps(writes[i], reads[j]))
                return fail(BN_ERR_INVALID, "%s overlaps %s", writes[i].name, reads[j].name);
        for (int j = i + 1; j < nw; ++j)
            if (overlaps(writes[i], writes[j]))
                return fail(BN_ERR_INVALID, "%s overlaps %s", writes[i].name, writes[j].name);
    }
    return BN_OK;
}

bn_status check_shape(int R, int T, int k, int H, bool fin)
{
    if (R < 1 || R > kMaxR) return fail(BN_ERR_INVALID, "R=%d outside [1, %d]", R, kMaxR);
    if (fin && (k < 1 || k > kMaxK)) return fail(BN_ERR_INVALID, "k=%d outside [1, %d]", k, kMaxK);
    if (T < 0) return fail(BN_ERR_INVALID, "T=%d is negative", T);
    if (H <= 0) return fail(BN_ERR_INVALID, "H=%d is not positive", H);
    if (H % 8 != 0) return fail(BN_ERR_INVALID, "H=%d is not a multiple of 8", H);
    return BN_OK;
}

// A valid shape that is not served is declined.  The fused entry points serve
// rows up to kMaxH; the unfused pieces, which the caller falls back to when a
// fused call declines, split a row over clusters of up to 16 CTAs and serve
// rows up to kMaxPieceH.
bn_status check_served(int R, int T, int k, int H, bool fin, bool piece = false)
{
    const int max_h = piece ? kMaxPieceH : kMaxH;
    if (H > max_h)
        return fail(BN_ERR_UNSUPPORTED, "H=%d above the served maximum %d of the %s", H, max_h,
                    piece ? "unfused pieces" : "fused entry points");
    if (fin && R * k > kMaxMeta)
        return fail(BN_ERR_UNSUPPORTED, "R*k=%d above the served maximum %d", R * k, kMaxMeta);
    if (fin && (long long)T * k >= (1LL << 31))
        return fail(BN_ERR_UNSUPPORTED, "T*k=%lld does not fit int32 row indices", (long long)T * k);
    (void)R;
    return BN_OK;
}

bn_status check_eps(float eps)
{
    if (!(eps >= 0.0f) || !std::isfinite(eps))
        return fail(BN_ERR_INVALID, "eps must be finite and non-negative");
    return BN_OK;
}

#define BN_REQUIRE(cond, ...)                                      \
    do {                                                           \
        if (!(cond)) return fail(BN_ERR_INVALID, __VA_ARGS__);     \
    } while (0)
#define BN_TRY(expr)                         \
    do {                                     \
        bn_status _st = (expr);              \
        if (_st != BN_OK) return _st;        \
    } while (0)

bn_status check_ptr16(const void *p, const char *name, bool required = true)
{
    if (!p) {
        if (required) return fail(BN_ERR_INVALID, "%s is NULL", name);
        return BN_OK;
    }
    if (!aligned(p, 16)) return fail(BN_ERR_INVALID, "%s is not 16-byte aligned", name);
    return BN_OK;
}

bn_status check_ptr4(const void *p, const char *name)
{
    if (!p) return fail(BN_ERR_INVALID, "%s is NULL", name);
    if (!aligned(p, 4)) return fail(BN_ERR_INVALID, "%s is not 4-byte aligned", name);
    return BN_OK;
}

// ---- launch shape ----------------------------------------------------------------

using LaunchFn = cudaError_t (*)(const Args &, const Launch &, cudaStream_t);
using OccFn = int (*)(const Launch &, cudaError_t *);

struct ModeOps {
    int mode;
    LaunchFn launch;
    OccFn occupancy;
    const char *name;
};

const ModeOps kOps[] = {
    {kModeReduceNorm, launch_reduce_norm, occupancy_reduce_norm, "reduce_norm"},
    {kModeFinReduceNorm, launch_fin_reduce_norm, occupancy_fin_reduce_norm, "finalize_reduce_norm"},
    {kModeReduceResNorm, launch_reduce_resnorm, occupancy_reduce_resnorm, "reduce_residual_norm"},
    {kModeFinReduceResNorm, launch_fin_reduce_resnorm, occupancy_fin_reduce_resnorm,
     "finalize_reduce_residual_norm"},
    {kModeReduceOnly, launch_reduce_only, occupancy_reduce_only, "reduce_only"},
    {kModeFinReduceOnly, launch_fin_reduce_only, occupancy_fin_reduce_only, "finalize_reduce_only"},
    {kModeNormOnly, launch_norm_only, occupancy_norm_only, "norm_only"},
    {kModeFinOnly, launch_fin_only, occupancy_fin_only, "finalize_only"},
    {kModeResNormOnly, launch_resnorm_only, occupancy_resnorm_only, "residual_norm_only"},
};

// The operations of bn_op, in its order.
const int kModeOfOp[] = {kModeReduceNorm,       kModeFinReduceNorm, kModeReduceResNorm,
                         kModeFinReduceResNorm, kModeReduceOnly,    kModeFinReduceOnly,
                         kModeNormOnly,         kModeFinOnly,       kModeResNormOnly};
constexpr int kNumOps = (int)(sizeof kModeOfOp / sizeof kModeOfOp[0]);

// The unfused pieces: the modes that write the FP32 sum or the finalize
// results, or that start from the FP32 sum.
bool is_piece(int mode) { return (mode & (F_SUM_OUT | F_Z_OUT | F_SUM_IN)) != 0; }

const ModeOps &ops_for(int mode)
{
    for (const ModeOps &o : kOps)
        if (o.mode == mode) return o;
    return kOps[0];
}

// Occupancy answers are cached: (device, mode, shape) -> resident clusters.
struct OccEntry {
    int dev, mode, split, full, cluster, consumers, cpt;
    size_t smem;
    int clusters;
};
constexpr int kOccCache = 256;
OccEntry g_occ[kOccCache];
int g_occ_n = 0;
std::mutex g_occ_mu;

bn_status resident_clusters(int mode, const Launch &l, int *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    {
        std::lock_guard<std::mutex> g(g_occ_mu);
        for (int i = 0; i < g_occ_n; ++i) {
            const OccEntry &o = g_occ[i];
            if (o.dev == dev && o.mode == mode && o.split == l.split && o.full == l.full &&
                o.cluster == l.cluster &&
                o.consumers == l.consumers && o.cpt == l.cpt && o.smem == l.smem) {
                *out = o.clusters;
                return BN_OK;
            }
        }
    }
    int n = ops_for(mode).occupancy(l, &e);
    if (e != cudaSuccess) {
        cudaGetLastError();  // occupancy queries leave no sticky error; clear the last one
        n = 0;
    }
    {
        std::lock_guard<std::mutex> g(g_occ_mu);
        if (g_occ_n < kOccCache)
            g_occ[g_occ_n++] = OccEntry{dev, mode, l.split, l.full, l.cluster, l.consumers, l.cpt, l.smem, n};
    }
    *out = n;
    return BN_OK;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// CTAs per token row for the finalize modes' column split (few finalize rows
// take the shard split instead).  A cluster splits a row only when the rows alone would
// leave SMs idle and a row is heavy enough (about 192 KB of copies per CTA)
// to repay the two cluster-wide exchanges; each CTA keeps at least 32 chunks.
int auto_cluster(int T, int nchunks, int sms, long long row_bytes)
{
    int by_rows = 1;
    while (by_rows < kMaxCluster && (long long)T * by_rows * 2 <= sms) by_rows *= 2;
    int by_bytes = 1;
    while (by_bytes < kMaxCluster && (long long)by_bytes * 2 * 192 * 1024 <= row_bytes) by_bytes *= 2;
    int cs = by_rows < by_bytes ? by_rows : by_bytes;
    while (cs > 1 && nchunks / cs < 32) cs /= 2;
    return cs;
}

// CTAs per token row for the reduce modes: while rows are few and heavy, a
// cluster splits each row so that more SMs work on it: up to 8 CTAs, each
// keeping at least 64 chunks, while T * CTAs * 1 KB stays within the bytes one
// row moves.  Measured on GB300 (us per call, CUDA graph, L2-cold; clusters
// of 1 / 2 / 4 / 8): R=8, H=8192 (180 KB a row) at T=12 6.24 / 5.74 / 5.33 /
// 5.20, T=24 6.30 / 5.81 / 5.46 / 5.49, T=40 6.40 / 6.05 / 6.15 / 6.50, T=64
// 6.56 / 6.53 / 7.16, T=100 7.33 / 9.57 / 8.48 / 10.48; R=4, H=5120 (70 KB)
// at T=12 3.99 / 4.15 / 3.78 / 3.90, T=24 4.29 / 4.67 / 4.35, T=40 4.38 /
// 4.83 / 4.66, T=64 4.50 / 4.96 / 4.98, T=100 4.79 / 5.36 / 6.03.  (T <= 8
// takes the cluster path of bn_cluster.cu where rows are heavy enough.)
int auto_cluster_reduce(int T, int nchunks, long long row_bytes)
{
    int cs = 1;
    while (cs < 8 && (long long)T * cs * 2 * 1024 <= row_bytes && nchunks / (cs * 2) >= 64) cs *= 2;
    return cs;
}

// Copies the producer of one CTA issues per token row (cs: the cluster size of
// a shard split, whose CTAs take R / cs shards each).
int loads_per_row(int mode, const Args &a, bool split, int cs)
{
    if (mode & F_SUM_IN) return 2;
    int n = (mode & F_FIN) ? (split ? a.R / cs : a.R) * (a.k + (a.shared ? 1 : 0)) : a.R;
    if (mode & F_RESNORM) n += 1;
    return n;
}

// Launch shape:
//   cluster   CTAs per row (automatic: split rows while rows alone leave SMs idle);
//   consumers up to `cap` threads per CTA (0: 256 for the reduce modes, 512
//             for the finalize modes), each owning CPT 16-byte chunks of the
//             CTA's slice;
//   CTAs/SM   as many as registers and threads allow (at most 4), so that the
//             per-row reductions of one CTA overlap another CTA's streaming,
//             but no more than the rows put on one SM when one CTA takes a row;
//   stages    the SM's shared memory split over those CTAs, capped at two rows
//             of copies ahead.
// Narrow rows take two chunks per thread down to this many consumer threads
// per CTA, and light reduce rows (at most kLightReduceMaxR shards) cap their
// CTAs at it (see shape_for).
constexpr int kNarrowMinConsumers = 128;
constexpr int kLightReduceMaxR = 4;

// One launch shape for a given row split.  Sets *resident to the clusters the
// device holds at once (0: this shape cannot be resident).
bn_status shape_for(int mode, Args *a, const DeviceInfo *d, bool split, int cs, int cap_in,
                    Launch *l, int *resident)
{
    const int H = a->H;
    const bool sum_in = (mode & F_SUM_IN) != 0;
    const bool fin = (mode & F_FIN) != 0;
    const int nchunks = H / 8;
    const int per_row = loads_per_row(mode, *a, split, cs);
    // measured on GB300: the finalize modes run best with 512 consumer threads
    // (one CTA per SM), the reduce modes with 256 and several CTAs per SM, and
    // the light reduce rows (R <= 4 shards summed, one CTA a row, more rows
    // than SMs) with 128 and up to 4 chunks a thread, which puts more rows in
    // flight per SM.  Light rows (us per call, T=4096, default / 128
    // threads): R=2 H=4096 38.9 / 32.6, R=4 H=4096 46.1 / 41.4, R=4 H=2048
    // 31.3 / 24.1; R=8 H=4096 is slower with 128 (56.6 / 61.2), and so is a
    // row that has an SM to itself (R=4 H=5120 T=64: 4.49 / 4.88).
    const bool light = !fin && !sum_in && (mode & F_RESNORM) && a->R <= kLightReduceMaxR &&
                       cs == 1 && a->T > d->sms;
    const int cap = g_tune_threads.load() > 0 ? g_tune_threads.load()
                    : cap_in > 0               ? cap_in
                    : fin                      ? kMaxConsumers
                    : light                    ? kNarrowMinConsumers
                                               : 256;
    const int want_stages = g_tune_stages.load();
    const int want_ctas = g_tune_ctas.load();
    *resident = 0;

    // chunks one CTA's threads must cover: the column slice, or the whole row
    // when a cluster splits rows by shard
    const int nch_max = split ? nchunks : (nchunks + cs - 1) / cs;
    // At most 4 chunks per thread (2 for the finalize modes): above that a
    // slice takes more threads (up to 512), then a larger cluster.  The
    // 8-chunk kernels spilled (finalize 900-1500 bytes, its 4-chunk kernels
    // 30-90) and lost to wider splits (see plan()).
    const int max_cpt = fin ? kMaxCptFin : kMaxCpt;
    int cpt = 1;
    while (cpt < max_cpt && (nch_max + cpt - 1) / cpt > cap) cpt *= 2;
    // Narrow rows (column split, threads automatic): two chunks per thread as
    // soon as a CTA still has 4 consumer warps, so that 2 to 4 CTAs share an
    // SM instead of one wide CTA.  Measured on GB300 (us per call; one CTA of
    // 1 chunk a thread / CTAs of 2): finalize R=8, k=8, T=1024 H=4096 143.3 /
    // 110.0 (T=4096 542 / 385), H=3072 135.4 / 89.4, H=2048 129.2 / 66.0
    // (3 CTAs of 128 threads); reduce R=8, H=2048, T=4096 38.9 / 30.8.  Reduce
    // rows split over a cluster, or with an SM each, keep one chunk a thread
    // (R=2, H=4096, T=16 over 2-CTA clusters: 3.38 / 3.54).
    const bool sums_rows = !sum_in && (fin || ((mode & F_RESNORM) != 0 && cs == 1 && a->T > d->sms));
    if (sums_rows && !split && cpt == 1 && max_cpt >= 2 && cap_in == 0 &&
        g_tune_threads.load() == 0 && nch_max >= 2 * kNarrowMinConsumers)
        cpt = 2;
    const int consumers = round_up((nch_max + cpt - 1) / cpt, 32);
    if (consumers > kMaxConsumers)
        return fail(BN_ERR_UNSUPPORTED, "row of %d chunks needs %d consumer threads", nch_max, consumers);
    const int item_bytes = round_up(nch_max * 16 * (sum_in ? 2 : 1), 128);
    const int slice = (nchunks + cs - 1) / cs;  // the largest column slice of the epilogue
    const int gamma_bytes = gamma_slot_bytes(mode, slice);
    // shard split: each CTA's z buffer holds R rows of its column slice
    const int zbuf_bytes =
        (split && !(mode & F_Z_OUT)) ? round_up(a->R * ((nchunks + cs - 1) / cs) * 16, 128) : 0;
    const int cta_max = d->smem_optin - 1024;  // room for the kernel's static shared memory

    Launch L;
    L.split = split ? 1 : 0;
    L.cluster = cs;
    L.consumers = consumers;
    L.cpt = cpt;
    L.pdl = 0;
    // every CTA's slice (the whole row for a shard split's finalize) exactly
    // cpt chunks per consumer thread: the kernel without those bounds checks
    L.full = split ? (nchunks == cpt * consumers ? 1 : 0)
                   : (nchunks % cs == 0 && nchunks / cs == cpt * consumers ? 1 : 0);
    L.tiny = a->tiny;
    // CTAs per SM that registers and threads allow (probe with the smallest
    // ring: two stages of one copy)
    Launch probe = L;
    probe.cluster = 1;
    probe.smem = SmemLayout::make(2, item_bytes, gamma_bytes, zbuf_bytes, fin).total;
    int resident_probe = 0;
    BN_TRY(resident_clusters(mode, probe, &resident_probe));
    int by_regs = resident_probe / (d->sms > 0 ? d->sms : 1);
    if (by_regs < 1) by_regs = 1;
    int ctas = want_ctas > 0 ? want_ctas : (by_regs < 4 ? by_regs : 4);
    if (ctas > by_regs) ctas = by_regs;
    // One CTA per row and fewer rows than CTA slots: the ring is sized for the
    // CTAs that will share an SM.  Measured on GB300, C1 (R=4, H=5120) at
    // T=256: 256 CTAs with rings sized for 3 per SM 8.69 us, for 2 per SM 6.94.
    if (!split && cs == 1 && want_ctas == 0 && want_stages == 0 && d->sms > 0) {
        const int fill = (a->T + d->sms - 1) / d->sms;
        if (fill >= 1 && fill < ctas) ctas = fill;
    }

    // One stage holds `group` row copies of item_bytes each.  Measured on
    // GB300: the finalize modes gain from about 48 KB of stages per SM (fewer
    // handshakes over their many gathered copies), split between the CTAs
    // that share it (R=8, k=8, H=4096, 2 CTAs: stages of 16, 24 and 32 KB
    // 111.2, 110.0 and 115.0 us); the reduce modes run best with one copy per
    // stage, and their kernels assume it (no item cursor).
    int group = g_tune_group.load() > 0 ? g_tune_group.load()
                                        : (fin ? (48 * 1024) / (ctas * item_bytes) : 1);
    if (!fin) group = 1;
    if (group > per_row) group = per_row;
    if (group < 1) group = 1;
    // A group is shrunk until two stages fit one CTA, or three when the group
    // is automatic (measured, shard split of C4 at T=64: 2 stages of 3 copies
    // 27.9 us, 3 stages of 2 copies 26.1 us).
    const int min_stages = g_tune_group.load() > 0 ? 2 : 3;
    while (group > 1 && (int)SmemLayout::make(min_stages, group * item_bytes, gamma_bytes, zbuf_bytes,
                                              fin).total > cta_max)
        --group;
    const int stage_bytes = group * item_bytes;
    const int stages_per_row = (per_row + group - 1) / group;
    const int overhead = (int)SmemLayout::make(0, stage_bytes, gamma_bytes, zbuf_bytes, fin).total;

    // the kernel's own static shared memory is 128 bytes; the occupancy check
    // below drops a stage if the estimate was one too many
    int per_cta = d->smem_per_sm / ctas - d->smem_reserved - 128;
    if (per_cta > cta_max) per_cta = cta_max;

    int stages;
    if (want_stages > 0) {
        stages = want_stages;
    } else {
        stages = (per_cta - overhead) / stage_bytes;
        const int ahead = 2 * stages_per_row + 2;
        if (stages > ahead) stages = ahead;
    }
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    while (stages > 2 &&
           (int)SmemLayout::make(stages, stage_bytes, gamma_bytes, zbuf_bytes, fin).total > cta_max)
        --stages;
    if ((int)SmemLayout::make(stages, stage_bytes, gamma_bytes, zbuf_bytes, fin).total > cta_max)
        return fail(BN_ERR_UNSUPPORTED, "stage of %d bytes does not fit shared memory", stage_bytes);
    L.smem = SmemLayout::make(stages, stage_bytes, gamma_bytes, zbuf_bytes, fin).total;

    BN_TRY(resident_clusters(mode, L, resident));
    // keep the intended CTAs per SM: one stage less if the ring estimate overshot
    if (want_stages == 0 && cs == 1 && stages > 2 && *resident < ctas * d->sms) {
        --stages;
        L.smem = SmemLayout::make(stages, stage_bytes, gamma_bytes, zbuf_bytes, fin).total;
        BN_TRY(resident_clusters(mode, L, resident));
    }
    if (*resident <= 0) return BN_OK;
    const int ncl = a->T < *resident ? a->T : *resident;
    L.grid = ncl * cs;
    // programmatic dependent launch: the launch and this kernel's setup
    // overlap the previous kernel in the stream (about 1 us per call measured)
    L.pdl = g_tune_pdl.load() == 1 ? 0 : 1;
    *l = L;
    a->stages = stages;
    a->stage_bytes = stage_bytes;
    a->group = group;
    a->item_bytes = item_bytes;
    a->gamma_bytes = gamma_bytes;
    a->gamma_stride = slice;
    a->zbuf_bytes = zbuf_bytes;
    a->spin_wait = g_tune_wait.load() == 2 ? 1 : 0;
    a->wait_polls = g_tune_polls.load();
    a->nchunks = nchunks;
    a->err = d->err;
    return BN_OK;
}

// Consumer threads one SM runs for a shape, and the most token rows one SM
// takes (rows per CTA on the busiest CTA times the CTAs that share an SM).
void sm_load(const Launch &l, int resident, int T, int sms, long long *threads, long long *rows)
{
    const int per_sm = resident / (sms > 0 ? sms : 1);
    const int grid = l.grid > 0 ? l.grid : 1;
    int sharing = (grid + sms - 1) / (sms > 0 ? sms : 1);
    if (sharing > per_sm) sharing = per_sm;
    if (sharing < 1) sharing = 1;
    *threads = (long long)l.consumers * sharing;
    *rows = (long long)((T + grid - 1) / grid) * sharing;
}

// Reduce rows with one CTA per row: the default shape (up to 256 consumer
// threads, several CTAs per SM) against one with up to 512 threads per CTA
// (at least 2 chunks per thread).  The wider shape is taken when an SM runs
// at least as many consumer threads with it and takes no more rows, and it
// is better on one of the two.  Measured on GB300 (us per call):
//   R=8, H=8192 (2 CTAs x 256 threads / 1 CTA x 512 per SM): T=256 12.24 /
//     12.51 (same threads and rows per SM: kept), T=1024 34.7 / 31.85,
//     T=4096 113.3 / 108.2;
//   R=8, H=16384, T=1024 (1 CTA x 256 threads of 8 chunks / 1 x 512 of 4):
//     93.5 / 67.3;
//   R=4, H=5120 keeps 3 CTAs x 160 threads against 1 x 320 (T=1024 18.0 /
//     20.4); R=8, H=4096 keeps 256 threads (512 would take 1 chunk each:
//     T=1024 19.1 / 24.2).
// With more rows than SMs, only heavy rows (at least kWideMinR shards) of at
// least kWideMinChunks chunks are offered the wider shape: elsewhere one CTA
// per SM left the row-wide reductions without a second CTA to overlap them,
// whatever the two figures said.  Measured (T=4096, default / wide): R=8
// H=7168 96.7 / 101.5, R=4 H=8192 78.5 / 88.2, R=4 H=7168 66.4 / 82.1, R=2
// H=8192 61.1 / 77.2.  A row with an SM to itself keeps the wider CTA
// (R=4, H=5120, T=64: 4.49 against 4.88 with 160 threads).
constexpr int kWideMinR = 8;
constexpr int kWideMinChunks = 1024;

bn_status wider_ctas(int mode, Args *a, const DeviceInfo *d, Launch *l, int resident)
{
    Args wa = *a;
    Launch wl{};
    int wres = 0;
    const bn_status st = shape_for(mode, &wa, d, false, 1, kMaxConsumers, &wl, &wres);
    if (st == BN_ERR_UNSUPPORTED || wres <= 0) return BN_OK;
    if (st != BN_OK) return st;
    if (wl.cpt < 2 || wl.consumers <= l->consumers) return BN_OK;
    long long th0, rows0, th1, rows1;
    sm_load(*l, resident, a->T, d->sms, &th0, &rows0);
    sm_load(wl, wres, a->T, d->sms, &th1, &rows1);
    if (th1 >= th0 && rows1 <= rows0 && (th1 > th0 || rows1 < rows0)) {
        *a = wa;
        *l = wl;
    }
    return BN_OK;
}

// Launch shape: the row split (by shard for finalize rows when rows are few,
// else by column slices over a cluster of `cs` CTAs), consumer threads, CTAs
// per SM and pipeline depth; see shape_for.
bn_status plan(int mode, Args *a, Launch *l)
{
    const DeviceInfo *d = nullptr;
    BN_TRY(device_info(&d));
    a->tiny = tiny_for(mode, a->eps);
    const int T = a->T, H = a->H;
    const int nchunks = H / 8;
    int resident = 0;

    // Shard split: finalize modes with an epilogue (or the finalize alone),
    // R >= 2, few rows.  The cluster takes the largest size cs dividing R
    // whose clusters all fit on the device at once for these T rows (one
    // wave); each CTA finalizes R / cs shards.  Measured on GB300 (R=8,
    // H=8192, k=10; shard / column split): T=1 12.1 / 30 us, T=16 22.0 / 28.5
    // us with cs=8 (15 resident clusters: two waves).
    const bool can_split = (mode & F_FIN) && (mode & (F_RESNORM | F_Z_OUT)) && a->R >= 2;
    const int pref = g_tune_split.load();
    if (can_split && (pref == 2 || (pref == 0 && (long long)T * a->R <= 512))) {
        const int want_cs = g_tune_cluster.load();
        for (int c = a->R < kMaxCluster ? a->R : kMaxCluster; c >= 2; --c) {
            if (a->R % c != 0 || (want_cs > 0 && c != want_cs)) continue;
            const bn_status st = shape_for(mode, a, d, true, c, 0, l, &resident);
            if (st == BN_ERR_UNSUPPORTED) continue;  // this cluster's CTAs do not fit
            if (st != BN_OK) return st;
            if (resident > 0 && (pref == 2 || T <= resident)) return BN_OK;
        }
    }

    const int want_cs = g_tune_cluster.load();
    int cs = want_cs;
    if (cs <= 0) {
        cs = (mode & F_FIN) ? auto_cluster(T, nchunks, d->sms, (long long)loads_per_row(mode, *a, false, 1) * 2 * H)
                            : auto_cluster_reduce(T, nchunks, ((long long)loads_per_row(mode, *a, false, 1) * 2 + 4) * H);
        // Wide rows split over a cluster until a CTA's slice is at most 1024
        // chunks (finalize) or 1536 (the others).  Measured on GB300 (us per
        // call, CUDA graph, L2-cold; the smallest cluster that fits shared
        // memory / this rule): reduce R=8 H=16384 T=1024 68.0 / 64.5, R=8
        // H=32768 T=300 63.4 / 42.1, R=4 H=24576 T=1024 146.7 / 74.6 (R=4
        // H=12288 stays one CTA a row: 33.5, against 38.0 with two);
        // finalize R=8 k=8 H=16384 T=256 135.4 / 114.7, R=8 k=4 H=32768 T=64
        // 46.8 / 37.8, R=4 k=2 H=12288 T=1024 87.6 / 84.3.
        const int max_slice = (mode & F_FIN) ? 1024 : 1536;
        while (cs < kMaxCluster && (nchunks + cs - 1) / cs > max_slice) cs *= 2;
    }
    if (cs > nchunks) cs = 1;
    // A slice too wide for one CTA's shared memory (gamma slots and two
    // stages: reduce rows above about 19 K elements at one CTA per row) takes
    // a larger cluster; a shape with no resident cluster takes a smaller one.
    for (int tried = 0; tried < 2 * kMaxCluster; ++tried) {
        const bn_status st = shape_for(mode, a, d, false, cs, 0, l, &resident);
        if (st == BN_OK && resident > 0) {
            if (!(mode & F_FIN) && cs == 1 && g_tune_threads.load() == 0 &&
                ((a->R >= kWideMinR && nchunks >= kWideMinChunks) || T <= d->sms))
                return wider_ctas(mode, a, d, l, resident);
            return BN_OK;
        }
        if (st != BN_OK && st != BN_ERR_UNSUPPORTED) return st;
        if (st == BN_ERR_UNSUPPORTED) {
            if (want_cs > 0 || cs * 2 > kMaxCluster || cs * 2 > nchunks) return st;
            cs *= 2;
        } else {
            if (cs <= 1) break;
            cs /= 2;
        }
    }
    return fail(BN_ERR_UNSUPPORTED, "no resident CTA for this shape");
}

// ---- the finalize with each row over a cluster, one task per thread --------------

// Token rows up to which the fused finalize entries take the cluster path
// when the planner leaves the choice to it, provided the clusters of all T
// rows fit on the device at once.  Measured on GB300 (us per call in a CUDA
// graph, L2-cold; cluster path with 16 CTAs a row / the default of the day):
// R=8, H=8192, k=10 at T=1 5.67 / 10.28 (shard split), T=4 6.75 / 10.47,
// T=12 10.34 / 11.59 (8-CTA clusters), T=16 20.5 / 14.3 (16-CTA clusters take
// two waves; with 8-CTA clusters 19.5, with 4 and four tasks a thread 17.1);
// R=8, H=6144, k=8 at T=1 5.07 / 8.85, T=16 18.4 / 12.1.
constexpr int kClusterFinMaxT = 15;
// The same for the fused reduce entry points, whose CTAs must also keep at
// least kClusterReduceMinTasks (shard, chunk) loads: light rows are faster on
// the main kernel.  Measured on GB300 (us per call, CUDA graph, L2-cold; main
// kernel / cluster path): R=8, H=8192 at T=1 4.55 / 3.34 (16 CTAs), T=8 5.03
// / 4.43 (8 CTAs); R=4, H=5120 at T=1 3.77 / 3.19 (8), T=8 3.83 / 3.48 (8);
// R=2, H=256 at T=8 2.60 / 2.83 (4); every case slower at T=64.
constexpr int kClusterReduceMaxT = 8;
constexpr int kClusterReduceMinTasks = 256;
// Past kClusterReduceMaxT rows, up to kClusterReduceMidMaxT, the reduce rows
// keep the cluster path with clusters of at most kClusterReduceMidMaxCs CTAs,
// all resident at once.  Measured on GB300 after the cluster kernels shrank
// (us per call, CUDA graph, L2-cold; main kernel / clusters of 8): R=8,
// H=8192 at T=16 5.52 / 4.61, T=24 5.37 / 4.88, T=32 5.90 / 4.96; R=4,
// H=5120 at T=16 3.69 / 3.05, T=32 4.49 / 4.16; R=8, H=4096 at T=16 5.05 /
// 3.44; R=2, H=8192 at T=16 3.40 / 3.11.  Clusters of 16 fell off between 192
// and 256 CTAs (R=8, H=8192: T=12 4.15, T=16 7.83), and at T=48 the clusters
// of 8 no longer fit at once (9.73 against 5.91).  Over R in {2, 4, 8}, H from
// 2048 to 12288 and T in {9, 12, 16, 24, 32} the rule lost to the main
// kernel by more than 3 % only at R=4, H=12288, T=24 and 32 (5.32 / 4.83,
// 5.50 / 4.96).  From kClusterReduceMidMaxT + 1 to kClusterReduceWideMaxT
// rows, rows of at least kClusterReduceWideMinR shards and at most 1024
// chunks take clusters of kClusterReduceMidMaxCs only, all resident at once
// (T=33: R=8, H=8192 5.48 / 5.00, R=8, H=4096 5.30 / 4.09; T=34, R=16,
// H=4096 7.40 / 4.87; T=36, R=8: H=8192 5.57 / 5.43, H=4096 5.58 / 4.78,
// H=2048 5.01 / 4.10).  Lighter rows lost at T=36 (R=4, H=5120 4.35 / 4.79;
// R=2, H=8192 4.20 / 4.76), wider ones too (R=4, H=12288: 4.99 / 6.29), and
// past 36 rows the clusters of 8 lost where they still fit (R=8, H=2048,
// T=64: 4.98 / 5.36); clusters of 4 or 2 lost by 0-11 % from T=40 on.
constexpr int kClusterReduceMidMaxT = 32;
constexpr int kClusterReduceWideMaxT = 36;
constexpr int kClusterReduceWideMinR = 8;
constexpr int kClusterReduceWideMaxChunks = 1024;
constexpr int kClusterReduceMidMaxCs = 8;
// Up to kClusterReduceMinTasks8MaxT rows, clusters of 8 take reduce rows down
// to kClusterReduceMinTasks8 tasks a CTA: R=2 rows of 5120 and 7168 (160 and
// 224 tasks) then take 8 CTAs instead of 4 (us per call: H=5120 T=1 2.90 ->
// 2.73, T=4 2.93 -> 2.79, T=12 3.02 -> 2.92; H=7168 T=2 2.95 -> 2.79, T=8
// 3.06 -> 2.89).  Past 12 rows the gain is gone (T=16: H=5120 3.04 -> 2.96,
// H=7168 3.09 -> 3.15; T=32, H=7168: 4.12 -> 4.21), and a cluster of 16
// below 256 tasks was slower from T=4 (R=4, H=5120, T=8: 3.16 against 2.96
// with 8).
constexpr int kClusterReduceMinTasks8 = 128;
constexpr int kClusterReduceMinTasks8MaxT = 12;
// Past kClusterFinMaxT rows the fused finalize entries keep the cluster path
// for narrow rows only: clusters of at most kClusterMidMaxCs CTAs whose
// CTAs, one per SM, hold all T rows at once with at most two tasks a thread.
// Measured on GB300 (us per call, CUDA graph, L2-cold; R=8, k=8; cluster
// path / the main kernel's shard or column split): H=2048 T=16 5.66 / 8.70,
// T=32 6.28 / 9.77 (4 CTAs a row), T=64 9.06 / 11.91 (2); H=4096 T=16 8.40
// / 11.33, T=32 9.27 / 12.32 (4).  Larger clusters lost (H=2048 T=16 with 8:
// 10.18), and so did wider rows (H=8192 T=16 with 8: 19.4 / 14.3).
constexpr int kClusterMidMaxCs = 4;

struct ClusterPlan {
    int cs, tpt, resident;
    size_t smem;
};

// The largest cluster (16, 8, 4 or 2 CTAs) whose CTAs take at most two
// (shard, chunk) tasks per thread (reduce rows: at least 256 tasks a CTA, or
// 128 in a cluster of 8 up to 12 rows) and
// whose clusters the device holds at once for the T rows (on request, any
// cluster that is resident at all); past kClusterFinMaxT finalize rows, a
// cluster of at most kClusterMidMaxCs CTAs with T * cs CTAs on distinct SMs;
// past kClusterReduceMaxT reduce rows, one of at most kClusterReduceMidMaxCs
// (past kClusterReduceMidMaxT rows, exactly that many, up to
// kClusterReduceWideMaxT rows, for rows of at least kClusterReduceWideMinR
// shards and at most kClusterReduceWideMaxChunks chunks).
bool plan_cluster_fin(int mode, const Args &a, const DeviceInfo *d, ClusterPlan *p)
{
    const bool fin = (mode & F_FIN) != 0;
    if (mode != kModeFinReduceNorm && mode != kModeFinReduceResNorm && mode != kModeReduceNorm &&
        mode != kModeReduceResNorm)
        return false;
    const int pref = g_tune_split.load();
    if (pref != 0 && pref != 3) return false;
    const bool mid = fin && pref == 0 && a.T > kClusterFinMaxT;
    const bool mid_reduce = !fin && pref == 0 && a.T > kClusterReduceMaxT;
    if (mid_reduce && a.T > kClusterReduceMidMaxT &&
        (a.T > kClusterReduceWideMaxT || a.R < kClusterReduceWideMinR ||
         a.H / 8 > kClusterReduceWideMaxChunks))
        return false;
    if (mid && (long long)a.T * 2 > d->sms) return false;
    const int want_cs = g_tune_cluster.load();
    const int nch = a.H / 8;
    for (int cs = mid ? kClusterMidMaxCs : kMaxCluster; cs >= 2; cs /= 2) {
        if (want_cs > 0 && cs != want_cs) continue;
        if (mid && (long long)a.T * cs > d->sms) continue;
        if (mid_reduce && cs > kClusterReduceMidMaxCs) continue;
        if (mid_reduce && a.T > kClusterReduceMidMaxT && cs != kClusterReduceMidMaxCs) continue;
        const int slice = (nch + cs - 1) / cs;
        if (nch < cs || slice > kClusterThreads) continue;
        const int tasks = a.R * slice;
        const int tpt = (tasks + kClusterThreads - 1) / kClusterThreads;
        if (tpt > kClusterMaxTpt) continue;
        if (!fin && pref == 0 && tasks < kClusterReduceMinTasks &&
            !(cs == kClusterReduceMidMaxCs && tasks >= kClusterReduceMinTasks8 &&
              a.T <= kClusterReduceMinTasks8MaxT))
            continue;
        const size_t smem = cluster_smem_bytes(a.R, slice);
        if ((long long)smem > (long long)d->smem_optin - 2048) continue;
        cudaError_t e = cudaSuccess;
        const int res = cluster_fin_resident(fin, a.k, (mode & F_POSTNORM) != 0, tpt,
                                             tiny_for(mode, a.eps) != 0, cs, smem, &e);
        if (e != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (res <= 0 || (pref == 0 && res < a.T)) continue;
        *p = ClusterPlan{cs, tpt, res, smem};
        return true;
    }
    return false;
}

bn_status run_cluster_fin(int mode, Args &a, const DeviceInfo *d, const ClusterPlan &cp,
                          void *stream)
{
    a.nchunks = a.H / 8;
    a.err = d->err;
    a.tiny = tiny_for(mode, a.eps);
    ClusterArgs c;
    c.a = a;
    c.tasks = a.R * ((a.nchunks + cp.cs - 1) / cp.cs);
    const cudaError_t e = launch_cluster_fin(c, (mode & F_FIN) != 0, (mode & F_POSTNORM) != 0,
                                             cp.tpt, cp.cs,
                                             g_tune_pdl.load() != 1,
                                             reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bn_cluster_fin_kernel");
    return BN_OK;
}

bn_status run(int mode, Args &a, void *stream)
{
    if (a.T == 0) return BN_OK;
    {
        const DeviceInfo *d = nullptr;
        BN_TRY(device_info(&d));
        ClusterPlan cp;
        if (plan_cluster_fin(mode, a, d, &cp)) return run_cluster_fin(mode, a, d, cp, stream);
    }
    Launch l;
    BN_TRY(plan(mode, &a, &l));
    cudaError_t e = ops_for(mode).launch(a, l, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, ops_for(mode).name);
    return BN_OK;
}

Args base_args(int R, int T, int k, int H, float eps)
{
    Args a;
    std::memset(&a, 0, sizeof a);
    a.R = R;
    a.T = T;
    a.k = k;
    a.H = H;
    a.eps = eps;
    return a;
}

void apply_debug(Args &a, const bn_debug *dbg)
{
    if (!dbg) return;
    a.sum_out = dbg->sum;
    a.ss_out = dbg->ss;
    a.z_out = dbg->z;
}

bn_status check_debug(const bn_debug *dbg, bool fin)
{
    if (!dbg) return BN_OK;
    BN_TRY(check_ptr16(dbg->sum, "dbg->sum", false));
    BN_TRY(check_ptr16(dbg->ss, "dbg->ss", false));  // 8-byte pairs; 16 keeps one rule
    if (fin) BN_TRY(check_ptr16(dbg->z, "dbg->z", false));
    return BN_OK;
}

void debug_ranges(const bn_debug *dbg, int R, int T, int H, bool fin, Range *w, int *nw)
{
    if (!dbg) return;
    const size_t th = (size_t)T * H;
    if (dbg->sum) w[(*nw)++] = Range{dbg->sum, th * 4, "dbg->sum"};
    if (dbg->ss) w[(*nw)++] = Range{dbg->ss, (size_t)T * 8, "dbg->ss"};
    if (fin && dbg->z) w[(*nw)++] = Range{dbg->z, (size_t)R * th * 2, "dbg->z"};
}

// ---- shared validation of the two source kinds ------------------------------------

bn_status check_reduce_sources(const uint16_t *partials, int R, int T, int H, Range *reads, int *nr)
{
    BN_TRY(check_ptr16(partials, "partials"));
    reads[(*nr)++] = Range{partials, (size_t)R * T * H * 2, "partials"};
    return BN_OK;
}

bn_status check_fin_sources(const uint16_t *expert_out, const int32_t *perm, const float *w,
                            const uint16_t *shared, int R, int T, int k, int H, Range *reads, int *nr)
{
    BN_TRY(check_ptr16(expert_out, "expert_out"));
    BN_TRY(check_ptr4(perm, "perm"));
    BN_TRY(check_ptr4(w, "w"));
    BN_TRY(check_ptr16(shared, "shared", false));
    const size_t rtk = (size_t)R * T * k;
    reads[(*nr)++] = Range{expert_out, rtk * H * 2, "expert_out"};
    reads[(*nr)++] = Range{perm, rtk * 4, "perm"};
    reads[(*nr)++] = Range{w, rtk * 4, "w"};
    if (shared) reads[(*nr)++] = Range{shared, (size_t)R * T * H * 2, "shared"};
    return BN_OK;
}

bn_status check_epilogue(uint16_t *residual, const float *gp, const float *gq, uint16_t *out,
                         float eps, int T, int H, Range *reads, int *nr, Range *writes, int *nw)
{
    BN_TRY(check_ptr16(residual, "residual"));
    BN_TRY(check_ptr16(gp, "gamma_post"));
    BN_TRY(check_ptr16(gq, "gamma_pre"));
    BN_TRY(check_ptr16(out, "out"));
    BN_TRY(check_eps(eps));
    const size_t th = (size_t)T * H;
    reads[(*nr)++] = Range{gp, (size_t)H * 4, "gamma_post"};
    if (gq != gp) reads[(*nr)++] = Range{gq, (size_t)H * 4, "gamma_pre"};
    writes[(*nw)++] = Range{residual, th * 2, "residual"};
    writes[(*nw)++] = Range{out, th * 2, "out"};
    return BN_OK;
}

// ---- the finalize with a workspace: token rows spread over many CTAs --------------

// Token rows up to which the many-CTA finalize serves.  Measured on GB300
// (us per call in a CUDA graph, L2-cold; one CTA or cluster per row / many
// CTAs per row): C4 (R=8, H=8192, k=10) T=1 10.1 / 7.78, T=4 10.5 / 9.0, T=8
// 11.1 / 10.0, T=16 14.4 / 14.7, T=64 24.7 / 39.0 (earlier versions); C3
// (R=8, H=6144, k=8) T=1 9.1 / 7.13, T=4 9.2 / 7.2, T=8 9.9 / 8.5, T=16 12.2
// / 12.1.  From T=16 on the rows themselves fill the SMs.
constexpr int kWideMaxT = 8;

bool wide_serves(int R, int T, int k, int H)
{
    return R >= 1 && R <= kMaxR && k >= 1 && k <= kMaxK && T >= 1 && T <= kWideMaxT && H > 0 &&
           H % 8 == 0 && H / 8 <= kWideThreads * kWideMaxCpt;
}

bn_status run_wide(Args &a, bool postnorm, void *workspace, void *stream)
{
    const DeviceInfo *d = nullptr;
    BN_TRY(device_info(&d));
    a.nchunks = a.H / 8;
    a.err = d->err;
    a.tiny = tiny_for(postnorm ? kModeFinReduceNorm : kModeFinReduceResNorm, a.eps);
    WideArgs w;
    w.a = a;
    w.count = static_cast<unsigned *>(workspace);
    w.zws = reinterpret_cast<uint16_t *>(static_cast<char *>(workspace) + wide_counter_bytes(a.T));
    // The fewest finalize tasks per CTA (a quarter, half or all of its
    // threads) with which all CTAs still fit in one wave: each SM then pulls
    // fewer gathered chunks at once.
    const int tasks_total = a.R * a.nchunks;
    w.tasks = kWideThreads;
    for (int tasks = kWideThreads / 4; tasks < kWideThreads; tasks *= 2) {
        const long long ctas = (long long)a.T * ((tasks_total + tasks - 1) / tasks);
        if (d->sms > 0 && ctas <= d->sms) {
            w.tasks = tasks;
            break;
        }
    }
    w.parts = (tasks_total + w.tasks - 1) / w.tasks;
    const int cpt = a.nchunks <= kWideThreads ? 1 : 2;
    const cudaError_t e = launch_wide(w, postnorm, cpt, g_tune_pdl.load() != 1,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bn_wide_kernel");
    return BN_OK;
}

// The two finalize entry points that take a workspace: the validation of the
// plain ones, plus the workspace (16-byte aligned, overlapping no other
// buffer) when it is large enough to be used.
bn_status fin_ws(bool postnorm, const uint16_t *expert_out, const int32_t *perm, const float *w,
                 const uint16_t *shared, int R, int T, int k, int H, uint16_t *residual,
                 const float *gamma_post, const float *gamma_pre, float eps, uint16_t *out,
                 const bn_debug *dbg, void *workspace, size_t workspace_bytes, void *stream)
{
    BN_TRY(check_shape(R, T, k, H, true));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_fin_sources(expert_out, perm, w, shared, R, T, k, H, reads, &nr));
    BN_TRY(check_epilogue(residual, gamma_post, gamma_pre, out, eps, T, H, reads, &nr, writes, &nw));
    BN_TRY(check_debug(dbg, true));
    debug_ranges(dbg, R, T, H, true, writes, &nw);
    const size_t need = wide_serves(R, T, k, H) ? wide_workspace_bytes(R, T, H) : 0;
    const bool wide = need > 0 && workspace != nullptr && workspace_bytes >= need;
    if (wide) {
        BN_TRY(check_ptr16(workspace, "workspace"));
        writes[nw++] = Range{workspace, need, "workspace"};
    }
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, k, H, true));
    Args a = base_args(R, T, k, H, eps);
    a.src = expert_out;
    a.perm = perm;
    a.w = w;
    a.shared = shared;
    a.residual = residual;
    a.gamma_post = gamma_post;
    a.gamma_pre = gamma_pre;
    a.out = out;
    apply_debug(a, dbg);
    if (wide) return run_wide(a, postnorm, workspace, stream);
    return run(postnorm ? kModeFinReduceNorm : kModeFinReduceResNorm, a, stream);
}

}  // namespace
}  // namespace bn

using namespace bn;

// ================================ C ABI ===========================================

extern "C" {

bn_status bn_reduce_norm(const uint16_t *partials, int R, int T, int H, uint16_t *residual,
                         const float *gamma_post, const float *gamma_pre, float eps, uint16_t *out,
                         const bn_debug *dbg, void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, 1, H, false));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_reduce_sources(partials, R, T, H, reads, &nr));
    BN_TRY(check_epilogue(residual, gamma_post, gamma_pre, out, eps, T, H, reads, &nr, writes, &nw));
    BN_TRY(check_debug(dbg, false));
    debug_ranges(dbg, R, T, H, false, writes, &nw);
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, 1, H, false));
    Args a = base_args(R, T, 0, H, eps);
    a.src = partials;
    a.residual = residual;
    a.gamma_post = gamma_post;
    a.gamma_pre = gamma_pre;
    a.out = out;
    apply_debug(a, dbg);
    return run(kModeReduceNorm, a, stream);
}

bn_status bn_finalize_reduce_norm(const uint16_t *expert_out, const int32_t *perm, const float *w,
                                  const uint16_t *shared, int R, int T, int k, int H,
                                  uint16_t *residual, const float *gamma_post,
                                  const float *gamma_pre, float eps, uint16_t *out,
                                  const bn_debug *dbg, void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, k, H, true));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_fin_sources(expert_out, perm, w, shared, R, T, k, H, reads, &nr));
    BN_TRY(check_epilogue(residual, gamma_post, gamma_pre, out, eps, T, H, reads, &nr, writes, &nw));
    BN_TRY(check_debug(dbg, true));
    debug_ranges(dbg, R, T, H, true, writes, &nw);
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, k, H, true));
    Args a = base_args(R, T, k, H, eps);
    a.src = expert_out;
    a.perm = perm;
    a.w = w;
    a.shared = shared;
    a.residual = residual;
    a.gamma_post = gamma_post;
    a.gamma_pre = gamma_pre;
    a.out = out;
    apply_debug(a, dbg);
    return run(kModeFinReduceNorm, a, stream);
}

bn_status bn_reduce_residual_norm(const uint16_t *partials, int R, int T, int H, uint16_t *residual,
                                  const float *gamma, float eps, uint16_t *out, const bn_debug *dbg,
                                  void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, 1, H, false));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_reduce_sources(partials, R, T, H, reads, &nr));
    BN_TRY(check_epilogue(residual, gamma, gamma, out, eps, T, H, reads, &nr, writes, &nw));
    BN_TRY(check_debug(dbg, false));
    debug_ranges(dbg, R, T, H, false, writes, &nw);
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, 1, H, false));
    Args a = base_args(R, T, 0, H, eps);
    a.src = partials;
    a.residual = residual;
    a.gamma_post = gamma;
    a.gamma_pre = gamma;
    a.out = out;
    apply_debug(a, dbg);
    return run(kModeReduceResNorm, a, stream);
}

bn_status bn_finalize_reduce_residual_norm(const uint16_t *expert_out, const int32_t *perm,
                                           const float *w, const uint16_t *shared, int R, int T,
                                           int k, int H, uint16_t *residual, const float *gamma,
                                           float eps, uint16_t *out, const bn_debug *dbg,
                                           void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, k, H, true));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_fin_sources(expert_out, perm, w, shared, R, T, k, H, reads, &nr));
    BN_TRY(check_epilogue(residual, gamma, gamma, out, eps, T, H, reads, &nr, writes, &nw));
    BN_TRY(check_debug(dbg, true));
    debug_ranges(dbg, R, T, H, true, writes, &nw);
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, k, H, true));
    Args a = base_args(R, T, k, H, eps);
    a.src = expert_out;
    a.perm = perm;
    a.w = w;
    a.shared = shared;
    a.residual = residual;
    a.gamma_post = gamma;
    a.gamma_pre = gamma;
    a.out = out;
    apply_debug(a, dbg);
    return run(kModeFinReduceResNorm, a, stream);
}

size_t bn_finalize_workspace_bytes(int R, int T, int k, int H)
{
    return wide_serves(R, T, k, H) ? wide_workspace_bytes(R, T, H) : 0;
}

bn_status bn_finalize_reduce_norm_ws(const uint16_t *expert_out, const int32_t *perm,
                                     const float *w, const uint16_t *shared, int R, int T, int k,
                                     int H, uint16_t *residual, const float *gamma_post,
                                     const float *gamma_pre, float eps, uint16_t *out,
                                     const bn_debug *dbg, void *workspace, size_t workspace_bytes,
                                     void *stream)
{
    g_msg[0] = '\0';
    return fin_ws(true, expert_out, perm, w, shared, R, T, k, H, residual, gamma_post, gamma_pre,
                  eps, out, dbg, workspace, workspace_bytes, stream);
}

bn_status bn_finalize_reduce_residual_norm_ws(const uint16_t *expert_out, const int32_t *perm,
                                              const float *w, const uint16_t *shared, int R, int T,
                                              int k, int H, uint16_t *residual, const float *gamma,
                                              float eps, uint16_t *out, const bn_debug *dbg,
                                              void *workspace, size_t workspace_bytes,
                                              void *stream)
{
    g_msg[0] = '\0';
    return fin_ws(false, expert_out, perm, w, shared, R, T, k, H, residual, gamma, gamma, eps, out,
                  dbg, workspace, workspace_bytes, stream);
}

// The many-CTA finalize for callers that cannot allocate: its workspace is the
// library's own static scratch (bn_noalloc.cu).  The checks are those of the
// workspace entry, then the scratch limit; the counters are cleared on the
// stream just before the kernel.
bn_status bn_finalize_reduce_norm_noalloc(const uint16_t *expert_out, const int32_t *perm,
                                          const float *w, const uint16_t *shared, int R, int T,
                                          int k, int H, uint16_t *residual,
                                          const float *gamma_post, const float *gamma_pre,
                                          float eps, uint16_t *out, const bn_debug *dbg,
                                          void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, k, H, true));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_fin_sources(expert_out, perm, w, shared, R, T, k, H, reads, &nr));
    BN_TRY(check_epilogue(residual, gamma_post, gamma_pre, out, eps, T, H, reads, &nr, writes, &nw));
    BN_TRY(check_debug(dbg, true));
    debug_ranges(dbg, R, T, H, true, writes, &nw);
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, k, H, true));
    if (!wide_serves(R, T, k, H))
        return fail(BN_ERR_UNSUPPORTED,
                    "bn_finalize_reduce_norm_noalloc serves 1 <= T <= %d and H <= %d (got T=%d, "
                    "H=%d); bn_finalize_reduce_norm needs no scratch for this shape",
                    kWideMaxT, kWideThreads * kWideMaxCpt * 8, T, H);
    const size_t need = wide_workspace_bytes(R, T, H);
    if (need > kNoAllocScratchBytes)
        return fail(BN_ERR_UNSUPPORTED,
                    "R=%d T=%d H=%d needs %zu bytes of scratch, above the library's static "
                    "maximum of %zu bytes",
                    R, T, H, need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "looking up the static scratch");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the row counters must start at zero (the z rows are written before they are read)
    e = cudaMemsetAsync(scratch, 0, wide_counter_bytes(T), st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch counters");
    Args a = base_args(R, T, k, H, eps);
    a.src = expert_out;
    a.perm = perm;
    a.w = w;
    a.shared = shared;
    a.residual = residual;
    a.gamma_post = gamma_post;
    a.gamma_pre = gamma_pre;
    a.out = out;
    apply_debug(a, dbg);
    return run_wide(a, true, scratch, stream);
}

bn_status bn_reduce_only(const uint16_t *partials, int R, int T, int H, float *sum_out, void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, 1, H, false));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[4], writes[2];
    int nr = 0, nw = 0;
    BN_TRY(check_reduce_sources(partials, R, T, H, reads, &nr));
    BN_TRY(check_ptr16(sum_out, "sum_out"));
    writes[nw++] = Range{sum_out, (size_t)T * H * 4, "sum_out"};
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, 1, H, false, true));
    Args a = base_args(R, T, 0, H, 0.f);
    a.src = partials;
    a.sum_out = sum_out;
    return run(kModeReduceOnly, a, stream);
}

bn_status bn_finalize_reduce_only(const uint16_t *expert_out, const int32_t *perm, const float *w,
                                  const uint16_t *shared, int R, int T, int k, int H, float *sum_out,
                                  void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, k, H, true));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[2];
    int nr = 0, nw = 0;
    BN_TRY(check_fin_sources(expert_out, perm, w, shared, R, T, k, H, reads, &nr));
    BN_TRY(check_ptr16(sum_out, "sum_out"));
    writes[nw++] = Range{sum_out, (size_t)T * H * 4, "sum_out"};
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, k, H, true, true));
    Args a = base_args(R, T, k, H, 0.f);
    a.src = expert_out;
    a.perm = perm;
    a.w = w;
    a.shared = shared;
    a.sum_out = sum_out;
    return run(kModeFinReduceOnly, a, stream);
}

bn_status bn_norm_only(const float *sum, int T, int H, uint16_t *residual, const float *gamma_post,
                       const float *gamma_pre, float eps, uint16_t *out, const bn_debug *dbg,
                       void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(1, T, 1, H, false));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_ptr16(sum, "sum"));
    reads[nr++] = Range{sum, (size_t)T * H * 4, "sum"};
    BN_TRY(check_epilogue(residual, gamma_post, gamma_pre, out, eps, T, H, reads, &nr, writes, &nw));
    if (dbg && dbg->ss) {
        BN_TRY(check_ptr16(dbg->ss, "dbg->ss"));
        writes[nw++] = Range{dbg->ss, (size_t)T * 8, "dbg->ss"};
    }
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(1, T, 1, H, false, true));
    Args a = base_args(1, T, 0, H, eps);
    a.sum_in = sum;
    a.residual = residual;
    a.gamma_post = gamma_post;
    a.gamma_pre = gamma_pre;
    a.out = out;
    if (dbg) a.ss_out = dbg->ss;
    return run(kModeNormOnly, a, stream);
}

bn_status bn_residual_norm_only(const float *sum, int T, int H, uint16_t *residual,
                                const float *gamma, float eps, uint16_t *out, const bn_debug *dbg,
                                void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(1, T, 1, H, false));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[8];
    int nr = 0, nw = 0;
    BN_TRY(check_ptr16(sum, "sum"));
    reads[nr++] = Range{sum, (size_t)T * H * 4, "sum"};
    BN_TRY(check_epilogue(residual, gamma, gamma, out, eps, T, H, reads, &nr, writes, &nw));
    if (dbg && dbg->ss) {
        BN_TRY(check_ptr16(dbg->ss, "dbg->ss"));
        writes[nw++] = Range{dbg->ss, (size_t)T * 8, "dbg->ss"};
    }
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(1, T, 1, H, false, true));
    Args a = base_args(1, T, 0, H, eps);
    a.sum_in = sum;
    a.residual = residual;
    a.gamma_post = gamma;
    a.gamma_pre = gamma;
    a.out = out;
    if (dbg) a.ss_out = dbg->ss;
    return run(kModeResNormOnly, a, stream);
}

bn_status bn_finalize_only(const uint16_t *expert_out, const int32_t *perm, const float *w,
                           const uint16_t *shared, int R, int T, int k, int H, uint16_t *z_out,
                           void *stream)
{
    g_msg[0] = '\0';
    BN_TRY(check_shape(R, T, k, H, true));
    if (T == 0) return BN_OK;  // nothing is read or written; pointers are not examined
    Range reads[8], writes[2];
    int nr = 0, nw = 0;
    BN_TRY(check_fin_sources(expert_out, perm, w, shared, R, T, k, H, reads, &nr));
    BN_TRY(check_ptr16(z_out, "z_out"));
    writes[nw++] = Range{z_out, (size_t)R * T * H * 2, "z_out"};
    BN_TRY(check_overlaps(writes, nw, reads, nr));
    BN_TRY(check_served(R, T, k, H, true, true));
    Args a = base_args(R, T, k, H, 0.f);
    a.src = expert_out;
    a.perm = perm;
    a.w = w;
    a.shared = shared;
    a.z_out = z_out;
    return run(kModeFinOnly, a, stream);
}

int bn_supports(int R, int T, int k, int H)
{
    const bool fin = k > 0;
    if (check_shape(R, T, fin ? k : 1, H, fin) != BN_OK) return 0;
    if (check_served(R, T, fin ? k : 1, H, fin) != BN_OK) return 0;
    g_msg[0] = '\0';
    return 1;
}

int bn_supports_op(bn_op op, int R, int T, int k, int H)
{
    if ((int)op < 0 || (int)op >= kNumOps) return 0;
    const int mode = kModeOfOp[(int)op];
    const bool fin = (mode & F_FIN) != 0;
    if (mode & F_SUM_IN) R = 1;  // the epilogue pieces read one FP32 row
    if (check_shape(R, T, fin ? k : 1, H, fin) != BN_OK) return 0;
    if (check_served(R, T, fin ? k : 1, H, fin, is_piece(mode)) != BN_OK) return 0;
    g_msg[0] = '\0';
    return 1;
}

bn_status bn_check_device_error(void *stream, unsigned *bits)
{
    g_msg[0] = '\0';
    if (bits) *bits = 0;
    const DeviceInfo *d = nullptr;
    BN_TRY(device_info(&d));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned v = 0;
    e = cudaMemcpy(&v, d->err, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (v != 0) {
        const unsigned zero = 0;
        e = cudaMemcpy(d->err, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    }
    if (bits) *bits = v;
    if (v != 0)
        return fail(BN_ERR_DEVICE, "device error bits 0x%x%s%s", v,
                    (v & BN_DEVERR_PERM_RANGE) ? " (perm index out of range)" : "",
                    (v & BN_DEVERR_TIMEOUT) ? " (pipeline wait timed out)" : "");
    return BN_OK;
}

const char *bn_last_error(void) { return g_msg; }

const char *bn_status_string(bn_status status)
{
    switch (status) {
    case BN_OK: return "BN_OK";
    case BN_ERR_INVALID: return "BN_ERR_INVALID";
    case BN_ERR_UNSUPPORTED: return "BN_ERR_UNSUPPORTED";
    case BN_ERR_CUDA: return "BN_ERR_CUDA";
    case BN_ERR_DEVICE: return "BN_ERR_DEVICE";
    }
    return "unknown status";
}

int bn_version(void) { return kVersion; }

void bn_shutdown(void) {}

bn_status bn_set_tuning(const bn_tuning *t)
{
    g_msg[0] = '\0';
    bn_tuning z;
    std::memset(&z, 0, sizeof z);
    if (!t) t = &z;
    const int cs = t->cluster_size;
    if (cs < 0 || cs > kMaxCluster)
        return fail(BN_ERR_INVALID, "cluster_size must be in [0, %d]", kMaxCluster);
    if (t->stages < 0 || t->stages > kMaxStages || t->stages == 1)
        return fail(BN_ERR_INVALID, "stages must be 0 or in [2, %d]", kMaxStages);
    if (t->threads < 0 || t->threads > kMaxConsumers || t->threads % 32 != 0)
        return fail(BN_ERR_INVALID, "threads must be 0 or a multiple of 32 up to %d", kMaxConsumers);
    if (t->ctas_per_sm < 0 || t->ctas_per_sm > 8)
        return fail(BN_ERR_INVALID, "ctas_per_sm must be in [0, 8]");
    if (t->wait_mode < 0 || t->wait_mode > 2)
        return fail(BN_ERR_INVALID, "wait_mode must be 0, 1 or 2");
    if (t->group < 0 || t->group > 64)
        return fail(BN_ERR_INVALID, "group must be in [0, 64]");
    if (t->split < 0 || t->split > 3)
        return fail(BN_ERR_INVALID, "split must be 0, 1, 2 or 3");
    if (t->dependent_launch < 0 || t->dependent_launch > 2)
        return fail(BN_ERR_INVALID, "dependent_launch must be 0, 1 or 2");
    if (t->wait_limit_polls < 0)
        return fail(BN_ERR_INVALID, "wait_limit_polls must not be negative");
    if (t->tiny_pass < 0 || t->tiny_pass > 2)
        return fail(BN_ERR_INVALID, "tiny_pass must be 0, 1 or 2");
    g_tune_cluster.store(cs);
    g_tune_stages.store(t->stages);
    g_tune_threads.store(t->threads);
    g_tune_ctas.store(t->ctas_per_sm);
    g_tune_wait.store(t->wait_mode);
    g_tune_group.store(t->group);
    g_tune_split.store(t->split);
    g_tune_pdl.store(t->dependent_launch);
    g_tune_polls.store(t->wait_limit_polls);
    g_tune_tiny.store(t->tiny_pass);
    return BN_OK;
}

bn_status bn_query_launch(bn_op op, int R, int T, int k, int H, int has_shared,
                          bn_launch_info *info)
{
    g_msg[0] = '\0';
    BN_REQUIRE(info != nullptr, "info is NULL");
    std::memset(info, 0, sizeof *info);
    BN_REQUIRE((int)op >= 0 && (int)op < kNumOps, "op=%d is not an operation", (int)op);
    const int mode = kModeOfOp[(int)op];
    const bool fin = (mode & F_FIN) != 0;
    if (mode & F_SUM_IN) R = 1;  // norm_only reads one FP32 row
    BN_TRY(check_shape(R, T, fin ? k : 1, H, fin));
    if (T == 0) return BN_OK;
    BN_TRY(check_served(R, T, fin ? k : 1, H, fin, is_piece(mode)));
    // the shape of a call with eps >= kTinyPassEps (the TINY kernels, which
    // may hold other registers, run only below it)
    Args a = base_args(R, T, fin ? k : 0, H, 1.0f);
    // only the presence of the shared rows matters to the shape; the address
    // is a marker that is never dereferenced (nothing is launched)
    static const uint16_t kSharedMarker[8] = {};
    a.shared = (fin && has_shared) ? kSharedMarker : nullptr;
    {
        const DeviceInfo *d = nullptr;
        BN_TRY(device_info(&d));
        ClusterPlan cp;
        if (plan_cluster_fin(mode, a, d, &cp)) {
            info->split = 2;
            info->cluster_size = cp.cs;
            info->threads = kClusterThreads;
            info->chunks_per_thread = cp.tpt;
            info->grid = T * cp.cs;
            info->resident_ctas = cp.resident * cp.cs;
            info->smem_bytes = (int)cp.smem;
            return BN_OK;
        }
    }
    Launch l;
    BN_TRY(plan(mode, &a, &l));
    int resident = 0;
    BN_TRY(resident_clusters(mode, l, &resident));
    info->split = l.split;
    info->cluster_size = l.cluster;
    info->threads = l.consumers + 32;
    info->chunks_per_thread = l.cpt;
    info->grid = l.grid;
    info->resident_ctas = resident * l.cluster;
    info->stages = a.stages;
    info->stage_bytes = a.stage_bytes;
    info->group = a.group;
    info->smem_bytes = (int)l.smem;
    return BN_OK;
}

}  // extern "C"
