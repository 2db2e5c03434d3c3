// bn_cluster.cu -- the finalize at small T with each token row spread over a
// thread-block cluster (see bn_cluster.h for the scheme).
//
// Operation: the one of the other kernels ("Fuse Beam's TP all-reduce with its
// sandwich norms", vLLM pull request 62366, section Claims: the finalize before
// the reduction keeps each shard's local BF16 rounding, then the FP32
// norm-residual-norm; section Details: no FMA contraction, -fmad=false), with
// the same instructions in the same order:
//   z[r]  = bf16(((w0*x0 + w1*x1) + ... + w(k-1)*x(k-1)) + shared[r])
//   s     = ((z[0] + z[1]) + ...) + z[R-1]            (FP32, rank order)
//   y     = (s * r1) * gamma_post,  r1 = 1/sqrt(sum(s^2)/H + eps)   (sandwich only)
//   h     = residual + y  ->  residual = bf16(h)
//   out   = bf16((h * r2) * gamma_pre),  r2 = 1/sqrt(sum(h^2)/H + eps)
// The sums of squares are the same compensated pairs, rounded once.
//
// Waits: only the two cluster exchanges wait, each bounded; every CTA still
// sends its pair, so they complete.  A final cluster barrier keeps every CTA
// alive until all remote stores into it have landed.
#include "bn_cluster.h"

#include <atomic>

#include "bn_device.cuh"

namespace bn {
namespace dev {
namespace {

constexpr int kCWarps = kClusterThreads / 32;

// Named barrier among the first nthreads threads (the slice's epilogue warps).
__device__ __forceinline__ void epilogue_sync(int nthreads)
{
    asm volatile("bar.sync 2, %0;" ::"r"(nthreads) : "memory");
}

// Row-wide sum of squares: the epilogue warps' compensated pairs, combined by
// a tree over the warps' pairs (lane w holding warp w's), then the CTAs'
// pairs exchanged across the cluster and combined by the same kind of tree
// (lane d holding CTA d's).  Every epilogue thread of every CTA gets the same
// value.  The trees replace loops over the pairs that the compiler unrolled
// into about a fifth of the kernels' code.
__device__ __forceinline__ float row_sum_squares_cl(f2 S2, f2 E2, float2 *red, float2 *xslot,
                                                    uint32_t xbar, uint32_t cs, uint32_t q,
                                                    int nwe, int warp, int lane, int tid,
                                                    const Ctl &ctl, bool &live)
{
    float S, E;
    fold2(S2, E2, S, E);
    warp_tree(S, E);
    if (lane == 0) red[warp] = make_float2(S, E);
    epilogue_sync(nwe * 32);
    small_tree(red, nwe, lane, S, E);
    if (cs > 1) {
        // thread d sends this CTA's pair into slot q of CTA d, counted in bytes
        // on CTA d's barrier; each CTA's own arrive expects cs * 8 bytes
        if (tid == 0) mbar_arrive_expect_tx(xbar, 8u * cs);
        if (tid < (int)cs) {
            const uint32_t d = (uint32_t)tid;
            st_async_f2(mapa(smem_addr(xslot + q), d), S, E, mapa(xbar, d));
        }
        if (!wait_phase<true, kDsmem>(xbar, 0u, ctl)) live = false;
        small_tree(xslot, (int)cs, lane, S, E);
    }
    return pair_value(S, E);
}

__device__ __forceinline__ void gamma8_regs(const float *g, f2 *out)
{
    const float4 x = __ldg(reinterpret_cast<const float4 *>(g));
    const float4 y = __ldg(reinterpret_cast<const float4 *>(g) + 1);
    out[0] = f2_make(x.x, x.y);
    out[1] = f2_make(x.z, x.w);
    out[2] = f2_make(y.x, y.y);
    out[3] = f2_make(y.z, y.w);
}

// Grid: T clusters of cs CTAs; cluster t works on token row t, CTA q of it on
// the chunks [c0, c0 + slice) of that row.  Thread i takes the tasks
// i + j * kClusterThreads (j < TPT) below R * slice: shard task / slice, chunk
// task % slice.  A task finalizes that chunk of that shard (FIN), or copies the
// shard's partial chunk (the reduce entry points).  The first `slice` threads
// then run the epilogue, one chunk each.
// KU: the expert slots a finalize task unrolls (k <= KU), 0 for the reduce
// entry points (cluster_slots).
template <int KU, bool POSTNORM, int TPT, bool TINY>
__global__ void __launch_bounds__(kClusterThreads, 1) bn_cluster_fin_kernel(const ClusterArgs ca)
{
    constexpr bool FIN = KU > 0;
    const Args &a = ca.a;
    extern __shared__ __align__(16) uint4 zsm[];  // [R][slice] BF16 finalize results
    // four row reductions at most: ss1, its rescale, ss2, its rescale; each
    // has its own warp slots, exchange slots and barrier (one phase each)
    __shared__ float2 red[4][kCWarps];
    __shared__ float2 xslot[4][kMaxCluster];
    __shared__ __align__(8) unsigned long long xbar[4];
    __shared__ int s_abort;
    const int tid = (int)threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t cs = cluster_nctarank();
    const uint32_t q = cluster_ctarank();
    const int t = (int)cluster_id_x();
    const int nch = a.nchunks;
    const int c0 = (int)(((long long)q * nch) / (long long)cs);
    const int slice = (int)(((long long)(q + 1) * nch) / (long long)cs) - c0;
    const int nwe = (slice + 31) >> 5;  // epilogue warps
    const size_t H = (size_t)a.H;
    const uint32_t xb[4] = {smem_addr(&xbar[0]), smem_addr(&xbar[1]), smem_addr(&xbar[2]),
                            smem_addr(&xbar[3])};
    // A kernel unrolled for fewer slots than k (the host never launches one)
    // returns at once, before any barrier, with the error bit set.
    if (FIN && a.k > KU) {
        griddep_wait();
        if (tid == 0) atomicOr(a.err, kErrTimeout);
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(xb[i], 1u);
        s_abort = 0;
    }
    fence_mbarrier_init();
    __syncthreads();
    if (cs > 1) cluster_sync_all();
    // Only shared memory so far: under a programmatic launch this overlaps the
    // previous kernel in the stream.  No global access comes before the wait.
    griddep_wait();
    const Ctl ctl{&s_abort, a.err, false, kMaxSpins};
    bool live = true;

    // the epilogue's operands first: their latency hides under the gathers
    const bool epi = tid < slice;
    const int gc = c0 + tid;  // this thread's epilogue chunk
    uint4 res = make_uint4(0u, 0u, 0u, 0u);
    f2 gpost[4] = {0ull, 0ull, 0ull, 0ull}, gpre[4] = {0ull, 0ull, 0ull, 0ull};
    if (epi) {
        res = __ldcg(reinterpret_cast<const uint4 *>(a.residual + (size_t)t * H) + gc);
        if constexpr (POSTNORM) gamma8_regs(a.gamma_post + (size_t)gc * 8, gpost);
        gamma8_regs(a.gamma_pre + (size_t)gc * 8, gpre);
    }

    // ---- the slice's finalize: one (shard, chunk) task at a time per thread ----
    const long long rows = (long long)a.T * a.k;  // expert rows per shard
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        const int task = tid + i * kClusterThreads;
        if (!FIN && task < a.R * slice) {
            const int r = task / slice;
            const int lc = task - r * slice;
            zsm[r * slice + lc] =
                __ldg(reinterpret_cast<const uint4 *>(a.src + ((size_t)r * a.T + t) * H) + c0 + lc);
        } else if (FIN && task < a.R * slice) {
            const int r = task / slice;
            const int lc = task - r * slice;
            const size_t meta = ((size_t)r * a.T + t) * (size_t)a.k;
            uint4 x[KU > 0 ? KU : 1];
            float wj[KU > 0 ? KU : 1];
#pragma unroll
            for (int j = 0; j < KU; ++j) {
                if (j < a.k) {
                    int p = __ldg(a.perm + meta + j);
                    if (p < 0 || (long long)p >= rows) {
                        atomicOr(a.err, kErrPerm);
                        p = 0;
                    }
                    wj[j] = __ldg(a.w + meta + j);
                    x[j] = __ldg(reinterpret_cast<const uint4 *>(
                                     a.src + ((size_t)r * (size_t)rows + (size_t)p) * H) +
                                 c0 + lc);
                }
            }
            uint4 sh = make_uint4(0u, 0u, 0u, 0u);
            if (a.shared != nullptr)
                sh = __ldg(reinterpret_cast<const uint4 *>(a.shared + ((size_t)r * a.T + t) * H) + c0 + lc);
            f2 acc[4];
            {
                f2 v[4];
                widen8(x[0], v);
                const f2 w2 = f2_make(wj[0], wj[0]);
#pragma unroll
                for (int m = 0; m < 4; ++m) acc[m] = mul_sep2(w2, v[m]);
            }
#pragma unroll
            for (int j = 1; j < KU; ++j) {
                if (j < a.k) {
                    f2 v[4];
                    widen8(x[j], v);
                    const f2 w2 = f2_make(wj[j], wj[j]);
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc[m] = add2(acc[m], mul_sep2(w2, v[m]));
                }
            }
            if (a.shared != nullptr) add_bf16x8(acc, sh);
            const uint4 z = round8(acc);
            zsm[r * slice + lc] = z;
            if (a.z_out != nullptr)
                reinterpret_cast<uint4 *>(a.z_out + ((size_t)r * a.T + t) * H)[c0 + lc] = z;
        }
    }
    __syncthreads();

    if (warp < nwe) {
        // ---- rank-ordered sum of the R finalize results of this thread's chunk ----
        f2 s[4] = {0ull, 0ull, 0ull, 0ull};
        if (epi) {
            widen8(zsm[tid], s);
            for (int r = 1; r < a.R; ++r) add_bf16x8(s, zsm[r * slice + tid]);
            if (a.sum_out != nullptr) {
                ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(a.sum_out + (size_t)t * H + (size_t)gc * 8);
                dst[0] = make_ulonglong2(s[0], s[1]);
                dst[1] = make_ulonglong2(s[2], s[3]);
            }
        }
        // ---- norm-residual-norm on the chunk ----
        float ss1 = 0.f;
        if constexpr (POSTNORM) {
            f2 S1 = 0ull, E1 = 0ull;
            if (epi) {
#pragma unroll
                for (int m = 0; m < 4; ++m) acc_square2(S1, E1, s[m]);
            }
            ss1 = row_sum_squares_cl(S1, E1, red[0], xslot[0], xb[0], cs, q, nwe, warp, lane, tid,
                                     ctl, live);
            if (TINY && needs_rescale(ss1)) {  // the same on every thread of the cluster
                const int kx = rescale_exp(ss1);
                const float up = pow2f(kx);
                float Sb = 0.f, Eb = 0.f;
                if (epi) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc_square_scaled(Sb, Eb, s[m], up);
                }
                const float r = row_sum_squares_cl(f2_make(Sb, 0.f), f2_make(Eb, 0.f), red[1], xslot[1],
                                                   xb[1], cs, q, nwe, warp, lane, tid, ctl, live);
                ss1 = mul_sep(mul_sep(r, pow2f(-kx)), pow2f(-kx));
            }
            const float r1 = rms_factor(ss1, a.H, a.eps);
            const f2 r1x2 = f2_make(r1, r1);
#pragma unroll
            for (int m = 0; m < 4; ++m) s[m] = mul_sep2(mul2(s[m], r1x2), gpost[m]);
        }
        f2 S2 = 0ull, E2 = 0ull;
        if (epi) {
            add_bf16x8(s, res);  // h = residual + y
#pragma unroll
            for (int m = 0; m < 4; ++m) acc_square2(S2, E2, s[m]);
            if (live) reinterpret_cast<uint4 *>(a.residual + (size_t)t * H)[gc] = round8(s);
        }
        float ss2 = row_sum_squares_cl(S2, E2, red[2], xslot[2], xb[2], cs, q, nwe, warp, lane,
                                       tid, ctl, live);
        if (TINY && needs_rescale(ss2)) {  // the same on every thread of the cluster
            const int kx = rescale_exp(ss2);
            const float up = pow2f(kx);
            float Sb = 0.f, Eb = 0.f;
            if (epi) {
#pragma unroll
                for (int m = 0; m < 4; ++m) acc_square_scaled(Sb, Eb, s[m], up);
            }
            const float r = row_sum_squares_cl(f2_make(Sb, 0.f), f2_make(Eb, 0.f), red[3], xslot[3],
                                               xb[3], cs, q, nwe, warp, lane, tid, ctl, live);
            ss2 = mul_sep(mul_sep(r, pow2f(-kx)), pow2f(-kx));
        }
        const float r2 = rms_factor(ss2, a.H, a.eps);
        const f2 r2x2 = f2_make(r2, r2);
        if (epi && live) {
            f2 o[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] = mul2(mul2(s[m], r2x2), gpre[m]);
            reinterpret_cast<uint4 *>(a.out + (size_t)t * H)[gc] = round8(o);
        }
        if (a.ss_out != nullptr && q == 0 && tid == 0 && live) {
            a.ss_out[2 * (size_t)t] = ss1;
            a.ss_out[2 * (size_t)t + 1] = ss2;
        }
    }
    griddep_launch_dependents();
    // The only accesses to another CTA's shared memory are remote stores (and
    // their byte counts) into the exchange slots, and every CTA waits for all
    // of those addressed to it before it gets here.  So a CTA leaves without a
    // cluster barrier (measured: 0.2 to 0.3 us less per call at few rows).
    // If one of its exchange waits gave up, stores from the other CTAs may
    // still be on their way: the threads that see it stay for the bounded
    // wait limit before leaving, and the CTA's shared memory lives as long as
    // they do.
    if (cs > 1 && (*(volatile int *)&s_abort & kAbortDsmem)) {
        const long long t0 = clock64();
        while (clock64() - t0 < kWaitLimitCycles) __nanosleep(1000);
    }
}

template <int KU, bool POSTNORM, bool TINY>
const void *cluster_kernel(int tpt)
{
    switch (tpt) {
    case 1: return reinterpret_cast<const void *>(&bn_cluster_fin_kernel<KU, POSTNORM, 1, TINY>);
    case 2: return reinterpret_cast<const void *>(&bn_cluster_fin_kernel<KU, POSTNORM, 2, TINY>);
    default: return nullptr;
    }
}

template <int KU, bool TINY>
const void *cluster_kernel(bool postnorm, int tpt)
{
    return postnorm ? cluster_kernel<KU, true, TINY>(tpt) : cluster_kernel<KU, false, TINY>(tpt);
}

template <bool TINY>
const void *cluster_kernel(int ku, bool postnorm, int tpt)
{
    switch (ku) {
    case 0: return cluster_kernel<0, TINY>(postnorm, tpt);
    case 4: return cluster_kernel<4, TINY>(postnorm, tpt);
    case 8: return cluster_kernel<8, TINY>(postnorm, tpt);
    case 10: return cluster_kernel<10, TINY>(postnorm, tpt);
    case kMaxK: return cluster_kernel<kMaxK, TINY>(postnorm, tpt);
    default: return nullptr;
    }
}

// position of a slot count in the table above
int slots_index(int ku) { return ku == 0 ? 0 : ku == 4 ? 1 : ku == 8 ? 2 : ku == 10 ? 3 : 4; }

// Function attributes are per device: dynamic shared memory above the 48 KB
// default and cluster sizes above 8, set once per kernel and device.
std::atomic<unsigned long long> g_cluster_ready[64];

cudaError_t prepare_cluster(const void *fn, int bit)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_cluster_ready[dev].load(std::memory_order_acquire) & (1ull << bit)) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    g_cluster_ready[dev].fetch_or(1ull << bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

const void *kernel_for(int ku, bool postnorm, int tpt, bool tiny, cudaError_t *e)
{
    const void *fn = tiny ? cluster_kernel<true>(ku, postnorm, tpt) : cluster_kernel<false>(ku, postnorm, tpt);
    if (!fn) {
        *e = cudaErrorInvalidValue;
        return nullptr;
    }
    *e = prepare_cluster(fn, ((slots_index(ku) * 2 + (tiny ? 1 : 0)) * 2 + (postnorm ? 1 : 0)) * 2 +
                                 (tpt == 2 ? 1 : 0));
    return *e == cudaSuccess ? fn : nullptr;
}

void fill(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int grid, int cs, size_t smem,
          bool pdl, cudaStream_t st)
{
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)kClusterThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    cudaLaunchAttribute &c = attr[cfg.numAttrs++];
    c.id = cudaLaunchAttributeClusterDimension;
    c.val.clusterDim.x = (unsigned)cs;
    c.val.clusterDim.y = 1;
    c.val.clusterDim.z = 1;
    if (pdl && st != nullptr) {
        cudaLaunchAttribute &p = attr[cfg.numAttrs++];
        p.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        p.val.programmaticStreamSerializationAllowed = 1;
    }
}

}  // namespace
}  // namespace dev

cudaError_t launch_cluster_fin(const ClusterArgs &c, bool fin, bool postnorm, int tpt, int cs,
                               bool pdl, cudaStream_t st)
{
    if (cs < 1 || cs > kMaxCluster || c.a.T < 1 || c.a.nchunks < cs ||
        c.tasks > kClusterThreads * tpt || (c.a.nchunks + cs - 1) / cs > kClusterThreads ||
        (fin && (c.a.k < 1 || c.a.k > kMaxK)))
        return cudaErrorInvalidValue;
    cudaError_t e;
    const void *fn = dev::kernel_for(cluster_slots(fin, c.a.k), postnorm, tpt, c.a.tiny != 0, &e);
    if (!fn) return e;
    const int slice = (c.a.nchunks + cs - 1) / cs;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    dev::fill(cfg, attr, c.a.T * cs, cs, cluster_smem_bytes(c.a.R, slice), pdl, st);
    void *args[] = {const_cast<ClusterArgs *>(&c)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int cluster_fin_resident(bool fin, int k, bool postnorm, int tpt, bool tiny, int cs, size_t smem,
                         cudaError_t *err)
{
    const void *fn = dev::kernel_for(cluster_slots(fin, k), postnorm, tpt, tiny, err);
    if (!fn) return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    dev::fill(cfg, attr, cs, cs, smem, false, nullptr);
    int n = 0;
    *err = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    return *err == cudaSuccess ? n : 0;
}

}  // namespace bn
