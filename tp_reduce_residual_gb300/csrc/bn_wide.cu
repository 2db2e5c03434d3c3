// bn_wide.cu -- the finalize at small T with each token row spread over many
// CTAs (see bn_wide.h for the scheme).
//
// Operation: the same as the one-CTA-per-row kernels of bn_device.cuh ("Fuse
// Beam's TP all-reduce with its sandwich norms", vLLM pull request 62366,
// section Claims: the finalize before the reduction keeps each shard's local
// BF16 rounding, then the FP32 norm-residual-norm; section Details: no FMA
// contraction, -fmad=false), with the same arithmetic in the same order:
//   z[r]  = bf16(((w0*x0 + w1*x1) + ... + w(k-1)*x(k-1)) + shared[r])
//   s     = ((z[0] + z[1]) + ...) + z[R-1]            (FP32, rank order)
//   y     = (s * r1) * gamma_post,  r1 = 1/sqrt(sum(s^2)/H + eps)   (sandwich only)
//   h     = residual + y  ->  residual = bf16(h)
//   out   = bf16((h * r2) * gamma_pre),  r2 = 1/sqrt(sum(h^2)/H + eps)
// The sums of squares are the same compensated pairs (TwoProduct and TwoSum
// errors carried in a second accumulator), combined in a fixed tree and
// rounded once, as in the main kernel; like them they are the FP32 rounding of
// the exact sum except right at a rounding boundary (they are as accurate as a
// sum carried in twice the precision).
//
// Memory ordering: a CTA barrier, then one device-scope fence by thread 0
// before its atomicInc on the row's counter (the fence is cumulative over the
// stores the barrier ordered before it); the CTA that takes the count to its
// end fences after the count and reads the z rows through L2 (ld.global.cg).  atomicInc wraps the counter back to zero, so a
// workspace whose counters start at zero is left at zero by every call.
#include "bn_wide.h"

#include <atomic>

#include "bn_device.cuh"

namespace bn {
namespace dev {
namespace {

constexpr int kWideWarps = kWideThreads / 32;

// Row-wide sum of squares over the CTA: each warp's tree, then the warps'
// pairs in a fixed order; every thread gets the value.
__device__ __forceinline__ float cta_sum_squares(f2 S2, f2 E2, float2 *red, int warp, int lane)
{
    float S, E;
    fold2(S2, E2, S, E);
    warp_tree(S, E);
    if (lane == 0) red[warp] = make_float2(S, E);
    __syncthreads();
    const float2 v = lane < kWideWarps ? red[lane] : make_float2(0.f, 0.f);
    S = v.x;
    E = v.y;
    warp_tree(S, E);
    S = __shfl_sync(0xffffffffu, S, 0);
    E = __shfl_sync(0xffffffffu, E, 0);
    return pair_value(S, E);
}

// 16 bytes global -> shared without a register round trip (completion: wait_all).
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The eight FP32 gammas of chunk lc (staged in shared memory) as four pairs.
__device__ __forceinline__ void gamma8_smem(const float4 *g, int lc, f2 *out)
{
    const float4 x = g[2 * lc];
    const float4 y = g[2 * lc + 1];
    out[0] = f2_make(x.x, x.y);
    out[1] = f2_make(x.z, x.w);
    out[2] = f2_make(y.x, y.y);
    out[3] = f2_make(y.z, y.w);
}

// Grid: T * parts CTAs; CTA b works on token row b / parts.  Its first
// w.tasks threads take the tasks q = (b % parts) * w.tasks + tid < R * nchunks
// of that row, task q being chunk q % nchunks of shard q / nchunks.
template <bool POSTNORM, int CPT, bool TINY>
__global__ void __launch_bounds__(kWideThreads, 1) bn_wide_kernel(const WideArgs w)
{
    const Args &a = w.a;
    extern __shared__ __align__(16) float4 gsm[];  // epilogue gammas: [post,] pre, 2 per chunk
    __shared__ float2 red[4][kWideWarps];  // ss1, its rescale, ss2, its rescale
    __shared__ int s_last;
    const int tid = (int)threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int t = (int)blockIdx.x / w.parts;
    const int part = (int)blockIdx.x - t * w.parts;
    const size_t H = (size_t)a.H;
    const int nch = a.nchunks;

    // The inputs, the workspace and its counters may come from the previous
    // kernel in the stream: nothing global is touched before this wait.
    griddep_wait();

    // ---- this CTA's share of the row's finalize ----
    const int q = part * w.tasks + tid;
    if (tid < w.tasks && q < a.R * nch) {
        const int r = q / nch;
        const int c = q - r * nch;
        const size_t meta = ((size_t)r * a.T + t) * (size_t)a.k;
        const long long rows = (long long)a.T * a.k;  // expert rows per shard
        // all k gathered chunks are loaded before any is used
        uint4 x[kMaxK];
        float wj[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < a.k) {
                int p = __ldg(a.perm + meta + j);
                if (p < 0 || (long long)p >= rows) {
                    atomicOr(a.err, kErrPerm);
                    p = 0;
                }
                wj[j] = __ldg(a.w + meta + j);
                x[j] = __ldg(reinterpret_cast<const uint4 *>(
                                 a.src + ((size_t)r * (size_t)rows + (size_t)p) * H) +
                             c);
            }
        }
        uint4 sh = make_uint4(0u, 0u, 0u, 0u);
        if (a.shared != nullptr)
            sh = __ldg(reinterpret_cast<const uint4 *>(a.shared + ((size_t)r * a.T + t) * H) + c);
        f2 acc[4];
        {
            f2 v[4];
            widen8(x[0], v);
            const f2 w2 = f2_make(wj[0], wj[0]);
#pragma unroll
            for (int m = 0; m < 4; ++m) acc[m] = mul_sep2(w2, v[m]);
        }
#pragma unroll
        for (int j = 1; j < kMaxK; ++j) {
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
        reinterpret_cast<uint4 *>(w.zws + ((size_t)t * a.R + r) * H)[c] = z;
        if (a.z_out != nullptr) reinterpret_cast<uint4 *>(a.z_out + ((size_t)r * a.T + t) * H)[c] = z;
    }

    // ---- count this CTA done on its row; the last one runs the epilogue ----
    // The barrier orders every thread's z stores before thread 0's fence,
    // which makes them visible device-wide before the count (the fence is
    // cumulative over what the barrier ordered); the counting CTA's fence
    // after the count orders its later loads after the other CTAs' stores.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned old = atomicInc(w.count + t, (unsigned)(w.parts - 1));
        __threadfence();
        s_last = old == (unsigned)(w.parts - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) {
        griddep_launch_dependents();
        return;
    }

    // Each thread stages the gammas of its own chunks in shared memory (it
    // alone reads them back), then loads the residual and the z rows: the
    // gammas' HBM latency is spent under the loads and the first reduction.
    float4 *gpre = gsm + (POSTNORM ? 2 * nch : 0);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int lc = tid + i * kWideThreads;
        if (lc < nch) {
            if constexpr (POSTNORM) {
                cp_async16(gsm + 2 * lc, a.gamma_post + (size_t)lc * 8);
                cp_async16(gsm + 2 * lc + 1, a.gamma_post + (size_t)lc * 8 + 4);
            }
            cp_async16(gpre + 2 * lc, a.gamma_pre + (size_t)lc * 8);
            cp_async16(gpre + 2 * lc + 1, a.gamma_pre + (size_t)lc * 8 + 4);
        }
    }
    cp_async_commit();
    f2 s[CPT][4];
    uint4 res[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
#pragma unroll
        for (int m = 0; m < 4; ++m) s[i][m] = 0ull;
        res[i] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int lc = tid + i * kWideThreads;
        if (lc < nch) res[i] = __ldcg(reinterpret_cast<const uint4 *>(a.residual + (size_t)t * H) + lc);
    }
    // rank-ordered sum of the row's R z rows, eight rows' loads in flight at once
    const uint4 *zrow = reinterpret_cast<const uint4 *>(w.zws + (size_t)t * a.R * H);
    for (int r0 = 0; r0 < a.R; r0 += 8) {
        uint4 zb[8][CPT];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int lc = tid + i * kWideThreads;
                zb[u][i] = make_uint4(0u, 0u, 0u, 0u);
                if (r0 + u < a.R && lc < nch) zb[u][i] = __ldcg(zrow + (size_t)(r0 + u) * nch + lc);
            }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int lc = tid + i * kWideThreads;
                if (r0 + u < a.R && lc < nch) {
                    if (r0 + u == 0)
                        widen8(zb[u][i], s[i]);
                    else
                        add_bf16x8(s[i], zb[u][i]);
                }
            }
    }
    if (a.sum_out != nullptr) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int lc = tid + i * kWideThreads;
            if (lc < nch) {
                ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(a.sum_out + (size_t)t * H + (size_t)lc * 8);
                dst[0] = make_ulonglong2(s[i][0], s[i][1]);
                dst[1] = make_ulonglong2(s[i][2], s[i][3]);
            }
        }
    }

    cp_async_wait_all();

    // ---- norm-residual-norm ----
    float ss1 = 0.f;
    if constexpr (POSTNORM) {
        f2 S1 = 0ull, E1 = 0ull;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int lc = tid + i * kWideThreads;
            if (lc < nch) {
#pragma unroll
                for (int m = 0; m < 4; ++m) acc_square2(S1, E1, s[i][m]);
            }
        }
        ss1 = cta_sum_squares(S1, E1, red[0], warp, lane);
        if (TINY && needs_rescale(ss1)) {  // the same on every thread of the CTA
            const int kx = rescale_exp(ss1);
            const float up = pow2f(kx);
            float Sb = 0.f, Eb = 0.f;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int lc = tid + i * kWideThreads;
                if (lc < nch) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc_square_scaled(Sb, Eb, s[i][m], up);
                }
            }
            const float r = cta_sum_squares(f2_make(Sb, 0.f), f2_make(Eb, 0.f), red[1], warp, lane);
            ss1 = mul_sep(mul_sep(r, pow2f(-kx)), pow2f(-kx));
        }
        const float r1 = rms_factor(ss1, a.H, a.eps);
        const f2 r1x2 = f2_make(r1, r1);
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int lc = tid + i * kWideThreads;
            if (lc < nch) {
                f2 g[4];
                gamma8_smem(gsm, lc, g);
#pragma unroll
                for (int m = 0; m < 4; ++m) s[i][m] = mul_sep2(mul2(s[i][m], r1x2), g[m]);
            }
        }
    }
    // residual add and write-back (s holds y, or the sum itself)
    f2 S2 = 0ull, E2 = 0ull;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int lc = tid + i * kWideThreads;
        if (lc < nch) {
            add_bf16x8(s[i], res[i]);
#pragma unroll
            for (int m = 0; m < 4; ++m) acc_square2(S2, E2, s[i][m]);
            reinterpret_cast<uint4 *>(a.residual + (size_t)t * H)[lc] = round8(s[i]);
        }
    }
    float ss2 = cta_sum_squares(S2, E2, red[2], warp, lane);
    if (TINY && needs_rescale(ss2)) {  // the same on every thread of the CTA
        const int kx = rescale_exp(ss2);
        const float up = pow2f(kx);
        float Sb = 0.f, Eb = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int lc = tid + i * kWideThreads;
            if (lc < nch) {
#pragma unroll
                for (int m = 0; m < 4; ++m) acc_square_scaled(Sb, Eb, s[i][m], up);
            }
        }
        const float r = cta_sum_squares(f2_make(Sb, 0.f), f2_make(Eb, 0.f), red[3], warp, lane);
        ss2 = mul_sep(mul_sep(r, pow2f(-kx)), pow2f(-kx));
    }
    const float r2 = rms_factor(ss2, a.H, a.eps);
    const f2 r2x2 = f2_make(r2, r2);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int lc = tid + i * kWideThreads;
        if (lc < nch) {
            f2 g[4], o[4];
            gamma8_smem(gpre, lc, g);
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] = mul2(mul2(s[i][m], r2x2), g[m]);
            reinterpret_cast<uint4 *>(a.out + (size_t)t * H)[lc] = round8(o);
        }
    }
    if (a.ss_out != nullptr && tid == 0) {
        a.ss_out[2 * (size_t)t] = ss1;
        a.ss_out[2 * (size_t)t + 1] = ss2;
    }
    griddep_launch_dependents();
}

template <bool POSTNORM, bool TINY>
const void *wide_kernel(int cpt)
{
    switch (cpt) {
    case 1: return reinterpret_cast<const void *>(&bn_wide_kernel<POSTNORM, 1, TINY>);
    case 2: return reinterpret_cast<const void *>(&bn_wide_kernel<POSTNORM, 2, TINY>);
    default: return nullptr;
    }
}

// The gammas take up to 64 KB of dynamic shared memory: above the default
// 48 KB the limit is raised once per kernel and device.
std::atomic<unsigned> g_wide_ready[64];

cudaError_t prepare_wide(const void *fn, int bit)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_wide_ready[dev].load(std::memory_order_acquire) & (1u << bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)wide_smem_bytes(true, kWideThreads * kWideMaxCpt * 8));
    if (e != cudaSuccess) return e;
    g_wide_ready[dev].fetch_or(1u << bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

}  // namespace
}  // namespace dev

cudaError_t launch_wide(const WideArgs &w, bool postnorm, int cpt, bool pdl, cudaStream_t st)
{
    const void *fn = w.a.tiny ? (postnorm ? dev::wide_kernel<true, true>(cpt) : dev::wide_kernel<false, true>(cpt))
                              : (postnorm ? dev::wide_kernel<true, false>(cpt) : dev::wide_kernel<false, false>(cpt));
    if (!fn || w.parts < 1 || w.a.T < 1 || w.a.H > kWideThreads * kWideMaxCpt * 8 ||
        w.tasks < 1 || w.tasks > kWideThreads)
        return cudaErrorInvalidValue;
    const cudaError_t e = dev::prepare_wide(fn, (w.a.tiny ? 4 : 0) + (postnorm ? 2 : 0) + (cpt == 2 ? 1 : 0));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)w.a.T * (unsigned)w.parts, 1, 1);
    cfg.blockDim = dim3((unsigned)kWideThreads, 1, 1);
    cfg.dynamicSmemBytes = wide_smem_bytes(postnorm, w.a.H);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    // programmatic dependent launch (created streams and graphs only)
    if (pdl && st != nullptr) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    void *args[] = {const_cast<WideArgs *>(&w)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace bn
