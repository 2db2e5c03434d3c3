// bn_kernels.cu -- instantiates the kernel template for one mode.
//
// Compiled once per mode with -DBN_MODE_NAME=<name> -DBN_MODE_VALUE=<bits>
// (the build compiles the nine modes as nine objects in parallel), always
// with -fmad=false: the FP32 epilogue must not be contracted into FMAs
// ("Fuse Beam's TP all-reduce with its sandwich norms", "Details", "Build").
#include <cuda_runtime.h>

#include <atomic>

#include "bn_device.cuh"

#if !defined(BN_MODE_NAME) || !defined(BN_MODE_VALUE)
#error "compile with -DBN_MODE_NAME=<name> -DBN_MODE_VALUE=<mode bits>"
#endif

#define BN_CAT2(a, b) a##b
#define BN_CAT(a, b) BN_CAT2(a, b)

namespace bn {
namespace {

constexpr int kMode = BN_MODE_VALUE;
constexpr int kMaxDevices = 64;

template <bool SPLIT, bool FULL, bool TINY>
const void *kernel_by_cpt(int cpt)
{
    switch (cpt) {
    case 1: return reinterpret_cast<const void *>(&dev::bn_kernel<kMode, 1, SPLIT, FULL, TINY>);
    case 2: return reinterpret_cast<const void *>(&dev::bn_kernel<kMode, 2, SPLIT, FULL, TINY>);
    case 4:
        // the planner takes at most kMaxCptFin chunks per thread in the finalize modes
        if constexpr ((kMode & F_FIN) == 0)
            return reinterpret_cast<const void *>(&dev::bn_kernel<kMode, 4, SPLIT, FULL, TINY>);
        return nullptr;
    default: return nullptr;
    }
}

// The second pass over rows of tiny values exists only where there are sums
// of squares (the modes with the norms).
constexpr bool kHasTiny = (kMode & F_RESNORM) != 0;

template <bool SPLIT, bool FULL>
const void *kernel_by_tiny(int cpt, int tiny)
{
    if (tiny) {
        if constexpr (kHasTiny) return kernel_by_cpt<SPLIT, FULL, true>(cpt);
        return nullptr;
    }
    return kernel_by_cpt<SPLIT, FULL, false>(cpt);
}

// The shard split exists for the finalize modes with an epilogue or the
// finalize alone; other modes have no such kernel.
constexpr bool kHasSplit = (kMode & F_FIN) && (kMode & (F_RESNORM | F_Z_OUT));

const void *kernel_for(const Launch &l)
{
    if (l.split) {
        if constexpr (kHasSplit)
            return l.full ? kernel_by_tiny<true, true>(l.cpt, l.tiny) : kernel_by_tiny<true, false>(l.cpt, l.tiny);
        return nullptr;
    }
    return l.full ? kernel_by_tiny<false, true>(l.cpt, l.tiny) : kernel_by_tiny<false, false>(l.cpt, l.tiny);
}

int cpt_index(const Launch &l)
{
    return (l.cpt == 1 ? 0 : l.cpt == 2 ? 1 : 2) + (l.split ? 4 : 0) + (l.full ? 8 : 0) + (l.tiny ? 16 : 0);
}

// Function attributes are per device: set them once per (device, kernel).
std::atomic<unsigned> g_prepared[kMaxDevices];

cudaError_t prepare(const void *fn, const Launch &l)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const unsigned bit = 1u << cpt_index(l);
    if (g_prepared[dev].load(std::memory_order_acquire) & bit) return cudaSuccess;
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
    g_prepared[dev].fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

void fill_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, const Launch &l, int grid,
                 cudaStream_t st)
{
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)(l.consumers + 32), 1, 1);
    cfg.dynamicSmemBytes = l.smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (l.cluster > 1) {
        cudaLaunchAttribute &c = attr[cfg.numAttrs++];
        c.id = cudaLaunchAttributeClusterDimension;
        c.val.clusterDim.x = (unsigned)l.cluster;
        c.val.clusterDim.y = 1;
        c.val.clusterDim.z = 1;
    }
    if (l.pdl && st != nullptr) {
        cudaLaunchAttribute &p = attr[cfg.numAttrs++];
        p.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        p.val.programmaticStreamSerializationAllowed = 1;
    }
    if (cfg.numAttrs == 0) cfg.attrs = nullptr;
}

}  // namespace

cudaError_t BN_CAT(launch_, BN_MODE_NAME)(const Args &a, const Launch &l, cudaStream_t st)
{
    const void *fn = kernel_for(l);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = prepare(fn, l);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, l, l.grid, st);
    void *args[] = {const_cast<Args *>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int BN_CAT(occupancy_, BN_MODE_NAME)(const Launch &l, cudaError_t *err)
{
    const void *fn = kernel_for(l);
    if (!fn) {
        *err = cudaErrorInvalidValue;
        return 0;
    }
    cudaError_t e = prepare(fn, l);
    if (e != cudaSuccess) {
        *err = e;
        return 0;
    }
    if (l.cluster <= 1) {
        int per_sm = 0, dev = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, l.consumers + 32, l.smem);
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        *err = e;
        return e == cudaSuccess ? per_sm * sms : 0;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    Launch one = l;
    one.pdl = 0;
    fill_config(cfg, attr, one, l.cluster, nullptr);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    *err = e;
    return e == cudaSuccess ? n : 0;
}

}  // namespace bn
