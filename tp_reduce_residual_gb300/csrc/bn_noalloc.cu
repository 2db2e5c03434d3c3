// bn_noalloc.cu -- library-owned scratch for bn_finalize_reduce_norm_noalloc,
// the many-CTA finalize for callers that cannot allocate device memory.
//
// The scratch is a file-scope static device array of kNoAllocScratchBytes.
// The device code of this file is loaded on a device the first time the
// array's address is looked up there; from then on the array stays reserved
// on that device until the process exits.  Host code cannot use the array's
// name as a device address (on the host it names a stand-in object), so the
// address is looked up once per device, with that device current, and handed
// to the kernel as a plain pointer.
#include <mutex>

#include <cuda_runtime.h>

#include "bn_wide.h"

static __device__ __align__(256) unsigned char g_bn_noalloc_scratch[bn::kNoAllocScratchBytes];

namespace bn {
namespace {

constexpr int kMaxScratchDevices = 64;

std::once_flag g_scratch_once[kMaxScratchDevices];
void *g_scratch_ptr[kMaxScratchDevices];
cudaError_t g_scratch_status[kMaxScratchDevices];

}  // namespace

cudaError_t noalloc_scratch(void **ptr)
{
    *ptr = nullptr;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::call_once(g_scratch_once[dev], [dev]() {
        void *p = nullptr;
        const cudaError_t st = cudaGetSymbolAddress(&p, g_bn_noalloc_scratch);
        g_scratch_ptr[dev] = st == cudaSuccess ? p : nullptr;
        g_scratch_status[dev] = st;
    });
    if (g_scratch_status[dev] != cudaSuccess) return g_scratch_status[dev];
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace bn
