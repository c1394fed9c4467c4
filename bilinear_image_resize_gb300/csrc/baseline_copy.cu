// The 1:1 copy baseline: before any resize arithmetic, the Volcanic page
// ("From Prototype to Performance: Optimizing OpenCV Resize on Volcanic
// GPUs", *Kernel evolution -> Baseline: simple 1:1 copy behavior*) runs a
// kernel that only moves the bytes, to see what a launch of that size can
// reach at all.  This is that kernel for sm_103a, in the launch shape of the
// exact-ratio resize kernels (direct.cu): 256-thread CTAs, one 16-byte
// streaming load and store per thread, a programmatic dependent launch, and
// (optionally) the CTA's source span prefetched into L2 before the wait on
// the previous grid.  A resize moving N bytes is compared with this copy
// moving N bytes (N / 2 read, N / 2 written).
#include <cuda_runtime.h>

#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) k_copy_baseline(const uint4 *src, uint4 *dst, long long n16,
                                                                 int prefetch)
{
    grid_launch_dependents();
    const long long i0 = static_cast<long long>(blockIdx.x) * kCopyThreads;
    if (prefetch && threadIdx.x == 0 && i0 < n16)
        l2_prefetch_span(reinterpret_cast<const uint8_t *>(src + i0), (min(i0 + kCopyThreads, n16) - i0) * 16);
    grid_dependency_wait();
    const long long i = i0 + threadIdx.x;
    if (i < n16)
        __stcs(dst + i, __ldcs(src + i));
}

}  // namespace
}  // namespace rz

extern "C" {

int resize_copy_baseline(const void *src, void *dst, size_t bytes, int flags, void *stream)
{
    if ((flags & ~(RZ_COPY_PDL | RZ_COPY_L2_PREFETCH)) != 0) return RZ_ERR_ARG;
    if (bytes == 0) return RZ_OK;
    if (!src || !dst || bytes % 16 != 0) return RZ_ERR_ARG;
    const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
    if ((s | d) % 16 != 0) return RZ_ERR_ARG;
    if (s < d + bytes && d < s + bytes) return RZ_ERR_ARG;   // overlapping ranges
    const long long n16 = static_cast<long long>(bytes / 16);
    const long long blocks = (n16 + rz::kCopyThreads - 1) / rz::kCopyThreads;
    if (blocks > 0x7fffffffLL) return RZ_ERR_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(rz::kCopyThreads, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (flags & RZ_COPY_PDL) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const int prefetch = (flags & RZ_COPY_L2_PREFETCH) ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, rz::k_copy_baseline, static_cast<const uint4 *>(src),
                                             static_cast<uint4 *>(dst), n16, prefetch);
    if (e != cudaSuccess) {
        rz::record_cuda_error(static_cast<int>(e));
        return RZ_ERR_CUDA;
    }
    return RZ_OK;
}

}  // extern "C"
