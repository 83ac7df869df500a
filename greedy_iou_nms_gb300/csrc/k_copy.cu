// Staging copy for callers whose input sits in pinned host memory mapped into
// the device's address space (the host pipeline's zero-copy mode): every SM
// takes a share of the bytes once, so the kernels after it read device
// memory.  Reading the input in place instead made each of the sort's CTAs
// fetch all scores across the host link.
#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int CP_THREADS = 256;

// dst[0..bytes) = src[0..bytes); 16-byte loads and stores when both pointers
// and the size allow, bytes otherwise.
__global__ void __launch_bounds__(CP_THREADS)
copy_kernel(unsigned char* __restrict__ dst, const unsigned char* __restrict__ src, size_t bytes, int wide)
{
    pdl_wait();     // an earlier kernel may still read dst
    pdl_release();  // the next kernel may be scheduled (it waits for this grid)
    const size_t t = static_cast<size_t>(blockIdx.x) * CP_THREADS + threadIdx.x;
    const size_t step = static_cast<size_t>(gridDim.x) * CP_THREADS;
    if (wide) {
        uint4* d = reinterpret_cast<uint4*>(dst);
        const uint4* s = reinterpret_cast<const uint4*>(src);
        for (size_t q = t; q < bytes / 16; q += step) d[q] = s[q];
    } else {
        for (size_t q = t; q < bytes; q += step) dst[q] = src[q];
    }
}

void launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t st)
{
    if (bytes == 0) return;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    const bool wide = (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                      bytes % 16 == 0;
    const size_t units = wide ? bytes / 16 : bytes;
    const size_t want = (units + CP_THREADS - 1) / CP_THREADS;
    const unsigned grid = static_cast<unsigned>(want < static_cast<size_t>(4 * sms) ? want : 4 * sms);
    launch_pdl(copy_kernel, dim3(grid), dim3(CP_THREADS), 0, st, static_cast<unsigned char*>(dst),
               static_cast<const unsigned char*>(src), bytes, wide ? 1 : 0);
}

}  // namespace gbnms
