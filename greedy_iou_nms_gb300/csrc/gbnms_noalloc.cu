// nms_resolve_mask_noalloc: the mask resolve with its scratch in a static
// device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run NMS:
// a plugin whose host framework owns every allocation and forbids allocating
// in the per-inference call, a real-time loop whose memory is planned once at
// start-up, or a certified deployment that bans dynamic allocation after
// initialisation.  They still own the inputs and the outputs; only the scratch
// has nowhere to live.  This entry point keeps that scratch in one file-scope
// __device__ array, so the call itself allocates nothing.
//
// The array is sized for NMS_NOALLOC_MAX_N boxes and exists on every GPU that
// loads the library until the process exits.  Host code cannot use its name
// as a device address (it is a host-side stand-in), so the device address is
// looked up with cudaGetSymbolAddress once per device, with that device
// current, on the first call made on that device.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gbnms {
namespace {

// Column-view band of the largest mask this entry point accepts:
// ceil(NMS_NOALLOC_MAX_N/64) tiles x (BAND_L+1) blocks x 64 words.
constexpr size_t kNoallocBandWords =
    static_cast<size_t>((NMS_NOALLOC_MAX_N + 63) / 64) * (BAND_L + 1) * 64;

static __device__ __align__(256) uint64_t g_noalloc_band[kNoallocBandWords];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
uint64_t* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_band on the current device (looked up once).
cudaError_t noalloc_band(uint64_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_band);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<uint64_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace gbnms

using namespace gbnms;

extern "C" nms_status nms_resolve_mask_noalloc(const uint64_t* mask, int64_t n, const int32_t* perm,
                                               int32_t max_out, int64_t* keep, int64_t* count,
                                               void* stream)
{
    if (n < 0) return NMS_ERR_INVALID_ARG;
    if (n > NMS_NOALLOC_MAX_N) return NMS_ERR_CAPACITY;
    if (!count || (n > 0 && (!mask || !keep))) return NMS_ERR_INVALID_ARG;
    if (n > 0 && reinterpret_cast<uintptr_t>(mask) % 16 != 0) return NMS_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    uint64_t* band = nullptr;
    if (noalloc_band(&band) != cudaSuccess) return NMS_ERR_CUDA;
    if (n == 0) {
        cudaMemsetAsync(count, 0, sizeof(int64_t), st);
        return cudaGetLastError() == cudaSuccess ? NMS_OK : NMS_ERR_CUDA;
    }
    // Every call rewrites every band block it reads (blocks above the first
    // row tile are written as zeros), so nothing left by an earlier call is
    // used and nothing needs clearing first.
    const int64_t ldw = nms_mask_row_words(n);
    launch_band_from_mask(mask, ldw, static_cast<int>(n), band, st);
    launch_resolve_single(mask, ldw, nullptr, 1, band, nullptr, nullptr, nullptr, nullptr,
                          static_cast<int>(n), perm, max_out, keep, count, nullptr, st);
    return cudaGetLastError() == cudaSuccess ? NMS_OK : NMS_ERR_CUDA;
}
