// nms_resolve_mask_noalloc: the mask resolve without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run NMS:
// a plugin whose host framework owns every allocation and forbids allocating
// in the per-inference call, a real-time loop whose memory is planned once at
// start-up, or a certified deployment that bans dynamic allocation after
// initialisation.  They still own the inputs and the outputs.  The walk keeps
// its removed-bitmap, its band windows (built from the mask itself) and its
// hand-over state in the shared memory of its one thread block, so the call
// needs no device scratch and allocates nothing.
#include "common.cuh"
#include "internal.h"

using namespace gbnms;

extern "C" nms_status nms_resolve_mask_noalloc(const uint64_t* mask, int64_t n, const int32_t* perm,
                                               int32_t max_out, int64_t* keep, int64_t* count,
                                               void* stream)
{
    if (n < 0) return NMS_ERR_INVALID_ARG;
    if (n > NMS_NOALLOC_MAX_N) return NMS_ERR_CAPACITY;
    // The resolve reads the mask with 16-byte loads and perm as int32, and
    // writes keep and count as int64: misaligned pointers are refused here.
    auto misaligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
    if (!count || misaligned(count, 8)) return NMS_ERR_INVALID_ARG;
    if (n > 0 && (!mask || !keep || misaligned(mask, 16) || misaligned(keep, 8) || (perm && misaligned(perm, 4))))
        return NMS_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    if (n == 0) {
        cudaMemsetAsync(count, 0, sizeof(int64_t), st);
        return cudaGetLastError() == cudaSuccess ? NMS_OK : NMS_ERR_CUDA;
    }
    launch_resolve_single(mask, nms_mask_row_words(n), nullptr, 1, nullptr, nullptr, 0u, nullptr, nullptr,
                          static_cast<int>(n), perm, max_out, keep, count, nullptr, st);
    return cudaGetLastError() == cudaSuccess ? NMS_OK : NMS_ERR_CUDA;
}
