// Ordered output of a kept bitmap; for Fast NMS of one image, the boxes no
// earlier box suppresses.
//
// "YOLOv5后处理GPU移植实战", section 2.2 稳定性增强方案: a box is suppressed
// when a box of higher priority (higher score, or equal score and lower
// index) has IoU above the threshold with it, whether or not that box was
// suppressed itself.  In sorted positions that is exactly bit p of the
// mask kernel's bitmap of boxes with an earlier neighbour over the threshold,
// so the answer is the clear bits, in order, mapped through the sort
// permutation.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int FE_THREADS = 1024;

// One CTA: warp w owns the 32-box words [w*wpw, (w+1)*wpw); a block prefix of
// the warps' kept counts places them, and within a word lane l writes box
// 32w+l (coalesced perm loads and keep stores).
// bits: 32-box words whose set bits (clear bits when `clear`) are the kept
// boxes; fs (optional): a value per sorted box written beside each kept one.
__global__ void __launch_bounds__(FE_THREADS)
bits_emit_kernel(const uint32_t* __restrict__ bits_in, int clear, const int* __restrict__ m_dev, int m_bound,
                 const int* __restrict__ perm, const float* __restrict__ fs, int max_out,
                 int64_t* __restrict__ keep, float* __restrict__ keep_fs, int64_t* __restrict__ counts)
{
    pdl_wait();
    pdl_release();
    __shared__ int scratch[32];
    const int n = m_dev ? *m_dev : m_bound;
    const int NW = (n + 31) / 32;
    const unsigned l = lane_id();
    const int warp = threadIdx.x >> 5;
    auto kept_word = [&](int w) {
        const uint32_t valid = (w == NW - 1 && (n & 31)) ? (1u << (n & 31)) - 1u : ~0u;
        return (clear ? ~bits_in[w] : bits_in[w]) & valid;
    };
    const int wpw = (NW + 31) / 32;
    const int a0 = min(warp * wpw, NW), a1 = min(a0 + wpw, NW);
    int c = 0;
    for (int w = a0 + static_cast<int>(l); w < a1; w += 32) c += __popc(kept_word(w));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(FULL, c, d);
    if (l == 0) scratch[warp] = c;
    __syncthreads();
    if (warp == 0) {
        int v = scratch[l];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(FULL, v, d);
            if (static_cast<int>(l) >= d) v += y;
        }
        scratch[l] = v;
    }
    __syncthreads();
    const int total = scratch[31];
    const int cap = max_out > 0 ? max_out : INT_MAX;
    int base = warp ? scratch[warp - 1] : 0;
    const uint32_t below = (1u << l) - 1u;
    constexpr int OW = 2;  // words per step (a short loop: its code is fetched cold after an L2 flush)
    for (int wb = a0; wb < a1 && base < cap; wb += OW) {
        uint32_t bits[OW];
        int v[OW];
        float f[OW];
#pragma unroll
        for (int u = 0; u < OW; ++u) {
            bits[u] = wb + u < a1 ? kept_word(wb + u) : 0u;
            const int j = 32 * (wb + u) + static_cast<int>(l);
            const bool k = (bits[u] >> l) & 1u;
            v[u] = k ? (perm ? perm[j] : j) : 0;
            f[u] = k && fs ? fs[j] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < OW; ++u) {
            const int pos = base + __popc(bits[u] & below);
            if (((bits[u] >> l) & 1u) && pos < cap) {
                keep[pos] = v[u];
                if (keep_fs) keep_fs[pos] = f[u];
            }
            base += __popc(bits[u]);
        }
    }
    if (threadIdx.x == 0) counts[0] = total < cap ? total : cap;
}

// With max_out, whether the leading k sorted boxes already hold max_out kept
// boxes (bits: 32-box words whose set bits, or clear bits when `clear`, are
// the kept ones).  For Fast NMS (the clear bits of the neighbour bitmap) and
// Matrix NMS (the kept bitmap) a box's decision depends only on the boxes
// before it, so once the prefix is done its decisions are final and the
// first max_out kept boxes are all among them.  Sets *done (also when the
// prefix is every box) so that the later stage returns at once.
__global__ void __launch_bounds__(FE_THREADS)
prefix_kernel(const uint32_t* __restrict__ bits, int clear, const int* __restrict__ m_dev, int m_bound, int k,
              int max_out, int* __restrict__ done)
{
    pdl_wait();
    pdl_release();
    __shared__ int wsum[FE_THREADS / 32];
    const int n = m_dev ? *m_dev : m_bound;
    const int kk = min(n, k);
    const int NW = (kk + 31) / 32;
    int c = 0;
    for (int w = threadIdx.x; w < NW; w += FE_THREADS) {
        const uint32_t valid = (w == NW - 1 && (kk & 31)) ? (1u << (kk & 31)) - 1u : ~0u;
        c += __popc((clear ? ~bits[w] : bits[w]) & valid);
    }
    c = __reduce_add_sync(FULL, c);
    if (lane_id() == 0) wsum[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x < 32) {
        const int t = __reduce_add_sync(FULL, wsum[threadIdx.x]);
        if (threadIdx.x == 0) *done = (n <= k || t >= max_out) ? 1 : 0;
    }
}

void launch_fast_prefix(const uint64_t* haspred, const int* m_dev, int m_bound, int k, int max_out, int* done,
                        cudaStream_t st)
{
    launch_pdl(prefix_kernel, dim3(1), dim3(FE_THREADS), 0, st, reinterpret_cast<const uint32_t*>(haspred), 1,
               m_dev, m_bound, k, max_out, done);
}

void launch_kept_prefix(const uint32_t* kept, const int* m_dev, int m_bound, int k, int max_out, int* done,
                        cudaStream_t st)
{
    launch_pdl(prefix_kernel, dim3(1), dim3(FE_THREADS), 0, st, kept, 0, m_dev, m_bound, k, max_out, done);
}

void launch_fast_emit(const uint64_t* haspred, const int* m_dev, int m_bound, const int* perm, int max_out,
                      int64_t* keep, int64_t* counts, cudaStream_t st)
{
    launch_pdl(bits_emit_kernel, dim3(1), dim3(FE_THREADS), 0, st, reinterpret_cast<const uint32_t*>(haspred), 1,
               m_dev, m_bound, perm, nullptr, max_out, keep, nullptr, counts);
}

void launch_bits_emit(const uint32_t* bits, const int* m_dev, int m_bound, const int* perm, const float* fs,
                      int max_out, int64_t* keep, float* keep_fs, int64_t* counts, cudaStream_t st)
{
    launch_pdl(bits_emit_kernel, dim3(1), dim3(FE_THREADS), 0, st, bits, 0, m_dev, m_bound, perm, fs, max_out, keep,
               keep_fs, counts);
}

}  // namespace gbnms
