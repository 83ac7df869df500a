// Single-image path, front end: optional score pre-filter (warp-aggregated
// atomics) and the stable descending sort by rank counting, fused with the
// gather of the sorted boxes.
//
// "NMS CUDA代码学习", section 算法与数据流 step 1 (sort by descending score,
// stable) and section "host 侧" (the sort permutation maps kept positions back
// to input indices); "Fastest Matrix NMS in the West (Part 2)", section
// "PyTorch extension" (stable descending sort, then the boxes gathered
// contiguous for the IoU kernel); "YOLOv5后处理GPU移植实战", section 1.2
// (atomic slot counters; per-warp aggregation cuts the contention).
#include "common.cuh"
#include "internal.h"

namespace gbnms {

// Pre-filter: candidates with score > score_thr, compacted with one atomic per
// warp.  The order of the compacted list is not deterministic; the rank sort
// below includes the input index in its key, so the result is.
__global__ void prefilter_kernel(const float* __restrict__ scores, int n, float score_thr,
                                 int* __restrict__ cand, int* __restrict__ m_count)
{
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    bool pass = i < n && scores[i] > score_thr;
    unsigned ballot = __ballot_sync(FULL, pass);
    if (!ballot) return;
    unsigned l = lane_id();
    int base = 0;
    if (l == static_cast<unsigned>(__ffs(ballot) - 1)) base = atomicAdd(m_count, __popc(ballot));
    base = __shfl_sync(FULL, base, __ffs(ballot) - 1);
    if (pass) cand[base + __popc(ballot & ((1u << l) - 1u))] = i;
}

// Rank sort.  A candidate's sorted position is the number of candidates whose
// (score key, index) is smaller; the keys are unique, so the positions form a
// permutation and the sort is stable by construction.  Each CTA ranks RS_I
// candidates against all of them: lane l of a warp owns 4 consecutive
// candidates (group l % 8) and takes every fourth 4-key group of the warp's
// share (subset l / 8), so one 16-byte shared-memory load feeds 16 compares.
//
// Without a pre-filter the candidate list is the input in index order, so a
// j before candidate i counts when key_j <= key_i and a j after it when key_j
// < key_i: one 32-bit compare per pair.  With a pre-filter the list order is
// arbitrary and the 64-bit (key, index) compare is used.
constexpr int RS_WARPS = 16;
constexpr int RS_I = 32;         // candidates ranked per CTA (8 lanes x 4)
constexpr int RS_SUB = 4;        // key subsets per warp (lanes / 8)
constexpr int RS_CHUNK = 4096;   // keys staged in shared memory per step

__global__ void __launch_bounds__(RS_WARPS * 32)
rank_sort_kernel(const float* __restrict__ scores, const float4* __restrict__ boxes,
                 const int* __restrict__ cand, const int* __restrict__ m_dev, int m_bound,
                 int* __restrict__ perm, float4* __restrict__ boxes_s, int32_t* status,
                 uint64_t* __restrict__ rowbits, int NB)
{
    __shared__ __align__(16) uint64_t keys64[RS_CHUNK];   // u32 keys use the first half
    __shared__ uint32_t part[RS_WARPS * RS_SUB][RS_I];
    uint32_t* keys32 = reinterpret_cast<uint32_t*>(keys64);

    const int m = m_dev ? *m_dev : m_bound;
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) *status = 0;
    const int i0 = blockIdx.x * RS_I;
    // Clear the mask's per-row chunk bitmaps of rows [i0, i0+RS_I) for the
    // mask kernel that follows.
    if (rowbits) {
        const int64_t q0 = static_cast<int64_t>(i0) * NB;
        const int64_t q1 = static_cast<int64_t>(min(i0 + RS_I, m_bound)) * NB;
        for (int64_t q = q0 + threadIdx.x; q < q1; q += blockDim.x) rowbits[q] = 0;
    }
    if (i0 >= m) return;

    const unsigned l = lane_id();
    const int w = threadIdx.x >> 5;
    const int ig = l & 7, js = l >> 3;
    const int sub = w * RS_SUB + js;           // this lane's share of the keys
    const int nsub = RS_WARPS * RS_SUB;
    int iv[4];
    uint32_t cnt[4] = {0, 0, 0, 0};
#pragma unroll
    for (int u = 0; u < 4; ++u) iv[u] = i0 + 4 * ig + u;

    if (!cand) {
        uint32_t kk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) kk[u] = iv[u] < m ? score_key(scores[iv[u]]) : 0xffffffffu;
        for (int c0 = 0; c0 < m; c0 += RS_CHUNK) {
            const int cn = min(RS_CHUNK, m - c0);
            __syncthreads();
            // Four scores per 16-byte load when the chunk start is aligned (all
            // loads of a thread in flight together); the ragged end pads with
            // the largest key.
            const bool vec = ((reinterpret_cast<uintptr_t>(scores + c0) & 15) == 0);
            if (vec) {
                const float4* s4 = reinterpret_cast<const float4*>(scores + c0);
                const int n4 = cn >> 2;
#pragma unroll 4
                for (int t = threadIdx.x; t < n4; t += blockDim.x) {
                    const float4 v = s4[t];
                    reinterpret_cast<uint4*>(keys32)[t] =
                        make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
                }
                for (int t = 4 * n4 + threadIdx.x; t < cn; t += blockDim.x) keys32[t] = score_key(scores[c0 + t]);
            } else {
#pragma unroll 4
                for (int t = threadIdx.x; t < cn; t += blockDim.x) keys32[t] = score_key(scores[c0 + t]);
            }
            for (int t = cn + threadIdx.x; t < ((cn + 3) & ~3); t += blockDim.x) keys32[t] = 0xffffffffu;
            __syncthreads();
            const uint4* k4 = reinterpret_cast<const uint4*>(keys32);
            for (int q = sub; 4 * q < cn; q += nsub) {
                const uint4 v = k4[q];
                const int j = c0 + 4 * q;
                if (j + 3 < i0) {               // all four before the block: ties count
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        cnt[u] += (v.x <= kk[u]) + (v.y <= kk[u]) + (v.z <= kk[u]) + (v.w <= kk[u]);
                } else if (j >= i0 + RS_I) {    // all after: strict
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        cnt[u] += (v.x < kk[u]) + (v.y < kk[u]) + (v.z < kk[u]) + (v.w < kk[u]);
                } else {
                    const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int jj = j + x;
                        if (jj < m) {
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                cnt[u] += (e[x] < kk[u]) || (e[x] == kk[u] && jj < iv[u]);
                        }
                    }
                }
            }
        }
    } else {
        int xv[4];
        uint64_t kk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            xv[u] = iv[u] < m ? cand[iv[u]] : 0;
            kk[u] = iv[u] < m ? order_key(scores[xv[u]], xv[u]) : ~0ull;
        }
        for (int c0 = 0; c0 < m; c0 += RS_CHUNK) {
            const int cn = min(RS_CHUNK, m - c0);
            __syncthreads();
            for (int t = threadIdx.x; t < cn; t += blockDim.x) {
                const int x = cand[c0 + t];
                keys64[t] = order_key(scores[x], x);
            }
            __syncthreads();
            for (int t = sub; t < cn; t += nsub) {
                const uint64_t k = keys64[t];
#pragma unroll
                for (int u = 0; u < 4; ++u) cnt[u] += k < kk[u];
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) part[sub][4 * ig + u] = cnt[u];
    __syncthreads();
    if (threadIdx.x < RS_I) {
        const int e = threadIdx.x;
        const int i = i0 + e;
        if (i < m) {
            uint32_t r = 0;
            for (int q = 0; q < nsub; ++q) r += part[q][e];
            const int x = cand ? cand[i] : i;
            perm[r] = x;
            boxes_s[r] = boxes[x];
        }
    }
}

void launch_prefilter(const float* scores, int n, float score_thr, int* cand, int* m_count,
                      cudaStream_t st)
{
    cudaMemsetAsync(m_count, 0, sizeof(int), st);
    if (n > 0) prefilter_kernel<<<(n + 255) / 256, 256, 0, st>>>(scores, n, score_thr, cand, m_count);
}

void launch_rank_sort(const float* scores, const float4* boxes, const int* cand, const int* m_dev,
                      int m_bound, int* perm, float4* boxes_s, int32_t* status, uint64_t* rowbits,
                      int NB, cudaStream_t st)
{
    int grid = (m_bound + RS_I - 1) / RS_I;
    if (grid < 1) grid = 1;
    rank_sort_kernel<<<grid, RS_WARPS * 32, 0, st>>>(scores, boxes, cand, m_dev, m_bound, perm,
                                                    boxes_s, status, rowbits, NB);
}

}  // namespace gbnms
