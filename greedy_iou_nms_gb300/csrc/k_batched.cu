// Batched, class-aware path: pre-filter + bucketing by (image, class)
// segment, per-segment greedy NMS, per-image merge in score order.
//
// "YOLOv5后处理GPU移植实战": section 1.1/1.2 (candidates above the confidence
// threshold claim slots with atomic counters; aggregating per warp before the
// global atomic cuts the contention), section 2.2 (suppression only between
// boxes of the same class, equal scores resolved by the lower index).
// "NMS CUDA代码学习", section 算法与数据流 (greedy in descending score order,
// strict IoU > threshold) and section Phase 1 (a warp's 32 lanes evaluate 32
// candidates and one ballot folds the votes into a mask word).
//
// A box never suppresses a box of another class or image, so each (image,
// class) segment is an independent greedy NMS; the image's answer is the
// union of its segments' answers in descending score order (ties by index),
// cut at max_out.
#include "common.cuh"
#include "internal.h"

namespace gbnms {

// ----------------------------------------------------------------- bucketing

// One CTA: zero the per-segment counters, check the image offsets.
__global__ void batched_setup_kernel(const int64_t* __restrict__ off, int batch, int64_t n,
                                     int S, int* __restrict__ seg_cnt, int* __restrict__ ok,
                                     int32_t* status)
{
    pdl_release();
    for (int s = threadIdx.x; s < S; s += blockDim.x) seg_cnt[s] = 0;
    int bad = 0;
    if (off) {
        for (int b = threadIdx.x; b <= batch; b += blockDim.x) {
            int64_t v = off[b];
            if (v < 0 || v > n) bad = 1;
            if (b == 0 && v != 0) bad = 1;
            if (b == batch && v != n) bad = 1;
            if (b < batch && off[b + 1] < v) bad = 1;
        }
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        *ok = !bad;
        *status = bad ? NMS_ERR_INVALID_ARG : NMS_OK;
    }
}

__device__ __forceinline__ int image_of(const int64_t* __restrict__ off, int batch, int64_t i)
{
    if (!off) return 0;
    int lo = 0, hi = batch;  // off[lo] <= i < off[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (off[mid] <= i) lo = mid; else hi = mid;
    }
    return lo;
}

// Candidates claim a slot in their segment; lanes of a warp that share a
// segment aggregate into one atomic.
__global__ void batched_count_kernel(const float* __restrict__ scores,
                                     const int32_t* __restrict__ cls, int C,
                                     const int64_t* __restrict__ off, int batch, int n,
                                     int use_thr, float score_thr, const int* __restrict__ img_rows,
                                     const int* __restrict__ ok, int* __restrict__ seg_cnt,
                                     int* __restrict__ seg_of, int* __restrict__ slot, int32_t* status)
{
    pdl_wait();
    pdl_release();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (!*ok) return;
    int seg = -1;
    if (i < n) {
        const int b = image_of(off, batch, i);
        // With img_rows, only the first img_rows[b] rows of image b take part.
        if (!img_rows || i - (off ? off[b] : 0) < img_rows[b]) {
            const int c = cls ? cls[i] : 0;
            if (c < 0 || c >= C) {
                set_status(status, NMS_ERR_INVALID_ARG);
            } else if (!use_thr || scores[i] > score_thr) {
                seg = b * C + c;
            }
        }
    }
    const unsigned active = __ballot_sync(FULL, seg >= 0);
    int my_slot = -1;
    if (seg >= 0) {
        const unsigned peers = __match_any_sync(active, seg);
        const int leader = __ffs(peers) - 1;
        int base = 0;
        if (static_cast<int>(lane_id()) == leader) base = atomicAdd(&seg_cnt[seg], __popc(peers));
        base = __shfl_sync(peers, base, leader);
        my_slot = base + __popc(peers & ((1u << lane_id()) - 1u));
    }
    if (i < n) {
        slot[i] = my_slot;
        seg_of[i] = seg;
    }
}

// One CTA: exclusive scan of the segment counters into segment offsets.
__global__ void batched_scan_kernel(const int* __restrict__ seg_cnt, int S,
                                    int* __restrict__ seg_off)
{
    pdl_wait();
    pdl_release();
    __shared__ int carry;
    __shared__ int warp_sums[32];
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const unsigned l = lane_id();
    const int wp = threadIdx.x >> 5;
    for (int s0 = 0; s0 < S; s0 += blockDim.x) {
        int s = s0 + threadIdx.x;
        int v = s < S ? seg_cnt[s] : 0;
        int x = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(FULL, x, d);
            if (static_cast<int>(l) >= d) x += y;
        }
        if (l == 31) warp_sums[wp] = x;
        __syncthreads();
        if (wp == 0) {
            int nw = blockDim.x >> 5;
            int ws = static_cast<int>(l) < nw ? warp_sums[l] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                int y = __shfl_up_sync(FULL, ws, d);
                if (static_cast<int>(l) >= d) ws += y;
            }
            warp_sums[l] = ws;  // inclusive
        }
        __syncthreads();
        int excl = carry + (wp > 0 ? warp_sums[wp - 1] : 0) + x - v;
        if (s < S) seg_off[s] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) seg_off[S] = carry;
}

// seg_of/slot are only written when the offsets passed the check, so the
// scatter must skip everything otherwise.
__global__ void batched_scatter_kernel(const int* __restrict__ seg_of, const int* __restrict__ slot,
                                       const int* __restrict__ seg_off, int n,
                                       const int* __restrict__ ok, int* __restrict__ cand)
{
    pdl_wait();
    pdl_release();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n || !*ok) return;
    const int s = seg_of[i];
    if (s >= 0) cand[seg_off[s] + slot[i]] = i;
}

// --------------------------------------------------- small segments (<= 64)
//
// One warp per segment: rank the (score key, index) keys inside the warp,
// stage the sorted boxes in shared memory, build the 64x64 mask in column view
// (each lane owns two candidates and collects which earlier boxes suppress
// them), resolve it (resolve_tile_col) and write the kept keys.
constexpr int SS_WARPS = 4;

__global__ void __launch_bounds__(SS_WARPS * 32)
seg_small_kernel(const float4* __restrict__ boxes, const float* __restrict__ scores,
                 const int* __restrict__ seg_off, const int* __restrict__ cand, int S,
                 const int* __restrict__ ok, float thr, int max_out, int fast,
                 uint64_t* __restrict__ kept_key, int* __restrict__ kept_cnt)
{
    pdl_wait();
    pdl_release();
    __shared__ float4 sbox[SS_WARPS][64];
    __shared__ float sarea[SS_WARPS][64];
    __shared__ uint64_t skey[SS_WARPS][64];
    const int wp = threadIdx.x >> 5;
    const int s = blockIdx.x * SS_WARPS + wp;
    if (s >= S || !*ok) return;
    const int lo = seg_off[s];
    const int m = seg_off[s + 1] - lo;
    if (m > 64) return;  // handled by seg_large_kernel
    const unsigned l = lane_id();
    if (m == 0) {
        if (l == 0) kept_cnt[s] = 0;
        return;
    }
    const bool ha = static_cast<int>(l) < m, hb = static_cast<int>(l) + 32 < m;
    const int xa = ha ? cand[lo + l] : 0;
    const int xb = hb ? cand[lo + 32 + l] : 0;
    // The boxes are loaded with the scores (one round of dependent loads).
    const float4 bxa = ha ? boxes[xa] : make_float4(0, 0, 0, 0);
    const float4 bxb = hb ? boxes[xb] : make_float4(0, 0, 0, 0);
    const uint64_t ka = ha ? order_key(scores[xa], xa) : ~0ull;
    const uint64_t kb = hb ? order_key(scores[xb], xb) : ~0ull;
    int ra = 0, rb = 0;
    for (int e = 0; e < m; ++e) {
        uint64_t ke = __shfl_sync(FULL, e < 32 ? ka : kb, e & 31);
        ra += ke < ka;
        rb += ke < kb;
    }
    if (ha) { sbox[wp][ra] = bxa; skey[wp][ra] = ka; }
    if (hb) { sbox[wp][rb] = bxb; skey[wp][rb] = kb; }
    __syncwarp();
    if (ha) sarea[wp][l] = box_area(sbox[wp][l]);
    if (hb) sarea[wp][l + 32] = box_area(sbox[wp][l + 32]);
    __syncwarp();
    const float4 ca = ha ? sbox[wp][l] : make_float4(0, 0, 0, 0);
    const float4 cb = hb ? sbox[wp][l + 32] : make_float4(0, 0, 0, 0);
    const float aa = ha ? sarea[wp][l] : 0.0f;
    const float ab = hb ? sarea[wp][l + 32] : 0.0f;
    // Column view of the segment's mask: bit r of colA is set iff sorted box r
    // suppresses sorted box l (r < l); colB likewise for box l+32.
    uint64_t colA = 0, colB = 0;
    if (m <= 32) {  // most segments: one column per lane
        for (int r = 0; r < m; ++r) {
            const bool va = ha && static_cast<int>(l) > r && suppress_exact(sbox[wp][r], sarea[wp][r], ca, aa, thr);
            colA |= static_cast<uint64_t>(va) << r;
        }
    } else {
        for (int r = 0; r < m; ++r) {
            const float4 rbx = sbox[wp][r];
            const float rar = sarea[wp][r];
            const bool va = ha && static_cast<int>(l) > r && suppress_exact(rbx, rar, ca, aa, thr);
            const bool vb = hb && static_cast<int>(l) + 32 > r && suppress_exact(rbx, rar, cb, ab, thr);
            colA |= static_cast<uint64_t>(va) << r;
            colB |= static_cast<uint64_t>(vb) << r;
        }
    }
    const uint64_t valid = m >= 64 ? ~0ull : ((1ull << m) - 1ull);
    // Greedy: resolve the column view; Fast NMS: keep the boxes no earlier
    // box suppresses.
    uint64_t K = fast ? ballot64(ha && colA == 0, hb && colB == 0) & valid : resolve_tile_col(valid, colA, colB);
    if (max_out > 0 && __popcll(K) > max_out) K = lowest_bits(K, max_out);
    if ((K >> l) & 1ull) kept_key[lo + __popcll(K & ((1ull << l) - 1ull))] = skey[wp][l];
    if ((K >> (l + 32)) & 1ull)
        kept_key[lo + __popcll(K & ((1ull << (l + 32)) - 1ull))] = skey[wp][l + 32];
    if (l == 0) kept_cnt[s] = __popcll(K);
}

// ------------------------------------------------------- large segments (> 64)
//
// A CTA per segment in turn, no mask in memory: the segment is ranked by counting,
// then walked tile by tile.  Each 64-candidate tile is first tested against
// every box kept so far (all threads), then its own 64x64 block is built (in
// column view) and resolved by warp 0.  Exact greedy; cost O(kept * m) IoUs on one SM.
constexpr int SL_THREADS = 512;
constexpr int SL_CACHE = 2048;  // kept boxes cached in shared memory (40 KB)

__global__ void __launch_bounds__(SL_THREADS)
seg_large_kernel(const float4* __restrict__ boxes, const float* __restrict__ scores,
                 const int* __restrict__ seg_off, const int* __restrict__ cand, int S,
                 const int* __restrict__ ok, float thr, int max_out, int fast,
                 uint64_t* __restrict__ sorted_key, float4* __restrict__ sorted_box,
                 uint64_t* __restrict__ kept_key, int* __restrict__ kept_cnt)
{
    __shared__ float4 kbox[SL_CACHE];
    __shared__ float karea[SL_CACHE];
    __shared__ uint64_t diag[64];
    __shared__ unsigned long long s_removed;
    __shared__ uint64_t s_kept;
    __shared__ int s_nk;

    pdl_release();  // runs beside the small-segment kernel, which ends before this grid does
    if (*ok) {
        // A few CTAs per SM take the segments in turn and skip the small ones
        // (the warp kernel's).
        for (int s = blockIdx.x; s < S; s += gridDim.x) {
            const int lo = seg_off[s];
            const int m = seg_off[s + 1] - lo;
            if (m <= 64) continue;
            __syncthreads();  // the previous segment's shared state is no longer read

            // Rank each candidate of the segment by counting smaller keys.
            for (int e = threadIdx.x; e < m; e += blockDim.x) {
                const int x = cand[lo + e];
                const uint64_t k = order_key(scores[x], x);
                int r = 0;
                for (int f = 0; f < m; ++f) {
                    const int y = cand[lo + f];
                    r += order_key(scores[y], y) < k;
                }
                sorted_key[lo + r] = k;
                sorted_box[lo + r] = boxes[x];
            }
            __syncthreads();

            int nk = 0;  // kept so far (uniform)
            const int cap = max_out > 0 ? max_out : m;
            const unsigned l = lane_id();
            for (int t0 = 0; t0 < m && nk < cap; t0 += 64) {
                const int tn = min(64, m - t0);
                if (threadIdx.x == 0) s_removed = 0;
                if (threadIdx.x < 64) diag[threadIdx.x] = 0;
                __syncthreads();
                // (a) candidates of the tile against every kept box (Fast NMS: every
                //     earlier box of the segment).
                {
                    const int cidx = threadIdx.x & 63;
                    const int slice = threadIdx.x >> 6;
                    const int nslice = blockDim.x >> 6;
                    if (cidx < tn) {
                        const float4 cbx = sorted_box[lo + t0 + cidx];
                        const float car = box_area(cbx);
                        bool hit = false;
                        if (fast) {
                            for (int k = slice; k < t0 && !hit; k += nslice) {
                                const float4 kb = sorted_box[lo + k];
                                hit = suppress_exact(kb, box_area(kb), cbx, car, thr);
                            }
                        }
                        for (int k = slice; !fast && k < nk && !hit; k += nslice) {
                            float4 kb;
                            float ka;
                            if (k < SL_CACHE) {
                                kb = kbox[k];
                                ka = karea[k];
                            } else {
                                // Beyond the cache: kept_key holds the kept box's sorted position.
                                kb = sorted_box[lo + static_cast<int>(kept_key[lo + k])];
                                ka = box_area(kb);
                            }
                            hit = suppress_exact(kb, ka, cbx, car, thr);
                        }
                        if (hit) atomicOr(&s_removed, 1ull << cidx);
                    }
                }
                // (b) the tile's own 64x64 block in column view: bit i of diag[j] set iff
                //     i < j and i suppresses j.
                for (int q = threadIdx.x; q < 64 * 64; q += blockDim.x) {
                    const int i = q >> 6, j = q & 63;
                    if (i < j && j < tn) {
                        const float4 bi = sorted_box[lo + t0 + i];
                        const float4 bj = sorted_box[lo + t0 + j];
                        if (suppress_exact(bi, box_area(bi), bj, box_area(bj), thr))
                            atomicOr(reinterpret_cast<unsigned long long*>(&diag[j]), 1ull << i);
                    }
                }
                __syncthreads();
                if (threadIdx.x < 32) {
                    const uint64_t valid = tn >= 64 ? ~0ull : ((1ull << tn) - 1ull);
                    const uint64_t cand = valid & ~static_cast<uint64_t>(s_removed);
                    uint64_t K = fast ? cand & ballot64(diag[l] == 0, diag[l + 32] == 0)
                                      : resolve_tile_col(cand, diag[l], diag[l + 32]);
                    const int room = cap - nk;
                    if (__popcll(K) > room) K = lowest_bits(K, room);
                    if (l == 0) { s_kept = K; s_nk = __popcll(K); }
                }
                __syncthreads();
                const uint64_t K = s_kept;
                // Append the tile's kept boxes in order: cache + record the sorted position.
                if (threadIdx.x < 64 && ((K >> threadIdx.x) & 1ull)) {
                    const int r = nk + __popcll(K & ((1ull << threadIdx.x) - 1ull));
                    const float4 b = sorted_box[lo + t0 + threadIdx.x];
                    if (r < SL_CACHE) { kbox[r] = b; karea[r] = box_area(b); }
                    // Temporarily store the sorted position; replaced by the key at the end.
                    kept_key[lo + r] = static_cast<uint64_t>(t0 + threadIdx.x);
                }
                nk += s_nk;
                __syncthreads();
            }
            // Replace the recorded sorted positions by the (score key, index) keys.
            __syncthreads();
            for (int r = threadIdx.x; r < nk; r += blockDim.x) {
                const int pos = static_cast<int>(kept_key[lo + r]);
                kept_key[lo + r] = sorted_key[lo + pos];
            }
            if (threadIdx.x == 0) kept_cnt[s] = nk;
        }
    }
    pdl_wait();  // the merge that follows also needs the small segments
}

// ------------------------------------------------------------ per-image merge
//
// One CTA per image: gather the kept keys of the image's segments into a
// contiguous run, sort them (a bitonic sort in shared memory up to MG_CHUNK
// keys, ranking by counting beyond) and write the indices of the first `cap`
// in order.
constexpr int MG_THREADS = 1024;
constexpr int MG_CHUNK = 4096;

// Ascending bitonic sort of the np (a power of two) unique keys in s (the
// padding keys, all ones, sort last), by the CTA.
__device__ __forceinline__ void bitonic_sort(uint64_t* s, int np)
{
    for (int k = 2; k <= np; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < np; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const uint64_t x = s[i], y = s[p];
                    if ((x > y) == ((i & k) == 0)) {
                        s[i] = y;
                        s[p] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Ascending bitonic sort of R * MG_THREADS unique keys held in registers:
// key e is v[e / MG_THREADS] of thread e % MG_THREADS.  Partners fewer than 32
// apart are in the same warp and swap by shuffles, partners MG_THREADS or more
// apart are in the same thread, and only the steps in between go through
// shared memory s (R * MG_THREADS keys), with two CTA barriers each.
template <int R>
__device__ __forceinline__ void bitonic_sort_regs(uint64_t (&v)[R], uint64_t* s)
{
    const int t = threadIdx.x;
    constexpr int NP = R * MG_THREADS;
    for (int k = 2; k <= NP; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= MG_THREADS) {
                const int jr = j / MG_THREADS;  // the partner is register r ^ jr of this thread
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int q = r + 1; q < R; ++q)
                        if (q == (r ^ jr)) {
                            const uint64_t x = v[r], y = v[q];
                            const bool asc = ((r * MG_THREADS + t) & k) == 0;
                            v[r] = asc ? min(x, y) : max(x, y);
                            v[q] = asc ? max(x, y) : min(x, y);
                        }
            } else if (j >= 32) {
#pragma unroll
                for (int r = 0; r < R; ++r) s[r * MG_THREADS + t] = v[r];
                __syncthreads();
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int e = r * MG_THREADS + t;
                    const uint64_t y = s[e ^ j];
                    const bool keep_min = ((e & j) == 0) == ((e & k) == 0);
                    v[r] = keep_min ? min(v[r], y) : max(v[r], y);
                }
                __syncthreads();
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int e = r * MG_THREADS + t;
                    const uint64_t y = __shfl_xor_sync(FULL, v[r], j);
                    const bool keep_min = ((e & j) == 0) == ((e & k) == 0);
                    v[r] = keep_min ? min(v[r], y) : max(v[r], y);
                }
            }
        }
    }
}

// Kept keys of the image's segments [s0, s0 + C) into registers (key e to
// v[e / MG_THREADS] of thread e % MG_THREADS, ~0 past tot), sorted, and the
// first cap written out.
template <int R>
__device__ __forceinline__ void merge_regs(const int* __restrict__ seg_off, const uint64_t* __restrict__ kept_key,
                                           const int* seg_pre, int s0, int C, int tot, int cap,
                                           int64_t* __restrict__ keep, int64_t out0, uint64_t* s)
{
    uint64_t v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int e = r * MG_THREADS + static_cast<int>(threadIdx.x);
        uint64_t k = ~0ull;
        if (e < tot) {
            int lo = 0, hi = C;  // last segment with prefix <= e
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (seg_pre[mid] <= e) lo = mid; else hi = mid;
            }
            k = kept_key[seg_off[s0 + lo] + (e - seg_pre[lo])];
        }
        v[r] = k;
    }
    bitonic_sort_regs<R>(v, s);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int e = r * MG_THREADS + static_cast<int>(threadIdx.x);
        if (e < cap) keep[out0 + e] = static_cast<int64_t>(v[r] & 0xffffffffu);
    }
}

__global__ void __launch_bounds__(MG_THREADS)
merge_kernel(const int* __restrict__ seg_off, const int* __restrict__ kept_cnt,
             const uint64_t* __restrict__ kept_key, int C, const int64_t* __restrict__ off,
             const int* __restrict__ ok, int max_out, uint64_t* __restrict__ stage,
             int64_t* __restrict__ keep, int64_t* __restrict__ counts)
{
    pdl_wait();
    pdl_release();
    __shared__ uint64_t ck[MG_CHUNK];
    __shared__ int seg_pre[MG_THREADS];
    __shared__ int s_tot;
    __shared__ int warp_sums[32];
    const int b = blockIdx.x;
    if (!*ok) {
        if (threadIdx.x == 0) counts[b] = 0;
        return;
    }
    const int s0 = b * C;
    const int base = seg_off[s0];  // the image's segments are contiguous
    const int64_t out0 = max_out > 0 ? static_cast<int64_t>(b) * max_out : off ? off[b] : 0;
    if (C <= MG_THREADS) {
        // Kept counts of the image's segments and their exclusive prefix in
        // shared memory; with at most MG_CHUNK keys each thread fetches keys
        // straight into the sort buffer (its segment by binary search).
        const int v = static_cast<int>(threadIdx.x) < C ? kept_cnt[s0 + threadIdx.x] : 0;
        int x = v;
        const unsigned ll = lane_id();
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(FULL, x, d);
            if (static_cast<int>(ll) >= d) x += y;
        }
        const int w = threadIdx.x >> 5;
        if (ll == 31) warp_sums[w] = x;
        __syncthreads();
        if (w == 0) {
            int ws = static_cast<int>(ll) < static_cast<int>(blockDim.x >> 5) ? warp_sums[ll] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(FULL, ws, d);
                if (static_cast<int>(ll) >= d) ws += y;
            }
            warp_sums[ll] = ws;
        }
        __syncthreads();
        const int pre = (w > 0 ? warp_sums[w - 1] : 0) + x - v;
        if (static_cast<int>(threadIdx.x) < C) seg_pre[threadIdx.x] = pre;
        const int tot = warp_sums[31];
        __syncthreads();
        if (tot <= MG_CHUNK) {
            const int cap = max_out > 0 ? min(max_out, tot) : tot;
            if (tot <= MG_THREADS) merge_regs<1>(seg_off, kept_key, seg_pre, s0, C, tot, cap, keep, out0, ck);
            else if (tot <= 2 * MG_THREADS) merge_regs<2>(seg_off, kept_key, seg_pre, s0, C, tot, cap, keep, out0, ck);
            else merge_regs<4>(seg_off, kept_key, seg_pre, s0, C, tot, cap, keep, out0, ck);
            if (threadIdx.x == 0) counts[b] = cap;
            return;
        }
    }
    // Exclusive scan of kept counts over the image's segments, then copy.
    if (threadIdx.x == 0) s_tot = 0;
    __syncthreads();
    const unsigned l = lane_id();
    const int wp = threadIdx.x >> 5;
    for (int c0 = 0; c0 < C; c0 += blockDim.x) {
        const int c = c0 + threadIdx.x;
        const int v = c < C ? kept_cnt[s0 + c] : 0;
        int x = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(FULL, x, d);
            if (static_cast<int>(l) >= d) x += y;
        }
        if (l == 31) warp_sums[wp] = x;
        __syncthreads();
        if (wp == 0) {
            int ws = static_cast<int>(l) < static_cast<int>(blockDim.x >> 5) ? warp_sums[l] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                int y = __shfl_up_sync(FULL, ws, d);
                if (static_cast<int>(l) >= d) ws += y;
            }
            warp_sums[l] = ws;
        }
        __syncthreads();
        const int start = s_tot + (wp > 0 ? warp_sums[wp - 1] : 0) + x - v;
        if (c < C) {
            const int src = seg_off[s0 + c];
            for (int e = 0; e < v; ++e) stage[base + start + e] = kept_key[src + e];
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) s_tot = start + v;
        __syncthreads();
    }
    const int tot = s_tot;
    const int cap = max_out > 0 ? min(max_out, tot) : tot;
    if (tot <= MG_CHUNK) {
        int np = 1;
        while (np < tot) np <<= 1;
        __syncthreads();
        for (int e = threadIdx.x; e < np; e += blockDim.x) ck[e] = e < tot ? stage[base + e] : ~0ull;
        __syncthreads();
        bitonic_sort(ck, np);
        for (int r = threadIdx.x; r < cap; r += blockDim.x) keep[out0 + r] = static_cast<int64_t>(ck[r] & 0xffffffffu);
        if (threadIdx.x == 0) counts[b] = cap;
        return;
    }
    // More than MG_CHUNK keys: rank by counting (keys are unique), staged
    // through shared memory.
    for (int e0 = 0; e0 < tot; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const uint64_t k = e < tot ? stage[base + e] : ~0ull;
        int r = 0;
        for (int f0 = 0; f0 < tot; f0 += MG_CHUNK) {
            const int fn = min(MG_CHUNK, tot - f0);
            __syncthreads();
            for (int f = threadIdx.x; f < fn; f += blockDim.x) ck[f] = stage[base + f0 + f];
            __syncthreads();
            for (int f = 0; f < fn; ++f) r += ck[f] < k;
        }
        if (e < tot && r < cap) keep[out0 + r] = static_cast<int64_t>(k & 0xffffffffu);
    }
    if (threadIdx.x == 0) counts[b] = cap;
}

// ------------------------------------------------------------------ launches

void launch_batched(const BatchedArgs& a, cudaStream_t st, const Stamps& stamps)
{
    const int n = a.n;
    const int S = a.S;
    stamps.record(0, st);
    batched_setup_kernel<<<1, 1024, 0, st>>>(a.off, a.batch, n, S, a.seg_cnt, a.ok, a.status);
    if (n > 0) {
        launch_pdl(batched_count_kernel, dim3((n + 255) / 256), dim3(256), 0, st, a.scores, a.cls, a.C, a.off,
                   a.batch, n, a.use_thr, a.score_thr, a.img_rows, a.ok, a.seg_cnt, a.seg_of, a.slot, a.status);
    }
    launch_pdl(batched_scan_kernel, dim3(1), dim3(1024), 0, st, a.seg_cnt, S, a.seg_off);
    if (n > 0)
        launch_pdl(batched_scatter_kernel, dim3((n + 255) / 256), dim3(256), 0, st, a.seg_of, a.slot, a.seg_off, n,
                   a.ok, a.cand);
    stamps.record(1, st);
    launch_pdl(seg_small_kernel, dim3((S + SS_WARPS - 1) / SS_WARPS), dim3(SS_WARPS * 32), 0, st, a.boxes, a.scores,
               a.seg_off, a.cand, S, a.ok, a.thr, a.max_out, a.fast, a.kept_key, a.kept_cnt);
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int large_grid = max(1, min(S, 2 * (sms > 0 ? sms : 1)));
    launch_pdl(seg_large_kernel, dim3(large_grid), dim3(SL_THREADS), 0, st, a.boxes, a.scores, a.seg_off, a.cand, S,
               a.ok, a.thr, a.max_out, a.fast, a.sorted_key, a.sorted_box, a.kept_key, a.kept_cnt);
    stamps.record(2, st);
    launch_pdl(merge_kernel, dim3(a.batch), dim3(MG_THREADS), 0, st, a.seg_off, a.kept_cnt, a.kept_key, a.C, a.off,
               a.ok, a.max_out, a.stage, a.keep, a.counts);
    stamps.record(3, st);
}

}  // namespace gbnms
