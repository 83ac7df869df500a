// Greedy NMS of lane candidates ("nms_kernel.cu 파일 분석 -2"): the page's
// candidate holds PROP_SIZE = 77 values, candidates are compared in score
// order through the sorted index, in 64-candidate tiles above the diagonal
// (sections row_start/col_start and 중복 비교 제거), and the comparison is
// symmetric, by absolute values, against a similarity threshold.  The page
// stops before the comparison; the reading (include/gbnms.h, nms_lane_run):
// two class scores, start row, start x, length and the x of 72 rows; a lane
// covers rows [floor(start), floor(start) + floor(length)) within [0, 72);
// the distance is the binary32 sum of |dx| over the common rows, lowest row
// first, over their number; a later lane goes when it is below the
// threshold.
//
// GB300 shape:
//   gather: the sorted lanes' x as 72 rows of n floats (row-major, so a
//           warp's lanes are contiguous), NaN in the rows a lane does not
//           cover, its row span, and a flag for a lane with a non-finite x
//           in a covered row; 32 lanes a CTA, transposed through shared
//           memory;
//   mask:   one CTA of 256 threads per run of 64 x 64 tiles along a row of
//           tiles of the upper triangle; thread (q, r) holds row lane r's 72
//           x in registers and takes 16 of each tile's 64 column lanes
//           (staged in shared memory row by row, the next tile by cp.async
//           while this one is compared) -- per row and pair of columns one
//           packed add, two maxes and one packed add:
//             acc += max(|x_c + (-x_r)|, 0)
//           (|x_c - x_r| = |x_r - x_c| exactly: binary32 subtraction is
//           antisymmetric)
//           max(NaN, 0) is 0, so a row either lane does not cover adds +0,
//           which leaves a non-negative sum unchanged: the sum is the
//           definition's sum over the common rows in row order.  Pairs with
//           a flagged lane take the definition's loop over the common rows
//           on the original values instead.  The words, the per-row chunk
//           bits, the neighbour bitmap and the pair list come out in the
//           layout of the box mask kernel, so the resolve is the same;
//   resolve: lane lists are dense cliques, so passes 0 and 1 of the graph
//           rounds run on all SMs first (launch_graph_prepass), then
//           launch_resolve_single (rounds over the pairs they leave, or the
//           walk).
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int LN_VALUES = NMS_LANE_VALUES;  // values of one candidate
constexpr int LN_ROWS = NMS_LANE_ROWS;      // x samples of one candidate
constexpr int LN_X0 = 5;                    // index of the first x sample
constexpr int LN_TILE = 64;                 // rows and columns of a mask tile
constexpr int LN_THREADS = 256;             // 64 row lanes x 4 column quarters
constexpr int LN_QCOLS = LN_TILE / (LN_THREADS / LN_TILE);  // column lanes per thread (16)
static_assert(LN_ROWS < 256, "a span packs two row indices into bytes");

// Row span [lo, hi) of a candidate, packed as lo | hi << 8 (0 for none).
__device__ __forceinline__ uint32_t lane_span(const float* __restrict__ p)
{
    const float s = p[2], l = p[4];
    if (!(s >= -1048576.0f && s <= 1048576.0f && l >= -1048576.0f && l <= 1048576.0f)) return 0u;
    int a = static_cast<int>(floorf(s));
    int b = a + static_cast<int>(floorf(l));
    a = max(a, 0);
    b = min(b, LN_ROWS);
    return b > a ? static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 8) : 0u;
}

// The definition's distance, row by row over the common rows, on the
// original values (pairs with a non-finite x in a covered row).
__device__ float lane_distance_exact(const float* __restrict__ a, const float* __restrict__ b, uint32_t sa,
                                     uint32_t sb)
{
    const int lo = max(static_cast<int>(sa & 255u), static_cast<int>(sb & 255u));
    const int hi = min(static_cast<int>(sa >> 8), static_cast<int>(sb >> 8));
    if (hi <= lo) return __int_as_float(0x7f800000);  // +inf: no common row
    float sum = 0.0f;
    for (int k = lo; k < hi; ++k) sum = __fadd_rn(sum, fabsf(__fsub_rn(a[LN_X0 + k], b[LN_X0 + k])));
    return __fdiv_rn(sum, static_cast<float>(hi - lo));
}

// Sorted lanes to the mask kernel's layout: xs[k * ld + p] = x_k of the lane
// at sorted position p (NaN where it does not cover row k), span[p], and
// flag[p] = 1 when a covered row holds a non-finite x.  A CTA takes 32 sorted
// lanes: its warps copy the lanes' 77-value records into shared memory
// (contiguous loads; the odd record length keeps the transposed reads
// conflict-free), then warp w writes rows w, w + 8, ... of all 32 lanes
// (128-byte stores).  Also zeroes z16 16-byte words at zero and the word
// *zcount (the graph prepass's state).
constexpr int LG_LANES = 32;
constexpr int LG_THREADS = 256;
static_assert(LN_TILE % LG_LANES == 0, "ld, a multiple of the tile, is a multiple of a CTA's lanes");
__global__ void __launch_bounds__(LG_THREADS)
lane_gather_kernel(const float* __restrict__ props, const int* __restrict__ perm, int n, int ld,
                   float* __restrict__ xs, uint32_t* __restrict__ span, uint32_t* __restrict__ flag,
                   uint4* __restrict__ zero, int z16, unsigned* __restrict__ zcount)
{
    __shared__ float rec[LG_LANES][LN_VALUES];
    __shared__ uint32_t bad_s[LG_LANES];
    static_assert(LN_VALUES % 2 == 1, "an odd record length spreads a column over the banks");
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x, warp = tid >> 5, l = tid & 31;
    const int g = blockIdx.x * LG_THREADS + tid;
    for (int q = g; q < z16; q += gridDim.x * LG_THREADS) zero[q] = make_uint4(0u, 0u, 0u, 0u);
    if (g == 0 && zcount) *zcount = 0u;
    const int p0 = blockIdx.x * LG_LANES;
    // Warp w stages lanes w, w + 8, w + 16, w + 24: their four perm loads,
    // then all their record loads, are in flight together.
    constexpr int RPW = LG_LANES / (LG_THREADS / 32);  // records a warp stages
    constexpr int CPR = (LN_VALUES + 31) / 32;          // loads a lane per record
    int src[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + i * (LG_THREADS / 32);
        src[i] = p0 + r < n ? perm[p0 + r] : -1;
    }
    float v[RPW][CPR];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int c = 0; c < CPR; ++c) {
            const int col = l + 32 * c;
            v[i][c] = src[i] >= 0 && col < LN_VALUES ? props[static_cast<int64_t>(src[i]) * LN_VALUES + col] : 0.0f;
        }
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int c = 0; c < CPR; ++c) {
            const int col = l + 32 * c;
            if (src[i] >= 0 && col < LN_VALUES) rec[warp + i * (LG_THREADS / 32)][col] = v[i][c];
        }
    if (tid < LG_LANES) bad_s[tid] = 0u;
    __syncthreads();
    const int p = p0 + l;  // < ld: the grid covers ld lanes exactly
    const bool real = p < n;
    const uint32_t sp = real ? lane_span(&rec[l][0]) : 0u;
    const int lo = static_cast<int>(sp & 255u), hi = static_cast<int>(sp >> 8);
    uint32_t bad = 0u;
    for (int k = warp; k < LN_ROWS; k += LG_THREADS / 32) {
        const bool cov = k >= lo && k < hi;  // never for a padding lane (sp = 0)
        const float x = cov ? rec[l][LN_X0 + k] : __int_as_float(0x7fc00000);
        if (cov && !(fabsf(x) <= 3.4028235e38f)) bad = 1u;
        xs[static_cast<int64_t>(k) * ld + p] = x;
    }
    if (bad) atomicOr(&bad_s[l], 1u);
    __syncthreads();
    if (warp == 0) {
        span[p] = sp;
        flag[p] = bad_s[l];
    }
}

// Row tile a and column tiles [c0, c1) of CTA b: each row of tiles of the
// upper triangle (column tiles a .. T-1) is cut into runs of K tiles, rows in
// order.
__device__ __forceinline__ void lane_run(int b, int T, int K, int& a, int& c0, int& c1)
{
    int left = b;
    for (a = 0; a < T - 1; ++a) {
        const int m = (T - a + K - 1) / K;
        if (left < m) break;
        left -= m;
    }
    c0 = a + left * K;
    c1 = min(T, c0 + K);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                     static_cast<unsigned>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// One CTA per run of K column tiles of one row tile: the row lanes' x stay
// in registers for the run, and the next column tile (its 72 x 64 x, spans
// and flags) is copied into the other half of a double buffer by 16-byte
// cp.async while the current one is compared.
__global__ void __launch_bounds__(LN_THREADS, 2)
lane_mask_kernel(const float* __restrict__ xs, const uint32_t* __restrict__ span,
                 const uint32_t* __restrict__ flag, const float* __restrict__ props, const int* __restrict__ perm,
                 int n, int ld, int K, float thr, uint64_t* __restrict__ mask, int64_t ldw,
                 unsigned long long* __restrict__ rowbits, int NB, uint32_t* __restrict__ edges,
                 unsigned* __restrict__ ecount, unsigned ecap, unsigned long long* __restrict__ haspred)
{
    __shared__ __align__(16) float s_x[2][LN_ROWS][LN_TILE];  // x of the column lanes, row by row
    __shared__ __align__(16) uint32_t s_span[2][LN_TILE];
    __shared__ __align__(16) uint32_t s_flag[2][LN_TILE];
    __shared__ uint16_t s_piece[LN_TILE][LN_THREADS / LN_TILE];
    __shared__ unsigned long long s_or[2];
    __shared__ int s_cnt[2];
    __shared__ int s_total;
    __shared__ unsigned s_base;

    pdl_wait();  // the gather has finished
    pdl_release();
    const int T = ld / LN_TILE;
    int ta, cA, cB;
    lane_run(blockIdx.x, T, K, ta, cA, cB);
    const int t = threadIdx.x;
    const int r = t & (LN_TILE - 1), q = t / LN_TILE;
    const int rbase = ta * LN_TILE;
    // Column tile c into half h of the buffer (one commit group).
    auto stage = [&](int h, int c) {
        const int cb = c * LN_TILE;
        for (int e = t; e < LN_ROWS * (LN_TILE / 4); e += LN_THREADS) {
            const int k = e / (LN_TILE / 4), v = 4 * (e % (LN_TILE / 4));
            cp_async16(&s_x[h][k][v], xs + static_cast<int64_t>(k) * ld + cb + v);
        }
        if (t < LN_TILE / 4)
            cp_async16(&s_span[h][4 * t], span + cb + 4 * t);
        else if (t < LN_TILE / 2)
            cp_async16(&s_flag[h][4 * t - LN_TILE], flag + cb + 4 * t - LN_TILE);
        cp_async_commit();
    };
    if (cA < cB) stage(0, cA);
    const int i = rbase + r;
    float nxr[LN_ROWS];  // the row lane's x, negated (NaN stays NaN)
#pragma unroll
    for (int k = 0; k < LN_ROWS; ++k) nxr[k] = -xs[static_cast<int64_t>(k) * ld + i];
    const uint32_t sr = span[i];
    const uint32_t fr = flag[i];
#pragma unroll 1
    for (int tc = cA; tc < cB; ++tc) {
        const int h = (tc - cA) & 1;
        if (tc + 1 < cB) {
            stage(h ^ 1, tc + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int cbase = tc * LN_TILE;
        uint32_t bits = 0u;
        const int c0 = q * LN_QCOLS;
#pragma unroll 1
        for (int g = 0; g < LN_QCOLS; g += 4) {
            float2 a01 = make_float2(0.0f, 0.0f), a23 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < LN_ROWS; ++k) {
                const float4 xc = *reinterpret_cast<const float4*>(&s_x[h][k][c0 + g]);
                const float2 nr = make_float2(nxr[k], nxr[k]);
                const float2 d01 = __fadd2_rn(make_float2(xc.x, xc.y), nr);  // x_c - x_r, two lanes
                const float2 d23 = __fadd2_rn(make_float2(xc.z, xc.w), nr);
                a01 = __fadd2_rn(a01, make_float2(fmaxf(fabsf(d01.x), 0.0f), fmaxf(fabsf(d01.y), 0.0f)));
                a23 = __fadd2_rn(a23, make_float2(fmaxf(fabsf(d23.x), 0.0f), fmaxf(fabsf(d23.y), 0.0f)));
            }
            const float acc[4] = {a01.x, a01.y, a23.x, a23.y};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int cl = c0 + g + u, j = cbase + cl;
                if (j <= i || j >= n || i >= n) continue;  // the upper triangle only
                const uint32_t sc = s_span[h][cl];
                const int lo = max(static_cast<int>(sr & 255u), static_cast<int>(sc & 255u));
                const int hi = min(static_cast<int>(sr >> 8), static_cast<int>(sc >> 8));
                if (hi <= lo) continue;  // no common row: +inf, never below the threshold
                float d;
                if (fr | s_flag[h][cl])
                    d = lane_distance_exact(props + static_cast<int64_t>(perm[i]) * LN_VALUES,
                                            props + static_cast<int64_t>(perm[j]) * LN_VALUES, sr, sc);
                else
                    d = __fdiv_rn(acc[u], static_cast<float>(hi - lo));
                if (d < thr) bits |= 1u << (g + u);
            }
        }
        s_piece[r][q] = static_cast<uint16_t>(bits);
        __syncthreads();
        // Threads 0..63 own the tile's rows: word, chunk bit, pair count.
        uint64_t w = 0;
        int cnt = 0;
        if (t < LN_TILE) {
#pragma unroll
            for (int k = 0; k < LN_THREADS / LN_TILE; ++k)
                w |= static_cast<uint64_t>(s_piece[t][k]) << (LN_QCOLS * k);
            const int row = rbase + t;
            if (row < n) {
                mask[static_cast<int64_t>(row) * ldw + tc] = w;
                if (w && rowbits) {
                    const int chunk = cbase >> 8;
                    atomicOr(rowbits + static_cast<int64_t>(row) * NB + (chunk >> 6), 1ull << (chunk & 63));
                }
            }
            cnt = __popcll(w);
            // Inclusive prefix of the counts within the warp.
            const unsigned l = lane_id();
            int x = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(FULL, x, d);
                if (static_cast<int>(l) >= d) x += y;
            }
            const unsigned long long o = __reduce_or_sync(FULL, static_cast<unsigned>(w)) |
                                         (static_cast<unsigned long long>(__reduce_or_sync(FULL,
                                              static_cast<unsigned>(w >> 32))) << 32);
            if (l == 31) {
                s_cnt[t >> 5] = x;
                s_or[t >> 5] = o;
            }
            cnt = x - cnt;  // exclusive prefix within the warp
        }
        __syncthreads();
        if (t == 0) {
            const unsigned long long o = s_or[0] | s_or[1];
            if (o && haspred) atomicOr(haspred + tc, o);
            const int total = s_cnt[0] + s_cnt[1];
            s_base = total && edges ? atomicAdd(ecount, static_cast<unsigned>(total)) : 0u;
            s_total = total;
        }
        __syncthreads();
        // The pair list: the tile's pairs land contiguously, row by row.  Past
        // the capacity the count still grows (the resolve then takes the walk)
        // and nothing is written.
        if (t < LN_TILE && edges && w) {
            const unsigned total = static_cast<unsigned>(s_total);
            const unsigned base = s_base;
            if (base <= ecap && total <= ecap - base) {
                uint32_t* dst = edges + base + cnt + (t >= 32 ? s_cnt[0] : 0);
                const uint32_t row = static_cast<uint32_t>(rbase + t);
                uint64_t x = w;
                while (x) {
                    const int b = __ffsll(static_cast<long long>(x)) - 1;
                    x &= x - 1;
                    *dst++ = (row << 16) | static_cast<uint32_t>(cbase + b);
                }
            }
        }
        __syncthreads();  // the buffer half and the tile's scratch are written again
    }
}

}  // namespace gbnms

namespace gbnms {

int lane_ld(int n) { return (n + LN_TILE - 1) / LN_TILE * LN_TILE; }

void launch_lane_mask(const float* props, const int* perm, int n, float thr, float* xs, uint32_t* span,
                      uint32_t* flag, uint64_t* mask, int64_t ldw, uint64_t* rowbits, int NB, uint32_t* edges,
                      unsigned* ecount, unsigned ecap, uint64_t* haspred, cudaStream_t st, void* zero,
                      size_t zero_bytes, unsigned* zcount)
{
    if (n <= 0) return;
    const int ld = lane_ld(n);
    launch_pdl(lane_gather_kernel, dim3(ld / LG_LANES), dim3(LG_THREADS), 0, st, props, perm, n, ld, xs, span, flag,
               static_cast<uint4*>(zero), zero ? static_cast<int>(zero_bytes / 16) : 0, zcount);
    // Runs of K column tiles: about one wave of 2 CTAs per SM, K at most 8.
    const int T = ld / LN_TILE;
    const long long tiles = static_cast<long long>(T) * (T + 1) / 2;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long slots = 2ll * (sms > 0 ? sms : 1);
    const int K = static_cast<int>(std::min<long long>(8, std::max<long long>(1, (tiles + slots - 1) / slots)));
    int runs = 0;
    for (int a = 0; a < T; ++a) runs += (T - a + K - 1) / K;
    launch_pdl(lane_mask_kernel, dim3(runs), dim3(LN_THREADS), 0, st, xs,
               static_cast<const uint32_t*>(span), static_cast<const uint32_t*>(flag), props, perm, n, ld, K, thr, mask,
               ldw, reinterpret_cast<unsigned long long*>(rowbits), NB, edges, ecount, ecap,
               reinterpret_cast<unsigned long long*>(haspred));
}

}  // namespace gbnms
