// Upper-triangular IoU suppression bitmask of score-sorted boxes.
//
// "NMS CUDA代码学习", section Phase 1: only j > i can be suppressed by i, one
// IoU per pair, bit k of a word always means box (word base + k) so rows stay
// aligned (the j_base rule), and 32 IoUs fold into one word write with no
// atomics.  "nms_kernel.cu 파일 분석 -2", sections row_start/col_start and
// 중복 비교 제거: a 2-D tiling where tiles below the diagonal do no work, and
// the column tile is staged in shared memory.  "Fastest Matrix NMS in the West
// (Part 2)", section "Optimization 1: tile the IoU matrix": coordinates loaded
// once per tile and reused by every row.
//
// GB300 shape: a CTA computes a 128-row x 256-column tile.  Each lane holds two
// row boxes in registers and walks the 256 staged column boxes (broadcast
// shared-memory reads), so a row's four words of the tile (one 32-byte
// sector) are built in registers and written with two 16-byte stores.  The
// triangle of tiles is enumerated column by column.  Each row also records,
// one bit per 256-column chunk, which of its chunks hold a set bit, and the
// 64x64 blocks within BAND_L tiles of the diagonal are also written in column
// view; the resolve uses the first to skip all-zero chunks and the second to
// decide a tile with lane-local tests.  When asked, every set bit is also
// appended to a list of (row, column) pairs, the sparse form of the same
// graph, as long as the list has room, and every column with a set bit is
// marked in a bitmap of boxes that have an earlier neighbour.  Pairs are
// decided by the
// division-free test of common.cuh and, for the rare pair it leaves open and
// for tiles holding a malformed box, by the exact binary32 division.
#include "common.cuh"
#include "internal.h"

#ifndef GBNMS_MASK_WARPS
#define GBNMS_MASK_WARPS 4
#endif
#ifndef GBNMS_MASK_UNROLL
#define GBNMS_MASK_UNROLL 8
#endif
namespace gbnms {
constexpr int kMaskUnroll = GBNMS_MASK_UNROLL;  // unroll of the 32-column inner loop
}

namespace gbnms {

constexpr int MT = 256;         // tile width (columns)
constexpr int M_WARPS = GBNMS_MASK_WARPS;  // warps of 64 rows per tile
constexpr int MR = M_WARPS * 64;  // tile height (rows)
constexpr int M_THREADS = M_WARPS * 32;

// Far-away zero-area box used to pad ragged tiles: overlaps nothing.
__device__ __forceinline__ float4 pad_box() { return make_float4(3e38f, 3e38f, 3e38f, 3e38f); }

// Linear index k of the tile triangle -> (row tile a, column tile c).  With
// r = MT/MR row tiles per column tile, column tile c meets row tiles
// a = 0 .. r(c+1)-1, so the tiles of columns before c number r c(c+1)/2;
// enumeration is column by column.
__device__ __forceinline__ void tri_coords(long long k, int& a, int& c)
{
    constexpr long long r = MT / MR;
    long long cc = static_cast<long long>((sqrt(8.0 * static_cast<double>(k) / r + 1.0) - 1.0) * 0.5);
    while (r * (cc + 1) * (cc + 2) / 2 <= k) ++cc;
    while (r * cc * (cc + 1) / 2 > k) --cc;
    c = static_cast<int>(cc);
    a = static_cast<int>(k - r * cc * (cc + 1) / 2);
}
static_assert(MT == 2 * MR || MT == MR, "tri_coords handles column tiles one or two row tiles wide");

// Sign bit of RN(k*s - a): set iff the exact k*s - a is negative, i.e.
// a > k*s (the product inside a fused multiply-add is not rounded).
__device__ __forceinline__ uint32_t sign_above(float k, float s, float a)
{
    return __float_as_uint(__fmaf_rn(k, s, -a));
}

// One 32-column half of the division-free test for one row: shifts the
// decision bits into `yes` and the "not surely below" bits into `maybe`,
// highest column first, so bit k ends up meaning column k.  For well-formed
// boxes and the constants of ThrParams, a > k_hi*s proves suppression and
// a <= k_lo*s proves no suppression (common.cuh); a pair with maybe and not
// yes is left to the exact division.  The intersection is fmax(w,0)*h with h
// unclamped: when h <= 0 the product is <= 0 and both tests say no, as the
// canonical (clamped) intersection 0 would.
__device__ __forceinline__ void half_fast(const float4* __restrict__ cb, const float* __restrict__ ca,
                                          float4 r, float ar, float khi, float klo, uint32_t& yes,
                                          uint32_t& maybe)
{
#pragma unroll kMaskUnroll
    for (int k = 31; k >= 0; --k) {
        const float4 c = cb[k];
        const float w = fmaxf(__fsub_rn(fminf(r.z, c.z), fmaxf(r.x, c.x)), 0.0f);
        const float h = __fsub_rn(fminf(r.w, c.w), fmaxf(r.y, c.y));
        const float a = __fmul_rn(w, h);
        const float s = __fadd_rn(ar, ca[k]);
        yes = __funnelshift_l(sign_above(khi, s, a), yes, 1);
        maybe = __funnelshift_l(sign_above(klo, s, a), maybe, 1);
    }
}

template <bool FAST>
__device__ __forceinline__ void tile_rows(const float4* __restrict__ cbox, const float* __restrict__ carea,
                                          float4 r0, float ar0, float4 r1, float ar1,
                                          const ThrParams& p, uint64_t (&w0)[4], uint64_t (&w1)[4],
                                          bool& unsure)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
        if (FAST) {
            uint32_t ml0 = 0, mh0 = 0, ml1 = 0, mh1 = 0;
            half_fast(cbox + q * 64, carea + q * 64, r0, ar0, p.k_hi, p.k_lo, lo0, ml0);
            half_fast(cbox + q * 64, carea + q * 64, r1, ar1, p.k_hi, p.k_lo, lo1, ml1);
            half_fast(cbox + q * 64 + 32, carea + q * 64 + 32, r0, ar0, p.k_hi, p.k_lo, hi0, mh0);
            half_fast(cbox + q * 64 + 32, carea + q * 64 + 32, r1, ar1, p.k_hi, p.k_lo, hi1, mh1);
            unsure |= ((ml0 & ~lo0) | (mh0 & ~hi0) | (ml1 & ~lo1) | (mh1 & ~hi1)) != 0;
        } else {
#pragma unroll 8
            for (int k = 0; k < 32; ++k) {
                const float4 c = cbox[q * 64 + k];
                const float ac = carea[q * 64 + k];
                lo0 |= static_cast<uint32_t>(suppress_exact(r0, ar0, c, ac, p.thr)) << k;
                lo1 |= static_cast<uint32_t>(suppress_exact(r1, ar1, c, ac, p.thr)) << k;
            }
#pragma unroll 8
            for (int k = 0; k < 32; ++k) {
                const float4 c = cbox[q * 64 + 32 + k];
                const float ac = carea[q * 64 + 32 + k];
                hi0 |= static_cast<uint32_t>(suppress_exact(r0, ar0, c, ac, p.thr)) << k;
                hi1 |= static_cast<uint32_t>(suppress_exact(r1, ar1, c, ac, p.thr)) << k;
            }
        }
        w0[q] = (static_cast<uint64_t>(hi0) << 32) | lo0;
        w1[q] = (static_cast<uint64_t>(hi1) << 32) | lo1;
    }
}

// Keep only bits j with j > i and j < n of the four words at column base cb.
__device__ __forceinline__ void clip_words(uint64_t (&w)[4], int i, int cb, int n)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        int j0 = cb + 64 * q;
        uint64_t keep = ~0ull;
        int lo = i + 1 - j0;                    // first allowed bit
        if (lo >= 64) keep = 0;
        else if (lo > 0) keep &= ~0ull << lo;
        int hi = n - j0;                        // bits >= hi are beyond n
        if (hi <= 0) keep = 0;
        else if (hi < 64) keep &= (1ull << hi) - 1ull;
        w[q] &= keep;
    }
}

// Append the set bits of row i's four words at column base cb as packed
// (i << 16 | j) pairs.
__device__ __forceinline__ uint32_t* emit_row(uint32_t* dst, const uint64_t (&w)[4], int i, int cb)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint64_t x = w[q];
        while (x) {
            const int b = __ffsll(static_cast<long long>(x)) - 1;
            x &= x - 1;
            *dst++ = (static_cast<uint32_t>(i) << 16) | static_cast<uint32_t>(cb + 64 * q + b);
        }
    }
    return dst;
}

__device__ __forceinline__ int popc4(const uint64_t (&w)[4])
{
    return __popcll(w[0]) + __popcll(w[1]) + __popcll(w[2]) + __popcll(w[3]);
}

__global__ void __launch_bounds__(M_THREADS)
iou_mask_kernel(const float4* __restrict__ boxes_s, const int* __restrict__ m_dev, int m_bound,
                ThrParams p, uint64_t* __restrict__ mask, int64_t ldw,
                unsigned long long* __restrict__ rowbits, int NB, ulonglong2* __restrict__ band,
                uint32_t* __restrict__ edges, unsigned* __restrict__ ecount, unsigned ecap,
                unsigned long long* __restrict__ haspred)
{
    __shared__ float4 cbox[MT];
    __shared__ float carea[MT];

    const int n = m_dev ? *m_dev : m_bound;
    int a, c;
    tri_coords(blockIdx.x, a, c);
    const int T = (n + MT - 1) / MT;
    if (c >= T || a * MR >= n) return;  // beyond the device-side count

    const int cb = c * MT;
    const int rbase = a * MR;
    bool ok = true;
    for (int t = threadIdx.x; t < MT; t += M_THREADS) {
        int j = cb + t;
        float4 b = j < n ? boxes_s[j] : pad_box();
        float ar = j < n ? box_area(b) : 0.0f;
        if (j < n) ok &= well_formed(b, ar);
        cbox[t] = b;
        carea[t] = ar;
    }
    const unsigned l = lane_id();
    const int wp = threadIdx.x >> 5;
    const int i0 = rbase + wp * 64 + l;
    const int i1 = i0 + 32;
    float4 r0 = i0 < n ? boxes_s[i0] : pad_box();
    float4 r1 = i1 < n ? boxes_s[i1] : pad_box();
    float ar0 = i0 < n ? box_area(r0) : 0.0f;
    float ar1 = i1 < n ? box_area(r1) : 0.0f;
    if (i0 < n) ok &= well_formed(r0, ar0);
    if (i1 < n) ok &= well_formed(r1, ar1);
    const bool fast = __syncthreads_and(ok) && p.fast_ok;

    uint64_t w0[4], w1[4];
    bool unsure = false;
    if (fast) {
        tile_rows<true>(cbox, carea, r0, ar0, r1, ar1, p, w0, w1, unsure);
        if (__any_sync(FULL, unsure)) {
            uint64_t e0[4], e1[4];
            bool dummy = false;
            if (unsure) {
                tile_rows<false>(cbox, carea, r0, ar0, r1, ar1, p, e0, e1, dummy);
#pragma unroll
                for (int q = 0; q < 4; ++q) { w0[q] = e0[q]; w1[q] = e1[q]; }
            }
        }
    } else {
        tile_rows<false>(cbox, carea, r0, ar0, r1, ar1, p, w0, w1, unsure);
    }

    if (rbase + MR > cb) {  // the tile meets the diagonal
        clip_words(w0, i0, cb, n);
        clip_words(w1, i1, cb, n);
    } else {
        clip_words(w0, -1, cb, n);
        clip_words(w1, -1, cb, n);
    }
    // Column view of the blocks within BAND_L tiles of the diagonal (64-row
    // tile R of this warp, 64-column tile C = 4c+q): a warp transpose of the
    // block's final words leaves columns l and l+32 in lane l.
    if (band) {
        const int R = rbase / 64 + wp;
        const int T64 = (n + 63) / 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int C = 4 * c + q;
            const int d = C - R;
            if (d < 0 || d > BAND_L || C >= T64) continue;  // warp-uniform
            uint64_t colA = w0[q], colB = w1[q];
            transpose64(colA, colB);
            band[(static_cast<int64_t>(C) * (BAND_L + 1) + d) * 32 + l] = make_ulonglong2(colA, colB);
        }
    }
    const int64_t wcol = static_cast<int64_t>(c) * 4;
    if (i0 < n) {
        uint64_t* dst = mask + static_cast<int64_t>(i0) * ldw + wcol;
        reinterpret_cast<ulonglong2*>(dst)[0] = make_ulonglong2(w0[0], w0[1]);
        reinterpret_cast<ulonglong2*>(dst)[1] = make_ulonglong2(w0[2], w0[3]);
        if (rowbits && (w0[0] | w0[1] | w0[2] | w0[3]))
            atomicOr(rowbits + static_cast<int64_t>(i0) * NB + (c >> 6), 1ull << (c & 63));
    }
    if (i1 < n) {
        uint64_t* dst = mask + static_cast<int64_t>(i1) * ldw + wcol;
        reinterpret_cast<ulonglong2*>(dst)[0] = make_ulonglong2(w1[0], w1[1]);
        reinterpret_cast<ulonglong2*>(dst)[1] = make_ulonglong2(w1[2], w1[3]);
        if (rowbits && (w1[0] | w1[1] | w1[2] | w1[3]))
            atomicOr(rowbits + static_cast<int64_t>(i1) * NB + (c >> 6), 1ull << (c & 63));
    }
    // Boxes with at least one earlier box over the threshold: the OR of the
    // warp's rows, one atomic per non-zero 64-column word.
    if (haspred) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint64_t v = (i0 < n ? w0[q] : 0ull) | (i1 < n ? w1[q] : 0ull);
            const unsigned lo = __reduce_or_sync(FULL, static_cast<unsigned>(v));
            const unsigned hi = __reduce_or_sync(FULL, static_cast<unsigned>(v >> 32));
            if (static_cast<int>(l) == q && (lo | hi))
                atomicOr(haspred + (cb >> 6) + q, (static_cast<unsigned long long>(hi) << 32) | lo);
        }
    }
    // Sparse form: one counter reservation per warp with any set bit; the
    // pairs of a warp land contiguously, lane by lane.  Past the capacity the
    // count still grows (it tells the resolve the list is incomplete) and
    // nothing is written.
    if (edges) {
        const int cnt = (i0 < n ? popc4(w0) : 0) + (i1 < n ? popc4(w1) : 0);
        int x = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(FULL, x, d);
            if (static_cast<int>(l) >= d) x += y;
        }
        const int total = __shfl_sync(FULL, x, 31);
        if (total) {
            unsigned base = 0;
            if (l == 31) base = atomicAdd(ecount, static_cast<unsigned>(total));
            base = __shfl_sync(FULL, base, 31);
            if (base <= ecap && static_cast<unsigned>(total) <= ecap - base) {
                uint32_t* dst = edges + base + (x - cnt);
                if (i0 < n) dst = emit_row(dst, w0, i0, cb);
                if (i1 < n) emit_row(dst, w1, i1, cb);
            }
        }
    }
}

int64_t mask_tiles(int64_t n)
{
    int64_t T = (n + MT - 1) / MT;
    return (MT / MR) * T * (T + 1) / 2;
}

void launch_iou_mask(const float4* boxes_s, const int* m_dev, int m_bound, const ThrParams& p,
                     uint64_t* mask, int64_t ldw, uint64_t* rowbits, int NB, uint64_t* band,
                     uint32_t* edges, unsigned* ecount, unsigned ecap, uint64_t* haspred,
                     cudaStream_t st)
{
    int64_t tiles = mask_tiles(m_bound);
    if (tiles == 0) return;
    iou_mask_kernel<<<static_cast<unsigned>(tiles), M_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, p,
                                                                        mask, ldw,
                                                                        reinterpret_cast<unsigned long long*>(rowbits), NB,
                                                                        reinterpret_cast<ulonglong2*>(band),
                                                                        edges, ecount, ecap,
                                                                        reinterpret_cast<unsigned long long*>(haspred));
}

}  // namespace gbnms
