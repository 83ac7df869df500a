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
// GB300 shape: a CTA computes a tile of M_WARPS*64 rows x MT columns.  Each
// lane holds two row boxes in registers and walks the MT staged column boxes
// (broadcast shared-memory reads), so a row's words of the tile are built in
// registers and written with 16-byte stores.  The
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
#define GBNMS_MASK_WARPS 2
#endif
#ifndef GBNMS_MASK_UNROLL
#define GBNMS_MASK_UNROLL 2
#endif
namespace gbnms {
constexpr int kMaskUnroll = GBNMS_MASK_UNROLL;  // unroll of the inner loop (4 columns per step)
}

namespace gbnms {

constexpr int MT = GBNMS_MASK_MT;  // tile width (columns)
constexpr int NQ = MT / 64;        // 64-bit words of a row per tile
static_assert(MT == MASK_TILE_W, "the tile width the host stages by");
static_assert(NQ == 1 || NQ == 2 || NQ == 4, "tile width of 64, 128 or 256 columns");
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
static_assert(MT % MR == 0, "a column tile spans a whole number of row tiles");

// Sign bit of RN(k*s - a): set iff the exact k*s - a is negative, i.e.
// a > k*s (the product inside a fused multiply-add is not rounded).
__device__ __forceinline__ uint32_t sign_above(float k, float s, float a)
{
    return __float_as_uint(__fmaf_rn(k, s, -a));
}

// One pair of the division-free test, shifted into the accumulators: `yes`
// takes the decision bit and `maybe` the "not surely below" bit.  For
// well-formed boxes and the constants of ThrParams, a > k_hi*s proves
// suppression and a <= k_lo*s proves no suppression (common.cuh); a pair with
// maybe and not yes is left to the exact division.  The test runs on doubled
// values: w + |w| = 2 max(w, 0) exactly, so a2 = (w + |w|) h = 2 a with h
// unclamped (when h <= 0 the product is <= 0 and both tests say no, as the
// canonical clamped intersection 0 would), compared against the doubled
// constants khi2 = 2 k_hi and klo2 = 2 k_lo.  Doubling is exact here: well-
// formed areas are at most 2^58, and an intersection small enough to round
// differently (below 2^-125) is far below k_lo * s >= 2^-78 either way.
__device__ __forceinline__ void pair_fast(float4 r, float ar, float4 c, float ac, float khi2, float klo2,
                                          uint32_t& yes, uint32_t& maybe)
{
    const float w = __fsub_rn(fminf(r.z, c.z), fmaxf(r.x, c.x));
    const float w2 = __fadd_rn(w, fabsf(w));
    const float h = __fsub_rn(fminf(r.w, c.w), fmaxf(r.y, c.y));
    const float a2 = __fmul_rn(w2, h);
    const float s = __fadd_rn(ar, ac);
    yes = __funnelshift_l(sign_above(khi2, s, a2), yes, 1);
    maybe = __funnelshift_l(sign_above(klo2, s, a2), maybe, 1);
}

// Both rows of a lane against 32 staged columns (cb, ca 16-byte aligned),
// highest column first so that bit k ends up meaning column k; one shared
// load of a column box feeds both rows, one 16-byte load brings 4 areas.
__device__ __forceinline__ void half_fast(const float4* __restrict__ cb, const float* __restrict__ ca,
                                          float4 r0, float ar0, float4 r1, float ar1, float khi2,
                                          float klo2, uint32_t& y0, uint32_t& m0, uint32_t& y1,
                                          uint32_t& m1)
{
    const float4* ca4 = reinterpret_cast<const float4*>(ca);
#pragma unroll kMaskUnroll
    for (int g = 7; g >= 0; --g) {
        const float4 a4 = ca4[g];
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int e = 3; e >= 0; --e) {
            const float4 c = cb[4 * g + e];
            pair_fast(r0, ar0, c, av[e], khi2, klo2, y0, m0);
            pair_fast(r1, ar1, c, av[e], khi2, klo2, y1, m1);
        }
    }
}

template <bool FAST>
__device__ __forceinline__ void tile_rows(const float4* __restrict__ cbox, const float* __restrict__ carea,
                                          float4 r0, float ar0, float4 r1, float ar1,
                                          const ThrParams& p, uint64_t (&w0)[NQ], uint64_t (&w1)[NQ],
                                          bool& unsure)
{
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        uint32_t lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
        if (FAST) {
            uint32_t ml0 = 0, mh0 = 0, ml1 = 0, mh1 = 0;
            const float khi2 = __fmul_rn(2.0f, p.k_hi), klo2 = __fmul_rn(2.0f, p.k_lo);
            half_fast(cbox + q * 64, carea + q * 64, r0, ar0, r1, ar1, khi2, klo2, lo0, ml0, lo1, ml1);
            half_fast(cbox + q * 64 + 32, carea + q * 64 + 32, r0, ar0, r1, ar1, khi2, klo2, hi0, mh0,
                      hi1, mh1);
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
__device__ __forceinline__ void clip_words(uint64_t (&w)[NQ], int i, int cb, int n)
{
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
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

// Append the set bits of row i's words at column base cb as packed
// (i << 16 | j) pairs.
__device__ __forceinline__ uint32_t* emit_row(uint32_t* dst, const uint64_t (&w)[NQ], int i, int cb)
{
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        uint64_t x = w[q];
        while (x) {
            const int b = __ffsll(static_cast<long long>(x)) - 1;
            x &= x - 1;
            *dst++ = (static_cast<uint32_t>(i) << 16) | static_cast<uint32_t>(cb + 64 * q + b);
        }
    }
    return dst;
}

__device__ __forceinline__ int popc_words(const uint64_t (&w)[NQ])
{
    int c = 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) c += __popcll(w[q]);
    return c;
}

__device__ __forceinline__ uint64_t or_words(const uint64_t (&w)[NQ])
{
    uint64_t v = 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) v |= w[q];
    return v;
}

// Row i's words of the tile: 16-byte stores (one 8-byte store for one word).
__device__ __forceinline__ void store_words(uint64_t* dst, const uint64_t (&w)[NQ])
{
    if constexpr (NQ == 1) {
        dst[0] = w[0];
    } else {
#pragma unroll
        for (int q = 0; q < NQ; q += 2) reinterpret_cast<ulonglong2*>(dst)[q / 2] = make_ulonglong2(w[q], w[q + 1]);
    }
}

__global__ void __launch_bounds__(M_THREADS)
iou_mask_kernel(const float4* __restrict__ boxes_s, const int* __restrict__ m_dev, int m_bound,
                ThrParams p, uint64_t* __restrict__ mask, int64_t ldw,
                unsigned long long* __restrict__ rowbits, int NB, ulonglong2* __restrict__ band,
                uint32_t* __restrict__ edges, unsigned* __restrict__ ecount, unsigned ecap,
                unsigned long long* __restrict__ haspred, int limit, long long tile_off,
                const int* __restrict__ done)
{
    __shared__ float4 cbox[MT];
    __shared__ __align__(16) float carea[MT];

    if (done && *done) return;  // an earlier stage already reached max_out
    const int n = min(m_dev ? *m_dev : m_bound, limit);
    int a, c;
    tri_coords(blockIdx.x + tile_off, a, c);
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

    uint64_t w0[NQ], w1[NQ];
    bool unsure = false;
    if (fast) {
        tile_rows<true>(cbox, carea, r0, ar0, r1, ar1, p, w0, w1, unsure);
        if (__any_sync(FULL, unsure)) {
            uint64_t e0[NQ], e1[NQ];
            bool dummy = false;
            if (unsure) {
                tile_rows<false>(cbox, carea, r0, ar0, r1, ar1, p, e0, e1, dummy);
#pragma unroll
                for (int q = 0; q < NQ; ++q) { w0[q] = e0[q]; w1[q] = e1[q]; }
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
        for (int q = 0; q < NQ; ++q) {
            const int C = cb / 64 + q;
            const int d = C - R;
            if (d < 0 || d > BAND_L || C >= T64) continue;  // warp-uniform
            uint64_t colA = w0[q], colB = w1[q];
            transpose64(colA, colB);
            band[(static_cast<int64_t>(C) * (BAND_L + 1) + d) * 32 + l] = make_ulonglong2(colA, colB);
        }
    }
    const int64_t wcol = cb / 64;
    const int chunk = cb >> 8;  // 256-column chunk of the per-row bitmap
    if (i0 < n) {
        if (mask) store_words(mask + static_cast<int64_t>(i0) * ldw + wcol, w0);
        if (rowbits && or_words(w0))
            atomicOr(rowbits + static_cast<int64_t>(i0) * NB + (chunk >> 6), 1ull << (chunk & 63));
    }
    if (i1 < n) {
        if (mask) store_words(mask + static_cast<int64_t>(i1) * ldw + wcol, w1);
        if (rowbits && or_words(w1))
            atomicOr(rowbits + static_cast<int64_t>(i1) * NB + (chunk >> 6), 1ull << (chunk & 63));
    }
    // Boxes with at least one earlier box over the threshold: the OR of the
    // warp's rows, one atomic per non-zero 64-column word.
    if (haspred) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
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
        const int cnt = (i0 < n ? popc_words(w0) : 0) + (i1 < n ? popc_words(w1) : 0);
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
                     cudaStream_t st, int col_lo, int col_hi, const int* done)
{
    // The triangle's tiles whose columns lie in [col_lo, col_hi) (multiples of
    // the tile width, or col_hi = m_bound), all rows above them.
    const int hi = min(col_hi, m_bound);
    const int64_t t0 = mask_tiles(col_lo), t1 = mask_tiles(hi);
    const int64_t tiles = t1 - t0;
    if (tiles <= 0) return;
    iou_mask_kernel<<<static_cast<unsigned>(tiles), M_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, p,
                                                                        mask, ldw,
                                                                        reinterpret_cast<unsigned long long*>(rowbits), NB,
                                                                        reinterpret_cast<ulonglong2*>(band),
                                                                        edges, ecount, ecap,
                                                                        reinterpret_cast<unsigned long long*>(haspred),
                                                                        hi, t0, done);
}

}  // namespace gbnms
