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
// GB300 shape: the triangle is cut into units of 64 rows x MT columns, each
// taken by one warp on its own (its column boxes staged in its own slice of
// shared memory, so no CTA barrier), enumerated column by column; warps
// stride over the units when the grid is smaller than the units.  Each lane holds two row boxes in
// registers and walks the MT staged column boxes (broadcast shared-memory
// reads of 4 columns at a time), so a row's words of the unit are built in
// registers and written with 16-byte stores.  Each row also records, one bit
// per 256-column chunk, which of its chunks hold a set bit (the walk skips
// all-zero chunks).  When asked, every set bit is also
// appended to a list of (row, column) pairs, the sparse form of the same
// graph, as long as the list has room, and every column with a set bit is
// marked in a bitmap of boxes that have an earlier neighbour.
//
// Deciding a pair takes two steps.  A filter, run on every pair, sets a
// "maybe" bit for a superset of the suppressing pairs: it bounds the
// intersection from above with packed two-column binary32 arithmetic (one
// instruction for two columns) and compares it against k_lo times the area
// sum, a comparison the canonical IoU > thr implies (see ThrParams), with the
// areas scaled once per box.  Only
// the maybe bits, a small fraction of the pairs, are then decided by the
// canonical IoU itself, so every stored bit is exactly the definition's.
// Tiles holding a malformed box, and thresholds outside the filter's range,
// send every pair of the tile to the canonical test.
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

#ifndef GBNMS_MASK_WARPS
#define GBNMS_MASK_WARPS 4
#endif
#ifndef GBNMS_MASK_ROWS
#define GBNMS_MASK_ROWS 2
#endif
#ifndef GBNMS_MASK_CTAS_PER_SM
#define GBNMS_MASK_CTAS_PER_SM 8
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
constexpr int M_WARPS = GBNMS_MASK_WARPS;  // warps per CTA, each on its own units
constexpr int RPL = GBNMS_MASK_ROWS;        // row boxes per lane
constexpr int UR = 32 * RPL;                // rows of a unit
static_assert(MT % UR == 0, "a column tile spans a whole number of row units");
constexpr int M_THREADS = M_WARPS * 32;
constexpr int M_CTAS_PER_SM = GBNMS_MASK_CTAS_PER_SM;  // resident CTAs per SM the grid is sized for

// Far-away zero-area box used to pad ragged tiles: overlaps nothing.
__device__ __forceinline__ float4 pad_box() { return make_float4(3e38f, 3e38f, 3e38f, 3e38f); }

// Linear index k of the unit triangle -> (UR-row tile a, MT-column tile c).
// Column tile c meets row tiles a = 0 .. r(c+1)-1 with r = MT/UR, so the
// units of columns before c number r c(c+1)/2; enumeration is column by
// column.
__device__ __forceinline__ void tri_coords(long long k, int& a, int& c)
{
    constexpr long long r = MT / UR;
    // A binary32 estimate (no binary64 on the hot path), made exact by the
    // integer corrections.
    long long cc = static_cast<long long>((sqrtf(8.0f * static_cast<float>(k) / r + 1.0f) - 1.0f) * 0.5f);
    if (cc < 0) cc = 0;
    while (r * (cc + 1) * (cc + 2) / 2 <= k) ++cc;
    while (cc > 0 && r * cc * (cc + 1) / 2 > k) --cc;
    c = static_cast<int>(cc);
    a = static_cast<int>(k - r * cc * (cc + 1) / 2);
}

// Column boxes of a tile in shared memory, one array per coordinate, with
// x1 and y2 negated so that every difference below is a sum.
struct ColsSoA {
    float* nx1;  // -x1
    float* x2;
    float* y1;
    float* ny2;  // -y2
    float* ka;   // RN(k2 * canonical area)
};

__device__ __forceinline__ float4 col_box(const ColsSoA& C, int t)
{
    return make_float4(-C.nx1[t], C.y1[t], C.x2[t], -C.ny2[t]);
}

// A row box spread over register pairs (both halves equal) for the packed
// instructions.
struct RowF2 {
    float2 z;   // (x2, x2)
    float2 nx;  // (-x1, -x1)
    float2 nw;  // (-y2, -y2)
    float2 y;   // (y1, y1)
    float2 ka;  // RN(k2 * area), twice
};

__device__ __forceinline__ float2 dup2(float v) { return make_float2(v, v); }

__device__ __forceinline__ RowF2 make_row(float4 b, float ka)
{
    RowF2 r;
    r.z = dup2(b.z);
    r.nx = dup2(-b.x);
    r.nw = dup2(-b.w);
    r.y = dup2(b.y);
    r.ka = dup2(ka);
    return r;
}

// The filter for one row and two adjacent columns, shifted into `acc`
// (second column first, so that bit k ends up meaning column k when the
// columns are walked from the highest down).
//   width bound  w' = min(RN(r.x2 - c.x1), RN(c.x2 - r.x1)) >= the canonical
//                w = RN(min(x2) - max(x1)) (both operands of each difference
//                are bounds and rounding is monotone); w2 = w' + |w'| =
//                2 max(w', 0)
//   height bound h' likewise, computed negated: -h' = max(RN(c.y1 - r.y2),
//                RN(r.y1 - c.y2))
//   maybe        RN(RN(w2 (-h') + kc) + kr) < 0, with kc = RN(k2 area_c),
//                kr = RN(k2 area_r) and k2 <= 2 k_lo (1 - 2^-20).
// Why every suppressing pair of well-formed boxes gets its bit: it has
// a = inter > k_lo s (ThrParams), w, h > 0 and so h' > 0.  With
// A = 2 k_lo (area_r + area_c) and u = 2^-24:
//   P = w2 h' >= 2 w h >= 2 a (1 - u) > 2 k_lo s (1 - u) >= A (1 - 2u),
//   kc + kr <= k2 (area_r + area_c)(1 + u) <= A (1 - 2^-20)(1 + u),
// so P - kc - kr > A (2^-20 - 3u) = 13 u A.  The first rounding, of
// kc - P < 0, moves it by at most u (P - kc), and kr <= A (1 + u), so
// t1 + kr < 0 still holds exactly and the second rounding keeps the sign
// (a negative sum rounds to a negative number or -0, both with the sign bit
// set).  A product past the binary32 range becomes -inf and sets the bit too.
// A negative h' gives a non-negative product and no bit, as the clamped
// canonical height 0 would give no suppression.
__device__ __forceinline__ void maybe2(const RowF2& r, float2 cnx1, float2 cx2, float2 cy1, float2 cny2, float2 ckc,
                                       uint32_t& acc)
{
    const float2 ax = __fadd2_rn(r.z, cnx1);  // r.x2 - c.x1
    const float2 bx = __fadd2_rn(cx2, r.nx);  // c.x2 - r.x1
    float2 w2;
    w2.x = fminf(ax.x, bx.x);
    w2.y = fminf(ax.y, bx.y);
    w2.x = __fadd_rn(w2.x, fabsf(w2.x));
    w2.y = __fadd_rn(w2.y, fabsf(w2.y));
    const float2 ay = __fadd2_rn(cy1, r.nw);  // c.y1 - r.y2
    const float2 by = __fadd2_rn(r.y, cny2);  // r.y1 - c.y2
    float2 nh;
    nh.x = fmaxf(ay.x, by.x);
    nh.y = fmaxf(ay.y, by.y);
    const float2 t = __fadd2_rn(__ffma2_rn(w2, nh, ckc), r.ka);
    acc = __funnelshift_l(__float_as_uint(t.y), acc, 1);
    acc = __funnelshift_l(__float_as_uint(t.x), acc, 1);
}

// The lane's RPL rows against 32 staged columns starting at `base` (a
// multiple of 4): one 16-byte shared load per coordinate brings 4 columns,
// shared by all the rows.
__device__ __forceinline__ void maybe_half(const ColsSoA& C, int base, const RowF2 (&r)[RPL], uint32_t (&m)[RPL])
{
#pragma unroll kMaskUnroll
    for (int g = 7; g >= 0; --g) {
        const int o = base + 4 * g;
        const float4 a = *reinterpret_cast<const float4*>(C.nx1 + o);
        const float4 b = *reinterpret_cast<const float4*>(C.x2 + o);
        const float4 c = *reinterpret_cast<const float4*>(C.y1 + o);
        const float4 d = *reinterpret_cast<const float4*>(C.ny2 + o);
        const float4 e = *reinterpret_cast<const float4*>(C.ka + o);
        const float2 ahi = make_float2(a.z, a.w), bhi = make_float2(b.z, b.w), chi = make_float2(c.z, c.w),
                     dhi = make_float2(d.z, d.w), ehi = make_float2(e.z, e.w);
        const float2 alo = make_float2(a.x, a.y), blo = make_float2(b.x, b.y), clo = make_float2(c.x, c.y),
                     dlo = make_float2(d.x, d.y), elo = make_float2(e.x, e.y);
#pragma unroll
        for (int k = 0; k < RPL; ++k) maybe2(r[k], ahi, bhi, chi, dhi, ehi, m[k]);
#pragma unroll
        for (int k = 0; k < RPL; ++k) maybe2(r[k], alo, blo, clo, dlo, elo, m[k]);
    }
}

// The maybe words of the lane's rows over the tile's NQ words.
__device__ __forceinline__ void maybe_rows(const ColsSoA& C, const RowF2 (&r)[RPL], uint64_t (&w)[RPL][NQ])
{
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        uint32_t lo[RPL], hi[RPL];
#pragma unroll
        for (int k = 0; k < RPL; ++k) lo[k] = hi[k] = 0;
        maybe_half(C, q * 64, r, lo);
        maybe_half(C, q * 64 + 32, r, hi);
#pragma unroll
        for (int k = 0; k < RPL; ++k) w[k][q] = (static_cast<uint64_t>(hi[k]) << 32) | lo[k];
    }
}

// Keeps the bits of `w` whose pair passes the canonical test.
__device__ __forceinline__ void verify_words(const ColsSoA& C, float4 b, float ar, float thr, uint64_t (&w)[NQ])
{
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        uint64_t x = w[q], keep = 0;
        while (x) {
            const int bit = __ffsll(static_cast<long long>(x)) - 1;
            x &= x - 1;
            const int t = 64 * q + bit;
            const float4 c = col_box(C, t);
            if (suppress_exact(b, ar, c, box_area(c), thr)) keep |= 1ull << bit;
        }
        w[q] = keep;
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

// The unit's outputs from its final words: the mask words, the per-row chunk
// bits, the neighbour bitmap and the pair list.
__device__ __forceinline__ void store_unit(const uint64_t (&w)[RPL][NQ], const int (&i)[RPL], int cb, int n,
                                           unsigned l, uint64_t* __restrict__ mask, int64_t ldw,
                                           unsigned long long* __restrict__ rowbits, int NB,
                                           uint32_t* __restrict__ edges, unsigned* __restrict__ ecount,
                                           unsigned ecap, unsigned long long* __restrict__ haspred)
{
    const int64_t wcol = cb / 64;
    const int chunk = cb >> 8;  // 256-column chunk of the per-row bitmap
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
        if (i[k] >= n) continue;
        if (mask) store_words(mask + static_cast<int64_t>(i[k]) * ldw + wcol, w[k]);
        if (rowbits && or_words(w[k]))
            atomicOr(rowbits + static_cast<int64_t>(i[k]) * NB + (chunk >> 6), 1ull << (chunk & 63));
    }
    // Boxes with at least one earlier box over the threshold: the OR of the
    // warp's rows, one atomic per non-zero 64-column word.
    if (haspred) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            uint64_t v = 0;
#pragma unroll
            for (int k = 0; k < RPL; ++k) v |= i[k] < n ? w[k][q] : 0ull;
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
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < RPL; ++k) cnt += i[k] < n ? popc_words(w[k]) : 0;
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
#pragma unroll
                for (int k = 0; k < RPL; ++k)
                    if (i[k] < n) dst = emit_row(dst, w[k], i[k], cb);
            }
        }
    }
}

__global__ void __launch_bounds__(M_THREADS, M_CTAS_PER_SM)
iou_mask_kernel(const float4* __restrict__ boxes_s, const int* __restrict__ m_dev, int m_bound,
                ThrParams p, uint64_t* __restrict__ mask, int64_t ldw,
                unsigned long long* __restrict__ rowbits, int NB,
                uint32_t* __restrict__ edges, unsigned* __restrict__ ecount, unsigned ecap,
                unsigned long long* __restrict__ haspred, int limit, long long u_begin, long long u_end,
                const int* __restrict__ done)
{
    __shared__ __align__(16) float s_cols[M_WARPS][5][MT];  // per warp: -x1, x2, y1, -y2, k2 area

    pdl_wait();     // the sort (or an earlier stage) has finished
    pdl_release();  // the resolve may be scheduled
    if (done && *done) return;  // an earlier stage already reached max_out
    const int n = min(m_dev ? *m_dev : m_bound, limit);
    const int T = (n + MT - 1) / MT;
    const unsigned l = lane_id();
    const int wp = threadIdx.x >> 5;
    const ColsSoA C{s_cols[wp][0], s_cols[wp][1], s_cols[wp][2], s_cols[wp][3], s_cols[wp][4]};
    const long long stride = static_cast<long long>(gridDim.x) * M_WARPS;
    for (long long u = u_begin + static_cast<long long>(blockIdx.x) * M_WARPS + wp; u < u_end; u += stride) {
        int a, c;
        tri_coords(u, a, c);
        if (c >= T || a * UR >= n) continue;  // beyond the device-side count (warp-uniform)
        const int cb = c * MT;
        const int rbase = a * UR;
        __syncwarp();  // the previous unit's reads of the staged columns are done
        bool ok = true;
#pragma unroll
        for (int t = static_cast<int>(l); t < MT; t += 32) {
            const int j = cb + t;
            const float4 b = j < n ? boxes_s[j] : pad_box();
            const float ar = j < n ? box_area(b) : 0.0f;
            if (j < n) ok &= well_formed(b, ar);
            C.nx1[t] = -b.x;
            C.x2[t] = b.z;
            C.y1[t] = b.y;
            C.ny2[t] = -b.w;
            C.ka[t] = __fmul_rn(p.k2, ar);
        }
        int i[RPL];
        float4 bx[RPL];
        float ar[RPL];
#pragma unroll
        for (int k = 0; k < RPL; ++k) {
            i[k] = rbase + static_cast<int>(l) + 32 * k;
            bx[k] = i[k] < n ? boxes_s[i[k]] : pad_box();
            ar[k] = i[k] < n ? box_area(bx[k]) : 0.0f;
            if (i[k] < n) ok &= well_formed(bx[k], ar[k]);
        }
        const bool fast = __all_sync(FULL, ok) && p.fast_ok;
        __syncwarp();  // the staged columns are visible to the whole warp

        uint64_t w[RPL][NQ];
        if (fast) {
            RowF2 r[RPL];
#pragma unroll
            for (int k = 0; k < RPL; ++k) r[k] = make_row(bx[k], __fmul_rn(p.k2, ar[k]));
            maybe_rows(C, r, w);
        } else {
#pragma unroll
            for (int k = 0; k < RPL; ++k)
#pragma unroll
                for (int q = 0; q < NQ; ++q) w[k][q] = ~0ull;
        }
        const bool diag = rbase + UR > cb;  // the unit meets the diagonal
#pragma unroll
        for (int k = 0; k < RPL; ++k) {
            if (diag) clip_words(w[k], i[k], cb, n);
            else if (cb + MT > n) clip_words(w[k], -1, cb, n);  // ragged last column tile
            if (i[k] >= n) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) w[k][q] = 0;
            }
            verify_words(C, bx[k], ar[k], p.thr, w[k]);
        }
        store_unit(w, i, cb, n, l, mask, ldw, rowbits, NB, edges, ecount, ecap, haspred);
    }
}

// Dynamic shared memory that holds the kernel to at most `cap` resident CTAs
// per SM (0 when the other limits already do), for the current device.
// Cached per (device, cap): the occupancy query runs once.
static size_t mask_smem_for_cap(int cap)
{
    static std::mutex mu;
    static std::map<std::pair<int, int>, size_t> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, cap});
    if (it != cache.end()) return it->second;
    int per_sm = 0, reserved = 0, optin = 0;
    cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, iou_mask_kernel);
    size_t dyn = 0;
    int blocks = 0;
    if (per_sm > 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, iou_mask_kernel, M_THREADS, 0) ==
                          cudaSuccess &&
        blocks > cap) {
        // The smallest CTA footprint (static + dynamic + reserved) of which
        // cap + 1 no longer fit, grown by 128 bytes until the query agrees.
        const long long need = static_cast<long long>(per_sm) / (cap + 1) + 1 - reserved -
                               static_cast<long long>(fa.sharedSizeBytes);
        dyn = need > 0 ? static_cast<size_t>(need) : 0;
        dyn = (dyn + 127) / 128 * 128;
        const size_t max_dyn = optin > static_cast<int>(fa.sharedSizeBytes) ? optin - fa.sharedSizeBytes : 0;
        for (int tries = 0; tries < 64 && dyn <= max_dyn; ++tries, dyn += 128) {
            ensure_dynamic_smem(reinterpret_cast<const void*>(iou_mask_kernel), dyn);
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, iou_mask_kernel, M_THREADS, dyn) !=
                cudaSuccess)
                break;
            if (blocks <= cap) break;
        }
        if (blocks > cap || dyn > max_dyn) dyn = 0;  // no footprint found: leave the placement to the hardware
        cudaGetLastError();
    }
    cache[{dev, cap}] = dyn;
    return dyn;
}

int64_t mask_tiles(int64_t n)
{
    int64_t T = (n + MT - 1) / MT;
    return (MT / UR) * T * (T + 1) / 2;
}

void launch_iou_mask(const float4* boxes_s, const int* m_dev, int m_bound, const ThrParams& p,
                     uint64_t* mask, int64_t ldw, uint64_t* rowbits, int NB,
                     uint32_t* edges, unsigned* ecount, unsigned ecap, uint64_t* haspred,
                     cudaStream_t st, int col_lo, int col_hi, const int* done)
{
    // The triangle's units whose columns lie in [col_lo, col_hi) (multiples of
    // the tile width, or col_hi = m_bound), all rows above them.
    const int hi = min(col_hi, m_bound);
    const int64_t u0 = mask_tiles(col_lo), u1 = mask_tiles(hi);
    if (u1 <= u0) return;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    // A unit per warp, the hardware balancing the CTAs; a launch that may find
    // its work already done (a later max_out stage) strides over the units
    // with one resident wave instead, so that finding the flag set costs a
    // few CTAs per SM.
    int64_t grid = (u1 - u0 + M_WARPS - 1) / M_WARPS;
    if (done) grid = min(grid, static_cast<int64_t>(sms) * M_CTAS_PER_SM);
    // A grid of one wave or less is held to ceil(grid / SMs) CTAs per SM.
    // The launch may be placed while the previous kernel still holds some
    // SMs (programmatic dependent launch); without the cap the free SMs
    // would take the full 8 CTAs each, finish last and set the kernel's time.
    size_t dyn = 0;
    const int64_t per_sm = (grid + sms - 1) / sms;
    if (!done && per_sm < M_CTAS_PER_SM) dyn = mask_smem_for_cap(static_cast<int>(per_sm));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(M_THREADS);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl_attr_count();
    cudaLaunchKernelEx(&cfg, iou_mask_kernel, boxes_s, m_dev, m_bound, p, mask, ldw,
                       reinterpret_cast<unsigned long long*>(rowbits), NB, edges, ecount, ecap,
                       reinterpret_cast<unsigned long long*>(haspred), hi, static_cast<long long>(u0),
                       static_cast<long long>(u1), done);
}

}  // namespace gbnms
