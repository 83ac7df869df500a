// Shared device helpers of the gbnms CUDA library.
//
// Box arithmetic follows one fixed binary32 operation order (the IoU
// definition in include/gbnms.h); every step is an explicit round-to-nearest
// intrinsic so no compiler flag can contract or reorder it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gbnms.h"

namespace gbnms {

constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------ score order key
//
// 32-bit key whose ascending order is the greedy visiting order ("NMS
// CUDA代码学习", section 算法与数据流: descending score, stable): -0 maps to
// +0, NaN maps to the largest key, ties are left to the index.
__host__ __device__ __forceinline__ uint32_t score_key(float s)
{
    if (s != s) return 0xffffffffu;            // NaN: after everything
    if (s == 0.0f) s = 0.0f;                   // -0 == +0
    uint32_t u;
#ifdef __CUDA_ARCH__
    u = __float_as_uint(s);
#else
    __builtin_memcpy(&u, &s, 4);
#endif
    uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending score
    uint32_t k = ~asc;                                           // descending score
    return k == 0xffffffffu ? 0xfffffffeu : k;                   // keep NaN strictly last
}

// 64-bit composite (score key, index): unique, ascending = visiting order.
__host__ __device__ __forceinline__ uint64_t order_key(float s, uint32_t idx)
{
    return (static_cast<uint64_t>(score_key(s)) << 32) | idx;
}

// ------------------------------------------------------------------- geometry

__device__ __forceinline__ float box_area(float4 b)
{
    return __fmul_rn(__fsub_rn(b.z, b.x), __fsub_rn(b.w, b.y));
}

// Canonical IoU, exactly the binary32 operation order of the definition.
__device__ __forceinline__ float iou_exact(float4 a, float area_a, float4 b, float area_b)
{
    float xx1 = fmaxf(a.x, b.x);
    float yy1 = fmaxf(a.y, b.y);
    float xx2 = fminf(a.z, b.z);
    float yy2 = fminf(a.w, b.w);
    float w = fmaxf(__fsub_rn(xx2, xx1), 0.0f);
    float h = fmaxf(__fsub_rn(yy2, yy1), 0.0f);
    float inter = __fmul_rn(w, h);
    float uni = __fsub_rn(__fadd_rn(area_a, area_b), inter);
    return __fdiv_rn(inter, uni);
}

__device__ __forceinline__ bool suppress_exact(float4 a, float area_a, float4 b, float area_b,
                                               float thr)
{
    return iou_exact(a, area_a, b, area_b) > thr;
}

// A box whose pairs may take the division-free test: finite coordinates,
// x2 >= x1, y2 >= y1, area in [2^-58, 2^58].  For two such boxes the union
// lies in [2^-59, 2^60], so every product in the test below is a normal
// binary32 number.
__device__ __forceinline__ bool well_formed(float4 b, float area)
{
    return b.z >= b.x && b.w >= b.y && area >= 0x1p-58f && area <= 0x1p58f &&
           fabsf(b.x) <= 0x1p100f && fabsf(b.y) <= 0x1p100f &&
           fabsf(b.z) <= 0x1p100f && fabsf(b.w) <= 0x1p100f;
}

// Threshold constant of the mask kernel's filter (computed on the host).
//   With s = area_a + area_b and a = inter as binary32 values, for well-formed
//   boxes and 2^-20 <= thr <= 2^20, and k_lo*s the exact real product:
//     a <= k_lo * s  implies  RN(a / RN(s - a)) <= thr   (no suppression)
//   so every suppressing pair has a > k_lo * s.
//   Proof sketch: q = a/(s-a) and the two roundings put the canonical IoU in
//   q(1 +- 2^-23); q <= T1 = thr(1-2^-21) <=> a <= s T1/(1+T1), and k_lo is
//   below that ratio by a factor 1-2^-22, so the rounded IoU cannot exceed thr.
//   The mask filter scales each box's area by k2 = 2 k_lo (1-2^-20), rounded
//   down, once per box, and its proof (iou_mask) spends the 2^-20 on the
//   roundings of those products.
struct ThrParams {
    float thr;     // the binary32 threshold
    float k_lo;    // <= (T1/(1+T1)) (1-2^-22), T1 = thr (1-2^-21)
    float k2;      // <= 2 k_lo (1-2^-20)
    int fast_ok;   // thr within [2^-20, 2^20]
};

// ------------------------------------------------------------- warp helpers

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// The lowest `k` set bits of `x` (k >= 0): binary search on prefix popcounts.
__device__ __forceinline__ uint64_t lowest_bits(uint64_t x, int k)
{
    if (k <= 0) return 0;
    if (k >= __popcll(x)) return x;
    int lo = 0, hi = 63;  // smallest p with popc(x & bits[0..p]) >= k
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__popcll(x & ((2ull << mid) - 1ull)) >= k) hi = mid; else lo = mid + 1;
    }
    return x & ((2ull << lo) - 1ull);  // lo < 63 here since k < popc(x)
}

__device__ __forceinline__ uint64_t ballot64(bool lo, bool hi)
{
    return static_cast<uint64_t>(__ballot_sync(FULL, lo)) |
           (static_cast<uint64_t>(__ballot_sync(FULL, hi)) << 32);
}

// Transpose of a 64x64 bit matrix spread over a warp: lane l holds rows l
// (a) and l+32 (b), bit c of a row meaning column c; afterwards lane l holds
// columns l and l+32 the same way (bit r meaning row r).  Recursive block
// swap: at step j the j x j blocks (rows with bit j clear, columns with bit j
// set) and (rows with bit j set, columns with bit j clear) trade places.
// j = 32 pairs a lane's own two rows; a smaller j pairs lane l with l ^ j.
__device__ __forceinline__ void transpose64(uint64_t& a, uint64_t& b)
{
    const uint64_t t = ((a >> 32) ^ b) & 0x00000000ffffffffull;
    b ^= t;
    a ^= t << 32;
    const unsigned l = lane_id();
    constexpr uint64_t kMask[5] = {0x0000ffff0000ffffull, 0x00ff00ff00ff00ffull, 0x0f0f0f0f0f0f0f0full,
                                   0x3333333333333333ull, 0x5555555555555555ull};
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int j = 16 >> s;
        const uint64_t m = kMask[s];
        const uint64_t pa = __shfl_xor_sync(FULL, a, j), pb = __shfl_xor_sync(FULL, b, j);
        if (l & j) {  // second row of the pair: takes the first row's high block
            a ^= ((pa >> j) ^ a) & m;
            b ^= ((pb >> j) ^ b) & m;
        } else {      // first row: takes the second row's low block
            a ^= (((a >> j) ^ pa) & m) << j;
            b ^= (((b >> j) ^ pb) & m) << j;
        }
    }
}

// Column-view tile resolve.  Lane l holds ca = C[l] and cb = C[l+32], where
// bit k of C[b] is set iff box k (k < b) of the tile suppresses box b.
// `cand` holds the tile's boxes no earlier kept box removed.  Each round, a
// candidate with a kept suppressor is removed and a candidate with no
// undecided or kept suppressor is kept; both tests are lane-local and two
// ballots publish them.  The lowest undecided box is always decided, so the
// loop ends (after a few rounds in practice, 64 at most).
__device__ __forceinline__ uint64_t resolve_tile_col(uint64_t cand, uint64_t ca, uint64_t cb)
{
    const unsigned l = lane_id();
    uint64_t kept = 0, und = cand;
    while (und) {
        const bool ua = (und >> l) & 1ull, ub = (und >> (l + 32)) & 1ull;
        const bool ra = ua && (ca & kept), rb = ub && (cb & kept);
        const bool sa = ua && !ra && !(ca & und), sb = ub && !rb && !(cb & und);
        const uint64_t rem = ballot64(ra, rb), safe = ballot64(sa, sb);
        und &= ~(rem | safe);
        kept |= safe;
    }
    return kept;
}

// Tiles below the diagonal whose 64x64 blocks the walk reads in column view
// (block (row tile C-d, column tile C) for d = 0..BAND_L).
constexpr int BAND_L = 16;

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may be scheduled while its predecessor in
// the stream still runs; it must wait here before reading what the
// predecessor writes (a no-op for an ordinary launch).  The predecessor lets
// it be scheduled early with pdl_release().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void set_status(int32_t* status, int code)
{
    atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

}  // namespace gbnms
