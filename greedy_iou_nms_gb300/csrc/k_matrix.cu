// Matrix NMS with Gaussian or linear decay, one image.
//
// "Fastest Matrix NMS in the West (Part 2)", section "What do we need to
// compute?": boxes sorted by score, O[i][j] the IoU of box j with its father
// i (i before j), O_max[i] the largest overlap of box i with its own fathers,
// decay exp((O_max[i]^2 - O[i][j]^2) / sigma), final score s'[j] = s[j] times
// the smallest decay over the fathers; section "Optimization 4": a box is
// dropped when its final score is below the threshold.
//
// The first box is a father of every other box and gives it a decay of at
// most 1; a father that does not overlap box j gives exp(O_max[i]^2 / sigma)
// >= 1.  So the smallest decay is min(1, smallest decay over the OVERLAPPING
// fathers), and only overlapping pairs (IoU > 0) need work.  Both passes walk
// the upper triangle in units of 64 rows x 128 columns, one warp per unit:
// a packed binary32 filter marks the pairs that may overlap (a superset, two
// columns per instruction), the warp queues those pairs in shared memory and
// takes them one per lane, and each unit folds its results per column in
// shared memory before one global atomic per column:
//   pass A: where two boxes overlap, the exact binary32 IoU, maxed into
//           O_max of the child;
//   pass B: for each overlapping pair the binary64 numerator
//           O_max[i]^2 - O[i][j]^2, minimised per child through an
//           order-preserving 64-bit key (dividing once per box by sigma > 0
//           afterwards gives the smallest quotient: correctly rounded
//           division by a positive number keeps the order); only pairs whose
//           binary32 bound can still be the column's minimum take the
//           binary64 value;
//   decide: per box (all SMs), s * exp(min(0, smallest exponent)) against
//           the threshold, decided in binary32 with expf when the result is
//           clear of the threshold by more than its error bound, in binary64
//           otherwise, into a kept bitmap and a final-score array;
//   emit:   the kept boxes in score order with their final scores.
//
// Linear decay (1 - O[i][j]) / (1 - O_max[i]): the same section of the page
// says the code holds a linear formula without printing it; this is the
// linear kernel with the same compensation.  A non-overlapping father gives
// 1 / (1 - O_max[i]) >= 1, so again only overlapping pairs count.  Pass B
// takes the binary64 quotient itself (a father with O_max = 1 gives x/0 or
// 0/0, which the minimum ignores), and the decide multiplies in binary64.

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace gbnms {

// Units of MU_ROWS rows x MU_COLS columns of the upper triangle, one per warp
// (columns staged in the warp's own slice of shared memory, no CTA barrier).
constexpr int MU_WARPS = 4;              // warps per CTA
constexpr int MU_ROWS = 64;              // rows of a unit: two per lane
constexpr int MU_COLS = 128;             // columns of a unit
constexpr int MU_Q = 128;                // queued pairs per warp and round
constexpr int MU_THREADS = 32 * MU_WARPS;

// Order-preserving key of a non-NaN binary64 value (-0 below +0).
__device__ __forceinline__ unsigned long long dkey(double x)
{
    const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(x));
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

__device__ __forceinline__ double dkey_value(unsigned long long k)
{
    const unsigned long long b = (k >> 63) ? (k & 0x7fffffffffffffffull) : ~k;
    return __longlong_as_double(static_cast<long long>(b));
}

// Order-preserving 32-bit key of a binary32 value (NaN not expected) and back.
__device__ __forceinline__ unsigned fkey(float x)
{
    const unsigned b = __float_as_uint(x);
    return (b >> 31) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned fkey_value(unsigned k) { return (k >> 31) ? (k & 0x7fffffffu) : ~k; }

// Linear index k of the triangle of units, column by column -> (row unit a,
// column tile c): column tile c meets row units 0 .. 2(c+1)-1.  A binary32
// estimate made exact by the integer corrections.
__device__ __forceinline__ void mu_coords(long long k, int& a, int& c)
{
    constexpr long long r = MU_COLS / MU_ROWS;
    long long cc = static_cast<long long>((sqrtf(8.0f * static_cast<float>(k) / r + 1.0f) - 1.0f) * 0.5f);
    if (cc < 0) cc = 0;
    while (r * (cc + 1) * (cc + 2) / 2 <= k) ++cc;
    while (cc > 0 && r * cc * (cc + 1) / 2 > k) --cc;
    c = static_cast<int>(cc);
    a = static_cast<int>(k - r * cc * (cc + 1) / 2);
}

constexpr int MX_LIST_MIN_N = 16384;  // boxes from which pass B takes the list

// About 96 overlapping pairs per box, plus a floor: beyond that pass B walks
// the units again.
unsigned matrix_list_cap(int64_t n)
{
    const unsigned long long all = n > 1 ? static_cast<unsigned long long>(n) * (n - 1) / 2 : 1ull;
    const unsigned long long c = std::min(all, 96ull * static_cast<unsigned long long>(n) + (1ull << 20));
    return static_cast<unsigned>(std::min(c, 1ull << 31));
}

long long matrix_units(long long n)
{
    const long long T = (n + MU_COLS - 1) / MU_COLS;
    return (MU_COLS / MU_ROWS) * T * (T + 1) / 2;
}

// A coordinate the packed overlap filter takes: 0, or a finite magnitude in
// [2^-40, 2^40].  Any nonzero difference of two such values is at least 2^-63
// and at most 2^41, so the product of two differences is a normal binary32
// number of the right sign (no underflow to 0, no overflow).
__device__ __forceinline__ bool filter_coord(float v)
{
    const float a = fabsf(v);
    return a == 0.0f || (a >= 0x1p-40f && a <= 0x1p40f);
}

__device__ __forceinline__ bool filter_box(float4 b)
{
    return filter_coord(b.x) && filter_coord(b.y) && filter_coord(b.z) && filter_coord(b.w);
}

// A row box spread over register pairs (both halves equal).
struct RowO {
    float2 x2, nx1, ny2, y1;
};

// The overlap filter for one row and two adjacent columns, shifted into acc
// (second column first).  A pair overlaps (the canonical w > 0 and h > 0)
// only if r.x2 > c.x1 and c.x2 > r.x1, i.e. both rounded differences
// ax = r.x2 - c.x1 and bx = c.x2 - r.x1 are positive and so is their product X
// (at most one of them is negative for boxes with x2 >= x1, and a product of
// a positive and a negative one is negative); likewise Y, the product of
// c.y1 - r.y2 and r.y1 - c.y2, both negative where they overlap in y.  The bit
// is the sign of max(-X, -Y): set where both products are positive (or -0 when
// X or Y is 0: a superset, which the exact test below sorts out).
__device__ __forceinline__ void overlap2(const RowO& r, float2 cnx1, float2 cx2, float2 cy1, float2 cny2,
                                         uint32_t& acc)
{
    const float2 ax = __fadd2_rn(r.x2, cnx1);
    const float2 bx = __fadd2_rn(cx2, r.nx1);
    const float2 ay = __fadd2_rn(cy1, r.ny2);
    const float2 by = __fadd2_rn(r.y1, cny2);
    const float2 X = __fmul2_rn(ax, bx);
    const float2 Y = __fmul2_rn(ay, by);
    const float tx = fmaxf(-X.x, -Y.x), ty = fmaxf(-X.y, -Y.y);
    acc = __funnelshift_l(__float_as_uint(ty), acc, 1);
    acc = __funnelshift_l(__float_as_uint(tx), acc, 1);
}

// Per-warp shared memory of the passes.
struct MxWarp {
    unsigned long long colmin[MU_COLS];  // passes 1, 2: smallest binary64 key per column
    float4 rows[MU_ROWS];                // the unit's row boxes
    float nx1[MU_COLS], x2[MU_COLS], y1[MU_COLS], ny2[MU_COLS];  // columns, x1 and y2 negated
    unsigned colacc[MU_COLS];            // pass 0: largest IoU bits; passes 1, 2: smallest upper-bound key
    uint32_t qe[MU_Q];                   // queued pairs: row << 8 | column
    float qo[MU_Q];                      // their IoU (0: no overlap)
    float qlo[MU_Q];                     // lower bound of their binary32 value (passes 1, 2)
    float om[MU_ROWS];                   // O_max of the rows (passes 1, 2)
};

// The binary32 bounds [lo, ub] of a pair's term in pass B (PASS 1: the
// numerator om^2 - o^2; PASS 2: the decay (1 - o) / (1 - om)); false when the
// pair contributes nothing (no overlap, or om = 1 in the linear decay).
template <int PASS>
__device__ __forceinline__ bool mx_bound(float o, float om, float& lo, float& ub)
{
    if (!(o > 0.0f)) return false;
    if (PASS == 2) {
        // binary32 quotient within a 2^-20 margin (three roundings of 2^-24)
        if (!(om < 1.0f)) return false;
        const float q = __fdiv_rn(__fsub_rn(1.0f, o), __fsub_rn(1.0f, om));
        const float eb = __fmul_rn(q, 0x1p-20f);
        lo = q - eb;
        ub = q + eb;
    } else {
        // within 2^-22 of om^2 + o^2 (three roundings) plus an absolute term
        // for tiny values
        const float aa = __fmul_rn(om, om), bb = __fmul_rn(o, o);
        const float eb = __fmul_rn(0x1p-22f, __fadd_rn(aa, bb)) + 0x1p-140f;
        const float xx = __fsub_rn(aa, bb);
        lo = xx - eb;
        ub = xx + eb;
    }
    return true;
}

// The pair's term in binary64: products exact and one rounding (Gaussian
// numerator), or the correctly rounded quotient (linear decay).
template <int PASS>
__device__ __forceinline__ double mx_value(float o, float om)
{
    const double od = static_cast<double>(o), omd = static_cast<double>(om);
    return PASS == 2 ? __ddiv_rn(__dsub_rn(1.0, od), __dsub_rn(1.0, omd))
                     : __dsub_rn(__dmul_rn(omd, omd), __dmul_rn(od, od));
}

// The list of overlapping pairs that pass A records for pass B: (i << 32 | j)
// and their IoU, count may grow past cap (the list is then incomplete and
// pass B walks the units again).
struct MxList {
    unsigned long long* ij;
    float* o;
    unsigned long long* count;  // 64-bit: the pairs of the largest inputs exceed 2^32
    unsigned cap;
};

// One unit (64 rows from rbase, 128 columns from cb) of a pass, by one warp.
// PASS 0: O_max; 1: smallest Gaussian numerator; 2: smallest linear decay.
template <int PASS>
__device__ __forceinline__ void matrix_unit(MxWarp& W, const float4* __restrict__ boxes_s, int n, int cb, int rbase,
                                            unsigned* __restrict__ omax_bits,
                                            unsigned long long* __restrict__ xmin_key, const MxList& L)
{
    const unsigned l = lane_id();
    bool ok = true;
#pragma unroll
    for (int t = static_cast<int>(l); t < MU_COLS; t += 32) {
        const int j = cb + t;
        const float4 b = j < n ? boxes_s[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        ok &= filter_box(b);
        W.nx1[t] = -b.x;
        W.x2[t] = b.z;
        W.y1[t] = b.y;
        W.ny2[t] = -b.w;
        W.colacc[t] = PASS == 0 ? 0u : 0xffffffffu;
        if (PASS) W.colmin[t] = ~0ull;
    }
    int i[2];
    float4 rb[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        i[k] = rbase + static_cast<int>(l) + 32 * k;
        rb[k] = i[k] < n ? boxes_s[i[k]] : make_float4(0.f, 0.f, 0.f, 0.f);
        ok &= filter_box(rb[k]);
        W.rows[l + 32 * k] = rb[k];
        if (PASS) W.om[l + 32 * k] = i[k] < n ? __uint_as_float(omax_bits[i[k]]) : 0.0f;
    }
    const bool fast = __all_sync(FULL, ok);
    __syncwarp();

    // Candidate bits: row k of the lane, 64-column word q.
    uint64_t w[2][2];
    if (fast) {
        RowO r[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            r[k].x2 = make_float2(rb[k].z, rb[k].z);
            r[k].nx1 = make_float2(-rb[k].x, -rb[k].x);
            r[k].ny2 = make_float2(-rb[k].w, -rb[k].w);
            r[k].y1 = make_float2(rb[k].y, rb[k].y);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t h[2][2] = {{0u, 0u}, {0u, 0u}};  // [half][row]
#pragma unroll
            for (int half = 1; half >= 0; --half) {
#pragma unroll 2
                for (int g = 7; g >= 0; --g) {
                    const int o = 64 * q + 32 * half + 4 * g;
                    const float4 A = *reinterpret_cast<const float4*>(W.nx1 + o);
                    const float4 B = *reinterpret_cast<const float4*>(W.x2 + o);
                    const float4 C = *reinterpret_cast<const float4*>(W.y1 + o);
                    const float4 D = *reinterpret_cast<const float4*>(W.ny2 + o);
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        overlap2(r[k], make_float2(A.z, A.w), make_float2(B.z, B.w), make_float2(C.z, C.w),
                                 make_float2(D.z, D.w), h[half][k]);
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        overlap2(r[k], make_float2(A.x, A.y), make_float2(B.x, B.y), make_float2(C.x, C.y),
                                 make_float2(D.x, D.y), h[half][k]);
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) w[k][q] = (static_cast<uint64_t>(h[1][k]) << 32) | h[0][k];
        }
    } else {
#pragma unroll
        for (int k = 0; k < 2; ++k) w[k][0] = w[k][1] = ~0ull;
    }
    // Only j > i, j < n.
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int j0 = cb + 64 * q;
            uint64_t keep = ~0ull;
            const int lo = i[k] + 1 - j0, hi = n - j0;
            if (i[k] >= n || lo >= 64 || hi <= 0) keep = 0;
            else {
                if (lo > 0) keep &= ~0ull << lo;
                if (hi < 64) keep &= (1ull << hi) - 1ull;
            }
            w[k][q] &= keep;
        }

    // The candidates of the warp, MU_Q at a time, one per lane: the exact
    // test and IoU, then the pass's reduction into the column accumulators.
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) cnt += __popcll(w[k][0]) + __popcll(w[k][1]);
    int x = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(FULL, x, d);
        if (static_cast<int>(l) >= d) x += y;
    }
    const int total = __shfl_sync(FULL, x, 31);
    int rk = x - cnt;  // rank of the lane's next candidate
    const int rend = x;
    for (int base = 0; base < total; base += MU_Q) {
        const int lim = min(rend, base + MU_Q);
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int q = 0; q < 2; ++q)
                while (w[k][q] && rk < lim) {
                    const int bit = __ffsll(static_cast<long long>(w[k][q])) - 1;
                    w[k][q] &= w[k][q] - 1;
                    W.qe[rk - base] = (static_cast<uint32_t>(32 * k + static_cast<int>(l)) << 8) |
                                      static_cast<uint32_t>(64 * q + bit);
                    ++rk;
                }
        __syncwarp();
        const int m = min(MU_Q, total - base);
        for (int e0 = 0; e0 < m; e0 += 32) {  // warp-uniform steps (the list reserves per warp)
            const int e = e0 + static_cast<int>(l);
            float o = 0.0f;
            int rl = 0, t = 0;
            if (e < m) {
                const uint32_t qe = W.qe[e];
                rl = static_cast<int>(qe >> 8);
                t = static_cast<int>(qe & 255u);
                const float4 r = W.rows[rl];
                const float4 cbx = make_float4(-W.nx1[t], W.y1[t], W.x2[t], -W.ny2[t]);
                // Overlap (IoU > 0) exactly as the canonical formula has it.
                const float ww = __fsub_rn(fminf(r.z, cbx.z), fmaxf(r.x, cbx.x));
                const float hh = __fsub_rn(fminf(r.w, cbx.w), fmaxf(r.y, cbx.y));
                if (ww > 0.0f && hh > 0.0f) {
                    o = iou_exact(r, box_area(r), cbx, box_area(cbx));
                    if (!(o > 0.0f)) o = 0.0f;
                }
            }
            if (PASS == 0) {
                if (o > 0.0f) atomicMax(&W.colacc[t], __float_as_uint(o));
                if (L.ij) {
                    const unsigned b = __ballot_sync(FULL, o > 0.0f);
                    unsigned long long base = 0;
                    if (l == 0 && b) base = atomicAdd(L.count, static_cast<unsigned long long>(__popc(b)));
                    base = __shfl_sync(FULL, base, 0) + static_cast<unsigned>(__popc(b & ((1u << l) - 1u)));
                    if (o > 0.0f && base < L.cap) {
                        L.ij[base] = (static_cast<unsigned long long>(rbase + rl) << 32) | static_cast<unsigned>(cb + t);
                        L.o[base] = o;
                    }
                }
            } else if (e < m) {
                const float om = W.om[rl];
                float lo = INFINITY, ub;
                if (mx_bound<PASS>(o, om, lo, ub)) atomicMin(&W.colacc[t], fkey(ub));
                else lo = INFINITY;
                W.qo[e] = o;
                W.qlo[e] = lo;
            }
        }
        if (PASS) {
            __syncwarp();
            // Candidates that can hold the column's minimum: the binary64
            // value, products exact and one rounding (Gaussian), or the
            // correctly rounded quotient (linear).
            for (int e = static_cast<int>(l); e < m; e += 32) {
                const float lo = W.qlo[e];
                const int t = static_cast<int>(W.qe[e] & 255u);
                if (lo == INFINITY || lo > __uint_as_float(fkey_value(W.colacc[t]))) continue;
                const double v = mx_value<PASS>(W.qo[e], W.om[W.qe[e] >> 8]);
                if (v == v) atomicMin(&W.colmin[t], dkey(v));
            }
        }
        __syncwarp();  // the queue is reused
    }
    // The unit's column results into the global ones.
#pragma unroll
    for (int t = static_cast<int>(l); t < MU_COLS; t += 32) {
        if (PASS == 0) {
            const unsigned v = W.colacc[t];
            if (v) atomicMax(omax_bits + cb + t, v);
        } else {
            const unsigned long long v = W.colmin[t];
            if (v != ~0ull) atomicMin(xmin_key + cb + t, v);
        }
    }
}

// A pass over the units [u_begin, u_end), one warp per unit; the grid strides
// over them when it is smaller.  A later max_out stage (done given) returns at
// once when the earlier stage has already found max_out kept boxes.
template <int PASS>
__global__ void __launch_bounds__(MU_THREADS, 8)
matrix_pass_kernel(const float4* __restrict__ boxes_s, const int* __restrict__ m_dev, int m_bound,
                   long long u_begin, long long u_end, const int* __restrict__ done,
                   unsigned* __restrict__ omax_bits, unsigned long long* __restrict__ xmin_key, MxList L)
{
    __shared__ __align__(16) MxWarp sw[MU_WARPS];
    if (done && *done) return;
    // Pass B with a list: the list kernels took the pairs unless it overflowed.
    if (PASS && L.count && *L.count <= L.cap) return;
    const int wp = threadIdx.x >> 5;
    const int n = m_dev ? *m_dev : m_bound;
    const long long stride = static_cast<long long>(gridDim.x) * MU_WARPS;
    for (long long u = u_begin + static_cast<long long>(blockIdx.x) * MU_WARPS + wp; u < u_end; u += stride) {
        int a, c;
        mu_coords(u, a, c);
        const int cb = c * MU_COLS, rbase = a * MU_ROWS;
        if (cb >= n || rbase >= n) continue;  // beyond the device-side count (warp-uniform)
        __syncwarp();  // the previous unit's use of the warp's shared memory is over
        matrix_unit<PASS>(sw[wp], boxes_s, n, cb, rbase, omax_bits, xmin_key, L);
    }
}

// Pass B over a complete list of overlapping pairs, in two sweeps: the
// smallest binary32 upper bound per child, then the binary64 term of the pairs
// whose lower bound does not exceed it, minimised per child.
template <int PASS>
__global__ void __launch_bounds__(256)
matrix_list_kernel(MxList L, int sweep, const unsigned* __restrict__ omax_bits, unsigned* __restrict__ colhi,
                   unsigned long long* __restrict__ xmin_key)
{
    const unsigned long long total = *L.count;
    if (total > L.cap) return;  // incomplete: the unit pass takes over
    const unsigned cnt = static_cast<unsigned>(total);
    for (unsigned e = blockIdx.x * blockDim.x + threadIdx.x; e < cnt; e += gridDim.x * blockDim.x) {
        const unsigned long long ij = L.ij[e];
        const int i = static_cast<int>(ij >> 32), j = static_cast<int>(ij & 0xffffffffu);
        const float o = L.o[e], om = __uint_as_float(omax_bits[i]);
        float lo, ub;
        if (!mx_bound<PASS>(o, om, lo, ub)) continue;
        if (sweep == 0) {
            atomicMin(colhi + j, fkey(ub));
        } else if (!(lo > __uint_as_float(fkey_value(colhi[j])))) {
            const double v = mx_value<PASS>(o, om);
            if (v == v) atomicMin(xmin_key + j, dkey(v));
        }
    }
}

// One thread per sorted box: its final score and whether it stays; lane l of
// a warp decides box 32w+l and the warp writes word w of the kept bitmap.
__global__ void __launch_bounds__(256)
matrix_decide_kernel(const float* __restrict__ scores, const int* __restrict__ perm,
                     const unsigned long long* __restrict__ xmin_key, const int* __restrict__ m_dev,
                     int m_bound, float sigma, int linear, float decay_thr, float* __restrict__ fs_out,
                     uint32_t* __restrict__ kept, int lo, const int* __restrict__ done)
{
    if (done && *done) return;  // an earlier max_out stage found enough kept boxes
    const int n = m_dev ? *m_dev : m_bound;
    const int j = lo + blockIdx.x * blockDim.x + threadIdx.x;  // lo: a multiple of 32
    if (j - static_cast<int>(lane_id()) >= n) return;  // whole warp past the end
    bool keep_j = false;
    if (j < n && linear) {
        // s * min(1, smallest decay) and the comparison, in binary64
        const float s = scores[perm[j]];
        const unsigned long long k = xmin_key[j];
        const double m = k == ~0ull ? 1.0 : fmin(dkey_value(k), 1.0);
        const double fd = __dmul_rn(static_cast<double>(s), m);
        fs_out[j] = static_cast<float>(fd);
        keep_j = !(fd < static_cast<double>(decay_thr));
    } else if (j < n) {
        const float s = scores[perm[j]];
        const unsigned long long k = xmin_key[j];
        // the smallest exponent is the smallest numerator over sigma (a
        // positive divisor keeps the order of correctly rounded quotients)
        const double x = k == ~0ull ? 0.0 : fmin(__ddiv_rn(dkey_value(k), static_cast<double>(sigma)), 0.0);
        const float x32 = static_cast<float>(x);
        const float f = __fmul_rn(s, expf(x32));
        // |f - s exp(x)| <= |f| (2^-22 (expf, 2 ulp) + 2^-24 (1 + |x|) (the
        // product and the exponent's rounding)) + 2^-126; a margin four times
        // that decides in binary32, anything closer in binary64.
        const float tol = fabsf(f) * (4.0f * (0x1p-22f + 0x1p-24f * (1.0f + fabsf(x32)))) + 0x1p-124f;
        float fs;
        if (fabsf(f - decay_thr) > tol) {
            fs = f;
            keep_j = !(f < decay_thr);
        } else {
            // The same binary64 comparison as the definition's evaluation on
            // the host, with CUDA's binary64 exp (at most 1 ulp from e^x) in
            // place of the C library's: the two can only disagree on a box
            // whose binary64 final score lies within about 2 ulp of the
            // threshold (a band of relative width 2^-51).
            const double fd = static_cast<double>(s) * exp(x);
            fs = static_cast<float>(fd);
            keep_j = !(fd < static_cast<double>(decay_thr));
        }
        fs_out[j] = fs;
    }
    const uint32_t w = __ballot_sync(FULL, keep_j);
    if (lane_id() == 0) kept[j >> 5] = w;
}

void launch_matrix(const float4* boxes_s, const float* scores, const int* perm, const int* m_dev, int m_bound,
                   float sigma, int linear, float decay_thr, int max_out, unsigned* omax_bits,
                   unsigned long long* xmin_key, float* fs, uint32_t* kept, int* done, unsigned long long* list_ij,
                   float* list_o, unsigned long long* list_count, unsigned list_cap, unsigned* colhi, int64_t* keep,
                   float* keep_scores, int64_t* count, cudaStream_t st)
{
    cudaMemsetAsync(omax_bits, 0, sizeof(unsigned) * static_cast<size_t>(m_bound), st);
    cudaMemsetAsync(xmin_key, 0xff, sizeof(unsigned long long) * static_cast<size_t>(m_bound), st);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    // Boxes [lo, hi): the passes over the units of columns [lo, hi) (all rows
    // above them) and the decisions of boxes [lo, hi).  A stage given `done`
    // strides over its units with one resident wave, so that finding the flag
    // set costs a few CTAs per SM.
    auto stage = [&](int lo, int hi, const int* dn, const MxList& L) {
        const long long u0 = matrix_units(lo), u1 = matrix_units(hi);
        if (u1 > u0) {
            long long g = (u1 - u0 + MU_WARPS - 1) / MU_WARPS;
            if (dn) g = std::min(g, static_cast<long long>(sms) * 8);
            const unsigned grid = static_cast<unsigned>(g);
            matrix_pass_kernel<0><<<grid, MU_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, u0, u1, dn, omax_bits,
                                                                xmin_key, L);
            // With a list, pass B takes its pairs in two flat sweeps, and the
            // unit pass (one resident wave, striding) returns at once unless
            // the list overflowed.
            const unsigned gb = L.ij ? static_cast<unsigned>(std::min(g, static_cast<long long>(sms) * 8)) : grid;
            if (L.ij) {
                const unsigned gl = static_cast<unsigned>(sms) * 8;
                for (int sweep = 0; sweep < 2; ++sweep) {
                    if (linear)
                        matrix_list_kernel<2><<<gl, 256, 0, st>>>(L, sweep, omax_bits, colhi, xmin_key);
                    else
                        matrix_list_kernel<1><<<gl, 256, 0, st>>>(L, sweep, omax_bits, colhi, xmin_key);
                }
            }
            if (linear)
                matrix_pass_kernel<2><<<gb, MU_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, u0, u1, dn, omax_bits,
                                                                  xmin_key, L);
            else
                matrix_pass_kernel<1><<<gb, MU_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, u0, u1, dn, omax_bits,
                                                                  xmin_key, L);
        }
        if (hi > lo)
            matrix_decide_kernel<<<(hi - lo + 255) / 256, 256, 0, st>>>(scores, perm, xmin_key, m_dev, m_bound,
                                                                        sigma, linear, decay_thr, fs, kept, lo, dn);
    };
    // With max_out, a box's decay depends only on the boxes before it, so the
    // first max_out kept boxes depend only on a prefix of the score order:
    // the leading 2*max_out boxes first, the rest only if they held fewer
    // than max_out kept boxes.
    const long long k = max_out > 0 ? (2LL * max_out + MU_COLS - 1) / MU_COLS * MU_COLS : m_bound;
    if (k >= m_bound) {
        // The list pays off when the unit walk of pass B is long; below
        // MX_LIST_MIN_N boxes its extra launches cost more than they save.
        const bool use_list = list_ij && m_bound >= MX_LIST_MIN_N;
        MxList L{use_list ? list_ij : nullptr, list_o, use_list ? list_count : nullptr, list_cap};
        if (use_list) {
            cudaMemsetAsync(list_count, 0, sizeof(unsigned long long), st);
            cudaMemsetAsync(colhi, 0xff, sizeof(unsigned) * static_cast<size_t>(m_bound), st);
        }
        stage(0, m_bound, nullptr, L);
    } else {
        const MxList none{nullptr, nullptr, nullptr, 0u};
        // The rest's decisions may be skipped: their kept words must read 0.
        cudaMemsetAsync(kept, 0, sizeof(uint32_t) * static_cast<size_t>((m_bound + 31) / 32), st);
        stage(0, static_cast<int>(k), nullptr, none);
        launch_kept_prefix(kept, m_dev, m_bound, static_cast<int>(k), max_out, done, st);
        stage(static_cast<int>(k), m_bound, done, none);
    }
    launch_bits_emit(kept, m_dev, m_bound, perm, fs, max_out, keep, keep_scores, count, st);
}

}  // namespace gbnms
