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
// fathers), and only overlapping pairs (IoU > 0) need work:
//   pass A: tiles of the upper triangle; where two boxes overlap, the exact
//           binary32 IoU, atomically maxed into O_max of the child;
//   pass B: the same tiles; for each overlapping pair the binary64 numerator
//           O_max[i]^2 - O[i][j]^2, atomically minimised per child through an
//           order-preserving 64-bit key (dividing once per box by sigma > 0
//           afterwards gives the smallest quotient: correctly rounded
//           division by a positive number keeps the order);
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

#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int MX_T = 128;             // tile rows and columns
constexpr int MX_THREADS = 64;        // 2 warps x 2 rows per lane = 128 rows

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

// Each warp reduces a column over its 64 rows before one atomic, and skips a
// column no lane overlaps with one vote.

// Order-preserving 32-bit key of a binary32 value (NaN not expected) and back.
__device__ __forceinline__ unsigned fkey(float x)
{
    const unsigned b = __float_as_uint(x);
    return (b >> 31) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned fkey_value(unsigned k) { return (k >> 31) ? (k & 0x7fffffffu) : ~k; }

// Linear index k of the triangle of MX_T x MX_T tiles, column by column ->
// (row tile a, column tile c), a <= c.  A binary32 estimate made exact by the
// integer corrections.
__device__ __forceinline__ void mx_coords(long long k, int& a, int& c)
{
    long long cc = static_cast<long long>((sqrtf(8.0f * static_cast<float>(k) + 1.0f) - 1.0f) * 0.5f);
    if (cc < 0) cc = 0;
    while ((cc + 1) * (cc + 2) / 2 <= k) ++cc;
    while (cc > 0 && cc * (cc + 1) / 2 > k) --cc;
    c = static_cast<int>(cc);
    a = static_cast<int>(k - cc * (cc + 1) / 2);
}

// Binary64 work of pass B, queued per warp: a candidate (child column j, the
// father's O_max, their IoU) is finished later with the other candidates of
// the warp, one per lane, so that each binary64 instruction serves up to 32
// candidates instead of the one or two rows a column leaves.
constexpr int MX_Q = 96;  // queue entries per warp: flushed at 32, one column adds at most 64

template <int PASS>
__device__ __forceinline__ void mx_flush(const int* qj, const float* qom, const float* qo, int cnt,
                                         unsigned long long* __restrict__ xmin_key)
{
    for (int e = static_cast<int>(lane_id()); e < cnt; e += 32) {
        const double om = static_cast<double>(qom[e]), od = static_cast<double>(qo[e]);
        const double x = PASS == 2 ? __ddiv_rn(__dsub_rn(1.0, od), __dsub_rn(1.0, om))
                                   : __dsub_rn(__dmul_rn(om, om), __dmul_rn(od, od));
        if (x == x) atomicMin(xmin_key + qj[e], dkey(x));
    }
}

// PASS 0: O_max; 1: smallest Gaussian numerator; 2: smallest linear decay.
template <int PASS>
__global__ void __launch_bounds__(MX_THREADS)
matrix_pass_kernel(const float4* __restrict__ boxes_s, const int* __restrict__ m_dev, int m_bound,
                   float sigma, unsigned* __restrict__ omax_bits, unsigned long long* __restrict__ xmin_key)
{
    __shared__ float4 cbox[MX_T];
    __shared__ float carea[MX_T];
    __shared__ int q_j[PASS ? MX_THREADS / 32 : 1][MX_Q];
    __shared__ float q_om[PASS ? MX_THREADS / 32 : 1][MX_Q], q_o[PASS ? MX_THREADS / 32 : 1][MX_Q];
    const int n = m_dev ? *m_dev : m_bound;
    int a, c;
    mx_coords(blockIdx.x, a, c);
    const int cb = c * MX_T, rb = a * MX_T;
    if (cb >= n) return;
    for (int t = threadIdx.x; t < MX_T; t += MX_THREADS) {
        const int j = cb + t;
        const float4 b = j < n ? boxes_s[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        cbox[t] = b;
        carea[t] = box_area(b);
    }
    const unsigned l = lane_id();
    const int i0 = rb + (threadIdx.x >> 5) * 64 + static_cast<int>(l), i1 = i0 + 32;
    const bool v0 = i0 < n, v1 = i1 < n;
    const float4 r0 = v0 ? boxes_s[i0] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 r1 = v1 ? boxes_s[i1] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float ar0 = box_area(r0), ar1 = box_area(r1);
    double om0 = 0.0, om1 = 0.0;
    if (PASS >= 1) {
        if (v0) om0 = static_cast<double>(__uint_as_float(omax_bits[i0]));
        if (v1) om1 = static_cast<double>(__uint_as_float(omax_bits[i1]));
    }
    __syncthreads();
    const int kend = min(MX_T, n - cb);
    // Row i's overlap with column box k, if any (IoU > 0, i before j).
    auto overlap = [&](int i, const float4& r, float ar, int k, float& o) -> bool {
        const float4 cbx = cbox[k];
        const float w = __fsub_rn(fminf(r.z, cbx.z), fmaxf(r.x, cbx.x));
        const float h = __fsub_rn(fminf(r.w, cbx.w), fmaxf(r.y, cbx.y));
        if (!(w > 0.0f && h > 0.0f && i < cb + k)) return false;
        o = iou_exact(r, ar, cbx, carea[k]);
        return o > 0.0f;
    };
    // The warp's queue of binary64 candidates (pass B).
    const int wq = PASS ? (threadIdx.x >> 5) : 0;
    int qn = 0;
    auto queue = [&](bool c0, bool c1, int j, float o0, float o1) {
        const unsigned b0 = __ballot_sync(FULL, c0), b1 = __ballot_sync(FULL, c1);
        const unsigned below = (1u << l) - 1u;
        if (c0) {
            const int e = qn + __popc(b0 & below);
            q_j[wq][e] = j;
            q_om[wq][e] = static_cast<float>(om0);
            q_o[wq][e] = o0;
        }
        if (c1) {
            const int e = qn + __popc(b0) + __popc(b1 & below);
            q_j[wq][e] = j;
            q_om[wq][e] = static_cast<float>(om1);
            q_o[wq][e] = o1;
        }
        qn += __popc(b0) + __popc(b1);
        if (qn >= 32) {
            __syncwarp();
            mx_flush<PASS>(q_j[wq], q_om[wq], q_o[wq], qn, xmin_key);
            __syncwarp();
            qn = 0;
        }
    };
    for (int k = 0; k < kend; ++k) {
        const float4 cbx = cbox[k];
        const bool maybe0 = v0 && fminf(r0.z, cbx.z) > fmaxf(r0.x, cbx.x) && fminf(r0.w, cbx.w) > fmaxf(r0.y, cbx.y);
        const bool maybe1 = v1 && fminf(r1.z, cbx.z) > fmaxf(r1.x, cbx.x) && fminf(r1.w, cbx.w) > fmaxf(r1.y, cbx.y);
        if (!__any_sync(FULL, maybe0 || maybe1)) continue;  // no lane overlaps column k
        float o0 = 0.0f, o1 = 0.0f;
        const bool ov0 = maybe0 && overlap(i0, r0, ar0, k, o0);
        const bool ov1 = maybe1 && overlap(i1, r1, ar1, k, o1);
        const int j = cb + k;
        if (PASS == 0) {
            // largest overlap of the column over the warp's rows, one atomic
            const unsigned m = max(ov0 ? __float_as_uint(o0) : 0u, ov1 ? __float_as_uint(o1) : 0u);
            const unsigned r = __reduce_max_sync(FULL, m);
            if (l == 0 && r) atomicMax(omax_bits + j, r);
        } else if (PASS == 2) {
            // Smallest decay (1 - O[i][j]) / (1 - O_max[i]) over the warp's
            // rows, one atomic.  Rows bound their quotient in binary32 (three
            // roundings, each within 2^-24 relative; a margin of 2^-20), and
            // only rows whose lower bound does not exceed the smallest upper
            // bound take the binary64 quotient.  O_max = 1 (a zero
            // denominator, the same in both precisions) contributes nothing.
            float lo0 = INFINITY, lo1 = INFINITY, ub = INFINITY;
            const bool d0 = ov0 && static_cast<float>(om0) < 1.0f, d1 = ov1 && static_cast<float>(om1) < 1.0f;
            if (d0) {
                const float q = __fdiv_rn(__fsub_rn(1.0f, o0), __fsub_rn(1.0f, static_cast<float>(om0)));
                const float e = __fmul_rn(q, 0x1p-20f);
                lo0 = q - e;
                ub = q + e;
            }
            if (d1) {
                const float q = __fdiv_rn(__fsub_rn(1.0f, o1), __fsub_rn(1.0f, static_cast<float>(om1)));
                const float e = __fmul_rn(q, 0x1p-20f);
                lo1 = q - e;
                ub = fminf(ub, q + e);
            }
            const float best = __uint_as_float(fkey_value(__reduce_min_sync(FULL, fkey(ub))));
            queue(d0 && !(lo0 > best), d1 && !(lo1 > best), j, o0, o1);
        } else {
            // Smallest numerator O_max[i]^2 - O[i][j]^2 (binary64, products
            // exact, one rounding) over the warp's rows, one atomic.  Only
            // rows that can hold the minimum compute it in binary64: each
            // overlapping row bounds its numerator in binary32 (three
            // roundings, each within 2^-24 of a term of magnitude at most
            // om^2 + o^2), the warp takes the smallest upper bound, and rows
            // whose lower bound does not exceed it are the candidates.
            float lo0 = INFINITY, lo1 = INFINITY, ub = INFINITY;
            if (ov0) {
                const float a = __fmul_rn(static_cast<float>(om0), static_cast<float>(om0)), b = __fmul_rn(o0, o0);
                const float e = __fmul_rn(0x1p-22f, __fadd_rn(a, b)) + 0x1p-140f;
                const float x = __fsub_rn(a, b);
                lo0 = x - e;
                ub = x + e;
            }
            if (ov1) {
                const float a = __fmul_rn(static_cast<float>(om1), static_cast<float>(om1)), b = __fmul_rn(o1, o1);
                const float e = __fmul_rn(0x1p-22f, __fadd_rn(a, b)) + 0x1p-140f;
                const float x = __fsub_rn(a, b);
                lo1 = x - e;
                ub = fminf(ub, x + e);
            }
            const float best = __uint_as_float(fkey_value(__reduce_min_sync(FULL, fkey(ub))));
            queue(ov0 && !(lo0 > best), ov1 && !(lo1 > best), j, o0, o1);
        }
    }
    if (PASS >= 1) {
        __syncwarp();
        mx_flush<PASS>(q_j[wq], q_om[wq], q_o[wq], qn, xmin_key);
    }
}

// One thread per sorted box: its final score and whether it stays; lane l of
// a warp decides box 32w+l and the warp writes word w of the kept bitmap.
__global__ void __launch_bounds__(256)
matrix_decide_kernel(const float* __restrict__ scores, const int* __restrict__ perm,
                     const unsigned long long* __restrict__ xmin_key, const int* __restrict__ m_dev,
                     int m_bound, float sigma, int linear, float decay_thr, float* __restrict__ fs_out,
                     uint32_t* __restrict__ kept)
{
    const int n = m_dev ? *m_dev : m_bound;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
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
                   unsigned long long* xmin_key, float* fs, uint32_t* kept, int64_t* keep, float* keep_scores,
                   int64_t* count, cudaStream_t st)
{
    cudaMemsetAsync(omax_bits, 0, sizeof(unsigned) * static_cast<size_t>(m_bound), st);
    cudaMemsetAsync(xmin_key, 0xff, sizeof(unsigned long long) * static_cast<size_t>(m_bound), st);
    const long long T = (m_bound + MX_T - 1) / MX_T;
    const long long tiles = T * (T + 1) / 2;
    if (tiles > 0) {
        matrix_pass_kernel<0><<<static_cast<unsigned>(tiles), MX_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, sigma,
                                                                                 omax_bits, xmin_key);
        if (linear)
            matrix_pass_kernel<2><<<static_cast<unsigned>(tiles), MX_THREADS, 0, st>>>(boxes_s, m_dev, m_bound,
                                                                                     sigma, omax_bits, xmin_key);
        else
            matrix_pass_kernel<1><<<static_cast<unsigned>(tiles), MX_THREADS, 0, st>>>(boxes_s, m_dev, m_bound,
                                                                                     sigma, omax_bits, xmin_key);
    }
    matrix_decide_kernel<<<(m_bound + 255) / 256, 256, 0, st>>>(scores, perm, xmin_key, m_dev, m_bound, sigma,
                                                                linear, decay_thr, fs, kept);
    launch_bits_emit(kept, m_dev, m_bound, perm, fs, max_out, keep, keep_scores, count, st);
}

}  // namespace gbnms
