// Matrix NMS with Gaussian decay, one image.
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
//   pass B: the same tiles; for each overlapping pair the binary64 exponent
//           (O_max[i]^2 - O[i][j]^2) / sigma, atomically minimised per child
//           through an order-preserving 64-bit key;
//   emit:   per box, s * exp(min(0, smallest exponent)) against the
//           threshold, decided in binary32 with expf when the result is
//           clear of the threshold by more than its error bound, in binary64
//           otherwise; the kept boxes in score order with their final scores.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int MX_T = 128;             // tile rows and columns
constexpr int MX_THREADS = 64;        // 2 warps x 2 rows per lane = 128 rows
constexpr int ME_THREADS = 1024;

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

// Linear index k of the triangle of MX_T x MX_T tiles, column by column ->
// (row tile a, column tile c), a <= c.
__device__ __forceinline__ void mx_coords(long long k, int& a, int& c)
{
    long long cc = static_cast<long long>((sqrt(8.0 * static_cast<double>(k) + 1.0) - 1.0) * 0.5);
    while ((cc + 1) * (cc + 2) / 2 <= k) ++cc;
    while (cc * (cc + 1) / 2 > k) --cc;
    c = static_cast<int>(cc);
    a = static_cast<int>(k - cc * (cc + 1) / 2);
}

template <int PASS>
__global__ void __launch_bounds__(MX_THREADS)
matrix_pass_kernel(const float4* __restrict__ boxes_s, const int* __restrict__ m_dev, int m_bound,
                   float sigma, unsigned* __restrict__ omax_bits, unsigned long long* __restrict__ xmin_key)
{
    __shared__ float4 cbox[MX_T];
    __shared__ float carea[MX_T];
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
    if (PASS == 1) {
        if (v0) om0 = static_cast<double>(__uint_as_float(omax_bits[i0]));
        if (v1) om1 = static_cast<double>(__uint_as_float(omax_bits[i1]));
    }
    __syncthreads();
    const int kend = min(MX_T, n - cb);
    auto pair = [&](int i, const float4& r, float ar, double om, int k) {
        const int j = cb + k;
        const float4 cbx = cbox[k];
        const float w = __fsub_rn(fminf(r.z, cbx.z), fmaxf(r.x, cbx.x));
        const float h = __fsub_rn(fminf(r.w, cbx.w), fmaxf(r.y, cbx.y));
        if (w > 0.0f && h > 0.0f && i < j) {
            const float o = iou_exact(r, ar, cbx, carea[k]);
            if (o > 0.0f) {
                if (PASS == 0) {
                    atomicMax(omax_bits + j, __float_as_uint(o));
                } else {
                    const double od = static_cast<double>(o);
                    const double x = __ddiv_rn(__dsub_rn(__dmul_rn(om, om), __dmul_rn(od, od)),
                                               static_cast<double>(sigma));
                    if (x == x) atomicMin(xmin_key + j, dkey(x));
                }
            }
        }
    };
    for (int k = 0; k < kend; ++k) {
        if (v0) pair(i0, r0, ar0, om0, k);
        if (v1) pair(i1, r1, ar1, om1, k);
    }
}

// One CTA: warp w owns the 32-box words [w*wpw, (w+1)*wpw); a block prefix of
// the kept counts places them; lane l decides box 32w+l.
__global__ void __launch_bounds__(ME_THREADS)
matrix_emit_kernel(const float* __restrict__ scores, const int* __restrict__ perm,
                   const unsigned long long* __restrict__ xmin_key, const int* __restrict__ m_dev,
                   int m_bound, float decay_thr, int max_out, int64_t* __restrict__ keep,
                   float* __restrict__ keep_scores, int64_t* __restrict__ count)
{
    __shared__ int scratch[32];
    const int n = m_dev ? *m_dev : m_bound;
    const int NW = (n + 31) / 32;
    const unsigned l = lane_id();
    const int warp = threadIdx.x >> 5;
    const int wpw = (NW + 31) / 32;
    const int a0 = min(warp * wpw, NW), a1 = min(a0 + wpw, NW);
    // Final score of sorted box j and whether it stays (>= the threshold).
    auto decide = [&](int j, float& fs) -> bool {
        if (j >= n) return false;
        const float s = scores[perm[j]];
        const unsigned long long k = xmin_key[j];
        const double x = k == ~0ull ? 0.0 : fmin(dkey_value(k), 0.0);
        const float x32 = static_cast<float>(x);
        const float f = __fmul_rn(s, expf(x32));
        // |f - s exp(x)| <= |f| (2^-22 (expf, 2 ulp) + 2^-24 (1 + |x|)
        // (product and the exponent's rounding)) + 2^-126; a margin four
        // times that decides in binary32, anything closer in binary64.
        const float tol = fabsf(f) * (4.0f * (0x1p-22f + 0x1p-24f * (1.0f + fabsf(x32)))) + 0x1p-124f;
        if (fabsf(f - decay_thr) > tol) {
            fs = f;
            return !(f < decay_thr);
        }
        const double fd = static_cast<double>(s) * exp(x);
        fs = static_cast<float>(fd);
        return !(fd < static_cast<double>(decay_thr));
    };
    int c = 0;
    for (int w = a0; w < a1; ++w) {
        float fs;
        c += __popc(__ballot_sync(FULL, decide(32 * w + static_cast<int>(l), fs)));
    }
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
    for (int w = a0; w < a1 && base < cap; ++w) {
        const int j = 32 * w + static_cast<int>(l);
        float fs = 0.0f;
        const bool kept = decide(j, fs);
        const uint32_t bits = __ballot_sync(FULL, kept);
        const int pos = base + __popc(bits & below);
        if (kept && pos < cap) {
            keep[pos] = perm[j];
            if (keep_scores) keep_scores[pos] = fs;
        }
        base += __popc(bits);
    }
    if (threadIdx.x == 0) count[0] = total < cap ? total : cap;
}

void launch_matrix(const float4* boxes_s, const float* scores, const int* perm, const int* m_dev, int m_bound,
                   float sigma, float decay_thr, int max_out, unsigned* omax_bits,
                   unsigned long long* xmin_key, int64_t* keep, float* keep_scores, int64_t* count,
                   cudaStream_t st)
{
    cudaMemsetAsync(omax_bits, 0, sizeof(unsigned) * static_cast<size_t>(m_bound), st);
    cudaMemsetAsync(xmin_key, 0xff, sizeof(unsigned long long) * static_cast<size_t>(m_bound), st);
    const long long T = (m_bound + MX_T - 1) / MX_T;
    const long long tiles = T * (T + 1) / 2;
    if (tiles > 0) {
        matrix_pass_kernel<0><<<static_cast<unsigned>(tiles), MX_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, sigma,
                                                                                 omax_bits, xmin_key);
        matrix_pass_kernel<1><<<static_cast<unsigned>(tiles), MX_THREADS, 0, st>>>(boxes_s, m_dev, m_bound, sigma,
                                                                                 omax_bits, xmin_key);
    }
    matrix_emit_kernel<<<1, ME_THREADS, 0, st>>>(scores, perm, xmin_key, m_dev, m_bound, decay_thr, max_out,
                                                 keep, keep_scores, count);
}

}  // namespace gbnms
