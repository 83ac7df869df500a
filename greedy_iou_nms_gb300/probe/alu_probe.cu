// Throughput probe of the SM's binary32 and integer instruction forms that
// the IoU test and the mask filter use, for the roofline denominators.
//
// Each thread runs kChains independent dependency chains of one instruction
// form (so latency is hidden by the chains and by the resident warps), the
// grid is exactly `ctas_per_sm` CTAs of 256 threads on every SM, and every
// CTA reads the SM clock (clock64) and the global timer (ns) before and after
// its loop, with a CTA barrier on both sides so the span covers all its warps.
// Lane operations per SM clock follow from the instruction count and the
// cycles, the clock from cycles per nanosecond; the caller's CUDA events give
// the rate per second.  The instructions are written as inline PTX, which the compiler
// neither folds nor removes (every result feeds the final store).
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int kThreads = 256;
constexpr int kChains = 8;
constexpr int kUnroll = 16;

enum Form : int {
    F_FFMA = 0,   // fma.rn.f32
    F_FADD = 1,   // add.rn.f32
    F_FMNMX = 2,  // min.f32
    F_FADD2 = 3,  // add.rn.f32x2 (two lane operations per instruction)
    F_FFMA2 = 4,  // fma.rn.f32x2 (two lane operations per instruction)
    F_SHF = 5,    // shf.l.wrap.b32
    F_MIX = 6,    // add.rn.f32x2 and min.f32 alternating (two pipes)
    F_FSET = 7,   // setp.lt.f32 feeding selp (compare and select)
    F_COUNT = 8
};

__device__ __forceinline__ float ffma(float a, float b, float c)
{
    float d;
    asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fadd(float a, float b)
{
    float d;
    asm("add.rn.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float fmin1(float a, float b)
{
    float d;
    asm("min.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint32_t shf(uint32_t lo, uint32_t hi)
{
    uint32_t d;
    asm("shf.l.wrap.b32 %0, %1, %2, 1;" : "=r"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ float fset(float a, float b, float c)
{
    float d;
    asm("{\n\t.reg .pred p;\n\tsetp.lt.f32 p, %1, %2;\n\tselp.f32 %0, %2, %3, p;\n\t}"
        : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint64_t pack2(float a, float b)
{
    return static_cast<uint64_t>(__float_as_uint(a)) | (static_cast<uint64_t>(__float_as_uint(b)) << 32);
}
__device__ __forceinline__ float unpack_sum(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v)) + __uint_as_float(static_cast<uint32_t>(v >> 32));
}

// Values stay finite and normal: the fma chains converge to c/(1-b), the add
// chains grow by 2^-20 a step, the min chains keep their starting values.
__device__ __forceinline__ long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return static_cast<long long>(t);
}

template <int F>
__global__ void __launch_bounds__(kThreads) probe_kernel(int iters, float seed, float* __restrict__ out,
                                                         long long* __restrict__ cycles, long long* __restrict__ ns)
{
    const float s = seed + 1e-3f * static_cast<float>(threadIdx.x & 31);
    float x[kChains];
    uint64_t y[kChains];
    uint32_t z[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        x[c] = s + static_cast<float>(c);
        y[c] = pack2(s + static_cast<float>(c), s - static_cast<float>(c));
        z[c] = __float_as_uint(s) + static_cast<uint32_t>(c) * 0x9e3779b9u;
    }
    const float b = 0.999f, cst = 0x1p-20f;
    const uint64_t b2 = pack2(b, b), c2 = pack2(cst, cst);
    __syncthreads();
    const long long t0 = clock64();
    const long long g0 = global_ns();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int c = 0; c < kChains; ++c) {
                if constexpr (F == F_FFMA) x[c] = ffma(x[c], b, cst);
                if constexpr (F == F_FADD) x[c] = fadd(x[c], cst);
                if constexpr (F == F_FMNMX) x[c] = fmin1(x[c], x[(c + 1) % kChains]);
                if constexpr (F == F_FADD2) y[c] = fadd2(y[c], c2);
                if constexpr (F == F_FFMA2) y[c] = ffma2(y[c], b2, c2);
                if constexpr (F == F_SHF) z[c] = shf(z[c], z[(c + 1) % kChains]);
                if constexpr (F == F_MIX) {
                    if (c & 1) x[c] = fmin1(x[c], x[c ^ 1]);
                    else y[c] = fadd2(y[c], c2);
                }
                if constexpr (F == F_FSET) x[c] = fset(x[c], x[(c + 1) % kChains], cst);
            }
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    const long long g1 = global_ns();
    float acc = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc += x[c] + unpack_sum(y[c]) + static_cast<float>(z[c] & 7u);
    out[static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x] = acc;
    if (threadIdx.x == 0) {
        cycles[blockIdx.x] = t1 - t0;
        ns[blockIdx.x] = g1 - g0;
    }
}

using Kern = void (*)(int, float, float*, long long*, long long*);
constexpr Kern kKernels[F_COUNT] = {probe_kernel<F_FFMA>,  probe_kernel<F_FADD>,  probe_kernel<F_FMNMX>,
                                    probe_kernel<F_FADD2>, probe_kernel<F_FFMA2>, probe_kernel<F_SHF>,
                                    probe_kernel<F_MIX>,   probe_kernel<F_FSET>};

}  // namespace

extern "C" {

// Number of instruction forms; form k's name and lane operations per
// instruction (2 for the packed forms; the compare-and-select form counts
// its two instructions as one operation, the mixed form averages 1.5).
int gbprobe_forms() { return F_COUNT; }

const char* gbprobe_form_name(int form)
{
    static const char* names[F_COUNT] = {"ffma",        "fadd",        "fmnmx", "fadd2",
                                         "ffma2",       "shf",         "fadd2+fmnmx", "fsetp+selp"};
    return form >= 0 && form < F_COUNT ? names[form] : "";
}

// Lane operations of one thread's run: iters x kUnroll x kChains instructions,
// each worth the form's lane operations.
double gbprobe_ops_per_thread(int form, int iters)
{
    const double ins = static_cast<double>(iters) * kUnroll * kChains;
    switch (form) {
        case F_FADD2:
        case F_FFMA2: return 2.0 * ins;
        case F_MIX: return 1.5 * ins;
        default: return ins;
    }
}

// Instructions (not operations) of one thread's run.
double gbprobe_insts_per_thread(int form, int iters)
{
    const double ins = static_cast<double>(iters) * kUnroll * kChains;
    return form == F_FSET ? 2.0 * ins : ins;
}

int gbprobe_threads_per_cta() { return kThreads; }

// Launches form `form` on `ctas` CTAs of 256 threads on `stream`.  `out` is
// a device buffer of ctas x 256 floats, `cycles` and `ns` device buffers of
// ctas long longs (each CTA's SM-clock cycles and global-timer nanoseconds
// for its loop).  Returns a cudaError_t value (0 on success); iters must be
// in [1, 2^24] and ctas in [1, 2^20].
int gbprobe_launch(int form, int ctas, int iters, float* out, long long* cycles, long long* ns, void* stream)
{
    if (form < 0 || form >= F_COUNT || ctas < 1 || ctas > (1 << 20) || iters < 1 || iters > (1 << 24) || !out ||
        !cycles || !ns)
        return static_cast<int>(cudaErrorInvalidValue);
    kKernels[form]<<<ctas, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, 1.25f, out, cycles, ns);
    return static_cast<int>(cudaGetLastError());
}

// Streaming multiprocessors of the current device (0 on error).
int gbprobe_sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // extern "C"
