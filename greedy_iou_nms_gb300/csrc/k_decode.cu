// Front end for YOLO-shaped outputs and NMS over the count-header buffer.
//
// "YOLOv5后处理GPU移植实战", section 1.1: a "count header + data body" buffer
// per image, float[1 + 7 * max_objects]: the number of candidates found, then
// one row of 7 floats per candidate (left, top, right, bottom, confidence,
// class, keep_flag).  Section 1.2: slots come from a counter, candidates past
// max_objects are dropped (the header still counts them), and the counter is
// reduced locally (per block) before the global step.  Section 2.2: NMS over
// the buffer ranks by confidence, then by the lower position, and only boxes
// of one class interact.
//
// Decode (the page gives the layout, not the decode): each prediction row
// (cx, cy, w, h, objectness, class scores) gives confidence RN(objectness x
// largest class score), the first class with that maximum, and the box
// centre +- half size; a row is a candidate when its confidence is >
// conf_thr.  Candidates take the rows in anchor order, so the buffer is the
// same on every run.
//
// GPU shape: one CTA per 128 anchors of an image stages their rows in shared
// memory with bulk copies (the rows are contiguous; the copy engine streams
// them, completing on a shared-memory barrier with a bounded wait), decodes
// one anchor per thread, compacts its candidates with a ballot per warp and a
// prefix over its 4 warps, and writes them and its count to a staging area
// (the local reduction).  One CTA per image then takes the prefix of the
// image's block counts, writes the header and copies the first max_objects
// candidates in order.  NMS over buffers gathers the rows into the batched path's inputs
// (per image at a fixed stride of max_objects rows, only the first
// min(header, max_objects) taking part), runs it, and writes keep_flag.
#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int DC_APB = 128;      // anchors per decode CTA

// The header and the first max_objects candidates of image b, in order, by
// the calling CTA (blockDim.x threads, `pre` shared scratch of nblk + 1 ints).
__device__ void emit_image(int b, const float* __restrict__ stage, const int* __restrict__ blk_cnt, int nblk,
                           int max_objects, float* __restrict__ out, int* pre, int* wsum)
{
    const int nt = blockDim.x;
    const int* cnt = blk_cnt + static_cast<int64_t>(b) * nblk;
    // Thread t sums a contiguous run of blocks, then a block-wide scan.
    const int per = (nblk + nt - 1) / nt;
    const int k0 = min(nblk, static_cast<int>(threadIdx.x) * per), k1 = min(nblk, k0 + per);
    int run = 0;
    for (int k = k0; k < k1; ++k) run += cnt[k];
    const unsigned l = lane_id();
    const int w = threadIdx.x >> 5;
    int x = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(FULL, x, d);
        if (static_cast<int>(l) >= d) x += y;
    }
    if (l == 31) wsum[w] = x;
    __syncthreads();
    int before = x - run;
    for (int q = 0; q < w; ++q) before += wsum[q];
    for (int k = k0; k < k1; ++k) {
        pre[k] = before;
        before += cnt[k];
    }
    if (static_cast<int>(threadIdx.x) == nt - 1) pre[nblk] = before;
    __syncthreads();
    const int total = pre[nblk];
    float* buf = out + static_cast<int64_t>(b) * (1 + 7 * static_cast<int64_t>(max_objects));
    if (threadIdx.x == 0) buf[0] = static_cast<float>(total);
    const int rows_out = min(total, max_objects);
    for (int r = threadIdx.x; r < rows_out; r += nt) {
        int lo = 0, hi = nblk;  // last block whose prefix is <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= r) lo = mid; else hi = mid;
        }
        const float* srow = stage + 7 * ((static_cast<int64_t>(b) * nblk + lo) * DC_APB + (r - pre[lo]));
        float* drow = buf + 1 + 7 * static_cast<int64_t>(r);
#pragma unroll
        for (int k = 0; k < 7; ++k) drow[k] = srow[k];
    }
}

constexpr unsigned long long DC_WAIT_NS = 10000000ull;  // 10 ms of global time before giving up
constexpr long long DC_WAIT_POLLS = 1ll << 26;              // and a poll count as a second bound
constexpr unsigned DC_COPY = 8192;                           // bytes per bulk copy (one per lane of warp 0)
// Every copy is issued by a lane of warp 0, the warp whose thread 0 set up the
// barrier (only a warp barrier lies between the two).
static_assert(4 * DC_APB * (5 + NMS_DECODE_MAX_CLASSES) <= 32 * DC_COPY,
              "a block's rows take at most 32 bulk copies");

__device__ __forceinline__ unsigned long long dc_now()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase 0 of the barrier at shared address sb: at most
// DC_WAIT_NS nanoseconds of the global timer (and DC_WAIT_POLLS polls).
__device__ __forceinline__ bool dc_wait(unsigned sb)
{
    const unsigned long long t0 = dc_now();
    for (long long k = 0; k < DC_WAIT_POLLS; ++k) {
        unsigned ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(sb)
            : "memory");
        if (ok) return true;
        if ((k & 15) == 15 && dc_now() - t0 > DC_WAIT_NS) break;
    }
    return false;
}

__global__ void __launch_bounds__(DC_APB)
decode_kernel(const float* __restrict__ preds, int anchors, int C, float conf_thr, int nblk,
              float* __restrict__ stage, int* __restrict__ blk_cnt, int32_t* status)
{
    extern __shared__ __align__(16) float rows[];  // DC_APB rows of 5 + C floats
    __shared__ int wcnt[DC_APB / 32];
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int s_ok;
    pdl_release();  // the emit may be scheduled; it waits for this grid
    const int b = blockIdx.y, blk = blockIdx.x;
    const int a0 = blk * DC_APB;
    const int na = min(DC_APB, anchors - a0);
    const int W = 5 + C;
    const float* src = preds + (static_cast<int64_t>(b) * anchors + a0) * W;
    const int nf = na * W;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (nf & 3) == 0) {
        // Bulk copies when the block's rows start on a 16-byte boundary (and
        // so, 16 bytes a row group, every copy's start and length): the whole
        // block's rows in flight at once, issued by a few lanes.  Thread 0
        // waits on the barrier (bounded) and the CTA barrier passes the rows
        // on; on a wait that gives up, the status says so, the copies still
        // in flight are waited for once more (bounded too) and the block
        // writes nothing.  If that second wait gives up as well, copies may
        // still be landing in the block's shared memory as it exits; the
        // call's buffers are then invalid, which NMS_ERR_TIMEOUT reports.
        const unsigned sb = static_cast<unsigned>(__cvta_generic_to_shared(&bar));
        const unsigned bytes = 4u * static_cast<unsigned>(nf);
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(sb));
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(sb), "r"(bytes) : "memory");
        }
        __syncwarp();
        const unsigned nch = (bytes + DC_COPY - 1) / DC_COPY;
        if (threadIdx.x < nch) {
            const unsigned off = threadIdx.x * DC_COPY, len = min(DC_COPY, bytes - off);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                    static_cast<unsigned>(__cvta_generic_to_shared(rows)) + off),
                "l"(reinterpret_cast<const char*>(src) + off), "r"(len), "r"(sb)
                : "memory");
        }
        if (threadIdx.x == 0) {
            const bool ok = dc_wait(sb);
            if (!ok) {
                set_status(status, NMS_ERR_TIMEOUT);
                dc_wait(sb);  // the copies in flight, once more
            }
            s_ok = ok;
        }
        __syncthreads();
        if (threadIdx.x == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(sb) : "memory");
        if (!s_ok) {
            if (threadIdx.x == 0) blk_cnt[static_cast<int64_t>(b) * nblk + blk] = 0;
            return;
        }
    } else {
#pragma unroll 4
        for (int e = threadIdx.x; e < nf; e += DC_APB) rows[e] = src[e];
    }
    __syncthreads();
    const int t = threadIdx.x;
    bool cand = false;
    float r[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (t < na) {
        const float* p = rows + t * W;
        int cls = 0;
        float best = p[5];
        for (int c = 1; c < C; ++c) {
            const float v = p[5 + c];
            if (v > best) {
                best = v;
                cls = c;
            }
        }
        const float conf = __fmul_rn(p[4], best);
        cand = conf > conf_thr;
        const float hw = __fmul_rn(p[2], 0.5f), hh = __fmul_rn(p[3], 0.5f);
        r[0] = __fsub_rn(p[0], hw);
        r[1] = __fsub_rn(p[1], hh);
        r[2] = __fadd_rn(p[0], hw);
        r[3] = __fadd_rn(p[1], hh);
        r[4] = conf;
        r[5] = static_cast<float>(cls);
    }
    const unsigned l = lane_id();
    const int w = t >> 5;
    const unsigned ball = __ballot_sync(FULL, cand);
    if (l == 0) wcnt[w] = __popc(ball);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int q = 0; q < DC_APB / 32; ++q) {
        before += q < w ? wcnt[q] : 0;
        total += wcnt[q];
    }
    const int64_t base = (static_cast<int64_t>(b) * nblk + blk) * DC_APB;
    if (cand) {
        float* dst = stage + 7 * (base + before + __popc(ball & ((1u << l) - 1u)));
#pragma unroll
        for (int k = 0; k < 6; ++k) dst[k] = r[k];
        dst[6] = 1.0f;
    }
    if (t == 0) blk_cnt[static_cast<int64_t>(b) * nblk + blk] = total;
}

// One CTA per image: its header and its first max_objects candidates (rows
// copied by many threads at once: each copy is a dependent L2 round trip).
constexpr int EM_THREADS = 1024;

__global__ void __launch_bounds__(EM_THREADS)
decode_emit_kernel(const float* __restrict__ stage, const int* __restrict__ blk_cnt, int nblk, int max_objects,
                   float* __restrict__ out)
{
    extern __shared__ int pre[];  // nblk + 1 prefixes
    __shared__ int wsum[EM_THREADS / 32];
    pdl_wait();
    emit_image(blockIdx.x, stage, blk_cnt, nblk, max_objects, out, pre, wsum);
}

__global__ void zero_headers_kernel(float* __restrict__ out, int batch, int max_objects)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) out[static_cast<int64_t>(b) * (1 + 7 * static_cast<int64_t>(max_objects))] = 0.0f;
}

int decode_blocks(int anchors) { return (anchors + DC_APB - 1) / DC_APB; }

void launch_decode(const float* preds, int batch, int anchors, int C, float conf_thr, int max_objects, float* out,
                   float* stage, int* blk_cnt, int32_t* status, cudaStream_t st)
{
    cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    const int nblk = decode_blocks(anchors);
    if (nblk == 0) {  // no anchors: every header is 0
        zero_headers_kernel<<<(batch + 255) / 256, 256, 0, st>>>(out, batch, max_objects);
        return;
    }
    const size_t smem = sizeof(float) * DC_APB * static_cast<size_t>(5 + C);
    ensure_dynamic_smem(reinterpret_cast<const void*>(decode_kernel), smem);
    decode_kernel<<<dim3(nblk, batch), DC_APB, smem, st>>>(preds, anchors, C, conf_thr, nblk, stage, blk_cnt,
                                                            status);
    const size_t esmem = sizeof(int) * (static_cast<size_t>(nblk) + 1);
    ensure_dynamic_smem(reinterpret_cast<const void*>(decode_emit_kernel), esmem);
    launch_pdl(decode_emit_kernel, dim3(batch), dim3(EM_THREADS), esmem, st, static_cast<const float*>(stage),
               static_cast<const int*>(blk_cnt), nblk, max_objects, out);
}

// ------------------------------------------------- NMS over count-header buffers

// Row r of image b -> batched inputs at b * max_objects + r.  Rows past
// min(header, max_objects) are placeholders that do not take part.  A class
// value that is not an integer in [0, C) becomes -1, which the batched path
// reports as NMS_ERR_INVALID_ARG.
__global__ void boxes7_gather_kernel(const float* __restrict__ bufs, int max_objects, int C,
                                     float4* __restrict__ boxes, float* __restrict__ scores,
                                     int32_t* __restrict__ cls, int64_t* __restrict__ off, int* __restrict__ img_rows,
                                     int batch)
{
    const int b = blockIdx.y;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    const float* buf = bufs + static_cast<int64_t>(b) * (1 + 7 * static_cast<int64_t>(max_objects));
    const float h = buf[0];
    const int m = h >= 1.0f ? static_cast<int>(fminf(h, static_cast<float>(max_objects))) : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        img_rows[b] = m;
        off[b] = static_cast<int64_t>(b) * max_objects;
        if (b == batch - 1) off[batch] = static_cast<int64_t>(batch) * max_objects;
    }
    if (r >= max_objects) return;
    const int64_t i = static_cast<int64_t>(b) * max_objects + r;
    if (r < m) {
        const float* row = buf + 1 + 7 * static_cast<int64_t>(r);
        boxes[i] = make_float4(row[0], row[1], row[2], row[3]);
        scores[i] = row[4];
        const float c = row[5];
        cls[i] = (c >= 0.0f && c < static_cast<float>(C) && c == floorf(c)) ? static_cast<int32_t>(c) : -1;
    } else {
        boxes[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        scores[i] = 0.0f;
        cls[i] = 0;
    }
}

// One CTA per image: keep_flag 0 for its live rows, then 1 for the kept ones.
__global__ void boxes7_flags_kernel(float* __restrict__ bufs, int max_objects, const int* __restrict__ img_rows,
                                    const int64_t* __restrict__ keep, const int64_t* __restrict__ counts)
{
    pdl_wait();
    const int b = blockIdx.x;
    float* buf = bufs + static_cast<int64_t>(b) * (1 + 7 * static_cast<int64_t>(max_objects));
    const int m = img_rows[b];
    for (int r = threadIdx.x; r < m; r += blockDim.x) buf[1 + 7 * static_cast<int64_t>(r) + 6] = 0.0f;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(b) * max_objects;
    const int64_t k = counts[b];
    for (int64_t q = threadIdx.x; q < k; q += blockDim.x) {
        const int64_t r = keep[base + q] - base;
        buf[1 + 7 * r + 6] = 1.0f;
    }
}

void launch_boxes7_gather(const float* bufs, int batch, int max_objects, int C, float4* boxes, float* scores,
                          int32_t* cls, int64_t* off, int* img_rows, cudaStream_t st)
{
    boxes7_gather_kernel<<<dim3((max_objects + 255) / 256 > 0 ? (max_objects + 255) / 256 : 1, batch), 256, 0, st>>>(
        bufs, max_objects, C, boxes, scores, cls, off, img_rows, batch);
}

void launch_boxes7_flags(float* bufs, int batch, int max_objects, const int* img_rows, const int64_t* keep,
                         const int64_t* counts, cudaStream_t st)
{
    launch_pdl(boxes7_flags_kernel, dim3(batch), dim3(256), 0, st, bufs, max_objects, img_rows, keep, counts);
}

}  // namespace gbnms
