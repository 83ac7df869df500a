// The C ABI of include/gbnms.h: argument checks, workspace layout and the
// launch sequence of each path.  No host synchronisation, no allocation.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace gbnms {

void ensure_dynamic_smem(const void* kernel, size_t bytes)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> limit;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = limit[{dev, kernel}];
    if (bytes <= have) return;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) ==
        cudaSuccess)
        have = bytes;
}

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Region offsets inside the caller's workspace.
struct Layout {
    size_t off[32] = {};
    size_t total = 0;
    int k = 0;
    size_t add(size_t bytes)
    {
        size_t o = total;
        total = align_up(total + (bytes ? bytes : 1));
        off[k++] = o;
        return o;
    }
};

struct SingleLayout {
    int64_t ldw = 0;
    int NB = 0;  // 64-bit words of the per-row chunk bitmap
    unsigned ecap = 0;   // pairs one CTA's graph path holds (0: no list, the walk resolves)
    unsigned lcap = 0;   // pairs the list holds (graph_list_cap: more than ecap when it fits)
    bool grid = false;   // the all-SM graph path exists at this size
    size_t status, m_count, ecount, done, cand, perm, boxes_s, keys, rowbits, edges, haspred, gstate,
        gctl, mask, total;
};

SingleLayout single_layout(int64_t n)
{
    SingleLayout s;
    const int64_t T = (n + 255) / 256;
    s.ldw = 4 * T;
    s.NB = static_cast<int>((T + 63) / 64 > 0 ? (T + 63) / 64 : 1);
    Layout L;
    s.ecap = graph_edge_cap(static_cast<int>(n));
    const unsigned gcap = graph_grid_cap(static_cast<int>(n));
    s.grid = gcap > s.ecap;
    s.lcap = graph_list_cap(static_cast<int>(n));
    s.status = L.add(4);
    s.m_count = L.add(4);
    s.ecount = L.add(4);
    s.done = L.add(4);
    s.cand = L.add(4 * static_cast<size_t>(n));
    s.perm = L.add(4 * static_cast<size_t>(n));
    s.boxes_s = L.add(16 * static_cast<size_t>(n));
    s.keys = L.add(sort_keys_bytes(static_cast<int>(n)));
    s.rowbits = L.add(8 * static_cast<size_t>(n) * static_cast<size_t>(s.NB));
    s.edges = L.add(4 * static_cast<size_t>(s.lcap));
    s.haspred = L.add(8 * static_cast<size_t>((n + 63) / 64));
    s.gstate = L.add(s.grid ? graph_grid_state_bytes(static_cast<int>(n)) : 0);
    s.gctl = L.add(s.grid ? graph_grid_ctl_bytes() : 0);
    s.mask = L.add(8 * static_cast<size_t>(n) * static_cast<size_t>(s.ldw));
    s.total = L.total;
    return s;
}

struct MatrixLayout {
    size_t status, m_count, cand, perm, boxes_s, keys, omax, xmin, fs, kept, done, list_count, colhi, list_ij,
        list_o, total;
};

MatrixLayout matrix_layout(int64_t n)
{
    MatrixLayout m;
    Layout L;
    const size_t N = static_cast<size_t>(n);
    m.status = L.add(4);
    m.m_count = L.add(4);
    m.cand = L.add(4 * N);
    m.perm = L.add(4 * N);
    m.boxes_s = L.add(16 * N);
    m.keys = L.add(sort_keys_bytes(static_cast<int>(n)));
    m.omax = L.add(4 * N);
    m.xmin = L.add(8 * N);
    m.fs = L.add(4 * N);
    m.kept = L.add(4 * ((N + 31) / 32 + 8));
    m.done = L.add(4);
    m.list_count = L.add(8);
    m.colhi = L.add(4 * N);
    m.list_ij = L.add(8 * static_cast<size_t>(matrix_list_cap(n)));
    m.list_o = L.add(4 * static_cast<size_t>(matrix_list_cap(n)));
    m.total = L.total;
    return m;
}

struct BatchedLayout {
    size_t status, ok, seg_cnt, seg_off, seg_of, slot, cand, kept_key, kept_cnt, sorted_key,
        sorted_box, stage, total;
};

BatchedLayout batched_layout(int64_t n, int64_t S)
{
    BatchedLayout b;
    Layout L;
    const size_t N = static_cast<size_t>(n);
    b.status = L.add(4);
    b.ok = L.add(4);
    b.seg_cnt = L.add(4 * static_cast<size_t>(S));
    b.seg_off = L.add(4 * static_cast<size_t>(S + 1));
    b.seg_of = L.add(4 * N);
    b.slot = L.add(4 * N);
    b.cand = L.add(4 * N);
    b.kept_key = L.add(8 * N);
    b.kept_cnt = L.add(4 * static_cast<size_t>(S));
    b.sorted_key = L.add(8 * N);
    b.sorted_box = L.add(16 * N);
    b.stage = L.add(8 * N);
    b.total = L.total;
    return b;
}

float next_down(float x) { return std::nextafter(x, -INFINITY); }

// Constants of the division-free test; the bounds are proved in common.cuh.
ThrParams make_thr(float thr)
{
    ThrParams p{};
    p.thr = thr;
    const double t = thr;
    p.fast_ok = (t >= 0x1p-20 && t <= 0x1p20) ? 1 : 0;
    p.k_lo = 0.0f;
    p.k2 = 0.0f;
    if (p.fast_ok) {
        const double T1 = t * (1.0 - 0x1p-21);
        const double k1 = T1 / (1.0 + T1) * (1.0 - 0x1p-22);
        float f1 = static_cast<float>(k1);
        if (static_cast<double>(f1) > k1) f1 = next_down(f1);
        p.k_lo = f1;
        const double k2 = 2.0 * static_cast<double>(f1) * (1.0 - 0x1p-20);  // exact in binary64
        float f2 = static_cast<float>(k2);
        if (static_cast<double>(f2) > k2) f2 = next_down(f2);
        p.k2 = f2;
    }
    return p;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename T>
T* at(void* base, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(base) + off); }

nms_status cuda_status()
{
    return cudaGetLastError() == cudaSuccess ? NMS_OK : NMS_ERR_CUDA;
}

}  // namespace
}  // namespace gbnms

using namespace gbnms;

extern "C" const char* nms_status_string(nms_status s)
{
    switch (s) {
        case NMS_OK: return "NMS_OK";
        case NMS_ERR_INVALID_ARG: return "NMS_ERR_INVALID_ARG";
        case NMS_ERR_WORKSPACE: return "NMS_ERR_WORKSPACE";
        case NMS_ERR_CAPACITY: return "NMS_ERR_CAPACITY";
        case NMS_ERR_CUDA: return "NMS_ERR_CUDA";
        case NMS_ERR_TIMEOUT: return "NMS_ERR_TIMEOUT";
    }
    return "NMS_ERR_UNKNOWN";
}

extern "C" nms_status nms_mapped_pointer(const void* host_ptr, void** device_ptr)
{
    if (!host_ptr || !device_ptr) return NMS_ERR_INVALID_ARG;
    *device_ptr = nullptr;
    cudaGetLastError();
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, host_ptr) != cudaSuccess) {
        cudaGetLastError();  // clear it: the pointer is simply not CUDA memory
        return NMS_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return NMS_ERR_INVALID_ARG;
    // The offset of host_ptr inside its allocation carries over to the mapping.
    const char* base_host = static_cast<const char*>(a.hostPointer);
    *device_ptr = static_cast<char*>(a.devicePointer) + (static_cast<const char*>(host_ptr) - base_host);
    return NMS_OK;
}

extern "C" nms_status nms_copy(void* dst, const void* src, size_t bytes, void* stream)
{
    if (bytes == 0) return NMS_OK;
    if (!dst || !src) return NMS_ERR_INVALID_ARG;
    cudaGetLastError();
    launch_copy(dst, src, bytes, static_cast<cudaStream_t>(stream));
    return cuda_status();
}

extern "C" nms_status nms_workspace_size(int64_t n, int32_t batch, int32_t num_classes,
                                         size_t* bytes)
{
    if (!bytes || n < 0 || n > INT32_MAX || batch < 0 || num_classes < 0) return NMS_ERR_INVALID_ARG;
    if (batch == 0 && num_classes == 0) {
        if (n > NMS_MAX_SINGLE_N) return NMS_ERR_CAPACITY;
        *bytes = single_layout(n).total;
        return NMS_OK;
    }
    const int64_t S = static_cast<int64_t>(batch > 0 ? batch : 1) * (num_classes > 0 ? num_classes : 1);
    if (S > INT32_MAX / 2) return NMS_ERR_INVALID_ARG;
    *bytes = batched_layout(n, S).total;
    return NMS_OK;
}

extern "C" int64_t nms_mask_row_words(int64_t n)
{
    return n <= 0 ? 0 : 4 * ((n + 255) / 256);
}

namespace {

nms_status run_impl(const float* boxes, const float* scores, int64_t n, const int32_t* class_ids,
                    int32_t num_classes, const int64_t* batch_offsets, int32_t batch, float iou_thr,
                    float score_thr, int32_t max_out, int64_t* keep, int64_t keep_cap,
                    int64_t* counts, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                    void* stream, const Stamps& stamps, bool fast = false)
{
    if (n < 0 || n > INT32_MAX) return NMS_ERR_INVALID_ARG;
    if (std::isnan(iou_thr) || std::isnan(score_thr)) return NMS_ERR_INVALID_ARG;
    if (n > 0 && (!boxes || !scores || !aligned(boxes, 16))) return NMS_ERR_INVALID_ARG;
    if (!keep || !counts) return NMS_ERR_INVALID_ARG;
    if (class_ids && num_classes < 1) return NMS_ERR_INVALID_ARG;
    if (batch_offsets && batch < 1) return NMS_ERR_INVALID_ARG;
    if (keep_cap < 0) return NMS_ERR_INVALID_ARG;
    const int B = batch_offsets ? batch : 1;
    const int C = class_ids ? num_classes : 1;
    const bool single = !class_ids && !batch_offsets;
    int64_t need = max_out > 0 ? static_cast<int64_t>(B) * max_out : n;
    if (single && max_out > 0) need = n < max_out ? n : max_out;
    if (keep_cap < need) return NMS_ERR_CAPACITY;
    if (single && n > NMS_MAX_SINGLE_N) return NMS_ERR_CAPACITY;
    const int64_t S64 = static_cast<int64_t>(B) * C;
    if (S64 > INT32_MAX / 2) return NMS_ERR_INVALID_ARG;
    size_t need_ws = 0;
    nms_status st0 = nms_workspace_size(n, batch_offsets ? batch : 0, class_ids ? num_classes : 0, &need_ws);
    if (st0 != NMS_OK) return st0;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < need_ws) return NMS_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();  // clear any stale error of this runtime
    const bool use_thr = !(std::isinf(score_thr) && score_thr < 0);

    if (single) {
        const SingleLayout L = single_layout(n);
        int32_t* status = dev_status ? dev_status : at<int32_t>(workspace, L.status);
        if (n == 0) {
            stamps.record(0, st);
            cudaMemsetAsync(counts, 0, sizeof(int64_t), st);
            cudaMemsetAsync(status, 0, sizeof(int32_t), st);
            for (int k = 1; k <= 3; ++k) stamps.record(k, st);
            return cuda_status();
        }
        const ThrParams p = make_thr(iou_thr);
        int* m_count = nullptr;
        int* cand = nullptr;
        stamps.record(0, st);
        if (use_thr) {
            m_count = at<int>(workspace, L.m_count);
            cand = at<int>(workspace, L.cand);
            launch_prefilter(scores, static_cast<int>(n), score_thr, cand, m_count, st);
        }
        int* perm = at<int>(workspace, L.perm);
        float4* boxes_s = at<float4>(workspace, L.boxes_s);
        uint64_t* mask = at<uint64_t>(workspace, L.mask);
        uint64_t* rowbits = at<uint64_t>(workspace, L.rowbits);
        uint64_t* haspred = at<uint64_t>(workspace, L.haspred);
        if (fast) {
            // Fast NMS ("YOLOv5后处理GPU移植实战" 2.2): the boxes with no earlier
            // box over the threshold, i.e. the clear bits of haspred.
            launch_sort(scores, reinterpret_cast<const float4*>(boxes), cand, m_count, static_cast<int>(n),
                        perm, boxes_s, sort_keys_bytes(static_cast<int>(n)) ? at<uint64_t>(workspace, L.keys)
                                                                            : nullptr,
                        status, nullptr, L.NB, nullptr, haspred, nullptr, st);
            stamps.record(1, st);
            // With max_out, the mask of the leading 2*max_out boxes first;
            // the rest only if that prefix held fewer than max_out kept boxes.
            const int64_t kf = max_out > 0 ? (2 * static_cast<int64_t>(max_out) + MASK_TILE_W - 1) /
                                                 MASK_TILE_W * MASK_TILE_W
                                           : n;
            if (kf >= n) {
                launch_iou_mask(boxes_s, m_count, static_cast<int>(n), p, nullptr, L.ldw, nullptr, L.NB, nullptr,
                                nullptr, 0u, haspred, st);
            } else {
                int* done = at<int>(workspace, L.done);
                const int k = static_cast<int>(kf), nb = static_cast<int>(n);
                launch_iou_mask(boxes_s, m_count, nb, p, nullptr, L.ldw, nullptr, L.NB, nullptr, nullptr, 0u,
                                haspred, st, 0, k);
                launch_fast_prefix(haspred, m_count, nb, k, max_out, done, st);
                launch_iou_mask(boxes_s, m_count, nb, p, nullptr, L.ldw, nullptr, L.NB, nullptr, nullptr, 0u,
                                haspred, st, k, nb, done);
            }
            stamps.record(2, st);
            launch_fast_emit(haspred, m_count, static_cast<int>(n), perm, max_out, keep, counts, st);
            stamps.record(3, st);
            return cuda_status();
        }
        uint32_t* edges = L.ecap ? at<uint32_t>(workspace, L.edges) : nullptr;
        unsigned* ecount = at<unsigned>(workspace, L.ecount);
        if (!L.ecap) haspred = nullptr;  // the walk needs no neighbour bitmap
        uint64_t* keys = sort_keys_bytes(static_cast<int>(n)) ? at<uint64_t>(workspace, L.keys) : nullptr;
        // The all-SM path's control block: its first 8 ints (barrier count,
        // round flags, per-stage "resolved" flags at 4..7) are zeroed by the sort.
        int* gctl = L.grid ? at<int>(workspace, L.gctl) : nullptr;
        launch_sort(scores, reinterpret_cast<const float4*>(boxes), cand, m_count, static_cast<int>(n),
                    perm, boxes_s, keys, status, rowbits, L.NB, ecount, haspred, gctl, st);
        stamps.record(1, st);
        const int nb = static_cast<int>(n);
        // With max_out, the first kept boxes depend only on a prefix of the
        // score order: mask and resolve the leading 2*max_out boxes first, and
        // the rest only if that prefix held fewer than max_out kept boxes (the
        // later launches find the device flag set and return at once).
        const int64_t k1 = max_out > 0 ? (2 * static_cast<int64_t>(max_out) + MASK_TILE_W - 1) /
                                             MASK_TILE_W * MASK_TILE_W
                                       : n;
        uint64_t* gstate = L.grid ? at<uint64_t>(workspace, L.gstate) : nullptr;
        // Resolve of one stage: with a list too long for one CTA, the all-SM
        // graph path first; one CTA's graph path or the walk otherwise.
        auto resolve = [&](int limit, const int* done_in, int* done_out, int stage) {
            const int* gd = nullptr;
            if (L.grid && limit > graph_grid_min_n()) {
                launch_graph_grid(edges, ecount, haspred, m_count, nb, perm, max_out, keep, counts, status, st,
                                  limit, done_in, done_out, gctl + 4 + stage, gstate, gctl);
                gd = gctl + 4 + stage;
            }
            launch_resolve_single(mask, L.ldw, rowbits, L.NB, edges, ecount, L.lcap, haspred, m_count, nb, perm,
                                  max_out, keep, counts, status, st, limit, done_in, done_out, gd);
        };
        if (k1 >= n) {
            launch_iou_mask(boxes_s, m_count, nb, p, mask, L.ldw, rowbits, L.NB, edges, ecount,
                            L.lcap, haspred, st);
            stamps.record(2, st);
            resolve(1 << 30, nullptr, nullptr, 0);
        } else {
            int* done = at<int>(workspace, L.done);
            const int k = static_cast<int>(k1);
            launch_iou_mask(boxes_s, m_count, nb, p, mask, L.ldw, rowbits, L.NB, edges, ecount,
                            L.lcap, haspred, st, 0, k);
            stamps.record(2, st);
            resolve(k, nullptr, done, 0);
            launch_iou_mask(boxes_s, m_count, nb, p, mask, L.ldw, rowbits, L.NB, edges, ecount,
                            L.lcap, haspred, st, k, nb, done);
            resolve(1 << 30, done, nullptr, 1);
        }
        stamps.record(3, st);
        return cuda_status();
    }

    const BatchedLayout L = batched_layout(n, S64);
    BatchedArgs a{};
    a.boxes = reinterpret_cast<const float4*>(boxes);
    a.scores = scores;
    a.cls = class_ids;
    a.C = C;
    a.off = batch_offsets;
    a.batch = B;
    a.n = static_cast<int>(n);
    a.S = static_cast<int>(S64);
    a.use_thr = use_thr ? 1 : 0;
    a.score_thr = score_thr;
    a.thr = iou_thr;
    a.max_out = max_out;
    a.fast = fast ? 1 : 0;
    a.seg_cnt = at<int>(workspace, L.seg_cnt);
    a.seg_off = at<int>(workspace, L.seg_off);
    a.seg_of = at<int>(workspace, L.seg_of);
    a.slot = at<int>(workspace, L.slot);
    a.cand = at<int>(workspace, L.cand);
    a.ok = at<int>(workspace, L.ok);
    a.kept_key = at<uint64_t>(workspace, L.kept_key);
    a.kept_cnt = at<int>(workspace, L.kept_cnt);
    a.sorted_key = at<uint64_t>(workspace, L.sorted_key);
    a.sorted_box = at<float4>(workspace, L.sorted_box);
    a.stage = at<uint64_t>(workspace, L.stage);
    a.keep = keep;
    a.counts = counts;
    a.status = dev_status ? dev_status : at<int32_t>(workspace, L.status);
    launch_batched(a, st, stamps);
    return cuda_status();
}

}  // namespace

extern "C" nms_status nms_run(const float* boxes, const float* scores, int64_t n,
                              const int32_t* class_ids, int32_t num_classes,
                              const int64_t* batch_offsets, int32_t batch, float iou_thr,
                              float score_thr, int32_t max_out, int64_t* keep, int64_t keep_cap,
                              int64_t* counts, int32_t* dev_status, void* workspace,
                              size_t workspace_bytes, void* stream)
{
    return run_impl(boxes, scores, n, class_ids, num_classes, batch_offsets, batch, iou_thr,
                    score_thr, max_out, keep, keep_cap, counts, dev_status, workspace,
                    workspace_bytes, stream, Stamps{});
}

extern "C" nms_status nms_fast_run(const float* boxes, const float* scores, int64_t n,
                                   const int32_t* class_ids, int32_t num_classes,
                                   const int64_t* batch_offsets, int32_t batch, float iou_thr,
                                   float score_thr, int32_t max_out, int64_t* keep, int64_t keep_cap,
                                   int64_t* counts, int32_t* dev_status, void* workspace,
                                   size_t workspace_bytes, void* stream)
{
    return run_impl(boxes, scores, n, class_ids, num_classes, batch_offsets, batch, iou_thr,
                    score_thr, max_out, keep, keep_cap, counts, dev_status, workspace,
                    workspace_bytes, stream, Stamps{}, true);
}

extern "C" nms_status nms_matrix_workspace_size(int64_t n, size_t* bytes)
{
    if (!bytes || n < 0) return NMS_ERR_INVALID_ARG;
    if (n > NMS_MAX_SINGLE_N) return NMS_ERR_CAPACITY;
    *bytes = matrix_layout(n).total;
    return NMS_OK;
}

extern "C" nms_status nms_matrix_run(const float* boxes, const float* scores, int64_t n, int32_t decay,
                                     float sigma, float score_thr, float decay_thr, int32_t max_out,
                                     int64_t* keep, float* keep_scores, int64_t keep_cap, int64_t* count,
                                     int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                     void* stream)
{
    if (n < 0) return NMS_ERR_INVALID_ARG;
    if (decay != NMS_DECAY_GAUSSIAN && decay != NMS_DECAY_LINEAR) return NMS_ERR_INVALID_ARG;
    if (decay == NMS_DECAY_GAUSSIAN && (!(sigma > 0.0f) || std::isinf(sigma))) return NMS_ERR_INVALID_ARG;
    if (std::isnan(score_thr) || std::isnan(decay_thr)) return NMS_ERR_INVALID_ARG;
    if (n > 0 && (!boxes || !scores || !aligned(boxes, 16))) return NMS_ERR_INVALID_ARG;
    if (!keep || !count || keep_cap < 0) return NMS_ERR_INVALID_ARG;
    if (n > NMS_MAX_SINGLE_N) return NMS_ERR_CAPACITY;
    const int64_t need = max_out > 0 ? (n < max_out ? n : max_out) : n;
    if (keep_cap < need) return NMS_ERR_CAPACITY;
    const MatrixLayout L = matrix_layout(n);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < L.total) return NMS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    int32_t* status = dev_status ? dev_status : at<int32_t>(workspace, L.status);
    if (n == 0) {
        cudaMemsetAsync(count, 0, sizeof(int64_t), st);
        cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        return cuda_status();
    }
    const bool use_thr = !(std::isinf(score_thr) && score_thr < 0);
    int* m_count = nullptr;
    int* cand = nullptr;
    if (use_thr) {
        m_count = at<int>(workspace, L.m_count);
        cand = at<int>(workspace, L.cand);
        launch_prefilter(scores, static_cast<int>(n), score_thr, cand, m_count, st);
    }
    int* perm = at<int>(workspace, L.perm);
    float4* boxes_s = at<float4>(workspace, L.boxes_s);
    uint64_t* keys = sort_keys_bytes(static_cast<int>(n)) ? at<uint64_t>(workspace, L.keys) : nullptr;
    launch_sort(scores, reinterpret_cast<const float4*>(boxes), cand, m_count, static_cast<int>(n), perm, boxes_s,
                keys, status, nullptr, 1, nullptr, nullptr, nullptr, st);
    launch_matrix(boxes_s, scores, perm, m_count, static_cast<int>(n), sigma, decay == NMS_DECAY_LINEAR ? 1 : 0,
                  decay_thr, max_out,
                  at<unsigned>(workspace, L.omax), at<unsigned long long>(workspace, L.xmin),
                  at<float>(workspace, L.fs), at<uint32_t>(workspace, L.kept), at<int>(workspace, L.done),
                  at<unsigned long long>(workspace, L.list_ij), at<float>(workspace, L.list_o),
                  at<unsigned long long>(workspace, L.list_count), matrix_list_cap(n),
                  at<unsigned>(workspace, L.colhi), keep,
                  keep_scores, count, st);
    return cuda_status();
}

namespace gbnms {
namespace {

struct DecodeLayout {
    size_t status, stage, blk_cnt, total;
};

DecodeLayout decode_layout(int32_t batch, int32_t anchors)
{
    DecodeLayout d;
    Layout L;
    const size_t slots = static_cast<size_t>(batch) * decode_blocks(anchors) * 128;
    d.status = L.add(sizeof(int32_t));
    d.stage = L.add(7 * sizeof(float) * slots);
    d.blk_cnt = L.add(sizeof(int) * static_cast<size_t>(batch) * decode_blocks(anchors));
    d.total = L.total;
    return d;
}

struct Boxes7Layout {
    BatchedLayout batched;
    size_t boxes, scores, cls, off, img_rows, keep, counts, total;
};

Boxes7Layout boxes7_layout(int32_t batch, int32_t max_objects, int32_t num_classes)
{
    Boxes7Layout b;
    const int64_t n = static_cast<int64_t>(batch) * max_objects;
    b.batched = batched_layout(n, static_cast<int64_t>(batch) * num_classes);
    Layout L;
    L.total = align_up(b.batched.total);
    const size_t N = static_cast<size_t>(n > 0 ? n : 1);
    b.boxes = L.add(16 * N);
    b.scores = L.add(4 * N);
    b.cls = L.add(4 * N);
    b.off = L.add(8 * (static_cast<size_t>(batch) + 1));
    b.img_rows = L.add(4 * static_cast<size_t>(batch));
    b.keep = L.add(8 * N);
    b.counts = L.add(8 * static_cast<size_t>(batch));
    b.total = L.total;
    return b;
}

}  // namespace
}  // namespace gbnms

extern "C" nms_status nms_decode_workspace_size(int32_t batch, int32_t anchors, size_t* bytes)
{
    if (!bytes || batch < 1 || anchors < 0) return NMS_ERR_INVALID_ARG;
    if (anchors > NMS_DECODE_MAX_ANCHORS || batch > NMS_DECODE_MAX_BATCH) return NMS_ERR_CAPACITY;
    *bytes = decode_layout(batch, anchors).total;
    return NMS_OK;
}

extern "C" nms_status nms_decode_boxes7(const float* preds, int32_t batch, int32_t anchors, int32_t num_classes,
                                        float conf_thr, int32_t max_objects, float* buffers, int32_t* dev_status,
                                        void* workspace, size_t workspace_bytes, void* stream)
{
    if (batch < 1 || anchors < 0 || num_classes < 1 || max_objects < 0 || std::isnan(conf_thr))
        return NMS_ERR_INVALID_ARG;
    if (anchors > NMS_DECODE_MAX_ANCHORS || num_classes > NMS_DECODE_MAX_CLASSES || batch > NMS_DECODE_MAX_BATCH)
        return NMS_ERR_CAPACITY;
    if (!buffers || (anchors > 0 && (!preds || !aligned(preds, 4)))) return NMS_ERR_INVALID_ARG;
    const DecodeLayout L = decode_layout(batch, anchors);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < L.total) return NMS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    launch_decode(preds, batch, anchors, num_classes, conf_thr, max_objects, buffers,
                  at<float>(workspace, L.stage), at<int>(workspace, L.blk_cnt),
                  dev_status ? dev_status : at<int32_t>(workspace, L.status), st);
    return cuda_status();
}

extern "C" nms_status nms_boxes7_workspace_size(int32_t batch, int32_t max_objects, int32_t num_classes,
                                                size_t* bytes)
{
    if (!bytes || batch < 1 || max_objects < 0 || num_classes < 1) return NMS_ERR_INVALID_ARG;
    if (static_cast<int64_t>(batch) * max_objects > INT32_MAX ||
        static_cast<int64_t>(batch) * num_classes > INT32_MAX / 2)
        return NMS_ERR_INVALID_ARG;
    if (batch > NMS_DECODE_MAX_BATCH) return NMS_ERR_CAPACITY;
    *bytes = boxes7_layout(batch, max_objects, num_classes).total;
    return NMS_OK;
}

extern "C" nms_status nms_boxes7_run(float* buffers, int32_t batch, int32_t max_objects, int32_t num_classes,
                                     float iou_thr, int32_t fast, int32_t* dev_status, void* workspace,
                                     size_t workspace_bytes, void* stream)
{
    size_t need = 0;
    const nms_status s0 = nms_boxes7_workspace_size(batch, max_objects, num_classes, &need);
    if (s0 != NMS_OK) return s0;
    if (!buffers || std::isnan(iou_thr) || (fast != 0 && fast != 1)) return NMS_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < need) return NMS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    const Boxes7Layout L = boxes7_layout(batch, max_objects, num_classes);
    float4* boxes = at<float4>(workspace, L.boxes);
    float* scores = at<float>(workspace, L.scores);
    int32_t* cls = at<int32_t>(workspace, L.cls);
    int64_t* off = at<int64_t>(workspace, L.off);
    int* img_rows = at<int>(workspace, L.img_rows);
    int64_t* keep = at<int64_t>(workspace, L.keep);
    int64_t* counts = at<int64_t>(workspace, L.counts);
    launch_boxes7_gather(buffers, batch, max_objects, num_classes, boxes, scores, cls, off, img_rows, st);
    const BatchedLayout& B = L.batched;
    BatchedArgs a{};
    a.boxes = boxes;
    a.scores = scores;
    a.cls = cls;
    a.C = num_classes;
    a.off = off;
    a.batch = batch;
    a.n = batch * max_objects;
    a.S = batch * num_classes;
    a.use_thr = 0;
    a.score_thr = 0.0f;
    a.thr = iou_thr;
    a.max_out = 0;
    a.fast = fast;
    a.img_rows = img_rows;
    a.seg_cnt = at<int>(workspace, B.seg_cnt);
    a.seg_off = at<int>(workspace, B.seg_off);
    a.seg_of = at<int>(workspace, B.seg_of);
    a.slot = at<int>(workspace, B.slot);
    a.cand = at<int>(workspace, B.cand);
    a.ok = at<int>(workspace, B.ok);
    a.kept_key = at<uint64_t>(workspace, B.kept_key);
    a.kept_cnt = at<int>(workspace, B.kept_cnt);
    a.sorted_key = at<uint64_t>(workspace, B.sorted_key);
    a.sorted_box = at<float4>(workspace, B.sorted_box);
    a.stage = at<uint64_t>(workspace, B.stage);
    a.keep = keep;
    a.counts = counts;
    a.status = dev_status ? dev_status : at<int32_t>(workspace, B.status);
    launch_batched(a, st, Stamps{});
    launch_boxes7_flags(buffers, batch, max_objects, img_rows, keep, counts, st);
    return cuda_status();
}

extern "C" nms_status nms_run_timed(const float* boxes, const float* scores, int64_t n,
                                    const int32_t* class_ids, int32_t num_classes,
                                    const int64_t* batch_offsets, int32_t batch, float iou_thr,
                                    float score_thr, int32_t max_out, int64_t* keep,
                                    int64_t keep_cap, int64_t* counts, int32_t* dev_status,
                                    void* workspace, size_t workspace_bytes, void* stream,
                                    void* const* events, int32_t nevents)
{
    Stamps sp;
    sp.ev = events;
    sp.n = events && nevents > 0 ? nevents : 0;
    // Plain launches between the stage events (see pdl_disabled).
    struct NoPdl {
        bool prev = pdl_disabled();
        NoPdl() { pdl_disabled() = true; }
        ~NoPdl() { pdl_disabled() = prev; }
    } no_pdl;
    return run_impl(boxes, scores, n, class_ids, num_classes, batch_offsets, batch, iou_thr,
                    score_thr, max_out, keep, keep_cap, counts, dev_status, workspace,
                    workspace_bytes, stream, sp);
}

namespace {

struct LaneLayout {
    SingleLayout s;
    size_t xs, span, flag, pre_planes, pre_count, pre_edges, total;
    size_t plane = 0;  // bytes of each prepass byte plane
};

LaneLayout lane_layout(int64_t n)
{
    LaneLayout L;
    L.s = single_layout(n);
    Layout X;
    X.total = L.s.total;
    const size_t ld = static_cast<size_t>(lane_ld(static_cast<int>(n)));
    L.xs = X.add(4 * static_cast<size_t>(NMS_LANE_ROWS) * ld);
    L.span = X.add(4 * ld);
    L.flag = X.add(4 * ld);
    // The graph prepass (lane lists are dense cliques): its removed and
    // blocked planes, its pair count and the pairs it leaves.
    L.plane = graph_pre_plane_bytes(static_cast<int>(n));
    L.pre_planes = X.add(2 * L.plane);
    L.pre_count = X.add(4);
    L.pre_edges = X.add(4 * static_cast<size_t>(L.s.lcap));
    L.total = X.total;
    return L;
}

}  // namespace

extern "C" nms_status nms_lane_workspace_size(int64_t n, size_t* bytes)
{
    if (!bytes || n < 0) return NMS_ERR_INVALID_ARG;
    if (n > NMS_LANE_MAX_N) return NMS_ERR_CAPACITY;
    *bytes = lane_layout(n).total;
    return NMS_OK;
}

extern "C" nms_status nms_lane_run(const float* props, const float* scores, int64_t n, float dist_thr,
                                   int32_t max_out, int64_t* keep, int64_t keep_cap, int64_t* count,
                                   int32_t* dev_status, void* workspace, size_t workspace_bytes, void* stream)
{
    if (n < 0 || std::isnan(dist_thr)) return NMS_ERR_INVALID_ARG;
    if (n > NMS_LANE_MAX_N) return NMS_ERR_CAPACITY;
    if (!count || !aligned(count, 8)) return NMS_ERR_INVALID_ARG;
    if (n > 0 && (!props || !scores || !keep || !aligned(props, 4) || !aligned(scores, 4) || !aligned(keep, 8)))
        return NMS_ERR_INVALID_ARG;
    if (dev_status && !aligned(dev_status, 4)) return NMS_ERR_INVALID_ARG;
    const int64_t need = max_out > 0 ? (n < max_out ? n : max_out) : n;
    if (keep_cap < need) return NMS_ERR_CAPACITY;
    const LaneLayout L = lane_layout(n);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < L.total) return NMS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    int32_t* status = dev_status ? dev_status : at<int32_t>(workspace, L.s.status);
    if (n == 0) {
        cudaMemsetAsync(count, 0, sizeof(int64_t), st);
        cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        return cuda_status();
    }
    const int nb = static_cast<int>(n);
    int* perm = at<int>(workspace, L.s.perm);
    uint64_t* mask = at<uint64_t>(workspace, L.s.mask);
    uint64_t* rowbits = at<uint64_t>(workspace, L.s.rowbits);
    uint64_t* haspred = at<uint64_t>(workspace, L.s.haspred);
    uint32_t* edges = L.s.ecap ? at<uint32_t>(workspace, L.s.edges) : nullptr;
    unsigned* ecount = at<unsigned>(workspace, L.s.ecount);
    uint64_t* keys = sort_keys_bytes(nb) ? at<uint64_t>(workspace, L.s.keys) : nullptr;
    // Sort only (no boxes to gather); it also zeroes the status, the pair
    // count, the per-row chunk bits and the neighbour bitmap.
    launch_sort(scores, nullptr, nullptr, nullptr, nb, perm, nullptr, keys, status, rowbits, L.s.NB, ecount,
                haspred, nullptr, st);
    GraphPre pre{};
    if (edges) {
        pre.edges = at<uint32_t>(workspace, L.pre_edges);
        pre.ecount = at<unsigned>(workspace, L.pre_count);
        pre.cap = L.s.lcap;
        pre.removed = at<uint8_t>(workspace, L.pre_planes);
        pre.blocked = pre.removed + L.plane;
    }
    launch_lane_mask(props, perm, nb, dist_thr, at<float>(workspace, L.xs), at<uint32_t>(workspace, L.span),
                     at<uint32_t>(workspace, L.flag), mask, L.s.ldw, rowbits, L.s.NB, edges, ecount, L.s.lcap,
                     L.s.ecap ? haspred : nullptr, st, edges ? pre.removed : nullptr, 2 * L.plane, pre.ecount);
    if (edges) launch_graph_prepass(edges, ecount, L.s.lcap, haspred, nb, pre, st);
    launch_resolve_single(mask, L.s.ldw, rowbits, L.s.NB, edges, ecount, L.s.lcap, L.s.ecap ? haspred : nullptr,
                          nullptr, nb, perm, max_out, keep, count, status, st, 1 << 30, nullptr, nullptr, nullptr,
                          edges ? &pre : nullptr);
    return cuda_status();
}

extern "C" nms_status nms_iou_mask(const float* boxes_sorted, int64_t n, float iou_thr,
                                   uint64_t* mask, int64_t mask_words, void* stream)
{
    if (n < 0 || std::isnan(iou_thr)) return NMS_ERR_INVALID_ARG;
    if (n > NMS_MAX_SINGLE_N) return NMS_ERR_CAPACITY;
    if (n == 0) return NMS_OK;
    if (!boxes_sorted || !mask || !aligned(boxes_sorted, 16) || !aligned(mask, 16))
        return NMS_ERR_INVALID_ARG;
    const int64_t ldw = nms_mask_row_words(n);
    if (mask_words < n * ldw) return NMS_ERR_CAPACITY;
    cudaGetLastError();
    launch_iou_mask(reinterpret_cast<const float4*>(boxes_sorted), nullptr, static_cast<int>(n),
                    make_thr(iou_thr), mask, ldw, nullptr, 1, nullptr, nullptr, 0u, nullptr,
                    static_cast<cudaStream_t>(stream));
    return cuda_status();
}

extern "C" nms_status nms_resolve_mask(const uint64_t* mask, int64_t n, const int32_t* perm,
                                       int32_t max_out, int64_t* keep, int64_t* count,
                                       void* workspace, size_t workspace_bytes, void* stream)
{
    if (n < 0) return NMS_ERR_INVALID_ARG;
    if (n > NMS_MAX_SINGLE_N) return NMS_ERR_CAPACITY;
    if (!count || !aligned(count, 8) || (n > 0 && (!mask || !keep || !aligned(mask, 16) || !aligned(keep, 8) ||
                                                   (perm && !aligned(perm, 4)))))
        return NMS_ERR_INVALID_ARG;
    const SingleLayout L = single_layout(n);
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < L.total) return NMS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    if (n == 0) {
        cudaMemsetAsync(count, 0, sizeof(int64_t), st);
        return cuda_status();
    }
    launch_resolve_single(mask, L.ldw, nullptr, 1, nullptr, nullptr, 0u, nullptr, nullptr,
                          static_cast<int>(n), perm, max_out, keep, count, nullptr, st);
    return cuda_status();
}
