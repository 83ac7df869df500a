// Host-side launchers shared between the translation units of the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gbnms {

struct ThrParams;

// Caller's stage events of nms_run_timed: record(k) records events[k] on the
// stream when present.
struct Stamps {
    void* const* ev = nullptr;
    int n = 0;
    void record(int k, cudaStream_t st) const
    {
        if (k < n && ev && ev[k]) cudaEventRecord(static_cast<cudaEvent_t>(ev[k]), st);
    }
};

// Launch attribute that lets a kernel be scheduled while its predecessor in
// the stream finishes (the kernel calls pdl_wait() before reading the
// predecessor's output).
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute a{};
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// Whether this host thread's launches leave out the programmatic-dependent
// launch attribute (nms_run_timed sets it for its call: its stage events sit
// between the kernels, so no kernel could start early anyway, and stage
// durations are then measured on plain launches).
inline bool& pdl_disabled()
{
    static thread_local bool off = false;
    return off;
}
inline unsigned pdl_attr_count() { return pdl_disabled() ? 0u : 1u; }

// Launch with pdl_attribute() (unless disabled for this thread).
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl_attr_count();
    cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the runtime is called only when the limit recorded for
// that (device, kernel) is lower, so repeated launches pay nothing.
void ensure_dynamic_smem(const void* kernel, size_t bytes);

void launch_prefilter(const float* scores, int n, float score_thr, int* cand, int* m_count,
                      cudaStream_t st);
size_t sort_keys_bytes(int m_bound);
// Sort of the candidates' score keys into perm; with boxes, their boxes are
// gathered into boxes_s in the same order (boxes may be NULL: perm only).
void launch_sort(const float* scores, const float4* boxes, const int* cand, const int* m_dev,
                 int m_bound, int* perm, float4* boxes_s, uint64_t* keys, int32_t* status,
                 uint64_t* rowbits, int NB, unsigned* ecount, uint64_t* haspred, int* zero8, cudaStream_t st);
int64_t mask_tiles(int64_t n);
// Tile width of the mask kernel (columns); stages of the max_out early exit
// start on a multiple of it.
#ifndef GBNMS_MASK_MT
#define GBNMS_MASK_MT 128
#endif
constexpr int MASK_TILE_W = GBNMS_MASK_MT;

// Mask tiles whose columns lie in [col_lo, min(col_hi, m_bound)); with `done`
// set on the device the launch does nothing.
void launch_iou_mask(const float4* boxes_s, const int* m_dev, int m_bound, const ThrParams& p,
                     uint64_t* mask, int64_t ldw, uint64_t* rowbits, int NB,
                     uint32_t* edges, unsigned* ecount, unsigned ecap, uint64_t* haspred,
                     cudaStream_t st, int col_lo = 0, int col_hi = 1 << 30, const int* done = nullptr);
size_t resolve_smem_bytes(int m_bound, int NB);
unsigned graph_edge_cap(int m_bound);
// Passes 0 and 1 of the graph resolve over all SMs (launch_graph_prepass):
// the pairs left after them (edges, up to cap, their count in *ecount), the
// removed byte of each box after pass 0 (removed) and a 3 for each box that
// pass 1 blocked (blocked).  removed and blocked hold 32 * ((n + 127) / 128
// * 4) bytes each; they and *ecount must be zero before the mask runs.
struct GraphPre {
    uint32_t* edges;
    unsigned* ecount;
    unsigned cap;
    uint8_t* removed;
    uint8_t* blocked;
};
inline size_t graph_pre_plane_bytes(int n) { return 32 * static_cast<size_t>(((n + 31) / 32 + 3) & ~3); }
// When the mask's list is complete (*ecount <= lcap) and longer than one
// CTA's shared memory (> graph_edge_cap): pass 0 stores removed = 1 for the
// target of every pair whose source has no source of its own; pass 1 keeps
// the pairs whose source has a source and is not removed, compacted into
// pre.edges, and stores blocked = 3 for their targets.  Otherwise nothing.
void launch_graph_prepass(const uint32_t* edges, const unsigned* ecount, unsigned lcap, const uint64_t* haspred,
                          int n, const GraphPre& pre, cudaStream_t st);

// Pairs the list of m_bound boxes holds: graph_grid_cap where the all-SM
// path exists, else up to 32 times graph_edge_cap (whose first passes the
// resolve runs from global memory).
unsigned graph_list_cap(int m_bound);
// Resolves boxes [0, min(n, limit)).  done_in set on the device: nothing to
// do; done_out: set to 1 when the call found max_out kept boxes or covered
// all n boxes (a later stage then has nothing to do).  lcap: the pairs the
// list edges holds; on the last stage, with no grid_done, a list longer than
// one CTA's shared memory is resolved from global memory (and compacted in
// place).  pre: launch_graph_prepass ran over the list (one stage, all n
// boxes), and the resolve starts from its results.
void launch_resolve_single(const uint64_t* mask, int64_t ldw, const uint64_t* rowbits, int NB,
                           uint32_t* edges, const unsigned* ecount, unsigned lcap,
                           const uint64_t* haspred, const int* m_dev, int m_bound, const int* perm,
                           int max_out, int64_t* keep, int64_t* counts, int32_t* status,
                           cudaStream_t st, int limit = 1 << 30, const int* done_in = nullptr,
                           int* done_out = nullptr, const int* grid_done = nullptr,
                           const GraphPre* pre = nullptr);

// Pair-list capacity of the all-SM graph path (0 below its size range) and
// its scratch: graph_grid_state_bytes of bitmaps and a control block.
unsigned graph_grid_cap(int m_bound);
size_t graph_grid_ctl_bytes();
int graph_grid_min_n();  // stages of at most this many boxes never take the all-SM path
// The control block starts with 8 ints that must be zero on entry (barrier
// count, round flags, per-stage "resolved" flags at ints 4..7).
inline size_t graph_grid_state_bytes(int m_bound) { return 16 * static_cast<size_t>(((m_bound + 31) / 32 + 3) & ~3); }
// Resolves boxes [0, min(n, limit)) over a pair list too long for one CTA
// (more than graph_edge_cap pairs, at most graph_grid_cap); on success sets
// *grid_done (and *done_out as launch_resolve_single would); otherwise leaves
// them for the walk.  The control block's barrier count and flags must be
// zero on entry.
void launch_graph_grid(uint32_t* edges, const unsigned* ecount, const uint64_t* haspred, const int* m_dev,
                       int m_bound, const int* perm, int max_out, int64_t* keep, int64_t* counts,
                       int32_t* status, cudaStream_t st, int limit, const int* done_in, int* done_out,
                       int* grid_done, uint64_t* state, void* ctl);

// Lane candidates (k_lane.cu): the SoA stride for n lanes, and the gather
// and mask launches over the sorted permutation (outputs in the layout of
// launch_iou_mask).  xs: 72 x lane_ld(n) floats; span, flag: lane_ld(n) each.
// The gather also zeroes zero_bytes (a multiple of 16, 16-byte aligned) at
// zero and *zcount.
int lane_ld(int n);
void launch_lane_mask(const float* props, const int* perm, int n, float thr, float* xs, uint32_t* span,
                      uint32_t* flag, uint64_t* mask, int64_t ldw, uint64_t* rowbits, int NB, uint32_t* edges,
                      unsigned* ecount, unsigned ecap, uint64_t* haspred, cudaStream_t st, void* zero = nullptr,
                      size_t zero_bytes = 0, unsigned* zcount = nullptr);

// Fast NMS output of one image: the boxes whose bit in haspred is clear, in
// sorted order, mapped through perm, cut at max_out.
void launch_kept_prefix(const uint32_t* kept, const int* m_dev, int m_bound, int k, int max_out, int* done,
                        cudaStream_t st);
void launch_fast_prefix(const uint64_t* haspred, const int* m_dev, int m_bound, int k, int max_out, int* done,
                        cudaStream_t st);
void launch_fast_emit(const uint64_t* haspred, const int* m_dev, int m_bound, const int* perm, int max_out,
                      int64_t* keep, int64_t* counts, cudaStream_t st);

// Ordered output of the set bits of `bits` (sorted positions) with fs[j]
// beside each (fs, keep_fs optional).
void launch_bits_emit(const uint32_t* bits, const int* m_dev, int m_bound, const int* perm, const float* fs,
                      int max_out, int64_t* keep, float* keep_fs, int64_t* counts, cudaStream_t st);

// Matrix NMS (Gaussian decay, or linear when `linear`) of the sorted boxes:
// zeroes its scratch, runs the two tiled passes, decides every box and writes
// the kept indices, their final scores and the count.  fs: n floats, kept:
// ceil(n/32) words of scratch.
void launch_matrix(const float4* boxes_s, const float* scores, const int* perm, const int* m_dev, int m_bound,
                   float sigma, int linear, float decay_thr, int max_out, unsigned* omax_bits,
                   unsigned long long* xmin_key, float* fs, uint32_t* kept, int* done, unsigned long long* list_ij,
                   float* list_o, unsigned long long* list_count, unsigned list_cap, unsigned* colhi, int64_t* keep,
                   float* keep_scores, int64_t* count, cudaStream_t st);
// Entries of the Matrix NMS list of overlapping pairs for n boxes.
unsigned matrix_list_cap(int64_t n);

// Front end (k_decode.cu): YOLO-shaped predictions to count-header buffers.
int decode_blocks(int anchors);
void launch_decode(const float* preds, int batch, int anchors, int C, float conf_thr, int max_objects, float* out,
                   float* stage, int* blk_cnt, int32_t* status, cudaStream_t st);
// NMS over count-header buffers: rows to batched inputs, then keep_flag.
void launch_boxes7_gather(const float* bufs, int batch, int max_objects, int C, float4* boxes, float* scores,
                          int32_t* cls, int64_t* off, int* img_rows, cudaStream_t st);
void launch_boxes7_flags(float* bufs, int batch, int max_objects, const int* img_rows, const int64_t* keep,
                         const int64_t* counts, cudaStream_t st);

struct BatchedArgs {
    const float4* boxes;
    const float* scores;
    const int32_t* cls;
    int C;
    const int64_t* off;
    int batch;
    int n;
    int S;
    int use_thr;
    float score_thr;
    float thr;
    int max_out;
    int fast;  // Fast NMS: drop a box any earlier box of its segment suppresses
    const int* img_rows;  // optional: only the first img_rows[b] rows of image b take part
    int* seg_cnt;
    int* seg_off;
    int* seg_of;
    int* slot;
    int* cand;
    int* ok;
    uint64_t* kept_key;
    int* kept_cnt;
    uint64_t* sorted_key;
    float4* sorted_box;
    uint64_t* stage;
    int64_t* keep;
    int64_t* counts;
    int32_t* status;
};

void launch_batched(const BatchedArgs& a, cudaStream_t st, const Stamps& stamps);

// dst[0..bytes) = src[0..bytes) by every SM (programmatic dependent launch;
// it waits for the previous kernel before writing dst).
void launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t st);

}  // namespace gbnms
