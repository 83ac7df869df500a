/*
 * gbnms: greedy IoU non-maximum suppression on GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; no PyTorch or C++ types cross it.
 * Every entry point returns an nms_status and never throws.  All device work
 * is enqueued on the caller's CUDA stream (`stream` is a cudaStream_t passed
 * as void*; NULL means the legacy default stream) and nms_run / nms_iou_mask
 * never synchronise the host.  The library never allocates device memory:
 * the caller owns every buffer, including the workspace.
 *
 * The operation (cited by page title and section):
 *   "NMS CUDA代码学习" (leetCUDA 14-nms), intro and section 算法与数据流:
 *     visit boxes from the highest score to the lowest (stable: equal scores
 *     keep input order), keep a box unless an already-kept box overlaps it
 *     with IoU strictly greater than the threshold, and return the survivors
 *     as original input indices; section "host 侧": int64 indices, on the
 *     input's device, in score order.
 *   "YOLOv5后处理GPU移植实战", section 1.1 (a device-side count next to the
 *     boxes), section 2.2 (equal scores: the lower index has priority;
 *     suppression only within one class).
 *
 * Conventions fixed by this library where the pages are silent:
 *   - boxes are xyxy fp32 [n][4], row-major, 16-byte aligned; scores fp32 [n].
 *   - IoU = inter / ((area_a + area_b) - inter) with area = (x2-x1)*(y2-y1),
 *     w = max(min(x2)-max(x1), 0), h likewise, every step one IEEE binary32
 *     operation with round-to-nearest-even, no fused multiply-add, no
 *     flush-to-zero; max/min return the non-NaN operand.  The test is
 *     iou > iou_thr in binary32 (strict).
 *   - score order: descending; -0 == +0; NaN after everything; ties (and NaNs
 *     among themselves) by lower input index.
 */
#ifndef GBNMS_H
#define GBNMS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nms_status {
    NMS_OK = 0,
    NMS_ERR_INVALID_ARG = 1, /* bad pointer, size, threshold, alignment, offsets or class id */
    NMS_ERR_WORKSPACE = 2,   /* workspace NULL or smaller than nms_workspace_size() */
    NMS_ERR_CAPACITY = 3,    /* keep_cap or mask capacity too small, or n beyond a limit */
    NMS_ERR_CUDA = 4,        /* a CUDA launch or copy failed */
    NMS_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (device status only) */
} nms_status;

/* Largest n of the single-image, single-class path (its mask is n*ceil(n/256)*32 bytes). */
#define NMS_MAX_SINGLE_N (1 << 18)

/* Human-readable name of a status code (static string; never NULL). */
const char* nms_status_string(nms_status s);

/*
 * Workspace bytes nms_run needs for n boxes.
 *   batch       = 0 when nms_run will get batch_offsets == NULL (one image),
 *                 else the number of images (>= 1).
 *   num_classes = 0 when nms_run will get class_ids == NULL (one class),
 *                 else the number of classes (>= 1).
 * The single-image single-class path (batch == 0 && num_classes == 0) holds
 * the full suppression bitmask: about n*n/8 bytes.  The batched path needs
 * O(n + batch*num_classes) bytes.  Pure host computation.
 * Errors: NMS_ERR_INVALID_ARG (n < 0, negative batch/num_classes, bytes NULL),
 *         NMS_ERR_CAPACITY (single path with n > NMS_MAX_SINGLE_N).
 */
nms_status nms_workspace_size(int64_t n, int32_t batch, int32_t num_classes, size_t* bytes);

/*
 * The device address of page-locked host memory that is mapped into the
 * device address space (memory from cudaHostAlloc or cudaMallocHost on a
 * system with unified addressing).  Every "device" pointer argument of this
 * library may be such an address: the kernels then read the input, or write
 * the output, across the host link themselves, so a caller with its data in
 * host memory needs no separate copies.
 *   host_ptr       any address inside such an allocation.
 *   device_ptr     receives the matching device address.
 * Errors: NMS_ERR_INVALID_ARG (NULL arguments, or host_ptr is not mapped
 *         page-locked host memory: device memory, pageable memory).  Pure
 *         host query; enqueues nothing.
 */
nms_status nms_mapped_pointer(const void* host_ptr, void** device_ptr);

/*
 * Copies bytes from src to dst with every SM, for a caller whose input sits in
 * mapped page-locked host memory (nms_mapped_pointer): one pass across the
 * host link into a device buffer, which nms_run then reads.  Read in place,
 * the same input would cross the link many times (each CTA of the score sort
 * reads every score).
 *   dst, src       device addresses (either may be mapped host memory); the
 *                  ranges must not overlap.  16-byte aligned pointers and a
 *                  size that is a multiple of 16 take 16-byte accesses.
 *   bytes          bytes to copy (0: nothing is enqueued).
 *   stream         cudaStream_t; the copy waits for the stream's previous
 *                  kernel before it writes dst (programmatic dependent launch).
 * Errors: NMS_ERR_INVALID_ARG (NULL dst or src with bytes > 0),
 *         NMS_ERR_CUDA.  Asynchronous; ownership stays with the caller.
 */
nms_status nms_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * Greedy IoU NMS.
 *
 *   boxes          device fp32 [n][4] xyxy, 16-byte aligned (see
 *                  nms_mapped_pointer for host memory).
 *   scores         device fp32 [n].
 *   n              number of boxes, 0 <= n < 2^31.
 *   class_ids      device int32 [n] with values in [0, num_classes), or NULL
 *                  (all boxes one class).  Boxes of different classes never
 *                  suppress each other.
 *   num_classes    >= 1 when class_ids != NULL; ignored otherwise.
 *   batch_offsets  device int64 [batch+1], 0 = off[0] <= off[1] <= ... <=
 *                  off[batch] = n: image b is boxes [off[b], off[b+1]).  NULL
 *                  means one image.  Boxes of different images never suppress
 *                  each other.
 *   batch          >= 1 when batch_offsets != NULL; ignored otherwise.
 *   iou_thr        fp32 IoU threshold (not NaN); a box is dropped when its IoU
 *                  with a kept box of the same image and class is > iou_thr.
 *   score_thr      pre-filter: only boxes with score > score_thr (strict; NaN
 *                  scores fail) take part.  -INFINITY disables the pre-filter
 *                  (then NaN and -inf scores take part and sort last).
 *   max_out        at most max_out outputs per image (the first ones in score
 *                  order); <= 0 means no cap.
 *   keep           device int64 output.  Image b's kept indices (global input
 *                  indices, descending score, ties by index, classes merged)
 *                  are written at keep[b * max_out] when max_out > 0, else at
 *                  keep[off[b]] (keep[0] for one image).
 *   keep_cap       entries available at keep: must be >= batch*max_out
 *                  (max_out > 0; min(n, max_out) for one image) or >= n.
 *   counts         device int64 [max(batch,1)]: kept boxes per image.
 *   dev_status     device int32 [1] or NULL.  Receives NMS_OK, or an error found
 *                  on the device (invalid batch_offsets or class ids:
 *                  NMS_ERR_INVALID_ARG; a bounded wait that gave up:
 *                  NMS_ERR_TIMEOUT).  On a device error, keep/counts of the
 *                  affected images are unspecified but all writes stay in
 *                  bounds.
 *   workspace      device scratch of >= nms_workspace_size(n, batch or 0,
 *                  num_classes or 0) bytes, 256-byte aligned; contents on entry
 *                  do not matter.  Reused freely between calls on one stream.
 *   stream         cudaStream_t.
 *
 * Host-detected errors return before anything is enqueued.  Asynchronous:
 * results are valid once the stream reaches the end of the call.
 */
nms_status nms_run(const float* boxes, const float* scores, int64_t n,
                   const int32_t* class_ids, int32_t num_classes,
                   const int64_t* batch_offsets, int32_t batch,
                   float iou_thr, float score_thr, int32_t max_out,
                   int64_t* keep, int64_t keep_cap, int64_t* counts,
                   int32_t* dev_status,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Row stride, in 64-bit words, of the bitmask nms_iou_mask writes: 4*ceil(n/256). */
int64_t nms_mask_row_words(int64_t n);

/*
 * The suppression bitmask of boxes already in score order
 * ("NMS CUDA代码学习", section Phase 1: warp-per-box ballot and the aligned
 * j_base rule): bit (j mod 64) of word j/64 of row i is set iff j > i, j < n
 * and IoU(box i, box j) > iou_thr.  Bit k of a word always means box
 * 64*word + k; in little-endian memory this equals the pages' 32-bit words.
 *
 *   boxes_sorted  device fp32 [n][4] xyxy, 16-byte aligned, highest score first.
 *   mask          device uint64 [n][nms_mask_row_words(n)], row-major.  For row
 *                 i, words w >= floor(i/64) are written (w < ceil(n/64) hold
 *                 the bits above, the padding words up to the stride are 0);
 *                 words below floor(i/64) are not part of the result.
 *   mask_words    capacity of mask in words (>= n * nms_mask_row_words(n)).
 * Errors: NMS_ERR_INVALID_ARG (NULL/unaligned pointers, n < 0, NaN threshold),
 *         NMS_ERR_CAPACITY (n > NMS_MAX_SINGLE_N or mask_words too small),
 *         NMS_ERR_CUDA.
 */
nms_status nms_iou_mask(const float* boxes_sorted, int64_t n, float iou_thr,
                        uint64_t* mask, int64_t mask_words, void* stream);

/*
 * Sequential resolve of a suppression bitmask in score order
 * ("NMS CUDA代码学习", section Phase 2: walk the boxes from the highest score
 * down, keep a box whose bit is not yet set in the removed-bitmap and OR its
 * mask row into the bitmap; section "host 侧": map kept positions back through
 * the sort permutation).  One thread block; the walk stops at max_out.
 *
 *   mask     device uint64 [n][nms_mask_row_words(n)] in the nms_iou_mask
 *            layout, 16-byte aligned.  Words w >= floor(i/64) of row i carry
 *            the bits; words below may be read but never change the result.
 *   perm     device int32 [n]: input index of each sorted position, or NULL
 *            (the output is then the kept sorted positions themselves).
 *   max_out  cap on the number of outputs; <= 0 means none.
 *   perm is 4-byte aligned when given.
 *   keep     device int64 [min(n, max_out) or n], 8-byte aligned: kept
 *            entries in order.
 *   count    device int64 [1], 8-byte aligned: number of kept entries.
 *   workspace device scratch of >= nms_workspace_size(n, 0, 0) bytes,
 *            256-byte aligned.  It is checked and reserved for the resolve,
 *            which at present keeps all its state (the removed-bitmap and
 *            the column view of the blocks near the diagonal, rebuilt from
 *            the mask) in the shared memory of its thread block and does not
 *            touch it.
 * Errors: NMS_ERR_INVALID_ARG (NULL or unaligned pointers with n > 0, an
 *         unaligned count, n < 0), NMS_ERR_CAPACITY (n > NMS_MAX_SINGLE_N),
 *         NMS_ERR_WORKSPACE, NMS_ERR_CUDA.
 */
nms_status nms_resolve_mask(const uint64_t* mask, int64_t n, const int32_t* perm,
                            int32_t max_out, int64_t* keep, int64_t* count,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Fast NMS ("YOLOv5后处理GPU移植实战", sections 2.1 and 2.2): a box is dropped
 * when any box of higher priority (higher score, or equal score and lower
 * index) of the same image and class has IoU > iou_thr with it, whether or
 * not that box was dropped itself.  It keeps a subset of what nms_run keeps,
 * in the same order, and needs no sequential resolve.  Arguments, output
 * layout, workspace and errors exactly as for nms_run.
 */
nms_status nms_fast_run(const float* boxes, const float* scores, int64_t n,
                        const int32_t* class_ids, int32_t num_classes,
                        const int64_t* batch_offsets, int32_t batch, float iou_thr,
                        float score_thr, int32_t max_out, int64_t* keep, int64_t keep_cap,
                        int64_t* counts, int32_t* dev_status, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Decay kernels of nms_matrix_run. */
#define NMS_DECAY_GAUSSIAN 0
#define NMS_DECAY_LINEAR 1

/*
 * Matrix NMS, one image ("Fastest Matrix NMS in the West (Part 2)", sections
 * "What do we need to compute?" and "Optimization 4").  Boxes in the greedy
 * order (descending score, ties to the lower index), O[i][j] the canonical
 * binary32 IoU of box j with a father i before it, O_max[i] the largest
 * overlap of box i with its own fathers (0 for none):
 *   s'[j] = s[j] * min over fathers i of d[i][j]   (1 without fathers)
 *   NMS_DECAY_GAUSSIAN: d = exp((O_max[i]^2 - O[i][j]^2) / sigma)
 *   NMS_DECAY_LINEAR:   d = (1 - O[i][j]) / (1 - O_max[i])
 * (the page names a linear decay without printing it; this is the linear
 * kernel with the same compensation), evaluated in binary64 from the binary32
 * IoUs and scores, NaN terms (a linear 0/0) ignored by the minimum; box j is
 * dropped when s'[j] < decay_thr.
 *   boxes, scores, n, score_thr, max_out, dev_status, stream: as nms_run
 *                  (one image, one class).
 *   decay          NMS_DECAY_GAUSSIAN or NMS_DECAY_LINEAR.
 *   sigma          Gaussian only: > 0, finite (the pages use 0.5); ignored
 *                  by the linear decay.
 *   decay_thr      threshold on the final scores (not NaN).
 *   keep           device int64 [keep_cap]: kept input indices in score order.
 *   keep_scores    device float [keep_cap] or NULL: their final scores, the
 *                  binary64 value rounded (linear), or within 4 binary32 ulp
 *                  of it (Gaussian; exactly it rounded when the score lies
 *                  near decay_thr).
 *   count          device int64 [1].
 *   workspace      >= nms_matrix_workspace_size(n) bytes, 256-byte aligned.
 * Errors: NMS_ERR_INVALID_ARG, NMS_ERR_CAPACITY (n > NMS_MAX_SINGLE_N or
 * keep_cap too small), NMS_ERR_WORKSPACE, NMS_ERR_CUDA.
 */
nms_status nms_matrix_workspace_size(int64_t n, size_t* bytes);
nms_status nms_matrix_run(const float* boxes, const float* scores, int64_t n, int32_t decay,
                          float sigma, float score_thr, float decay_thr, int32_t max_out,
                          int64_t* keep, float* keep_scores, int64_t keep_cap, int64_t* count,
                          int32_t* dev_status, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * nms_run with stage timing, for measurement: the same call, plus up to
 * nevents caller-created CUDA events (cudaEvent_t, created with timing
 * enabled) that it records on `stream`: events[0] before its first kernel and
 * events[k] when stage k has been enqueued.
 *   One image:  1 = pre-filter, sort and gather; 2 = IoU mask (with the pair
 *               list; with max_out, of the leading 2*max_out boxes); 3 =
 *               resolve and output (with max_out, also the rest of the mask
 *               and a second resolve when the leading boxes held fewer than
 *               max_out kept boxes).
 *   Batched:    1 = pre-filter and bucketing into (image, class) segments;
 *               2 = per-segment NMS; 3 = per-image merge and output.
 * NULL entries and entries past nevents are skipped (nevents may be 0).  The
 * events are only recorded, never synchronised.  Arguments, errors and
 * results otherwise as for nms_run.
 */
nms_status nms_run_timed(const float* boxes, const float* scores, int64_t n,
                         const int32_t* class_ids, int32_t num_classes,
                         const int64_t* batch_offsets, int32_t batch, float iou_thr,
                         float score_thr, int32_t max_out, int64_t* keep, int64_t keep_cap,
                         int64_t* counts, int32_t* dev_status, void* workspace,
                         size_t workspace_bytes, void* stream, void* const* events,
                         int32_t nevents);

/* Limits of the front end for YOLO-shaped outputs. */
#define NMS_DECODE_MAX_ANCHORS (1 << 20)
#define NMS_DECODE_MAX_CLASSES 384
/* Largest batch of the front end and of NMS over count-header buffers (the
 * images are one dimension of the launch grids). */
#define NMS_DECODE_MAX_BATCH 65535

/*
 * Front end for YOLO-shaped outputs: the "count header + data body" buffer of
 * "YOLOv5后处理GPU移植实战" (section 1.1), one per image,
 *   float buffers[batch][1 + 7 * max_objects]:
 *   element 0     the number of candidates found (may exceed max_objects:
 *                 section 1.2 drops a candidate past max_objects but still
 *                 counts it; a reader takes min(count, max_objects) rows);
 *   rows of 7     left, top, right, bottom, confidence, class, keep_flag.
 * The page prints the layout, not the decode.  Readings: preds is
 * [batch][anchors][5 + num_classes] binary32 (cx, cy, w, h, objectness, class
 * scores; activations already applied), confidence = RN(objectness x largest
 * class score), class = the first class with that maximum (as a float), a
 * row is a candidate when confidence > conf_thr, the box is centre +- half
 * size in binary32, keep_flag = 1, and candidates take the rows in anchor
 * order (so the buffer is the same on every run).  Rows past the candidates
 * are left as they are.
 *   preds        device, 4-byte aligned.
 *   batch        in [1, NMS_DECODE_MAX_BATCH]; anchors in [0, NMS_DECODE_MAX_ANCHORS];
 *   num_classes  in [1, NMS_DECODE_MAX_CLASSES].
 *   conf_thr     not NaN.
 *   max_objects  >= 0 rows per image.
 *   buffers      device float[batch * (1 + 7 * max_objects)].
 *   dev_status   device int32 [1] or NULL (then a word of the workspace):
 *                NMS_OK, or NMS_ERR_TIMEOUT if a block's bounded wait for its
 *                staged rows gave up (the buffers are then unspecified).
 *   workspace    >= nms_decode_workspace_size() bytes, 256-byte aligned.
 * Errors: NMS_ERR_INVALID_ARG, NMS_ERR_CAPACITY (limits), NMS_ERR_WORKSPACE,
 * NMS_ERR_CUDA (host side); the device status above.
 */
nms_status nms_decode_workspace_size(int32_t batch, int32_t anchors, size_t* bytes);
nms_status nms_decode_boxes7(const float* preds, int32_t batch, int32_t anchors, int32_t num_classes,
                             float conf_thr, int32_t max_objects, float* buffers, int32_t* dev_status,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * NMS in place over count-header buffers (layout as above): for each image
 * the first min(count, max_objects) rows take part (a count below 1 or NaN:
 * none); boxes of one class interact; rows rank by confidence, then by the
 * lower position ("YOLOv5后处理GPU移植实战", section 2.2); keep_flag of each
 * taking-part row becomes 1 (kept) or 0.  fast = 0: exact greedy NMS (IoU >
 * iou_thr, canonical binary32 IoU); fast = 1: the page's Fast NMS (a row goes
 * when any higher-ranked row of its class, kept or not, overlaps it beyond
 * iou_thr).  Rows past the taking-part ones are not touched.
 *   num_classes   class values must be integers in [0, num_classes); any
 *                 other value sets NMS_ERR_INVALID_ARG in the device status
 *                 (dev_status, or the workspace's status word) and leaves
 *                 that row out.
 *   batch <= NMS_DECODE_MAX_BATCH (else NMS_ERR_CAPACITY);
 *   batch * max_objects <= INT32_MAX; batch * num_classes <= INT32_MAX / 2.
 *   workspace     >= nms_boxes7_workspace_size() bytes, 256-byte aligned.
 * Errors: NMS_ERR_INVALID_ARG, NMS_ERR_WORKSPACE, NMS_ERR_CUDA (host side);
 * the device status as for nms_run.
 */
nms_status nms_boxes7_workspace_size(int32_t batch, int32_t max_objects, int32_t num_classes, size_t* bytes);
nms_status nms_boxes7_run(float* buffers, int32_t batch, int32_t max_objects, int32_t num_classes, float iou_thr,
                          int32_t fast, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Lane candidates of nms_lane_run. */
#define NMS_LANE_VALUES 77
#define NMS_LANE_ROWS 72
#define NMS_LANE_MAX_N 16384

/*
 * Greedy NMS of lane candidates ("nms_kernel.cu 파일 분석 -2": a candidate
 * holds PROP_SIZE = 77 values; candidates are compared in score order in
 * 64-candidate tiles above the diagonal; the comparison is symmetric, by
 * absolute values, against the threshold that says whether two lanes are
 * alike).  The page stops before the comparison; the reading taken:
 *   values   0, 1: class scores (not used here); 2: start row; 3: start x
 *            (not used here); 4: length in rows; 5..76: the lane's x at
 *            rows 0..71;
 *   rows     a lane covers rows [floor(start), floor(start) + floor(length))
 *            within [0, 72); a NaN, infinite or beyond 2^20 start or length
 *            covers none;
 *   distance of two lanes: over the rows both cover, the binary32 sum of
 *            |x_a - x_b|, added from the lowest row up, divided by the
 *            number of those rows (+inf without any);
 *   rule     greedy NMS in descending score (ties to the lower index): a
 *            lane is dropped when its distance to a kept lane is strictly
 *            below dist_thr (a NaN distance never drops).
 *
 *   props    device float [n][77], row-major, 4-byte aligned.
 *   scores   device float [n]: the NMS order (descending; -0 = +0; NaN last).
 *   n        0 <= n <= NMS_LANE_MAX_N.
 *   max_out  at most this many outputs (<= 0: no cap).
 *   keep     device int64 [keep_cap] (8-byte aligned), keep_cap >=
 *            min(n, max_out) with max_out, else >= n: kept input indices in
 *            score order.
 *   count    device int64 [1] (8-byte aligned): their number.
 *   dev_status optional device int32: NMS_ERR_TIMEOUT when a bounded wait
 *            of the resolve gave up.
 *   workspace device scratch of >= nms_lane_workspace_size(n) bytes,
 *            256-byte aligned, owned by the caller.
 * Asynchronous on `stream`; the library allocates nothing.
 * Errors: NMS_ERR_INVALID_ARG (n < 0, NaN dist_thr, NULL or misaligned
 *         pointers), NMS_ERR_CAPACITY (n > NMS_LANE_MAX_N, keep_cap too
 *         small), NMS_ERR_WORKSPACE, NMS_ERR_CUDA.
 */
nms_status nms_lane_workspace_size(int64_t n, size_t* bytes);
nms_status nms_lane_run(const float* props, const float* scores, int64_t n, float dist_thr, int32_t max_out,
                        int64_t* keep, int64_t keep_cap, int64_t* count, int32_t* dev_status, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Largest n nms_resolve_mask_noalloc accepts. */
#define NMS_NOALLOC_MAX_N 16384

/*
 * nms_resolve_mask without a workspace: the same resolve, which keeps all its
 * state in the shared memory of one thread block, so it needs no device
 * scratch at all.  The pages have no counterpart to this entry point; it
 * exists for callers that cannot allocate device memory where they run NMS
 * (a plugin whose host framework owns every allocation, a real-time loop
 * whose memory is planned at start-up, a deployment that bans allocation
 * after initialisation).
 *
 *   mask, perm, max_out, keep, count: as for nms_resolve_mask (with the
 *            same alignment); n must be <= NMS_NOALLOC_MAX_N.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine) and holds nothing between calls, so calls on any streams, host
 * threads or devices may overlap.
 * Errors: NMS_ERR_INVALID_ARG (n < 0, NULL or unaligned pointers),
 *         NMS_ERR_CAPACITY (n > NMS_NOALLOC_MAX_N), NMS_ERR_CUDA.
 */
nms_status nms_resolve_mask_noalloc(const uint64_t* mask, int64_t n, const int32_t* perm,
                                    int32_t max_out, int64_t* keep, int64_t* count, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBNMS_H */
