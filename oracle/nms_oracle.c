/*
 * Greedy IoU NMS oracle: TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg may load, call or run this code.  It shares no code, header, table or
 * helper with the CUDA library in greedy_iou_nms_gb300/csrc; the two never
 * import each other.
 *
 * What it computes is the plain definition of greedy hard NMS, written out as
 * a slow loop with no bitmask, no tiling and no reordering:
 *
 *   "NMS CUDA代码学习" (leetCUDA 14-nms), intro and section 算法与数据流:
 *     boxes are visited from the highest score to the lowest (stable sort, so
 *     equal scores keep input order); a box is dropped when it overlaps an
 *     already-kept box with IoU strictly greater than the threshold; the
 *     survivors are returned as original input indices (section "host 侧:
 *     zeros、映射回原索引、返回类型": int64 indices, in score order).
 *
 *   "YOLOv5后处理GPU移植实战", section 2.2 稳定性增强方案: among equal scores the
 *     lower index has priority, and suppression only happens between boxes of
 *     the same class.
 *
 * Readings where the pages are silent:
 *   - IoU on continuous xyxy coordinates, no "+1"; every step in IEEE binary32
 *     with round-to-nearest-even, in the fixed order of oracle_iou() below, no
 *     fused multiply-add (this file must be built with -ffp-contract=off and
 *     without -ffast-math), no flush-to-zero.  max/min are C fmaxf/fminf.
 *   - The threshold is an fp32 value and the test is iou > thr (strict).
 *   - Score order: descending; -0 equals +0; NaN scores go after every other
 *     score (including -inf); ties (and NaNs among themselves) by lower index.
 *   - Optional pre-filter keeps score > score_thr (strict; NaN fails).
 *   - max_out caps the number of outputs per image (first max_out kept in score
 *     order); max_out <= 0 means no cap.
 *   - Batched class-aware mode: images are the ranges
 *     [batch_offsets[b], batch_offsets[b+1]); within an image, boxes suppress
 *     only boxes of the same class; the output of image b is written at
 *     keep[b * max_out] when max_out > 0, else at keep[batch_offsets[b]], in
 *     score order across classes, and counts[b] holds its length.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Canonical IoU of two xyxy boxes, in the fixed binary32 operation order. */
float oracle_iou(const float* a, const float* b)
{
    float area_a = (a[2] - a[0]) * (a[3] - a[1]);
    float area_b = (b[2] - b[0]) * (b[3] - b[1]);
    float xx1 = fmaxf(a[0], b[0]);
    float yy1 = fmaxf(a[1], b[1]);
    float xx2 = fminf(a[2], b[2]);
    float yy2 = fminf(a[3], b[3]);
    float w = fmaxf(xx2 - xx1, 0.0f);
    float h = fmaxf(yy2 - yy1, 0.0f);
    float inter = w * h;
    float uni = (area_a + area_b) - inter;
    return inter / uni;
}

/* Score order used for sorting: returns <0 when candidate (sa, ia) comes
 * before (sb, ib).  Descending score, NaN last, ties by lower index. */
static int score_before(float sa, int64_t ia, float sb, int64_t ib)
{
    int na = isnan(sa), nb = isnan(sb);
    if (na != nb) return na ? 1 : -1;
    if (!na) {
        if (sa > sb) return -1;
        if (sa < sb) return 1;
    }
    if (ia < ib) return -1;
    if (ia > ib) return 1;
    return 0;
}

static const float* g_scores; /* comparator context (single-threaded oracle) */

static int cmp_index(const void* pa, const void* pb)
{
    int64_t ia = *(const int64_t*)pa, ib = *(const int64_t*)pb;
    return score_before(g_scores[ia], ia, g_scores[ib], ib);
}

/* Sort idx[0..m) into greedy visiting order (stable descending score). */
void oracle_score_order(const float* scores, int64_t* idx, int64_t m)
{
    g_scores = scores;
    qsort(idx, (size_t)m, sizeof(int64_t), cmp_index);
}

/*
 * Greedy NMS over one image [lo, hi) of the input.
 * Writes kept original indices (score order) to out, returns their number.
 * order/kept are caller-provided scratch of at least hi-lo entries.
 */
static int64_t greedy_image(const float* boxes, const float* scores, const int32_t* class_ids,
                            int64_t lo, int64_t hi, float iou_thr, int use_score_thr,
                            float score_thr, int32_t max_out, int64_t* order, int64_t* out)
{
    int64_t m = 0;
    for (int64_t i = lo; i < hi; ++i)
        if (!use_score_thr || scores[i] > score_thr) order[m++] = i;
    oracle_score_order(scores, order, m);

    int64_t nkept = 0;
    for (int64_t p = 0; p < m; ++p) {
        int64_t i = order[p];
        int suppressed = 0;
        for (int64_t q = 0; q < nkept && !suppressed; ++q) {
            int64_t k = out[q];
            if (class_ids && class_ids[k] != class_ids[i]) continue;
            if (oracle_iou(boxes + 4 * k, boxes + 4 * i) > iou_thr) suppressed = 1;
        }
        if (suppressed) continue;
        out[nkept++] = i;
        if (max_out > 0 && nkept == max_out) break;
    }
    return nkept;
}

/*
 * Full oracle entry.  boxes: [n][4] xyxy fp32; scores: [n]; class_ids: [n] or
 * NULL (one class); batch_offsets: [batch+1] or NULL (one image, batch must be
 * 1).  keep must hold batch*max_out entries when max_out > 0, else n.
 * counts: [batch].  Returns the total number of kept boxes, or -1 on bad input.
 */
int64_t oracle_nms(const float* boxes, const float* scores, int64_t n,
                   const int32_t* class_ids, const int64_t* batch_offsets, int32_t batch,
                   float iou_thr, int use_score_thr, float score_thr, int32_t max_out,
                   int64_t* keep, int64_t* counts)
{
    if (n < 0 || batch < 1) return -1;
    if (!batch_offsets && batch != 1) return -1;
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!order) return -1;
    int64_t total = 0;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t lo = batch_offsets ? batch_offsets[b] : 0;
        int64_t hi = batch_offsets ? batch_offsets[b + 1] : n;
        if (lo < 0 || hi < lo || hi > n) { free(order); return -1; }
        int64_t base = (max_out > 0) ? (int64_t)b * max_out : lo;
        counts[b] = greedy_image(boxes, scores, class_ids, lo, hi, iou_thr, use_score_thr,
                                 score_thr, max_out, order, keep + base);
        total += counts[b];
    }
    free(order);
    return total;
}

/*
 * Fast NMS over one image [lo, hi): a box is dropped when ANY box before it
 * in the priority order (same class) overlaps it with IoU > thr, whether or
 * not that box was itself dropped.
 *
 *   "YOLOv5后处理GPU移植实战", section 2.2 稳定性增强方案: each box is tested
 *     against every other box of its class; it is suppressed when a box of
 *     higher priority (higher score, or equal score and lower index) has
 *     IoU above the threshold.  Section 2.1: without the index tie-break,
 *     equal-score overlapping boxes would all drop each other.
 *
 * Readings: the output is the kept indices in the same
 * priority order as greedy NMS, cut at max_out; the pre-filter and the batch
 * layout are those of oracle_nms.
 */
static int64_t fast_image(const float* boxes, const float* scores, const int32_t* class_ids,
                          int64_t lo, int64_t hi, float iou_thr, int use_score_thr, float score_thr,
                          int32_t max_out, int64_t* order, int64_t* out)
{
    int64_t m = 0;
    for (int64_t i = lo; i < hi; ++i)
        if (!use_score_thr || scores[i] > score_thr) order[m++] = i;
    oracle_score_order(scores, order, m);

    int64_t nkept = 0;
    for (int64_t p = 0; p < m; ++p) {
        int64_t i = order[p];
        int suppressed = 0;
        for (int64_t q = 0; q < p && !suppressed; ++q) {
            int64_t k = order[q];
            if (class_ids && class_ids[k] != class_ids[i]) continue;
            if (oracle_iou(boxes + 4 * k, boxes + 4 * i) > iou_thr) suppressed = 1;
        }
        if (suppressed) continue;
        out[nkept++] = i;
        if (max_out > 0 && nkept == max_out) break;
    }
    return nkept;
}

/* Fast NMS entry: arguments, output layout and return value as oracle_nms. */
int64_t oracle_fast_nms(const float* boxes, const float* scores, int64_t n,
                        const int32_t* class_ids, const int64_t* batch_offsets, int32_t batch,
                        float iou_thr, int use_score_thr, float score_thr, int32_t max_out,
                        int64_t* keep, int64_t* counts)
{
    if (n < 0 || batch < 1) return -1;
    if (!batch_offsets && batch != 1) return -1;
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!order) return -1;
    int64_t total = 0;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t lo = batch_offsets ? batch_offsets[b] : 0;
        int64_t hi = batch_offsets ? batch_offsets[b + 1] : n;
        if (lo < 0 || hi < lo || hi > n) { free(order); return -1; }
        int64_t base = (max_out > 0) ? (int64_t)b * max_out : lo;
        counts[b] = fast_image(boxes, scores, class_ids, lo, hi, iou_thr, use_score_thr, score_thr,
                               max_out, order, keep + base);
        total += counts[b];
    }
    free(order);
    return total;
}

/*
 * Matrix NMS, one image, Gaussian (linear == 0) or linear (linear != 0) decay:
 *
 *   "Fastest Matrix NMS in the West (Part 2)", section "What do we need to
 *   compute?": with boxes sorted by score (highest first), O[i][j] is the IoU
 *   of box j with a higher-scoring father box i (i before j), O_max[i] the
 *   largest overlap of box i with its own fathers, the decay that father i
 *   gives box j is exp((O_max[i]^2 - O[i][j]^2) / sigma), and the final score
 *   is s'[j] = s[j] * min over fathers i of that decay.  Section
 *   "Optimization 4": a box is dropped when its final score is below the
 *   threshold t.  The same section says the code also holds a linear decay;
 *   the page does not print it.  The reading taken is the linear kernel of
 *   the Matrix NMS method with the same compensation by the father's own
 *   largest overlap: the decay is (1 - O[i][j]) / (1 - O_max[i]).
 *
 * Readings: the sort is the stable descending one of
 * greedy NMS (ties to the lower index) over the pre-filtered candidates; IoUs
 * are the canonical binary32 ones; a box with no father (the first) keeps
 * s[j] (the minimum over no fathers is 1); the exponent, the exponential, the
 * product and the comparison are evaluated in binary64 from those binary32
 * values, with NaN decays (the linear 0/0 of a father that fully overlaps
 * its own father and the box) ignored by the minimum; the output is the kept
 * indices in score order with their final scores rounded to binary32, cut at
 * max_out.  This is the literal O(n^2) evaluation.
 */
int64_t oracle_matrix_nms(const float* boxes, const float* scores, int64_t n, float sigma, int linear,
                          int use_score_thr, float score_thr, float decay_thr, int32_t max_out,
                          int64_t* keep, float* out_scores)
{
    if (n < 0) return -1;
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    float* omax = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    if (!order || !omax) { free(order); free(omax); return -1; }
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i)
        if (!use_score_thr || scores[i] > score_thr) order[m++] = i;
    oracle_score_order(scores, order, m);
    for (int64_t p = 0; p < m; ++p) {
        float best = 0.0f;
        for (int64_t q = 0; q < p; ++q) {
            float o = oracle_iou(boxes + 4 * order[q], boxes + 4 * order[p]);
            if (o > best) best = o;
        }
        omax[p] = best;
    }
    int64_t nkept = 0;
    for (int64_t p = 0; p < m && !(max_out > 0 && nkept == max_out); ++p) {
        double dmin = 1.0;
        for (int64_t q = 0; q < p; ++q) {
            float o = oracle_iou(boxes + 4 * order[q], boxes + 4 * order[p]);
            double d;
            if (linear) {
                d = (1.0 - (double)o) / (1.0 - (double)omax[q]);
            } else {
                double x = ((double)omax[q] * (double)omax[q] - (double)o * (double)o) / (double)sigma;
                d = exp(x);
            }
            if (d < dmin) dmin = d;
        }
        double fs = (double)scores[order[p]] * dmin;
        if (fs < (double)decay_thr) continue;
        keep[nkept] = order[p];
        if (out_scores) out_scores[nkept] = (float)fs;
        ++nkept;
    }
    free(order);
    free(omax);
    return nkept;
}

/*
 * Matrix NMS decisions at chosen sorted positions, for images too large for
 * oracle_matrix_nms to finish in a test.  Same definition, evaluated box by
 * box: without max_out every box is decided on its own (its final score
 * depends only on its fathers and theirs, never on another decision).
 *
 * For the box at sorted position p (positions[k], among the m candidates
 * that pass the pre-filter, in the order of oracle_score_order):
 *   final = s[j] * min over fathers q < p of the decay of (O[q][p], O_max[q]),
 * kept when final >= t, exactly as oracle_matrix_nms computes them.  A father
 * with O[q][p] = 0 gives the Gaussian decay exp(O_max[q]^2 / sigma) >= 1 and
 * the linear decay 1 / (1 - O_max[q]) >= 1 (or +inf), and a NaN overlap a NaN
 * decay; none of them can lower the minimum, which starts at 1, so only the
 * fathers with O[q][p] > 0 are visited, and O_max[q] is computed for those
 * alone (the largest overlap of box q with its own fathers, as above).  The
 * result is the same value bit for bit.
 *
 * Out, per requested position: index[k] the input index there, kept[k] 0 or
 * 1, final_scores[k] the final score rounded to binary32.  Returns m, or -1
 * on invalid arguments (a position outside [0, m)).
 */
int64_t oracle_matrix_decide_at(const float* boxes, const float* scores, int64_t n, float sigma, int linear,
                                int use_score_thr, float score_thr, float decay_thr, const int64_t* positions,
                                int64_t npos, int64_t* index, int32_t* kept, float* final_scores)
{
    if (n < 0 || npos < 0) return -1;
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!order) return -1;
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i)
        if (!use_score_thr || scores[i] > score_thr) order[m++] = i;
    oracle_score_order(scores, order, m);
    for (int64_t k = 0; k < npos; ++k) {
        const int64_t p = positions[k];
        if (p < 0 || p >= m) { free(order); return -1; }
        const float* bp = boxes + 4 * order[p];
        double dmin = 1.0;
        for (int64_t q = 0; q < p; ++q) {
            const float* bq = boxes + 4 * order[q];
            float o = oracle_iou(bq, bp);
            if (!(o > 0.0f)) continue;
            float omax = 0.0f;  /* O_max of father q */
            for (int64_t r = 0; r < q; ++r) {
                float oq = oracle_iou(boxes + 4 * order[r], bq);
                if (oq > omax) omax = oq;
            }
            double d;
            if (linear) {
                d = (1.0 - (double)o) / (1.0 - (double)omax);
            } else {
                double x = ((double)omax * (double)omax - (double)o * (double)o) / (double)sigma;
                d = exp(x);
            }
            if (d < dmin) dmin = d;
        }
        double fs = (double)scores[order[p]] * dmin;
        index[k] = order[p];
        kept[k] = fs < (double)decay_thr ? 0 : 1;
        final_scores[k] = (float)fs;
    }
    free(order);
    return m;
}

/*
 * Lane-proposal NMS ("nms_kernel.cu 파일 분석 -2"): the same greedy NMS over
 * lane candidates instead of boxes.  The page gives: a candidate holds
 * PROP_SIZE = 77 values; candidates are visited in score order through idx
 * (the sorted order), each compared with every later one; the comparison is
 * symmetric ("A against B is the same as B against A, because it compares by
 * absolute value"); nms_overlap_thresh is the threshold that decides whether
 * two lanes are alike.  The page stops before the comparison itself.
 *
 * Readings taken:
 *   - the 77 values: two class scores, the start row, the start x, the
 *     length (in rows), then the lane's x at 72 fixed image rows, row 0
 *     first (the distance uses only the start row, the length and the x's;
 *     the NMS order comes from the scores passed beside the candidates);
 *   - a lane's rows are [floor(start), floor(start) + floor(length)) clipped
 *     to [0, 72); a NaN, infinite or larger than 2^20 start or length gives
 *     no rows;
 *   - the distance of two lanes: over the rows both cover, the sum of
 *     |x_a - x_b| in binary32, added row by row from the lowest row, then
 *     divided by the number of those rows (binary32, round to nearest); no
 *     common row gives +inf;
 *   - a later lane is suppressed when its distance to a kept lane is
 *     strictly below the threshold (a NaN distance never suppresses).
 * Order, ties, max_out and the output are those of greedy NMS above.
 */
#define LANE_VALUES 77
#define LANE_ROWS 72
#define LANE_X0 5

static void lane_rows(const float* p, int* lo, int* hi)
{
    const float s = p[2], l = p[4];
    *lo = 0;
    *hi = 0;
    if (!(s >= -1048576.0f && s <= 1048576.0f && l >= -1048576.0f && l <= 1048576.0f)) return;
    int a = (int)floorf(s);
    int b = a + (int)floorf(l);
    if (a < 0) a = 0;
    if (b > LANE_ROWS) b = LANE_ROWS;
    if (b > a) {
        *lo = a;
        *hi = b;
    }
}

float oracle_lane_distance(const float* a, const float* b)
{
    int la, ha, lb, hb;
    lane_rows(a, &la, &ha);
    lane_rows(b, &lb, &hb);
    const int lo = la > lb ? la : lb, hi = ha < hb ? ha : hb;
    if (hi <= lo) return INFINITY;
    float sum = 0.0f;
    for (int k = lo; k < hi; ++k) sum = sum + fabsf(a[LANE_X0 + k] - b[LANE_X0 + k]);
    return sum / (float)(hi - lo);
}

int64_t oracle_lane_nms(const float* props, const float* scores, int64_t n, float thr, int32_t max_out,
                        int64_t* keep)
{
    if (n < 0) return -1;
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!order) return -1;
    for (int64_t i = 0; i < n; ++i) order[i] = i;
    oracle_score_order(scores, order, n);
    int64_t nk = 0;
    for (int64_t p = 0; p < n; ++p) {
        if (max_out > 0 && nk == max_out) break;
        const float* cand = props + LANE_VALUES * order[p];
        int suppressed = 0;
        for (int64_t k = 0; k < nk && !suppressed; ++k)
            if (oracle_lane_distance(props + LANE_VALUES * keep[k], cand) < thr) suppressed = 1;
        if (!suppressed) keep[nk++] = order[p];
    }
    free(order);
    return nk;
}

/*
 * Suppression bitmask of boxes that are already in score order, as the pages
 * define it ("NMS CUDA代码学习", section Phase 1): bit (j mod 64) of word
 * j/64 in row i is set iff j > i and IoU(i, j) > thr.  Row-major [n][W]
 * uint64 words, W = ceil(n/64), every word written (zero where no bit).
 * Used only by tests that check the library's mask entry point.
 */
void oracle_mask(const float* boxes_sorted, int64_t n, float iou_thr, uint64_t* mask)
{
    int64_t W = (n + 63) / 64;
    memset(mask, 0, sizeof(uint64_t) * (size_t)(n * W));
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = i + 1; j < n; ++j)
            if (oracle_iou(boxes_sorted + 4 * i, boxes_sorted + 4 * j) > iou_thr)
                mask[i * W + j / 64] |= (uint64_t)1 << (j % 64);
}

/*
 * Front end for YOLO-shaped outputs: the "count header + data body" buffer of
 * "YOLOv5后处理GPU移植实战", section 1.1, filled from the head's predictions.
 *
 * Per image the buffer is float[1 + 7 * max_objects]: element 0 the number
 * of candidates found, then one row of 7 floats per candidate: left, top,
 * right, bottom, confidence, class, keep_flag.  Section 1.2: a slot is taken
 * with an atomic counter and a candidate beyond max_objects is dropped, so
 * the header may exceed max_objects and a reader takes min(header,
 * max_objects) rows.
 *
 * The page gives the layout but not the decode itself.  Readings: preds is
 * [batch][anchors][5 + num_classes] binary32, each row (cx, cy, w, h,
 * objectness, class scores) as an exported detector emits it (activations
 * already applied); the confidence is RN(objectness * max class score), the
 * class is the first class with that maximum, a row is a candidate when its
 * confidence is > conf_thr (strict, as the score pre-filter), the box is
 * (RN(cx - RN(w / 2)), RN(cy - RN(h / 2)), RN(cx + RN(w / 2)), RN(cy +
 * RN(h / 2))) and keep_flag starts at 1; candidates take the rows in anchor
 * order (the order the page's atomic counter hands out when slots are taken
 * in order: one valid outcome, and the reproducible one).  Unused rows are
 * left as they are.
 */
void oracle_decode_boxes7(const float* preds, int32_t batch, int32_t anchors, int32_t num_classes,
                          float conf_thr, int32_t max_objects, float* out)
{
    const int64_t rowlen = 5 + (int64_t)num_classes;
    const int64_t stride = 1 + 7 * (int64_t)max_objects;
    for (int32_t b = 0; b < batch; ++b) {
        float* buf = out + b * stride;
        int64_t count = 0;
        for (int32_t a = 0; a < anchors; ++a) {
            const float* p = preds + ((int64_t)b * anchors + a) * rowlen;
            int32_t cls = 0;
            float best = p[5];
            for (int32_t c = 1; c < num_classes; ++c)
                if (p[5 + c] > best) { best = p[5 + c]; cls = c; }
            float conf = p[4] * best;
            if (!(conf > conf_thr)) continue;
            if (count < max_objects) {
                float* r = buf + 1 + 7 * count;
                float hw = p[2] / 2.0f, hh = p[3] / 2.0f;
                r[0] = p[0] - hw;
                r[1] = p[1] - hh;
                r[2] = p[0] + hw;
                r[3] = p[1] + hh;
                r[4] = conf;
                r[5] = (float)cls;
                r[6] = 1.0f;
            }
            ++count;
        }
        buf[0] = (float)count;
    }
}
