/*
 * Multi-core CPU greedy NMS: the stronger CPU baseline that bench.py times
 * beside the GPU path (TEST AND BENCHMARK INFRASTRUCTURE ONLY, like the
 * oracle: only tests/ and bench.py's CPU-baseline leg load it).  It shares no
 * code with the oracle (nms_oracle.c) or with the CUDA library: its own
 * order, IoU, bitmask and resolve, written for the host's cores.
 *
 * The method is the bitmask form of "NMS CUDA代码学习", sections 算法与数据流,
 * Phase 1 and Phase 2, run with OpenMP:
 *   1. order: descending score, ties to the lower index, -0 equal to +0,
 *      NaN after everything (one sort of 64-bit keys);
 *   2. mask: row i of the score-sorted boxes gets bit j (j > i) when
 *      IoU(i, j) > thr, 64-bit words, computed a block of 64 rows at a
 *      time over the threads and only for rows no earlier block removed;
 *   3. resolve: one thread walks each block's rows in order, keeps a box
 *      whose bit is clear in the removed-bitmap and ORs its row into it,
 *      stopping at max_out; kept positions map back to input indices.
 * Batched input (class ids, image offsets, a score pre-filter) runs steps
 * 1-3 for every (image, class) segment, segments spread over the threads,
 * then merges each image's kept boxes by (score desc, index asc) and cuts at
 * max_out per image.
 *
 * The IoU is the continuous xyxy one in binary32, one rounding per
 * operation in the order min/max, sides, clamp at 0, product, area sum,
 * minus the intersection, division; built with -ffp-contract=off so no
 * multiply-add is fused.  The comparison is strict (IoU == thr keeps).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------ ordering */

/* 32-bit key whose ascending order is descending score (-0 as +0, NaN last). */
static uint32_t desc_key(float s)
{
    if (s != s) return 0xffffffffu;
    if (s == 0.0f) s = 0.0f;
    uint32_t u;
    memcpy(&u, &s, 4);
    uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    uint32_t k = ~asc;
    return k == 0xffffffffu ? 0xfffffffeu : k;
}

/* 64 flags (bytes of 0 or 1) to the bits of a word, flag b to bit b: per
 * 8 flags read as a little-endian word v, the product v * 0x0102040810204080
 * puts flag b at bit 56 + b (the partial products are distinct powers of
 * two, so nothing carries into the top byte). */
static uint64_t pack_flags(const unsigned char* f)
{
    uint64_t bits = 0;
    for (int q = 0; q < 8; ++q) {
        uint64_t v;
        memcpy(&v, f + 8 * q, 8);
        bits |= ((v * 0x0102040810204080ull) >> 56) << (8 * q);
    }
    return bits;
}

static int cmp_u64(const void* a, const void* b)
{
    uint64_t x = *(const uint64_t*)a, y = *(const uint64_t*)b;
    return x < y ? -1 : (x > y ? 1 : 0);
}


/* Greedy NMS of the m boxes idx[0..m) (input indices, already in score
 * order), writing at most cap kept input indices to out; returns the count
 * (-1 when out of memory).  sb: scratch of 4 m floats for the sorted boxes.
 *
 * The rows go in blocks of 64.  A block first computes, for each of its
 * rows that no earlier block removed, the row's bits over the columns after
 * it (rows x column chunks spread over the threads when `parallel` is set);
 * then one thread resolves the block in order: a row still clear is kept and
 * ORs its bits into the removed-bitmap.  Rows an earlier block removed are
 * never computed, so the work is about (kept + 63 per block) rows rather
 * than the whole triangle.  The IoU is the continuous xyxy one in binary32
 * (see the file header), both areas formed as (x2 - x1) * (y2 - y1). */
static int64_t greedy_sorted(const float* boxes, const int64_t* idx, int64_t m, float thr, int64_t cap,
                             int parallel, float* sb, int64_t* out)
{
    if (m <= 0 || cap <= 0) return 0;
    const int64_t W = (m + 63) / 64;
    /* the sorted boxes as four coordinate arrays (unit-stride loads in the
     * column loop, which the compiler can run several columns at a time) */
    float *X1 = sb, *Y1 = sb + m, *X2 = sb + 2 * m, *Y2 = sb + 3 * m;
    for (int64_t p = 0; p < m; ++p) {
        const float* b = boxes + 4 * idx[p];
        X1[p] = b[0];
        Y1[p] = b[1];
        X2[p] = b[2];
        Y2[p] = b[3];
    }
    uint64_t* rows = (uint64_t*)malloc(sizeof(uint64_t) * 64 * (size_t)W);  /* one block's rows */
    uint64_t* removed = (uint64_t*)calloc((size_t)W, sizeof(uint64_t));
    if (!rows || !removed) {
        free(rows);
        free(removed);
        return -1;
    }
    const int64_t CH = 16;  /* words (1024 columns) per task */
    int64_t k = 0;
    int stop = 0;
    /* One parallel region for the whole image: per block, the (live row,
     * column chunk) tasks split statically over the threads, then one
     * thread resolves the block; the barriers of `omp for` and `omp single`
     * order the two, and every thread reads k and stop after them. */
#pragma omp parallel if (parallel)
    {
        int64_t lr[64];
        for (int64_t blk = 0; blk < W && !stop; ++blk) {
            const uint64_t live = ~removed[blk];
            const int64_t nr = m - 64 * blk < 64 ? m - 64 * blk : 64;
            const int64_t nch = (W - blk + CH - 1) / CH;
            int64_t nl = 0;
            for (int64_t r = 0; r < nr; ++r)
                if (live >> r & 1) lr[nl++] = r;
#pragma omp for schedule(static)
            for (int64_t t = 0; t < nl * nch; ++t) {
                const int64_t r = lr[t / nch], c = t % nch;
                const int64_t i = 64 * blk + r;
                const float bx1 = X1[i], by1 = Y1[i], bx2 = X2[i], by2 = Y2[i];
                const float ai = (bx2 - bx1) * (by2 - by1);
                const int64_t w1 = blk + (c + 1) * CH < W ? blk + (c + 1) * CH : W;
                for (int64_t w = blk + c * CH; w < w1; ++w) {
                    const int64_t j0 = w << 6;
                    const int64_t jlo = j0 > i ? j0 : i + 1;
                    const int64_t jhi = j0 + 64 < m ? j0 + 64 : m;
                    unsigned char f[64] = {0};
                    for (int64_t j = jlo; j < jhi; ++j) {
                        float xx1 = fmaxf(bx1, X1[j]), yy1 = fmaxf(by1, Y1[j]);
                        float xx2 = fminf(bx2, X2[j]), yy2 = fminf(by2, Y2[j]);
                        float ww = fmaxf(xx2 - xx1, 0.0f), hh = fmaxf(yy2 - yy1, 0.0f);
                        float inter = ww * hh;
                        float aj = (X2[j] - X1[j]) * (Y2[j] - Y1[j]);
                        float uni = (ai + aj) - inter;
                        f[j - j0] = (inter / uni) > thr;
                    }
                    rows[r * W + w] = pack_flags(f);
                }
            }
#pragma omp single
            {
                for (int64_t r = 0; r < nr && k < cap; ++r) {
                    const int64_t i = 64 * blk + r;
                    if (removed[blk] >> r & 1) continue;
                    out[k++] = idx[i];
                    const uint64_t* row = rows + r * W;
                    for (int64_t w = blk; w < W; ++w) removed[w] |= row[w];
                }
                if (k >= cap) stop = 1;
            }
        }
    }
    free(rows);
    free(removed);
    return k;
}

/* ------------------------------------------------------------ entry points */

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int cpu_baseline_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Greedy NMS of one image or a batch, as the library's nms_run defines it:
 *   boxes [n][4] xyxy binary32, scores [n]; class_ids [n] or NULL;
 *   offsets [batch+1] or NULL (one image); a candidate needs score >
 *   score_thr when use_score_thr; max_out per image (<= 0: none).
 * Output: keep holds image b's kept input indices at b * max_out (with
 * max_out) or at offsets[b] (without), counts[b] their number (one image:
 * keep from 0, counts[0]).  Returns the total kept, or -1 on bad arguments
 * or memory exhaustion.
 */
int64_t cpu_baseline_nms(const float* boxes, const float* scores, int64_t n, const int32_t* class_ids,
                         const int64_t* offsets, int32_t batch, float iou_thr, int use_score_thr,
                         float score_thr, int32_t max_out, int64_t* keep, int64_t* counts)
{
    if (n < 0 || (offsets && batch < 1)) return -1;
    const int B = offsets ? batch : 1;
    /* (segment, key, index) order: segment = image * C' + class, where C'
     * covers the largest class id; keys sort descending score, ties by index. */
    int64_t cmax = 0;
    if (class_ids)
        for (int64_t i = 0; i < n; ++i) {
            if (class_ids[i] < 0) return -1;
            if (class_ids[i] > cmax) cmax = class_ids[i];
        }
    const int64_t C = cmax + 1;
    uint64_t* sk = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(n > 0 ? n : 1));
    int64_t* seg = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!sk || !seg) {
        free(sk);
        free(seg);
        return -1;
    }
    int64_t m = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t lo = offsets ? offsets[b] : 0, hi = offsets ? offsets[b + 1] : n;
        if (lo < 0 || hi < lo || hi > n) {
            free(sk);
            free(seg);
                return -1;
        }
        for (int64_t i = lo; i < hi; ++i) {
            if (use_score_thr && !(scores[i] > score_thr)) continue;
            seg[m] = (int64_t)b * C + (class_ids ? class_ids[i] : 0);
            sk[m] = ((uint64_t)desc_key(scores[i]) << 32) | (uint64_t)(i - lo);
            ++m;
        }
    }
    /* Candidates are bucketed by segment (a counting pass), then each
     * segment's keys are sorted on their own. */
    int64_t* perm = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
    uint64_t* rec = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(m > 0 ? m : 1));
    if (!perm || !rec) {
        free(sk);
        free(seg);
        free(perm);
        free(rec);
        return -1;
    }
    for (int64_t r = 0; r < m; ++r) perm[r] = r;
    /* segment-major counting pass, then a key sort inside each segment */
    const int64_t S = (int64_t)B * C;
    int64_t* soff = (int64_t*)calloc((size_t)(S + 1), sizeof(int64_t));
    int64_t* sidx = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
    if (!soff || !sidx) {
        free(sk);
        free(seg);
        free(perm);
        free(rec);
        free(soff);
        free(sidx);
        return -1;
    }
    for (int64_t r = 0; r < m; ++r) soff[seg[r] + 1]++;
    for (int64_t s = 0; s < S; ++s) soff[s + 1] += soff[s];
    {
        int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)(S > 0 ? S : 1));
        if (!fill) {
            free(sk);
            free(seg);
                free(perm);
            free(rec);
            free(soff);
            free(sidx);
            return -1;
        }
        memcpy(fill, soff, sizeof(int64_t) * (size_t)S);
        for (int64_t r = 0; r < m; ++r) sidx[fill[seg[r]]++] = r;
        free(fill);
    }
    /* per segment: sort its keys (score key above, index within the image below) */
    int64_t* kept = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
    int64_t* kcnt = (int64_t*)calloc((size_t)(S > 0 ? S : 1), sizeof(int64_t));
    int err = 0;
    if (!kept || !kcnt) err = 1;
    const int parallel_rows = S <= 1;
#pragma omp parallel for schedule(dynamic, 1) if (!parallel_rows) reduction(| : err)
    for (int64_t s = 0; s < S; ++s) {
        if (err) continue;
        const int64_t lo = soff[s], cnt = soff[s + 1] - lo;
        if (cnt == 0) continue;
        uint64_t* keys = rec + lo;  /* the segment's slice of the key scratch */
        for (int64_t t = 0; t < cnt; ++t) keys[t] = sk[sidx[lo + t]];
        qsort(keys, (size_t)cnt, sizeof(uint64_t), cmp_u64);
        int64_t* ord = perm + lo;
        for (int64_t t = 0; t < cnt; ++t) {
            /* the slot is the index within the image: back to the input index */
            const int64_t b = s / C;
            const int64_t base = offsets ? offsets[b] : 0;
            ord[t] = base + (int64_t)(uint32_t)keys[t];
        }
        float* sb = (float*)malloc(sizeof(float) * 4 * (size_t)cnt);
        if (!sb) {
            err = 1;
            continue;
        }
        const int64_t cap = (!offsets && !class_ids && max_out > 0) ? max_out : cnt;
        const int64_t k = greedy_sorted(boxes, ord, cnt, iou_thr, cap, parallel_rows, sb, kept + lo);
        free(sb);
        if (k < 0) err = 1;
        else kcnt[s] = k;
    }
    int64_t total = 0;
    if (!err) {
        /* per image: merge its segments' kept boxes by (score key, index) */
        uint64_t* mk = (uint64_t*)rec;  /* reuse: at most m keys */
        for (int b = 0; b < B; ++b) {
            int64_t q = 0;
            for (int64_t s = (int64_t)b * C; s < (int64_t)(b + 1) * C; ++s)
                for (int64_t t = 0; t < kcnt[s]; ++t) mk[q++] = (uint64_t)soff[s] + (uint64_t)t;
            /* sort the positions by the kept box's (score key, index) */
            uint64_t* pk = (uint64_t*)malloc(sizeof(uint64_t) * 2 * (size_t)(q > 0 ? q : 1));
            if (!pk) {
                err = 1;
                break;
            }
            const int64_t base = offsets ? offsets[b] : 0;
            for (int64_t t = 0; t < q; ++t) {
                const int64_t i = kept[mk[t]];
                pk[t] = ((uint64_t)desc_key(scores[i]) << 32) | (uint64_t)(uint32_t)(i - base);
            }
            qsort(pk, (size_t)q, sizeof(uint64_t), cmp_u64);
            int64_t c = q;
            if (max_out > 0 && c > max_out) c = max_out;
            int64_t* dst = keep + (max_out > 0 ? (int64_t)b * max_out : base);
            for (int64_t t = 0; t < c; ++t) dst[t] = base + (int64_t)(uint32_t)pk[t];
            free(pk);
            counts[b] = c;
            total += c;
        }
    }
    free(sk);
    free(seg);
    free(perm);
    free(rec);
    free(soff);
    free(sidx);
    free(kept);
    free(kcnt);
    return err ? -1 : total;
}
