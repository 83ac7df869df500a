// Single-image path, front end: optional score pre-filter (warp-aggregated
// atomics) and the stable descending sort, a merge sort of (score key, index)
// keys, fused with the gather of the sorted boxes.
//
// "NMS CUDA代码学习", section 算法与数据流 step 1 (sort by descending score,
// stable) and section "host 侧" (the sort permutation maps kept positions back
// to input indices); "Fastest Matrix NMS in the West (Part 2)", section
// "PyTorch extension" (stable descending sort, then the boxes gathered
// contiguous for the IoU kernel); "YOLOv5后处理GPU移植实战", section 1.2
// (atomic slot counters; per-warp aggregation cuts the contention).
#include "common.cuh"
#include "internal.h"

namespace gbnms {

// Pre-filter: candidates with score > score_thr, compacted with one atomic per
// warp.  The order of the compacted list is not deterministic; the sort below
// includes the input index in its key, so the result is.
__global__ void prefilter_kernel(const float* __restrict__ scores, int n, float score_thr,
                                 int* __restrict__ cand, int* __restrict__ m_count)
{
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    bool pass = i < n && scores[i] > score_thr;
    unsigned ballot = __ballot_sync(FULL, pass);
    if (!ballot) return;
    unsigned l = lane_id();
    int base = 0;
    if (l == static_cast<unsigned>(__ffs(ballot) - 1)) base = atomicAdd(m_count, __popc(ballot));
    base = __shfl_sync(FULL, base, __ffs(ballot) - 1);
    if (pass) cand[base + __popc(ballot & ((1u << l) - 1u))] = i;
}

// Sort on 64-bit (score key << 32 | input index) keys.  The keys are unique,
// so any correct sort of them is the stable descending score order (ties by
// lower index); 0xffff...ff pads and sorts after every real key.
//
// Chunks of MS_CHUNK keys are sorted by bucketed ranking (below), every
// chunk by many CTAs.  Larger inputs then merge pairs of sorted runs in
// global memory, one launch per doubling: a CTA produces one ML_TILE tile of
// the output, loads the two input ranges it covers (found by a 32-way
// search) into shared memory, and each thread merges MS_P outputs after a
// merge-path search for its first one.  Shared memory keeps one spare slot
// per MS_P keys so that lanes MS_P keys apart do not share banks.  The last
// step writes the permutation and the gathered boxes instead of keys.
constexpr int MS_P = 8;                        // keys merged per thread
constexpr int MS_CHUNK = 8192;                 // keys of a bucket-ranked chunk
constexpr uint64_t MS_PAD = ~0ull;

// Shared-memory slot of logical key i: one spare slot after every MS_P keys,
// so the lanes of a warp, MS_P keys apart, hit different banks.
__device__ __forceinline__ int sk(int i) { return i + i / MS_P; }
constexpr int ML_THREADS = 256;                // merge level: threads per CTA
constexpr int ML_TILE = ML_THREADS * MS_P;     // merge level: outputs per CTA
constexpr int ML_SLOTS = ML_TILE + ML_TILE / MS_P;
static_assert(MS_CHUNK % ML_TILE == 0, "merge tiles split the runs evenly");

// Number of A elements among the first d outputs of merge(A, B) (A first on
// ties), A = keys [a0, a0+na) and B = keys [b0, b0+nb) of the skewed buffer.
__device__ __forceinline__ int merge_path(const uint64_t* buf, int a0, int na, int b0, int nb, int d)
{
    int lo = max(0, d - nb), hi = min(d, na);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (buf[sk(a0 + mid)] <= buf[sk(b0 + d - 1 - mid)]) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// MS_P outputs of merge(A, B) starting at output d, into out[].
__device__ __forceinline__ void merge_p(const uint64_t* buf, int a0, int na, int b0, int nb, int d,
                                        uint64_t (&out)[MS_P])
{
    int i = merge_path(buf, a0, na, b0, nb, d), j = d - i;
    uint64_t a = i < na ? buf[sk(a0 + i)] : MS_PAD, b = j < nb ? buf[sk(b0 + j)] : MS_PAD;
#pragma unroll
    for (int u = 0; u < MS_P; ++u) {
        const bool takeA = j >= nb || (i < na && a <= b);
        out[u] = takeA ? a : b;
        if (takeA) { ++i; a = i < na ? buf[sk(a0 + i)] : MS_PAD; }
        else { ++j; b = j < nb ? buf[sk(b0 + j)] : MS_PAD; }
    }
}

// Sorted position r holds key k: the permutation entry and the gathered box
// (no box when the caller sorts without boxes).
__device__ __forceinline__ void emit_sorted(uint64_t k, int r, int m, const float4* __restrict__ boxes,
                                            int* __restrict__ perm, float4* __restrict__ boxes_s)
{
    if (r < m) {
        const int x = static_cast<int>(static_cast<uint32_t>(k));
        perm[r] = x;
        if (boxes) boxes_s[r] = boxes[x];
    }
}

// Bucketed rank within a chunk of MS_CHUNK candidates (positions
// [c*MS_CHUNK, ...), c = blockIdx.y).  A key's sorted position in its chunk
// is the number of smaller keys.  Every CTA of the chunk histograms all of the
// chunk's keys into BR_BUCKETS buckets, scatters them into bucket order in
// shared memory (order inside a bucket does not matter) and then counts, for
// each of its BR_CAND candidates, the smaller keys of its own bucket: the
// work per CTA is linear in the chunk plus the candidates' bucket sizes.
// The bucket of a key is its offset in the [lo, hi] range of the keys of the
// chunk's finite scores, shifted right so that the range fits the buckets
// (keys beyond the range, i.e. of +inf, -inf and NaN, go to the end
// buckets); it is monotone in the key, so buckets come in key order.  The
// range is of whole keys, score and index, so that a run of equal scores
// spreads over buckets by index instead of filling one.
// With one chunk the kernel writes perm and boxes_s (the candidates' boxes
// are loaded with their scores, at the start), otherwise the chunk's
// sorted keys for the merge levels.  It also clears what the mask kernel
// accumulates into: the status, the pair counter, the bitmap of boxes with an
// earlier neighbour and the per-row chunk bitmaps of its candidates' rows.
// Threads of a ranking CTA: 1024 when the input is one chunk (half the
// unrolled code per thread, which is fetched cold after an L2 flush, and the
// chunk's loads spread over more threads), 512 with several chunks (two CTAs
// per SM, so that the chunks' CTAs fit in one wave).
constexpr int BR_THREADS_ONE = 1024;
constexpr int BR_THREADS_MULTI = 512;
constexpr int BR_CAND = 128;                   // candidates ranked per CTA
constexpr int BR_BUCKETS = 4096;

constexpr int BR_SOLO = 64;                    // buckets a single lane scans alone

struct BucketMap {
    uint64_t lo, hi;  // key range of the finite scores
    int shift;        // (hi - lo) >> shift < BR_BUCKETS
    __device__ __forceinline__ int operator()(uint64_t key) const
    {
        if (key < lo) return 0;
        if (key > hi) return BR_BUCKETS - 1;
        return static_cast<int>((key - lo) >> shift);
    }
};

__device__ __forceinline__ uint64_t warp_min_u64(uint64_t v)
{
#pragma unroll
    for (int d = 16; d; d >>= 1) {
        const uint64_t o = __shfl_xor_sync(FULL, v, d);
        v = o < v ? o : v;
    }
    return v;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v)
{
#pragma unroll
    for (int d = 16; d; d >>= 1) {
        const uint64_t o = __shfl_xor_sync(FULL, v, d);
        v = o > v ? o : v;
    }
    return v;
}

template <int BR_THREADS>
__global__ void __launch_bounds__(BR_THREADS)
bucket_rank_kernel(const float* __restrict__ scores, const float4* __restrict__ boxes,
                   const int* __restrict__ cand, const int* __restrict__ m_dev, int m_bound,
                   uint64_t* __restrict__ keys_out, int* __restrict__ perm, float4* __restrict__ boxes_s,
                   int32_t* status, uint64_t* __restrict__ rowbits, int NB, unsigned* __restrict__ ecount,
                   uint64_t* __restrict__ haspred, int* __restrict__ zero8)
{
    constexpr int BR_KPT = MS_CHUNK / BR_THREADS;  // chunk keys per thread
    extern __shared__ __align__(16) uint64_t list[];                 // MS_CHUNK keys, bucket order
    int* start = reinterpret_cast<int*>(list + MS_CHUNK);            // [BR_BUCKETS + 1]
    int* cur = start + BR_BUCKETS + 1;                               // [BR_BUCKETS]
    __shared__ int wsum[BR_THREADS / 32];
    __shared__ uint64_t wlo[BR_THREADS / 32], whi[BR_THREADS / 32];
    __shared__ uint64_t ckey[BR_CAND];  // this CTA's candidates
    __shared__ int crank[BR_CAND];
    pdl_release();  // the mask kernel may be scheduled (it waits for this grid's results)
    pdl_wait();     // a kernel before nms_run (a staging copy, a previous call) has finished
    const int tid = threadIdx.x;
    const int c0 = blockIdx.y * MS_CHUNK;
    const int q0 = c0 + blockIdx.x * BR_CAND;  // this CTA's candidates [q0, q0 + BR_CAND)
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        if (tid == 0) {
            if (status) *status = 0;
            if (ecount) *ecount = 0;
        }
        if (zero8 && tid < 8) zero8[tid] = 0;  // the resolve's flags and barrier counter
    }
    const int r1 = min(q0 + BR_CAND, m_bound);
    if (haspred && (q0 & 63) == 0)
        for (int w = q0 / 64 + tid; w < (r1 + 63) / 64; w += BR_THREADS) haspred[w] = 0;
    if (rowbits)
        for (int64_t q = static_cast<int64_t>(q0) * NB + tid; q < static_cast<int64_t>(r1) * NB; q += BR_THREADS)
            rowbits[q] = 0;
    const int m = m_dev ? *m_dev : m_bound;
    const int cn = min(MS_CHUNK, m - c0);     // keys of this chunk (may be <= 0)
    const bool multi = gridDim.y > 1;
    if (!multi && q0 >= m) return;

    for (int b = tid; b < BR_BUCKETS; b += BR_THREADS) start[b] = 0;
    float4 cbox = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < BR_CAND) {
        const int p = q0 + tid;
        uint64_t key = MS_PAD;
        if (p < m && p < c0 + MS_CHUNK) {
            const int xi = cand ? cand[p] : p;
            key = order_key(scores[xi], static_cast<uint32_t>(xi));
            if (!multi && boxes) cbox = boxes[xi];
        }
        ckey[tid] = key;
    }
    // The chunk's keys, BR_KPT per thread: all index loads, then all score
    // loads, so that each round of loads is in flight at once.
    uint64_t k[BR_KPT];
    int xs[BR_KPT];
    float sc[BR_KPT];
#pragma unroll
    for (int u = 0; u < BR_KPT; ++u) {
        const int t = tid + u * BR_THREADS;
        xs[u] = t < cn ? (cand ? cand[c0 + t] : c0 + t) : -1;
    }
#pragma unroll
    for (int u = 0; u < BR_KPT; ++u) sc[u] = xs[u] >= 0 ? scores[xs[u]] : 0.0f;
    uint64_t lo = ~0ull, hi = 0ull;
#pragma unroll
    for (int u = 0; u < BR_KPT; ++u) {
        k[u] = xs[u] >= 0 ? order_key(sc[u], static_cast<uint32_t>(xs[u])) : MS_PAD;
        if (xs[u] >= 0 && isfinite(sc[u])) {
            lo = min(lo, k[u]);
            hi = max(hi, k[u]);
        }
    }
    const unsigned l = lane_id();
    lo = warp_min_u64(lo);
    hi = warp_max_u64(hi);
    if (l == 0) {
        wlo[tid >> 5] = lo;
        whi[tid >> 5] = hi;
    }
    __syncthreads();
    BucketMap bm;
    constexpr int NWARP = BR_THREADS / 32;
    bm.lo = warp_min_u64(l < NWARP ? wlo[l] : ~0ull);
    bm.hi = warp_max_u64(l < NWARP ? whi[l] : 0ull);
    if (bm.lo > bm.hi) bm.lo = bm.hi = 0ull;  // no finite score
    // Smallest shift with (hi - lo) >> shift < BR_BUCKETS (a power of two).
    static_assert((BR_BUCKETS & (BR_BUCKETS - 1)) == 0, "power-of-two bucket count");
    const int span_bits = 64 - __clzll(static_cast<long long>(bm.hi - bm.lo));
    bm.shift = max(0, span_bits - (31 - __clz(BR_BUCKETS)));
#pragma unroll
    for (int u = 0; u < BR_KPT; ++u)
        if (k[u] != MS_PAD) atomicAdd(&start[bm(k[u])], 1);
    __syncthreads();
    // Exclusive prefix of the bucket counts: thread t owns buckets [8t, 8t+8).
    constexpr int BPT = BR_BUCKETS / BR_THREADS;
    int v[BPT], run = 0;
#pragma unroll
    for (int u = 0; u < BPT; ++u) {
        v[u] = start[tid * BPT + u];
        run += v[u];
    }
    int x = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(FULL, x, d);
        if (static_cast<int>(l) >= d) x += y;
    }
    if (l == 31) wsum[tid >> 5] = x;
    __syncthreads();
    int before = x - run + __reduce_add_sync(FULL, static_cast<int>(l) < (tid >> 5) ? wsum[l] : 0);
#pragma unroll
    for (int u = 0; u < BPT; ++u) {
        start[tid * BPT + u] = before;
        cur[tid * BPT + u] = before;
        before += v[u];
    }
    if (tid == BR_THREADS - 1) start[BR_BUCKETS] = before;
    __syncthreads();
    // Slots in bucket order: every atomic first, then the stores.
    int slot[BR_KPT];
#pragma unroll
    for (int u = 0; u < BR_KPT; ++u) slot[u] = k[u] != MS_PAD ? atomicAdd(&cur[bm(k[u])], 1) : -1;
#pragma unroll
    for (int u = 0; u < BR_KPT; ++u)
        if (slot[u] >= 0) list[slot[u]] = k[u];
    __syncthreads();
    // Rank: thread e < BR_CAND counts the smaller keys of its candidate's
    // bucket alone; a bucket of more than BR_SOLO keys is counted by the
    // candidate's whole warp, lanes splitting it.
    if (tid < BR_CAND) {
        const uint64_t key = ckey[tid];
        int r = q0 + tid - c0;                 // pads keep their place at the end
        bool big = false;
        int s0 = 0, s1 = 0;
        if (key != MS_PAD) {
            const int b = bm(key);
            s0 = start[b];
            s1 = start[b + 1];
            big = s1 - s0 > BR_SOLO;
            if (!big) {
                int c = 0;
#pragma unroll 4
                for (int i = s0; i < s1; ++i) c += list[i] < key;
                r = s0 + c;
            }
        }
        unsigned todo = __ballot_sync(FULL, big);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const uint64_t kk = __shfl_sync(FULL, key, src);
            const int b0 = __shfl_sync(FULL, s0, src), b1 = __shfl_sync(FULL, s1, src);
            int c = 0;
            for (int i = b0 + static_cast<int>(l); i < b1; i += 32) c += list[i] < kk;
            c = __reduce_add_sync(FULL, c);
            if (static_cast<int>(l) == src) r = b0 + c;
        }
        crank[tid] = r;
    }
    __syncthreads();
    if (tid < BR_CAND && q0 + tid < c0 + MS_CHUNK) {
        if (multi) keys_out[c0 + crank[tid]] = ckey[tid];
        else if (crank[tid] < m) {
            perm[crank[tid]] = static_cast<int>(static_cast<uint32_t>(ckey[tid]));
            if (boxes) boxes_s[crank[tid]] = cbox;
        }
    }
}

// Warp-cooperative merge-path search in global memory: the number of A
// elements among the first d outputs of merge(A[0..na), B[0..nb)).  Each step
// probes 32 evenly spaced candidates and keeps the interval where the
// predicate A[i] <= B[d-1-i] changes.
__device__ __forceinline__ int merge_path_warp(const uint64_t* __restrict__ A, int na,
                                               const uint64_t* __restrict__ B, int nb, int d)
{
    int lo = max(0, d - nb), hi = min(d, na);  // answer in [lo, hi]
    const int l = static_cast<int>(lane_id());
    while (hi - lo > 0) {
        const int span = hi - lo;
        const int step = (span + 31) / 32;
        const int mid = lo + l * step;  // probe: is the answer > mid?
        const bool beyond = mid < hi && A[mid] <= B[d - 1 - mid];
        const unsigned ball = __ballot_sync(FULL, beyond);
        // predicate is true for a prefix of probes; the answer lies after the
        // last true probe and at or before the first false one
        const int t = __popc(ball);
        const int nlo = t ? lo + (t - 1) * step + 1 : lo;
        const int nhi = t < 32 ? min(hi, lo + t * step) : hi;
        lo = nlo;
        hi = nhi;
        if (step == 1) break;
    }
    return lo;
}

// One doubling of the global merge: pairs of sorted runs of `run` keys from
// keys_in into keys_out (or, when `last`, into perm and boxes_s).  CTA b makes
// output tile [b*ML_TILE, (b+1)*ML_TILE).
__global__ void __launch_bounds__(ML_THREADS)
merge_level_kernel(const uint64_t* __restrict__ keys_in, uint64_t* __restrict__ keys_out, int run,
                   int last, const int* __restrict__ m_dev, int m_bound,
                   const float4* __restrict__ boxes, int* __restrict__ perm,
                   float4* __restrict__ boxes_s)
{
    __shared__ __align__(16) uint64_t buf[ML_SLOTS];  // ML_TILE keys, A part then B part, skewed
    __shared__ int split[2];
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x;
    const int o0 = blockIdx.x * ML_TILE;
    const int pb = o0 & ~(2 * run - 1);       // start of the merge pair
    const uint64_t* A = keys_in + pb;
    const uint64_t* B = A + run;
    const int warp = tid >> 5;
    if (warp < 2) {
        const int d = o0 - pb + warp * ML_TILE;
        const int i = merge_path_warp(A, run, B, run, d);
        if (lane_id() == 0) split[warp] = i;
    }
    __syncthreads();
    const int d0 = o0 - pb;
    const int ia = split[0], ib = split[1];
    const int ja = d0 - ia, jb = d0 + ML_TILE - ib;
    const int na = ib - ia, nb = jb - ja;
    for (int t = tid; t < na; t += ML_THREADS) buf[sk(t)] = A[ia + t];
    for (int t = tid; t < nb; t += ML_THREADS) buf[sk(na + t)] = B[ja + t];
    __syncthreads();
    uint64_t k[MS_P];
    merge_p(buf, 0, na, na, nb, tid * MS_P, k);
    if (last) {
        const int m = m_dev ? *m_dev : m_bound;
#pragma unroll
        for (int u = 0; u < MS_P; ++u) emit_sorted(k[u], o0 + tid * MS_P + u, m, boxes, perm, boxes_s);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(keys_out + o0 + tid * MS_P);
#pragma unroll
        for (int u = 0; u < MS_P; u += 2)
            dst[u / 2] = make_uint4(static_cast<uint32_t>(k[u]), static_cast<uint32_t>(k[u] >> 32),
                                    static_cast<uint32_t>(k[u + 1]), static_cast<uint32_t>(k[u + 1] >> 32));
    }
}

void launch_prefilter(const float* scores, int n, float score_thr, int* cand, int* m_count,
                      cudaStream_t st)
{
    cudaMemsetAsync(m_count, 0, sizeof(int), st);
    if (n > 0) prefilter_kernel<<<(n + 255) / 256, 256, 0, st>>>(scores, n, score_thr, cand, m_count);
}

int sort_chunks(int m_bound)
{
    int c = (m_bound + MS_CHUNK - 1) / MS_CHUNK;
    int p = 1;
    while (p < c) p *= 2;
    return m_bound > 0 ? p : 1;
}

size_t sort_keys_bytes(int m_bound)
{
    const int c = sort_chunks(m_bound);
    return c > 1 ? 2 * sizeof(uint64_t) * static_cast<size_t>(c) * MS_CHUNK : 0;
}

void launch_sort(const float* scores, const float4* boxes, const int* cand, const int* m_dev,
                 int m_bound, int* perm, float4* boxes_s, uint64_t* keys, int32_t* status,
                 uint64_t* rowbits, int NB, unsigned* ecount, uint64_t* haspred, int* zero8, cudaStream_t st)
{
    const int chunks = sort_chunks(m_bound);
    const int per_chunk = chunks > 1 ? MS_CHUNK / BR_CAND : (m_bound + BR_CAND - 1) / BR_CAND;
    const size_t rank_smem = sizeof(uint64_t) * MS_CHUNK + sizeof(int) * (2 * BR_BUCKETS + 1);
    const size_t half = static_cast<size_t>(chunks) * MS_CHUNK;
    uint64_t* k0 = keys;
    uint64_t* k1 = keys ? keys + half : nullptr;
    const dim3 grid(per_chunk > 0 ? per_chunk : 1, chunks);
    if (chunks == 1) {
        ensure_dynamic_smem(reinterpret_cast<const void*>(bucket_rank_kernel<BR_THREADS_ONE>), rank_smem);
        launch_pdl(bucket_rank_kernel<BR_THREADS_ONE>, grid, dim3(BR_THREADS_ONE), rank_smem, st, scores, boxes,
                   cand, m_dev, m_bound, k0, perm, boxes_s, status, rowbits, NB, ecount, haspred, zero8);
    } else {
        ensure_dynamic_smem(reinterpret_cast<const void*>(bucket_rank_kernel<BR_THREADS_MULTI>), rank_smem);
        launch_pdl(bucket_rank_kernel<BR_THREADS_MULTI>, grid, dim3(BR_THREADS_MULTI), rank_smem, st, scores, boxes,
                   cand, m_dev, m_bound, k0, perm, boxes_s, status, rowbits, NB, ecount, haspred, zero8);
    }
    if (chunks == 1) return;
    const int tiles = chunks * (MS_CHUNK / ML_TILE);
    for (int run = MS_CHUNK; run < chunks * MS_CHUNK; run *= 2) {
        const bool last = 2 * run >= chunks * MS_CHUNK;
        launch_pdl(merge_level_kernel, dim3(tiles), dim3(ML_THREADS), 0, st, k0, k1, run, last ? 1 : 0, m_dev,
                   m_bound, boxes, perm, boxes_s);
        uint64_t* t = k0;
        k0 = k1;
        k1 = t;
    }
}

}  // namespace gbnms
