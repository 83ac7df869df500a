// Resolve of the suppression graph in score order, with the map back to input
// indices.
//
// Two ways to the same result, chosen on the device per call:
//
// Graph path (the sparse pair list fits in shared memory).  Greedy NMS
// decides box j as soon as every earlier box that overlaps it beyond the
// threshold is decided: j is removed when one of them is kept, and kept when
// all of them are removed.  Deciding, in rounds, every box whose earlier
// neighbours are all decided therefore gives exactly the greedy result
// (induction over the score order), in as many rounds as the longest chain of
// such dependencies.  For detector-like inputs that chain is a handful of
// links even when the walk below would take thousands of steps.  One CTA
// keeps a byte per box (the last pass that blocked it), a removed byte per
// box and the live pairs in shared memory; a round is one pass over the pairs
// whose source is still open and one barrier (graph_resolve).  Launched as
// a cluster, four CTAs share passes 0 and 1 and CTA 0 goes on alone
// (graph_cluster_prologue).  Up to 16384
// boxes, the first passes over a longer list run from global memory
// (global_passes) until the rest fits; passes 0 and 1, which need no barrier
// inside, can also run on every SM first (graph_pass0_kernel,
// graph_pass1_kernel).  Lists beyond one CTA above 16384 boxes go to
// graph_grid_kernel, the same rounds on every SM with grid barriers.
//
// Walk (everything else, and a caller's own mask):
// "NMS CUDA代码学习", section Phase 2: one thread block walks the boxes from
// the highest score down with the removed-bitmap in shared memory; a box not
// yet removed is kept and its mask row is ORed into the bitmap, each decision
// visible to the next.  Section "host 侧": the kept sorted positions are
// mapped back through the sort permutation to int64 input indices.
//
// GB300 shape: one CTA, three roles, 64-box tiles.  Whether box b of tile t
// is removed by a kept box depends on
//   (a) the kept sets of tiles t-1 .. t-RV_DR,          -> the resolver warp,
//   (b) the kept sets of tiles t-RV_DR-1 .. t-BAND_L,   -> helper warps,
//   (c) the kept sets of tiles <= t-BAND_L-1,           -> worker warp groups.
// (a) and (b) use the column views of the blocks (tile t-d, tile t) for
// d <= BAND_L, which the helper of tile t builds from the row-major mask (a
// warp transpose per block): lane l ANDs its two boxes' columns with the kept
// sets and one pair of ballots gives the removed word.  (c) ORs the
// kept rows of the row-major mask into a shared removed-bitmap with shared
// atomics, skipping the 256-column chunks the per-row chunk bitmap marks
// all-zero.
//
// A helper folds (b) and (c) into the tile's candidates and also decides the
// tile on them (tile_greedy): a speculative kept set that ignores (a).  The
// resolver then only tests (a): if no box of the speculative kept set is hit,
// the speculation is the answer (boxes hit by (a) were not kept, and a box
// that is not kept suppresses nothing); otherwise it re-decides the tile
// without the boxes (a) removed.  Its critical path per tile is the (a) test
// and the hand-over of the kept set.
//
// The windows arrive by lane-parallel 8-byte cp.async copies of mask words
// (bulk copies cost ~200 cycles of issue each on this SM, too much for one
// small window per tile) into the helpers' shared-memory rings, where the
// helper turns them into column view; the resolver reads the blocks it needs
// from the helper's slot, so it issues no global memory operation of its own.  Every hand-over between roles is
// an mbarrier, waiters off the critical path nap between attempts, and every
// wait is bounded and gives up with NMS_ERR_TIMEOUT.  The resolver owns a
// scheduler partition: the warps that share warp 0's partition (4, 8, ...)
// stay idle.  Kept sets go to shared memory; the output list is written by
// the whole CTA after the walk.
#include <climits>
#include <cstddef>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace gbnms {

constexpr int RV_L = BAND_L;               // tiles covered by the column-view windows
constexpr int RV_DR = 4;                   // distances the resolver tests itself
constexpr int RV_HW = RV_L + 1;            // blocks of a window: the whole band of one tile
constexpr int RV_NH = 4;                   // helper warps (tiles round-robin)
constexpr int RV_HR = 3;                   // window slots per helper
constexpr int RV_WARPS = 32;
constexpr int RV_THREADS = RV_WARPS * 32;
constexpr int RV_WPG = 2;                  // warps per worker group
constexpr int RV_GT = RV_WPG * 32;
constexpr int RV_G = 10;                   // worker groups at most (fewer when the bitmaps are wide)
constexpr int RV_FL_BUDGET = 40 * 1024;    // shared bytes for the workers' chunk bitmaps
constexpr int RV_KR = 32;                  // ring of per-tile hand-overs
constexpr int RV_BATCH = 8;                // kept rows whose loads a worker lane issues together
constexpr int RV_SERIAL = 2;               // conflicts resolved one by one before rounds
constexpr long long RV_WAIT_LIMIT = 1ll << 24;  // wait attempts before giving up
#ifndef GBNMS_RV_NAP_HELPER
#define GBNMS_RV_NAP_HELPER 32
#endif
#ifndef GBNMS_RV_NAP_WORKER
#define GBNMS_RV_NAP_WORKER 256
#endif
constexpr unsigned RV_NAP_HELPER = GBNMS_RV_NAP_HELPER;  // ns between wait attempts (helpers)
constexpr unsigned RV_NAP_WORKER = GBNMS_RV_NAP_WORKER;  // ns between wait attempts (workers)

static_assert(RV_KR >= RV_L + RV_NH, "hand-over ring must outlive the band and the helpers");
static_assert(RV_DR + 1 <= RV_L, "helpers cover at least one distance");
static_assert(RV_G <= 15 && RV_NH + RV_G * RV_WPG <= RV_WARPS - RV_WARPS / 4, "warp roles");

// Worker groups that fit the chunk-bitmap budget for NB words per row.
__host__ __device__ __forceinline__ int resolve_groups(int NB)
{
    const int g = RV_FL_BUDGET / (64 * 8 * (NB > 0 ? NB : 1));
    return g < 1 ? 1 : (g > RV_G ? RV_G : g);
}

struct ResolveShared {
    unsigned long long pub[RV_KR];     // kept set of tile t published (resolver)
    unsigned long long ready[RV_KR];   // speculation for tile t ready (helper)
    unsigned long long done[RV_KR];    // kept rows of tile t applied (worker group)
    uint64_t cand[RV_KR];              // candidates of tile t without distances <= RV_DR
    uint64_t spec[RV_KR];              // greedy kept set of those candidates
    int stop;
    int ntiles;                        // tiles decided (the walk may stop early at max_out)
};

__device__ __forceinline__ int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

__device__ __forceinline__ unsigned smem_addr(const void* p)
{
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* b, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(b)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* b)
{
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_addr(b))
                 : "memory");
}

// One wait attempt for the phase with the given parity.
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* b, unsigned parity)
{
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of use `k` of barrier b; gives up (returns
// false) after RV_WAIT_LIMIT attempts or when `stop` is raised.  try_wait may
// return at once instead of suspending the warp, so waiters off the critical
// path sleep `nap` ns between attempts to leave the issue slots to the warps
// that work.
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, int k, const int* stop,
                                          unsigned nap = 0)
{
    long long w = 0;
    while (!mbar_try_wait(b, static_cast<unsigned>(k) & 1u)) {
        if ((stop && vload(stop)) || ++w > RV_WAIT_LIMIT) return false;
        if (nap) __nanosleep(nap);
    }
    return true;
}

// The band window of tile tt, straight from the row-major mask: the words of
// column tile tt in the 64 rows of each tile tt-d, d = 0..RV_L, one 8-byte
// copy per row, so lane l's pair of slots (2l, 2l+1) of block d holds rows l
// and l+32.  Rows before the first tile or past n are zero-filled.
// commit_group() closes a window.
__device__ __forceinline__ void window_from_mask(uint64_t* dst, const uint64_t* __restrict__ mask, int64_t ldw,
                                                 int tt, int n, unsigned l)
{
#pragma unroll
    for (int d = 0; d <= RV_L; ++d) {
        const int R = tt - d;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = static_cast<int64_t>(R) * 64 + l + 32 * h;
            const bool ok = R >= 0 && row < n;
            const uint64_t* src = ok ? mask + row * ldw + tt : mask;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(smem_addr(dst + d * 64 + 2 * l + h)),
                         "l"(src), "r"(ok ? 8u : 0u)
                         : "memory");
        }
    }
}

// In place: each block of a window from window_from_mask turned into column
// view (lane l's slot pair then holds columns l and l+32: bit r set iff row r
// suppresses that column), keeping only bits above the diagonal in block 0.
__device__ __forceinline__ void window_to_columns(uint64_t* win, unsigned l)
{
    ulonglong2* wv = reinterpret_cast<ulonglong2*>(win);
#pragma unroll 1
    for (int d = 0; d <= RV_L; ++d) {
        const ulonglong2 v = wv[d * 32 + l];
        uint64_t a = v.x, b = v.y;
        if (d == 0) {
            a &= ~0ull << (l + 1);
            b &= l + 33 < 64 ? ~0ull << (l + 33) : 0ull;
        }
        transpose64(a, b);
        wv[d * 32 + l] = make_ulonglong2(a, b);
    }
}
__device__ __forceinline__ void commit_group() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void wait_groups() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void group_bar(int g)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(g + 1), "n"(RV_GT));
}

// Barrier of one worker group that also ORs a predicate over the group.
__device__ __forceinline__ bool group_bar_or(int g, bool v)
{
    unsigned r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(static_cast<unsigned>(v)), "r"(g + 1), "n"(RV_GT));
    return r != 0;
}

// The greedy kept set of one tile.  Lane l holds ca = C[l], cb = C[l+32]
// (column view of the diagonal block: bit k of C[b] set iff box k < b
// suppresses box b) and `cand` the boxes no earlier kept box removed.  A
// candidate with no candidate suppressor inside the tile is kept outright;
// the others ("conflicts") are decided in ascending order, each against the
// boxes kept so far, or by resolve_tile_col when there are many.
__device__ __forceinline__ uint64_t tile_greedy(uint64_t cand, uint64_t ca, uint64_t cb)
{
    const unsigned l = lane_id();
    const bool ia = (cand >> l) & 1ull, ib = (cand >> (l + 32)) & 1ull;
    const uint64_t X = ballot64(ia && (ca & cand) != 0, ib && (cb & cand) != 0);
    if (__popcll(X) > RV_SERIAL) return resolve_tile_col(cand, ca, cb);
    uint64_t kept = cand & ~X;
    uint64_t rest = X;
    while (rest) {
        const int b = __ffsll(static_cast<long long>(rest)) - 1;
        rest &= rest - 1;
        const uint64_t cbits = __shfl_sync(FULL, b < 32 ? ca : cb, b & 31);
        if (!(cbits & kept)) kept |= 1ull << b;
    }
    return kept;
}

// Words of the shared removed-bitmap: the used words plus a 256-column chunk
// of slack, rounded to a multiple of 4.
__host__ __device__ __forceinline__ int resolve_bitmap_words(int m_bound)
{
    return ((m_bound + 63) / 64 + 4 + 3) & ~3;
}

struct ResolveLayout {
    size_t removed, hwin, fl, wlist, kept, opre, total;  // offsets in 64-bit words / bytes
};

__host__ __device__ __forceinline__ ResolveLayout resolve_layout(int m_bound, int NB)
{
    ResolveLayout L;
    const size_t tiles = static_cast<size_t>((m_bound + 63) / 64);
    L.removed = 0;
    L.hwin = L.removed + static_cast<size_t>(resolve_bitmap_words(m_bound));
    L.fl = L.hwin + static_cast<size_t>(RV_NH) * RV_HR * RV_HW * 64;
    L.wlist = L.fl + static_cast<size_t>(resolve_groups(NB)) * 64 * NB;  // bytes [worker warps][64]
    L.kept = L.wlist + static_cast<size_t>(RV_G) * RV_WPG * 64 / 8;
    L.opre = L.kept + tiles;                                     // int[tiles] after kept
    L.total = 8 * L.opre + 4 * tiles;                            // bytes
    return L;
}

// ---------------------------------------------------------------- graph path
constexpr int GR_SMEM = 200 * 1024;   // shared bytes the graph path may take
constexpr int GR_MAX_N = 65536;       // a pair packs two 16-bit sorted positions
constexpr int GR_HEAD = 64;           // words: block-prefix scratch [0,32), barriers at 32 and 34, counts 36..38
constexpr int GR_COPY = 32 * 1024;    // bytes per bulk copy of the pair list

// 32-bit bitmap words for m_bound boxes, rounded up to a multiple of 4 so the
// pair list that follows starts 16-byte aligned.
__host__ __device__ __forceinline__ int graph_words(int m_bound) { return ((m_bound + 31) / 32 + 3) & ~3; }

// Above GR_GRID_MIN_N boxes a list larger than one CTA's shared memory is
// resolved by graph_grid_kernel (all SMs, the list in global memory), up to
// GR_GRID_MAX_PAIRS pairs.
constexpr int GR_GRID_MIN_N = 16384;
// Up to GR_GRID_MIN_N boxes the list holds GR_LIST_X times one CTA's pairs;
// the first passes over a longer list than one CTA holds run from global
// memory.
constexpr unsigned GR_LIST_X = 32;
// The resolve of the box path is launched as a cluster of GR_CLUSTER CTAs,
// which share passes 0 and 1 of lists of GR_CLUSTER_MIN_PAIRS pairs or more
// (graph_cluster_prologue).
constexpr int GR_CLUSTER = 4;
constexpr unsigned GR_CLUSTER_MIN_PAIRS = 2048;
constexpr unsigned GR_GRID_MAX_PAIRS = 1u << 24;
constexpr int GG_THREADS = 1024;

unsigned graph_grid_cap(int m_bound)
{
    if (m_bound <= GR_GRID_MIN_N || m_bound > GR_MAX_N) return 0;
    const unsigned long long all = static_cast<unsigned long long>(m_bound) * (m_bound - 1) / 2;
    return static_cast<unsigned>(all < GR_GRID_MAX_PAIRS ? ((all + 3) & ~3ull) : GR_GRID_MAX_PAIRS);
}

unsigned graph_edge_cap(int m_bound)
{
    if (m_bound <= 0 || m_bound > GR_MAX_N) return 0;
    const long long room = GR_SMEM - 4ll * GR_HEAD - 64ll * graph_words(m_bound);
    return room > 0 ? static_cast<unsigned>((room / 4) & ~3ll) : 0u;
}

unsigned graph_list_cap(int m_bound)
{
    const unsigned e = graph_edge_cap(m_bound), g = graph_grid_cap(m_bound);
    if (g > e) return g;
    const unsigned long long all = static_cast<unsigned long long>(m_bound) * (m_bound - 1) / 2;
    const unsigned long long x = static_cast<unsigned long long>(GR_LIST_X) * e;
    const unsigned long long r = ((all + 3) & ~3ull) < x ? ((all + 3) & ~3ull) : x;
    return r > e ? static_cast<unsigned>(r) : e;
}

size_t graph_smem_bytes(int m_bound)
{
    return 4 * GR_HEAD + 64 * static_cast<size_t>(graph_words(m_bound)) +
           4 * static_cast<size_t>(graph_edge_cap(m_bound));
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* b, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(b)), "r"(bytes)
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from global to shared memory,
// completing on mbarrier b.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* b)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(b))
        : "memory");
}

// Thread-block cluster: this CTA's rank and the cluster's size, a shared
// address of the CTA of rank r (mapa), stores and an add into it, and the
// cluster barrier as its two halves (arrive with release, wait with acquire;
// every thread of every CTA takes both).
__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_size()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_map(const void* p, unsigned rank)
{
    unsigned r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_u8(unsigned addr, unsigned v)
{
    asm volatile("st.shared::cluster.u8 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(unsigned addr, unsigned v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_cluster_v4(unsigned addr)
{
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ unsigned atom_cluster_add(unsigned addr, unsigned v)
{
    unsigned old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;\n" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Kept bits of 32-box word w (lane l: box 32w + l) once the rounds are over.
__device__ __forceinline__ uint32_t kept_word(const uint8_t* RMb, int w, int n, unsigned l)
{
    const int j = 32 * w + static_cast<int>(l);
    return __ballot_sync(FULL, j < n && RMb[j] == 0);
}

// Writes the kept boxes of 32-box words [w0, w1) at positions base, base+1,
// ... (below cap), lane l taking box 32w + l: OW words a step, their ballots
// first and then all their permutation loads (from global memory when the
// permutation did not fit in shared memory), so those latencies overlap.
template <int OW>
__device__ __forceinline__ void write_kept(const uint8_t* RMb, int w0, int w1, int n, unsigned l, int base, int cap,
                                           const int* perm_s, const int* __restrict__ perm,
                                           int64_t* __restrict__ keep)
{
    const uint32_t below = (1u << l) - 1u;
    for (int wb = w0; wb < w1 && base < cap; wb += OW) {
        uint32_t bits[OW];
        int v[OW];
#pragma unroll
        for (int u = 0; u < OW; ++u) bits[u] = wb + u < w1 ? kept_word(RMb, wb + u, n, l) : 0u;
#pragma unroll
        for (int u = 0; u < OW; ++u) {
            const int j = 32 * (wb + u) + static_cast<int>(l);
            v[u] = ((bits[u] >> l) & 1u) ? (perm_s ? perm_s[j] : perm ? perm[j] : j) : 0;
        }
#pragma unroll
        for (int u = 0; u < OW; ++u) {
            const int pos = base + __popc(bits[u] & below);
            if (((bits[u] >> l) & 1u) && pos < cap) keep[pos] = v[u];
            base += __popc(bits[u]);
        }
    }
}

// Passes start, start + 1, ... of graph_resolve over a list too long for
// shared memory, straight from global memory (the per-box bytes FL and RMb
// stay in shared memory).  Thread t owns the 16-byte quads t, t + RV_THREADS, ... of gedges
// and packs its survivors in place into the pair slots of those quads (slot
// s: quad t + RV_THREADS * (s / 4), element s % 4).  Four quads, sixteen
// pairs, are taken a step, and the next step's quads are loaded before this
// step's survivors are stored: a step stores only into quads it or an
// earlier step has loaded.  The body is that of the rounds in shared memory
// for every pass (in pass 0 an open source's store of 2 finds 2 already).
// After each pass a block prefix counts the survivors; once they fit in cap
// pairs each thread copies its own into Es at its prefix.  Returns the next
// pass (*total: the pairs now in Es), or -1 after RV_GLOBAL_PASSES passes,
// or at max_rounds, with too many left.
constexpr int RV_GLOBAL_PASSES = 8;
constexpr int GP_Q = 4;  // quads a step
__device__ __forceinline__ uint32_t quad_at(const uint4& v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ int global_passes(uint32_t* __restrict__ gedges, unsigned E, unsigned cap, uint8_t* FL,
                                             uint8_t* RMb, uint32_t* Es, int* scratch, int start,
                                             int max_rounds, unsigned* total)
{
    const int tid = threadIdx.x;
    const unsigned l = lane_id();
    const int warp = tid >> 5;
    uint4* Q = reinterpret_cast<uint4*>(gedges);
    uint4* Qt = Q + tid;  // the thread's quads, RV_THREADS apart
    // The thread's pairs: four per quad, less the padding of the last quad.
    const unsigned nq = (E + 3) / 4;
    const unsigned mine = nq > static_cast<unsigned>(tid) ? (nq - tid + RV_THREADS - 1) / RV_THREADS : 0u;
    int live = static_cast<int>(4 * mine);
    if (nq && (nq - 1) % RV_THREADS == static_cast<unsigned>(tid)) live -= static_cast<int>(4 * nq - E);
    for (int round = start; round < start + RV_GLOBAL_PASSES && round < max_rounds; ++round) {
        const uint32_t kept_f = static_cast<uint32_t>(round) & 0xffu;
        const uint8_t blk_f = static_cast<uint8_t>(round + 2);
        const int lq = (live + 3) >> 2;  // quads holding live pairs
        uint4 cur[GP_Q];
#pragma unroll
        for (int u = 0; u < GP_Q; ++u) cur[u] = u < lq ? Qt[RV_THREADS * u] : make_uint4(0u, 0u, 0u, 0u);
        int nl = 0;
        for (int k0 = 0; k0 < lq; k0 += GP_Q) {
            uint4 nxt[GP_Q];
#pragma unroll
            for (int u = 0; u < GP_Q; ++u)
                nxt[u] = k0 + GP_Q + u < lq ? Qt[RV_THREADS * (k0 + GP_Q + u)] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 4 * GP_Q; ++u) {
                if (4 * k0 + u >= live) break;
                const uint32_t e = quad_at(cur[u >> 2], u & 3);
                const uint32_t src = e >> 16, j = e & 0xffffu;
                if (RMb[src]) continue;  // a removed source no longer matters
                if (FL[src] == kept_f) {  // kept: the removal is final
                    RMb[j] = 1;
                    continue;
                }
                FL[j] = blk_f;  // open: blocks its target, the pair stays
                gedges[4 * (tid + RV_THREADS * (nl >> 2)) + (nl & 3)] = e;
                ++nl;
            }
#pragma unroll
            for (int u = 0; u < GP_Q; ++u) cur[u] = nxt[u];
        }
        live = nl;
        int x = nl;  // inclusive prefix of the survivors over the warp
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(FULL, x, d);
            if (static_cast<int>(l) >= d) x += y;
        }
        if (l == 31) scratch[warp] = x;
        __syncthreads();
        int before = 0, tot = 0;
#pragma unroll 8
        for (int w = 0; w < RV_WARPS; ++w) {
            const int v = scratch[w];
            before += w < warp ? v : 0;
            tot += v;
        }
        __syncthreads();  // scratch is written again after the next pass
        if (static_cast<unsigned>(tot) <= cap) {
            uint32_t* dst = Es + (before + x - nl);
            const int sq = (nl + 3) >> 2;
            for (int k0 = 0; k0 < sq; k0 += GP_Q) {
                uint4 v[GP_Q];
#pragma unroll
                for (int u = 0; u < GP_Q; ++u)
                    v[u] = k0 + u < sq ? Qt[RV_THREADS * (k0 + u)] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4 * GP_Q; ++u)
                    if (4 * k0 + u < nl) dst[4 * k0 + u] = quad_at(v[u >> 2], u & 3);
            }
            __syncthreads();
            *total = static_cast<unsigned>(tot);
            return round + 1;
        }
    }
    return -1;
}

// Passes 0 and 1 of graph_resolve shared by the C CTAs of a cluster, each
// over its own staged pairs Es[0, Eloc) in warp shares as in the rounds.
// Neither pass needs a barrier inside (pass 0 keeps exactly the sources
// without a source; in pass 1 every byte is 0 or 2, so it keeps nothing), so
// a cluster barrier after each is enough.  Pass 0 stores its removals into
// this CTA's plane; after the barrier each CTA ORs the other CTAs' planes
// into its own (16-byte loads of their shared memory; a plane read while its
// owner merges holds at least the owner's removals, and every bit is a
// removal of pass 0, so the merged planes are all the same).  Pass 1 reads
// the full plane, blocks its targets in CTA 0 and gathers the pairs left at
// CTA 0's Es2 (one reservation per CTA on the count at word 36 of CTA 0).
// gave_up: this CTA's copy did not arrive (word 37 of CTA 0 is raised).
// Every CTA takes the three cluster barriers (the first arrived at by the
// caller).  Returns whether this is CTA 0, which goes on with the rounds
// from pass 2.
__device__ __forceinline__ bool graph_cluster_prologue(uint32_t* Es, unsigned Eloc, bool gave_up, uint8_t* FL,
                                                       uint8_t* RMb, int NWp, uint32_t* Es2, uint32_t* sm,
                                                       unsigned C, unsigned crank)
{
    const int tid = threadIdx.x;
    const unsigned l = lane_id();
    const int warp = tid >> 5;
    const uint32_t lt = (1u << l) - 1u;
    int* scratch = reinterpret_cast<int*>(sm);
    cluster_wait();  // barrier 0: every CTA's planes and CTA 0's counts are set up
    if (gave_up && tid == 0) st_cluster_u32(cluster_map(sm + 37, 0), 1u);
    const unsigned chunk = (Eloc + 32u * RV_WARPS - 1) / (32u * RV_WARPS) * 32u;
    const unsigned wbeg = min(Eloc, static_cast<unsigned>(warp) * chunk);
    unsigned cnt = min(Eloc, wbeg + chunk) - wbeg;
    uint32_t* Ew = Es + wbeg;
    unsigned out = 0;
    for (unsigned k = 0; k < cnt; k += 32) {
        const bool have = k + l < cnt;
        const uint32_t e = have ? Ew[k + l] : 0u;
        const bool kept = have && FL[e >> 16] == 0;
        if (kept) RMb[e & 0xffffu] = 1;
        const bool stay = have && !kept;
        const uint32_t b = __ballot_sync(FULL, stay);  // every lane has read its pair
        if (stay) Ew[out + __popc(b & lt)] = e;
        out += __popc(b);
    }
    cnt = out;
    cluster_arrive();
    cluster_wait();  // barrier 1: every CTA's removals of pass 0 are in its plane
    uint4* R4 = reinterpret_cast<uint4*>(RMb);
    for (int w = tid; w < 2 * NWp; w += RV_THREADS) {
        uint4 v = R4[w];
        for (unsigned q = 1; q < C; ++q) {
            const uint4 o = ld_cluster_v4(cluster_map(R4 + w, (crank + q) % C));
            v = make_uint4(v.x | o.x, v.y | o.y, v.z | o.z, v.w | o.w);
        }
        R4[w] = v;
    }
    __syncthreads();
    const unsigned fl0 = cluster_map(FL, 0);
    out = 0;
    for (unsigned k = 0; k < cnt; k += 32) {
        const bool have = k + l < cnt;
        const uint32_t e = have ? Ew[k + l] : 0u;
        const bool stay = have && RMb[e >> 16] == 0;
        if (stay) st_cluster_u8(fl0 + (e & 0xffffu), 3u);  // blocked in pass 1
        const uint32_t b = __ballot_sync(FULL, stay);
        if (stay) Ew[out + __popc(b & lt)] = e;
        out += __popc(b);
    }
    cnt = out;
    if (l == 0) scratch[warp] = static_cast<int>(cnt);
    __syncthreads();
    const int wc = scratch[l];
    const int total = __reduce_add_sync(FULL, wc);
    const int before = __reduce_add_sync(FULL, static_cast<int>(l) < warp ? wc : 0);
    if (tid == 0) sm[38] = total ? atom_cluster_add(cluster_map(sm + 36, 0), static_cast<unsigned>(total)) : 0u;
    __syncthreads();
    const unsigned dst = cluster_map(Es2, 0) + 4u * (sm[38] + static_cast<unsigned>(before));
    for (unsigned k = l; k < cnt; k += 32) st_cluster_u32(dst + 4u * k, Ew[k]);
    cluster_arrive();
    cluster_wait();  // barrier 2: CTA 0 holds every pair left and every block of pass 1
    return crank == 0;
}

// Rounds over the pair list gedges[0..E) of n sorted boxes (haspred: bit j
// set iff box j has a pair).  Returns false, with nothing written, when the
// rounds outnumber the walk's tiles plus 16 (a long chain of dependencies:
// the walk is then the faster way).
//
// Shared layout: the head of GR_HEAD words (block-prefix scratch at [0, 32),
// the copy barrier at 32, the permutation's own barrier at 34 and the
// cluster's counts at 36..38), then one byte per box holding the last pass
// that blocked it (plus 2, mod 256), then one "removed" byte per box, then
// the live pairs.  Byte planes keep a warp's
// stores conflict-free: its pairs come from one 128-column tile of the mask,
// so their targets are 128 consecutive bytes.  Each warp owns an equal
// contiguous share of the list and compacts it in place.
//
// One pass per round and one barrier: a source is kept in pass r when it is
// not removed and no open box blocked it in pass r - 1.  A box blocked in
// pass r was blocked in pass r - 1 too (its pairs only leave and an open
// source was open before), so a byte written in pass r changes no reader's
// decision in that pass; and a kept source's pairs all leave in the first
// pass that finds it kept, so a live source's byte is r, r + 1 or r + 2 (mod
// 256) and the wrap is harmless.  A pair leaves the list once its source is
// decided; when none is left, the kept boxes are the ones not removed.
//
// Pass 0 is known in advance: a source without a source of its own is kept
// and every other one is open, so a box with a source ends pass 0 removed or
// blocked.  Its byte therefore starts at 2 (blocked in pass 0; 0 for a box
// without a source), and pass 0 only removes: it reads no removed byte
// (nothing is removed before it) and stores no block.
//
// kLong: the list is longer than cap_words and is not staged; its first
// passes run from global memory (global_passes), the rest here once the
// survivors fit.  kPre: passes 0 and 1 were done over all SMs
// (graph_pass0_kernel, graph_pass1_kernel): gedges holds the pairs left
// after them, pre->removed the removed bytes and pre->blocked a 3 for each
// box blocked in pass 1; the rounds start at pass 2.  kCluster: the CTAs of
// this thread-block cluster share passes 0 and 1 (graph_cluster_prologue
// below), and CTA 0 goes on alone.  Separate instances keep the common one's
// code as it is.
template <bool kLong, bool kPre, bool kCluster = false>
__device__ __forceinline__ bool graph_resolve(uint32_t* __restrict__ gedges, unsigned E, unsigned cap_words,
                              const uint32_t* __restrict__ haspred, int n, int NWp, uint32_t hp_tid,
                              const int* __restrict__ perm, int max_out, int64_t* __restrict__ keep,
                              int64_t* __restrict__ counts, int32_t* status, uint32_t* sm,
                              int* done_out, const uint8_t* __restrict__ pre_rm = nullptr,
                              const uint8_t* __restrict__ pre_blk = nullptr)
{
    int* scratch = reinterpret_cast<int*>(sm);
    unsigned long long* bar = reinterpret_cast<unsigned long long*>(sm + 32);
    unsigned long long* pbar = reinterpret_cast<unsigned long long*>(sm + 34);  // kCluster: the permutation
    uint8_t* FL = reinterpret_cast<uint8_t*>(sm + GR_HEAD);
    uint8_t* RMb = FL + 32 * NWp;
    uint32_t* Es = sm + GR_HEAD + 16 * NWp;
    const int tid = threadIdx.x;
    const unsigned l = lane_id();
    const int warp = tid >> 5;
    const int NW = (n + 31) / 32;

    // Stage the list with bulk copies (the list is 16-byte aligned and padded
    // to a multiple of 4 pairs) while the bitmaps are set up; the sort
    // permutation follows it when both fit (the output then maps positions
    // from shared memory).
    //
    // kCluster: CTA crank of C stages pairs [my0, my0 + Eloc) of the list
    // (shares of S pairs, a multiple of 4); CTA 0 also stages the permutation
    // after its share, when its share, the permutation and all E pairs fit
    // (the pairs left after pass 1 gather after them, at Es2), on a barrier
    // of its own that only the output waits for.
    const unsigned C = kCluster ? cluster_size() : 1u;
    const unsigned crank = kCluster ? cluster_rank() : 0u;
    const unsigned S = kCluster ? (((E + C - 1) / C + 3) & ~3u) : E;
    const unsigned my0 = kCluster ? min(E, crank * S) : 0u;
    const unsigned Eloc = kCluster ? min(E, my0 + S) - my0 : E;
    const unsigned bytes = kLong ? 0u : 16u * ((Eloc + 3) / 4);
    const unsigned ncopy = (bytes + GR_COPY - 1) / GR_COPY;
    const unsigned pbytes = 16u * ((static_cast<unsigned>(n) + 3) / 4);
    const bool perm0 = kCluster && perm && S + pbytes / 4 + E <= cap_words;
    uint32_t* Es2 = Es + S + (perm0 ? pbytes / 4 : 0u);
    const bool perm_here =
        kCluster ? perm0 && crank == 0 : !kLong && perm && (bytes + pbytes) / 4 <= cap_words;
    const unsigned pofs = kCluster ? 4u * S : bytes;  // byte offset of the permutation
    const int* perm_s = perm_here ? reinterpret_cast<const int*>(reinterpret_cast<const char*>(Es) + pofs) : nullptr;
    const unsigned pcopy = perm_here ? (pbytes + GR_COPY - 1) / GR_COPY : 0u;
    if (tid == 0) {
        mbar_init(bar, 1);
        if (kCluster) mbar_init(pbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    const unsigned tx = bytes + (perm_here && !kCluster ? pbytes : 0u);  // bytes the barrier waits for
    if (tid == 0 && tx) mbar_expect_tx(bar, tx);
    if (kCluster && tid == 0 && perm_here) mbar_expect_tx(pbar, pbytes);
    __syncwarp();
    if (warp == 0 && l < ncopy) {
        const unsigned off = l * GR_COPY;
        const unsigned len = min(static_cast<unsigned>(GR_COPY), bytes - off);
        bulk_g2s(reinterpret_cast<char*>(Es) + off, reinterpret_cast<const char*>(gedges + my0) + off, len, bar);
    }
    if (warp == 1 && l < pcopy) {
        const unsigned off = l * GR_COPY;
        const unsigned len = min(static_cast<unsigned>(GR_COPY), pbytes - off);
        bulk_g2s(reinterpret_cast<char*>(Es) + pofs + off, reinterpret_cast<const char*>(perm) + off, len,
                 kCluster ? pbar : bar);
    }
    for (int w = tid; w < NW; w += RV_THREADS) {
        // A box with a source starts blocked in pass 0 (word tid was loaded
        // with the pair count).
        const uint32_t hp = w == tid ? hp_tid : haspred[w];
        uint32_t bx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) bx[q] = (((hp >> (4 * q)) & 0xfu) * 0x00204081u & 0x01010101u) << 1;  // bits -> 0/2
        uint4* fq = reinterpret_cast<uint4*>(FL + 32 * w);
        uint4* rq = reinterpret_cast<uint4*>(RMb + 32 * w);
        if (kPre) {  // 2 | 3 = 3: a box blocked in pass 1 has a source
            const uint4* bq = reinterpret_cast<const uint4*>(pre_blk + 32 * w);
            const uint4 b0 = bq[0], b1 = bq[1];
            fq[0] = make_uint4(bx[0] | b0.x, bx[1] | b0.y, bx[2] | b0.z, bx[3] | b0.w);
            fq[1] = make_uint4(bx[4] | b1.x, bx[5] | b1.y, bx[6] | b1.z, bx[7] | b1.w);
            const uint4* pq = reinterpret_cast<const uint4*>(pre_rm + 32 * w);
            rq[0] = pq[0];
            rq[1] = pq[1];
        } else {
            fq[0] = make_uint4(bx[0], bx[1], bx[2], bx[3]);
            fq[1] = make_uint4(bx[4], bx[5], bx[6], bx[7]);
            rq[0] = make_uint4(0u, 0u, 0u, 0u);
            rq[1] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (kCluster) {
        if (tid == 0) {
            sm[36] = 0u;  // CTA 0: pairs gathered at Es2
            sm[37] = 0u;  // CTA 0: some CTA's copy gave up
        }
        cluster_arrive();  // this CTA's planes are set up (barrier 0, waited for below)
    }
    bool copied = true;
    if (tx) {
        long long tries = 0;
        while (!mbar_try_wait(bar, 0)) {
            if (++tries > RV_WAIT_LIMIT) { copied = false; break; }
            __nanosleep(64);
        }
    }
    const bool all_copied = __syncthreads_and(copied);
    if (tid == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_addr(bar)) : "memory");
    if (!kCluster && !all_copied) {
        if (tid == 0) {
            if (status) set_status(status, NMS_ERR_TIMEOUT);
            counts[0] = 0;
        }
        return true;
    }
    // kCluster, CTA 0: waits for the permutation's copy; on giving up raises
    // the status, writes a zero count and returns false.
    auto perm_ready = [&]() -> bool {
        bool got = true;
        long long tries = 0;
        while (!mbar_try_wait(pbar, 0)) {
            if (++tries > RV_WAIT_LIMIT) { got = false; break; }
            __nanosleep(64);
        }
        const bool all_got = __syncthreads_and(got);
        if (tid == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_addr(pbar)) : "memory");
        if (!all_got && tid == 0) {
            if (status) set_status(status, NMS_ERR_TIMEOUT);
            counts[0] = 0;
        }
        return all_got;
    };
    const int max_rounds = (n + 63) / 64 + 16;
    int round0 = kPre ? 2 : 0;  // the first pass over the list in shared memory
    uint32_t* Eb = Es;          // the list the rounds run over
    if (kCluster) {
        if (!graph_cluster_prologue(Es, all_copied ? Eloc : 0u, !all_copied, FL, RMb, NWp, Es2, sm, C, crank))
            return true;  // CTAs 1 .. C-1 are done
        if (sm[37]) {     // a copy gave up: nothing is decided
            if (perm_here) perm_ready();  // no copy into this CTA stays in flight
            if (tid == 0) {
                if (status) set_status(status, NMS_ERR_TIMEOUT);
                counts[0] = 0;
            }
            return true;
        }
        E = sm[36];
        Eb = Es2;
        round0 = 2;
    }
    if (kLong) {
        unsigned left = 0;
        round0 = global_passes(gedges, E, cap_words, FL, RMb, Es, scratch, round0, max_rounds, &left);
        if (round0 < 0) return false;
        E = left;
    }
    // Warp w owns the pairs [wbeg, wbeg + cnt): 32 a step, one a lane, its
    // survivors packed in place at the front by a ballot.  A live pair in
    // pass r: a removed source no longer matters; a source that no open box
    // blocked in the previous pass (its byte == r mod 256) is kept and removes
    // its target at once (the removal is final, so other pairs may see it in
    // this same pass); any other source is still open, blocks its target for
    // this pass (in pass 0 the target's byte already says so) and its pair
    // stays.  Both are plain byte stores (every writer of a byte in one pass
    // stores the same value).
    const unsigned chunk = (E + 32u * RV_WARPS - 1) / (32u * RV_WARPS) * 32u;
    const unsigned wbeg = min(E, static_cast<unsigned>(warp) * chunk);
    unsigned cnt = min(E, wbeg + chunk) - wbeg;
    uint32_t* Ew = Eb + wbeg;
    const uint32_t lt = (1u << l) - 1u;
    // Pass 0: a source without a source of its own (byte 0) is kept and
    // removes its target; every other pair stays.
    bool any = E > 0u;
    if (round0 == 0) {
        unsigned out = 0;
        for (unsigned k = 0; k < cnt; k += 32) {
            const bool have = k + l < cnt;
            const uint32_t e = have ? Ew[k + l] : 0u;
            const bool kept = have && FL[e >> 16] == 0;
            if (kept) RMb[e & 0xffffu] = 1;
            const bool stay = have && !kept;
            const uint32_t b = __ballot_sync(FULL, stay);  // every lane has read its pair
            if (stay) Ew[out + __popc(b & lt)] = e;
            out += __popc(b);
        }
        cnt = out;
        any = __syncthreads_or(cnt > 0u);
    }
    for (int round = round0 > 0 ? round0 : 1; any; ++round) {
        if (round == max_rounds) {
            // kCluster: the walk reuses the shared memory the permutation's
            // copy may still be writing.
            if (kCluster && perm_here && !perm_ready()) return true;
            return false;
        }
        const uint32_t kept_f = static_cast<uint32_t>(round) & 0xffu;
        const uint8_t blk_f = static_cast<uint8_t>(round + 2);
        unsigned out = 0;
        for (unsigned k = 0; k < cnt; k += 32) {
            const bool have = k + l < cnt;
            const uint32_t e = have ? Ew[k + l] : 0u;
            const uint32_t src = e >> 16, j = e & 0xffffu;
            const uint32_t rm = have ? RMb[src] : 1u;
            const uint32_t f = have ? FL[src] : 0u;
            const bool kept = rm == 0u && f == kept_f;
            const bool open = rm == 0u && f != kept_f;
            if (kept) RMb[j] = 1;
            if (open) FL[j] = blk_f;
            const uint32_t b = __ballot_sync(FULL, open);  // every lane has read its pair
            if (open) Ew[out + __popc(b & lt)] = e;
            out += __popc(b);
        }
        cnt = out;
        any = __syncthreads_or(cnt > 0u);
    }
    if (kCluster && perm_here && !perm_ready()) return true;
    // Output: warp w owns 32-box words [w*wpw, (w+1)*wpw); a block-wide
    // prefix of the warps' kept counts places them, and within a word lane l
    // writes box 32w+l, so loads of perm and stores of keep are coalesced.
    const int wpw = (NW + 31) / 32;
    const int w0 = min(warp * wpw, NW), w1 = min(w0 + wpw, NW);
    // Kept = boxes of the warp's words less the removed ones; a removed byte
    // is 0 or 1 and no box past n is ever removed, so popcounts of 16-byte
    // loads count them.
    int c = static_cast<int>(l) == 0 ? max(0, min(32 * w1, n) - 32 * w0) : 0;
    for (int j0 = 32 * w0 + 16 * static_cast<int>(l); j0 < 32 * w1; j0 += 512) {
        const uint4 q = *reinterpret_cast<const uint4*>(RMb + j0);
        c -= __popc(q.x) + __popc(q.y) + __popc(q.z) + __popc(q.w);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(FULL, c, d);
    if (l == 0) scratch[warp] = c;
    __syncthreads();
    // Every warp sums the counts of the warps before it (one barrier).
    const int wc = scratch[l];
    const int total = __reduce_add_sync(FULL, wc);
    const int cap = max_out > 0 ? max_out : INT_MAX;
    const int base = __reduce_add_sync(FULL, static_cast<int>(l) < warp ? wc : 0);
    // Words [w0, w1) in steps of eight when the warp has that many, else two
    // (a short body, fetched cold after an L2 flush).
    if (w1 - w0 >= 8)
        write_kept<8>(RMb, w0, w1, n, l, base, cap, perm_s, perm, keep);
    else
        write_kept<2>(RMb, w0, w1, n, l, base, cap, perm_s, perm, keep);
    if (tid == 0) {
        counts[0] = total < cap ? total : cap;
        if (done_out && total >= cap) *done_out = 1;
    }
    return true;
}

// kPre: passes 0 and 1 over a list longer than ecap ran on all SMs first
// (launch_graph_prepass), their results in pre.
template <bool kPre>
__global__ void __launch_bounds__(RV_THREADS, 1)
resolve_single_kernel(const uint64_t* __restrict__ mask, int64_t ldw,
                      const uint64_t* __restrict__ rowbits, int NB,
                      uint32_t* __restrict__ edges, const unsigned* __restrict__ ecount,
                      unsigned ecap, unsigned lcap, const uint32_t* __restrict__ haspred,
                      const int* __restrict__ m_dev, int m_bound, const int* __restrict__ perm,
                      int max_out, int64_t* __restrict__ keep, int64_t* __restrict__ counts,
                      int32_t* status, int limit, const int* __restrict__ done_in, int* done_out,
                      const int* __restrict__ grid_done, GraphPre pre)
{
    extern __shared__ __align__(128) uint64_t smem[];
    __shared__ ResolveShared S;

    pdl_wait();  // the mask (or an earlier kernel) has finished
    // Everything read from the earlier kernels, loaded together before any
    // store: the stage flags, the box and pair counts, and the neighbour
    // bitmap's word of this thread.
    const int was_done = done_in ? *done_in : 0;
    const int grid_did = grid_done ? *grid_done : 0;
    const int n_all = m_dev ? *m_dev : m_bound;
    const unsigned E = edges ? *ecount : 0u;
    const unsigned E2 = kPre && edges ? *pre.ecount : 0u;
    const uint32_t hp_tid =
        edges && haspred && static_cast<int>(threadIdx.x) < (m_bound + 31) / 32 ? haspred[threadIdx.x] : 0u;
    if (was_done) return;  // an earlier stage already finished
    if (grid_did) return;  // graph_grid_kernel resolved this stage
    const int n = min(n_all, limit);
    // Launched as a cluster, CTAs 1 .. C-1 only help with passes 0 and 1 of
    // the graph path; everything else is CTA 0's.
    const unsigned crank = cluster_rank();
    if (done_out && threadIdx.x == 0 && crank == 0) *done_out = n >= n_all;  // raised below on max_out
    if (edges) {
        // A list beyond shared memory is compacted in place by the first
        // passes: only the last stage may do that, and only when no all-SM
        // pass ran over it before.
        uint32_t* sm = reinterpret_cast<uint32_t*>(smem);
        const int NWp = graph_words(m_bound);
        const unsigned C = cluster_size();
        const bool shared = !kPre && C > 1 && E >= GR_CLUSTER_MIN_PAIRS && E <= ecap &&
                            (((E + C - 1) / C + 3) & ~3u) + E <= ecap;
        if (shared) {
            // Only CTA 0 comes back, when the rounds outnumber the limit.
            if (graph_resolve<false, false, true>(edges, E, ecap, haspred, n, NWp, hp_tid, perm, max_out, keep,
                                                  counts, status, sm, done_out))
                return;
        } else if (crank != 0) {
            return;
        } else if (E <= ecap) {
            if (graph_resolve<false, false>(edges, E, ecap, haspred, n, NWp, hp_tid, perm, max_out, keep, counts,
                                            status, sm, done_out))
                return;
        } else if (kPre && E <= lcap) {
            // The pairs left after passes 0 and 1 (the list was complete).
            if (E2 <= ecap) {
                if (graph_resolve<false, true>(pre.edges, E2, ecap, haspred, n, NWp, hp_tid, perm, max_out, keep,
                                               counts, status, sm, done_out, pre.removed, pre.blocked))
                    return;
            } else if (E2 <= pre.cap) {
                if (graph_resolve<true, true>(pre.edges, E2, ecap, haspred, n, NWp, hp_tid, perm, max_out, keep,
                                              counts, status, sm, done_out, pre.removed, pre.blocked))
                    return;
            }
        } else if (!kPre && E <= lcap && !grid_done && n >= n_all) {
            if (graph_resolve<true, false>(edges, E, ecap, haspred, n, NWp, hp_tid, perm, max_out, keep, counts,
                                           status, sm, done_out))
                return;
        }
        __syncthreads();  // the walk reuses the shared memory
    }
    if (crank != 0) return;
    const int T = (n + 63) / 64;              // tiles
    const int T256 = (n + 255) / 256;         // 256-column chunks
    const ResolveLayout LY = resolve_layout(m_bound, NB);
    const int G = resolve_groups(NB);         // worker groups
    uint64_t* removed = smem + LY.removed;
    uint64_t* hwin = smem + LY.hwin;          // [RV_NH][RV_HR][RV_HW*64]
    uint64_t* fl = smem + LY.fl;              // [G][64][NB]
    unsigned char* wlist = reinterpret_cast<unsigned char*>(smem + LY.wlist);  // per worker warp
    uint64_t* kept = smem + LY.kept;          // [tiles]
    int* opre = reinterpret_cast<int*>(smem + LY.opre);

    const int Wpad = resolve_bitmap_words(m_bound);
    for (int w = threadIdx.x; w < Wpad; w += blockDim.x) removed[w] = 0;
    if (threadIdx.x < RV_KR) {
        mbar_init(&S.pub[threadIdx.x], 1);
        mbar_init(&S.ready[threadIdx.x], 1);
        mbar_init(&S.done[threadIdx.x], 1);
    }
    if (threadIdx.x == 0) { S.stop = 0; S.ntiles = 0; }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    __syncthreads();

    const unsigned l = lane_id();
    const int warp = threadIdx.x >> 5;

    const int role = (warp & 3) == 0 ? -1 : warp - 1 - warp / 4;  // index among non-idle warps
    if (warp == 0) {
        // ------------------------------------------------------------ resolver
        uint64_t Kh[RV_DR + 1];  // Kh[d] = kept set of tile t-d (0 before the first tile)
#pragma unroll
        for (int d = 0; d <= RV_DR; ++d) Kh[d] = 0;
        int count = 0, t = 0;
        bool timeout = false;
        for (; t < T; ++t) {
            if (!mbar_wait(&S.ready[t % RV_KR], t / RV_KR, nullptr)) { timeout = true; break; }
            // The helper of tile t left the tile's band window in its slot.
            const int hh = t % RV_NH, hi = t / RV_NH;
            const ulonglong2* wv = reinterpret_cast<const ulonglong2*>(
                hwin + (static_cast<size_t>(hh) * RV_HR + hi % RV_HR) * RV_HW * 64);
            uint64_t xa = 0, xb = 0;
#pragma unroll
            for (int d = 1; d <= RV_DR; ++d) {
                const ulonglong2 v = wv[d * 32 + l];
                xa |= v.x & Kh[d];
                xb |= v.y & Kh[d];
            }
            const uint64_t near = ballot64(xa != 0, xb != 0);
            uint64_t K = S.spec[t % RV_KR];
            if (K & near) {  // the speculation kept a box a recent tile removes: re-decide
                const ulonglong2 dg = wv[l];
                K = resolve_tile_col(S.cand[t % RV_KR] & ~near, dg.x, dg.y);
            }
            const int nk = __popcll(K);
            const bool last = max_out > 0 && count + nk >= max_out;
            if (last) K = lowest_bits(K, max_out - count);
            count += nk;
            if (l == 0) {
                kept[t] = K;
                mbar_arrive(&S.pub[t % RV_KR]);  // release: kept[t] visible
            }
            if (last) { ++t; break; }
#pragma unroll
            for (int d = RV_DR; d > 1; --d) Kh[d] = Kh[d - 1];
            Kh[1] = K;
        }
        if (l == 0) {
            S.ntiles = t;
            if (timeout && status) set_status(status, NMS_ERR_TIMEOUT);
            __threadfence_block();
            *reinterpret_cast<volatile int*>(&S.stop) = 1;
        }
    } else if (role >= 0 && role < RV_NH) {
        // ------------------------------------------------------------- helpers
        const int h = role;
        uint64_t* myw = hwin + static_cast<size_t>(h) * RV_HR * RV_HW * 64;
        auto fill = [&](int i) {  // own tile i: its whole band window into slot i % RV_HR
            const int tt = h + RV_NH * i;
            if (tt < T) window_from_mask(myw + static_cast<size_t>(i % RV_HR) * RV_HW * 64, mask, ldw, tt, n, l);
            commit_group();
        };
        for (int i = 0; i < RV_HR - 1; ++i) fill(i);
        for (int i = 0; h + RV_NH * i < T; ++i) {
            const int t = h + RV_NH * i;
            // The slot of own tile i-1 (tile t-RV_NH) is free once the resolver
            // has published that tile; refill it with own tile i+RV_HR-1.
            if (i > 0 && !mbar_wait(&S.pub[(t - RV_NH) % RV_KR], (t - RV_NH) / RV_KR, &S.stop, RV_NAP_HELPER))
                break;
            fill(i + RV_HR - 1);
            // Kept sets of tiles <= t-RV_DR-1, and the workers' part of word t:
            // worker groups finish tiles out of order, so wait for every tile
            // since this helper's previous tile (t-RV_NH): together with that
            // tile's waits, all tiles <= t-RV_L-1 are applied.
            if (t - RV_DR - 1 >= 0 &&
                !mbar_wait(&S.pub[(t - RV_DR - 1) % RV_KR], (t - RV_DR - 1) / RV_KR, &S.stop, RV_NAP_HELPER))
                break;
            bool ok = true;
            for (int f = max(t - RV_L - RV_NH, 0); ok && f <= t - RV_L - 1; ++f)
                ok = mbar_wait(&S.done[f % RV_KR], f / RV_KR, &S.stop, RV_NAP_HELPER);
            if (!ok) break;
            wait_groups<RV_HR - 1>();
            __syncwarp();
            window_to_columns(myw + static_cast<size_t>(i % RV_HR) * RV_HW * 64, l);
            __syncwarp();
            const ulonglong2* wv =
                reinterpret_cast<const ulonglong2*>(myw + static_cast<size_t>(i % RV_HR) * RV_HW * 64);
            uint64_t xa = 0, xb = 0;
#pragma unroll
            for (int d = RV_DR + 1; d <= RV_L; ++d) {
                const uint64_t Kd = t - d >= 0 ? kept[t - d] : 0ull;
                const ulonglong2 v = wv[d * 32 + l];
                xa |= v.x & Kd;
                xb |= v.y & Kd;
            }
            const int rem = n - t * 64;
            const uint64_t valid = rem >= 64 ? ~0ull : ((1ull << rem) - 1ull);
            const uint64_t cand = ~(removed[t] | ballot64(xa != 0, xb != 0)) & valid;
            const ulonglong2 dg = wv[l];
            const uint64_t spec = tile_greedy(cand, dg.x, dg.y);
            if (l == 0) {
                S.cand[t % RV_KR] = cand;
                S.spec[t % RV_KR] = spec;
                mbar_arrive(&S.ready[t % RV_KR]);
            }
            __syncwarp();
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (role >= RV_NH && (role - RV_NH) / RV_WPG < G) {
        // ------------------------------------------------------------- workers
        const int wk = role - RV_NH;  // index among worker warps
        const int g = wk / RV_WPG;
        const int wg = wk % RV_WPG;
        const int gt = wg * 32 + static_cast<int>(l);
        uint64_t* gfl = fl + static_cast<size_t>(g) * 64 * NB;
        for (int r = g; r < T; r += G) {
            // Chunk bitmaps of the tile's 64 rows (independent of the decision).
            if (rowbits) {
                for (int q = gt; q < 64 * NB; q += RV_GT) {
                    const int64_t i = static_cast<int64_t>(r) * 64 + q / NB;
                    gfl[q] = i < n ? rowbits[i * NB + q % NB] : 0ull;
                }
            }
            const bool stop = group_bar_or(g, !mbar_wait(&S.pub[r % RV_KR], r / RV_KR, &S.stop, RV_NAP_WORKER));
            if (stop) break;
            const uint64_t K = kept[r];
            // Warp wg of the group takes the kept rows of rank wg, wg+RV_WPG, ...:
            // a warp-parallel compaction writes them to the warp's row list.
            unsigned char* rows = wlist + static_cast<size_t>(wk) * 64;
            int nmine = 0;
            {
                const int nlo = __popc(static_cast<unsigned>(K));
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int b = static_cast<int>(l) + 32 * hh;
                    const bool set = (K >> b) & 1ull;
                    const int rank = __popcll(K & ((1ull << b) - 1ull));
                    if (set && rank % RV_WPG == wg) rows[rank / RV_WPG] = static_cast<unsigned char>(b);
                }
                const int nk = nlo + __popc(static_cast<unsigned>(K >> 32));
                nmine = nk > wg ? (nk - wg + RV_WPG - 1) / RV_WPG : 0;
                __syncwarp();
            }
            const int c0 = (r + 1) >> 2;
            // Chunks any of the warp's rows has a bit in (all of them when the
            // bitmaps are absent); lane l takes chunks 64q+l and 64q+l+32.
            const int NQ = rowbits ? NB : (T256 + 63) / 64;
            for (int q = 0; nmine && q < NQ; ++q) {
              uint64_t un = ~0ull;
              if (rowbits) {
                  un = 0;
                  for (int j = 0; j < nmine; ++j) un |= gfl[rows[j] * NB + q];
              }
              for (int hh = 0; hh < 2; ++hh) {
                const int cq = 64 * q + static_cast<int>(l) + 32 * hh;
                if (!((un >> (cq & 63)) & 1ull) || cq < c0 || cq >= T256) continue;
                uint64_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
                for (int j0 = 0; j0 < nmine; j0 += RV_BATCH) {
                    // Up to RV_BATCH rows per round, all loads in flight together.
                    int rb[RV_BATCH];
#pragma unroll
                    for (int u = 0; u < RV_BATCH; ++u) {
                        const int b = j0 + u < nmine ? rows[j0 + u] : -1;
                        rb[u] = (b >= 0 && (!rowbits || ((gfl[b * NB + (cq >> 6)] >> (cq & 63)) & 1ull)))
                                    ? b : -1;
                    }
                    ulonglong2 x[RV_BATCH], y[RV_BATCH];
#pragma unroll
                    for (int u = 0; u < RV_BATCH; ++u) {
                        x[u] = make_ulonglong2(0, 0);
                        y[u] = make_ulonglong2(0, 0);
                        if (rb[u] >= 0) {
                            const ulonglong2* src = reinterpret_cast<const ulonglong2*>(
                                mask + (static_cast<int64_t>(r) * 64 + rb[u]) * ldw + 4 * cq);
                            x[u] = src[0];
                            y[u] = src[1];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < RV_BATCH; ++u) {
                        a0 |= x[u].x; a1 |= x[u].y; a2 |= y[u].x; a3 |= y[u].y;
                    }
                }
                unsigned long long* dst = reinterpret_cast<unsigned long long*>(removed + 4 * cq);
                if (a0) atomicOr(dst + 0, a0);
                if (a1) atomicOr(dst + 1, a1);
                if (a2) atomicOr(dst + 2, a2);
                if (a3) atomicOr(dst + 3, a3);
              }
            }
            group_bar(g);
            if (gt == 0) {
                __threadfence_block();
                mbar_arrive(&S.done[r % RV_KR]);
            }
        }
    }
    __syncthreads();
    // Output: exclusive prefix of the kept counts over the decided tiles, then
    // each warp writes whole tiles, mapping sorted positions through perm.
    const int nt = S.ntiles;
    if (warp == 0) {
        int carry = 0;
        for (int t0 = 0; t0 < nt; t0 += 32) {
            const int t = t0 + static_cast<int>(l);
            const int c = t < nt ? __popcll(kept[t]) : 0;
            int x = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(FULL, x, d);
                if (static_cast<int>(l) >= d) x += y;
            }
            if (t < nt) opre[t] = carry + x - c;
            carry += __shfl_sync(FULL, x, 31);
        }
        if (l == 0) {
            counts[0] = carry;
            if (done_out && max_out > 0 && carry >= max_out) *done_out = 1;
        }
    }
    __syncthreads();
    for (int t = warp; t < nt; t += RV_WARPS) {
        const uint64_t K = kept[t];
        const int p0 = opre[t];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int b = static_cast<int>(l) + 32 * hh;
            if ((K >> b) & 1ull) {
                const int pos = t * 64 + b;
                keep[p0 + __popcll(K & ((1ull << b) - 1ull))] = perm ? perm[pos] : pos;
            }
        }
    }
}


// ------------------------------------------------------- graph path, all SMs
// The rounds of graph_resolve over a pair list too long for one CTA's shared
// memory, by one CTA per SM (a cooperative launch: all CTAs are resident, so
// a barrier over the grid is safe).  The (kept, removed) and (hit, blocked)
// bitmaps live in global memory; CTA b owns a range of their words and a
// contiguous slice of the list, which its threads compact in place.  A round:
// the owners update their words; grid barrier; every CTA copies the (kept,
// removed) bitmap into shared memory, passes over its live pairs marking hit
// and blocked targets in shared memory, and ORs its non-zero mark words into
// the global bitmaps; grid barrier.  Cross-CTA data is read through L2
// (__ldcg), and the barrier orders it with fences.  Returns without output
// (the walk then runs) when the rounds outnumber the walk's tiles plus 16.
struct GridCtl {
    unsigned count, gen;  // barrier arrivals, generation
    int more[2];          // "some box still open", by round parity
    int resolved[4];      // per stage: this path decided it (the walk then returns)
    int cnt[1024];        // kept boxes per CTA
};
static_assert(offsetof(GridCtl, resolved) == 16, "stage flags at ints 4..7 of the control block");

__device__ __forceinline__ bool grid_barrier(GridCtl* ctl, unsigned nblocks, int* ok_s)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned* vgen = &ctl->gen;
        const unsigned g = *vgen;
        __threadfence();
        bool ok = true;
        if (atomicAdd(&ctl->count, 1u) == nblocks - 1) {
            atomicExch(&ctl->count, 0u);
            __threadfence();
            atomicAdd(&ctl->gen, 1u);
        } else {
            long long tries = 0;
            while (*vgen == g) {
                if (++tries > RV_WAIT_LIMIT) { ok = false; break; }
                __nanosleep(32);
            }
        }
        __threadfence();
        *ok_s = ok;
    }
    __syncthreads();
    return *ok_s != 0;
}

__global__ void __launch_bounds__(GG_THREADS, 1)
graph_grid_kernel(uint32_t* __restrict__ edges, const unsigned* __restrict__ ecount, unsigned ecap_smem,
                  unsigned ecap_list, const uint32_t* __restrict__ haspred, const int* __restrict__ m_dev,
                  int m_bound, int limit, const int* __restrict__ perm, int max_out,
                  int64_t* __restrict__ keep, int64_t* __restrict__ counts, int32_t* status,
                  const int* __restrict__ done_in, int* done_out, int* grid_done, uint2* KRg, uint2* HBg,
                  GridCtl* ctl)
{
    extern __shared__ __align__(16) uint2 gsm[];  // (kept, removed) copy, then local (hit, blocked)
    __shared__ int ok_s;
    __shared__ int scratch[32];
    if (done_in && *done_in) return;
    const unsigned E = *ecount;
    if (E <= ecap_smem || E > ecap_list) return;  // one CTA's path, or the walk
    const int n_all = m_dev ? *m_dev : m_bound;
    const int n = min(n_all, limit);
    const int NW = (n + 31) / 32;
    uint2* KRs = gsm;
    uint2* HBs = gsm + NW;
    const unsigned nb = gridDim.x, b = blockIdx.x;
    const int tid = threadIdx.x;
    const unsigned l = lane_id();
    const int warp = tid >> 5;
    const int wpb = (NW + static_cast<int>(nb) - 1) / static_cast<int>(nb);
    const int w0 = min(static_cast<int>(b) * wpb, NW), w1 = min(w0 + wpb, NW);
    const unsigned epb = (E + nb - 1) / nb;
    const unsigned e0 = min(b * epb, E), e1 = min(e0 + epb, E);
    int live = e1 > e0 + tid ? static_cast<int>((e1 - e0 - tid + GG_THREADS - 1) / GG_THREADS) : 0;

    for (int w = w0 + tid; w < w1; w += GG_THREADS) {
        KRg[w] = make_uint2(0u, 0u);
        HBg[w] = make_uint2(0u, haspred[w]);  // before the first round every target is blocked
    }
    if (!grid_barrier(ctl, nb, &ok_s)) goto fail;
    {
        const int max_rounds = (n + 63) / 64 + 16;
        for (int round = 0;; ++round) {
            bool more = false;
            for (int w = w0 + tid; w < w1; w += GG_THREADS) {
                const uint2 kr = __ldcg(KRg + w);
                const uint32_t valid = (w == NW - 1 && (n & 31)) ? (1u << (n & 31)) - 1u : ~0u;
                const uint32_t open = ~(kr.x | kr.y) & valid;
                if (open) {
                    const uint2 hb = __ldcg(HBg + w);
                    KRg[w] = make_uint2(kr.x | (open & ~hb.x & ~hb.y), kr.y | (open & hb.x));
                    HBg[w] = make_uint2(0u, 0u);
                    more |= (open & ~hb.x & hb.y) != 0;
                }
            }
            if (__syncthreads_or(more) && tid == 0) atomicOr(&ctl->more[round & 1], 1);
            if (!grid_barrier(ctl, nb, &ok_s)) goto fail;
            if (!__ldcg(&ctl->more[round & 1])) break;
            if (round == max_rounds) return;  // no output: the walk decides
            if (b == 0 && tid == 0) ctl->more[(round + 1) & 1] = 0;
            for (int w = tid; w < NW; w += GG_THREADS) {
                KRs[w] = __ldcg(KRg + w);
                HBs[w] = make_uint2(0u, 0u);
            }
            __syncthreads();
            int nl = 0;
            for (int k0 = 0; k0 < live; k0 += 4) {
                uint32_t e[4];
                uint2 ki[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    e[u] = k0 + u < live ? edges[e0 + tid + GG_THREADS * (k0 + u)] : 0xffffffffu;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (e[u] != 0xffffffffu) ki[u] = KRs[e[u] >> 21];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (e[u] == 0xffffffffu) continue;
                    const uint32_t j = e[u] & 0xffffu;
                    const uint32_t bi = 1u << ((e[u] >> 16) & 31);
                    if (ki[u].x & bi) {
                        atomicOr(&HBs[j >> 5].x, 1u << (j & 31));
                    } else if (!(ki[u].y & bi)) {
                        atomicOr(&HBs[j >> 5].y, 1u << (j & 31));
                        edges[e0 + tid + GG_THREADS * nl++] = e[u];
                    }
                }
            }
            live = nl;
            __syncthreads();
            for (int w = tid; w < NW; w += GG_THREADS) {
                const uint2 hb = HBs[w];
                if (hb.x) atomicOr(&HBg[w].x, hb.x);
                if (hb.y) atomicOr(&HBg[w].y, hb.y);
            }
            if (!grid_barrier(ctl, nb, &ok_s)) goto fail;
        }
        // Output of the owned words in score order: kept counts per CTA, a
        // prefix over the CTAs, then lane l of a warp writes box 32w+l.
        const int nown = w1 - w0;
        const int wpw = (nown + 31) / 32;
        const int a0 = min(w0 + warp * wpw, w1), a1 = min(a0 + wpw, w1);
        int c = 0;
        for (int w = a0 + static_cast<int>(l); w < a1; w += 32) c += __popc(__ldcg(&KRg[w].x));
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(FULL, c, d);
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
            if (l == 31) ctl->cnt[b] = v;
        }
        if (!grid_barrier(ctl, nb, &ok_s)) goto fail;
        int total = 0, cbase = 0;
        for (unsigned q = 0; q < nb; ++q) {
            const int v = __ldcg(&ctl->cnt[q]);
            if (q < b) cbase += v;
            total += v;
        }
        const int cap = max_out > 0 ? max_out : INT_MAX;
        int base = cbase + (warp ? scratch[warp - 1] : 0);
        const uint32_t below = (1u << l) - 1u;
        for (int w = a0; w < a1 && base < cap; ++w) {
            const uint32_t bits = __ldcg(&KRg[w].x);
            if ((bits >> l) & 1u) {
                const int pos = base + __popc(bits & below);
                const int j = 32 * w + static_cast<int>(l);
                if (pos < cap) keep[pos] = perm ? perm[j] : j;
            }
            base += __popc(bits);
        }
        if (b == 0 && tid == 0) {
            counts[0] = total < cap ? total : cap;
            if (done_out) *done_out = (n >= n_all) || (max_out > 0 && total >= max_out);
            *grid_done = 1;
        }
        return;
    }
fail:
    if (tid == 0 && status) set_status(status, NMS_ERR_TIMEOUT);
}

size_t graph_grid_smem(int m_bound) { return 2 * sizeof(uint2) * static_cast<size_t>(graph_words(m_bound)); }
size_t graph_grid_ctl_bytes() { return sizeof(GridCtl); }
int graph_grid_min_n() { return GR_GRID_MIN_N; }

void launch_graph_grid(uint32_t* edges, const unsigned* ecount, const uint64_t* haspred, const int* m_dev,
                       int m_bound, const int* perm, int max_out, int64_t* keep, int64_t* counts,
                       int32_t* status, cudaStream_t st, int limit, const int* done_in, int* done_out,
                       int* grid_done, uint64_t* state, void* ctl)
{
    const unsigned ecap_list = graph_grid_cap(m_bound);
    if (!ecap_list) return;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) return;
    const size_t smem = graph_grid_smem(m_bound);
    ensure_dynamic_smem(reinterpret_cast<const void*>(graph_grid_kernel), smem);
    uint2* KRg = reinterpret_cast<uint2*>(state);
    uint2* HBg = KRg + graph_words(m_bound);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms < 1024 ? sms : 1024));
    cfg.blockDim = dim3(GG_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, graph_grid_kernel, edges, ecount, graph_edge_cap(m_bound), ecap_list,
                       reinterpret_cast<const uint32_t*>(haspred), m_dev, m_bound, limit, perm, max_out, keep,
                       counts, status, done_in, done_out, grid_done, KRg, HBg, static_cast<GridCtl*>(ctl));
}

// Passes 0 and 1 of graph_resolve over all SMs, for a list longer than one
// CTA's shared memory.  Neither needs a barrier inside: pass 0 keeps exactly
// the sources without a source of their own (the clear bits of haspred) and
// removes their targets; pass 1 keeps nothing (every box's byte is then 0 or
// 2, never 1), drops the pairs whose source pass 0 removed and blocks the
// targets of the rest.  Both are plain byte stores of one value.
constexpr int GP_THREADS = 512;

__device__ __forceinline__ bool has_source(const uint32_t* __restrict__ haspred, uint32_t i)
{
    return (haspred[i >> 5] >> (i & 31u)) & 1u;
}

__global__ void __launch_bounds__(GP_THREADS)
graph_pass0_kernel(const uint32_t* __restrict__ edges, const unsigned* __restrict__ ecount, unsigned ecap,
                   unsigned lcap, const uint32_t* __restrict__ haspred, uint8_t* __restrict__ removed)
{
    pdl_wait();  // the mask has finished
    pdl_release();
    const unsigned E = *ecount;
    if (E <= ecap || E > lcap) return;  // one CTA holds it, or the list is incomplete
    const unsigned nq = (E + 3) / 4;
    const uint4* Q = reinterpret_cast<const uint4*>(edges);
    for (unsigned q = blockIdx.x * GP_THREADS + threadIdx.x; q < nq; q += gridDim.x * GP_THREADS) {
        const uint4 v = Q[q];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t e = quad_at(v, u);
            if (4 * q + u < E && !has_source(haspred, e >> 16)) removed[e & 0xffffu] = 1;
        }
    }
}

// One tile of GP_THREADS quads a step: the kept pairs are counted by a block
// prefix, one reservation in out per tile, and stored (none past ocap; the
// count still grows, so the resolve sees the overflow).
__global__ void __launch_bounds__(GP_THREADS)
graph_pass1_kernel(const uint32_t* __restrict__ edges, const unsigned* __restrict__ ecount, unsigned ecap,
                   unsigned lcap, const uint32_t* __restrict__ haspred, const uint8_t* __restrict__ removed,
                   uint32_t* __restrict__ out, unsigned* __restrict__ ocount, unsigned ocap,
                   uint8_t* __restrict__ blocked)
{
    constexpr int NWARP = GP_THREADS / 32;
    __shared__ int wsum[NWARP];
    __shared__ unsigned s_base;
    pdl_wait();  // pass 0 has finished
    pdl_release();
    const unsigned E = *ecount;
    if (E <= ecap || E > lcap) return;
    const unsigned nq = (E + 3) / 4;
    const unsigned tiles = (nq + GP_THREADS - 1) / GP_THREADS;
    const uint4* Q = reinterpret_cast<const uint4*>(edges);
    const unsigned l = lane_id();
    const int warp = static_cast<int>(threadIdx.x) >> 5;
    for (unsigned t = blockIdx.x; t < tiles; t += gridDim.x) {
        const unsigned q = t * GP_THREADS + threadIdx.x;
        const uint4 v = q < nq ? Q[q] : make_uint4(0u, 0u, 0u, 0u);
        uint32_t stay = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t e = quad_at(v, u), i = e >> 16;
            if (q < nq && 4 * q + u < E && has_source(haspred, i) && !removed[i]) stay |= 1u << u;
        }
        const int c = __popc(stay);
        int x = c;  // inclusive prefix over the warp
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(FULL, x, d);
            if (static_cast<int>(l) >= d) x += y;
        }
        if (l == 31) wsum[warp] = x;
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            const int s = wsum[w];
            before += w < warp ? s : 0;
            total += s;
        }
        if (threadIdx.x == 0) s_base = total ? atomicAdd(ocount, static_cast<unsigned>(total)) : 0u;
        __syncthreads();
        const unsigned base = s_base;
        const bool room = base <= ocap && static_cast<unsigned>(total) <= ocap - base;
        unsigned o = base + static_cast<unsigned>(before + x - c);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!((stay >> u) & 1u)) continue;
            const uint32_t e = quad_at(v, u);
            blocked[e & 0xffffu] = 3;
            if (room) out[o] = e;
            ++o;
        }
        __syncthreads();  // wsum and s_base are written again
    }
}

void launch_graph_prepass(const uint32_t* edges, const unsigned* ecount, unsigned lcap, const uint64_t* haspred,
                          int n, const GraphPre& pre, cudaStream_t st)
{
    if (n <= 0 || !edges || !ecount || !haspred || !pre.edges || !pre.ecount || !pre.removed || !pre.blocked)
        return;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) return;
    const unsigned ecap = graph_edge_cap(n);
    const uint32_t* hp = reinterpret_cast<const uint32_t*>(haspred);
    launch_pdl(graph_pass0_kernel, dim3(2 * sms), dim3(GP_THREADS), 0, st, edges, ecount, ecap, lcap, hp,
               pre.removed);
    launch_pdl(graph_pass1_kernel, dim3(2 * sms), dim3(GP_THREADS), 0, st, edges, ecount, ecap, lcap, hp,
               static_cast<const uint8_t*>(pre.removed), pre.edges, pre.ecount, pre.cap, pre.blocked);
}

size_t resolve_smem_bytes(int m_bound, int NB) { return resolve_layout(m_bound, NB).total; }

// GR_CLUSTER when a cluster of that many resolve CTAs with `smem` bytes each
// can be resident on the current device at all, else 1 (the kernel then runs
// passes 0 and 1 in one CTA).  Asked once per device and size.
unsigned resolve_cluster_size(size_t smem)
{
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, unsigned> known;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1u;
    std::lock_guard<std::mutex> lock(mu);
    const auto it = known.find({dev, smem});
    if (it != known.end()) return it->second;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(GR_CLUSTER);
    cfg.blockDim = dim3(RV_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = GR_CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    const bool fits =
        cudaOccupancyMaxActiveClusters(&clusters, resolve_single_kernel<false>, &cfg) == cudaSuccess && clusters >= 1;
    cudaGetLastError();  // a refused query leaves no error behind
    const unsigned c = fits ? static_cast<unsigned>(GR_CLUSTER) : 1u;
    known[{dev, smem}] = c;
    return c;
}

void launch_resolve_single(const uint64_t* mask, int64_t ldw, const uint64_t* rowbits, int NB,
                           uint32_t* edges, const unsigned* ecount, unsigned lcap,
                           const uint64_t* haspred, const int* m_dev, int m_bound, const int* perm,
                           int max_out, int64_t* keep, int64_t* counts, int32_t* status,
                           cudaStream_t st, int limit, const int* done_in, int* done_out,
                           const int* grid_done, const GraphPre* pre)
{
    size_t smem = resolve_smem_bytes(m_bound, NB);
    const unsigned ecap = edges ? graph_edge_cap(m_bound) : 0u;
    if (edges && graph_smem_bytes(m_bound) > smem) smem = graph_smem_bytes(m_bound);
    if (!edges) pre = nullptr;
    ensure_dynamic_smem(pre ? reinterpret_cast<const void*>(resolve_single_kernel<true>)
                            : reinterpret_cast<const void*>(resolve_single_kernel<false>),
                        smem);
    cudaLaunchConfig_t cfg{};
    // The box path with a pair list: a cluster of GR_CLUSTER CTAs (passes 0
    // and 1 shared; CTA 0 does the rest) where the device can hold one.
    const unsigned csize = edges && !pre ? resolve_cluster_size(smem) : 1u;
    cfg.gridDim = dim3(csize);
    cfg.blockDim = dim3(RV_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 1u + static_cast<unsigned>(pdl_attr_count());
    const uint32_t* hp = reinterpret_cast<const uint32_t*>(haspred);
    const unsigned lc = edges ? lcap : 0u;
    if (pre)
        cudaLaunchKernelEx(&cfg, resolve_single_kernel<true>, mask, ldw, rowbits, NB, edges, ecount, ecap, lc, hp,
                           m_dev, m_bound, perm, max_out, keep, counts, status, limit, done_in, done_out, grid_done,
                           *pre);
    else
        cudaLaunchKernelEx(&cfg, resolve_single_kernel<false>, mask, ldw, rowbits, NB, edges, ecount, ecap, lc,
                           hp, m_dev, m_bound, perm, max_out, keep, counts, status, limit, done_in, done_out,
                           grid_done, GraphPre{});
}

}  // namespace gbnms
