// bfs_device.cuh -- device code of the level-synchronous frontier BFS.
//
// One persistent cooperative kernel runs the level loop ("a device-resident
// level loop" replacing the per-level launch plus device->host count copy
// that "100 Days of GPU, Day 38" measures in its host loop, and the remedy
// the PMPP ch. 15 notes name in section 15.7: grid-wide synchronisation
// inside one kernel). Every level:
//
//   S2 direction: push (top-down, sparse queue) or pull (bottom-up, bitmap),
//      chosen from exact device counters with the rule of PMPP ch. 15 notes,
//      section 15.7 (pull when the frontier's edges outnumber the unvisited
//      vertices), evaluated again at every level.
//   S3/S4 push advance, load-balanced either by degree bins (thread / warp /
//      CTA per vertex, PMPP ch. 15 notes section 15.7; the three size classes
//      of the Gunrock paper's section 4.4 as quoted on the Gunrock reading
//      page, step 4) or edge-balanced (merge-path: an exclusive prefix of the
//      frontier's degrees plus a search per CTA and per edge; Gunrock reading
//      page steps 4-5, and "The Frontier Model for Parallel BFS" section 22.3).
//   S5 discovery: atomicOr on a visited bitmap, or atomicCAS on dist
//      (Day 38 claimVertex; ch. 22 sections 22.1-22.2); exactly one winner
//      per vertex writes dist and parent.
//   S6 compaction: winners are staged in shared memory and flushed with one
//      global atomic per CTA batch (the privatised queue of PMPP ch. 15 notes,
//      section 15.6, without its silent drop on overflow: a full stage makes
//      the thread append directly).
//   S7 pull level over a frontier bitmap, one warp per 32-vertex word: no
//      atomics, dedupe by construction (Gunrock reading page, step 6).
//   S8 representation switches queue <-> bitmap when the direction changes.
//   S9 a bounded grid barrier ends each phase; the loop stops on an empty
//      frontier (Gunrock's convergence test, read on the device).
//
// The exclusive prefix the merge-path search needs is produced for free by
// the compaction: a CTA reserves its queue slots and its edge range with one
// 64-bit atomicAdd on a packed (count, edges) counter, so queue order and
// edge order agree and qoff[] is a valid exclusive scan of the degrees.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "bfs_csr.h"

namespace fbc {

constexpr int kItems = 4;        // edges per thread per merge-path round
constexpr int kSlots = 4;        // rotating per-level counter slots
constexpr int kMaxBlock = 1024;
constexpr unsigned kFull = 0xffffffffu;

// Counters describing one frontier F_k. Level k - 1 accumulates them (all
// CTAs, atomically); level k reads them after the barrier. CTA 0 writes
// `unvisited` and `dir` of slot k at the start of level k; they are read at
// level k + 1. Slot (k + 2) % 4 is cleared by CTA 0 during level k.
struct __align__(16) LevelSlot {
    unsigned long long qpack;   // (queue count << eb) | queue edge total
    unsigned long long found;   // |F_k|, every discovered vertex
    unsigned long long fedges;  // sum of out-degrees over F_k
    unsigned long long maxdeg;  // largest out-degree in F_k
    long long unvisited;        // U_k: non-isolated vertices unreached at level k
    int dir;                    // direction used at level k
    int adv;                    // advance used at level k (push levels)
};

struct __align__(128) Ctl {
    unsigned long long bar;     // barrier arrivals in the current launch
    unsigned long long pad0[15];
    unsigned int exit_count;    // CTAs that left the current launch
    int status;                 // BFS_CSR_OK or a device error code
    int done;                   // the search has ended
    int level;                  // next level to run (persists across launches)
    int num_levels;             // non-empty frontiers, valid once done
    int pad1[27];
    LevelSlot slot[kSlots];
    unsigned long long t_end_ns;
    long long nonisolated;      // vertices of nonzero degree (set at create)
    int validate_flags;         // bit 0 row_ptr bad, bit 1 col out of range
    int pad2[27];
};

template <typename RowT>
struct Params {
    const RowT* __restrict__ row_ptr;
    const int32_t* __restrict__ col;
    int32_t n;
    int32_t words;              // ceil(n / 32)
    int32_t* dist;
    int32_t* parent;            // may be null
    uint32_t* visited;
    uint32_t* fb[2];            // frontier bitmaps, F_k in fb[k & 1]
    int32_t* qv[2];             // frontier queues, F_k in qv[k & 1]
    RowT* qbeg[2];              // row start of each queued vertex
    RowT* qoff[2];              // exclusive prefix of queued degrees
    Ctl* ctl;
    bfs_csr_level_stat* stats;
    int32_t stats_cap;
    int32_t* num_levels_out;    // may be null
    int eb;                     // edge bits of LevelSlot::qpack
    int direction, advance, discovery;
    int small_max, cta_min, mp_min_frontier, binned_max_deg;
    double pull_ratio;
    int max_depth;
    int symmetric;
    int level_budget;           // levels this launch may run
    long long timeout_ns;
    int unreachable_barrier;
};

// ------------------------------------------------------------ primitives

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Loads of data other CTAs write during the kernel go to L2 (.cg) so that a
// stale L1 line can never be read.
template <typename T>
__device__ __forceinline__ T ldcg(const T* p) { return __ldcg(p); }

__device__ __forceinline__ unsigned long long ldcg_u64(const unsigned long long* p)
{
    return __ldcg(p);
}

// Grid-wide barrier with a bounded wait. All CTAs of the cooperative launch
// call it the same number of times. Thread 0 publishes the CTA's writes
// (fence), arrives, and polls the arrival counter with acquire loads until
// every CTA has arrived or the time limit passes; on expiry it records
// BFS_CSR_ETIMEOUT. Returns false when the run must stop.
template <typename RowT>
__device__ __forceinline__ bool grid_barrier(const Params<RowT>& p, unsigned long long& target)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        target += gridDim.x;
        const unsigned long long want = target + (unsigned long long)p.unreachable_barrier;
        __threadfence();
        atomicAdd(&p.ctl->bar, 1ull);
        const unsigned long long t0 = global_timer_ns();
        unsigned int spins = 0;
        int ok = 1;
        while (ld_acquire_u64(&p.ctl->bar) < want) {
            if ((++spins & 255u) == 0u) {
                if (global_timer_ns() - t0 > (unsigned long long)p.timeout_ns || spins > (1u << 30)) {
                    atomicCAS(&p.ctl->status, BFS_CSR_OK, BFS_CSR_ETIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        if (ok && ldcg(&p.ctl->status) != BFS_CSR_OK)
            ok = 0;
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Inclusive warp scan.
template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T x)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const T y = __shfl_up_sync(kFull, x, d);
        if (lane >= d)
            x += y;
    }
    return x;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T x)
{
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        x += __shfl_xor_sync(kFull, x, d);
    return x;
}

template <typename T>
__device__ __forceinline__ T warp_max(T x)
{
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const T y = __shfl_xor_sync(kFull, x, d);
        x = y > x ? y : x;
    }
    return x;
}

// Block-wide exclusive scan of one value per thread; *total gets the sum.
// Uses s_tmp[32]. Every thread of the block must call it.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T x, T* total, T* s_tmp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const T inc = warp_inclusive_scan(x);
    if (lane == 31)
        s_tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        T w = lane < nwarps ? s_tmp[lane] : T(0);
        const T winc = warp_inclusive_scan(w);
        s_tmp[lane] = winc - w;  // exclusive prefix of warp totals
        if (lane == 31)
            s_tmp[32] = winc;
    }
    __syncthreads();
    const T out = s_tmp[warp] + inc - x;
    *total = s_tmp[32];
    __syncthreads();
    return out;
}

// ------------------------------------------------------------ shared state

template <typename RowT>
struct Smem {
    // compaction stage (S6)
    int32_t* sv;      // vertex
    RowT* sb;         // row start
    RowT* sd;         // degree
    int cap;
    // merge-path window (S4)
    RowT* woff;
    RowT* wbeg;
    int32_t* wu;
    int wcap;
    // CTA-per-vertex list of the binned advance
    int32_t* lu;
    RowT* lb;
    RowT* ld;
};

struct __align__(16) SmemScalars {
    int stage_n;
    int nlarge;
    int cur;
    int i0;
    unsigned long long base;
    unsigned long long ebase;
    long long tmp_ll[33];
};

// Per-thread tallies of the vertices this thread discovered in a level.
struct Tally {
    unsigned long long found;
    unsigned long long edges;
    unsigned long long maxdeg;
};

// ------------------------------------------------------------ S6 compaction

// Append one discovered vertex (degree > 0) to the next queue directly with a
// single packed atomic. Used only when the shared-memory stage is full.
template <typename RowT>
__device__ __noinline__ void append_direct(const Params<RowT>& p, LevelSlot* nxt, int qsel,
                                           int32_t v, RowT b, RowT deg)
{
    const unsigned long long old = atomicAdd(&nxt->qpack, (1ull << p.eb) | (unsigned long long)deg);
    const unsigned long long slot = old >> p.eb;
    const unsigned long long eoff = old & ((1ull << p.eb) - 1ull);
    p.qv[qsel][slot] = v;
    p.qbeg[qsel][slot] = b;
    p.qoff[qsel][slot] = (RowT)eoff;
}

template <typename RowT>
__device__ __forceinline__ void stage_push(const Params<RowT>& p, const Smem<RowT>& sm,
                                           SmemScalars& ss, LevelSlot* nxt, int qsel,
                                           int32_t v, RowT b, RowT deg)
{
    const int pos = atomicAdd(&ss.stage_n, 1);
    if (pos < sm.cap) {
        sm.sv[pos] = v;
        sm.sb[pos] = b;
        sm.sd[pos] = deg;
    } else {
        append_direct(p, nxt, qsel, v, b, deg);
    }
}

// Block-wide: move the staged vertices to the next queue with one packed
// atomic per CTA. Every thread calls it; the stage is empty afterwards.
template <typename RowT>
__device__ void stage_flush(const Params<RowT>& p, const Smem<RowT>& sm, SmemScalars& ss,
                            LevelSlot* nxt, int qsel)
{
    __syncthreads();
    const int cnt = min(ss.stage_n, sm.cap);
    if (cnt > 0) {
        const int bd = blockDim.x;
        const int per = (cnt + bd - 1) / bd;
        const int lo = min(threadIdx.x * per, cnt), hi = min(lo + per, cnt);
        long long sum = 0;
        for (int i = lo; i < hi; ++i)
            sum += (long long)sm.sd[i];
        long long total;
        const long long excl = block_exclusive_scan(sum, &total, ss.tmp_ll);
        if (threadIdx.x == 0) {
            const unsigned long long add = ((unsigned long long)cnt << p.eb) | (unsigned long long)total;
            const unsigned long long old = atomicAdd(&nxt->qpack, add);
            ss.base = old >> p.eb;
            ss.ebase = old & ((1ull << p.eb) - 1ull);
        }
        __syncthreads();
        const unsigned long long base = ss.base;
        RowT run = (RowT)(ss.ebase + (unsigned long long)excl);
        int32_t* qv = p.qv[qsel];
        RowT* qb = p.qbeg[qsel];
        RowT* qo = p.qoff[qsel];
        for (int i = lo; i < hi; ++i) {
            qv[base + i] = sm.sv[i];
            qb[base + i] = sm.sb[i];
            qo[base + i] = run;
            run += sm.sd[i];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        ss.stage_n = 0;
    __syncthreads();
}

// End of a level: one atomic per CTA for each frontier statistic.
template <typename RowT>
__device__ void publish_tally(const Tally& t, LevelSlot* nxt, SmemScalars& ss)
{
    long long tot_found, tot_edges;
    block_exclusive_scan((long long)t.found, &tot_found, ss.tmp_ll);
    block_exclusive_scan((long long)t.edges, &tot_edges, ss.tmp_ll);
    unsigned long long m = warp_max(t.maxdeg);
    __shared__ unsigned long long s_max[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        s_max[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long mm = 0;
        for (int w = 0; w < (int)((blockDim.x + 31) >> 5); ++w)
            mm = s_max[w] > mm ? s_max[w] : mm;
        if (tot_found > 0) {
            atomicAdd(&nxt->found, (unsigned long long)tot_found);
            atomicAdd(&nxt->fedges, (unsigned long long)tot_edges);
            atomicMax(&nxt->maxdeg, mm);
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------ S5 discovery

// The claim of vertex v by frontier vertex u at level k. Exactly one caller
// per v gets true; the winner writes dist[v] and parent[v].
template <typename RowT>
__device__ __forceinline__ bool claim(const Params<RowT>& p, int k, int32_t v, int32_t u)
{
    if (p.discovery == BFS_CSR_DISC_CAS) {
        if (ldcg(&p.dist[v]) != -1)
            return false;
        if (atomicCAS(&p.dist[v], -1, k + 1) != -1)
            return false;
        atomicOr(&p.visited[v >> 5], 1u << (v & 31));  // keeps pull levels exact
    } else {
        const uint32_t bit = 1u << (v & 31);
        uint32_t* w = p.visited + (v >> 5);
        if (ldcg(w) & bit)
            return false;
        if (atomicOr(w, bit) & bit)
            return false;
        p.dist[v] = k + 1;
    }
    if (p.parent != nullptr)
        p.parent[v] = u;
    return true;
}

// After a win: read v's row, count it, and queue it when it has edges.
template <typename RowT>
__device__ __forceinline__ void after_win(const Params<RowT>& p, const Smem<RowT>& sm,
                                          SmemScalars& ss, LevelSlot* nxt, int qsel, Tally& t,
                                          int32_t v)
{
    const RowT b = p.row_ptr[v];
    const RowT deg = p.row_ptr[v + 1] - b;
    t.found += 1;
    t.edges += (unsigned long long)deg;
    t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg : t.maxdeg;
    if (deg > 0)
        stage_push(p, sm, ss, nxt, qsel, v, b, deg);
}

// ------------------------------------------------------------ S4 push levels

// Degree-binned advance: thread per vertex below small_max, warp per vertex
// below cta_min, whole CTA per vertex above. Frontier entry i belongs to
// CTA i % G so that small frontiers spread over every SM.
template <typename RowT>
__device__ void push_binned(const Params<RowT>& p, int k, int qn, RowT qm, const Smem<RowT>& sm,
                            SmemScalars& ss, LevelSlot* nxt, Tally& t)
{
    const int cs = k & 1, ns = cs ^ 1;
    const int32_t* qv = p.qv[cs];
    const RowT* qb = p.qbeg[cs];
    const RowT* qo = p.qoff[cs];
    const int G = gridDim.x, bd = blockDim.x, lane = threadIdx.x & 31;
    const int mine = qn > (int)blockIdx.x ? (qn - (int)blockIdx.x + G - 1) / G : 0;
    for (int base = 0; base < mine; base += bd) {
        const int li = base + threadIdx.x;
        const bool valid = li < mine;
        const int i = (int)blockIdx.x + li * G;
        int32_t u = 0;
        RowT b = 0, deg = 0;
        if (valid) {
            u = ldcg(qv + i);
            b = ldcg(qb + i);
            const RowT o = ldcg(qo + i);
            deg = (i + 1 < qn ? ldcg(qo + i + 1) : qm) - o;
        }
        // thread per vertex
        if (valid && deg < (RowT)p.small_max) {
            RowT j = 0;
            for (; j + 4 <= deg; j += 4) {
                const int32_t v0 = p.col[b + j], v1 = p.col[b + j + 1];
                const int32_t v2 = p.col[b + j + 2], v3 = p.col[b + j + 3];
                if (claim(p, k, v0, u)) after_win(p, sm, ss, nxt, ns, t, v0);
                if (claim(p, k, v1, u)) after_win(p, sm, ss, nxt, ns, t, v1);
                if (claim(p, k, v2, u)) after_win(p, sm, ss, nxt, ns, t, v2);
                if (claim(p, k, v3, u)) after_win(p, sm, ss, nxt, ns, t, v3);
            }
            for (; j < deg; ++j) {
                const int32_t v = p.col[b + j];
                if (claim(p, k, v, u)) after_win(p, sm, ss, nxt, ns, t, v);
            }
        }
        // warp per vertex
        unsigned mm = __ballot_sync(kFull, valid && deg >= (RowT)p.small_max && deg < (RowT)p.cta_min);
        while (mm) {
            const int src = __ffs(mm) - 1;
            mm &= mm - 1;
            const int32_t wu = __shfl_sync(kFull, u, src);
            const RowT wb = __shfl_sync(kFull, b, src);
            const RowT wd = __shfl_sync(kFull, deg, src);
            for (RowT j = lane; j < wd; j += 32) {
                const int32_t v = p.col[wb + j];
                if (claim(p, k, v, wu)) after_win(p, sm, ss, nxt, ns, t, v);
            }
        }
        // CTA per vertex
        if (valid && deg >= (RowT)p.cta_min) {
            const int pos = atomicAdd(&ss.nlarge, 1);
            sm.lu[pos] = u;
            sm.lb[pos] = b;
            sm.ld[pos] = deg;
        }
        __syncthreads();
        const int nl = ss.nlarge;
        for (int L = 0; L < nl; ++L) {
            const int32_t cu = sm.lu[L];
            const RowT cb = sm.lb[L], cd = sm.ld[L];
            for (RowT j0 = 0; j0 < cd; j0 += bd) {
                const RowT j = j0 + threadIdx.x;
                if (j < cd) {
                    const int32_t v = p.col[cb + j];
                    if (claim(p, k, v, cu)) after_win(p, sm, ss, nxt, ns, t, v);
                }
                if (__syncthreads_or(ss.stage_n > sm.cap / 2))
                    stage_flush(p, sm, ss, nxt, ns);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0)
            ss.nlarge = 0;
        stage_flush(p, sm, ss, nxt, ns);
    }
}

// Merge-path advance: CTA c owns the edge range [c*M/G, (c+1)*M/G) of the
// frontier's concatenated adjacency lists. One 32-ary search over qoff finds
// the first vertex; each round then stages the offsets of at most TILE + 1
// vertices in shared memory (every queued vertex has at least one edge) and
// each thread binary-searches the window for the owner of its edges.
template <typename RowT>
__device__ void push_merge_path(const Params<RowT>& p, int k, int qn, RowT qm,
                                const Smem<RowT>& sm, SmemScalars& ss, LevelSlot* nxt, Tally& t)
{
    const int cs = k & 1, ns = cs ^ 1;
    const int32_t* qv = p.qv[cs];
    const RowT* qb = p.qbeg[cs];
    const RowT* qo = p.qoff[cs];
    const int bd = blockDim.x, lane = threadIdx.x & 31;
    const unsigned long long G = gridDim.x;
    const RowT e_lo = (RowT)((unsigned long long)qm * blockIdx.x / G);
    const RowT e_hi = (RowT)((unsigned long long)qm * (blockIdx.x + 1) / G);
    if (e_lo >= e_hi)
        return;
    const int tile = bd * kItems;

    if (threadIdx.x < 32) {
        // last i in [0, qn) with qoff[i] <= e_lo; qoff[0] = 0 <= e_lo
        int lo = 0, hi = qn;
        while (hi - lo > 1) {
            const int step = (hi - lo + 31) / 32;
            const int probe = lo + lane * step;
            const bool le = lane > 0 && probe < hi && ldcg(qo + probe) <= e_lo;
            const unsigned bal = __ballot_sync(kFull, le);
            if (bal == 0u) {
                hi = min(hi, lo + step);
            } else {
                const int top = 31 - __clz(bal);
                lo = lo + top * step;
                hi = min(hi, lo + step);
            }
        }
        if (lane == 0)
            ss.cur = lo;
    }
    __syncthreads();

    for (RowT r0 = e_lo; r0 < e_hi; r0 += tile) {
        const RowT r1 = r0 + (RowT)tile < e_hi ? r0 + (RowT)tile : e_hi;
        const int cur = ss.cur;
        const int win = min(tile + 1, qn - cur);
        for (int x = threadIdx.x; x < win; x += bd) {
            sm.woff[x] = ldcg(qo + cur + x);
            sm.wbeg[x] = ldcg(qb + cur + x);
            sm.wu[x] = ldcg(qv + cur + x);
        }
        __syncthreads();
        int32_t vv[kItems], uu[kItems];
        int lo = 0;
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const RowT e = r0 + (RowT)(it * bd + threadIdx.x);
            vv[it] = -1;
            uu[it] = 0;
            if (e < r1) {
                int hi = win;
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (sm.woff[mid] <= e)
                        lo = mid;
                    else
                        hi = mid;
                }
                uu[it] = sm.wu[lo];
                vv[it] = p.col[sm.wbeg[lo] + (e - sm.woff[lo])];
            }
        }
        bool won[kItems];
#pragma unroll
        for (int it = 0; it < kItems; ++it)
            won[it] = vv[it] >= 0 && claim(p, k, vv[it], uu[it]);
#pragma unroll
        for (int it = 0; it < kItems; ++it)
            if (won[it])
                after_win(p, sm, ss, nxt, ns, t, vv[it]);
        if (threadIdx.x == 0 && r1 < e_hi) {
            int a = 0, c = win;  // last window index with woff <= r1
            while (c - a > 1) {
                const int mid = (a + c) >> 1;
                if (sm.woff[mid] <= r1)
                    a = mid;
                else
                    c = mid;
            }
            ss.cur = cur + a;
        }
        stage_flush(p, sm, ss, nxt, ns);
    }
}

// ------------------------------------------------------------ S7 pull level

// One warp per 32-vertex word of the visited bitmap; lane i owns vertex
// 32w + i. An unvisited vertex scans its neighbours in CSR order and stops at
// the first one whose bit is set in the frontier bitmap fb[k & 1]. The warp
// is the only writer of its visited word and of the next-frontier word, so no
// atomics are needed; every next-frontier word is written, so the bitmap
// needs no clearing.
template <typename RowT>
__device__ void pull_level(const Params<RowT>& p, int k, Tally& t)
{
    const uint32_t* fcur = p.fb[k & 1];
    uint32_t* fnext = p.fb[(k + 1) & 1];
    const int lane = threadIdx.x & 31;
    const int gwarp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    for (int w = gwarp; w < p.words; w += nwarps) {
        const uint32_t vis = ldcg(p.visited + w);
        uint32_t found = 0;
        if (vis != kFull) {
            const int32_t v = (w << 5) + lane;
            int32_t par = -1;
            RowT deg = 0;
            if (!((vis >> lane) & 1u)) {
                const RowT b = p.row_ptr[v];
                const RowT e = p.row_ptr[v + 1];
                deg = e - b;
                RowT j = b;
                for (; j + 2 <= e && par < 0; j += 2) {
                    const int32_t u0 = p.col[j], u1 = p.col[j + 1];
                    const uint32_t w0 = ldcg(fcur + (u0 >> 5)), w1 = ldcg(fcur + (u1 >> 5));
                    if ((w0 >> (u0 & 31)) & 1u)
                        par = u0;
                    else if ((w1 >> (u1 & 31)) & 1u)
                        par = u1;
                }
                if (par < 0 && j < e) {
                    const int32_t u0 = p.col[j];
                    if ((ldcg(fcur + (u0 >> 5)) >> (u0 & 31)) & 1u)
                        par = u0;
                }
            }
            found = __ballot_sync(kFull, par >= 0);
            if (par >= 0) {
                p.dist[v] = k + 1;
                if (p.parent != nullptr)
                    p.parent[v] = par;
                t.found += 1;
                t.edges += (unsigned long long)deg;
                t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg : t.maxdeg;
            }
            if (lane == 0 && found != 0u)
                __stcg(p.visited + w, vis | found);
        }
        if (lane == 0)
            __stcg(fnext + w, found);
    }
}

// ------------------------------------------------------------ S8 switches

// F_k from queue to bitmap: clear fb[k & 1], then set one bit per queued
// vertex. The caller puts a grid barrier between the two halves.
template <typename RowT>
__device__ void queue_to_bitmap_clear(const Params<RowT>& p, int k)
{
    uint32_t* f = p.fb[k & 1];
    const int stride = gridDim.x * blockDim.x;
    for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < p.words; w += stride)
        __stcg(f + w, 0u);
}

template <typename RowT>
__device__ void queue_to_bitmap_set(const Params<RowT>& p, int k, int qn)
{
    uint32_t* f = p.fb[k & 1];
    const int32_t* qv = p.qv[k & 1];
    const int stride = gridDim.x * blockDim.x;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < qn; i += stride) {
        const int32_t v = ldcg(qv + i);
        atomicOr(f + (v >> 5), 1u << (v & 31));
    }
}

// F_k from bitmap to queue (with row starts and the degree prefix), through
// the same stage as push levels; counts go to the current slot's qpack.
template <typename RowT>
__device__ void bitmap_to_queue(const Params<RowT>& p, int k, const Smem<RowT>& sm,
                                SmemScalars& ss, LevelSlot* cur)
{
    const uint32_t* f = p.fb[k & 1];
    const int sel = k & 1;
    const int bd = blockDim.x;
    const int stride = gridDim.x * bd;
    for (int base = blockIdx.x * bd; base < p.words; base += stride) {
        const int w = base + threadIdx.x;
        if (w < p.words) {
            uint32_t bits = ldcg(f + w);
            while (bits) {
                const int bit = __ffs(bits) - 1;
                bits &= bits - 1;
                const int32_t v = (w << 5) + bit;
                const RowT b = p.row_ptr[v];
                const RowT deg = p.row_ptr[v + 1] - b;
                if (deg > 0)
                    stage_push(p, sm, ss, cur, sel, v, b, deg);
            }
        }
        if (__syncthreads_or(ss.stage_n > sm.cap / 2))
            stage_flush(p, sm, ss, cur, sel);
    }
    stage_flush(p, sm, ss, cur, sel);
}

// ------------------------------------------------------------ kernels

template <typename RowT>
__device__ __forceinline__ Smem<RowT> carve_smem(unsigned char* raw, int bd)
{
    Smem<RowT> sm;
    const int tile = bd * kItems;
    unsigned char* q = raw;
    sm.cap = tile;
    sm.wcap = tile + 1;
    sm.sb = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.cap;
    sm.sd = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.cap;
    sm.woff = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.wcap;
    sm.wbeg = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.wcap;
    sm.lb = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * bd;
    sm.ld = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * bd;
    sm.sv = reinterpret_cast<int32_t*>(q); q += sizeof(int32_t) * sm.cap;
    sm.wu = reinterpret_cast<int32_t*>(q); q += sizeof(int32_t) * sm.wcap;
    sm.lu = reinterpret_cast<int32_t*>(q);
    return sm;
}

template <typename RowT>
__host__ __device__ inline size_t level_smem_bytes(int bd)
{
    const size_t tile = (size_t)bd * kItems;
    return sizeof(RowT) * (2 * tile + 2 * (tile + 1) + 2 * (size_t)bd) +
           sizeof(int32_t) * (tile + (tile + 1) + (size_t)bd) + 16;
}

// The persistent level loop (S2-S9).
template <typename RowT>
__global__ void __launch_bounds__(512, 2) level_kernel(Params<RowT> p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ SmemScalars ss;
    const Smem<RowT> sm = carve_smem<RowT>(smem_raw, blockDim.x);
    if (threadIdx.x == 0) {
        ss.stage_n = 0;
        ss.nlarge = 0;
    }
    unsigned long long target = 0;
    int k = ldcg(&p.ctl->level);
    int budget = p.level_budget;
    const bool leader = blockIdx.x == 0 && threadIdx.x == 0;
    __syncthreads();

    while (ldcg(&p.ctl->done) == 0) {
        LevelSlot* cur = &p.ctl->slot[k & 3];
        LevelSlot* nxt = &p.ctl->slot[(k + 1) & 3];
        const LevelSlot* prv = &p.ctl->slot[(k + 3) & 3];
        const long long F = (long long)ldcg_u64(&cur->found);
        if (F == 0 || (p.max_depth >= 0 && k >= p.max_depth)) {
            if (leader) {
                const int nl = F == 0 ? k : k + 1;
                p.ctl->num_levels = nl;
                p.ctl->t_end_ns = global_timer_ns();
                if (p.num_levels_out != nullptr)
                    *p.num_levels_out = nl;
                __threadfence();
                p.ctl->done = 1;
            }
            break;
        }
        if (budget <= 0)
            break;
        const unsigned long long t_level = leader ? global_timer_ns() : 0ull;
        const long long mF = (long long)ldcg_u64(&cur->fedges);
        const unsigned long long maxdeg = ldcg_u64(&cur->maxdeg);
        const long long U = ldcg(&prv->unvisited) - F;
        const int prev_dir = ldcg(&prv->dir);
        int dir;
        if (!p.symmetric || p.direction == BFS_CSR_DIR_PUSH)
            dir = BFS_CSR_DIR_PUSH;
        else if (p.direction == BFS_CSR_DIR_PULL)
            dir = BFS_CSR_DIR_PULL;
        else
            dir = (double)mF > p.pull_ratio * (double)U ? BFS_CSR_DIR_PULL : BFS_CSR_DIR_PUSH;
        Tally t = {0ull, 0ull, 0ull};
        int adv = 0;

        if (dir == BFS_CSR_DIR_PULL) {
            if (leader) {
                LevelSlot* z = &p.ctl->slot[(k + 2) & 3];
                z->qpack = 0ull; z->found = 0ull; z->fedges = 0ull; z->maxdeg = 0ull;
                cur->unvisited = U;
                cur->dir = dir;
                cur->adv = 0;
            }
            if (prev_dir != BFS_CSR_DIR_PULL) {
                const int qn = (int)(ldcg_u64(&cur->qpack) >> p.eb);
                queue_to_bitmap_clear(p, k);
                if (!grid_barrier(p, target)) break;
                queue_to_bitmap_set(p, k, qn);
                if (!grid_barrier(p, target)) break;
            }
            pull_level(p, k, t);
        } else {
            if (prev_dir == BFS_CSR_DIR_PULL) {
                bitmap_to_queue(p, k, sm, ss, cur);
                if (!grid_barrier(p, target)) break;
            }
            const unsigned long long qp = ldcg_u64(&cur->qpack);
            const int qn = (int)(qp >> p.eb);
            const RowT qm = (RowT)(qp & ((1ull << p.eb) - 1ull));
            if (p.advance == BFS_CSR_ADV_BINNED)
                adv = BFS_CSR_ADV_BINNED;
            else if (p.advance == BFS_CSR_ADV_MERGE_PATH)
                adv = BFS_CSR_ADV_MERGE_PATH;
            else
                adv = (qn >= p.mp_min_frontier || maxdeg >= (unsigned long long)p.binned_max_deg)
                          ? BFS_CSR_ADV_MERGE_PATH : BFS_CSR_ADV_BINNED;
            if (leader) {
                LevelSlot* z = &p.ctl->slot[(k + 2) & 3];
                z->qpack = 0ull; z->found = 0ull; z->fedges = 0ull; z->maxdeg = 0ull;
                cur->unvisited = U;
                cur->dir = dir;
                cur->adv = adv;
            }
            if (adv == BFS_CSR_ADV_MERGE_PATH)
                push_merge_path(p, k, qn, qm, sm, ss, nxt, t);
            else
                push_binned(p, k, qn, qm, sm, ss, nxt, t);
        }
        if (leader && k < p.stats_cap) {
            bfs_csr_level_stat st;
            st.level = k;
            st.direction = dir;
            st.advance = adv;
            st.reserved = 0;
            st.frontier = F;
            st.frontier_edges = mF;
            st.unvisited = U;
            st.max_degree = (long long)maxdeg;
            st.t_start_ns = (long long)t_level;
            p.stats[k] = st;
        }
        publish_tally<RowT>(t, nxt, ss);
        if (!grid_barrier(p, target)) break;
        ++k;
        --budget;
    }

    // Leave: the last CTA out resets the barrier for the next launch.
    __syncthreads();
    if (threadIdx.x == 0) {
        if (blockIdx.x == 0)
            p.ctl->level = k;
        __threadfence();
        const unsigned int prev = atomicAdd(&p.ctl->exit_count, 1u);
        if (prev == gridDim.x - 1) {
            p.ctl->bar = 0ull;
            p.ctl->exit_count = 0u;
            __threadfence();
        }
    }
}

// S1: reset the run state and seed the source. dist and parent are filled
// with -1 (source: 0 and itself), visited starts as the dead bitmap (vertices
// of degree 0 and padding bits beyond n) plus the source bit, and slot 0
// holds F_0 = {source}.
template <typename RowT>
__global__ void init_kernel(Params<RowT> p, const uint32_t* __restrict__ dead, int32_t source,
                            int use_dead)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int32_t n = p.n;
    const int64_t n4 = n / 4;
    int4* d4 = reinterpret_cast<int4*>(p.dist);
    int4* p4 = reinterpret_cast<int4*>(p.parent);
    const int4 neg = make_int4(-1, -1, -1, -1);
    const bool aligned = (reinterpret_cast<uintptr_t>(p.dist) & 15u) == 0 &&
                         (p.parent == nullptr || (reinterpret_cast<uintptr_t>(p.parent) & 15u) == 0);
    if (aligned) {
        for (int64_t i = tid; i < n4; i += stride) {
            int4 dv = neg, pv = neg;
            if (source / 4 == i) {
                (&dv.x)[source & 3] = 0;
                (&pv.x)[source & 3] = source;
            }
            d4[i] = dv;
            if (p.parent != nullptr)
                p4[i] = pv;
        }
        for (int64_t i = n4 * 4 + tid; i < n; i += stride) {
            p.dist[i] = i == source ? 0 : -1;
            if (p.parent != nullptr)
                p.parent[i] = i == source ? source : -1;
        }
    } else {
        for (int64_t i = tid; i < n; i += stride) {
            p.dist[i] = i == source ? 0 : -1;
            if (p.parent != nullptr)
                p.parent[i] = i == source ? source : -1;
        }
    }
    for (int64_t w = tid; w < p.words; w += stride) {
        uint32_t x = use_dead ? dead[w] : 0u;
        if (!use_dead && w == p.words - 1 && (n & 31))
            x |= ~((1u << (n & 31)) - 1u);  // padding bits beyond n
        if (w == (source >> 5))
            x |= 1u << (source & 31);
        p.visited[w] = x;
    }
    if (tid == 0) {
        Ctl* c = p.ctl;
        const RowT b = p.row_ptr[source];
        const RowT deg = p.row_ptr[source + 1] - b;
        c->bar = 0ull;
        c->exit_count = 0u;
        c->status = BFS_CSR_OK;
        c->done = 0;
        c->level = 0;
        c->num_levels = 0;
        c->t_end_ns = 0ull;
        for (int s = 0; s < kSlots; ++s) {
            c->slot[s].qpack = 0ull;
            c->slot[s].found = 0ull;
            c->slot[s].fedges = 0ull;
            c->slot[s].maxdeg = 0ull;
            c->slot[s].unvisited = 0;
            c->slot[s].dir = BFS_CSR_DIR_PUSH;
            c->slot[s].adv = 0;
        }
        c->slot[0].found = 1ull;
        c->slot[0].fedges = (unsigned long long)deg;
        c->slot[0].maxdeg = (unsigned long long)deg;
        if (deg > 0) {
            c->slot[0].qpack = (1ull << p.eb) | (unsigned long long)deg;
            p.qv[0][0] = source;
            p.qbeg[0][0] = b;
            p.qoff[0][0] = 0;
        }
        // U_0 = nonisolated vertices other than the source: slot 3 holds U_{-1}
        // such that U_0 = U_{-1} - |F_0|.
        c->slot[3].unvisited = c->nonisolated - (deg > 0 ? 1 : 0) + 1;
        c->slot[3].dir = BFS_CSR_DIR_PUSH;
    }
}

// S0: CSR checks (row_ptr[0] = 0, row_ptr[n] = nnz, non-decreasing, col in
// range). Flags: bit 0 row_ptr, bit 1 col.
template <typename RowT>
__global__ void validate_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                                int64_t n, int64_t nnz, int* flags)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int bad = 0;
    if (tid == 0 && (row_ptr[0] != 0 || (int64_t)row_ptr[n] != nnz))
        bad |= 1;
    for (int64_t i = tid; i < n; i += stride)
        if (row_ptr[i + 1] < row_ptr[i])
            bad |= 1;
    for (int64_t e = tid; e < nnz; e += stride) {
        const int32_t v = col[e];
        if (v < 0 || (int64_t)v >= n)
            bad |= 2;
    }
    if (bad)
        atomicOr(flags, bad);
}

// Vertices of out-degree 0 (and padding bits beyond n) as a bitmap, and the
// count of the others. For a symmetric CSR such vertices are isolated.
template <typename RowT>
__global__ void dead_kernel(const RowT* __restrict__ row_ptr, int32_t n, int32_t words,
                            uint32_t* dead, long long* nonisolated)
{
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    long long live = 0;
    for (int64_t w = gw; w < words; w += nw) {
        const int64_t v = (w << 5) + lane;
        const bool d = v >= n || row_ptr[v + 1] == row_ptr[v];
        const unsigned m = __ballot_sync(kFull, d);
        if (lane == 0) {
            dead[w] = m;
            live += 32 - __popc(m);
        }
    }
    if (lane == 0 && live)
        atomicAdd(reinterpret_cast<unsigned long long*>(nonisolated), (unsigned long long)live);
}

}  // namespace fbc
