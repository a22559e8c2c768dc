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
//      frontier's degrees plus a search per warp and per edge; Gunrock
//      reading page steps 4-5, and "The Frontier Model for Parallel BFS"
//      section 22.3).
//   S5 discovery: atomicOr on a visited bitmap, or atomicCAS on dist
//      (Day 38 claimVertex; ch. 22 sections 22.1-22.2); exactly one winner
//      per vertex writes dist and parent.
//   S6 compaction: winners are staged in shared memory and flushed with one
//      global atomic per CTA (or, in the merge path, per warp) batch (the
//      privatised queue of PMPP ch. 15 notes,
//      section 15.6, without its silent drop on overflow: a full stage makes
//      the thread append directly).
//   S7 pull level over a frontier bitmap, one warp per 32-vertex word: no
//      atomics, dedupe by construction (Gunrock reading page, step 6).
//   S8 representation switches queue <-> bitmap when the direction changes.
//   S9 a bounded grid barrier ends each phase; the loop stops on an empty
//      frontier (Gunrock's convergence test, read on the device).
//
// The exclusive prefix the merge-path search needs is produced for free by
// the compaction: a CTA or warp reserves its queue slots and its edge range
// with one 64-bit atomicAdd on a packed (count, edges) counter, so queue
// order and edge order agree and qoff[] is a valid exclusive scan of the
// degrees.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_runtime.h>

#include "bfs_csr.h"

namespace fbc {

constexpr int kItems = 4;        // edges per thread per single-CTA level round

// Single-CTA level capacities, in entries. The stage holds the next frontier
// (and is the CTA stage of the grid-wide compaction); a single-CTA level's
// edges are bounded by it, so its winners always fit. The window holds the
// current frontier. Both are one round of kItems entries per thread (the
// window three with 8-byte row offsets, see window_cap): a wider
// stage (7,168 entries with 4-byte row offsets, several rounds per level)
// made the lattice's levels slower on one CTA than on the whole grid, and
// its shared memory took L1 capacity from the other configurations.
template <typename RowT>
__host__ __device__ constexpr int stage_cap(int bd)
{
    return kItems * bd;
}

template <typename RowT>
__host__ __device__ constexpr int window_cap(int bd)
{
    // three rounds for 8-byte row offsets, so that two CTAs' shared memory
    // leaves the SM a 124 KB L1 (the window's frontier of single-CTA levels
    // is then at most 3 * bd - 1 vertices)
    return (sizeof(RowT) == 8 ? 3 : kItems) * bd;
}
constexpr int kSlots = 4;        // rotating per-level counter slots
// Threads per CTA of the level kernel (its largest and default block), two
// CTAs per SM, so the register file gives each thread 65536 / (2 * block)
// registers: 384 threads (80 registers, no spills) with 4-byte row offsets,
// 512 threads (64 registers) with 8-byte ones. Measured on GB300: 384 is
// 8-12 % faster on the graphs of up to 2^22 vertices, 512 is 4-5 % faster on
// R-MAT scale 25 with two searches in flight.
template <typename RowT>
__host__ __device__ constexpr int level_block()
{
    return sizeof(RowT) == 4 ? 384 : 512;
}
constexpr int kLevelBlockMax = 512;

// A push level below the merge-path frontier threshold still takes the merge
// path when its rows average at least this many entries: short rows (a
// lattice's) are walked fastest one thread per vertex, longer ones are
// balanced better edge by edge.
constexpr long long kMergePathMinAvgDegree = 8;
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
    unsigned int work_next;     // (unused) chunk counter
    unsigned int pad_slot;
    long long unvisited_edges;  // m_U at level k: out-degree sum of U_k
};

struct __align__(128) Ctl {
    unsigned long long bar;     // barrier arrivals in the current launch
    unsigned long long pad0[15];
    unsigned int exit_count;    // CTAs that left the current launch
    int status;                 // BFS_CSR_OK or a device error code
    int done;                   // the search has ended
    int level;                  // next level to run (persists across launches)
    int num_levels;             // non-empty frontiers, valid once done
    int solo_resume;            // first level after a single-CTA session
    int pad1[26];
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
    // Hop code per vertex while a search runs (bitmap discovery only): the
    // low 7 bits are 0 unreached, d + 1 for a distance d < kHopDirect,
    // kHopFar when the distance itself went straight to dist; the top bit
    // says the parent is the vertex's probe neighbour (probe[]) and was not
    // stored. dist and parent are written from the codes once, coalesced,
    // when the search ends.
    uint8_t* hop;
    int defer_dist;             // 1: discoveries write hop codes (bitmap discovery)
    // 1 (only with defer_dist): a pull level's probe hits store no parent;
    // the end-of-search pass writes every parent from the hop-code flags. Set
    // when the parent array is too large for the L2 to absorb scattered
    // stores into it.
    int defer_parent;
    uint32_t* visited;
    const uint32_t* dead;       // degree-0 vertices and padding bits (symmetric CSR)
    // Per vertex: its probe neighbour (the highest-degree one among the row's
    // first entries) in bits 0-30, kProbeNone for a row without entries,
    // and bit 31 set when that neighbour is the row's only entry.
    const uint32_t* probe;
    int vec_out;                // dist and parent are 16-byte aligned
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
    double pull_alpha;
    int push_beta;
    long long nnz;
    int max_depth;
    int symmetric;
    int level_budget;           // levels this launch may run
    long long timeout_ns;
    int unreachable_barrier;
    int narrow_max;             // single-CTA levels: frontier edges (and vertices) <= this
    long long* stamps;          // may be null: global timer at init, level-loop start and end
    // BFS_CSR_FRONTIER_*: how a push level hands its winners to the next
    // level; the padded modes use pad[] (max(nnz, 1) entries each).
    int frontier_output;
    int32_t* pad[2];
    int32_t* wq;                // winners of a large push level, before their degrees
    // A pull level that starts with at most this many unvisited vertices also
    // appends what it finds to the next queue, so that a push level after it
    // needs no bitmap-to-queue pass.
    long long emit_max;
    // Graph loop mode: the conditional handle of the CUDA graph's while node
    // whose body launches this kernel once per level (0 otherwise).
    unsigned long long graph_cond;
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

__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// Grid-wide barrier with a bounded wait. All CTAs of the cooperative launch
// call it the same number of times. After the CTA's own barrier, thread 0
// arrives with a release add (publishing every write the CTA made before the
// barrier) and polls the arrival counter with acquire loads until every CTA
// has arrived or the time limit passes; on expiry it records
// BFS_CSR_ETIMEOUT and the caller stops. A status set by another CTA is
// picked up at the next level start.
template <typename RowT>
__device__ __forceinline__ bool grid_barrier(const Params<RowT>& p, unsigned long long& target)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        target += gridDim.x;
        const unsigned long long want = target + (unsigned long long)p.unreachable_barrier;
        red_release_add_u64(&p.ctl->bar, 1ull);
        int ok = 1;
        if (ld_acquire_u64(&p.ctl->bar) < want) {
            const unsigned long long t0 = global_timer_ns();
            unsigned int spins = 0;
            while (ld_acquire_u64(&p.ctl->bar) < want) {
                if ((++spins & 63u) == 0u &&
                    (global_timer_ns() - t0 > (unsigned long long)p.timeout_ns || spins > (1u << 30))) {
                    atomicCAS(&p.ctl->status, BFS_CSR_OK, BFS_CSR_ETIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
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
    int32_t* sd;      // degree (a row holds fewer than 2^31 entries)
    int cap;
    // single-CTA level frontier (offsets, row starts, vertices)
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
    unsigned long long solo_found, solo_edges, solo_maxdeg;
    long long tmp_ll[33];
};

// Per-thread tallies of the vertices this thread discovered in a level.
// Push levels count the found vertices' out-degrees in `edges`; pull levels
// count there the out-degrees of the unvisited vertices they did not find.
struct Tally {
    unsigned long long found;
    unsigned long long edges;
    unsigned long long maxdeg;
};

// ------------------------------------------------------------ S6 compaction

// Append one discovered vertex (degree > 0) to the next queue directly with a
// single packed atomic. Used only when the shared-memory stage is full.
template <typename RowT>
__device__ void append_direct(const Params<RowT>& p, LevelSlot* nxt, int qsel,
                                           int32_t v, RowT b, RowT deg)
{
    const unsigned long long old = atomicAdd(&nxt->qpack, (1ull << p.eb) | (unsigned long long)deg);
    const unsigned long long slot = old >> p.eb;
    const unsigned long long eoff = old & ((1ull << p.eb) - 1ull);
    p.qv[qsel][slot] = v;
    p.qbeg[qsel][slot] = b;
    p.qoff[qsel][slot] = (RowT)eoff;
}

// Stage v (row start b, degree deg) when take is set. Every converged lane
// of the warp calls it; one shared atomic per warp reserves the slots of all
// its taking lanes (a per-lane atomic on the one counter serialises when
// most edges discover). A slot past the stage's capacity goes straight to
// the queue.
template <typename RowT>
__device__ __forceinline__ void stage_push(const Params<RowT>& p, const Smem<RowT>& sm,
                                           SmemScalars& ss, LevelSlot* nxt, int qsel,
                                           int32_t v, RowT b, RowT deg, bool take)
{
    const unsigned act = __activemask();
    const unsigned m = __ballot_sync(act, take);
    if (m == 0u)
        return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader)
        base = atomicAdd(&ss.stage_n, __popc(m));
    base = __shfl_sync(act, base, leader);
    if (take) {
        const int pos = base + __popc(m & ((1u << lane) - 1u));
        if (pos < sm.cap) {
            sm.sv[pos] = v;
            sm.sb[pos] = b;
            sm.sd[pos] = (int32_t)deg;
        } else {
            append_direct(p, nxt, qsel, v, b, deg);
        }
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

// End of a level: one atomic per CTA for each frontier statistic. After a
// pull level (`pulled`) fedges accumulates minus the edges of the vertices
// left unvisited, so that the next level reads m_F = m_U - that sum: the
// unvisited vertices at the level's start are exactly the ones it found plus
// the ones it did not.
template <typename RowT>
__device__ void publish_tally(const Tally& t, LevelSlot* nxt, SmemScalars& ss, bool pulled)
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
        if (tot_found > 0)
            atomicAdd(&nxt->found, (unsigned long long)tot_found);
        if (pulled) {
            if (tot_edges != 0)
                atomicAdd(&nxt->fedges, (unsigned long long)(-tot_edges));
        } else if (tot_found > 0) {
            atomicAdd(&nxt->fedges, (unsigned long long)tot_edges);
            atomicMax(&nxt->maxdeg, mm);
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------ S5 discovery

// Distances below kHopDirect are kept as one byte per vertex during the
// search: a discovery then touches one byte of an array an eighth the size
// of dist (it mostly stays in L2) instead of a 4-byte slot of a 32-byte DRAM
// sector that must be read, merged and written back. Larger distances (long
// paths, lattices) go to dist directly and are marked kHopFar. The top bit,
// kHopProbe, marks a vertex whose parent is its probe neighbour: almost
// every vertex a pull level finds (the probe is the one neighbour it tests
// first), so its parent costs no scattered store either and is written by
// the end-of-search pass from probe[], sequentially.
constexpr int kHopDirect = 126;
constexpr uint8_t kHopFar = 127;
constexpr uint8_t kHopProbe = 0x80;
constexpr uint32_t kProbeNone = 0x7fffffffu;

template <typename RowT>
__device__ __forceinline__ void record_dist(const Params<RowT>& p, int32_t v, int d,
                                            bool probe_parent = false)
{
    if (p.defer_dist) {
        const uint8_t flag = probe_parent ? kHopProbe : (uint8_t)0;
        if (d < kHopDirect) {
            p.hop[v] = (uint8_t)(d + 1) | flag;
        } else {
            p.hop[v] = kHopFar | flag;
            p.dist[v] = d;
        }
    } else {
        p.dist[v] = d;
    }
}

// The claim of vertex v by frontier vertex u at level k. Exactly one caller
// per v gets true; the winner writes dist[v] and parent[v]. With
// BFS_CSR_DISC_MIN the claim is an atomic minimum of dist[v], read as an
// unsigned word so that the unvisited -1 is the largest value: the first
// caller sees the old -1 and wins, any later one sees level + 1 and loses
// (the Gunrock page, step 2); min is idempotent, so every interleaving
// leaves the same dist.
__device__ __forceinline__ unsigned int* as_unsigned(int32_t* x)
{
    return reinterpret_cast<unsigned int*>(x);
}

template <typename RowT>
__device__ __forceinline__ bool claim(const Params<RowT>& p, int k, int32_t v, int32_t u,
                                      bool precheck)
{
    if (p.discovery == BFS_CSR_DISC_CAS) {
        if (precheck && ldcg(&p.dist[v]) != -1)
            return false;
        if (atomicCAS(&p.dist[v], -1, k + 1) != -1)
            return false;
        atomicOr(&p.visited[v >> 5], 1u << (v & 31));  // keeps pull levels exact
    } else if (p.discovery == BFS_CSR_DISC_MIN) {
        const unsigned int d = (unsigned int)(k + 1);
        if (precheck && (unsigned int)ldcg(&p.dist[v]) <= d)
            return false;
        if (!(d < atomicMin(as_unsigned(p.dist + v), d)))
            return false;
        atomicOr(&p.visited[v >> 5], 1u << (v & 31));  // keeps pull levels exact
    } else {
        const uint32_t bit = 1u << (v & 31);
        uint32_t* w = p.visited + (v >> 5);
        if (precheck && (ldcg(w) & bit))
            return false;
        if (atomicOr(w, bit) & bit)
            return false;
        record_dist(p, v, k + 1);
    }
    if (p.parent != nullptr)
        p.parent[v] = u;
    return true;
}

// N claims at once: every load and atomic of the batch is issued before any
// result is used, so their round trips overlap. v[i] < 0 marks an empty lane
// of the batch.
template <typename RowT, int N>
__device__ __forceinline__ void claim_batch(const Params<RowT>& p, int k, const int32_t (&v)[N],
                                            const int32_t (&u)[N], bool precheck, bool (&won)[N])
{
    if (p.discovery == BFS_CSR_DISC_CAS) {
        int32_t seen[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            seen[i] = (v[i] >= 0 && precheck) ? ldcg(&p.dist[v[i]]) : -1;
#pragma unroll
        for (int i = 0; i < N; ++i)
            won[i] = v[i] >= 0 && seen[i] == -1 && atomicCAS(&p.dist[v[i]], -1, k + 1) == -1;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (won[i])
                atomicOr(&p.visited[v[i] >> 5], 1u << (v[i] & 31));
    } else if (p.discovery == BFS_CSR_DISC_MIN) {
        const unsigned int d = (unsigned int)(k + 1);
        unsigned int seen[N], old[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            seen[i] = (v[i] >= 0 && precheck) ? (unsigned int)ldcg(&p.dist[v[i]]) : 0xffffffffu;
#pragma unroll
        for (int i = 0; i < N; ++i)
            old[i] = (v[i] >= 0 && seen[i] > d) ? atomicMin(as_unsigned(p.dist + v[i]), d) : 0u;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            won[i] = v[i] >= 0 && d < old[i];
            if (won[i])
                atomicOr(&p.visited[v[i] >> 5], 1u << (v[i] & 31));
        }
    } else {
        uint32_t seen[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            seen[i] = (v[i] >= 0 && precheck) ? ldcg(p.visited + (v[i] >> 5)) : 0u;
        uint32_t old[N];
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const uint32_t bit = 1u << (v[i] & 31);
            old[i] = bit;
            if (v[i] >= 0 && !(seen[i] & bit))
                old[i] = atomicOr(p.visited + (v[i] >> 5), bit);
        }
#pragma unroll
        for (int i = 0; i < N; ++i) {
            won[i] = v[i] >= 0 && !(old[i] & (1u << (v[i] & 31)));
            if (won[i])
                record_dist(p, v[i], k + 1);
        }
    }
    if (p.parent != nullptr) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (won[i])
                p.parent[v[i]] = u[i];
    }
}

// After a claim: a winner reads v's row, counts it, and is queued when it
// has edges. Every converged lane calls it (won false for the others).
template <typename RowT>
__device__ __forceinline__ void after_win(const Params<RowT>& p, const Smem<RowT>& sm,
                                          SmemScalars& ss, LevelSlot* nxt, int qsel, Tally& t,
                                          int32_t v, bool won)
{
    RowT b = 0, deg = 0;
    if (won) {
        b = p.row_ptr[v];
        deg = p.row_ptr[v + 1] - b;
        t.found += 1;
        t.edges += (unsigned long long)deg;
        t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg : t.maxdeg;
    }
    stage_push(p, sm, ss, nxt, qsel, v, b, deg, won && deg > 0);
}

// after_win for a batch: the row offsets of all winners are loaded together.
template <typename RowT, int N>
__device__ __forceinline__ void after_win_batch(const Params<RowT>& p, const Smem<RowT>& sm,
                                                SmemScalars& ss, LevelSlot* nxt, int qsel,
                                                Tally& t, const int32_t (&v)[N],
                                                const bool (&won)[N])
{
    RowT b[N], e[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        b[i] = 0;
        e[i] = 0;
        if (won[i]) {
            b[i] = p.row_ptr[v[i]];
            e[i] = p.row_ptr[v[i] + 1];
        }
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const RowT deg = e[i] - b[i];
        if (won[i]) {
            t.found += 1;
            t.edges += (unsigned long long)deg;
            t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg : t.maxdeg;
        }
        stage_push(p, sm, ss, nxt, qsel, v[i], b[i], deg, won[i] && deg > 0);
    }
}

// ------------------------------------------------------------ S4 push levels

// Degree-binned advance: thread per vertex below small_max, warp per vertex
// below cta_min, whole CTA per vertex above. Frontier entry i belongs to
// CTA i % G so that small frontiers spread over every SM.
template <typename RowT>
__device__ void push_binned(const Params<RowT>& p, int k, int qn, RowT qm, const Smem<RowT>& sm,
                            SmemScalars& ss, LevelSlot* nxt, Tally& t, bool pre)
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
            for (RowT j = 0; j < deg; j += 4) {
                int32_t vv[4], uu[4];
                bool won[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    vv[i] = j + i < deg ? p.col[b + j + i] : -1;
                    uu[i] = u;
                }
                claim_batch(p, k, vv, uu, pre, won);
                after_win_batch(p, sm, ss, nxt, ns, t, vv, won);
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
                after_win(p, sm, ss, nxt, ns, t, v, claim(p, k, v, wu, pre));
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
                    after_win(p, sm, ss, nxt, ns, t, v, claim(p, k, v, cu, pre));
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

// Warp-level merge path. The level's edge range [0, m_F) is split evenly over
// all warps of the grid; a warp walks its share in batches of up to kWItems
// items of 32 consecutive edges, with no CTA-wide barrier, so every warp is
// an independent chain of loads (a CTA-wide tile loop gives the SM only as
// many chains as it has CTAs, and every tile waits for the slowest warp).
// The warp keeps a window of 32 queue entries in registers, one per lane:
// the entry's edge offset, row start and vertex, and the end of its range.
// For an item starting at edge e, the entry of e is the first lane whose
// range ends after e, and lane l's entry is that one plus the number of
// entries starting in (e, e + l], read from one OR-reduction of start bits.
// 32 consecutive edges span at most 32 entries (every queued vertex has an
// edge), so a window whose first entry holds e covers a whole item. Winners
// go to the warp's own slice of the stage; a flush moves it to the next
// queue with one packed atomic per warp.
constexpr int kWarpStage = 224;  // stage entries per warp
constexpr int kWItems = 4;       // 32-edge items per warp batch

template <typename RowT>
struct WarpStage {
    RowT* b;
    int32_t* v;
    int32_t* d;
};

template <typename RowT>
__device__ __forceinline__ WarpStage<RowT> warp_stage(unsigned char* raw)
{
    unsigned char* q = raw + (size_t)(threadIdx.x >> 5) * kWarpStage * (sizeof(RowT) + 8);
    WarpStage<RowT> w;
    w.b = reinterpret_cast<RowT*>(q);
    w.v = reinterpret_cast<int32_t*>(q + sizeof(RowT) * kWarpStage);
    w.d = w.v + kWarpStage;
    return w;
}

// Move the warp's n staged vertices to the next queue: one packed atomic
// reserves their slots and edge range; they are written 32 at a time with
// the exclusive prefix of their degrees.
template <typename RowT>
__device__ void warp_flush(const Params<RowT>& p, const WarpStage<RowT>& ws, int n,
                           LevelSlot* nxt, int qsel)
{
    __syncwarp();
    const int lane = threadIdx.x & 31;
    unsigned long long sum = 0ull;
    for (int i = lane; i < n; i += 32)
        sum += (unsigned long long)ws.d[i];
    sum = warp_sum(sum);
    unsigned long long old = 0ull;
    if (lane == 0)
        old = atomicAdd(&nxt->qpack, ((unsigned long long)n << p.eb) | sum);
    old = __shfl_sync(kFull, old, 0);
    const unsigned long long base = old >> p.eb;
    unsigned long long run = old & ((1ull << p.eb) - 1ull);
    int32_t* qv = p.qv[qsel];
    RowT* qb = p.qbeg[qsel];
    RowT* qo = p.qoff[qsel];
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const unsigned long long d = i < n ? (unsigned long long)ws.d[i] : 0ull;
        const unsigned long long inc = warp_inclusive_scan(d);
        if (i < n) {
            qv[base + i] = ws.v[i];
            qb[base + i] = ws.b[i];
            qo[base + i] = (RowT)(run + inc - d);
        }
        run += __shfl_sync(kFull, inc, 31);
    }
    __syncwarp();
}

// Large push levels (at least kIdsMinEdges frontier edges) keep the winners'
// row offsets out of the claim chain: the merge path stages only the winners'
// ids (ids_flush appends them to wq, counted in the next slot's work_next),
// and after a grid barrier queue_from_ids loads their row offsets with many
// loads in flight and builds the queue of F_{k+1}.
constexpr long long kIdsMinEdges = 1ll << 20;

template <typename RowT>
__device__ void ids_flush(const Params<RowT>& p, const WarpStage<RowT>& ws, int n, LevelSlot* nxt)
{
    __syncwarp();
    const int lane = threadIdx.x & 31;
    unsigned int base = 0u;
    if (lane == 0)
        base = atomicAdd(&nxt->work_next, (unsigned int)n);
    base = __shfl_sync(kFull, base, 0);
    for (int i = lane; i < n; i += 32)
        p.wq[base + i] = ws.v[i];
    __syncwarp();
}

template <typename RowT, bool kIds>
__device__ void push_warp_mp(const Params<RowT>& p, int k, int qn, RowT qm, unsigned char* raw,
                             LevelSlot* nxt, Tally& t, bool pre)
{
    const int cs = k & 1, ns = cs ^ 1;
    const int32_t* qv = p.qv[cs];
    const RowT* qb = p.qbeg[cs];
    const RowT* qo = p.qoff[cs];
    const int lane = threadIdx.x & 31;
    const unsigned long long W = (unsigned long long)gridDim.x * (blockDim.x >> 5);
    const unsigned long long gw =
        (unsigned long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    // Edge positions in 64 bits: e + 32 * j never overflows an int32 row_ptr.
    const long long e_lo = (long long)((unsigned long long)qm * gw / W);
    const long long e_hi = (long long)((unsigned long long)qm * (gw + 1) / W);
    if (e_lo >= e_hi)
        return;
    const WarpStage<RowT> ws = warp_stage<RowT>(raw);

    // First entry: the last i with qoff[i] <= e_lo (qoff[0] = 0), 32-ary search.
    int cur = 0;
    {
        int hi = qn;
        while (hi - cur > 1) {
            const int step = (hi - cur + 31) / 32;
            const int probe = cur + lane * step;
            const bool le = lane > 0 && probe < hi && ldcg(qo + probe) <= e_lo;
            const unsigned bal = __ballot_sync(kFull, le);
            if (bal == 0u) {
                hi = min(hi, cur + step);
            } else {
                cur = cur + (31 - __clz(bal)) * step;
                hi = min(hi, cur + step);
            }
        }
    }
    RowT off, beg, end;
    int32_t vtx;
    // Window of entries [c, c + 32); lanes past the queue hold empty ranges
    // at m_F.
    auto load_window = [&](int c) {
        const int i = c + lane;
        if (i < qn) {
            off = ldcg(qo + i);
            beg = ldcg(qb + i);
            vtx = ldcg(qv + i);
        } else {
            off = qm;
            beg = 0;
            vtx = -1;
        }
        RowT nx = __shfl_down_sync(kFull, off, 1);
        if (lane == 31)
            nx = c + 32 < qn ? ldcg(qo + c + 32) : qm;
        end = nx;
    };
    load_window(cur);
    long long e = e_lo;
    int cnt = 0;  // staged entries (the same in every lane)
    while (e < e_hi) {
        const long long wend = (long long)__shfl_sync(kFull, end, 31);
        if (e >= wend) {  // e is the first edge of entry cur + 32
            cur += 32;
            load_window(cur);
            continue;
        }
        const int x0 = __ffs(__ballot_sync(kFull, (long long)end > e)) - 1;
        int n = 0;
#pragma unroll
        for (int j = 0; j < kWItems; ++j) {
            const long long first = e + 32 * j;
            const long long last = first + 31 < e_hi - 1 ? first + 31 : e_hi - 1;
            if (n == j && first < e_hi && last < wend)
                n = j + 1;
        }
        if (n < kWItems && x0 > 0 && e + 32 * n < e_hi) {
            cur += x0;  // slide the window to the entry of e and look again
            load_window(cur);
            continue;
        }
        if (cnt + 32 * n > kWarpStage) {
            if constexpr (kIds)
                ids_flush(p, ws, cnt, nxt);
            else
                warp_flush(p, ws, cnt, nxt, ns);
            cnt = 0;
        }
        int32_t vv[kWItems], uu[kWItems];
#pragma unroll
        for (int j = 0; j < kWItems; ++j) {
            vv[j] = -1;
            uu[j] = 0;
            if (j < n) {
                const long long e0 = e + 32 * j;
                const int xf = __ffs(__ballot_sync(kFull, (long long)end > e0)) - 1;
                const long long rel = (long long)off - e0;
                const unsigned starts =
                    __reduce_or_sync(kFull, (rel > 0 && rel < 32) ? 1u << (int)rel : 0u);
                const int xl = xf + __popc(starts & ((2u << lane) - 1u));
                const RowT o = __shfl_sync(kFull, off, xl);
                const RowT bg = __shfl_sync(kFull, beg, xl);
                const int32_t u = __shfl_sync(kFull, vtx, xl);
                const long long ej = e0 + lane;
                if (ej < e_hi) {
                    uu[j] = u;
                    vv[j] = p.col[bg + (RowT)(ej - (long long)o)];
                }
            }
        }
        bool won[kWItems];
        claim_batch(p, k, vv, uu, pre, won);
        if (p.frontier_output == BFS_CSR_FRONTIER_PADDED_FILTER) {
            // Every edge of the level writes its slot of the padded output:
            // the neighbour it claimed, or the sentinel -1 (the filter pass
            // compacts them).
#pragma unroll
            for (int j = 0; j < kWItems; ++j) {
                const long long ej = e + 32 * j + lane;
                if (j < n && ej < e_hi)
                    p.pad[0][ej] = won[j] ? vv[j] : -1;
            }
            e += 32 * n;
            continue;
        }
        if constexpr (kIds) {
            // winners' ids only; their degrees come later (queue_from_ids)
#pragma unroll
            for (int j = 0; j < kWItems; ++j) {
                if (won[j])
                    t.found += 1;
                const unsigned m = __ballot_sync(kFull, won[j]);
                if (won[j])
                    ws.v[cnt + __popc(m & ((1u << lane) - 1u))] = vv[j];
                cnt += __popc(m);
            }
        } else {
            RowT wb[kWItems], we[kWItems];
#pragma unroll
            for (int j = 0; j < kWItems; ++j) {
                wb[j] = 0;
                we[j] = 0;
                if (won[j]) {
                    wb[j] = p.row_ptr[vv[j]];
                    we[j] = p.row_ptr[vv[j] + 1];
                }
            }
#pragma unroll
            for (int j = 0; j < kWItems; ++j) {
                const RowT deg = we[j] - wb[j];
                if (won[j]) {
                    t.found += 1;
                    t.edges += (unsigned long long)deg;
                    t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg
                                                                  : t.maxdeg;
                }
                const bool take = won[j] && deg > 0;
                const unsigned m = __ballot_sync(kFull, take);
                if (take) {
                    const int pos = cnt + __popc(m & ((1u << lane) - 1u));
                    ws.v[pos] = vv[j];
                    ws.b[pos] = wb[j];
                    ws.d[pos] = (int32_t)deg;
                }
                cnt += __popc(m);
            }
        }
        e += 32 * n;
    }
    if (cnt > 0) {
        if constexpr (kIds)
            ids_flush(p, ws, cnt, nxt);
        else
            warp_flush(p, ws, cnt, nxt, ns);
    }
}

// The queue of F_{k+1} from the winners' ids in wq (nxt->work_next of them):
// every warp takes an even share, loads kIdsBatch ids and their row offsets
// per lane at a time, stages the vertices with edges and flushes them with
// the packed atomic of the merge path. Adds the degrees to the tally (the
// push level counted the winners).
template <typename RowT>
__device__ void queue_from_ids(const Params<RowT>& p, int k, unsigned char* raw, LevelSlot* nxt,
                               Tally& t)
{
    constexpr int kIdsBatch = 4;
    const long long total = (long long)ldcg(&nxt->work_next);
    const long long W = (long long)gridDim.x * (blockDim.x >> 5);
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long long lo = total * gw / W, hi = total * (gw + 1) / W;
    const WarpStage<RowT> ws = warp_stage<RowT>(raw);
    const int lane = threadIdx.x & 31;
    const int ns = (k + 1) & 1;
    for (long long c0 = lo; c0 < hi; c0 += kWarpStage) {
        const int m = (int)(hi - c0 < kWarpStage ? hi - c0 : kWarpStage);
        int cnt = 0;
        for (int j0 = 0; j0 < m; j0 += 32 * kIdsBatch) {
            int32_t v[kIdsBatch];
            RowT b[kIdsBatch], e[kIdsBatch];
#pragma unroll
            for (int u = 0; u < kIdsBatch; ++u) {
                const int j = j0 + 32 * u + lane;
                v[u] = j < m ? ldcg(p.wq + c0 + j) : -1;
            }
#pragma unroll
            for (int u = 0; u < kIdsBatch; ++u) {
                b[u] = v[u] >= 0 ? p.row_ptr[v[u]] : (RowT)0;
                e[u] = v[u] >= 0 ? p.row_ptr[v[u] + 1] : (RowT)0;
            }
#pragma unroll
            for (int u = 0; u < kIdsBatch; ++u) {
                const RowT deg = e[u] - b[u];
                const bool take = v[u] >= 0 && deg > 0;
                if (take) {
                    t.edges += (unsigned long long)deg;
                    t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg
                                                                  : t.maxdeg;
                }
                const unsigned tm = __ballot_sync(kFull, take);
                if (take) {
                    const int pos = cnt + __popc(tm & ((1u << lane) - 1u));
                    ws.v[pos] = v[u];
                    ws.b[pos] = b[u];
                    ws.d[pos] = (int32_t)deg;
                }
                cnt += __popc(tm);
            }
        }
        if (cnt > 0)
            warp_flush(p, ws, cnt, nxt, ns);
    }
}

// ------------------------------------------------------------ padded frontiers

// The filter of the Gunrock page, step 2: the padded output pad[0][0, L) of
// a push level (one slot per frontier edge: a claimed neighbour or -1) is
// compacted into the next queue through the CTA stage, and the new
// frontier's statistics are counted. Every thread of the grid calls it.
template <typename RowT>
__device__ void filter_padded(const Params<RowT>& p, unsigned long long L, const Smem<RowT>& sm,
                              SmemScalars& ss, LevelSlot* nxt, int qsel, Tally& t)
{
    const int32_t* in = p.pad[0];
    const unsigned long long bd = blockDim.x;
    const unsigned long long stride = (unsigned long long)gridDim.x * bd;
    for (unsigned long long base = blockIdx.x * bd; base < L; base += stride) {
        const unsigned long long i = base + threadIdx.x;
        const int32_t v = i < L ? ldcg(in + i) : -1;
        RowT b = 0, deg = 0;
        if (v >= 0) {
            b = p.row_ptr[v];
            deg = p.row_ptr[v + 1] - b;
            t.found += 1;
            t.edges += (unsigned long long)deg;
            t.maxdeg = (unsigned long long)deg > t.maxdeg ? (unsigned long long)deg : t.maxdeg;
        }
        stage_push(p, sm, ss, nxt, qsel, v, b, deg, v >= 0 && deg > 0);
        if (__syncthreads_or(ss.stage_n > sm.cap / 2))
            stage_flush(p, sm, ss, nxt, qsel);
    }
    stage_flush(p, sm, ss, nxt, qsel);
}

// A push level without the filter: the frontier is the padded array
// pad[k & 1][0, L) of the previous level, sentinels included, and each
// thread takes one slot and walks its vertex's whole row (the thread-mapped
// advance of the Gunrock page, step 3). A warp reserves the output slots of
// its 32 rows with one atomic add on the next level's length (the edge bits
// of nxt->qpack); every entry of a row writes its slot of pad[(k + 1) & 1],
// the claimed neighbour or -1.
template <typename RowT>
__device__ void push_padded(const Params<RowT>& p, int k, unsigned long long L, LevelSlot* nxt,
                            Tally& t, bool pre)
{
    const int32_t* in = p.pad[k & 1];
    int32_t* out = p.pad[(k + 1) & 1];
    const int lane = threadIdx.x & 31;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    const unsigned long long emask = (1ull << p.eb) - 1ull;
    for (unsigned long long i0 = (unsigned long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31u);
         i0 < L; i0 += stride) {
        const unsigned long long i = i0 + lane;
        const int32_t v = i < L ? ldcg(in + i) : -1;
        RowT b = 0, deg = 0;
        if (v >= 0) {
            b = p.row_ptr[v];
            deg = p.row_ptr[v + 1] - b;
        }
        const unsigned long long d = (unsigned long long)deg;
        const unsigned long long inc = warp_inclusive_scan(d);
        const unsigned long long tot = __shfl_sync(kFull, inc, 31);
        unsigned long long base = 0ull;
        if (lane == 31 && tot != 0ull)
            base = atomicAdd(&nxt->qpack, tot) & emask;
        base = __shfl_sync(kFull, base, 31) + inc - d;
        for (RowT j = 0; j < deg; ++j) {
            const int32_t w = p.col[b + j];
            const bool won = claim(p, k, w, v, pre);
            out[base + (unsigned long long)j] = won ? w : -1;
            if (won) {
                const RowT wd = p.row_ptr[w + 1] - p.row_ptr[w];
                t.found += 1;
                t.edges += (unsigned long long)wd;
                t.maxdeg = (unsigned long long)wd > t.maxdeg ? (unsigned long long)wd : t.maxdeg;
            }
        }
    }
}

// ------------------------------------------------------------ S7 pull level

constexpr int kHeadVerts = 4;    // probe tests per lane in flight
constexpr int kPullVerts = 2;    // miss rows per lane in flight
constexpr int kRoundEntries = 4; // entries of a row tested per round (in flight together)
constexpr int kPullRounds = 4;   // rounds before the whole warp takes a row
constexpr int kTailEntries = 1;  // entries per lane per step of the whole-warp row scan
constexpr int kPullList = 1024;  // per-warp list of unvisited vertices
constexpr int kPullWin = 128;    // visited-bitmap words per warp window (4,096 vertices)
// The list grows 32 visited words (up to 1,024 vertices) at a time, and its
// entries are 16-bit offsets within the window.
static_assert(kPullList >= 32 * 32, "one 32-word step must fit an empty list");
static_assert(kPullWin * 32 <= 65536, "window offsets must fit 16 bits");

// Pull level over the frontier bitmap fb[k & 1] (bit u set iff u is in F_k).
// Every warp owns a contiguous range of visited-bitmap words and walks it in
// windows of kPullWin words: it stages the window's visited words in shared
// memory, compacts the unvisited vertices into a per-warp list (processing
// the list whenever the next 32 words would overflow it), and at the window's
// end writes the window's visited and next-frontier words. A sparse level
// (few unvisited vertices) thus costs one list pass per window, not one per
// 32 words.
//
// A list pass (pull_list) first tests, for every entry, the probe neighbour
// stored in the probe array (read nearly sequentially, with the flag that
// marks a one-entry row; kHeadVerts entries per lane in flight, so their
// probe -> frontier-bitmap chains overlap); most rows found by a wide pull
// level resolve there, never touch row_ptr or col, and need no parent
// store. Rows that miss are scanned in CSR order, kRoundEntries entries per
// round and kPullVerts rows per lane; one still unresolved after kPullRounds
// rounds is scanned by the whole warp, 32 * kTailEntries entries per step,
// and the first hit in CSR order gives the first frontier neighbour, as the
// per-lane scan does. The parent is thus the probe neighbour when it is
// in F_k, else the first neighbour in F_k in CSR order. The warp is the only
// writer of its words of the visited and next-frontier bitmaps, so no global
// atomics are needed for them (a level that starts with at most emit_max
// unvisited vertices also appends its finds to the next queue, one packed
// atomic per window), and every next-frontier word is written, so that bitmap
// needs no clearing.

// x is found at level k with parent par. A parent that is x's probe
// neighbour is only flagged in the hop code (the end-of-search pass writes
// it); any other parent is stored now.
template <typename RowT>
__device__ __forceinline__ void pull_resolve(const Params<RowT>& p, int k, Tally& t,
                                             uint32_t* wfound, int w0, int32_t x, int32_t par,
                                             bool par_is_probe)
{
    const bool flag = par_is_probe && p.defer_parent;
    record_dist(p, x, k + 1, flag);
    if (p.parent != nullptr && !flag)
        p.parent[x] = par;
    atomicOr(&wfound[(x >> 5) - w0], 1u << (x & 31));
    t.found += 1;
}

// The finds of one window (wfound, words a .. a + nwin) appended to the queue
// of F_{k+1} (slot nxt, queue (k + 1) & 1). They are gathered as 16-bit
// window offsets into the warp's list (free once the window's passes are
// done), at most kPullList at a time; a first pass loads their rows' starts
// and degrees with kEmitBatch loads per lane in flight and sums them, one
// packed atomic reserves the list's slots and edge range, and a second pass
// (its loads served by L1) writes the entries. Slot order and degree-prefix
// order agree as in the CTA stage.
constexpr int kEmitBatch = 4;

template <typename RowT>
__device__ void emit_window(const Params<RowT>& p, int k, LevelSlot* nxt,
                            const uint32_t* wfound, int a, int nwin, uint16_t* wlist)
{
    const int lane = threadIdx.x & 31;
    uint32_t fw[kPullWin / 32];
    int cnt = 0;
#pragma unroll
    for (int jj = 0; jj < kPullWin / 32; ++jj) {
        const int i = 32 * jj + lane;
        fw[jj] = i < nwin ? wfound[i] : 0u;
        cnt += __popc(fw[jj]);
    }
    const int incl = warp_inclusive_scan(cnt);
    const int tot = __shfl_sync(kFull, incl, 31);
    const int32_t v0 = a << 5;
    const int qs = (k + 1) & 1;
    const unsigned long long emask = (1ull << p.eb) - 1ull;
    for (int b0 = 0; b0 < tot; b0 += kPullList) {
        int pos = incl - cnt;
        __syncwarp();
#pragma unroll
        for (int jj = 0; jj < kPullWin / 32; ++jj) {
            uint32_t f = fw[jj];
            while (f != 0u) {
                const int bit = __ffs(f) - 1;
                f &= f - 1u;
                if (pos >= b0 && pos < b0 + kPullList)
                    wlist[pos - b0] = (uint16_t)(((32 * jj + lane) << 5) + bit);
                ++pos;
            }
        }
        __syncwarp();
        const int m = min(kPullList, tot - b0);
        unsigned long long edges = 0ull, md = 0ull;
        int taken = 0;
        for (int j0 = 0; j0 < m; j0 += 32 * kEmitBatch) {
            RowT bb[kEmitBatch], ee[kEmitBatch];
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u) {
                const int j = j0 + 32 * u + lane;
                const int32_t v = j < m ? v0 + (int32_t)wlist[j] : -1;
                bb[u] = v >= 0 ? p.row_ptr[v] : (RowT)0;
                ee[u] = v >= 0 ? p.row_ptr[v + 1] : (RowT)0;
            }
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u) {
                const unsigned long long deg = (unsigned long long)(ee[u] - bb[u]);
                if (deg > 0ull) {
                    edges += deg;
                    md = deg > md ? deg : md;
                    ++taken;
                }
            }
        }
        edges = warp_sum(edges);
        md = warp_max(md);
        taken = warp_sum(taken);
        unsigned long long old = 0ull;
        if (lane == 0 && taken > 0) {
            old = atomicAdd(&nxt->qpack, ((unsigned long long)taken << p.eb) | edges);
            atomicMax(&nxt->maxdeg, md);
        }
        old = __shfl_sync(kFull, old, 0);
        unsigned long long slot = old >> p.eb, run = old & emask;
        for (int j0 = 0; j0 < m; j0 += 32) {
            const int j = j0 + lane;
            const int32_t v = j < m ? v0 + (int32_t)wlist[j] : -1;
            const RowT b = v >= 0 ? p.row_ptr[v] : (RowT)0;
            const RowT deg = v >= 0 ? p.row_ptr[v + 1] - b : (RowT)0;
            const bool take = deg > 0;
            const unsigned tm = __ballot_sync(kFull, take);
            const unsigned long long d = take ? (unsigned long long)deg : 0ull;
            const unsigned long long inc = warp_inclusive_scan(d);
            if (take) {
                const unsigned long long sl = slot + __popc(tm & ((1u << lane) - 1u));
                p.qv[qs][sl] = v;
                p.qbeg[qs][sl] = b;
                p.qoff[qs][sl] = (RowT)(run + inc - d);
            }
            slot += __popc(tm);
            run += __shfl_sync(kFull, inc, 31);
        }
    }
    __syncwarp();
}

// One pass over the warp's list wlist[0, total) of unvisited vertices, all in
// the window whose first visited-bitmap word is w0, each held as its offset
// from the window's first vertex 32 * w0 (a window spans 32 * kPullWin
// vertices, so 16 bits): phase 1 (probe tests) then phase 2 (row scans of
// the misses). Found vertices get their bit in wfound (indexed by word - w0).
template <typename RowT>
__device__ void pull_list(const Params<RowT>& p, int k, Tally& t, uint16_t* wlist, int total,
                          uint32_t* wfound, int w0)
{
    const uint32_t* fcur = p.fb[k & 1];
    const int lane = threadIdx.x & 31;
    const int32_t v0 = w0 << 5;
    // Phase 1: every list entry's probe neighbour, kHeadVerts per lane in
    // flight. Hits resolve here. A miss whose row is that one neighbour is
    // not found at this level (its one edge counts toward the unvisited
    // edges); any other miss is written back to the front of the list
    // (never past an entry already read), so phase 2 scans rows for those
    // misses only and no lane of a round idles behind a hit.
    int nmiss = 0;
    for (int base = 0; base < total; base += 32 * kHeadVerts) {
        int32_t hv[kHeadVerts];
        uint32_t hc[kHeadVerts];
        uint32_t hf[kHeadVerts];
#pragma unroll
        for (int b = 0; b < kHeadVerts; ++b) {
            const int j = base + b * 32 + lane;
            hv[b] = j < total ? v0 + (int32_t)wlist[j] : -1;
            hc[b] = hv[b] >= 0 ? __ldg(p.probe + hv[b]) : kProbeNone;
        }
#pragma unroll
        for (int b = 0; b < kHeadVerts; ++b) {
            const uint32_t u = hc[b] & kProbeNone;
            hf[b] = u != kProbeNone ? ldcg(fcur + (u >> 5)) : 0u;
        }
        __syncwarp();
#pragma unroll
        for (int b = 0; b < kHeadVerts; ++b) {
            const uint32_t u = hc[b] & kProbeNone;
            const bool hit = u != kProbeNone && ((hf[b] >> (u & 31)) & 1u);
            if (hit)
                pull_resolve(p, k, t, wfound, w0, hv[b], (int32_t)u, true);
            else if (hv[b] >= 0 && (hc[b] >> 31))
                t.edges += 1ull;  // the only edge leads outside F_k
            const bool miss = hv[b] >= 0 && !hit && u != kProbeNone && !(hc[b] >> 31);
            const unsigned mm = __ballot_sync(kFull, miss);
            if (miss)
                wlist[nmiss + __popc(mm & ((1u << lane) - 1u))] = (uint16_t)(hv[b] - v0);
            nmiss += __popc(mm);
        }
        __syncwarp();
    }
    // Phase 2: the misses' rows in CSR order, kRoundEntries entries per round.
    for (int base = 0; base < nmiss; base += 32 * kPullVerts) {
        int32_t v[kPullVerts], par[kPullVerts], deg[kPullVerts];
        RowT cur[kPullVerts], end[kPullVerts];
#pragma unroll
        for (int b = 0; b < kPullVerts; ++b) {
            const int j = base + b * 32 + lane;
            v[b] = j < nmiss ? v0 + (int32_t)wlist[j] : -1;
            par[b] = -1;
            cur[b] = 0;
            end[b] = 0;
            deg[b] = 0;
            if (v[b] >= 0) {
                cur[b] = p.row_ptr[v[b]];
                end[b] = p.row_ptr[v[b] + 1];
                deg[b] = (int32_t)(end[b] - cur[b]);
            }
        }
        for (int round = 0; round < kPullRounds; ++round) {
            bool any = false;
#pragma unroll
            for (int b = 0; b < kPullVerts; ++b)
                any |= par[b] < 0 && cur[b] < end[b];
            if (!__any_sync(kFull, any))
                break;
            int32_t u[kPullVerts][kRoundEntries];
            uint32_t f[kPullVerts][kRoundEntries];
#pragma unroll
            for (int b = 0; b < kPullVerts; ++b) {
                const bool open = par[b] < 0 && cur[b] < end[b];
#pragma unroll
                for (int j = 0; j < kRoundEntries; ++j)
                    u[b][j] = open && cur[b] + j < end[b] ? p.col[cur[b] + j] : -1;
            }
#pragma unroll
            for (int b = 0; b < kPullVerts; ++b)
#pragma unroll
                for (int j = 0; j < kRoundEntries; ++j)
                    f[b][j] = u[b][j] >= 0 ? ldcg(fcur + (u[b][j] >> 5)) : 0u;
            bool more = false;
#pragma unroll
            for (int b = 0; b < kPullVerts; ++b) {
                if (u[b][0] >= 0) {
                    // the first of the round's entries (in CSR order) that hit
#pragma unroll
                    for (int j = kRoundEntries - 1; j >= 0; --j)
                        if (u[b][j] >= 0 && ((f[b][j] >> (u[b][j] & 31)) & 1u))
                            par[b] = u[b][j];
                    if (par[b] < 0)
                        cur[b] += kRoundEntries;
                }
                more |= par[b] < 0 && cur[b] < end[b];
            }
            if (!__any_sync(kFull, more))
                break;
        }
        // Rows still open: the whole warp scans kTailEntries * 32 entries per
        // step, entry q + 32 j + lane in lane `lane` (coalesced col loads, all
        // col and frontier-bitmap loads of a step in flight together); the
        // first hit in CSR order is the lowest lane of the lowest j that hit.
#pragma unroll
        for (int b = 0; b < kPullVerts; ++b) {
            unsigned mm = __ballot_sync(kFull, par[b] < 0 && cur[b] < end[b]);
            while (mm) {
                const int src = __ffs(mm) - 1;
                mm &= mm - 1;
                const RowT cp = __shfl_sync(kFull, cur[b], src);
                const RowT ce = __shfl_sync(kFull, end[b], src);
                int32_t hitv = -1;
                for (RowT q = cp; q < ce && hitv < 0; q += 32 * kTailEntries) {
                    int32_t u[kTailEntries];
                    uint32_t f[kTailEntries];
#pragma unroll
                    for (int j = 0; j < kTailEntries; ++j) {
                        const RowT e = q + 32 * j + lane;
                        u[j] = e < ce ? p.col[e] : -1;
                    }
#pragma unroll
                    for (int j = 0; j < kTailEntries; ++j)
                        f[j] = u[j] >= 0 ? ldcg(fcur + (u[j] >> 5)) : 0u;
#pragma unroll
                    for (int j = 0; j < kTailEntries; ++j) {
                        const bool hit = u[j] >= 0 && ((f[j] >> (u[j] & 31)) & 1u);
                        const unsigned hm = __ballot_sync(kFull, hit);
                        if (hm != 0u && hitv < 0)
                            hitv = __shfl_sync(kFull, u[j], __ffs(hm) - 1);
                    }
                }
                if (lane == src) {
                    par[b] = hitv;
                    cur[b] = ce;
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kPullVerts; ++b) {
            if (par[b] >= 0)
                pull_resolve(p, k, t, wfound, w0, v[b], par[b], false);
            else if (v[b] >= 0)
                t.edges += (unsigned long long)deg[b];  // stays unvisited
        }
    }
}

template <typename RowT>
__device__ void pull_level(const Params<RowT>& p, int k, Tally& t, uint16_t* wlist,
                           uint32_t* wfound, uint32_t* wvis, LevelSlot* emit)
{
    uint32_t* fnext = p.fb[(k + 1) & 1];
    const int lane = threadIdx.x & 31;
    const long long gwarp = (long long)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const long long nwarps = (long long)((gridDim.x * blockDim.x) >> 5);
    const int wlo = (int)((long long)p.words * gwarp / nwarps);
    const int whi = (int)((long long)p.words * (gwarp + 1) / nwarps);
    for (int a = wlo; a < whi; a += kPullWin) {
        const int nwin = min(kPullWin, whi - a);
        // Stage the window's visited words (padding words read as visited).
#pragma unroll
        for (int j = 0; j < kPullWin / 32; ++j) {
            const int i = 32 * j + lane;
            wvis[i] = i < nwin ? ldcg(p.visited + a + i) : kFull;
            wfound[i] = 0u;
        }
        __syncwarp();
        // Compact 32 words at a time; a step whose vertices would overflow
        // the list runs the pass on the list first. One call site.
        int j = 0, nl = 0;
        for (;;) {
            bool run = j >= kPullWin / 32;
            if (!run) {
                const uint32_t todo = ~wvis[32 * j + lane];
                const int cnt = __popc(todo);
                const int incl = warp_inclusive_scan(cnt);
                const int tot = __shfl_sync(kFull, incl, 31);
                if (nl + tot <= kPullList) {
                    int pos = nl + incl - cnt;
                    uint32_t m = todo;
                    const int w = a + 32 * j + lane;
                    while (m) {
                        const int bit = __ffs(m) - 1;
                        m &= m - 1;
                        wlist[pos++] = (uint16_t)(((w - a) << 5) + bit);
                    }
                    nl += tot;
                    ++j;
                    continue;
                }
                run = true;
            }
            __syncwarp();
            if (nl > 0)
                pull_list(p, k, t, wlist, nl, wfound, a);
            __syncwarp();
            nl = 0;
            if (j >= kPullWin / 32)
                break;
        }
        // Few unvisited vertices at the level's start: the window's finds also
        // go to the next queue.
        if (emit != nullptr)
            emit_window(p, k, emit, wfound, a, nwin, wlist);
#pragma unroll
        for (int jj = 0; jj < kPullWin / 32; ++jj) {
            const int i = 32 * jj + lane;
            if (i < nwin) {
                const uint32_t f = wfound[i];
                if (f != 0u)
                    __stcg(p.visited + a + i, wvis[i] | f);
                __stcg(fnext + a + i, f);
            }
        }
        __syncwarp();
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

// F_k from the hop codes: bit v of fb[k & 1] is set iff v's code holds
// distance k (every vertex of F_k was recorded with that code by level k - 1;
// codes are exact below kHopDirect). One coalesced pass that writes every
// word, for large queues where an atomic per queued vertex costs more than
// reading a byte per vertex; it also needs no clearing pass before it.
__device__ __forceinline__ uint32_t hop_match4(uint32_t x, uint32_t code4)
{
    const uint32_t m = __vcmpeq4(x & 0x7f7f7f7fu, code4);  // 0xff per matching byte
    return ((m >> 7) & 1u) | ((m >> 14) & 2u) | ((m >> 21) & 4u) | ((m >> 28) & 8u);
}

template <typename RowT>
__device__ void hop_to_bitmap(const Params<RowT>& p, int k)
{
    uint32_t* f = p.fb[k & 1];
    const uint32_t code = (uint32_t)(k + 1);
    const uint32_t code4 = code * 0x01010101u;
    const int full = p.n >> 5;  // words whose 32 vertices all exist
    const uint4* h4 = reinterpret_cast<const uint4*>(p.hop);  // 256-byte aligned
    const int stride = gridDim.x * blockDim.x;
    for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < p.words; w += stride) {
        uint32_t bits = 0u;
        if (w < full) {
            const uint4 a = ldcg(h4 + 2 * w);
            const uint4 b = ldcg(h4 + 2 * w + 1);
            bits = hop_match4(a.x, code4) | hop_match4(a.y, code4) << 4 |
                   hop_match4(a.z, code4) << 8 | hop_match4(a.w, code4) << 12 |
                   hop_match4(b.x, code4) << 16 | hop_match4(b.y, code4) << 20 |
                   hop_match4(b.z, code4) << 24 | hop_match4(b.w, code4) << 28;
        } else {
            for (int i = 0; i < 32; ++i) {
                const int v = (w << 5) + i;
                if (v < p.n && (uint32_t)(ldcg(p.hop + v) & 0x7f) == code)
                    bits |= 1u << i;
            }
        }
        __stcg(f + w, bits);
    }
}

// F_k from bitmap to queue (with row starts and the degree prefix), through
// the same stage as push levels; counts go to the current slot's qpack, and
// the largest degree of F_k (which a pull level does not count) to its
// maxdeg.
template <typename RowT>
__device__ void bitmap_to_queue(const Params<RowT>& p, int k, const Smem<RowT>& sm,
                                SmemScalars& ss, LevelSlot* cur)
{
    unsigned long long md = 0ull;
    constexpr int kBatch = 4;  // bitmap words per thread loaded together
    const uint32_t* f = p.fb[k & 1];
    const int sel = k & 1;
    const int bd = blockDim.x;
    const int stride = gridDim.x * bd;
    for (int base = blockIdx.x * bd; base < p.words; base += stride * kBatch) {
        uint32_t bits[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int w = base + i * stride + threadIdx.x;
            bits[i] = w < p.words ? ldcg(f + w) : 0u;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int w = base + i * stride + threadIdx.x;
            uint32_t b = bits[i];
            while (b) {
                const int bit = __ffs(b) - 1;
                b &= b - 1;
                const int32_t v = (w << 5) + bit;
                const RowT rb = p.row_ptr[v];
                const RowT deg = p.row_ptr[v + 1] - rb;
                md = (unsigned long long)deg > md ? (unsigned long long)deg : md;
                stage_push(p, sm, ss, cur, sel, v, rb, deg, deg > 0);
            }
        }
        if (__syncthreads_or(ss.stage_n > sm.cap / 2))
            stage_flush(p, sm, ss, cur, sel);
    }
    stage_flush(p, sm, ss, cur, sel);
    md = warp_max(md);
    if ((threadIdx.x & 31) == 0 && md != 0ull)
        atomicMax(&cur->maxdeg, md);
}

// S2: the direction of level k. Only symmetric graphs may pull. In AUTO
// mode this is the direction-optimising rule with exact device counts: after
// a push level, pull once the frontier's edges m_F exceed m_U / pull_alpha
// (m_U = edges of the vertices not reached yet); after a pull level, return
// to push once |F| falls below N / push_beta (N = vertices of nonzero
// degree). The pages' rule compares |F| * average degree with |U| (PMPP
// ch. 15 notes, section 15.7); exact m_F and m_U make the comparison robust to
// frontiers whose degrees are far from the average (hub-heavy levels).
template <typename RowT>
__device__ __forceinline__ int choose_direction(const Params<RowT>& p, int prev_dir, long long F,
                                                long long mF, long long mU, long long nonisolated)
{
    if (!p.symmetric || p.direction == BFS_CSR_DIR_PUSH ||
        p.frontier_output == BFS_CSR_FRONTIER_PADDED)
        return BFS_CSR_DIR_PUSH;
    if (p.direction == BFS_CSR_DIR_PULL)
        return BFS_CSR_DIR_PULL;
    if (prev_dir == BFS_CSR_DIR_PULL && p.push_beta > 0)
        return (double)F * (double)p.push_beta < (double)nonisolated ? BFS_CSR_DIR_PUSH
                                                                      : BFS_CSR_DIR_PULL;
    return (double)mF * p.pull_alpha > (double)mU ? BFS_CSR_DIR_PULL : BFS_CSR_DIR_PUSH;
}

// ------------------------------------------------------------ S9 narrow levels

constexpr int kSoloMaxLevels = 4096;  // levels per single-CTA session

// Narrow push levels on CTA 0 alone (the other CTAs wait at the level's grid
// barrier). The frontier lives in shared memory (vertex, row start, degree
// prefix); each level is an edge-balanced pass of at most TILE edges with
// block barriers only, so the per-level cost is the chain of dependent loads
// (col, visited atomic, row offsets of the winners) instead of a grid-wide
// barrier. The session ends at the first level that is empty, too wide, due
// for a pull, at the depth bound, or after kSoloMaxLevels levels; that level
// k' is published to the slots and queues exactly as a grid level would have
// produced it, and its number is left in ctl->solo_resume.
template <typename RowT>
__device__ void solo_levels(const Params<RowT>& p, int k, int qn, RowT qm, long long F, long long U,
                            long long mU, unsigned long long maxdeg, const Smem<RowT>& sm,
                            SmemScalars& ss, unsigned long long bar_base, long long nonisolated)
{
    const int bd = blockDim.x;
    const int tid = threadIdx.x;
    int32_t* cv = sm.wu;
    RowT* cb = sm.wbeg;
    RowT* co = sm.woff;
    {
        const int cs = k & 1;
        for (int i = tid; i < qn; i += bd) {
            cv[i] = ldcg(p.qv[cs] + i);
            cb[i] = ldcg(p.qbeg[cs] + i);
            co[i] = ldcg(p.qoff[cs] + i);
        }
        if (tid == 0) {
            co[qn] = qm;
            ss.stage_n = 0;
            ss.solo_found = 0ull;
            ss.solo_edges = 0ull;
            ss.solo_maxdeg = 0ull;
        }
    }
    __syncthreads();
    int j = k;
    long long Fj = F;
    long long Uj = U;               // unvisited at level j's start
    long long mUj = mU;             // their edges
    unsigned long long mdj = maxdeg;
    for (;;) {
        const unsigned long long t0 = tid == 0 ? global_timer_ns() : 0ull;
        const RowT M = co[qn];
        // expand in rounds of kItems edges per thread, the loads of a round
        // batched; M is at most the stage capacity, so every winner fits it
        unsigned long long f_loc = 0ull, e_loc = 0ull, m_loc = 0ull;
        for (RowT r0 = 0; r0 < M; r0 += (RowT)(kItems * bd)) {
            int32_t vv[kItems], uu[kItems];
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const RowT e = r0 + (RowT)(it * bd + tid);
                vv[it] = -1;
                uu[it] = 0;
                if (e < M) {
                    int lo = 0, hi = qn;
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (co[mid] <= e)
                            lo = mid;
                        else
                            hi = mid;
                    }
                    uu[it] = cv[lo];
                    vv[it] = p.col[cb[lo] + (e - co[lo])];
                }
            }
            bool won[kItems];
            claim_batch(p, j, vv, uu, false, won);
            RowT wb[kItems], we[kItems];
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                wb[it] = 0;
                we[it] = 0;
                if (won[it]) {
                    wb[it] = p.row_ptr[vv[it]];
                    we[it] = p.row_ptr[vv[it] + 1];
                }
            }
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const RowT deg = we[it] - wb[it];
                if (won[it]) {
                    f_loc += 1ull;
                    e_loc += (unsigned long long)deg;
                    m_loc = (unsigned long long)deg > m_loc ? (unsigned long long)deg : m_loc;
                }
                stage_push(p, sm, ss, nullptr, 0, vv[it], wb[it], deg, won[it] && deg > 0);
            }
        }
        // Tallies per warp, then one shared atomic per warp and counter; the
        // level has at most one stage of winners, so no slot overflows.
        f_loc = warp_sum(f_loc);
        e_loc = warp_sum(e_loc);
        m_loc = warp_max(m_loc);
        if ((tid & 31) == 0 && f_loc != 0ull) {
            atomicAdd(&ss.solo_found, f_loc);
            atomicAdd(&ss.solo_edges, e_loc);
            atomicMax(&ss.solo_maxdeg, m_loc);
        }
        __syncthreads();
        const long long Fn = (long long)ss.solo_found;
        const unsigned long long en = ss.solo_edges;
        const unsigned long long mdn = ss.solo_maxdeg;
        const int nq = ss.stage_n;
        if (tid == 0 && j < p.stats_cap) {
            bfs_csr_level_stat st;
            st.level = j;
            st.direction = BFS_CSR_DIR_PUSH;
            st.advance = BFS_CSR_ADV_SINGLE_CTA;
            st.reserved = 0;
            st.frontier = Fj;
            st.frontier_edges = (long long)M;
            st.unvisited = Uj;
            st.max_degree = (long long)mdj;
            st.t_start_ns = (long long)t0;
            st.t_work_ns = (long long)global_timer_ns();
            p.stats[j] = st;
        }
        const long long Un = Uj - Fn;   // unvisited at level j + 1's start
        const long long mUn = mUj - (long long)en;
        bool stop = Fn == 0 || (p.max_depth >= 0 && j + 1 >= p.max_depth) ||
                    (long long)en > (long long)p.narrow_max || nq >= sm.wcap ||
                    j + 1 - k >= kSoloMaxLevels;
        if (!stop && choose_direction(p, BFS_CSR_DIR_PUSH, Fn, (long long)en, mUn, nonisolated) !=
                         BFS_CSR_DIR_PUSH)
            stop = true;
        if (stop) {
            // Publish F_{j+1}: its queue (staged), its counters, and the
            // state the grid level j + 1 expects to find. The slots written
            // here may be the ones the other CTAs read at level k's start, so
            // first wait (bounded) until every other CTA has arrived at level
            // k's barrier, which each does right after those reads.
            const int jn = j + 1;
            if (tid == 0) {
                const unsigned long long want = bar_base + gridDim.x - 1;
                const unsigned long long t0w = global_timer_ns();
                unsigned int spins = 0;
                while (ld_acquire_u64(&p.ctl->bar) < want) {
                    if ((++spins & 63u) == 0u &&
                        (global_timer_ns() - t0w > (unsigned long long)p.timeout_ns ||
                         spins > (1u << 30))) {
                        atomicCAS(&p.ctl->status, BFS_CSR_OK, BFS_CSR_ETIMEOUT);
                        break;
                    }
                }
            }
            __syncthreads();
            if (tid == 0) {
                LevelSlot* sn = &p.ctl->slot[jn & 3];
                LevelSlot* sp = &p.ctl->slot[j & 3];
                LevelSlot* sa = &p.ctl->slot[(jn + 1) & 3];
                sn->qpack = 0ull;
                sn->found = (unsigned long long)Fn;
                sn->fedges = en;
                sn->maxdeg = mdn;
                sp->unvisited = Uj;
                sp->unvisited_edges = mUj;
                sp->dir = BFS_CSR_DIR_PUSH;
                sp->adv = BFS_CSR_ADV_SINGLE_CTA;
                sa->qpack = 0ull;
                sa->found = 0ull;
                sa->fedges = 0ull;
                sa->maxdeg = 0ull;
                sa->work_next = 0u;
                sn->work_next = 0u;
                p.ctl->solo_resume = jn;
                if (jn < p.stats_cap)
                    p.stats[jn].t_work_ns = 0;
            }
            stage_flush(p, sm, ss, &p.ctl->slot[jn & 3], jn & 1);
            return;
        }
        // F_{j+1} becomes the current frontier (degree prefix by block scan).
        {
            const int per = (nq + bd - 1) / bd;
            const int lo = min(tid * per, nq), hi = min(lo + per, nq);
            long long sum = 0;
            for (int i = lo; i < hi; ++i)
                sum += (long long)sm.sd[i];
            long long total;
            const long long excl = block_exclusive_scan(sum, &total, ss.tmp_ll);
            RowT run = (RowT)excl;
            for (int i = lo; i < hi; ++i) {
                cv[i] = sm.sv[i];
                cb[i] = sm.sb[i];
                co[i] = run;
                run += sm.sd[i];
            }
            if (tid == 0) {
                co[nq] = (RowT)total;
                ss.stage_n = 0;
                ss.solo_found = 0ull;
                ss.solo_edges = 0ull;
                ss.solo_maxdeg = 0ull;
            }
        }
        __syncthreads();
        qn = nq;
        Fj = Fn;
        Uj = Un;
        mUj = mUn;
        mdj = mdn;
        ++j;
    }
}

// ------------------------------------------------------------ S10 output

// dist and parent from the hop codes, once the search has ended. A warp
// converts 1,024 consecutive vertices per step: lane l reads the 4 codes of
// vertices base + 128 q + 4 l (q = 0..7) as one word each and writes their
// distances and parents as one 16-byte store each, so every store
// instruction of the warp covers 512 contiguous bytes and all eight code
// loads are in flight together. With defer_parent the parents are written
// the same way: those of flagged codes come from probe[] (four at a time,
// 16-byte loads), a reached vertex without the flag kept the parent its
// discovery stored, an unreached one gets -1. Codes of kHopFar keep the
// distance their discovery wrote to dist.
__device__ __forceinline__ int32_t hop_to_dist(uint32_t c, const int32_t* dist, int64_t v)
{
    const uint32_t d = c & 0x7fu;
    return d == 0u ? -1 : (d == kHopFar ? ldcg(dist + v) : (int32_t)d - 1);
}

__device__ __forceinline__ int32_t hop_to_parent(uint32_t c, uint32_t probe, const int32_t* parent,
                                                 int64_t v)
{
    if ((c & 0x7fu) == 0u)
        return -1;
    return (c & kHopProbe) ? (int32_t)(probe & kProbeNone) : ldcg(parent + v);
}

template <typename RowT>
__device__ void write_outputs(const Params<RowT>& p)
{
    constexpr int kQ = 8;
    const int64_t n = p.n;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t* h4 = reinterpret_cast<const uint32_t*>(p.hop);  // 16-byte aligned
    const bool vec = p.vec_out != 0;
    const bool par = p.parent != nullptr && p.defer_parent;
    const int64_t nfull = vec ? n / (128 * kQ) : 0;   // steps with every vertex < n
    for (int64_t st = gw; st < nfull; st += nw) {
        const int64_t base = st * 128 * kQ;
        uint32_t c[kQ];
#pragma unroll
        for (int q = 0; q < kQ; ++q)
            c[q] = ldcg(h4 + ((base + 128 * q) >> 2) + lane);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const int64_t v = base + 128 * q + 4 * lane;
            int4 o;
            o.x = hop_to_dist(c[q] & 0xffu, p.dist, v);
            o.y = hop_to_dist((c[q] >> 8) & 0xffu, p.dist, v + 1);
            o.z = hop_to_dist((c[q] >> 16) & 0xffu, p.dist, v + 2);
            o.w = hop_to_dist(c[q] >> 24, p.dist, v + 3);
            *reinterpret_cast<int4*>(p.dist + v) = o;
        }
        if (par) {
            uint4 pr[kQ];
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                const int64_t v = base + 128 * q + 4 * lane;
                pr[q] = (c[q] & 0x80808080u) ? __ldg(reinterpret_cast<const uint4*>(p.probe + v))
                                             : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                const int64_t v = base + 128 * q + 4 * lane;
                int4 o;
                o.x = hop_to_parent(c[q] & 0xffu, pr[q].x, p.parent, v);
                o.y = hop_to_parent((c[q] >> 8) & 0xffu, pr[q].y, p.parent, v + 1);
                o.z = hop_to_parent((c[q] >> 16) & 0xffu, pr[q].z, p.parent, v + 2);
                o.w = hop_to_parent(c[q] >> 24, pr[q].w, p.parent, v + 3);
                *reinterpret_cast<int4*>(p.parent + v) = o;
            }
        }
    }
    // The rest (or everything when the outputs are not 16-byte aligned), one
    // vertex per thread.
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = nfull * 128 * kQ + tid; v < n; v += stride) {
        const uint32_t c = ldcg(p.hop + v);
        p.dist[v] = hop_to_dist(c, p.dist, v);
        if (par)
            p.parent[v] = hop_to_parent(c, (c & kHopProbe) ? __ldg(p.probe + v) : 0u, p.parent, v);
    }
}

// ------------------------------------------------------------ kernels

// Dynamic shared memory: the compaction stage (row starts, degrees, vertices)
// and, after it, one region used either as the single-CTA levels' frontier
// (offsets, row starts, vertices) or as the binned advance's CTA-per-vertex
// list; pull levels reuse the whole buffer for their per-warp lists and the
// warp-level merge path for its per-warp stages.
template <typename RowT>
__device__ __forceinline__ Smem<RowT> carve_smem(unsigned char* raw, int bd)
{
    Smem<RowT> sm;
    unsigned char* q = raw;
    sm.cap = stage_cap<RowT>(bd);
    sm.wcap = window_cap<RowT>(bd) + 1;
    sm.sb = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.cap;
    sm.sd = reinterpret_cast<int32_t*>(q); q += sizeof(int32_t) * sm.cap;
    sm.sv = reinterpret_cast<int32_t*>(q); q += sizeof(int32_t) * sm.cap;
    unsigned char* x = q;
    sm.woff = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.wcap;
    sm.wbeg = reinterpret_cast<RowT*>(q); q += sizeof(RowT) * sm.wcap;
    sm.wu = reinterpret_cast<int32_t*>(q);
    sm.lb = reinterpret_cast<RowT*>(x);
    sm.ld = sm.lb + bd;
    sm.lu = reinterpret_cast<int32_t*>(sm.ld + bd);
    return sm;
}

template <typename RowT>
__host__ __device__ inline size_t level_smem_bytes(int bd)
{
    const size_t scap = (size_t)stage_cap<RowT>(bd), wcap = (size_t)window_cap<RowT>(bd);
    const size_t push = (sizeof(RowT) + 8) * scap + (2 * sizeof(RowT) + 4) * (wcap + 1) + 16;
    const size_t pull = (size_t)(bd / 32) *
                        (kPullList * sizeof(uint16_t) + 2 * kPullWin * sizeof(uint32_t));
    const size_t wstage = (size_t)(bd / 32) * kWarpStage * (sizeof(RowT) + 8);
    const size_t m = push > pull ? push : pull;
    return m > wstage ? m : wstage;
}

// The persistent level loop (S2-S9).
template <typename RowT>
__global__ void __launch_bounds__(level_block<RowT>(), 2) level_kernel(Params<RowT> p)
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
    if (p.stamps != nullptr && k == 0 && blockIdx.x == 0 && threadIdx.x == 0)
        p.stamps[1] = (long long)global_timer_ns();
    const long long nonisolated = ldcg(&p.ctl->nonisolated);
    const bool leader = blockIdx.x == 0 && threadIdx.x == 0;
    bool finished = false;      // this launch saw the search end
    __syncthreads();

    for (;;) {
        LevelSlot* cur = &p.ctl->slot[k & 3];
        LevelSlot* nxt = &p.ctl->slot[(k + 1) & 3];
        const LevelSlot* prv = &p.ctl->slot[(k + 3) & 3];
        // Everything the level start needs, as one batch of independent loads.
        const unsigned long long found = ldcg_u64(&cur->found);
        const unsigned long long fedges = ldcg_u64(&cur->fedges);
        const unsigned long long maxdeg = ldcg_u64(&cur->maxdeg);
        // F_k's queue counter, final here unless this level builds the queue
        // from the frontier bitmap (then it is read again after that pass)
        const unsigned long long qpack0 = ldcg_u64(&cur->qpack);
        const long long uprev = ldcg(&prv->unvisited);
        const long long ueprev = ldcg(&prv->unvisited_edges);
        const int prev_dir = ldcg(&prv->dir);
        const int done = ldcg(&p.ctl->done);
        const int status = ldcg(&p.ctl->status);
        if (done != 0 || status != BFS_CSR_OK) {
            // done may also come from CTA 0 ending the search in this very
            // iteration; the hop codes are final either way.
            finished = done != 0 && status == BFS_CSR_OK;
            break;
        }
        const long long F = (long long)found;
        // m_F: counted directly by a push level; after a pull level, the
        // unvisited edges at its start minus those it left unvisited.
        const long long mF = prev_dir == BFS_CSR_DIR_PULL ? ueprev + (long long)fedges
                                                          : (long long)fedges;
        if (F == 0 || (p.max_depth >= 0 && k >= p.max_depth)) {
            if (leader) {
                const int nl = F == 0 ? k : k + 1;
                const unsigned long long t_end = global_timer_ns();
                if (F != 0 && k < p.stats_cap) {
                    // Depth bound: F_k counts as a level but is not expanded.
                    bfs_csr_level_stat st;
                    st.level = k;
                    st.direction = 0;
                    st.advance = 0;
                    st.reserved = 0;
                    st.frontier = F;
                    st.frontier_edges = mF;
                    st.unvisited = uprev - F;
                    st.max_degree = (long long)maxdeg;
                    st.t_start_ns = (long long)t_end;
                    st.t_work_ns = (long long)t_end;
                    p.stats[k] = st;
                }
                p.ctl->num_levels = nl;
                p.ctl->t_end_ns = t_end;
                if (p.num_levels_out != nullptr)
                    *p.num_levels_out = nl;
                __threadfence();
                p.ctl->done = 1;
            }
            finished = true;
            break;
        }
        if (budget <= 0)
            break;
        const unsigned long long t_level = leader ? global_timer_ns() : 0ull;
        const long long U = uprev - F;
        const long long mU = ueprev - mF;
        const int dir = choose_direction(p, prev_dir, F, mF, mU, nonisolated);
        Tally t = {0ull, 0ull, 0ull};
        int adv = 0;
        unsigned long long md = maxdeg;  // largest degree in F_k (known to push levels)

        // Narrow push level: CTA 0 runs it (and the following narrow ones)
        // alone; everyone meets at the barrier and resumes where it stopped.
        if (dir == BFS_CSR_DIR_PUSH && prev_dir != BFS_CSR_DIR_PULL && p.narrow_max > 0 &&
            p.level_budget == INT_MAX && p.frontier_output == BFS_CSR_FRONTIER_COMPACT) {
            const int qn0 = (int)(qpack0 >> p.eb);
            const long long qm0 = (long long)(qpack0 & ((1ull << p.eb) - 1ull));
            if (qm0 <= (long long)p.narrow_max && qn0 < sm.wcap) {
                if (blockIdx.x == 0)
                    solo_levels(p, k, qn0, (RowT)qm0, F, U, mU, maxdeg, sm, ss, target,
                                nonisolated);
                if (!grid_barrier(p, target)) break;
                k = ldcg(&p.ctl->solo_resume);
                continue;
            }
        }

        if (dir == BFS_CSR_DIR_PULL) {
            if (leader) {
                LevelSlot* z = &p.ctl->slot[(k + 2) & 3];
                z->qpack = 0ull; z->found = 0ull; z->fedges = 0ull; z->maxdeg = 0ull;
                z->work_next = 0u;
                cur->unvisited = U;
                cur->unvisited_edges = mU;
                cur->dir = dir;
                cur->adv = 0;
            }
            if (prev_dir != BFS_CSR_DIR_PULL) {
                const int qn = (int)(qpack0 >> p.eb);
                if (p.defer_dist && k + 1 < kHopDirect && 64ll * qn >= (long long)p.n) {
                    hop_to_bitmap(p, k);
                } else {
                    queue_to_bitmap_clear(p, k);
                    if (!grid_barrier(p, target)) break;
                    queue_to_bitmap_set(p, k, qn);
                }
                if (!grid_barrier(p, target)) break;
            }
            {
                const int wid = threadIdx.x >> 5;
                uint16_t* wlist = reinterpret_cast<uint16_t*>(smem_raw) + wid * kPullList;
                uint32_t* wfound =
                    reinterpret_cast<uint32_t*>(smem_raw + (size_t)(blockDim.x >> 5) * kPullList *
                                                               sizeof(uint16_t)) +
                    wid * 2 * kPullWin;
                pull_level(p, k, t, wlist, wfound, wfound + kPullWin,
                           U <= p.emit_max ? nxt : nullptr);
            }
        } else {
            // After a pull level that started with few unvisited vertices
            // (uprev is that count) the queue of F_k was built as it found
            // them; otherwise it is built from the frontier bitmap now.
            unsigned long long qp = qpack0;
            if (prev_dir == BFS_CSR_DIR_PULL && uprev > p.emit_max) {
                bitmap_to_queue(p, k, sm, ss, cur);
                if (!grid_barrier(p, target)) break;
                md = ldcg_u64(&cur->maxdeg);
                qp = ldcg_u64(&cur->qpack);
            }
            const int qn = (int)(qp >> p.eb);
            const RowT qm = (RowT)(qp & ((1ull << p.eb) - 1ull));
            if (p.frontier_output == BFS_CSR_FRONTIER_PADDED)
                adv = BFS_CSR_ADV_PADDED;
            else if (p.frontier_output == BFS_CSR_FRONTIER_PADDED_FILTER)
                adv = BFS_CSR_ADV_MERGE_PATH;
            else if (p.advance == BFS_CSR_ADV_BINNED)
                adv = BFS_CSR_ADV_BINNED;
            else if (p.advance == BFS_CSR_ADV_MERGE_PATH)
                adv = BFS_CSR_ADV_MERGE_PATH;
            else
                adv = (qn >= p.mp_min_frontier || md >= (unsigned long long)p.binned_max_deg ||
                       (long long)qm >= kMergePathMinAvgDegree * (long long)qn)
                          ? BFS_CSR_ADV_MERGE_PATH : BFS_CSR_ADV_BINNED;
            if (leader) {
                LevelSlot* z = &p.ctl->slot[(k + 2) & 3];
                z->qpack = 0ull; z->found = 0ull; z->fedges = 0ull; z->maxdeg = 0ull;
                z->work_next = 0u;
                cur->unvisited = U;
                cur->unvisited_edges = mU;
                cur->dir = dir;
                cur->adv = adv;
            }
            // The plain pre-load of a target's visited word saves an atomic
            // when most targets are already visited (late, wide levels) and
            // costs a round trip otherwise.
            const bool pre = (long long)qm >= 65536 && 2 * U < nonisolated;
            if (adv == BFS_CSR_ADV_PADDED) {
                // qm is the length of the padded frontier here
                push_padded(p, k, qp & ((1ull << p.eb) - 1ull), nxt, t, pre);
            } else if (adv == BFS_CSR_ADV_MERGE_PATH &&
                       p.frontier_output == BFS_CSR_FRONTIER_COMPACT &&
                       (long long)qm >= kIdsMinEdges) {
                push_warp_mp<RowT, true>(p, k, qn, qm, smem_raw, nxt, t, pre);
                // every winner's id is in wq before its row offsets are read
                if (!grid_barrier(p, target)) break;
                queue_from_ids(p, k, smem_raw, nxt, t);
            } else if (adv == BFS_CSR_ADV_MERGE_PATH) {
                push_warp_mp<RowT, false>(p, k, qn, qm, smem_raw, nxt, t, pre);
                if (p.frontier_output == BFS_CSR_FRONTIER_PADDED_FILTER) {
                    // every slot of the padded output is written before the
                    // filter reads it
                    if (!grid_barrier(p, target)) break;
                    filter_padded(p, (unsigned long long)qm, sm, ss, nxt, (k + 1) & 1, t);
                }
            } else {
                push_binned(p, k, qn, qm, sm, ss, nxt, t, pre);
            }
        }
        // The level's record. Every CTA stamps the end of its share of the
        // work (the latest stamp wins); the next level's stamp is cleared
        // here, before the barrier after which CTAs write it.
        if (threadIdx.x == 0 && k < p.stats_cap)
            atomicMax(reinterpret_cast<unsigned long long*>(&p.stats[k].t_work_ns),
                      global_timer_ns());
        if (leader && k < p.stats_cap) {
            bfs_csr_level_stat* st = &p.stats[k];
            st->level = k;
            st->direction = dir;
            st->advance = adv;
            st->reserved = 0;
            st->frontier = F;
            st->frontier_edges = mF;
            st->unvisited = U;
            st->max_degree = (long long)md;
            st->t_start_ns = (long long)t_level;
            if (k + 1 < p.stats_cap)
                p.stats[k + 1].t_work_ns = 0;
        }
        publish_tally<RowT>(t, nxt, ss, dir == BFS_CSR_DIR_PULL);
        if (!grid_barrier(p, target)) break;
        ++k;
        --budget;
    }

    // S10: every CTA saw the same empty (or depth-bounded) frontier after
    // the last grid barrier, so all hop codes are final.
    if (finished && p.defer_dist)
        write_outputs(p);

    // Leave: the last CTA out resets the barrier for the next launch.
    __syncthreads();
    if (threadIdx.x == 0) {
        if (blockIdx.x == 0)
            p.ctl->level = k;
        __threadfence();
        const unsigned int prev = atomicAdd(&p.ctl->exit_count, 1u);
        if (prev == gridDim.x - 1) {
            if (p.stamps != nullptr && finished)
                p.stamps[2] = (long long)global_timer_ns();
            p.ctl->bar = 0ull;
            p.ctl->exit_count = 0u;
            if (p.graph_cond != 0ull) {
                // The graph's while loop runs another launch until the search
                // has ended or failed. Every launch either runs a level or
                // ends the search, so more than n + 1 launches would mean a
                // fault: it ends the loop with an error instead of spinning.
                bool stop = ldcg(&p.ctl->done) != 0 || ldcg(&p.ctl->status) != BFS_CSR_OK;
                if (!stop && (long long)ldcg(&p.ctl->level) > (long long)p.n + 1) {
                    atomicCAS(&p.ctl->status, BFS_CSR_OK, BFS_CSR_EDEVICE);
                    stop = true;
                }
                if (stop)
                    cudaGraphSetConditional(p.graph_cond, 0u);
            }
            __threadfence();
        }
    }
}

// S1: reset the run state and seed the source. With bitmap discovery the hop
// codes are cleared (source: distance 0) and dist is left to the end of the
// search; so is parent when defer_parent is set (then only parent[source] =
// source is stored). Whatever is not deferred is filled with -1 here (the
// source: distance 0, parent itself).
// visited starts as the dead bitmap (vertices of degree 0 and padding bits
// beyond n) plus the source bit, and slot 0 holds F_0 = {source}.
template <typename RowT>
__global__ void init_kernel(Params<RowT> p, const uint32_t* __restrict__ dead, int32_t source,
                            int use_dead)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int32_t n = p.n;
    const bool fill = !p.defer_dist;
    const bool fill_parent = !p.defer_parent;
    if (p.stamps != nullptr && tid == 0)
        p.stamps[0] = (long long)global_timer_ns();
    if (!fill_parent && p.parent != nullptr && tid == 0)
        p.parent[source] = source;
    int32_t* outs[2] = {fill ? p.dist : nullptr, fill_parent ? p.parent : nullptr};
    const int32_t seed[2] = {0, source};
    for (int o = 0; o < 2; ++o) {
        int32_t* a = outs[o];
        if (a == nullptr)
            continue;
        if ((reinterpret_cast<uintptr_t>(a) & 15u) == 0) {
            const int64_t n4 = n / 4;
            int4* a4 = reinterpret_cast<int4*>(a);
            for (int64_t i = tid; i < n4; i += stride) {
                int4 x = make_int4(-1, -1, -1, -1);
                if (source / 4 == i)
                    (&x.x)[source & 3] = seed[o];
                a4[i] = x;
            }
            for (int64_t i = n4 * 4 + tid; i < n; i += stride)
                a[i] = i == source ? seed[o] : -1;
        } else {
            for (int64_t i = tid; i < n; i += stride)
                a[i] = i == source ? seed[o] : -1;
        }
    }
    if (p.defer_dist) {
        // The hop region is 16-byte aligned and padded to a multiple of 16.
        uint4* h16 = reinterpret_cast<uint4*>(p.hop);
        const int64_t n16 = ((int64_t)n + 15) / 16;
        for (int64_t i = tid; i < n16; i += stride) {
            uint4 z = make_uint4(0u, 0u, 0u, 0u);
            if (source / 16 == i)
                (&z.x)[(source & 15) >> 2] = 1u << (8 * (source & 3));
            h16[i] = z;
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
            c->slot[s].unvisited_edges = 0;
            c->slot[s].dir = BFS_CSR_DIR_PUSH;
            c->slot[s].adv = 0;
            c->slot[s].work_next = 0u;
        }
        if (p.stats != nullptr && p.stats_cap > 0)
            p.stats[0].t_work_ns = 0;
        c->slot[0].found = 1ull;
        c->slot[0].fedges = (unsigned long long)deg;
        c->slot[0].maxdeg = (unsigned long long)deg;
        if (p.frontier_output == BFS_CSR_FRONTIER_PADDED) {
            // F_0 as a padded frontier of one slot
            p.pad[0][0] = source;
            c->slot[0].qpack = 1ull;
        } else if (deg > 0) {
            c->slot[0].qpack = (1ull << p.eb) | (unsigned long long)deg;
            p.qv[0][0] = source;
            p.qbeg[0][0] = b;
            p.qoff[0][0] = 0;
        }
        // U_0 = nonisolated vertices other than the source: slot 3 holds U_{-1}
        // such that U_0 = U_{-1} - |F_0|.
        c->slot[3].unvisited = c->nonisolated - (deg > 0 ? 1 : 0) + 1;
        c->slot[3].unvisited_edges = p.nnz;
        c->slot[3].dir = BFS_CSR_DIR_PUSH;
    }
}

// S0: CSR checks (row_ptr[0] = 0, row_ptr[n] = nnz, non-decreasing with rows
// shorter than 2^31 entries, col in range). Flags: bit 0 row_ptr, bit 1 col.
template <typename RowT>
__global__ void validate_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                                int64_t n, int64_t nnz, int* flags)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int bad = 0;
    if (tid == 0 && (row_ptr[0] != 0 || (int64_t)row_ptr[n] != nnz))
        bad |= 1;
    for (int64_t i = tid; i < n; i += stride) {
        const int64_t d = (int64_t)row_ptr[i + 1] - (int64_t)row_ptr[i];
        if (d < 0 || d > (int64_t)INT32_MAX)
            bad |= 1;  // decreasing, or a row too long for 32-bit degrees
    }
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

// Per vertex, its probe neighbour: the one of highest degree among the
// row's first kHeadScan entries (the earliest on ties), with bit 31 set when
// it is the row's only entry, kProbeNone for an empty row. A pull level
// tests this one likely parent of each unvisited vertex first, from a
// sequential 4-byte array instead of a row_ptr entry and a random col
// block: high-degree vertices are reached first in a search from almost any
// source, so for a vertex a pull level finds that neighbour is nearly always
// in the current frontier (on R-MAT inputs the first neighbour in CSR
// order, the plain choice, is there for only about a third of them). A
// vertex found through its probe needs no parent store (its hop code is
// flagged). Derived from the CSR at create time; rows are never copied.
constexpr int kHeadScan = 64;

template <typename RowT>
__global__ void probe_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                             int32_t n, uint32_t* probe)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += stride) {
        const RowT b = row_ptr[v];
        const RowT d = row_ptr[v + 1] - b;
        int32_t best = d > 0 ? col[b] : -1;
        if (d > 1) {
            const int m = d < (RowT)kHeadScan ? (int)d : kHeadScan;
            RowT best_deg = -1;
            for (int i = 0; i < m; i += 8) {
                int32_t u[8];
                RowT du[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    u[j] = i + j < m ? col[b + i + j] : -1;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    du[j] = u[j] >= 0 ? row_ptr[u[j] + 1] - row_ptr[u[j]] : (RowT)-1;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (du[j] > best_deg) {
                        best_deg = du[j];
                        best = u[j];
                    }
                }
            }
        }
        probe[v] = d == 0 ? kProbeNone : ((uint32_t)best | (d == 1 ? 0x80000000u : 0u));
    }
}

}  // namespace fbc
