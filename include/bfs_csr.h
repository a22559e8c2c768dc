/*
 * bfs_csr.h -- level-synchronous frontier BFS over a CSR graph on one GPU.
 *
 * Given row_ptr/col, a vertex count and a source vertex, a run produces
 *   dist[v]   = number of hops from the source to v, or -1 if v is unreached;
 *   parent[v] = a BFS-tree parent of v: an in-neighbour u with
 *               dist[u] = dist[v] - 1 (parent[source] = source, -1 if unreached).
 * The problem statement (CSR in, per-vertex hop count out, -1 = not reached)
 * is that of "100 Days of GPU, Day 38: Graph traversal on a GPU" (section
 * "What a level-synchronous search actually launches") and of "The Frontier
 * Model for Parallel Breadth-First Search" (ch. 22, section 22.1). The pages
 * define no parent array; any in-neighbour one level closer is equally valid
 * ("Gunrock: advance, filter, and the ragged-frontier problem", "Done when").
 *
 * All functions are C-ABI, thread-compatible (one handle must not be used by
 * two host threads at once) and return a status code; none prints or exits.
 * Device pointers are CUDA global-memory addresses of the current device.
 * `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 */
#ifndef FRONTIER_BFS_CSR_H
#define FRONTIER_BFS_CSR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */
#define BFS_CSR_OK 0
#define BFS_CSR_EINVAL 1        /* bad argument or malformed CSR */
#define BFS_CSR_ENOMEM 2        /* a device or host allocation failed */
#define BFS_CSR_ECUDA 3         /* a CUDA call failed; see bfs_csr_last_cuda_error */
#define BFS_CSR_ETIMEOUT 4      /* a bounded device-wide wait expired */
#define BFS_CSR_EUNSUPPORTED 5  /* option or size the library cannot serve */
#define BFS_CSR_EDEVICE 6       /* a device-side consistency check failed */

/* ----------------------------------------------------------------- options */
/* Direction of a level. Pull (bottom-up) scans unvisited vertices for a
 * neighbour in the frontier bitmap; it needs in-edges, so it is only
 * available for a symmetric CSR (PMPP ch. 15 notes, section 15.3 push/pull
 * and section 15.7 direction-optimised BFS). */
#define BFS_CSR_DIR_AUTO 0      /* direction-optimising rule, see pull_alpha / push_beta */
#define BFS_CSR_DIR_PUSH 1
#define BFS_CSR_DIR_PULL 2      /* every level is bottom-up */

/* Load balance of a top-down (push) level. */
#define BFS_CSR_ADV_AUTO 0      /* merge-path when |F| >= merge_path_min_frontier
                                   (the Gunrock paper's static hybrid threshold), when
                                   the largest frontier degree >= binned_max_degree, or
                                   when the frontier's rows average 8 entries or more;
                                   binned otherwise */
#define BFS_CSR_ADV_BINNED 1    /* thread / warp / CTA per vertex by degree */
#define BFS_CSR_ADV_MERGE_PATH 2 /* edge-balanced: degree prefix + search */
#define BFS_CSR_ADV_SINGLE_CTA 3 /* (level records only) a narrow level run by one CTA */
#define BFS_CSR_ADV_PADDED 4     /* (level records only) one thread per slot of a
                                    sentinel-padded frontier, see BFS_CSR_FRONTIER_PADDED */

/* How a top-down level decides who discovered a vertex. */
#define BFS_CSR_DISC_BITMAP 0   /* atomicOr on a visited bitmap */
#define BFS_CSR_DISC_CAS 1      /* atomicCAS on dist (-1 -> level + 1) */
#define BFS_CSR_DISC_MIN 2      /* atomicMin on dist read as unsigned (-1 = UINT_MAX); the
                                   claim is won when level + 1 is below the old value
                                   ("Gunrock: advance, filter, and the ragged-frontier
                                   problem", step 2) */

/* What a push level writes for the next frontier ("Gunrock: advance, filter,
 * and the ragged-frontier problem", step 2: the advance writes every
 * neighbour it claims, or an invalid sentinel in its place; an optional
 * filter removes the sentinels). */
#define BFS_CSR_FRONTIER_COMPACT 0       /* winners go straight to the next queue
                                            (block-aggregated compaction) */
#define BFS_CSR_FRONTIER_PADDED_FILTER 1 /* every frontier edge writes its neighbour or -1
                                            into an edge-indexed array (merge-path
                                            advance); a filter pass compacts it into the
                                            next queue. No single-CTA levels */
#define BFS_CSR_FRONTIER_PADDED 2        /* no filter: the padded array is the next
                                            frontier, walked one thread per slot (the
                                            thread-mapped advance), sentinels skipped.
                                            Push levels only, no single-CTA levels */

/* Where a pull level's parents go (bitmap discovery). Almost every vertex a
 * pull level finds has its probe neighbour (see bfs_csr_create) as parent;
 * END_PASS only flags those in the one-byte hop code and writes every parent
 * once, in order, when the search ends, instead of one scattered 4-byte store
 * each (and no -1 fill at init). AUTO picks END_PASS when the parent array
 * (4n bytes) exceeds half of the device's L2, below which scattered stores
 * stay in the L2. */
#define BFS_CSR_PARENT_AUTO 0
#define BFS_CSR_PARENT_END_PASS 1
#define BFS_CSR_PARENT_AT_DISCOVERY 2

/* Where the level loop runs. */
#define BFS_CSR_LOOP_PERSISTENT 0 /* one cooperative kernel runs every level */
#define BFS_CSR_LOOP_HOST 1       /* one launch plus one device->host read per level */
#define BFS_CSR_LOOP_GRAPH 2      /* one CUDA graph launch per search: a while node, driven
                                     from the device, whose body launches one level; the
                                     host loop without its per-level round trip (PMPP ch. 15
                                     notes, section 15.7, on per-level launch cost) */

typedef struct bfs_csr_options {
    int32_t direction;               /* BFS_CSR_DIR_*, default AUTO */
    int32_t advance;                 /* BFS_CSR_ADV_*, default AUTO */
    int32_t discovery;               /* BFS_CSR_DISC_*, default BITMAP */
    int32_t loop_mode;               /* BFS_CSR_LOOP_*, default PERSISTENT */
    int32_t small_max_degree;        /* binned: degree < this -> thread per vertex (32) */
    int32_t cta_min_degree;          /* binned: degree >= this -> CTA per vertex (256) */
    int32_t merge_path_min_frontier; /* auto advance threshold on |F| (4096) */
    int32_t binned_max_degree;       /* auto advance threshold on max degree (8192) */
    double pull_alpha;               /* auto direction after a push level: pull iff
                                        m_F * pull_alpha > m_U, the edges of the vertices
                                        not reached yet (14) */
    int32_t max_depth;               /* label only vertices within this many hops; <0: all */
    int32_t validate;                /* nonzero: check the CSR at create (O(nnz)) */
    int32_t block_threads;           /* CTA size of the level kernel, a multiple of 32 from
                                        64; 0 = default and largest: 384 with int32
                                        row_ptr, 512 with int64 (create fails with
                                        BFS_CSR_EINVAL above it) */
    int32_t grid_blocks;             /* CTAs of the level kernel; 0 = fill every SM */
    int64_t barrier_timeout_ns;      /* limit of any device-wide wait (10 s) */
    int32_t test_unreachable_barrier;/* diagnostics only: nonzero makes the first
                                        device-wide barrier wait for one CTA more than
                                        exists, so the run ends with BFS_CSR_ETIMEOUT */
    int32_t push_beta;               /* auto direction after a pull level: push again iff
                                        |F| * push_beta < vertices of nonzero degree (24);
                                        0: apply the pull_alpha rule instead */
    int32_t narrow_max_edges;        /* push levels whose frontier has at most this many
                                        edges (and vertices) run on one CTA without grid
                                        barriers; 0 disables; capped at the CTA's stage
                                        (block_threads * 4); default 2048 */
    int32_t lanes;                   /* searches bfs_csr_run_batch keeps in flight at once,
                                        1..8 (0 means 1); each has its own search state
                                        in the workspace and 1/lanes of the level
                                        kernel's CTAs; default 1 */
    int32_t parent_pass;             /* BFS_CSR_PARENT_*: where parents found through a
                                        pull level's probe neighbour are written; default
                                        AUTO */
    int32_t frontier_output;         /* BFS_CSR_FRONTIER_*, default COMPACT; the padded
                                        modes add two arrays of max(nnz, 1) int32 to the
                                        workspace of each lane */
    int32_t reserved[2];             /* zero */
} bfs_csr_options;

/* Per-level record, kept when the run completes (see bfs_csr_level_stats). */
typedef struct bfs_csr_level_stat {
    int32_t level;           /* k: the frontier holds the vertices at distance k */
    int32_t direction;       /* BFS_CSR_DIR_PUSH or BFS_CSR_DIR_PULL; 0 for the
                                last frontier of a run cut by max_depth, which
                                counts as a level but is not expanded */
    int32_t advance;         /* push levels: BFS_CSR_ADV_BINNED, _MERGE_PATH or
                                _SINGLE_CTA; 0 otherwise */
    int32_t reserved;
    int64_t frontier;        /* |F_k| */
    int64_t frontier_edges;  /* m_F: sum of out-degrees over F_k */
    int64_t unvisited;       /* non-isolated vertices not yet reached at level start */
    int64_t max_degree;      /* largest out-degree in F_k; 0 when F_k was found by
                                a pull level and level k pulls too (a pull level
                                does not look at the degrees of what it finds) */
    int64_t t_start_ns;      /* device global timer at the level's start */
    int64_t t_work_ns;       /* device global timer when the last CTA finished the
                                level's work, before the barrier that ends it
                                (t_work_ns - t_start_ns is the level's busy time;
                                the rest, up to the next level's start, is its
                                synchronisation cost) */
} bfs_csr_level_stat;

typedef struct bfs_csr_t *bfs_csr_handle;

/* Fill *opt with the defaults listed above. */
int bfs_csr_default_options(bfs_csr_options *opt);

/* Bytes of device workspace a handle needs for a graph of n vertices and
 * nnz entries (row_ptr of int64 when row_ptr_64 != 0). opt may be NULL. */
int bfs_csr_workspace_bytes(int64_t n, int64_t nnz, int row_ptr_64,
                            const bfs_csr_options *opt, size_t *bytes);

/*
 * Adopt a device CSR. d_row_ptr holds n + 1 offsets (int32, or int64 when
 * row_ptr_64 != 0) with row_ptr[0] = 0 and row_ptr[n] = nnz; d_col holds nnz
 * int32 vertex ids. Both are borrowed: they must stay unchanged and alive
 * until bfs_csr_destroy. symmetric != 0 declares that the CSR is its own
 * transpose (every u->v has v->u), which enables pull levels. d_workspace may
 * be NULL (the library allocates and frees it) or caller memory of at least
 * bfs_csr_workspace_bytes, 256-byte aligned, owned by the caller. With
 * opt->validate the CSR is checked on the device; a malformed CSR gives
 * BFS_CSR_EINVAL. The call then derives, in the workspace, a bitmap of the
 * degree-0 vertices and a probe array (per vertex, 4 bytes: one probe
 * neighbour, the highest-degree one among the row's first 64 entries, and
 * whether it is the row's only entry) in one pass over the rows. Limits: 1 <= n < 2^31, nnz < 2^31 for int32
 * row_ptr. The call synchronises `stream`.
 */
int bfs_csr_create(bfs_csr_handle *out, int64_t n, int64_t nnz,
                   const void *d_row_ptr, int row_ptr_64, const int32_t *d_col,
                   int symmetric, void *d_workspace, size_t workspace_bytes,
                   const bfs_csr_options *opt, void *stream);

/*
 * Enqueue one search from `source` on `stream`: the level-synchronous search
 * of "100 Days of GPU, Day 38: Graph traversal on a GPU" (its host loop
 * `runBfs`: reset, then one frontier expansion per level until a level
 * discovers nothing) and of "The Frontier Model for Parallel Breadth-First
 * Search" (ch. 22, sections 22.1-22.2: expand every frontier vertex's CSR
 * row, claim each unvisited neighbour once, the claimed vertices form the
 * next frontier), with the levels run on the device. d_dist (n int32, required),
 * d_parent (n int32, may be NULL) and d_num_levels (one int32, may be NULL:
 * the number of non-empty frontiers, i.e. the source's eccentricity + 1 when
 * no depth bound cuts it short) are caller-owned device memory. The call is
 * asynchronous in the persistent loop mode; in the host loop mode it
 * synchronises `stream` once per level. Device-side failures (a wait that
 * timed out) are reported by bfs_csr_sync. Returns BFS_CSR_EINVAL for a
 * source outside [0, n) or a NULL d_dist, BFS_CSR_EUNSUPPORTED for forced
 * pull on a non-symmetric graph.
 */
int bfs_csr_run(bfs_csr_handle h, int64_t source, int32_t *d_dist,
                int32_t *d_parent, int32_t *d_num_levels, void *stream);

/*
 * The two halves of bfs_csr_run, for callers that time or schedule them
 * separately: bfs_csr_run_init resets the run state and seeds `source`
 * (one kernel: parent filled with -1 and the source's set to itself, the
 * per-search state cleared; dist is written by the level loop when the
 * search ends, or, with BFS_CSR_DISC_CAS, filled with -1 here);
 * bfs_csr_run_levels then runs the level loop (one cooperative kernel, or
 * one launch per level in the host loop mode) on the outputs given to the
 * preceding bfs_csr_run_init of this handle. Same arguments, errors and
 * asynchrony as bfs_csr_run; calling run_levels without a preceding
 * run_init gives BFS_CSR_EINVAL.
 */
int bfs_csr_run_init(bfs_csr_handle h, int64_t source, int32_t *d_dist,
                     int32_t *d_parent, void *stream);
int bfs_csr_run_levels(bfs_csr_handle h, int32_t *d_num_levels, void *stream);

/* Wait for the handle's last run on `stream`; return its device status and
 * store the level count in *num_levels (may be NULL). This is the one
 * device->host read a search needs: Day 38's `runBfs` reads the next
 * frontier's size back after every level ("What a level-synchronous search
 * actually launches"); here the level loop runs on the device and only its
 * end state (status, done, level count) is read, once. A search that ended
 * without reaching its end state gives BFS_CSR_EDEVICE. */
int bfs_csr_sync(bfs_csr_handle h, void *stream, int32_t *num_levels);

/*
 * Search from each of num_sources sources (host array) and wait. Source i's
 * dist and parent go to row i of d_dist and d_parent (device, num_sources x n
 * int32, row-major; d_parent may be NULL) and its level count to
 * d_num_levels[i] (device, may be NULL). The searches run on the handle's
 * opt.lanes lanes: lane j takes sources j, j + lanes, ... in order, on a
 * stream of its own forked from and joined back to `stream`, with its own
 * search state and 1/lanes of the level kernel's CTAs, so searches on
 * different lanes overlap: while one runs its narrow, latency-bound levels or
 * grid barriers, another keeps the memory system busy. Not a construct of the
 * pages, whose searches run one at a time; an independent search per source,
 * each with the result a single bfs_csr_run would give. d_stamps (device,
 * 3 x num_sources int64, may be NULL) receives, per search, the device
 * global timer (ns) when its init kernel, its level loop and the end of its
 * level loop ran. With lanes = 1 or the host loop mode the searches run one
 * after another on `stream`. Returns the first failing search's status
 * (every search is run), BFS_CSR_EINVAL for a NULL or out-of-range argument.
 * The level records of bfs_csr_level_stats are not kept for batch searches.
 */
int bfs_csr_run_batch(bfs_csr_handle h, int32_t num_sources, const int64_t *sources,
                      int32_t *d_dist, int32_t *d_parent, int32_t *d_num_levels,
                      int64_t *d_stamps, void *stream);

/* Copy up to cap per-level records of the last synchronised run to host
 * memory; *count receives the number of levels the run had. The records are
 * the columns of the level table of "100 Days of GPU, Day 38" ("What a
 * level-synchronous search actually launches": level, frontier size, edges,
 * largest degree) plus the direction, advance, unvisited count and device
 * timer stamps of each level; their frontier sizes sum to the reached count,
 * the page's check against a vertex queued twice ("Pitfalls"). */
int bfs_csr_level_stats(bfs_csr_handle h, bfs_csr_level_stat *host_buf,
                        int32_t cap, int32_t *count);

/*
 * Host-memory variant for callers whose graph and results live on the host.
 * bfs_csr_create_host allocates device copies of the CSR, the workspace and
 * the outputs, uploads the CSR and validates it as bfs_csr_create does.
 * bfs_csr_run_host then (1) re-uploads the CSR from h_row_ptr/h_col when they
 * are non-NULL (same n and nnz; checked again when validation is on) and
 * re-derives the per-vertex data create builds from it (the degree-0 bitmap
 * and the probe array: one pass over the rows), (2)
 * runs the search, (3) copies dist, parent (if h_parent != NULL) and the level
 * count back, and synchronises `stream` before returning the run's status.
 * Pinned host memory makes the copies asynchronous and fast.
 */
int bfs_csr_create_host(bfs_csr_handle *out, int64_t n, int64_t nnz,
                        const void *h_row_ptr, int row_ptr_64,
                        const int32_t *h_col, int symmetric,
                        const bfs_csr_options *opt, void *stream);
int bfs_csr_run_host(bfs_csr_handle h, int64_t source, const void *h_row_ptr,
                     const int32_t *h_col, int32_t *h_dist, int32_t *h_parent,
                     int32_t *h_num_levels, void *stream);

/*
 * Host-memory batch: one call searches from every source of sources[0 ..
 * num_sources) on a bfs_csr_create_host handle. When h_row_ptr/h_col are
 * non-NULL the CSR is first re-uploaded and re-derived as in
 * bfs_csr_run_host. Search i writes row i of h_dist (and of h_parent when it
 * is non-NULL): num_sources x n int32, row-major, caller-owned host memory
 * (pinned, so that the copies run asynchronously). The copy-back of search i
 * overlaps search i + 1: the handle keeps two device output slots and a copy
 * stream (allocated on the first call: 8n bytes more). h_num_levels
 * (num_sources int32, may be NULL) receives each search's level count. The
 * call synchronises before returning and returns the first failing search's
 * status, BFS_CSR_OK when all succeeded. BFS_CSR_EINVAL for a NULL argument,
 * num_sources <= 0 or a source outside [0, n); nothing runs then.
 */
int bfs_csr_run_host_batch(bfs_csr_handle h, int32_t num_sources, const int64_t *sources,
                           const void *h_row_ptr, const int32_t *h_col,
                           int32_t *h_dist, int32_t *h_parent, int32_t *h_num_levels,
                           void *stream);

/*
 * The isolated neighbour walk of one frontier, the measurement of "100 Days
 * of GPU, Day 38: Graph traversal on a GPU", section "Measuring the mapping
 * without measuring the launch": the handle's CSR rows of the frontier's
 * vertices are read `repeats` times with no claims, no frontier build and no
 * distance writes, so that one level's mapping can be timed on its own. For
 * slot i of d_frontier (device, frontier_size int32 vertex ids, 0 <=
 * frontier_size <= n) with vertex u, d_out[i] (device, frontier_size uint32)
 * receives
 *     sum over r < repeats and over e in [row_ptr[u], row_ptr[u + 1]) of
 *     (col[e] XOR r), modulo 2^32,
 * the same value for every mapping (unsigned addition wraps and commutes),
 * which a caller predicts exactly on the host. An entry outside [0, n)
 * walks nothing (its slot gets 0).
 * mapping: BFS_CSR_WALK_THREAD one thread per vertex, _WARP one warp per
 * vertex (the page's two mappings), _BINNED thread / warp / CTA by degree
 * with the handle's small_max_degree and cta_min_degree (the push levels'
 * mapping), _EDGE edge-balanced over the prefix of the frontier's degrees
 * (the merge path's mapping; the prefix is built first, on the device, in
 * the handle's workspace). Asynchronous on `stream`; it uses the workspace
 * of the handle's first lane, so it must not overlap a search on the same
 * handle. BFS_CSR_EINVAL for a NULL pointer (with frontier_size > 0), a
 * size outside [0, n], repeats < 0 or an unknown mapping.
 */
#define BFS_CSR_WALK_THREAD 0
#define BFS_CSR_WALK_WARP 1
#define BFS_CSR_WALK_BINNED 2
#define BFS_CSR_WALK_EDGE 3
int bfs_csr_walk(bfs_csr_handle h, const int32_t *d_frontier, int32_t frontier_size,
                 int32_t repeats, int32_t mapping, uint32_t *d_out, void *stream);

/* Release everything the library allocated for the handle. */
int bfs_csr_destroy(bfs_csr_handle h);

/* Static text for a status code. */
const char *bfs_csr_status_string(int status);

/* The last CUDA error code recorded on the handle (0 if none). */
int bfs_csr_last_cuda_error(bfs_csr_handle h);

/*
 * A search that allocates nothing, for callers that cannot call cudaMalloc:
 * for example a process whose device memory already belongs to another
 * allocator (a framework's caching pool that reserved the device), or a
 * latency-critical path where the implicit synchronisation of
 * cudaMalloc/cudaFree is not allowed. The pages have no counterpart; this is
 * a deployment variant of bfs_csr_run.
 *
 * Instead of a handle and a workspace it uses one scratch array that lives
 * in the library's own device memory (a file-scope __device__ array, about
 * 37 MB, held on every GPU that loads the library until the process exits).
 * That bounds the graph: n <= 1,048,576 vertices and an int32 row_ptr
 * (nnz < 2^31); larger inputs are rejected with BFS_CSR_EUNSUPPORTED before
 * any work. The caller still provides the device CSR (d_row_ptr: n + 1
 * int32, d_col: nnz int32), d_dist (n int32, required), d_parent (n int32,
 * may be NULL) and d_num_levels (one int32 on the device, may be NULL).
 * opt may be NULL (defaults). No cudaMalloc, cudaFree or other allocating
 * call is made, on the host or the device.
 *
 * The call runs synchronously on `stream`: it validates the CSR when
 * opt->validate is set, searches, waits for the stream and returns the
 * search's status (*num_levels, when not NULL, receives the level count on
 * the host). The first call on a device looks up the scratch array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture. The address is kept for the life of the
 * process: after a cudaDeviceReset of that device this entry point must not
 * be called again in the same process. Every call shares the one scratch
 * array and resets the parts that must start from zero; calls that overlap
 * on the GPU (from two host threads or two streams) race on it and must not
 * be issued. One search at a time: opt->lanes above 1 gives
 * BFS_CSR_EUNSUPPORTED.
 */
#define BFS_CSR_NOALLOC_MAX_VERTICES 1048576
int bfs_csr_run_noalloc(int64_t n, int64_t nnz, const int32_t *d_row_ptr,
                        const int32_t *d_col, int symmetric, int64_t source,
                        int32_t *d_dist, int32_t *d_parent,
                        int32_t *d_num_levels, int32_t *num_levels,
                        const bfs_csr_options *opt, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FRONTIER_BFS_CSR_H */
