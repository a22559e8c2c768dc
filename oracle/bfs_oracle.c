/*
 * bfs_oracle.c -- the CPU oracle for level-synchronous BFS over CSR.
 *
 * TEST INFRASTRUCTURE. This file is the yardstick the CUDA path is checked
 * against. It is plain, sequential C with no blocking, no parallelism and no
 * shortcuts. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it; the product library never does, and
 * the two share no code, header or table.
 *
 * Definitions followed (pages are named by title and section):
 *
 *  oracle_bfs
 *    The textbook FIFO-queue breadth-first search the pages check every GPU
 *    result against: "100 Days of GPU, Day 38: Graph traversal on a GPU"
 *    (section "Measuring the mapping without measuring the launch", the host
 *    BFS and its exact-distance gate) and "The Frontier Model for Parallel
 *    Breadth-First Search" (DSA CUDA from first principles, ch. 22, section
 *    22.1 "The Sequential (CPU) Baseline"). Distances start at -1 (the
 *    not-reached mark), the source gets 0 and enters an explicit array queue
 *    with head and tail indices; each dequeued u walks its out-edges in CSR
 *    order and every neighbour still at -1 gets dist[u] + 1 and is enqueued.
 *    The pages define no parent array; the oracle records the first
 *    discoverer in FIFO order, and sets parent[source] = source.
 *
 *  oracle_bfs_depth
 *    The same search cut off at a depth bound: vertices farther than
 *    max_depth hops stay at -1. Section 22.1 of the ch. 22 page prints the
 *    state after level 1's frontier has been expanded (every vertex within
 *    two hops labelled, vertex 5 still -1); that is max_depth = 2 here.
 *
 *  oracle_check_dist
 *    A certificate check of a distance array that needs no second BFS. A
 *    dist[] is the exact hop distance from s if and only if
 *      (1) dist[s] = 0 and every other entry is -1 or >= 1,
 *      (2) for every edge u->v with dist[u] >= 0: dist[v] >= 0 and
 *          dist[v] <= dist[u] + 1,
 *      (3) every v != s with dist[v] >= 0 has an in-neighbour u with
 *          dist[u] = dist[v] - 1.
 *    (3) gives a path of length dist[v] from s, so hop(v) <= dist[v]; (2)
 *    applied along a shortest path gives dist[v] <= hop(v) and labels every
 *    reachable vertex. On a symmetric graph (2) reduces to the
 *    |dist[u] - dist[v]| <= 1 rule on every edge between reached vertices.
 *
 *  oracle_check_parent
 *    Validity of a BFS tree, the one output where several answers are
 *    right ("Gunrock: advance, filter, and the ragged-frontier problem",
 *    the "Done when" answer on a lost race: at a given level every
 *    candidate parent is equally valid). parent[s] = s; an unreached vertex
 *    has -1; every other reached v has parent[v] = u with u->v an edge of
 *    the CSR and dist[u] = dist[v] - 1.
 *
 *  oracle_level_sizes
 *    Per-level frontier sizes |{v : dist[v] = k}| and the walked-edge count
 *    sum of deg(v) over reached v (the page's "edges to walk" total in the
 *    Day 38 level table). The sizes summing to the reached count is the
 *    gate that sees a vertex enqueued twice (Day 38, "Pitfalls").
 *
 *  oracle_walk_checksum
 *    What the isolated neighbour walk of one frontier must return ("100 Days
 *    of GPU, Day 38", section "Measuring the mapping without measuring the
 *    launch"): for each frontier slot, the neighbour ids of its vertex's
 *    row XORed with the repeat counter r and summed over every repeat into
 *    an unsigned 32-bit accumulator, where overflow wraps. Plain loops in
 *    CSR order, repeat by repeat.
 *
 * Every function takes the CSR as (n, row_ptr, row_ptr_64, col): row_ptr
 * holds n + 1 entries, int64 when row_ptr_64 is nonzero and int32
 * otherwise; col holds row_ptr[n] int32 vertex ids. Return codes: 0 means
 * success (or "check passed"), a negative value a bad argument or no
 * memory, a positive value a failed check; *bad receives the first
 * offending vertex where there is one.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EARG (-1)
#define ORACLE_ENOMEM (-2)

static int64_t row_at(const void *row_ptr, int row_ptr_64, int64_t i)
{
    if (row_ptr_64)
        return ((const int64_t *)row_ptr)[i];
    return (int64_t)((const int32_t *)row_ptr)[i];
}

/* FIFO BFS bounded by max_depth (negative: no bound). */
int oracle_bfs_depth(int64_t n, const void *row_ptr, int row_ptr_64,
                     const int32_t *col, int64_t source, int64_t max_depth,
                     int32_t *dist, int32_t *parent, int64_t *num_levels)
{
    int32_t *queue;
    int64_t head = 0, tail = 0, v;

    if (n <= 0 || n > INT32_MAX || row_ptr == NULL || dist == NULL)
        return ORACLE_EARG;
    if (source < 0 || source >= n)
        return ORACLE_EARG;
    if (row_at(row_ptr, row_ptr_64, n) > 0 && col == NULL)
        return ORACLE_EARG;
    queue = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    if (queue == NULL)
        return ORACLE_ENOMEM;

    for (v = 0; v < n; ++v) {
        dist[v] = -1;
        if (parent != NULL)
            parent[v] = -1;
    }
    dist[source] = 0;
    if (parent != NULL)
        parent[source] = (int32_t)source;
    queue[tail++] = (int32_t)source;

    while (head < tail) {
        const int32_t u = queue[head++];
        const int64_t first = row_at(row_ptr, row_ptr_64, u);
        const int64_t last = row_at(row_ptr, row_ptr_64, (int64_t)u + 1);
        int64_t e;
        if (max_depth >= 0 && dist[u] >= max_depth)
            continue; /* its neighbours would lie beyond the bound */
        for (e = first; e < last; ++e) {
            const int32_t w = col[e];
            if (dist[w] == -1) {
                dist[w] = dist[u] + 1;
                if (parent != NULL)
                    parent[w] = u;
                queue[tail++] = w;
            }
        }
    }
    /* FIFO order is level order, so the last vertex enqueued is the
     * deepest one: the number of non-empty frontiers is its depth + 1. */
    if (num_levels != NULL)
        *num_levels = (int64_t)dist[queue[tail - 1]] + 1;
    free(queue);
    return ORACLE_OK;
}

int oracle_bfs(int64_t n, const void *row_ptr, int row_ptr_64,
               const int32_t *col, int64_t source, int32_t *dist,
               int32_t *parent, int64_t *num_levels)
{
    return oracle_bfs_depth(n, row_ptr, row_ptr_64, col, source, -1, dist,
                            parent, num_levels);
}

/* Certificate check (1)-(3) above. */
int oracle_check_dist(int64_t n, const void *row_ptr, int row_ptr_64,
                      const int32_t *col, int64_t source, const int32_t *dist,
                      int64_t *bad)
{
    unsigned char *supported;
    int64_t u, v;
    int rc = ORACLE_OK;

    if (n <= 0 || row_ptr == NULL || dist == NULL || source < 0 || source >= n)
        return ORACLE_EARG;
    if (bad != NULL)
        *bad = -1;
    /* (1) */
    if (dist[source] != 0) {
        if (bad != NULL)
            *bad = source;
        return 1;
    }
    for (v = 0; v < n; ++v) {
        if (v != source && !(dist[v] == -1 || dist[v] >= 1)) {
            if (bad != NULL)
                *bad = v;
            return 1;
        }
    }
    supported = (unsigned char *)calloc((size_t)n, 1);
    if (supported == NULL)
        return ORACLE_ENOMEM;
    /* (2), and collect the support of (3) in the same sweep over edges. */
    for (u = 0; u < n && rc == ORACLE_OK; ++u) {
        const int64_t first = row_at(row_ptr, row_ptr_64, u);
        const int64_t last = row_at(row_ptr, row_ptr_64, u + 1);
        int64_t e;
        if (dist[u] < 0)
            continue;
        for (e = first; e < last; ++e) {
            const int32_t w = col[e];
            if (w < 0 || w >= n) {
                rc = ORACLE_EARG;
                break;
            }
            if (dist[w] < 0 || dist[w] > dist[u] + 1) {
                if (bad != NULL)
                    *bad = w;
                rc = 2;
                break;
            }
            if (dist[w] == dist[u] + 1)
                supported[w] = 1;
        }
    }
    /* (3) */
    for (v = 0; v < n && rc == ORACLE_OK; ++v) {
        if (v != source && dist[v] >= 1 && !supported[v]) {
            if (bad != NULL)
                *bad = v;
            rc = 3;
        }
    }
    free(supported);
    return rc;
}

/* BFS-tree validity, given a distance array already known to be exact. */
int oracle_check_parent(int64_t n, const void *row_ptr, int row_ptr_64,
                        const int32_t *col, int64_t source,
                        const int32_t *dist, const int32_t *parent,
                        int64_t *bad)
{
    unsigned char *confirmed;
    int64_t u, v;
    int rc = ORACLE_OK;

    if (n <= 0 || row_ptr == NULL || dist == NULL || parent == NULL ||
        source < 0 || source >= n)
        return ORACLE_EARG;
    if (bad != NULL)
        *bad = -1;
    confirmed = (unsigned char *)calloc((size_t)n, 1);
    if (confirmed == NULL)
        return ORACLE_ENOMEM;
    /* An edge u->w confirms w when parent[w] names u and u sits exactly one
     * level above w. One sweep over the edges, so hubs cost nothing extra. */
    for (u = 0; u < n; ++u) {
        const int64_t first = row_at(row_ptr, row_ptr_64, u);
        const int64_t last = row_at(row_ptr, row_ptr_64, u + 1);
        int64_t e;
        if (dist[u] < 0)
            continue;
        for (e = first; e < last; ++e) {
            const int32_t w = col[e];
            if (w >= 0 && w < n && parent[w] == u && dist[w] == dist[u] + 1)
                confirmed[w] = 1;
        }
    }
    for (v = 0; v < n; ++v) {
        int ok;
        if (v == source)
            ok = (parent[v] == (int32_t)source);
        else if (dist[v] < 0)
            ok = (parent[v] == -1);
        else
            ok = confirmed[v];
        if (!ok) {
            if (bad != NULL)
                *bad = v;
            rc = 4;
            break;
        }
    }
    free(confirmed);
    return rc;
}

/* Level sizes (capped at level_cap entries) and the walked-edge count. */
int oracle_level_sizes(int64_t n, const void *row_ptr, int row_ptr_64,
                       const int32_t *dist, int64_t *level_sizes,
                       int64_t level_cap, int64_t *num_levels,
                       int64_t *reached, int64_t *edges_walked)
{
    int64_t v, deepest = -1, count = 0, edges = 0, k;

    if (n <= 0 || row_ptr == NULL || dist == NULL)
        return ORACLE_EARG;
    for (k = 0; k < level_cap && level_sizes != NULL; ++k)
        level_sizes[k] = 0;
    for (v = 0; v < n; ++v) {
        const int32_t d = dist[v];
        if (d < 0)
            continue;
        ++count;
        edges += row_at(row_ptr, row_ptr_64, v + 1) -
                 row_at(row_ptr, row_ptr_64, v);
        if (d > deepest)
            deepest = d;
        if (level_sizes != NULL && d < level_cap)
            ++level_sizes[d];
    }
    if (num_levels != NULL)
        *num_levels = deepest + 1;
    if (reached != NULL)
        *reached = count;
    if (edges_walked != NULL)
        *edges_walked = edges;
    return ORACLE_OK;
}

/* Walk checksum of every frontier slot; an entry outside [0, n) gets 0. */
int oracle_walk_checksum(int64_t n, const void *row_ptr, int row_ptr_64,
                         const int32_t *col, const int32_t *frontier,
                         int64_t size, int64_t repeats, uint32_t *out)
{
    int64_t i, r, e;

    if (n <= 0 || row_ptr == NULL || size < 0 || repeats < 0)
        return ORACLE_EARG;
    if (size > 0 && (frontier == NULL || out == NULL))
        return ORACLE_EARG;
    for (i = 0; i < size; ++i) {
        const int32_t u = frontier[i];
        uint32_t acc = 0u;
        if (u >= 0 && u < n) {
            const int64_t first = row_at(row_ptr, row_ptr_64, u);
            const int64_t last = row_at(row_ptr, row_ptr_64, u + 1);
            for (r = 0; r < repeats; ++r)
                for (e = first; e < last; ++e)
                    acc += (uint32_t)col[e] ^ (uint32_t)r;
        }
        out[i] = acc;
    }
    return ORACLE_OK;
}
