/*
 * graphgen.c -- seeded synthetic graph generators and a CSR builder.
 *
 * These are the inputs both sides of the parity tests consume: the oracle and
 * the CUDA path read the same CSR arrays. Nothing here walks a graph or
 * computes a distance; it only draws edges and sorts them into CSR.
 *
 * Random numbers come from one counter-based generator: the SplitMix64
 * output function (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) applied to key + (counter + 1) * gamma,
 * gamma = 0x9E3779B97F4A7C15. Every draw is addressed by (key, counter), so
 * results do not depend on the thread count or the machine.
 *
 * Build: gcc -std=c11 -O3 -fopenmp -shared -fPIC graphgen.c
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GG_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t gg_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of an independent stream: one mixing of (seed, stream). */
uint64_t gg_key(uint64_t seed, uint64_t stream)
{
    return gg_mix(seed * GG_GAMMA + gg_mix(stream + 1));
}

static inline uint64_t gg_draw(uint64_t key, uint64_t ctr)
{
    return gg_mix(key + (ctr + 1) * GG_GAMMA);
}

/* Uniform double in [0, 1) from the top 53 bits. */
static inline double gg_unit(uint64_t x)
{
    return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

/* Uniform integer in [0, bound) by the multiply-high method. */
static inline uint64_t gg_below(uint64_t x, uint64_t bound)
{
    return (uint64_t)(((unsigned __int128)x * bound) >> 64);
}

/* Fill out[i] = gg_draw(key, first + i): exposes the generator for tests. */
void gg_draws(uint64_t key, uint64_t first, int64_t count, uint64_t *out)
{
    int64_t i;
    for (i = 0; i < count; ++i)
        out[i] = gg_draw(key, first + (uint64_t)i);
}

/*
 * R-MAT edges (Chakrabarti, Zhan and Faloutsos, SDM 2004): each edge picks one
 * of four quadrants with probabilities (a, b, c, 1-a-b-c), once per bit of
 * the vertex id, most significant bit first, with no noise. Each level uses a
 * 32-bit uniform: edge i takes draws i*16 .. i*16+15 of `key`, high half for
 * even levels and low half for odd ones; the quadrant thresholds are a,
 * a+b and a+b+c scaled to 2^32.
 */
void gg_rmat_edges(int scale, int64_t m, double a, double b, double c,
                   uint64_t key, uint32_t *src, uint32_t *dst)
{
    const uint64_t ta = (uint64_t)(a * 4294967296.0);
    const uint64_t tab = (uint64_t)((a + b) * 4294967296.0);
    const uint64_t tabc = (uint64_t)((a + b + c) * 4294967296.0);
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < m; ++i) {
        uint32_t u = 0, v = 0;
        uint64_t word = 0;
        int level;
        for (level = 0; level < scale; ++level) {
            uint64_t r;
            uint32_t ubit, vbit;
            if ((level & 1) == 0) {
                word = gg_draw(key, (uint64_t)i * 16 + (uint64_t)(level >> 1));
                r = word >> 32;
            } else {
                r = word & 0xFFFFFFFFULL;
            }
            ubit = r >= tab;
            vbit = (r >= ta && r < tab) || r >= tabc;
            u = (u << 1) | ubit;
            v = (v << 1) | vbit;
        }
        src[i] = u;
        dst[i] = v;
    }
}

/* Uniform endpoint pairs: edge i draws u from counter 2i and v from 2i+1. */
void gg_uniform_edges(int64_t n, int64_t m, uint64_t key, uint32_t *src,
                      uint32_t *dst)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < m; ++i) {
        src[i] = (uint32_t)gg_below(gg_draw(key, 2 * (uint64_t)i), (uint64_t)n);
        dst[i] = (uint32_t)gg_below(gg_draw(key, 2 * (uint64_t)i + 1), (uint64_t)n);
    }
}

/* A uniformly random permutation of 0..n-1 (Fisher-Yates, draws i = n-1..1). */
void gg_permutation(int64_t n, uint64_t key, uint32_t *perm)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        perm[i] = (uint32_t)i;
    for (i = n - 1; i > 0; --i) {
        const uint64_t j = gg_below(gg_draw(key, (uint64_t)i), (uint64_t)i + 1);
        const uint32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
}

/* Relabel both endpoints of every edge through perm. */
void gg_relabel(int64_t m, const uint32_t *perm, uint32_t *src, uint32_t *dst)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < m; ++i) {
        src[i] = perm[src[i]];
        dst[i] = perm[dst[i]];
    }
}

/*
 * rows x cols 4-neighbour lattice, vertex id r*cols + c. Candidate edges are
 * enumerated horizontal first, then vertical, each in row-major order; edge k
 * survives when the k-th draw is >= p_delete. Returns the number kept.
 */
int64_t gg_grid_edges(int64_t rows, int64_t cols, double p_delete, uint64_t key,
                      uint32_t *src, uint32_t *dst)
{
    int64_t k = 0, kept = 0, r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c + 1 < cols; ++c, ++k)
            if (gg_unit(gg_draw(key, (uint64_t)k)) >= p_delete) {
                src[kept] = (uint32_t)(r * cols + c);
                dst[kept] = (uint32_t)(r * cols + c + 1);
                ++kept;
            }
    for (r = 0; r + 1 < rows; ++r)
        for (c = 0; c < cols; ++c, ++k)
            if (gg_unit(gg_draw(key, (uint64_t)k)) >= p_delete) {
                src[kept] = (uint32_t)(r * cols + c);
                dst[kept] = (uint32_t)((r + 1) * cols + c);
                ++kept;
            }
    return kept;
}

/*
 * Chung-Lu graph (Chung and Lu, PNAS 2002): pair {i, j}, i < j, is an edge
 * with probability min(1, w_i w_j / sum(w)); pair (i, j) uses counter
 * i*n + j. Writes at most cap edges and returns how many pairs were kept
 * (which may exceed cap, in which case the caller retries with more room).
 */
int64_t gg_chung_lu_edges(int64_t n, const double *w, uint64_t key, int64_t cap,
                          uint32_t *src, uint32_t *dst)
{
    double total = 0.0;
    int64_t i, j, kept = 0;
    for (i = 0; i < n; ++i)
        total += w[i];
    for (i = 0; i < n; ++i)
        for (j = i + 1; j < n; ++j) {
            double p = w[i] * w[j] / total;
            if (p > 1.0)
                p = 1.0;
            if (gg_unit(gg_draw(key, (uint64_t)(i * n + j))) < p) {
                if (kept < cap) {
                    src[kept] = (uint32_t)i;
                    dst[kept] = (uint32_t)j;
                }
                ++kept;
            }
        }
    return kept;
}

static void radix_sort_u32(uint32_t *a, uint32_t *scratch, int64_t len)
{
    int pass;
    for (pass = 0; pass < 4; ++pass) {
        const int shift = 8 * pass;
        int64_t count[257], i;
        memset(count, 0, sizeof(count));
        for (i = 0; i < len; ++i)
            ++count[((a[i] >> shift) & 0xFF) + 1];
        for (i = 0; i < 256; ++i)
            count[i + 1] += count[i];
        for (i = 0; i < len; ++i)
            scratch[count[(a[i] >> shift) & 0xFF]++] = a[i];
        memcpy(a, scratch, (size_t)len * sizeof(uint32_t));
    }
}

/* Sort one adjacency row in place; returns 0, or -2 when out of memory. */
static int sort_row(uint32_t *a, int64_t len)
{
    int64_t i, j;
    if (len > 64) {
        uint32_t *scratch = (uint32_t *)malloc((size_t)len * sizeof(uint32_t));
        if (scratch == NULL)
            return -2;
        radix_sort_u32(a, scratch, len);
        free(scratch);
        return 0;
    }
    for (i = 1; i < len; ++i) {
        const uint32_t x = a[i];
        for (j = i; j > 0 && a[j - 1] > x; --j)
            a[j] = a[j - 1];
        a[j] = x;
    }
    return 0;
}

/*
 * Edge list -> CSR with sorted adjacency lists. With `symmetric` every edge
 * (u, v) is stored in both directions; `drop_loops` discards u == v and
 * `dedupe` keeps one copy of each repeated (u, v). row_ptr receives n + 1
 * int64 offsets and col up to col_cap entries; the entry count is returned,
 * or -1 when col_cap is too small, -2 when memory runs out and -3 for an
 * endpoint outside [0, n).
 *
 * Method: entries are partitioned by the high bits of their row into at most
 * 4096 buckets using per-thread counts over a fixed split of the edge list
 * (no shared counters); each bucket is then counting-sorted by row, each row
 * sorted and deduplicated, and the rows compacted into col.
 */
int64_t gg_build_csr(int64_t n, int64_t m, const uint32_t *src,
                     const uint32_t *dst, int symmetric, int drop_loops,
                     int dedupe, int64_t *row_ptr, int32_t *col, int64_t col_cap)
{
    int nthreads = 1, shift = 0, bad = 0;
    int64_t nbuckets, total, i, acc;
    int64_t *counts = NULL, *bstart = NULL, *rstart = NULL;
    uint64_t *keys = NULL;
    uint32_t *vals = NULL;

    if (n <= 0)
        return -3;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (i = 0; i < m; ++i)
        if (src[i] >= (uint64_t)n || dst[i] >= (uint64_t)n)
            bad = 1;
    if (bad)
        return -3;
#ifdef _OPENMP
    nthreads = omp_get_max_threads();
#endif
    while (((n - 1) >> shift) >= 4096)
        ++shift;
    nbuckets = ((n - 1) >> shift) + 1;

    counts = (int64_t *)calloc((size_t)(nthreads * nbuckets), sizeof(int64_t));
    bstart = (int64_t *)malloc((size_t)(nbuckets + 1) * sizeof(int64_t));
    rstart = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    if (counts == NULL || bstart == NULL || rstart == NULL)
        goto oom;
#pragma omp parallel num_threads(nthreads)
    {
        int t = 0;
        int64_t k, lo, hi;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        lo = m * t / nthreads;
        hi = m * (t + 1) / nthreads;
        for (k = lo; k < hi; ++k) {
            const uint32_t u = src[k], w = dst[k];
            if (drop_loops && u == w)
                continue;
            ++counts[(int64_t)t * nbuckets + (u >> shift)];
            if (symmetric)
                ++counts[(int64_t)t * nbuckets + (w >> shift)];
        }
    }
    acc = 0; /* exclusive offsets in (bucket, thread) order */
    for (i = 0; i < nbuckets; ++i) {
        int t;
        bstart[i] = acc;
        for (t = 0; t < nthreads; ++t) {
            const int64_t c = counts[(int64_t)t * nbuckets + i];
            counts[(int64_t)t * nbuckets + i] = acc;
            acc += c;
        }
    }
    bstart[nbuckets] = acc;
    total = acc;

    keys = (uint64_t *)malloc((size_t)(total > 0 ? total : 1) * sizeof(uint64_t));
    vals = (uint32_t *)malloc((size_t)(total > 0 ? total : 1) * sizeof(uint32_t));
    if (keys == NULL || vals == NULL)
        goto oom;
#pragma omp parallel num_threads(nthreads)
    {
        int t = 0;
        int64_t k, lo, hi, *cur;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        cur = counts + (int64_t)t * nbuckets;
        lo = m * t / nthreads;
        hi = m * (t + 1) / nthreads;
        for (k = lo; k < hi; ++k) {
            const uint32_t u = src[k], w = dst[k];
            if (drop_loops && u == w)
                continue;
            keys[cur[u >> shift]++] = ((uint64_t)u << 32) | w;
            if (symmetric)
                keys[cur[w >> shift]++] = ((uint64_t)w << 32) | u;
        }
    }
    free(counts);
    counts = NULL;

    /* Per bucket: counting sort by row into vals, then sort and dedupe each
     * row in place. rstart[v] = start of row v in vals, row_ptr[v + 1] = its
     * kept length (turned into offsets afterwards). */
    row_ptr[0] = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (i = 0; i < nbuckets; ++i) {
        const int64_t lo = bstart[i], hi = bstart[i + 1];
        const int64_t vlo = i << shift;
        const int64_t vhi = ((i + 1) << shift) < n ? ((i + 1) << shift) : n;
        const int64_t width = vhi - vlo;
        int64_t *fill = (int64_t *)calloc((size_t)(width + 1), sizeof(int64_t));
        int64_t k, r;
        if (fill == NULL) {
            bad = 1;
            continue;
        }
        for (k = lo; k < hi; ++k)
            ++fill[(int64_t)(keys[k] >> 32) - vlo + 1];
        for (r = 0; r < width; ++r) {
            fill[r + 1] += fill[r];
            rstart[vlo + r] = lo + fill[r];
        }
        for (k = lo; k < hi; ++k)
            vals[lo + fill[(int64_t)(keys[k] >> 32) - vlo]++] = (uint32_t)keys[k];
        /* fill[r] is now the end of row r (relative to lo) */
        for (r = 0; r < width; ++r) {
            uint32_t *row = vals + rstart[vlo + r];
            const int64_t len = lo + fill[r] - rstart[vlo + r];
            int64_t j, out = 0;
            if (sort_row(row, len) != 0) {
                bad = 1;
                break;
            }
            for (j = 0; j < len; ++j)
                if (!dedupe || out == 0 || row[out - 1] != row[j])
                    row[out++] = row[j];
            row_ptr[vlo + r + 1] = out;
        }
        free(fill);
    }
    free(keys);
    keys = NULL;
    if (bad)
        goto oom;
    for (i = 0; i < n; ++i)
        row_ptr[i + 1] += row_ptr[i];
    if (row_ptr[n] > col_cap) {
        free(bstart);
        free(rstart);
        free(vals);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 4096)
    for (i = 0; i < n; ++i)
        memcpy(col + row_ptr[i], vals + rstart[i],
               (size_t)(row_ptr[i + 1] - row_ptr[i]) * sizeof(uint32_t));
    total = row_ptr[n];
    free(bstart);
    free(rstart);
    free(vals);
    return total;
oom:
    free(counts);
    free(bstart);
    free(rstart);
    free(keys);
    free(vals);
    return -2;
}

/* Order-sensitive 64-bit fingerprint of a CSR (chunked so it parallelises). */
uint64_t gg_fingerprint(int64_t n, const int64_t *row_ptr, int64_t nnz,
                        const int32_t *col)
{
    const int64_t chunk = 1 << 20;
    const int64_t nchunks_col = (nnz + chunk - 1) / chunk;
    const int64_t nchunks_row = (n + 1 + chunk - 1) / chunk;
    uint64_t h = gg_mix((uint64_t)n * GG_GAMMA ^ gg_mix((uint64_t)nnz));
    int64_t c;
#pragma omp parallel for schedule(static) reduction(^ : h)
    for (c = 0; c < nchunks_col + nchunks_row; ++c) {
        uint64_t acc = gg_mix((uint64_t)c + 17);
        int64_t i, lo, hi;
        if (c < nchunks_col) {
            lo = c * chunk;
            hi = lo + chunk < nnz ? lo + chunk : nnz;
            for (i = lo; i < hi; ++i)
                acc = gg_mix(acc ^ ((uint64_t)(uint32_t)col[i] + (uint64_t)i * GG_GAMMA));
        } else {
            lo = (c - nchunks_col) * chunk;
            hi = lo + chunk < n + 1 ? lo + chunk : n + 1;
            for (i = lo; i < hi; ++i)
                acc = gg_mix(acc ^ ((uint64_t)row_ptr[i] * 31 + (uint64_t)i));
        }
        h ^= gg_mix(acc + (uint64_t)c * GG_GAMMA);
    }
    return h;
}

/*
 * Up to `count` distinct vertices of nonzero degree, drawn uniformly with
 * counters 0, 1, 2, ... of `key` (rejection of zero-degree and repeated
 * draws). Returns how many were found within max_draws draws.
 */
int64_t gg_pick_sources(int64_t n, const int64_t *row_ptr, int64_t count,
                        uint64_t key, int64_t max_draws, int32_t *out)
{
    int64_t found = 0, t, k;
    for (t = 0; t < max_draws && found < count; ++t) {
        const int64_t v = (int64_t)gg_below(gg_draw(key, (uint64_t)t), (uint64_t)n);
        int repeat = 0;
        if (row_ptr[v + 1] == row_ptr[v])
            continue;
        for (k = 0; k < found; ++k)
            if (out[k] == v) {
                repeat = 1;
                break;
            }
        if (!repeat)
            out[found++] = (int32_t)v;
    }
    return found;
}
