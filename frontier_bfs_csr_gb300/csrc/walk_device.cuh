// walk_device.cuh -- the isolated neighbour walk of one frontier.
//
// "100 Days of GPU, Day 38: Graph traversal on a GPU", section "Measuring the
// mapping without measuring the launch", times one level's neighbour walk on
// its own: no claims, no frontier build, no distance writes, the walk
// repeated inside the kernel so that it outlasts a launch. Every mapping
// computes, for each frontier slot i with vertex u = frontier[i],
//
//     out[i] = sum over r < repeats, e in row(u) of (col[e] XOR r)   (mod 2^32)
//
// Unsigned addition wraps and commutes, so every mapping returns the same
// value whatever order its lanes visit the entries in, and a walk the
// compiler shortened returns a wrong value rather than a fast one; the XOR
// with r keeps the inner sum from being loop invariant (same section).
//
// A frontier entry outside [0, n) walks nothing (its slot gets 0), so a bad
// entry can never read outside row_ptr.
//
// Mappings:
//   thread   one thread per frontier vertex (the page's first mapping);
//   warp     one warp per frontier vertex, lanes striding the row (the page's
//            second mapping), reduced with a shuffle ladder;
//   binned   this library's push mapping: a thread for rows below small_max,
//            a warp below cta_min, the whole CTA above (PMPP ch. 15 notes,
//            section 15.7; the Gunrock reading page, step 4);
//   edge     edge-balanced: the level's entries are split evenly over every
//            warp of the grid using the exclusive prefix of the frontier's
//            degrees (the Gunrock reading page, steps 4-5; "The Frontier
//            Model for Parallel BFS", section 22.3); a row cut between warps
//            gets its partial sums added atomically.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fbc {

template <typename RowT>
__device__ __forceinline__ uint32_t walk_row(const int32_t* __restrict__ col, RowT b, RowT e,
                                             RowT start, RowT step, int repeats)
{
    uint32_t acc = 0u;
    for (int r = 0; r < repeats; ++r)
        for (RowT x = b + start; x < e; x += step)
            acc += (uint32_t)col[x] ^ (uint32_t)r;
    return acc;
}

template <typename RowT>
__global__ void walk_thread_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                                   int32_t n, const int32_t* __restrict__ frontier, int32_t size,
                                   int repeats, uint32_t* __restrict__ out)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < size) {
        const int32_t u = frontier[t];
        out[t] = (uint32_t)u < (uint32_t)n
                     ? walk_row(col, row_ptr[u], row_ptr[u + 1], (RowT)0, (RowT)1, repeats)
                     : 0u;
    }
}

template <typename RowT>
__global__ void walk_warp_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                                 int32_t n, const int32_t* __restrict__ frontier, int32_t size,
                                 int repeats, uint32_t* __restrict__ out)
{
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t acc = 0u;
    // w is the same in every lane: the branch is warp uniform and every lane
    // reaches the shuffles below.
    if (w < size) {
        const int32_t u = frontier[w];
        if ((uint32_t)u < (uint32_t)n)
            acc = walk_row(col, row_ptr[u], row_ptr[u + 1], (RowT)lane, (RowT)32, repeats);
    }
    for (int d = 16; d > 0; d >>= 1)
        acc += __shfl_down_sync(0xffffffffu, acc, d);
    if (w < size && lane == 0)
        out[w] = acc;
}

// Degree-binned: entry i belongs to CTA i % gridDim.x (small frontiers spread
// over every SM, as in the push levels). Rows of fewer than small_max
// entries are walked by their own thread, rows below cta_min by a warp, the
// rest by the whole CTA.
template <typename RowT>
__global__ void walk_binned_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                                   int32_t n, const int32_t* __restrict__ frontier, int32_t size,
                                   int repeats, int small_max, int cta_min,
                                   uint32_t* __restrict__ out)
{
    __shared__ int32_t s_big[1024];
    __shared__ int s_nbig;
    __shared__ uint32_t s_part[32];
    const int G = gridDim.x, bd = blockDim.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int mine = size > (int)blockIdx.x ? (size - (int)blockIdx.x + G - 1) / G : 0;
    if (threadIdx.x == 0)
        s_nbig = 0;
    __syncthreads();
    for (int base = 0; base < mine; base += bd) {
        const int li = base + threadIdx.x;
        const bool valid = li < mine;
        const int i = (int)blockIdx.x + li * G;
        RowT b = 0, e = 0;
        if (valid) {
            const int32_t u = frontier[i];
            if ((uint32_t)u < (uint32_t)n) {
                b = row_ptr[u];
                e = row_ptr[u + 1];
            }
        }
        const RowT deg = e - b;
        if (valid && deg < (RowT)small_max)
            out[i] = walk_row(col, b, e, (RowT)0, (RowT)1, repeats);
        unsigned mm = __ballot_sync(0xffffffffu, valid && deg >= (RowT)small_max && deg < (RowT)cta_min);
        while (mm) {
            const int src = __ffs(mm) - 1;
            mm &= mm - 1;
            const RowT wb = __shfl_sync(0xffffffffu, b, src);
            const RowT we = __shfl_sync(0xffffffffu, e, src);
            const int wi = __shfl_sync(0xffffffffu, i, src);
            uint32_t acc = walk_row(col, wb, we, (RowT)lane, (RowT)32, repeats);
            for (int d = 16; d > 0; d >>= 1)
                acc += __shfl_down_sync(0xffffffffu, acc, d);
            if (lane == 0)
                out[wi] = acc;
        }
        if (valid && deg >= (RowT)cta_min)
            s_big[atomicAdd(&s_nbig, 1)] = i;
        __syncthreads();
        const int nb = s_nbig;
        for (int q = 0; q < nb; ++q) {
            const int ci = s_big[q];
            const int32_t u = frontier[ci];  // in range: only such rows reach this list
            uint32_t acc = walk_row(col, row_ptr[u], row_ptr[u + 1], (RowT)threadIdx.x, (RowT)bd,
                                    repeats);
            for (int d = 16; d > 0; d >>= 1)
                acc += __shfl_down_sync(0xffffffffu, acc, d);
            if (lane == 0)
                s_part[warp] = acc;
            __syncthreads();
            if (threadIdx.x == 0) {
                uint32_t tot = 0u;
                for (int w = 0; w < (bd >> 5); ++w)
                    tot += s_part[w];
                out[ci] = tot;
            }
            __syncthreads();
        }
        if (threadIdx.x == 0)
            s_nbig = 0;
        __syncthreads();
    }
}

// Exclusive prefix of the frontier's degrees (offs[0 .. size]), one CTA: each
// thread sums a contiguous chunk, a block scan gives the chunk bases, and
// the chunk is written out. Also clears out[] for the atomic partial sums.
template <typename RowT>
__global__ void walk_prefix_kernel(const RowT* __restrict__ row_ptr, int32_t n,
                                   const int32_t* __restrict__ frontier, int32_t size,
                                   RowT* __restrict__ offs, uint32_t* __restrict__ out)
{
    __shared__ unsigned long long s_w[32];
    __shared__ unsigned long long s_tot;
    const int bd = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (size + bd - 1) / bd;
    const int lo = min(tid * per, size), hi = min(lo + per, size);
    unsigned long long sum = 0ull;
    for (int i = lo; i < hi; ++i) {
        const int32_t u = frontier[i];
        if ((uint32_t)u < (uint32_t)n)
            sum += (unsigned long long)(row_ptr[u + 1] - row_ptr[u]);
        out[i] = 0u;
    }
    unsigned long long inc = sum;
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d)
            inc += y;
    }
    if (lane == 31)
        s_w[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long x = lane < (bd >> 5) ? s_w[lane] : 0ull;
        unsigned long long wi = x;
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d)
                wi += y;
        }
        s_w[lane] = wi - x;
        if (lane == 31)
            s_tot = wi;
    }
    __syncthreads();
    unsigned long long run = s_w[warp] + inc - sum;
    for (int i = lo; i < hi; ++i) {
        offs[i] = (RowT)run;
        const int32_t u = frontier[i];
        if ((uint32_t)u < (uint32_t)n)
            run += (unsigned long long)(row_ptr[u + 1] - row_ptr[u]);
    }
    if (tid == 0)
        offs[size] = (RowT)s_tot;
}

// Edge-balanced walk: warp g of W takes entries [M g / W, M (g + 1) / W) of
// the level's M = offs[size] entries, finds the frontier slot of its first
// entry by binary search in offs, and walks slot by slot, 32 entries a step;
// each slot's partial sum goes to out[] with one atomic add per warp.
template <typename RowT>
__global__ void walk_edge_kernel(const RowT* __restrict__ row_ptr, const int32_t* __restrict__ col,
                                 int32_t n, const int32_t* __restrict__ frontier, int32_t size,
                                 int repeats, const RowT* __restrict__ offs,
                                 uint32_t* __restrict__ out)
{
    const int lane = threadIdx.x & 31;
    const unsigned long long W = (unsigned long long)gridDim.x * (blockDim.x >> 5);
    const unsigned long long g = ((unsigned long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const unsigned long long M = (unsigned long long)offs[size];
    const unsigned long long lo = M * g / W, hi = M * (g + 1) / W;
    if (lo >= hi)
        return;
    // last slot s with offs[s] <= lo
    int a = 0, b = size;
    while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if ((unsigned long long)offs[mid] <= lo)
            a = mid;
        else
            b = mid;
    }
    unsigned long long pos = lo;
    for (int s = a; s < size && pos < hi; ++s) {
        const unsigned long long s_beg = (unsigned long long)offs[s];
        const unsigned long long s_end = (unsigned long long)offs[s + 1];
        if (s_end <= pos)
            continue;
        const unsigned long long from = pos, to = s_end < hi ? s_end : hi;
        const int32_t u = frontier[s];  // in range: other slots have no entries
        const RowT rb = row_ptr[u];
        const RowT b0 = rb + (RowT)(from - s_beg), b1 = rb + (RowT)(to - s_beg);
        uint32_t acc = walk_row(col, b0, b1, (RowT)lane, (RowT)32, repeats);
        for (int d = 16; d > 0; d >>= 1)
            acc += __shfl_down_sync(0xffffffffu, acc, d);
        if (lane == 0)
            atomicAdd(out + s, acc);
        pos = to;
    }
}

}  // namespace fbc
