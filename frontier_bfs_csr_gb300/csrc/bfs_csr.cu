// bfs_csr.cu -- the C-ABI library: handle, workspace, launches.
//
// The device work lives in bfs_device.cuh; this file validates arguments,
// carves the workspace, sizes the cooperative grid and drives the level loop
// either once per run (persistent mode) or once per level with a
// device-to-host read of the loop state in between (host mode, the
// structure of the host loop in "100 Days of GPU, Day 38").
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <new>

#include "bfs_csr.h"
#include "bfs_device.cuh"
#include "walk_device.cuh"

using fbc::Ctl;
using fbc::Params;

namespace {

constexpr int kStatsCap = 1 << 16;


constexpr int kMaxLanes = 8;

// Workspace: the graph part (dead bitmap, probe array), derived once per CSR,
// then one search part per lane; the offsets below are lane 0's, lane j's
// are `search` bytes further on.
struct Layout {
    size_t dead, probe;
    size_t ctl, visited, hop, fb0, fb1, qv0, qv1, qbeg0, qbeg1, qoff0, qoff1, wq, stats, pad0, pad1;
    size_t pad_entries;
    size_t search, total;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// pad_entries: length of each padded-frontier array (0 without the padded
// frontier modes).
Layout make_layout(int64_t n, int row_ptr_64, int lanes = 1, size_t pad_entries = 0)
{
    Layout L;
    const size_t words = (size_t)((n + 31) / 32);
    const size_t R = row_ptr_64 ? 8 : 4;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.dead = take(words * 4);
    L.probe = take((size_t)n * 4);
    const size_t search0 = off;
    L.ctl = take(sizeof(Ctl));
    L.visited = take(words * 4);
    L.hop = take(align_up((size_t)n, 16));
    L.fb0 = take(words * 4);
    L.fb1 = take(words * 4);
    L.qv0 = take((size_t)n * 4);
    L.qv1 = take((size_t)n * 4);
    L.qbeg0 = take((size_t)n * R);
    L.qbeg1 = take((size_t)n * R);
    L.qoff0 = take((size_t)n * R);
    L.qoff1 = take((size_t)n * R);
    L.wq = take((size_t)n * 4);
    L.stats = take((size_t)kStatsCap * sizeof(bfs_csr_level_stat));
    L.pad_entries = pad_entries;
    L.pad0 = pad_entries ? take(pad_entries * 4) : 0;
    L.pad1 = pad_entries ? take(pad_entries * 4) : 0;
    L.search = off - search0;
    L.total = off + (size_t)(lanes - 1) * L.search;
    return L;
}

size_t pad_entries_for(const bfs_csr_options& o, int64_t nnz)
{
    if (o.frontier_output == BFS_CSR_FRONTIER_COMPACT)
        return 0;
    return (size_t)(nnz > 0 ? nnz : 1);
}

}  // namespace

struct bfs_csr_t {
    int64_t n = 0, nnz = 0;
    int row_ptr_64 = 0;
    const void* row_ptr = nullptr;
    const int32_t* col = nullptr;
    int symmetric = 0;
    bfs_csr_options opt{};
    unsigned char* ws = nullptr;
    size_t ws_bytes = 0;
    bool own_ws = false;
    Layout L{};
    int words = 0;
    int eb = 0;
    int device = 0;
    int sm_count = 0;
    int l2_bytes = 0;
    int block = 0;
    int grid = 0;
    size_t smem = 0;
    int last_cuda_error = 0;
    int last_status = BFS_CSR_OK;
    int last_num_levels = 0;
    // outputs of the last bfs_csr_run_init, consumed by bfs_csr_run_levels
    int32_t pending_source = -1;
    int32_t* pending_dist = nullptr;
    int32_t* pending_parent = nullptr;
    // host-memory variant
    bool host_mode = false;
    void* d_row_ptr_own = nullptr;
    int32_t* d_col_own = nullptr;
    int32_t* d_dist_own = nullptr;
    int32_t* d_parent_own = nullptr;
    int32_t* d_levels_own = nullptr;
    // host-memory batches: a second output slot, per-search level counts and
    // end states, and a copy stream with its events (made on first use)
    int32_t* d_dist_b = nullptr;
    int32_t* d_parent_b = nullptr;
    int32_t* d_batch = nullptr;   // per search: status, done, level, num_levels
    int32_t batch_cap = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_search[2] = {nullptr, nullptr};
    cudaEvent_t ev_copy[2] = {nullptr, nullptr};
    // graph loop mode: one instantiated graph per (lane, outputs, stamps),
    // made on first use and kept until destroy
    struct LoopGraph {
        int lane = 0, grid = 0;
        const void *dist = nullptr, *parent = nullptr, *levels = nullptr, *stamps = nullptr;
        cudaGraph_t graph = nullptr;
        cudaGraphExec_t exec = nullptr;
    };
    std::vector<LoopGraph> graphs;
    // device batches: one stream per lane and the fork/join events (made on
    // first use)
    int lanes = 1;
    cudaStream_t lane_stream[kMaxLanes] = {};
    cudaEvent_t ev_fork = nullptr;
    cudaEvent_t ev_join[kMaxLanes] = {};
};

namespace {

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int cuda_fail(bfs_csr_t* h, cudaError_t e)
{
    if (h != nullptr)
        h->last_cuda_error = (int)e;
    return e == cudaErrorMemoryAllocation ? BFS_CSR_ENOMEM : BFS_CSR_ECUDA;
}

#define FBC_CUDA(h, call)                         \
    do {                                          \
        cudaError_t e_ = (call);                  \
        if (e_ != cudaSuccess)                    \
            return cuda_fail((h), e_);            \
    } while (0)

int check_options(const bfs_csr_options& o)
{
    if (o.direction < BFS_CSR_DIR_AUTO || o.direction > BFS_CSR_DIR_PULL) return BFS_CSR_EINVAL;
    if (o.advance < BFS_CSR_ADV_AUTO || o.advance > BFS_CSR_ADV_MERGE_PATH) return BFS_CSR_EINVAL;
    if (o.discovery < BFS_CSR_DISC_BITMAP || o.discovery > BFS_CSR_DISC_MIN) return BFS_CSR_EINVAL;
    if (o.frontier_output < BFS_CSR_FRONTIER_COMPACT || o.frontier_output > BFS_CSR_FRONTIER_PADDED)
        return BFS_CSR_EINVAL;
    if (o.loop_mode < BFS_CSR_LOOP_PERSISTENT || o.loop_mode > BFS_CSR_LOOP_GRAPH) return BFS_CSR_EINVAL;
    if (o.small_max_degree < 1 || o.cta_min_degree < o.small_max_degree) return BFS_CSR_EINVAL;
    if (o.merge_path_min_frontier < 0 || o.binned_max_degree < 1) return BFS_CSR_EINVAL;
    if (!(o.pull_alpha >= 0.0) || o.push_beta < 0) return BFS_CSR_EINVAL;
    if (o.block_threads != 0 &&
        (o.block_threads < 64 || o.block_threads > fbc::kLevelBlockMax || o.block_threads % 32))
        return BFS_CSR_EINVAL;
    if (o.grid_blocks < 0 || o.barrier_timeout_ns <= 0 || o.narrow_max_edges < 0)
        return BFS_CSR_EINVAL;
    if (o.lanes < 0 || o.lanes > kMaxLanes)
        return BFS_CSR_EINVAL;
    if (o.parent_pass < BFS_CSR_PARENT_AUTO || o.parent_pass > BFS_CSR_PARENT_AT_DISCOVERY)
        return BFS_CSR_EINVAL;
    return BFS_CSR_OK;
}

// Bits of the packed (count, edges) counter given to the edge total.
int edge_bits(int64_t n, int64_t nnz, int row_ptr_64)
{
    if (!row_ptr_64)
        return 32;
    int vb = 1;
    while (vb < 63 && (int64_t(1) << vb) <= n)
        ++vb;
    const int eb = 64 - vb;
    if (eb >= 63 || nnz < (int64_t(1) << eb))
        return eb;
    return -1;
}

template <typename RowT>
void* level_kernel_ptr() { return reinterpret_cast<void*>(&fbc::level_kernel<RowT>); }

template <typename RowT>
int configure_grid(bfs_csr_t* h)
{
    h->block = h->opt.block_threads ? h->opt.block_threads : fbc::level_block<RowT>();
    if (h->block > fbc::level_block<RowT>())
        return BFS_CSR_EINVAL;  // above the kernel's launch bound for this row_ptr width
    h->smem = fbc::level_smem_bytes<RowT>(h->block);
    FBC_CUDA(h, cudaFuncSetAttribute(fbc::level_kernel<RowT>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->smem));
    int per_sm = 0;
    FBC_CUDA(h, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fbc::level_kernel<RowT>,
                                                              h->block, h->smem));
    if (per_sm < 1)
        return BFS_CSR_EUNSUPPORTED;
    const int full = per_sm * h->sm_count;
    h->grid = h->opt.grid_blocks ? (h->opt.grid_blocks < full ? h->opt.grid_blocks : full) : full;
    return BFS_CSR_OK;
}

template <typename RowT>
Params<RowT> make_params(bfs_csr_t* h, int32_t* d_dist, int32_t* d_parent, int32_t* d_levels,
                         int lane = 0)
{
    Params<RowT> p;
    std::memset(&p, 0, sizeof(p));
    unsigned char* g = h->ws;                                // graph part
    unsigned char* w = h->ws + (size_t)lane * h->L.search;   // this lane's search part
    p.row_ptr = static_cast<const RowT*>(h->row_ptr);
    p.col = h->col;
    p.n = (int32_t)h->n;
    p.words = h->words;
    p.dist = d_dist;
    p.parent = d_parent;
    p.visited = reinterpret_cast<uint32_t*>(w + h->L.visited);
    p.dead = reinterpret_cast<const uint32_t*>(g + h->L.dead);
    p.probe = reinterpret_cast<const uint32_t*>(g + h->L.probe);
    p.hop = reinterpret_cast<uint8_t*>(w + h->L.hop);
    p.defer_dist = h->opt.discovery == BFS_CSR_DISC_BITMAP ? 1 : 0;
    // A parent array within half of the L2 takes scattered stores without
    // DRAM read-modify-writes; a larger one is written once, whole, by the
    // end-of-search pass (R-MAT scale 25: 134 MB against a 129 MB L2).
    const bool big = (size_t)h->n * 4 > (size_t)h->l2_bytes / 2;
    p.defer_parent = p.defer_dist && (h->opt.parent_pass == BFS_CSR_PARENT_END_PASS ||
                                      (h->opt.parent_pass == BFS_CSR_PARENT_AUTO && big)) ? 1 : 0;
    p.vec_out = ((reinterpret_cast<uintptr_t>(d_dist) & 15u) == 0 &&
                 (reinterpret_cast<uintptr_t>(d_parent) & 15u) == 0) ? 1 : 0;
    p.fb[0] = reinterpret_cast<uint32_t*>(w + h->L.fb0);
    p.fb[1] = reinterpret_cast<uint32_t*>(w + h->L.fb1);
    p.qv[0] = reinterpret_cast<int32_t*>(w + h->L.qv0);
    p.qv[1] = reinterpret_cast<int32_t*>(w + h->L.qv1);
    p.qbeg[0] = reinterpret_cast<RowT*>(w + h->L.qbeg0);
    p.qbeg[1] = reinterpret_cast<RowT*>(w + h->L.qbeg1);
    p.qoff[0] = reinterpret_cast<RowT*>(w + h->L.qoff0);
    p.qoff[1] = reinterpret_cast<RowT*>(w + h->L.qoff1);
    p.ctl = reinterpret_cast<Ctl*>(w + h->L.ctl);
    p.frontier_output = h->opt.frontier_output;
    p.emit_max = 65536;
    p.wq = reinterpret_cast<int32_t*>(w + h->L.wq);
    p.pad[0] = h->L.pad_entries ? reinterpret_cast<int32_t*>(w + h->L.pad0) : nullptr;
    p.pad[1] = h->L.pad_entries ? reinterpret_cast<int32_t*>(w + h->L.pad1) : nullptr;
    p.stats = reinterpret_cast<bfs_csr_level_stat*>(w + h->L.stats);
    p.stats_cap = kStatsCap;
    p.num_levels_out = d_levels;
    p.eb = h->eb;
    p.direction = h->opt.direction;
    p.advance = h->opt.advance;
    p.discovery = h->opt.discovery;
    p.small_max = h->opt.small_max_degree;
    p.cta_min = h->opt.cta_min_degree;
    p.mp_min_frontier = h->opt.merge_path_min_frontier;
    p.binned_max_deg = h->opt.binned_max_degree;
    p.pull_alpha = h->opt.pull_alpha;
    p.push_beta = h->opt.push_beta;
    p.nnz = h->nnz;
    p.max_depth = h->opt.max_depth;
    p.symmetric = h->symmetric;
    p.level_budget = INT_MAX;
    p.timeout_ns = h->opt.barrier_timeout_ns;
    p.unreachable_barrier = h->opt.test_unreachable_barrier ? 1 : 0;
    {
        const int cap = fbc::stage_cap<RowT>(h->block);
        p.narrow_max = h->opt.narrow_max_edges < cap ? h->opt.narrow_max_edges : cap;
    }
    return p;
}

int init_grid(bfs_csr_t* h) { return h->sm_count * 8; }

template <typename RowT>
int prepare(bfs_csr_t* h, cudaStream_t s)
{
    unsigned char* w = h->ws;
    Ctl* ctl = reinterpret_cast<Ctl*>(w + h->L.ctl);
    for (int j = 0; j < h->lanes; ++j)
        FBC_CUDA(h, cudaMemsetAsync(w + (size_t)j * h->L.search + h->L.ctl, 0, sizeof(Ctl), s));
    const RowT* rp = static_cast<const RowT*>(h->row_ptr);
    if (h->opt.validate) {
        fbc::validate_kernel<RowT><<<init_grid(h), 256, 0, s>>>(rp, h->col, h->n, h->nnz,
                                                                 &ctl->validate_flags);
        FBC_CUDA(h, cudaGetLastError());
        int flags = 0;
        FBC_CUDA(h, cudaMemcpyAsync(&flags, &ctl->validate_flags, sizeof(int),
                                    cudaMemcpyDeviceToHost, s));
        FBC_CUDA(h, cudaStreamSynchronize(s));
        if (flags != 0)
            return BFS_CSR_EINVAL;
    }
    fbc::dead_kernel<RowT><<<init_grid(h), 256, 0, s>>>(
        rp, (int32_t)h->n, h->words, reinterpret_cast<uint32_t*>(w + h->L.dead), &ctl->nonisolated);
    FBC_CUDA(h, cudaGetLastError());
    // Every lane's control block carries the non-isolated count.
    for (int j = 1; j < h->lanes; ++j) {
        Ctl* cj = reinterpret_cast<Ctl*>(w + (size_t)j * h->L.search + h->L.ctl);
        FBC_CUDA(h, cudaMemcpyAsync(&cj->nonisolated, &ctl->nonisolated, sizeof(long long),
                                    cudaMemcpyDeviceToDevice, s));
    }
    fbc::probe_kernel<RowT><<<init_grid(h), 256, 0, s>>>(rp, h->col, (int32_t)h->n,
                                                          reinterpret_cast<uint32_t*>(w + h->L.probe));
    FBC_CUDA(h, cudaGetLastError());
    FBC_CUDA(h, cudaStreamSynchronize(s));
    return configure_grid<RowT>(h);
}

template <typename RowT>
int launch_init(bfs_csr_t* h, int32_t source, int32_t* d_dist, int32_t* d_parent, cudaStream_t s,
                int lane = 0, long long* stamps = nullptr)
{
    Params<RowT> p = make_params<RowT>(h, d_dist, d_parent, nullptr, lane);
    p.stamps = stamps;
    const uint32_t* dead = reinterpret_cast<const uint32_t*>(h->ws + h->L.dead);
    fbc::init_kernel<RowT><<<init_grid(h), 256, 0, s>>>(p, dead, source, h->symmetric ? 1 : 0);
    FBC_CUDA(h, cudaGetLastError());
    return BFS_CSR_OK;
}

constexpr size_t kMaxLoopGraphs = 64;

// Graph loop mode: a CUDA graph whose one node is a while loop; its body is
// one cooperative launch of the level kernel with a budget of one level.
// The kernel's last CTA sets the loop's condition to 0 once the search has
// ended (or failed), so one graph launch runs the whole level loop with no
// host round trip. The graph holds the kernel's parameters (outputs and
// stamps included), so it is made once per set of them and kept.
template <typename RowT>
int loop_graph(bfs_csr_t* h, int32_t* d_dist, int32_t* d_parent, int32_t* d_levels, int lane,
               int grid, long long* stamps, cudaGraphExec_t* out)
{
    for (const auto& g : h->graphs) {
        if (g.lane == lane && g.grid == grid && g.dist == d_dist && g.parent == d_parent &&
            g.levels == d_levels && g.stamps == stamps) {
            *out = g.exec;
            return BFS_CSR_OK;
        }
    }
    if (h->graphs.size() >= kMaxLoopGraphs) {
        auto& old = h->graphs.front();
        cudaGraphExecDestroy(old.exec);
        cudaGraphDestroy(old.graph);
        h->graphs.erase(h->graphs.begin());
    }
    bfs_csr_t::LoopGraph lg;
    lg.lane = lane;
    lg.grid = grid;
    lg.dist = d_dist;
    lg.parent = d_parent;
    lg.levels = d_levels;
    lg.stamps = stamps;
    FBC_CUDA(h, cudaGraphCreate(&lg.graph, 0));
    auto fail = [&](cudaError_t e) {
        cudaGraphDestroy(lg.graph);
        return cuda_fail(h, e);
    };
    cudaGraphConditionalHandle cond = 0;
    cudaError_t e = cudaGraphConditionalHandleCreate(&cond, lg.graph, 1u, cudaGraphCondAssignDefault);
    if (e != cudaSuccess)
        return fail(e);
    // cudaGraphNodeParams has no default constructor (its union holds dim3s):
    // build it in zeroed storage, as its reserved fields require.
    alignas(cudaGraphNodeParams) unsigned char cbuf[sizeof(cudaGraphNodeParams)] = {};
    cudaGraphNodeParams& cp = *reinterpret_cast<cudaGraphNodeParams*>(cbuf);
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = cond;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    cudaGraphNode_t cnode = nullptr;
    e = cudaGraphAddNode(&cnode, lg.graph, nullptr, nullptr, 0, &cp);
    if (e != cudaSuccess)
        return fail(e);
    cudaGraph_t body = cp.conditional.phGraph_out[0];
    Params<RowT> p = make_params<RowT>(h, d_dist, d_parent, d_levels, lane);
    p.stamps = stamps;
    p.level_budget = 1;
    p.graph_cond = cond;
    void* args[] = {&p};
    alignas(cudaGraphNodeParams) unsigned char kbuf[sizeof(cudaGraphNodeParams)] = {};
    cudaGraphNodeParams& kp = *reinterpret_cast<cudaGraphNodeParams*>(kbuf);
    kp.type = cudaGraphNodeTypeKernel;
    kp.kernel.func = level_kernel_ptr<RowT>();
    kp.kernel.gridDim = dim3(grid);
    kp.kernel.blockDim = dim3(h->block);
    kp.kernel.sharedMemBytes = (unsigned)h->smem;
    kp.kernel.kernelParams = args;
    cudaGraphNode_t knode = nullptr;
    e = cudaGraphAddNode(&knode, body, nullptr, nullptr, 0, &kp);
    if (e != cudaSuccess)
        return fail(e);
    cudaLaunchAttributeValue coop;
    std::memset(&coop, 0, sizeof(coop));
    coop.cooperative = 1;
    e = cudaGraphKernelNodeSetAttribute(knode, cudaLaunchAttributeCooperative, &coop);
    if (e != cudaSuccess)
        return fail(e);
    e = cudaGraphInstantiate(&lg.exec, lg.graph, 0);
    if (e != cudaSuccess)
        return fail(e);
    h->graphs.push_back(lg);
    *out = lg.exec;
    return BFS_CSR_OK;
}

template <typename RowT>
int launch_levels(bfs_csr_t* h, int32_t* d_dist, int32_t* d_parent, int32_t* d_levels,
                  cudaStream_t s, int lane = 0, int grid = 0, long long* stamps = nullptr)
{
    Params<RowT> p = make_params<RowT>(h, d_dist, d_parent, d_levels, lane);
    p.stamps = stamps;
    void* args[] = {&p};
    if (grid <= 0)
        grid = h->grid;
    if (h->opt.loop_mode == BFS_CSR_LOOP_PERSISTENT) {
        FBC_CUDA(h, cudaLaunchCooperativeKernel(level_kernel_ptr<RowT>(), dim3(grid),
                                                dim3(h->block), args, h->smem, s));
        return BFS_CSR_OK;
    }
    if (h->opt.loop_mode == BFS_CSR_LOOP_GRAPH) {
        cudaGraphExec_t exec = nullptr;
        const int rc = loop_graph<RowT>(h, d_dist, d_parent, d_levels, lane, grid, stamps, &exec);
        if (rc != BFS_CSR_OK)
            return rc;
        FBC_CUDA(h, cudaGraphLaunch(exec, s));
        return BFS_CSR_OK;
    }
    // Host loop: one launch per level and a device->host read of the state.
    Ctl* ctl = reinterpret_cast<Ctl*>(h->ws + (size_t)lane * h->L.search + h->L.ctl);
    p.level_budget = 1;
    for (;;) {
        FBC_CUDA(h, cudaLaunchCooperativeKernel(level_kernel_ptr<RowT>(), dim3(grid),
                                                dim3(h->block), args, h->smem, s));
        int state[2] = {0, 0};  // status, done
        FBC_CUDA(h, cudaMemcpyAsync(state, &ctl->status, sizeof(state), cudaMemcpyDeviceToHost, s));
        FBC_CUDA(h, cudaStreamSynchronize(s));
        if (state[0] != BFS_CSR_OK || state[1] != 0)
            break;
    }
    return BFS_CSR_OK;
}

int create_common(bfs_csr_t* h, void* d_workspace, size_t workspace_bytes, cudaStream_t s)
{
    h->lanes = h->opt.lanes > 1 ? h->opt.lanes : 1;
    h->L = make_layout(h->n, h->row_ptr_64, h->lanes, pad_entries_for(h->opt, h->nnz));
    h->words = (int)((h->n + 31) / 32);
    if (d_workspace != nullptr) {
        if (workspace_bytes < h->L.total || (reinterpret_cast<uintptr_t>(d_workspace) & 255u))
            return BFS_CSR_EINVAL;
        h->ws = static_cast<unsigned char*>(d_workspace);
        h->ws_bytes = workspace_bytes;
        h->own_ws = false;
    } else {
        void* p = nullptr;
        FBC_CUDA(h, cudaMalloc(&p, h->L.total));
        h->ws = static_cast<unsigned char*>(p);
        h->ws_bytes = h->L.total;
        h->own_ws = true;
    }
    return h->row_ptr_64 ? prepare<int64_t>(h, s) : prepare<int32_t>(h, s);
}

int validate_shape(int64_t n, int64_t nnz, int row_ptr_64, const bfs_csr_options* opt)
{
    if (n < 1 || n >= (int64_t(1) << 31) || nnz < 0)
        return BFS_CSR_EINVAL;
    if (!row_ptr_64 && nnz >= (int64_t(1) << 31))
        return BFS_CSR_EINVAL;
    if (edge_bits(n, nnz, row_ptr_64) < 0)
        return BFS_CSR_EUNSUPPORTED;
    if (opt != nullptr)
        return check_options(*opt);
    return BFS_CSR_OK;
}

void release(bfs_csr_t* h)
{
    if (h == nullptr)
        return;
    if (h->own_ws && h->ws != nullptr)
        cudaFree(h->ws);
    if (h->d_row_ptr_own) cudaFree(h->d_row_ptr_own);
    if (h->d_col_own) cudaFree(h->d_col_own);
    if (h->d_dist_own) cudaFree(h->d_dist_own);
    if (h->d_parent_own) cudaFree(h->d_parent_own);
    if (h->d_levels_own) cudaFree(h->d_levels_own);
    if (h->d_dist_b) cudaFree(h->d_dist_b);
    if (h->d_parent_b) cudaFree(h->d_parent_b);
    if (h->d_batch) cudaFree(h->d_batch);
    for (int i = 0; i < 2; ++i) {
        if (h->ev_search[i]) cudaEventDestroy(h->ev_search[i]);
        if (h->ev_copy[i]) cudaEventDestroy(h->ev_copy[i]);
    }
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    for (int j = 0; j < kMaxLanes; ++j) {
        if (h->lane_stream[j]) cudaStreamDestroy(h->lane_stream[j]);
        if (h->ev_join[j]) cudaEventDestroy(h->ev_join[j]);
    }
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    for (auto& g : h->graphs) {
        if (g.exec) cudaGraphExecDestroy(g.exec);
        if (g.graph) cudaGraphDestroy(g.graph);
    }
    delete h;
}

int init_handle(bfs_csr_t* h, int64_t n, int64_t nnz, int row_ptr_64, int symmetric,
                const bfs_csr_options* opt)
{
    h->n = n;
    h->nnz = nnz;
    h->row_ptr_64 = row_ptr_64 ? 1 : 0;
    h->symmetric = symmetric ? 1 : 0;
    if (opt != nullptr)
        h->opt = *opt;
    else
        bfs_csr_default_options(&h->opt);
    h->eb = edge_bits(n, nnz, h->row_ptr_64);
    FBC_CUDA(h, cudaGetDevice(&h->device));
    FBC_CUDA(h, cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device));
    FBC_CUDA(h, cudaDeviceGetAttribute(&h->l2_bytes, cudaDevAttrL2CacheSize, h->device));
    int coop = 0;
    FBC_CUDA(h, cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device));
    if (!coop)
        return BFS_CSR_EUNSUPPORTED;
    return BFS_CSR_OK;
}

// Host CSR -> the handle's device copy (same n and nnz), then the checks and
// per-vertex data create derives from it.
int upload_host_csr(bfs_csr_t* h, const void* h_row_ptr, const int32_t* h_col, cudaStream_t s)
{
    const size_t rp_bytes = (size_t)(h->n + 1) * (h->row_ptr_64 ? 8 : 4);
    FBC_CUDA(h, cudaMemcpyAsync(h->d_row_ptr_own, h_row_ptr, rp_bytes, cudaMemcpyHostToDevice, s));
    if (h->nnz > 0)
        FBC_CUDA(h, cudaMemcpyAsync(h->d_col_own, h_col, (size_t)h->nnz * 4,
                                    cudaMemcpyHostToDevice, s));
    // A new CSR: validate it and re-derive the dead bitmap, the non-isolated
    // count and the probe array, as create does.
    return h->row_ptr_64 ? prepare<int64_t>(h, s) : prepare<int32_t>(h, s);
}

}  // namespace

extern "C" {

int bfs_csr_default_options(bfs_csr_options* o)
{
    if (o == nullptr)
        return BFS_CSR_EINVAL;
    std::memset(o, 0, sizeof(*o));
    o->direction = BFS_CSR_DIR_AUTO;
    o->advance = BFS_CSR_ADV_AUTO;
    o->discovery = BFS_CSR_DISC_BITMAP;
    o->loop_mode = BFS_CSR_LOOP_PERSISTENT;
    o->small_max_degree = 32;
    o->cta_min_degree = 256;
    o->merge_path_min_frontier = 4096;
    o->binned_max_degree = 8192;
    o->pull_alpha = 14.0;
    o->push_beta = 24;
    o->max_depth = -1;
    o->validate = 1;
    o->block_threads = 0;
    o->grid_blocks = 0;
    o->barrier_timeout_ns = 10ll * 1000 * 1000 * 1000;
    o->test_unreachable_barrier = 0;
    o->narrow_max_edges = 2048;
    o->lanes = 1;
    return BFS_CSR_OK;
}

int bfs_csr_workspace_bytes(int64_t n, int64_t nnz, int row_ptr_64, const bfs_csr_options* opt,
                            size_t* bytes)
{
    if (bytes == nullptr)
        return BFS_CSR_EINVAL;
    const int rc = validate_shape(n, nnz, row_ptr_64, opt);
    if (rc != BFS_CSR_OK)
        return rc;
    const int lanes = opt != nullptr && opt->lanes > 1 ? opt->lanes : 1;
    bfs_csr_options d;
    bfs_csr_default_options(&d);
    *bytes = make_layout(n, row_ptr_64, lanes, pad_entries_for(opt != nullptr ? *opt : d, nnz)).total;
    return BFS_CSR_OK;
}

int bfs_csr_create(bfs_csr_handle* out, int64_t n, int64_t nnz, const void* d_row_ptr,
                   int row_ptr_64, const int32_t* d_col, int symmetric, void* d_workspace,
                   size_t workspace_bytes, const bfs_csr_options* opt, void* stream)
{
    if (out == nullptr)
        return BFS_CSR_EINVAL;
    *out = nullptr;
    int rc = validate_shape(n, nnz, row_ptr_64, opt);
    if (rc != BFS_CSR_OK)
        return rc;
    if (d_row_ptr == nullptr || (nnz > 0 && d_col == nullptr))
        return BFS_CSR_EINVAL;
    bfs_csr_t* h = new (std::nothrow) bfs_csr_t();
    if (h == nullptr)
        return BFS_CSR_ENOMEM;
    rc = init_handle(h, n, nnz, row_ptr_64, symmetric, opt);
    if (rc == BFS_CSR_OK) {
        h->row_ptr = d_row_ptr;
        h->col = d_col;
        rc = create_common(h, d_workspace, workspace_bytes, as_stream(stream));
    }
    if (rc != BFS_CSR_OK) {
        release(h);
        return rc;
    }
    *out = h;
    return BFS_CSR_OK;
}

int bfs_csr_run_init(bfs_csr_handle h, int64_t source, int32_t* d_dist, int32_t* d_parent,
                     void* stream)
{
    if (h == nullptr || d_dist == nullptr || source < 0 || source >= h->n)
        return BFS_CSR_EINVAL;
    if (h->opt.direction == BFS_CSR_DIR_PULL && !h->symmetric)
        return BFS_CSR_EUNSUPPORTED;
    h->pending_source = -1;
    const int rc = h->row_ptr_64
                       ? launch_init<int64_t>(h, (int32_t)source, d_dist, d_parent, as_stream(stream))
                       : launch_init<int32_t>(h, (int32_t)source, d_dist, d_parent, as_stream(stream));
    if (rc == BFS_CSR_OK) {
        h->pending_source = (int32_t)source;
        h->pending_dist = d_dist;
        h->pending_parent = d_parent;
    }
    h->last_status = rc;
    return rc;
}

int bfs_csr_run_levels(bfs_csr_handle h, int32_t* d_num_levels, void* stream)
{
    if (h == nullptr || h->pending_source < 0)
        return BFS_CSR_EINVAL;
    const int rc = h->row_ptr_64
                       ? launch_levels<int64_t>(h, h->pending_dist, h->pending_parent, d_num_levels,
                                                as_stream(stream))
                       : launch_levels<int32_t>(h, h->pending_dist, h->pending_parent, d_num_levels,
                                                as_stream(stream));
    h->pending_source = -1;
    h->last_status = rc;
    return rc;
}

int bfs_csr_run(bfs_csr_handle h, int64_t source, int32_t* d_dist, int32_t* d_parent,
                int32_t* d_num_levels, void* stream)
{
    const int rc = bfs_csr_run_init(h, source, d_dist, d_parent, stream);
    if (rc != BFS_CSR_OK)
        return rc;
    return bfs_csr_run_levels(h, d_num_levels, stream);
}

int bfs_csr_sync(bfs_csr_handle h, void* stream, int32_t* num_levels)
{
    if (h == nullptr)
        return BFS_CSR_EINVAL;
    cudaStream_t s = as_stream(stream);
    FBC_CUDA(h, cudaStreamSynchronize(s));
    FBC_CUDA(h, cudaGetLastError());
    const Ctl* ctl = reinterpret_cast<const Ctl*>(h->ws + h->L.ctl);
    int state[5] = {0, 0, 0, 0, 0};  // status, done, level, num_levels (+pad)
    FBC_CUDA(h, cudaMemcpy(state, &ctl->status, 4 * sizeof(int), cudaMemcpyDeviceToHost));
    h->last_status = state[0];
    h->last_num_levels = state[3];
    if (num_levels != nullptr)
        *num_levels = state[3];
    if (state[0] == BFS_CSR_OK && state[1] == 0)
        return BFS_CSR_EDEVICE;  // the loop ended without reaching its end state
    return state[0];
}

int bfs_csr_level_stats(bfs_csr_handle h, bfs_csr_level_stat* host_buf, int32_t cap,
                        int32_t* count)
{
    if (h == nullptr || count == nullptr || cap < 0 || (cap > 0 && host_buf == nullptr))
        return BFS_CSR_EINVAL;
    *count = h->last_num_levels;
    int take = h->last_num_levels < cap ? h->last_num_levels : cap;
    if (take > kStatsCap)
        take = kStatsCap;
    if (take > 0)
        FBC_CUDA(h, cudaMemcpy(host_buf, h->ws + h->L.stats,
                               (size_t)take * sizeof(bfs_csr_level_stat), cudaMemcpyDeviceToHost));
    return BFS_CSR_OK;
}

int bfs_csr_create_host(bfs_csr_handle* out, int64_t n, int64_t nnz, const void* h_row_ptr,
                        int row_ptr_64, const int32_t* h_col, int symmetric,
                        const bfs_csr_options* opt, void* stream)
{
    if (out == nullptr)
        return BFS_CSR_EINVAL;
    *out = nullptr;
    int rc = validate_shape(n, nnz, row_ptr_64, opt);
    if (rc != BFS_CSR_OK)
        return rc;
    if (h_row_ptr == nullptr || (nnz > 0 && h_col == nullptr))
        return BFS_CSR_EINVAL;
    bfs_csr_t* h = new (std::nothrow) bfs_csr_t();
    if (h == nullptr)
        return BFS_CSR_ENOMEM;
    cudaStream_t s = as_stream(stream);
    rc = init_handle(h, n, nnz, row_ptr_64, symmetric, opt);
    const size_t rp_bytes = (size_t)(n + 1) * (row_ptr_64 ? 8 : 4);
    const size_t col_bytes = (size_t)(nnz > 0 ? nnz : 1) * 4;
    auto alloc = [&](void** p, size_t b) {
        if (rc != BFS_CSR_OK)
            return;
        const cudaError_t e = cudaMalloc(p, b);
        if (e != cudaSuccess)
            rc = cuda_fail(h, e);
    };
    alloc(&h->d_row_ptr_own, rp_bytes);
    alloc(reinterpret_cast<void**>(&h->d_col_own), col_bytes);
    alloc(reinterpret_cast<void**>(&h->d_dist_own), (size_t)n * 4);
    alloc(reinterpret_cast<void**>(&h->d_parent_own), (size_t)n * 4);
    alloc(reinterpret_cast<void**>(&h->d_levels_own), 4);
    if (rc == BFS_CSR_OK) {
        cudaError_t e = cudaMemcpyAsync(h->d_row_ptr_own, h_row_ptr, rp_bytes,
                                        cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess && nnz > 0)
            e = cudaMemcpyAsync(h->d_col_own, h_col, (size_t)nnz * 4, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess)
            rc = cuda_fail(h, e);
    }
    if (rc == BFS_CSR_OK) {
        h->host_mode = true;
        h->row_ptr = h->d_row_ptr_own;
        h->col = h->d_col_own;
        rc = create_common(h, nullptr, 0, s);
    }
    if (rc != BFS_CSR_OK) {
        release(h);
        return rc;
    }
    *out = h;
    return BFS_CSR_OK;
}

int bfs_csr_run_host(bfs_csr_handle h, int64_t source, const void* h_row_ptr, const int32_t* h_col,
                     int32_t* h_dist, int32_t* h_parent, int32_t* h_num_levels, void* stream)
{
    if (h == nullptr || !h->host_mode || h_dist == nullptr || source < 0 || source >= h->n)
        return BFS_CSR_EINVAL;
    if (h_row_ptr == nullptr && h_col != nullptr)
        return BFS_CSR_EINVAL;
    if (h_row_ptr != nullptr && h->nnz > 0 && h_col == nullptr)
        return BFS_CSR_EINVAL;
    cudaStream_t s = as_stream(stream);
    if (h_row_ptr != nullptr) {
        const int prc = upload_host_csr(h, h_row_ptr, h_col, s);
        if (prc != BFS_CSR_OK)
            return prc;
    }
    int rc = bfs_csr_run(h, source, h->d_dist_own, h_parent ? h->d_parent_own : nullptr,
                         h->d_levels_own, stream);
    if (rc != BFS_CSR_OK)
        return rc;
    FBC_CUDA(h, cudaMemcpyAsync(h_dist, h->d_dist_own, (size_t)h->n * 4, cudaMemcpyDeviceToHost, s));
    if (h_parent != nullptr)
        FBC_CUDA(h, cudaMemcpyAsync(h_parent, h->d_parent_own, (size_t)h->n * 4,
                                    cudaMemcpyDeviceToHost, s));
    int32_t levels = 0;
    rc = bfs_csr_sync(h, stream, &levels);
    if (h_num_levels != nullptr)
        *h_num_levels = levels;
    return rc;
}

int bfs_csr_run_host_batch(bfs_csr_handle h, int32_t num_sources, const int64_t* sources,
                           const void* h_row_ptr, const int32_t* h_col, int32_t* h_dist,
                           int32_t* h_parent, int32_t* h_num_levels, void* stream)
{
    if (h == nullptr || !h->host_mode || num_sources <= 0 || sources == nullptr ||
        h_dist == nullptr)
        return BFS_CSR_EINVAL;
    if (h_row_ptr == nullptr && h_col != nullptr)
        return BFS_CSR_EINVAL;
    if (h_row_ptr != nullptr && h->nnz > 0 && h_col == nullptr)
        return BFS_CSR_EINVAL;
    for (int32_t i = 0; i < num_sources; ++i)
        if (sources[i] < 0 || sources[i] >= h->n)
            return BFS_CSR_EINVAL;
    cudaStream_t s = as_stream(stream);
    const size_t out_bytes = (size_t)h->n * 4;
    // First batch: the second output slot, the copy stream and its events.
    if (h->copy_stream == nullptr) {
        FBC_CUDA(h, cudaMalloc(&h->d_dist_b, out_bytes));
        FBC_CUDA(h, cudaMalloc(&h->d_parent_b, out_bytes));
        FBC_CUDA(h, cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking));
        for (int i = 0; i < 2; ++i) {
            FBC_CUDA(h, cudaEventCreateWithFlags(&h->ev_search[i], cudaEventDisableTiming));
            FBC_CUDA(h, cudaEventCreateWithFlags(&h->ev_copy[i], cudaEventDisableTiming));
        }
    }
    if (num_sources > h->batch_cap) {
        if (h->d_batch != nullptr) {
            FBC_CUDA(h, cudaFree(h->d_batch));
            h->d_batch = nullptr;
            h->batch_cap = 0;
        }
        FBC_CUDA(h, cudaMalloc(&h->d_batch, (size_t)num_sources * 4 * sizeof(int32_t)));
        h->batch_cap = num_sources;
    }
    if (h_row_ptr != nullptr) {
        const int prc = upload_host_csr(h, h_row_ptr, h_col, s);
        if (prc != BFS_CSR_OK)
            return prc;
    }
    int32_t* slot_dist[2] = {h->d_dist_own, h->d_dist_b};
    int32_t* slot_parent[2] = {h->d_parent_own, h->d_parent_b};
    const Ctl* ctl = reinterpret_cast<const Ctl*>(h->ws + h->L.ctl);
    cudaStream_t cs = h->copy_stream;
    // Search i writes slot i % 2 on `stream`; its copy-back runs on the copy
    // stream while search i + 1 runs, and search i + 2 waits for it.
    for (int32_t i = 0; i < num_sources; ++i) {
        const int sl = i & 1;
        if (i >= 2)
            FBC_CUDA(h, cudaStreamWaitEvent(s, h->ev_copy[sl], 0));
        const int rc = bfs_csr_run(h, sources[i], slot_dist[sl],
                                   h_parent != nullptr ? slot_parent[sl] : nullptr, nullptr, s);
        if (rc != BFS_CSR_OK) {
            cudaStreamSynchronize(s);
            cudaStreamSynchronize(cs);
            return rc;
        }
        // The run's end state (status, done, level, level count) for the check below.
        FBC_CUDA(h, cudaMemcpyAsync(h->d_batch + 4 * i, &ctl->status, 4 * sizeof(int32_t),
                                    cudaMemcpyDeviceToDevice, s));
        FBC_CUDA(h, cudaEventRecord(h->ev_search[sl], s));
        FBC_CUDA(h, cudaStreamWaitEvent(cs, h->ev_search[sl], 0));
        FBC_CUDA(h, cudaMemcpyAsync(h_dist + (size_t)i * h->n, slot_dist[sl], out_bytes,
                                    cudaMemcpyDeviceToHost, cs));
        if (h_parent != nullptr)
            FBC_CUDA(h, cudaMemcpyAsync(h_parent + (size_t)i * h->n, slot_parent[sl], out_bytes,
                                        cudaMemcpyDeviceToHost, cs));
        FBC_CUDA(h, cudaEventRecord(h->ev_copy[sl], cs));
    }
    std::vector<int32_t> st((size_t)num_sources * 4);
    FBC_CUDA(h, cudaMemcpyAsync(st.data(), h->d_batch, st.size() * sizeof(int32_t),
                                cudaMemcpyDeviceToHost, s));
    FBC_CUDA(h, cudaStreamSynchronize(s));
    FBC_CUDA(h, cudaStreamSynchronize(cs));
    int first_bad = BFS_CSR_OK;
    for (int32_t i = 0; i < num_sources; ++i) {
        const int status = st[4 * i], done = st[4 * i + 1];
        if (h_num_levels != nullptr)
            h_num_levels[i] = st[4 * i + 3];
        const int r = status != BFS_CSR_OK ? status : (done == 0 ? BFS_CSR_EDEVICE : BFS_CSR_OK);
        if (r != BFS_CSR_OK && first_bad == BFS_CSR_OK)
            first_bad = r;
    }
    h->last_status = st[4 * (num_sources - 1)];
    h->last_num_levels = st[4 * (num_sources - 1) + 3];
    return first_bad;
}

int bfs_csr_run_batch(bfs_csr_handle h, int32_t num_sources, const int64_t* sources,
                      int32_t* d_dist, int32_t* d_parent, int32_t* d_num_levels,
                      int64_t* d_stamps, void* stream)
{
    if (h == nullptr || num_sources <= 0 || sources == nullptr || d_dist == nullptr)
        return BFS_CSR_EINVAL;
    for (int32_t i = 0; i < num_sources; ++i)
        if (sources[i] < 0 || sources[i] >= h->n)
            return BFS_CSR_EINVAL;
    if (h->opt.direction == BFS_CSR_DIR_PULL && !h->symmetric)
        return BFS_CSR_EUNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    const bool concurrent = h->lanes > 1 && h->opt.loop_mode == BFS_CSR_LOOP_PERSISTENT;
    const int lanes = concurrent ? h->lanes : 1;
    if (concurrent && h->ev_fork == nullptr) {
        FBC_CUDA(h, cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming));
        for (int j = 0; j < h->lanes; ++j) {
            FBC_CUDA(h, cudaStreamCreateWithFlags(&h->lane_stream[j], cudaStreamNonBlocking));
            FBC_CUDA(h, cudaEventCreateWithFlags(&h->ev_join[j], cudaEventDisableTiming));
        }
    }
    if (num_sources > h->batch_cap) {
        if (h->d_batch != nullptr) {
            FBC_CUDA(h, cudaFree(h->d_batch));
            h->d_batch = nullptr;
            h->batch_cap = 0;
        }
        FBC_CUDA(h, cudaMalloc(&h->d_batch, (size_t)num_sources * 4 * sizeof(int32_t)));
        h->batch_cap = num_sources;
    }
    // Each lane's level kernel gets an equal share of the cooperative grid.
    const int grid = concurrent ? (h->grid / lanes > 0 ? h->grid / lanes : 1) : h->grid;
    if (concurrent) {
        FBC_CUDA(h, cudaEventRecord(h->ev_fork, s));
        for (int j = 0; j < lanes; ++j)
            FBC_CUDA(h, cudaStreamWaitEvent(h->lane_stream[j], h->ev_fork, 0));
    }
    int rc = BFS_CSR_OK;
    for (int32_t i = 0; i < num_sources && rc == BFS_CSR_OK; ++i) {
        const int j = i % lanes;
        cudaStream_t ls = concurrent ? h->lane_stream[j] : s;
        const size_t row = (size_t)i * (size_t)h->n;
        int32_t* dd = d_dist + row;
        int32_t* dp = d_parent != nullptr ? d_parent + row : nullptr;
        int32_t* dl = d_num_levels != nullptr ? d_num_levels + i : nullptr;
        long long* st = d_stamps != nullptr ? reinterpret_cast<long long*>(d_stamps) + 3 * i
                                            : nullptr;
        rc = h->row_ptr_64 ? launch_init<int64_t>(h, (int32_t)sources[i], dd, dp, ls, j, st)
                           : launch_init<int32_t>(h, (int32_t)sources[i], dd, dp, ls, j, st);
        if (rc == BFS_CSR_OK)
            rc = h->row_ptr_64 ? launch_levels<int64_t>(h, dd, dp, dl, ls, j, grid, st)
                               : launch_levels<int32_t>(h, dd, dp, dl, ls, j, grid, st);
        if (rc == BFS_CSR_OK) {
            // The search's end state (status, done, level, level count).
            const Ctl* cj = reinterpret_cast<const Ctl*>(h->ws + (size_t)j * h->L.search + h->L.ctl);
            const cudaError_t e = cudaMemcpyAsync(h->d_batch + 4 * i, &cj->status,
                                                  4 * sizeof(int32_t), cudaMemcpyDeviceToDevice, ls);
            if (e != cudaSuccess)
                rc = cuda_fail(h, e);
        }
    }
    if (concurrent) {
        for (int j = 0; j < lanes; ++j) {
            cudaError_t e = cudaEventRecord(h->ev_join[j], h->lane_stream[j]);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(s, h->ev_join[j], 0);
            if (e != cudaSuccess && rc == BFS_CSR_OK)
                rc = cuda_fail(h, e);
        }
    }
    std::vector<int32_t> st((size_t)num_sources * 4, 0);
    if (rc == BFS_CSR_OK) {
        cudaError_t e = cudaMemcpyAsync(st.data(), h->d_batch, st.size() * sizeof(int32_t),
                                        cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess)
            rc = cuda_fail(h, e);
    }
    const cudaError_t se = cudaStreamSynchronize(s);
    if (se != cudaSuccess && rc == BFS_CSR_OK)
        rc = cuda_fail(h, se);
    h->last_num_levels = 0;   // batch searches keep no level records
    if (rc != BFS_CSR_OK) {
        h->last_status = rc;
        return rc;
    }
    int first_bad = BFS_CSR_OK;
    for (int32_t i = 0; i < num_sources; ++i) {
        const int status = st[4 * i], done = st[4 * i + 1];
        const int r = status != BFS_CSR_OK ? status : (done == 0 ? BFS_CSR_EDEVICE : BFS_CSR_OK);
        if (r != BFS_CSR_OK && first_bad == BFS_CSR_OK)
            first_bad = r;
    }
    h->last_status = first_bad;
    return first_bad;
}

}  // extern "C"

namespace {

template <typename RowT>
int launch_walk(bfs_csr_t* h, const int32_t* frontier, int32_t size, int32_t repeats,
                int32_t mapping, uint32_t* out, cudaStream_t s)
{
    const RowT* rp = static_cast<const RowT*>(h->row_ptr);
    const int32_t n = (int32_t)h->n;
    switch (mapping) {
    case BFS_CSR_WALK_THREAD:
        fbc::walk_thread_kernel<RowT><<<(size + 255) / 256, 256, 0, s>>>(rp, h->col, n, frontier,
                                                                        size, repeats, out);
        break;
    case BFS_CSR_WALK_WARP: {
        const int64_t threads = (int64_t)size * 32;
        fbc::walk_warp_kernel<RowT><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
            rp, h->col, n, frontier, size, repeats, out);
        break;
    }
    case BFS_CSR_WALK_BINNED:
        fbc::walk_binned_kernel<RowT><<<h->sm_count * 4, 256, 0, s>>>(
            rp, h->col, n, frontier, size, repeats, h->opt.small_max_degree,
            h->opt.cta_min_degree, out);
        break;
    default: {  // BFS_CSR_WALK_EDGE
        // The frontier's degree prefix goes to the lane-0 queue offset
        // arrays, which are consecutive in the workspace and hold at least
        // n + 1 entries together.
        RowT* offs = reinterpret_cast<RowT*>(h->ws + h->L.qoff0);
        fbc::walk_prefix_kernel<RowT><<<1, 1024, 0, s>>>(rp, n, frontier, size, offs, out);
        FBC_CUDA(h, cudaGetLastError());
        fbc::walk_edge_kernel<RowT><<<h->sm_count * 8, 256, 0, s>>>(rp, h->col, n, frontier, size,
                                                                    repeats, offs, out);
        break;
    }
    }
    FBC_CUDA(h, cudaGetLastError());
    return BFS_CSR_OK;
}

}  // namespace

extern "C" {

int bfs_csr_walk(bfs_csr_handle h, const int32_t* d_frontier, int32_t frontier_size,
                 int32_t repeats, int32_t mapping, uint32_t* d_out, void* stream)
{
    if (h == nullptr || frontier_size < 0 || (int64_t)frontier_size > h->n || repeats < 0 ||
        mapping < BFS_CSR_WALK_THREAD || mapping > BFS_CSR_WALK_EDGE)
        return BFS_CSR_EINVAL;
    if (frontier_size == 0)
        return BFS_CSR_OK;
    if (d_frontier == nullptr || d_out == nullptr)
        return BFS_CSR_EINVAL;
    cudaStream_t s = as_stream(stream);
    return h->row_ptr_64 ? launch_walk<int64_t>(h, d_frontier, frontier_size, repeats, mapping,
                                                d_out, s)
                         : launch_walk<int32_t>(h, d_frontier, frontier_size, repeats, mapping,
                                                d_out, s);
}

int bfs_csr_destroy(bfs_csr_handle h)
{
    if (h == nullptr)
        return BFS_CSR_EINVAL;
    release(h);
    return BFS_CSR_OK;
}

const char* bfs_csr_status_string(int status)
{
    switch (status) {
    case BFS_CSR_OK: return "ok";
    case BFS_CSR_EINVAL: return "invalid argument or malformed CSR";
    case BFS_CSR_ENOMEM: return "out of memory";
    case BFS_CSR_ECUDA: return "CUDA error";
    case BFS_CSR_ETIMEOUT: return "a device-wide wait timed out";
    case BFS_CSR_EUNSUPPORTED: return "unsupported option or size";
    case BFS_CSR_EDEVICE: return "device-side check failed";
    default: return "unknown status";
    }
}

int bfs_csr_last_cuda_error(bfs_csr_handle h)
{
    return h == nullptr ? 0 : h->last_cuda_error;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The allocation-free variant. Its scratch is one device array of the library
// itself, laid out exactly like a handle's workspace for the largest graph it
// accepts; the host side keeps nothing but that array's per-device address.

namespace {

constexpr int64_t kNoAllocMaxN = BFS_CSR_NOALLOC_MAX_VERTICES;

// Upper bound of make_layout(kNoAllocMaxN, 0).total: every region rounded up
// to 256 bytes.
constexpr size_t kNoAllocBytes =
    (sizeof(Ctl) + 256) + 4 * ((size_t)kNoAllocMaxN / 8 + 256) +
    ((size_t)kNoAllocMaxN * 4 + 256) + ((size_t)kNoAllocMaxN + 256) +
    3 * ((size_t)kNoAllocMaxN * 4 + 256) + 4 * ((size_t)kNoAllocMaxN * 4 + 256) +
    ((size_t)kStatsCap * sizeof(bfs_csr_level_stat) + 256);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::atomic<void*> g_noalloc_addr[kNoAllocMaxDevices];

// Device address of the scratch array on the current device (looked up once
// per device; a host-side stand-in is never passed to a kernel).
int noalloc_scratch(int device, void** out)
{
    if (device < 0 || device >= kNoAllocMaxDevices)
        return BFS_CSR_EUNSUPPORTED;
    void* p = g_noalloc_addr[device].load(std::memory_order_acquire);
    if (p == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return BFS_CSR_ECUDA;
        g_noalloc_addr[device].store(p, std::memory_order_release);
    }
    *out = p;
    return BFS_CSR_OK;
}

}  // namespace

extern "C" int bfs_csr_run_noalloc(int64_t n, int64_t nnz, const int32_t* d_row_ptr,
                                   const int32_t* d_col, int symmetric, int64_t source,
                                   int32_t* d_dist, int32_t* d_parent, int32_t* d_num_levels,
                                   int32_t* num_levels, const bfs_csr_options* opt, void* stream)
{
    if (n > kNoAllocMaxN)
        return BFS_CSR_EUNSUPPORTED;
    int rc = validate_shape(n, nnz, 0, opt);
    if (rc != BFS_CSR_OK)
        return rc;
    if (d_row_ptr == nullptr || (nnz > 0 && d_col == nullptr) || d_dist == nullptr ||
        source < 0 || source >= n)
        return BFS_CSR_EINVAL;
    bfs_csr_t h;  // on the stack: nothing is allocated
    rc = init_handle(&h, n, nnz, 0, symmetric, opt);
    if (rc != BFS_CSR_OK)
        return rc;
    if (h.opt.direction == BFS_CSR_DIR_PULL && !h.symmetric)
        return BFS_CSR_EUNSUPPORTED;
    if (h.opt.lanes > 1)
        return BFS_CSR_EUNSUPPORTED;  // the scratch array holds one search's state
    if (h.opt.loop_mode == BFS_CSR_LOOP_GRAPH)
        return BFS_CSR_EUNSUPPORTED;  // a graph is a resource this entry point cannot keep
    if (h.opt.frontier_output != BFS_CSR_FRONTIER_COMPACT)
        return BFS_CSR_EUNSUPPORTED;  // the padded arrays (nnz entries each) do not fit the scratch
    void* scratch = nullptr;
    rc = noalloc_scratch(h.device, &scratch);
    if (rc != BFS_CSR_OK)
        return rc;
    h.row_ptr = d_row_ptr;
    h.col = d_col;
    h.L = make_layout(n, 0);
    if (h.L.total > kNoAllocBytes)
        return BFS_CSR_EUNSUPPORTED;
    h.words = (int)((n + 31) / 32);
    h.ws = static_cast<unsigned char*>(scratch);
    h.ws_bytes = kNoAllocBytes;
    h.own_ws = false;
    cudaStream_t s = as_stream(stream);
    rc = prepare<int32_t>(&h, s);  // clears the control block, validates, dead bitmap
    if (rc == BFS_CSR_OK)
        rc = launch_init<int32_t>(&h, (int32_t)source, d_dist, d_parent, s);
    if (rc == BFS_CSR_OK)
        rc = launch_levels<int32_t>(&h, d_dist, d_parent, d_num_levels, s);
    if (rc != BFS_CSR_OK)
        return rc;
    int32_t levels = 0;
    rc = bfs_csr_sync(&h, stream, &levels);
    if (num_levels != nullptr)
        *num_levels = levels;
    return rc;
}
