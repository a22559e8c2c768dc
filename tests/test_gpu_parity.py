"""GPU parity: the CUDA path through the C-ABI against the CPU oracle.

dist must equal the oracle's bit for bit (BFS distances are unique); parent
must be a valid BFS tree (checked by the oracle's checker, since several
trees are correct); the level count and the per-level frontier sizes must
equal the oracle's (the sizes summing to the reached count is the gate that
catches a vertex queued twice, "100 Days of GPU, Day 38", "Pitfalls").
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import graphgen
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fbc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import frontier_bfs_csr_gb300
    return frontier_bfs_csr_gb300


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def check_against_oracle(fbc, g, sources, bfs=None, max_depth=-1, stats=True):
    """Run each source on the GPU and compare with the oracle."""
    own = bfs is None
    if own:
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), symmetric=g.symmetric)
    for s in sources:
        s = int(s)
        dist, parent, levels = bfs.search(s)
        dist_h = dist.cpu().numpy()
        parent_h = parent.cpu().numpy()
        want, _, want_levels = oracle.bfs(g.row_ptr, g.col, s, max_depth=max_depth,
                                          want_parent=False)
        if not np.array_equal(dist_h, want):
            bad = np.nonzero(dist_h != want)[0]
            raise AssertionError("%s source %d: dist differs at %d vertices, first %d "
                                 "(gpu %d, oracle %d)" % (g.name, s, bad.size, bad[0],
                                                          dist_h[bad[0]], want[bad[0]]))
        assert levels == want_levels, (g.name, s, levels, want_levels)
        code, where = oracle.check_parent(g.row_ptr, g.col, s, dist_h, parent_h)
        assert code == 0, "%s source %d: invalid parent at %d" % (g.name, s, where)
        if stats:
            sizes, _, reached, _ = oracle.level_sizes(g.row_ptr, want)
            rec = bfs.level_stats()
            assert len(rec) == want_levels
            got = [r["frontier"] for r in rec]
            assert got == sizes.tolist(), (g.name, s)
            assert sum(got) == reached
            # m_F of every level (after a pull level the kernel derives it
            # from the edges the pull left unvisited)
            deg = np.diff(g.row_ptr.astype(np.int64))
            want_mf = [int(deg[want == k].sum()) for k in range(want_levels)]
            assert [r["frontier_edges"] for r in rec] == want_mf, (g.name, s)
    if own:
        bfs.close()


def check_rows_against_oracle(g, srcs, dist_rows, parent_rows, levels):
    """Row i of dist_rows/parent_rows (host arrays) and levels[i] are source
    srcs[i]'s search. Every row is compared element by element with the
    oracle's distances and every parent row is tree-checked; the oracle runs
    for several sources at once (its ctypes calls release the GIL)."""
    def one(i):
        s = int(srcs[i])
        want, _, want_levels = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
        d = dist_rows[i]
        bad = np.nonzero(d != want)[0]
        first = (int(bad[0]), int(d[bad[0]]), int(want[bad[0]])) if bad.size else None
        pcode, pwhere = (oracle.check_parent(g.row_ptr, g.col, s, d, parent_rows[i])
                         if parent_rows is not None else (0, -1))
        return s, bad.size, first, int(levels[i]), want_levels, pcode, pwhere

    workers = max(1, min(16, os.cpu_count() or 1, len(srcs)))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(one, range(len(srcs))))
    for s, nbad, first, lev, want_levels, pcode, pwhere in results:
        assert nbad == 0, "%s source %d: dist differs at %d vertices, first (v, gpu, oracle) %s" % (
            g.name, s, nbad, first)
        assert lev == want_levels, (g.name, s, lev, want_levels)
        assert pcode == 0, "%s source %d: invalid parent at %d" % (g.name, s, pwhere)


def run_batch_rows(fbc, g, srcs, lanes, **over):
    """bfs_csr_run_batch over srcs on `lanes` lanes; host copies of the rows."""
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), symmetric=g.symmetric,
                     options=fbc.default_options(lanes=lanes, **over))
    k = len(srcs)
    dist = torch.empty((k, g.n), dtype=torch.int32, device="cuda")
    parent = torch.empty_like(dist)
    levels = torch.empty(k, dtype=torch.int32, device="cuda")
    bfs.run_batch([int(s) for s in srcs], dist, parent, levels)
    out = dist.cpu().numpy(), parent.cpu().numpy(), levels.cpu().numpy()
    bfs.close()
    del dist, parent, levels
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- goldens

def test_six_vertex_directed_golden(fbc, golden):
    gx = golden("six_vertex_directed.json")
    g = graphgen.from_csr(np.array(gx["row_ptr"], np.int32), np.array(gx["col"], np.int32),
                          symmetric=False, name="six")
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), symmetric=False)
    dist, parent, levels = bfs.search(0)
    assert dist.cpu().tolist() == gx["dist"]
    assert levels == gx["num_levels"]
    assert oracle.check_parent(g.row_ptr, g.col, 0, dist.cpu().numpy(), parent.cpu().numpy())[0] == 0
    assert [r["frontier"] for r in bfs.level_stats()] == [len(f) for f in gx["levels"]]
    bfs.close()
    opt = fbc.default_options(max_depth=gx["after_level_1"]["max_depth"])
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), symmetric=False, options=opt)
    dist, _, levels = bfs.search(0)
    assert dist.cpu().tolist() == gx["after_level_1"]["dist"] and levels == 3
    bfs.close()


def test_four_vertex_golden(fbc, golden):
    gx = golden("four_vertex_undirected.json")
    rp, col = np.array(gx["row_ptr"], np.int32), np.array(gx["col"], np.int32)
    for direction in (fbc.BFS_CSR_DIR_PUSH, fbc.BFS_CSR_DIR_PULL, fbc.BFS_CSR_DIR_AUTO):
        bfs = fbc.BfsCsr(_dev(rp), _dev(col), True, fbc.default_options(direction=direction))
        for s, want in gx["dist_from"].items():
            dist, parent, levels = bfs.search(int(s))
            assert dist.cpu().tolist() == want and levels == max(want) + 1
            assert oracle.check_parent(rp, col, int(s), dist.cpu().numpy(),
                                       parent.cpu().numpy())[0] == 0
        bfs.close()


# ---------------------------------------------------------------- small graphs

def test_random_small_graphs_every_source(fbc):
    for k in range(120):
        n = 1 + (k % 12)
        directed = bool(k % 2)
        g = graphgen.random_graph(n, [0.15, 0.3, 0.5][k % 3], 300 + k, directed=directed,
                                  loops=directed and k % 3 == 0)
        check_against_oracle(fbc, g, range(n))


def test_many_back_to_back_small_searches(fbc):
    """Tiny searches finish in a few microseconds, so CTAs that start late
    overlap with CTA 0's single-CTA levels. Many in a row, every direction,
    must all end correctly (a slot race between them once surfaced as a
    barrier timeout)."""
    graphs = [graphgen.from_csr(np.array([0, 2, 4, 7, 8], np.int32),
                                np.array([1, 2, 0, 2, 0, 1, 3, 2], np.int32), True),
              graphgen.path_graph(9), graphgen.star_graph(17), graphgen.clique_graph(5)]
    for g in graphs:
        for direction in (0, 1, 2):
            bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True,
                             fbc.default_options(direction=direction,
                                                 barrier_timeout_ns=2_000_000_000))
            want = [oracle.bfs(g.row_ptr, g.col, s, want_parent=False) for s in range(g.n)]
            for rep in range(25):
                for s in range(g.n):
                    dist, _, levels = bfs.search(s, want_parent=False)
                    assert np.array_equal(dist.cpu().numpy(), want[s][0]), (g.name, s, rep)
                    assert levels == want[s][2]
            bfs.close()


def test_corner_cases(fbc):
    cases = [
        (graphgen.from_edges(1, [], []), [0]),
        (graphgen.from_edges(5, [], []), [0, 4]),
        (graphgen.from_edges(6, [0, 3], [1, 4]), [0, 2, 3, 5]),
        (graphgen.path_graph(2000), [0, 1000, 1999]),
        (graphgen.star_graph(5000), [0, 17]),
        (graphgen.clique_graph(64), [0, 63]),
        (graphgen.grid(30, 50, 0.0, 0), [0, 777]),
    ]
    for g, srcs in cases:
        check_against_oracle(fbc, g, srcs)


def test_distances_past_the_hop_byte(fbc):
    """Distances of 126 and more do not fit the hop code's 7 distance bits and
    go to dist directly (the code's top bit flags a probe-neighbour parent);
    here they are reached by push and by pull levels: a 300-vertex path ends
    in a dense random cluster (so the automatic rule pulls at depth ~300),
    plus isolated vertices; every direction mode, with parents stored at
    discovery and written by the end-of-search pass."""
    rng = np.random.default_rng(17)
    path = 300
    cl = 4000
    src = list(range(path - 1))
    dst = list(range(1, path))
    a = rng.integers(path, path + cl, 60000)
    b = rng.integers(path, path + cl, 60000)
    src += [path - 1] * 8 + a.tolist()
    dst += rng.integers(path, path + cl, 8).tolist() + b.tolist()
    g = graphgen.from_edges(path + cl + 50, src, dst, name="path_then_cluster")
    for over in (dict(), dict(direction=1), dict(direction=2), dict(loop_mode=1),
                 dict(parent_pass=1), dict(parent_pass=1, direction=2)):
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), symmetric=True,
                         options=fbc.default_options(**over))
        check_against_oracle(fbc, g, [150, path + 5, 0], bfs=bfs)  # source 0 last: its records
        rec = bfs.level_stats()
        if over.get("direction", 0) != 1:
            assert any(r["direction"] == fbc.BFS_CSR_DIR_PULL and r["level"] >= 126
                       for r in rec), over
        bfs.close()


def test_self_loops_and_duplicate_edges(fbc):
    rng = np.random.default_rng(5)
    src = rng.integers(0, 300, 3000)
    dst = rng.integers(0, 300, 3000)
    g = graphgen.from_edges(300, src, dst, symmetric=False, drop_loops=False, dedupe=False)
    assert (np.repeat(np.arange(300), np.diff(g.row_ptr)) == g.col).any()
    check_against_oracle(fbc, g, [0, 5, 299])
    gs = graphgen.from_edges(300, np.concatenate([src, dst]), np.concatenate([dst, src]),
                             symmetric=False, drop_loops=False, dedupe=False)
    gs.symmetric = True  # every edge is present in both directions
    check_against_oracle(fbc, gs, [0, 5, 299])


def test_int64_row_ptr(fbc):
    g = graphgen.rmat(12, 8, 11, row_ptr_64=True)
    assert g.row_ptr.dtype == np.int64
    check_against_oracle(fbc, g, graphgen.pick_sources(g, 6, 11))


# ---------------------------------------------------------------- configs

def test_config1_all_sources(fbc):
    g = graphgen.config(1)
    deg = g.degrees()
    cand = np.nonzero(deg)[0]
    ecc = [(oracle.bfs(g.row_ptr, g.col, int(s), want_parent=False)[2], int(s)) for s in cand]
    best = max(ecc, key=lambda t: (t[0], -t[1]))[1]
    check_against_oracle(fbc, g, [best] + list(g.sources))


@pytest.mark.parametrize("cfg", [2, 3])
def test_configs_2_and_3_every_source(fbc, cfg):
    """All 64 sources of the uniform random graph and of R-MAT scale 22: the
    batch path on two lanes (the benchmark's configuration) element by
    element against the oracle, every parent row tree-checked; the first
    six also through single runs with their per-level records."""
    g = graphgen.config(cfg)
    assert len(g.sources) == 64
    check_against_oracle(fbc, g, g.sources[:6])
    dist, parent, levels = run_batch_rows(fbc, g, g.sources, lanes=2)
    check_rows_against_oracle(g, g.sources, dist, parent, levels)


def test_config4_grid_corner(fbc):
    g = graphgen.config(4)
    check_against_oracle(fbc, g, g.sources[:1])
    dist, parent, levels = run_batch_rows(fbc, g, g.sources[:1], lanes=1)
    check_rows_against_oracle(g, g.sources[:1], dist, parent, levels)


def test_large_level_paths_on_rmat22(fbc):
    """The paths that only large levels take, shown to run and checked
    against the oracle on R-MAT scale 22: with pushes only, merge-path levels
    of at least 2^20 frontier edges (winners staged as ids, their queue built
    after a grid barrier); by default, a pull level right after a push whose
    queue holds at least n/64 vertices (frontier bitmap from the hop codes)."""
    g = graphgen.config(3)
    srcs = g.sources[:3]
    for over, want in ((dict(direction=1, advance=2), "ids"), (dict(), "hop")):
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, fbc.default_options(**over))
        check_against_oracle(fbc, g, srcs, bfs=bfs)
        seen = False
        for s in srcs:
            bfs.search(int(s))
            rec = bfs.level_stats()
            for a, b in zip(rec, rec[1:]):
                if want == "ids":
                    seen |= (a["direction"] == fbc.BFS_CSR_DIR_PUSH and
                             a["advance"] == fbc.BFS_CSR_ADV_MERGE_PATH and
                             a["frontier_edges"] >= 1 << 20)
                else:
                    seen |= (a["direction"] == fbc.BFS_CSR_DIR_PUSH and
                             b["direction"] == fbc.BFS_CSR_DIR_PULL and
                             64 * b["frontier"] >= g.n)
        bfs.close()
        assert seen, want


def test_config5_rmat25_single_runs(fbc):
    """R-MAT scale 25 (int64 row_ptr) through single runs: dist, parent,
    level count and per-level records of two sources against the oracle."""
    g = graphgen.config(5)
    assert g.row_ptr.dtype == np.int64 and g.n == 1 << 25
    check_against_oracle(fbc, g, g.sources[:2])


def test_config5_rmat25_every_source_on_two_lanes(fbc):
    """The benchmark's step at full size: bfs_csr_run_batch with two lanes
    over all 16 sources of R-MAT scale 25; every dist row equal to the
    oracle's element by element, every parent row a valid BFS tree, every
    level count equal to the oracle's."""
    g = graphgen.config(5)
    assert len(g.sources) == 16
    dist, parent, levels = run_batch_rows(fbc, g, g.sources, lanes=2)
    check_rows_against_oracle(g, g.sources, dist, parent, levels)


# ---------------------------------------------------------------- option matrix

OPTION_MATRIX = [
    dict(direction=1, advance=1), dict(direction=1, advance=2), dict(direction=2),
    dict(direction=0, advance=1), dict(direction=0, advance=2), dict(discovery=1),
    dict(discovery=1, direction=1, advance=2), dict(loop_mode=1), dict(loop_mode=1, direction=1),
    dict(block_threads=64), dict(block_threads=256, advance=2), dict(grid_blocks=1),
    dict(grid_blocks=3, advance=1), dict(grid_blocks=7, advance=2, direction=1),
    dict(small_max_degree=1, cta_min_degree=2, advance=1),
    dict(small_max_degree=4, cta_min_degree=64, advance=1, direction=1),
    dict(merge_path_min_frontier=0), dict(merge_path_min_frontier=100000, binned_max_degree=64),
    dict(pull_alpha=0.0), dict(pull_alpha=1e9),
    dict(push_beta=0), dict(push_beta=1000000, pull_alpha=1.0),
    dict(narrow_max_edges=0), dict(narrow_max_edges=8), dict(narrow_max_edges=2048, advance=2),
    dict(narrow_max_edges=100000, block_threads=128), dict(narrow_max_edges=64, discovery=1),
    dict(loop_mode=2), dict(loop_mode=2, direction=1, advance=1), dict(loop_mode=2, direction=2),
    dict(loop_mode=2, discovery=1),
    dict(parent_pass=1), dict(parent_pass=1, direction=2), dict(parent_pass=1, loop_mode=1),
    dict(parent_pass=1, block_threads=64, grid_blocks=3), dict(parent_pass=2),
    dict(parent_pass=1, discovery=1),
    dict(discovery=2), dict(discovery=2, direction=1, advance=2), dict(discovery=2, direction=2),
    dict(discovery=2, loop_mode=1, advance=1),
    dict(frontier_output=1), dict(frontier_output=1, discovery=2),
    dict(frontier_output=1, grid_blocks=3, direction=1), dict(frontier_output=2),
    dict(frontier_output=2, discovery=2), dict(frontier_output=2, loop_mode=1, discovery=1),
    dict(frontier_output=2, grid_blocks=1),
]


@pytest.mark.parametrize("over", OPTION_MATRIX, ids=lambda d: ",".join(
    "%s=%s" % kv for kv in sorted(d.items())))
def test_option_matrix(fbc, over):
    opt = fbc.default_options(**over)
    for cfg in (1, 3):
        g = graphgen.config(cfg)
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, opt)
        check_against_oracle(fbc, g, g.sources[:3], bfs=bfs)
        bfs.close()
    g = graphgen.random_graph(11, 0.3, 42, directed=True)
    if over.get("direction") != 2:
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), False, opt)
        check_against_oracle(fbc, g, range(11), bfs=bfs)
        bfs.close()


@pytest.mark.parametrize("depth", [0, 1, 2, 3, 5])
def test_depth_bound_with_level_records(fbc, depth):
    """max_depth = d: dist matches the oracle's depth-bounded search, the
    level count includes the last (unexpanded) frontier F_d, and its record
    has direction 0 and the right size."""
    for cfg in (1, 3):
        g = graphgen.config(cfg)
        for over in (dict(), dict(direction=1), dict(narrow_max_edges=0)):
            opt = fbc.default_options(max_depth=depth, **over)
            bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, opt)
            check_against_oracle(fbc, g, g.sources[:2], bfs=bfs, max_depth=depth)
            rec = bfs.level_stats()
            want, _, levels = oracle.bfs(g.row_ptr, g.col, int(g.sources[1]), max_depth=depth,
                                         want_parent=False)
            if levels == depth + 1:
                assert rec[-1]["direction"] == 0 and rec[-1]["level"] == depth
                assert rec[-1]["frontier"] == int((want == depth).sum())
            assert all(r["direction"] in (1, 2) for r in rec[:levels - 1])
            bfs.close()


def test_graph_loop_mode(fbc):
    """The CUDA-graph level loop (a device-driven while node, one level per
    body launch): the 2048 x 2048 grid (4,094 levels), a 3,000-level path,
    the power-law graph from several sources into different outputs (one
    graph per output set, reused on repeats), a depth bound, and a batch."""
    opt = fbc.default_options(loop_mode=fbc.BFS_CSR_LOOP_GRAPH)
    for g, srcs in ((graphgen.config(4), graphgen.config(4).sources[:1]),
                    (graphgen.path_graph(3000), [0, 2999, 1500])):
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, opt)
        check_against_oracle(fbc, g, srcs, bfs=bfs)
        bfs.close()
    g = graphgen.config(1)
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, opt)
    outs = [torch.empty(g.n, dtype=torch.int32, device="cuda") for _ in range(3)]
    for rep in range(3):
        for i, s in enumerate(g.sources[:3]):
            bfs.run(int(s), outs[i])
            bfs.sync()
    for i, s in enumerate(g.sources[:3]):
        want = oracle.bfs(g.row_ptr, g.col, int(s), want_parent=False)[0]
        assert np.array_equal(outs[i].cpu().numpy(), want)
    bfs.close()
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True,
                     fbc.default_options(loop_mode=fbc.BFS_CSR_LOOP_GRAPH, max_depth=3))
    check_against_oracle(fbc, g, g.sources[:2], bfs=bfs, max_depth=3)
    bfs.close()
    dist, parent, levels = run_batch_rows(fbc, g, g.sources[:6], lanes=2,
                                          loop_mode=fbc.BFS_CSR_LOOP_GRAPH)
    check_rows_against_oracle(g, g.sources[:6], dist, parent, levels)


def test_padded_frontier_records(fbc):
    """The sentinel-padded frontier without a filter: every level is a push
    level walked one thread per slot (advance code BFS_CSR_ADV_PADDED), and
    with the filter a push level takes the merge path and never the
    single-CTA mode; both agree with the oracle on the power-law graph and
    the grid."""
    for cfg in (1, 4):
        g = graphgen.config(cfg)
        for fo, disc in ((2, 2), (1, 2), (2, 0)):
            bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True,
                             fbc.default_options(frontier_output=fo, discovery=disc))
            check_against_oracle(fbc, g, g.sources[:2], bfs=bfs)
            rec = bfs.level_stats()
            if fo == 2:
                assert all(r["direction"] == fbc.BFS_CSR_DIR_PUSH and
                           r["advance"] == fbc.BFS_CSR_ADV_PADDED for r in rec)
            else:
                assert all(r["advance"] != fbc.BFS_CSR_ADV_SINGLE_CTA for r in rec)
            bfs.close()


def test_stage_overflow_path(fbc):
    """One CTA, binned advance: a level where 3,000 frontier vertices each
    discover 20 new leaves overflows the shared-memory stage; the overflow
    vertices must be appended, never dropped (the privatised queue of the
    PMPP ch. 15 notes, section 15.6, drops them)."""
    hub, mids, leaves = 0, np.arange(1, 3001), 20
    src = [np.zeros(3000, np.int64)]
    dst = [mids]
    nxt = 3001
    for m in mids:
        src.append(np.full(leaves, m))
        dst.append(np.arange(nxt, nxt + leaves))
        nxt += leaves
    g = graphgen.from_edges(nxt, np.concatenate(src), np.concatenate(dst))
    for over in (dict(grid_blocks=1, advance=1), dict(grid_blocks=1, advance=2),
                 dict(grid_blocks=2, direction=1, advance=1, small_max_degree=8,
                      cta_min_degree=16)):
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, fbc.default_options(**over))
        check_against_oracle(fbc, g, [hub, 5], bfs=bfs)
        bfs.close()


# ---------------------------------------------------------------- API behaviour

def test_errors(fbc):
    g = graphgen.config(1)
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True)
    dist = torch.empty(g.n, dtype=torch.int32, device="cuda")
    for bad_src in (-1, g.n, g.n + 100):
        with pytest.raises(fbc.BfsError) as e:
            bfs.run(bad_src, dist)
        assert e.value.status == fbc.BFS_CSR_EINVAL
    bfs.close()
    rp = g.row_ptr.copy()
    rp[10], rp[11] = rp[11], rp[10] - 1  # non-monotone
    with pytest.raises(fbc.BfsError) as e:
        fbc.BfsCsr(_dev(rp), _dev(g.col), True)
    assert e.value.status == fbc.BFS_CSR_EINVAL
    col = g.col.copy()
    col[7] = g.n  # out of range
    with pytest.raises(fbc.BfsError) as e:
        fbc.BfsCsr(_dev(g.row_ptr), _dev(col), True)
    assert e.value.status == fbc.BFS_CSR_EINVAL
    # a CTA size above the level kernel's bound for int32 row offsets (384)
    with pytest.raises(fbc.BfsError) as e:
        fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, fbc.default_options(block_threads=512))
    assert e.value.status == fbc.BFS_CSR_EINVAL
    d = graphgen.random_graph(8, 0.4, 3, directed=True)
    bfs = fbc.BfsCsr(_dev(d.row_ptr), _dev(d.col), False, fbc.default_options(direction=2))
    with pytest.raises(fbc.BfsError) as e:
        bfs.run(0, torch.empty(8, dtype=torch.int32, device="cuda"))
    assert e.value.status == fbc.BFS_CSR_EUNSUPPORTED
    bfs.close()


def test_barrier_timeout_is_reported_and_recoverable(fbc):
    """A barrier that waits for one CTA more than exists must give up after
    the time limit, report BFS_CSR_ETIMEOUT, and leave the context usable."""
    g = graphgen.config(1)
    opt = fbc.default_options(test_unreachable_barrier=1, barrier_timeout_ns=50_000_000)
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, opt)
    dist = torch.empty(g.n, dtype=torch.int32, device="cuda")
    bfs.run(int(g.sources[0]), dist)
    with pytest.raises(fbc.BfsError) as e:
        bfs.sync()
    assert e.value.status == fbc.BFS_CSR_ETIMEOUT
    bfs.close()
    check_against_oracle(fbc, g, g.sources[:2])


def test_output_without_parent_and_device_level_count(fbc):
    g = graphgen.config(1)
    bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True)
    s = int(g.sources[1])
    dist = torch.empty(g.n, dtype=torch.int32, device="cuda")
    nl = torch.zeros(1, dtype=torch.int32, device="cuda")
    bfs.run(s, dist, None, nl)
    levels = bfs.sync()
    want, _, want_levels = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
    assert np.array_equal(dist.cpu().numpy(), want)
    assert levels == want_levels == int(nl.item())
    bfs.close()


def test_caller_workspace_and_streams(fbc):
    g = graphgen.config(1)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        bfs = fbc.BfsCsr(_dev(g.row_ptr), _dev(g.col), True, stream=stream)
        outs = []
        for s in g.sources[:4]:
            dist = torch.empty(g.n, dtype=torch.int32, device="cuda")
            bfs.run(int(s), dist, stream=stream)
            bfs.sync(stream)
            outs.append(dist.cpu().numpy())
    for s, d in zip(g.sources[:4], outs):
        assert np.array_equal(d, oracle.bfs(g.row_ptr, g.col, int(s), want_parent=False)[0])
    bfs.close()


def test_host_memory_api(fbc):
    g = graphgen.config(1)
    h = fbc.BfsCsrHost(g.row_ptr, g.col, True)
    for s in g.sources[:4]:
        dist = np.empty(g.n, np.int32)
        parent = np.empty(g.n, np.int32)
        levels = h.run(int(s), dist, parent, row_ptr=g.row_ptr, col=g.col)
        want, _, want_levels = oracle.bfs(g.row_ptr, g.col, int(s), want_parent=False)
        assert np.array_equal(dist, want) and levels == want_levels
        assert oracle.check_parent(g.row_ptr, g.col, int(s), dist, parent)[0] == 0
        levels = h.run(int(s), dist)  # resident CSR, no parent
        assert np.array_equal(dist, want) and levels == want_levels
    h.close()


def test_host_memory_batch(fbc):
    """bfs_csr_run_host_batch: row i of the outputs is source i's search (odd
    and even batch sizes exercise both output slots), with and without a CSR
    re-upload, parent and level counts; bad arguments run nothing."""
    for cfg in (1, 3):
        g = graphgen.config(cfg)
        h = fbc.BfsCsrHost(g.row_ptr, g.col, True)
        for k in (1, 2, 3, 5):
            srcs = [int(x) for x in g.sources[:k]][::-1]
            dist = np.full((k, g.n), -7, np.int32)
            par = np.full((k, g.n), -7, np.int32)
            lev = np.zeros(k, np.int32)
            up = k == 3
            h.run_batch(srcs, dist, par, lev, row_ptr=g.row_ptr if up else None,
                        col=g.col if up else None)
            for i, s in enumerate(srcs):
                want, _, want_levels = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
                assert np.array_equal(dist[i], want), (cfg, k, i)
                assert lev[i] == want_levels
                assert oracle.check_parent(g.row_ptr, g.col, s, dist[i], par[i])[0] == 0
        dist = np.empty((2, g.n), np.int32)
        h.run_batch(g.sources[:2], dist)
        for i in range(2):
            want, _, _ = oracle.bfs(g.row_ptr, g.col, int(g.sources[i]), want_parent=False)
            assert np.array_equal(dist[i], want)
        for bad in ([], [g.n], [-1]):
            with pytest.raises(fbc.BfsError):
                h.run_batch(bad, np.empty((len(bad), g.n), np.int32))
        h.close()


def test_device_batch_on_concurrent_lanes(fbc):
    """bfs_csr_run_batch: row i is source i's search whatever lane ran it
    (1, 2 and 3 lanes, odd and even batch sizes, with and without parent),
    equal to the oracle; the device stamps are ordered per search; the host
    loop mode runs the batch one search at a time; bad arguments run
    nothing."""
    for cfg in (1, 3):
        g = graphgen.config(cfg)
        rp, col = _dev(g.row_ptr), _dev(g.col)
        for lanes, extra in ((1, {}), (2, {}), (3, {}), (2, dict(loop_mode=1)),
                             (2, dict(direction=2))):
            bfs = fbc.BfsCsr(rp, col, True, options=fbc.default_options(lanes=lanes, **extra))
            for k in (1, 5, 8):
                srcs = [int(x) for x in g.sources[:k]][::-1]
                dist = torch.full((k, g.n), -7, dtype=torch.int32, device="cuda")
                par = torch.full((k, g.n), -7, dtype=torch.int32, device="cuda")
                lev = torch.zeros(k, dtype=torch.int32, device="cuda")
                stamps = torch.zeros(3 * k, dtype=torch.int64, device="cuda")
                bfs.run_batch(srcs, dist, par if k != 5 else None, lev, stamps)
                dist_h, par_h, lev_h = dist.cpu().numpy(), par.cpu().numpy(), lev.cpu().numpy()
                st = stamps.cpu().numpy().reshape(k, 3)
                for i, s in enumerate(srcs):
                    want, _, want_levels = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
                    assert np.array_equal(dist_h[i], want), (cfg, lanes, extra, k, i)
                    assert lev_h[i] == want_levels
                    if k != 5:
                        assert oracle.check_parent(g.row_ptr, g.col, s, dist_h[i], par_h[i])[0] == 0
                    else:
                        assert (par_h[i] == -7).all()
                    assert 0 < st[i, 0] <= st[i, 1] <= st[i, 2], (cfg, lanes, st[i])
            # a single search on the same handle still works after a batch
            check_against_oracle(fbc, g, g.sources[:2], bfs=bfs)
            for bad in ([g.n], [-1]):
                with pytest.raises(fbc.BfsError):
                    bfs.run_batch(bad, torch.empty((1, g.n), dtype=torch.int32, device="cuda"))
            bfs.close()


def test_host_memory_api_new_csr_of_the_same_size(fbc):
    """Each upload of a different CSR with the same n and nnz is searched as
    that graph: the degree-0 bitmap and the head array are re-derived."""
    n = 5000
    v = np.arange(n - 1, dtype=np.uint32)
    cyc = np.arange(n - 1, dtype=np.uint32)
    graphs = [graphgen.star_graph(n), graphgen.path_graph(n),
              graphgen.from_edges(n, cyc, (cyc + 1) % (n - 1)),  # vertex n-1 isolated
              graphgen.from_edges(n, np.full(n - 1, n - 1, np.uint32), v)]  # star at n-1
    assert len({g.nnz for g in graphs}) == 1
    h = fbc.BfsCsrHost(graphs[0].row_ptr, graphs[0].col, True)
    for g in graphs:
        for s in (0, 1, n // 2):
            dist = np.empty(n, np.int32)
            parent = np.empty(n, np.int32)
            levels = h.run(s, dist, parent, row_ptr=g.row_ptr, col=g.col)
            want, _, want_levels = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
            assert np.array_equal(dist, want) and levels == want_levels, g.name
            assert oracle.check_parent(g.row_ptr, g.col, s, dist, parent)[0] == 0
    h.close()
