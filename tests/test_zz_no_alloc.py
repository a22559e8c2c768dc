"""bfs_csr_run_noalloc: the search for callers that cannot call cudaMalloc
(their device memory belongs to another allocator, or the path must not take
cudaMalloc's implicit synchronisation). It runs on the library's own fixed
scratch array instead of a handle's workspace.

Checked through the C-ABI against the regular entry point (bfs_csr_create +
bfs_csr_run) on the same inputs, two calls in a row: dist must be identical
(distances are unique), parent must be a valid BFS tree (several are
correct, so it is checked, not compared) and the level counts must agree.
This file is collected last and also passes on its own in a fresh process.
"""
import ctypes

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


def _noalloc(fbc, row_ptr, col, n, nnz, source, symmetric=True, want_parent=True, opt=None):
    dist = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    parent = torch.full((n,), -7, dtype=torch.int32, device="cuda") if want_parent else None
    dlev = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlev = ctypes.c_int32(0)
    stream = torch.cuda.current_stream().cuda_stream
    status = fbc.bfs_csr_run_noalloc(n, nnz, row_ptr.data_ptr(),
                                     col.data_ptr() if nnz else None, int(symmetric),
                                     int(source), dist.data_ptr(),
                                     parent.data_ptr() if want_parent else None,
                                     dlev.data_ptr(), ctypes.byref(hlev),
                                     ctypes.byref(opt) if opt is not None else None, stream)
    return status, dist, parent, int(hlev.value), int(dlev.item())


def _compare(fbc, g, sources, **over):
    rp = torch.from_numpy(g.row_ptr).cuda()
    col = torch.from_numpy(g.col).cuda()
    opt = fbc.default_options(**over) if over else None
    ref = fbc.BfsCsr(rp, col, symmetric=g.symmetric, options=opt)
    for s in sources:
        s = int(s)
        status, dist, parent, hlev, dlev = _noalloc(fbc, rp, col, g.n, g.nnz, s, g.symmetric,
                                                    opt=opt)
        assert status == fbc.BFS_CSR_OK, fbc.bfs_csr_status_string(status)
        want_dist, _, want_levels = ref.search(s)
        assert torch.equal(dist, want_dist)
        assert hlev == dlev == want_levels
        code, bad = oracle.check_parent(g.row_ptr, g.col, s, dist.cpu().numpy(),
                                        parent.cpu().numpy())
        assert code == 0, "invalid parent at %d" % bad
    ref.close()


def test_noalloc_matches_regular_entry_point_small(fbc):
    g = graphgen.config(1)
    _compare(fbc, g, g.sources[:2])          # two calls in a row
    _compare(fbc, g, [g.sources[0]] * 2)     # same source twice: state is reset


def test_noalloc_matches_regular_entry_point_at_the_size_limit(fbc):
    g = graphgen.config(2)                   # exactly 2^20 vertices
    assert g.n == fbc.BFS_CSR_NOALLOC_MAX_VERTICES
    _compare(fbc, g, g.sources[:2])


def test_noalloc_directed_and_without_parent(fbc):
    g = graphgen.random_graph(12, 0.3, 8, directed=True)
    _compare(fbc, g, [0, 5])
    rp = torch.from_numpy(g.row_ptr).cuda()
    col = torch.from_numpy(g.col).cuda()
    status, dist, _, hlev, _ = _noalloc(fbc, rp, col, g.n, g.nnz, 3, False, want_parent=False)
    assert status == fbc.BFS_CSR_OK
    want, _, levels = oracle.bfs(g.row_ptr, g.col, 3, want_parent=False)
    assert np.array_equal(dist.cpu().numpy(), want) and hlev == levels


def test_noalloc_rejects_sizes_beyond_the_limit(fbc):
    n = fbc.BFS_CSR_NOALLOC_MAX_VERTICES + 1
    rp = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    col = torch.zeros(1, dtype=torch.int32, device="cuda")
    status, *_ = _noalloc(fbc, rp, col, n, 0, 0)
    assert status == fbc.BFS_CSR_EUNSUPPORTED
    status, *_ = _noalloc(fbc, rp, col, 10, 0, 10)    # source out of range
    assert status == fbc.BFS_CSR_EINVAL


@pytest.mark.parametrize("over", [dict(loop_mode=1, discovery=1), dict(direction=2),
                                  dict(direction=1, advance=2, discovery=1)],
                         ids=["host_loop+cas", "pull", "push+merge_path+cas"])
def test_noalloc_options_match_regular_entry_point(fbc, over):
    """The host level loop, CAS discovery (dist written at discovery instead
    of through the hop codes) and forced directions on the shared scratch,
    each against the regular entry point with the same options."""
    g = graphgen.config(1)
    _compare(fbc, g, g.sources[:2], **over)


def test_noalloc_malformed_csr_then_recovers(fbc):
    """A malformed CSR is rejected by the validation pass with EINVAL; the
    next call on a good graph, on the same shared scratch, is still right.
    Several lanes are refused (the scratch holds one search), and so are the
    graph loop mode (a graph is a resource the entry point cannot keep) and
    the padded frontiers (their arrays do not fit the scratch)."""
    g = graphgen.config(1)
    bad = g.row_ptr.copy()
    bad[10], bad[11] = bad[11], bad[10] - 1      # row_ptr decreases
    rp_bad = torch.from_numpy(bad).cuda()
    col = torch.from_numpy(g.col).cuda()
    status, *_ = _noalloc(fbc, rp_bad, col, g.n, g.nnz, int(g.sources[0]))
    assert status == fbc.BFS_CSR_EINVAL
    status, *_ = _noalloc(fbc, torch.from_numpy(g.row_ptr).cuda(), col, g.n, g.nnz,
                          int(g.sources[0]), opt=fbc.default_options(lanes=2))
    assert status == fbc.BFS_CSR_EUNSUPPORTED
    status, *_ = _noalloc(fbc, torch.from_numpy(g.row_ptr).cuda(), col, g.n, g.nnz,
                          int(g.sources[0]), opt=fbc.default_options(loop_mode=2))
    assert status == fbc.BFS_CSR_EUNSUPPORTED
    status, *_ = _noalloc(fbc, torch.from_numpy(g.row_ptr).cuda(), col, g.n, g.nnz,
                          int(g.sources[0]), opt=fbc.default_options(frontier_output=1))
    assert status == fbc.BFS_CSR_EUNSUPPORTED
    _compare(fbc, g, g.sources[2:4])
