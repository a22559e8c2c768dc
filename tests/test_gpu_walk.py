"""The isolated neighbour walk ("100 Days of GPU, Day 38", section "Measuring
the mapping without measuring the launch") through the C-ABI: every mapping
(thread, warp, degree-binned, edge-balanced) must return, slot by slot, the
wrapping 32-bit checksum the oracle predicts on the host."""
import numpy as np
import pytest

import graphgen
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MAPPINGS = ("thread", "warp", "binned", "edge")


@pytest.fixture(scope="module")
def fbc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import frontier_bfs_csr_gb300
    return frontier_bfs_csr_gb300


def _walk_all(fbc, bfs, g, frontier, repeats):
    fr = torch.from_numpy(np.ascontiguousarray(frontier, dtype=np.int32)).cuda()
    want = oracle.walk_checksum(g.row_ptr, g.col, frontier, repeats)
    for m, name in enumerate(MAPPINGS):
        out = torch.full((len(frontier),), 7, dtype=torch.int32, device="cuda")
        bfs.walk(fr, repeats, m, out)
        got = out.cpu().numpy().view(np.uint32)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, "%s %s repeats %d: slot %d got %d want %d" % (
            g.name, name, repeats, bad[0], got[bad[0]], want[bad[0]])


def _eccentric_source(g):
    deg = g.degrees()
    best, best_levels = None, -1
    for s in np.nonzero(deg)[0]:
        levels = oracle.bfs(g.row_ptr, g.col, int(s), want_parent=False)[2]
        if levels > best_levels:
            best, best_levels = int(s), levels
    return best


def test_walk_every_level_of_the_power_law_graph(fbc):
    """Config 1 from its most eccentric source, every level (frontier in
    vertex order), 64 repeats as on the page and 3 (not a power of two)."""
    g = graphgen.config(1)
    s = _eccentric_source(g)
    dist, _, levels = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
    bfs = fbc.BfsCsr(torch.from_numpy(g.row_ptr).cuda(), torch.from_numpy(g.col).cuda(), True)
    for k in range(levels):
        frontier = np.nonzero(dist == k)[0].astype(np.int32)
        for repeats in (64, 3):
            _walk_all(fbc, bfs, g, frontier, repeats)
    # the whole vertex set (degree-0 vertices included), shuffled, plus ids
    # outside [0, n) that must walk nothing
    every = np.random.default_rng(3).permutation(g.n).astype(np.int32)
    _walk_all(fbc, bfs, g, every, 2)
    _walk_all(fbc, bfs, g, np.array([-1, 0, g.n, 5, g.n + 7], np.int32), 64)
    bfs.close()


def test_walk_wide_level_and_int64_rows(fbc):
    """A wide R-MAT scale-22 level (hundreds of thousands of vertices, hubs of
    ~10^5 entries) and an int64 row_ptr graph."""
    g = graphgen.config(3)
    s = int(g.sources[0])
    dist, _, _ = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
    sizes = np.bincount(dist[dist >= 0])
    k = int(np.argmax(sizes))
    frontier = np.nonzero(dist == k)[0].astype(np.int32)
    hubs = np.argsort(g.degrees())[-3:].astype(np.int32)
    bfs = fbc.BfsCsr(torch.from_numpy(g.row_ptr).cuda(), torch.from_numpy(g.col).cuda(), True)
    _walk_all(fbc, bfs, g, frontier, 1)
    _walk_all(fbc, bfs, g, hubs, 5)
    bfs.close()
    g = graphgen.rmat(12, 8, 11, row_ptr_64=True)
    bfs = fbc.BfsCsr(torch.from_numpy(g.row_ptr).cuda(), torch.from_numpy(g.col).cuda(), True)
    _walk_all(fbc, bfs, g, np.arange(g.n, dtype=np.int32), 4)
    bfs.close()


def test_walk_argument_errors(fbc):
    g = graphgen.config(1)
    bfs = fbc.BfsCsr(torch.from_numpy(g.row_ptr).cuda(), torch.from_numpy(g.col).cuda(), True)
    fr = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    for args in ((fr.data_ptr(), 4, -1, 0), (fr.data_ptr(), 4, 1, 4), (fr.data_ptr(), 4, 1, -1),
                 (fr.data_ptr(), g.n + 1, 1, 0), (None, 4, 1, 0), (fr.data_ptr(), -1, 1, 0)):
        assert fbc.bfs_csr_walk(bfs.handle, args[0], args[1], args[2], args[3],
                                out.data_ptr(), None) == fbc.BFS_CSR_EINVAL, args
    assert fbc.bfs_csr_walk(bfs.handle, None, 0, 1, 0, None, None) == fbc.BFS_CSR_OK
    bfs.close()
