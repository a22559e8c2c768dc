"""The seeded input generators: determinism, CSR well-formedness, recipes."""
import numpy as np

import graphgen


def _well_formed(g, symmetric=True):
    rp = g.row_ptr.astype(np.int64)
    assert rp[0] == 0 and rp[-1] == g.nnz and np.all(np.diff(rp) >= 0)
    assert g.col.dtype == np.int32
    if g.nnz:
        assert g.col.min() >= 0 and g.col.max() < g.n
    src = np.repeat(np.arange(g.n, dtype=np.int64), np.diff(rp))
    assert np.all(src != g.col), "self-loop kept"
    key = src * g.n + g.col
    assert np.all(np.diff(key) > 0), "rows not sorted or repeats kept"
    if symmetric:
        rev = np.sort(g.col.astype(np.int64) * g.n + src)
        assert np.array_equal(rev, key)


def test_generator_is_counter_based():
    k = graphgen.key(7, 1)
    a = graphgen.draws(k, 0, 1000)
    b = graphgen.draws(k, 500, 500)
    assert np.array_equal(a[500:], b)
    assert len(np.unique(a)) == 1000
    # SplitMix64 reference value: mix(0x9E3779B97F4A7C15) for key 0, counter 0
    assert int(graphgen.draws(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_small_configs_deterministic_and_well_formed():
    for cfg in (1, 2, 4):
        g1 = graphgen.config(cfg, cache=False)
        g2 = graphgen.config(cfg, cache=False)
        assert g1.fingerprint() == g2.fingerprint()
        assert np.array_equal(g1.sources, g2.sources)
        _well_formed(g1)
        deg = g1.degrees()
        assert np.all(deg[g1.sources] > 0)
        assert len(np.unique(g1.sources)) == len(g1.sources)


def test_config1_shape():
    st = graphgen.config(1, cache=False).stats()
    assert st["n"] == 3485
    assert st["median_degree"] == 3.0
    assert 8.0 < st["mean_degree"] < 10.5
    assert 1150 < st["max_degree"] < 1400
    assert 900 < st["second_degree"] < 1150


def test_er_shape():
    g = graphgen.config(2, cache=False)
    st = g.stats()
    assert st["n"] == 1 << 20
    assert abs(st["mean_degree"] - 16.0) < 0.05


def test_grid_shape():
    g = graphgen.config(4, cache=False)
    assert g.n == 2048 * 2048
    full = 2 * (2048 * 2047 * 2)
    assert abs(g.nnz / full - 0.9) < 0.002
    assert int(g.sources[0]) in (0, 2047, 2048 * 2047, 2048 * 2048 - 1)


def test_rmat_quadrant_frequencies():
    lib = graphgen._load()
    m = 1 << 18
    src = np.empty(m, dtype=np.uint32)
    dst = np.empty(m, dtype=np.uint32)
    lib.gg_rmat_edges(10, m, 0.57, 0.19, 0.19, graphgen.key(9, 1), graphgen._p(src),
                      graphgen._p(dst))
    for bit in (9, 4, 0):
        u = (src >> bit) & 1
        v = (dst >> bit) & 1
        freq = [np.mean((u == a) & (v == b)) for a, b in ((0, 0), (0, 1), (1, 0), (1, 1))]
        assert np.allclose(freq, [0.57, 0.19, 0.19, 0.05], atol=0.005)


def test_from_edges_options():
    g = graphgen.from_edges(3, [0, 0, 1, 2], [1, 1, 1, 0], symmetric=False, drop_loops=False,
                            dedupe=False)
    assert g.row_ptr.tolist() == [0, 2, 3, 4] and g.col.tolist() == [1, 1, 1, 0]
    g = graphgen.from_edges(3, [0, 0, 1, 2], [1, 1, 1, 0])
    assert g.row_ptr.tolist() == [0, 2, 3, 4] and g.col.tolist() == [1, 2, 0, 0]
    g = graphgen.from_edges(3, [0], [2], row_ptr_64=True)
    assert g.row_ptr.dtype == np.int64


def test_random_permutation_is_a_permutation():
    lib = graphgen._load()
    n = 100000
    perm = np.empty(n, dtype=np.uint32)
    lib.gg_permutation(n, graphgen.key(2, 2), graphgen._p(perm))
    assert np.array_equal(np.sort(perm), np.arange(n, dtype=np.uint32))
