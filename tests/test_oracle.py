"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: the checks use the pages'
printed worked examples (tests/golden), library shortest-path routines
(scipy, networkx) on small random graphs, closed forms on structured graphs,
an exhaustive search over every candidate distance array on tiny graphs, and
mutants of the oracle source that these pins must reject.
"""
import itertools
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import graphgen
import oracle

scipy_csgraph = pytest.importorskip("scipy.sparse.csgraph")
import scipy.sparse as sp  # noqa: E402


def _hops_scipy(g, source):
    n = g.n
    a = sp.csr_matrix((np.ones(g.nnz), g.col.astype(np.int64), g.row_ptr.astype(np.int64)),
                      shape=(n, n))
    d = scipy_csgraph.shortest_path(a, directed=True, unweighted=True, indices=source)
    out = np.where(np.isinf(d), -1, d).astype(np.int32)
    return out


def _hops_networkx(g, source):
    nx = pytest.importorskip("networkx")
    G = nx.DiGraph()
    G.add_nodes_from(range(g.n))
    rp = g.row_ptr.astype(np.int64)
    for u in range(g.n):
        for e in range(rp[u], rp[u + 1]):
            G.add_edge(u, int(g.col[e]))
    d = np.full(g.n, -1, dtype=np.int32)
    for v, k in nx.single_source_shortest_path_length(G, source).items():
        d[v] = k
    return d


# ----------------------------------------------------------- worked examples

def test_six_vertex_golden(golden):
    gx = golden("six_vertex_directed.json")
    rp, col = np.array(gx["row_ptr"]), np.array(gx["col"])
    dist, parent, levels = oracle.bfs(rp, col, gx["source"])
    assert dist.tolist() == gx["dist"]
    assert parent.tolist() == gx["fifo_parent"]
    assert levels == gx["num_levels"]
    sizes, nl, reached, _ = oracle.level_sizes(rp, dist)
    assert sizes.tolist() == [len(f) for f in gx["levels"]]
    assert nl == gx["num_levels"] and reached == 6
    for k, frontier in enumerate(gx["levels"]):
        assert sorted(np.nonzero(dist == k)[0].tolist()) == sorted(frontier)


def test_six_vertex_after_level_one(golden):
    gx = golden("six_vertex_directed.json")
    st = gx["after_level_1"]
    dist, _, levels = oracle.bfs(np.array(gx["row_ptr"]), np.array(gx["col"]), gx["source"],
                                 max_depth=st["max_depth"])
    assert dist.tolist() == st["dist"]
    assert levels == 3


def test_six_vertex_edge_parallel_bookkeeping(golden):
    """The exclusive scan of frontier degrees and the edge -> (src, dst) map
    printed for frontier {3, 4}: derived from the CSR and the oracle's dist."""
    gx = golden("six_vertex_directed.json")
    rp, col = np.array(gx["row_ptr"]), np.array(gx["col"])
    dist, _, _ = oracle.bfs(rp, col, gx["source"])
    frontier = sorted(np.nonzero(dist == 2)[0].tolist())
    ep = gx["edge_parallel"]
    assert frontier == ep["frontier"]
    deg = [int(rp[v + 1] - rp[v]) for v in frontier]
    assert deg == ep["degrees"]
    offs = np.concatenate([[0], np.cumsum(deg)]).tolist()
    assert offs == ep["offsets"]
    pairs = []
    for e in range(offs[-1]):
        i = int(np.searchsorted(offs, e, side="right") - 1)
        pairs.append([frontier[i], int(col[rp[frontier[i]] + e - offs[i]])])
    assert pairs == ep["assignments"]
    assert np.nonzero(dist == 3)[0].tolist() == ep["next_frontier"]


def test_four_vertex_golden(golden):
    gx = golden("four_vertex_undirected.json")
    rp, col = np.array(gx["row_ptr"]), np.array(gx["col"])
    assert col[rp[2]:rp[3]].tolist() == gx["neighbours_of_2"]
    for s, want in gx["dist_from"].items():
        dist, parent, levels = oracle.bfs(rp, col, int(s))
        assert dist.tolist() == want
        assert levels == max(want) + 1
        assert oracle.check_parent(rp, col, int(s), dist, parent)[0] == 0


def test_day38_table_bookkeeping(golden):
    t = golden("day38_level_table.json")
    assert sum(t["frontier"]) == t["reached"]
    assert sum(t["edges"]) == t["edges_walked"]
    assert len(t["frontier"]) == t["levels"]
    assert sum(t["lane_slots"]) == t["lane_slots_total"]
    for w, md, slots in zip(t["warps"], t["max_degree"], t["lane_slots"]):
        if w == 1:
            assert slots == 32 * md


# --------------------------------------------------------- brute force, n <= 12

def _small_graphs(count, seed0):
    for k in range(count):
        n = 1 + (k % 12)
        p = [0.1, 0.2, 0.35, 0.6][k % 4]
        directed = bool(k % 2)
        loops = directed and (k % 3 == 0)
        yield graphgen.random_graph(n, p, seed0 + k, directed=directed, loops=loops)


def test_bfs_matches_scipy_on_random_small_graphs():
    checked = 0
    for g in _small_graphs(1200, 1000):
        for s in range(g.n):
            dist, parent, levels = oracle.bfs(g.row_ptr, g.col, s)
            want = _hops_scipy(g, s)
            assert np.array_equal(dist, want), (g.name, s)
            assert levels == int(want.max()) + 1
            checked += 1
    assert checked > 5000


def test_bfs_matches_networkx_on_random_small_graphs():
    for g in _small_graphs(200, 5000):
        for s in range(g.n):
            dist, _, _ = oracle.bfs(g.row_ptr, g.col, s, want_parent=False)
            assert np.array_equal(dist, _hops_networkx(g, s)), (g.name, s)


def test_parent_is_fifo_first_discoverer_and_valid():
    """Parent validity by enumeration: the set of valid parents of v is every
    in-neighbour one hop closer to the source (from scipy's distances)."""
    for g in _small_graphs(400, 9000):
        rp = g.row_ptr.astype(np.int64)
        for s in range(g.n):
            dist, parent, _ = oracle.bfs(g.row_ptr, g.col, s)
            d = _hops_scipy(g, s)
            for v in range(g.n):
                if v == s:
                    assert parent[v] == s
                elif d[v] < 0:
                    assert parent[v] == -1
                else:
                    valid = {u for u in range(g.n) if d[u] == d[v] - 1
                             and v in g.col[rp[u]:rp[u + 1]]}
                    assert parent[v] in valid


def test_max_depth_truncation_matches_scipy():
    for g in _small_graphs(300, 12000):
        for s in range(g.n):
            full = _hops_scipy(g, s)
            for depth in range(0, 4):
                dist, _, levels = oracle.bfs(g.row_ptr, g.col, s, max_depth=depth,
                                             want_parent=False)
                want = np.where((full >= 0) & (full <= depth), full, -1)
                assert np.array_equal(dist, want)
                assert levels == int(want.max()) + 1


# --------------------------------------------------------- closed forms

def test_closed_forms():
    n = 10
    g = graphgen.path_graph(n)
    dist, parent, levels = oracle.bfs(g.row_ptr, g.col, 0)
    assert dist.tolist() == list(range(n)) and levels == n
    assert parent.tolist() == [0] + list(range(n - 1))
    dist, _, levels = oracle.bfs(g.row_ptr, g.col, 4)
    assert dist.tolist() == [abs(v - 4) for v in range(n)] and levels == 6

    g = graphgen.star_graph(7)
    dist, parent, levels = oracle.bfs(g.row_ptr, g.col, 0)
    assert dist.tolist() == [0] + [1] * 6 and parent.tolist() == [0] * 7 and levels == 2
    dist, parent, levels = oracle.bfs(g.row_ptr, g.col, 3)
    assert dist.tolist() == [1, 2, 2, 0, 2, 2, 2] and levels == 3
    assert parent.tolist() == [3, 0, 0, 3, 0, 0, 0]

    g = graphgen.clique_graph(6)
    dist, _, levels = oracle.bfs(g.row_ptr, g.col, 2)
    assert dist.tolist() == [1, 1, 0, 1, 1, 1] and levels == 2

    g = graphgen.from_edges(1, [], [])
    dist, parent, levels = oracle.bfs(g.row_ptr, g.col, 0)
    assert dist.tolist() == [0] and parent.tolist() == [0] and levels == 1

    g = graphgen.from_edges(5, [0, 3], [1, 4])  # two components and an isolated vertex
    dist, parent, levels = oracle.bfs(g.row_ptr, g.col, 3)
    assert dist.tolist() == [-1, -1, -1, 0, 1] and parent.tolist() == [-1, -1, -1, 3, 3]
    assert levels == 2

    rows, cols = 5, 7  # full lattice: Manhattan distance from the corner
    g = graphgen.grid(rows, cols, 0.0, 0)
    dist, _, levels = oracle.bfs(g.row_ptr, g.col, 0)
    assert dist.tolist() == [r + c for r in range(rows) for c in range(cols)]
    assert levels == rows + cols - 1


def test_self_loops_and_duplicates_do_not_change_distances():
    src = [0, 0, 0, 1, 1, 2, 2, 3]
    dst = [0, 1, 1, 1, 2, 2, 3, 3]
    g_multi = graphgen.from_edges(4, src, dst, symmetric=False, drop_loops=False, dedupe=False)
    g_simple = graphgen.from_edges(4, src, dst, symmetric=False)
    assert g_multi.nnz == 8 and g_simple.nnz == 3
    for s in range(4):
        d1, p1, l1 = oracle.bfs(g_multi.row_ptr, g_multi.col, s)
        d2, _, l2 = oracle.bfs(g_simple.row_ptr, g_simple.col, s)
        assert np.array_equal(d1, d2) and l1 == l2
        assert oracle.check_parent(g_multi.row_ptr, g_multi.col, s, d1, p1)[0] == 0


def test_int64_row_ptr_same_as_int32():
    g = graphgen.random_graph(12, 0.3, 77)
    rp64 = g.row_ptr.astype(np.int64)
    for s in range(g.n):
        a = oracle.bfs(g.row_ptr, g.col, s)
        b = oracle.bfs(rp64, g.col, s)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


# --------------------------------------------------------- the checkers

def test_check_dist_is_exact_certificate_exhaustive():
    """On tiny graphs, check_dist accepts exactly one array out of every
    candidate in {-1, 0, .., n-1}^n: the true hop distances."""
    graphs = [graphgen.random_graph(4, 0.4, s, directed=bool(s % 2)) for s in range(6)]
    graphs.append(graphgen.from_csr([0, 2, 4, 7, 8], [1, 2, 0, 2, 0, 1, 3, 2], True))
    for g in graphs:
        n = g.n
        for s in range(n):
            truth = _hops_scipy(g, s)
            accepted = []
            for cand in itertools.product(range(-1, n), repeat=n):
                c = np.array(cand, dtype=np.int32)
                if oracle.check_dist(g.row_ptr, g.col, s, c)[0] == 0:
                    accepted.append(c)
            assert len(accepted) == 1 and np.array_equal(accepted[0], truth)


def test_check_parent_accepts_exactly_valid_trees():
    for g in _small_graphs(150, 20000):
        rp = g.row_ptr.astype(np.int64)
        for s in range(min(g.n, 3)):
            d = _hops_scipy(g, s)
            choices = []
            for v in range(g.n):
                if v == s:
                    choices.append([s])
                elif d[v] < 0:
                    choices.append([-1])
                else:
                    choices.append(sorted({u for u in range(g.n) if d[u] == d[v] - 1
                                           and v in g.col[rp[u]:rp[u + 1]]}))
            rng = np.random.default_rng(s)
            for _ in range(5):
                par = np.array([rng.choice(c) for c in choices], dtype=np.int32)
                assert oracle.check_parent(g.row_ptr, g.col, s, d, par)[0] == 0
                v = int(rng.integers(g.n))
                for wrong in range(-1, g.n):
                    if wrong in choices[v]:
                        continue
                    bad = par.copy()
                    bad[v] = wrong
                    code, where = oracle.check_parent(g.row_ptr, g.col, s, d, bad)
                    assert code != 0 and where == v


def test_level_sizes_and_edges_walked():
    g = graphgen.powerlaw_3485(0)
    deg = g.degrees()
    s = int(np.argmax(deg))
    dist, _, levels = oracle.bfs(g.row_ptr, g.col, s)
    sizes, nl, reached, edges = oracle.level_sizes(g.row_ptr, dist)
    assert nl == levels and sizes.sum() == reached == (dist >= 0).sum()
    assert edges == int(deg[dist >= 0].sum())
    assert np.array_equal(sizes, np.bincount(dist[dist >= 0], minlength=nl))


def test_edges_walked_pinned_to_the_worked_examples(golden):
    """The walked-edge count (the TEPS numerator: CSR entries of the reached
    vertices) on graphs where the pages or a closed form fix it.

    ch. 22 section 22.1's six-vertex graph from source 0 reaches all six
    vertices, so all 9 printed CSR entries are walked; cut at depth 2 (the
    state the section prints after level 1) vertex 5 stays unreached but has
    no out-edges, so still 9. PMPP 15.1's four-vertex graph is connected: 8
    entries from every source. A path of m vertices walks 2(m - 1) entries
    from any vertex; a graph of two components walks only the source's one.
    """
    gx = golden("six_vertex_directed.json")
    rp, col = np.array(gx["row_ptr"]), np.array(gx["col"])
    dist, _, _ = oracle.bfs(rp, col, gx["source"])
    assert oracle.level_sizes(rp, dist)[3] == 9 == len(gx["col"])
    d2, _, _ = oracle.bfs(rp, col, gx["source"], max_depth=gx["after_level_1"]["max_depth"])
    assert oracle.level_sizes(rp, d2)[2:] == (5, 9)
    # from vertex 3 only {3, 4, 5} are reached: rows of 2 + 1 + 0 entries
    d3, _, _ = oracle.bfs(rp, col, 3)
    assert oracle.level_sizes(rp, d3)[2:] == (3, 3)
    g4 = golden("four_vertex_undirected.json")
    rp4, col4 = np.array(g4["row_ptr"]), np.array(g4["col"])
    for s in range(4):
        d, _, _ = oracle.bfs(rp4, col4, s)
        assert oracle.level_sizes(rp4, d)[2:] == (4, 8)
    for m in (1, 2, 7, 100):
        g = graphgen.path_graph(m)
        for s in (0, m // 2, m - 1):
            d, _, _ = oracle.bfs(g.row_ptr, g.col, s)
            assert oracle.level_sizes(g.row_ptr, d)[2:] == (m, 2 * (m - 1))
    # a 5-clique beside a 4-vertex path: 20 entries or 6
    src = [a for a in range(5) for b in range(5) if a != b] + [5, 6, 7]
    dst = [b for a in range(5) for b in range(5) if a != b] + [6, 7, 8]
    g = graphgen.from_edges(9, src, dst)
    assert g.nnz == 20 + 6
    for s, want in ((0, (5, 20)), (4, (5, 20)), (5, (4, 6)), (8, (4, 6))):
        d, _, _ = oracle.bfs(g.row_ptr, g.col, s)
        assert oracle.level_sizes(g.row_ptr, d)[2:] == want


def _xor_sum_by_bits(c: int, repeats: int) -> int:
    """sum over r < repeats of (c XOR r), counted bit by bit: bit b of c ^ r is
    set for every r whose bit b differs from c's, and among 0 .. R-1 the
    number of r with bit b set is (R >> (b+1)) << b plus the overhang of the
    last partial period. Independent of the oracle's loop."""
    total = 0
    for b in range(40):
        period = 1 << (b + 1)
        ones = (repeats // period) * (1 << b) + max(0, repeats % period - (1 << b))
        n_set = repeats - ones if (c >> b) & 1 else ones
        total += n_set << b
    return total


def test_walk_checksum_pins(golden):
    """The walk checksum against values fixed without the oracle's loop.

    One repeat (r = 0) is the plain sum of the neighbour ids: on the ch. 22
    six-vertex graph the rows [1 2] [2 3] [3 4] [4 5] [5] [] sum to 3, 5, 7,
    9, 5, 0. For a power-of-two repeat count P, XOR with r < P permutes the
    low bits, so each entry c contributes P * (c with its low log2 P bits
    cleared) + P (P - 1) / 2; the page's 64 repeats fall under this. Other
    counts are checked bit by bit; the sum wraps modulo 2^32, and an id
    outside [0, n) walks nothing."""
    gx = golden("six_vertex_directed.json")
    rp, col = np.array(gx["row_ptr"]), np.array(gx["col"])
    assert oracle.walk_checksum(rp, col, [0, 1, 2, 3, 4, 5], 1).tolist() == [3, 5, 7, 9, 5, 0]
    assert oracle.walk_checksum(rp, col, [0, 5, 0], 0).tolist() == [0, 0, 0]
    assert oracle.walk_checksum(rp, col, [6, -1, 2], 1).tolist() == [0, 0, 7]
    g = graphgen.config(1)
    fr = np.arange(g.n, dtype=np.int32)
    rp1 = g.row_ptr.astype(np.int64)
    for P in (1, 2, 64, 256):
        want = [(sum(P * (int(c) & ~(P - 1)) + P * (P - 1) // 2
                     for c in g.col[rp1[u]:rp1[u + 1]])) % (1 << 32) for u in range(0, g.n, 7)]
        assert oracle.walk_checksum(g.row_ptr, g.col, fr[::7], P).tolist() == want, P
    for R in (3, 5, 37, 100):
        want = [sum(_xor_sum_by_bits(int(c), R) for c in g.col[rp1[u]:rp1[u + 1]]) % (1 << 32)
                for u in range(0, g.n, 11)]
        assert oracle.walk_checksum(g.row_ptr, g.col, fr[::11], R).tolist() == want, R
    # wrap-around: 40 entries of id 3 over 2^22 repeats sum to ~2^48
    P = 1 << 22
    rpw = np.array([0, 40, 40, 40, 40, 40], dtype=np.int64)
    colw = np.full(40, 3, dtype=np.int32)
    exact = 40 * (P * (3 & ~(P - 1)) + P * (P - 1) // 2)
    assert exact >= 1 << 40
    assert oracle.walk_checksum(rpw, colw, [0, 4], P).tolist() == [exact % (1 << 32), 0]


def test_config1_eccentric_source_levels_equal_ecc_plus_one():
    g = graphgen.config(1)
    n = g.n
    a = sp.csr_matrix((np.ones(g.nnz), g.col.astype(np.int64), g.row_ptr.astype(np.int64)),
                      shape=(n, n))
    deg = g.degrees()
    cand = np.nonzero(deg)[0][:400]
    d = scipy_csgraph.shortest_path(a, directed=False, unweighted=True, indices=cand)
    d[np.isinf(d)] = -1
    for row, s in zip(d, cand):
        dist, _, levels = oracle.bfs(g.row_ptr, g.col, int(s), want_parent=False)
        assert np.array_equal(dist, row.astype(np.int32))
        assert levels == int(row.max()) + 1
        assert oracle.check_dist(g.row_ptr, g.col, int(s), dist)[0] == 0


# --------------------------------------------------------- mutants

MUTANTS = [
    ("dist[w] = dist[u] + 1;", "dist[w] = dist[u] + 2;"),       # wrong level increment
    ("if (dist[w] == -1) {", "if (dist[w] <= 0) {"),             # re-discovers the source
    ("parent[w] = u;", "parent[w] = w;"),                        # wrong parent
    ("queue[tail++] = w;", "queue[tail++] = u;"),                # enqueues the wrong vertex
    ("if (max_depth >= 0 && dist[u] >= max_depth)",
     "if (max_depth >= 0 && dist[u] > max_depth)"),              # off-by-one depth bound
    ("e < last; ++e) {\n            const int32_t w = col[e];\n            if (dist[w] == -1)",
     "e + 1 < last; ++e) {\n            const int32_t w = col[e];\n            if (dist[w] == -1)"),
    ("edges += row_at(row_ptr, row_ptr_64, v + 1) -",
     "edges += row_at(row_ptr, row_ptr_64, v + 1) + 0 *"),  # walked count without the row start
    ("row_at(row_ptr, row_ptr_64, v);\n        if (d > deepest)",
     "row_at(row_ptr, row_ptr_64, 0);\n        if (d > deepest)"),  # wrong row start
    ("acc += (uint32_t)col[e] ^ (uint32_t)r;", "acc += (uint32_t)col[e] ^ (uint32_t)(r + 1);"),
    ("acc += (uint32_t)col[e] ^ (uint32_t)r;", "acc += (uint32_t)col[e];"),  # XOR dropped
]


@pytest.mark.parametrize("old,new", MUTANTS)
def test_pins_reject_oracle_mutants(old, new, golden, monkeypatch):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "bfs_oracle.c")).read()
    assert old in src, "mutation site vanished"
    build_dir = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "_build")
    os.makedirs(build_dir, exist_ok=True)
    tmp = tempfile.mkdtemp(dir=build_dir)
    try:
        pkg = os.path.join(tmp, "oracle")
        shutil.copytree(os.path.dirname(oracle.__file__), pkg,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
        with open(os.path.join(pkg, "bfs_oracle.c"), "w") as f:
            f.write(src.replace(old, new, 1))
        gdir = os.path.join(os.path.dirname(__file__), "golden")
        code = (
            "import json, os, sys, numpy as np\n"
            "sys.path.insert(0, %r)\n"
            "import oracle\n"
            "gx = json.load(open(os.path.join(%r, 'six_vertex_directed.json')))\n"
            "rp, col = np.array(gx['row_ptr']), np.array(gx['col'])\n"
            "d, p, L = oracle.bfs(rp, col, 0)\n"
            "ok = d.tolist() == gx['dist'] and p.tolist() == gx['fifo_parent'] and L == 4\n"
            "d2, _, _ = oracle.bfs(rp, col, 0, max_depth=2)\n"
            "ok = ok and d2.tolist() == gx['after_level_1']['dist']\n"
            "g4 = json.load(open(os.path.join(%r, 'four_vertex_undirected.json')))\n"
            "for s, want in g4['dist_from'].items():\n"
            "    d, p, L = oracle.bfs(np.array(g4['row_ptr']), np.array(g4['col']), int(s))\n"
            "    ok = ok and d.tolist() == want and L == max(want) + 1\n"
            "    ok = ok and oracle.level_sizes(np.array(g4['row_ptr']), d)[3] == 8\n"
            "d3, _, _ = oracle.bfs(rp, col, 3)\n"
            "ok = ok and oracle.level_sizes(rp, d3)[2:] == (3, 3)\n"
            "ok = ok and oracle.walk_checksum(rp, col, [0, 3], 1).tolist() == [3, 9]\n"
            "ok = ok and oracle.walk_checksum(rp, col, [0], 64).tolist() == [2 * 2016]\n"
            "print('PASS' if ok else 'FAIL')\n" % (tmp, gdir, gdir))
        out = subprocess.run(["python", "-c", code], capture_output=True, text=True,
                             timeout=120)
        assert "FAIL" in out.stdout or out.returncode != 0, out.stdout + out.stderr
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
