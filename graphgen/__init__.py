"""Seeded synthetic CSR graphs shared by the tests and the benchmark.

This module only draws edges and sorts them into CSR (``graphgen.c``); it
walks no graph and computes no distance, so neither the oracle nor the CUDA
path depends on the other through it. Every random number comes from one
counter-based generator (the SplitMix64 output function on
``key + (counter + 1) * 0x9E3779B97F4A7C15``), so a graph is the same on any
machine and thread count.

The five workloads (sizes, degree structure and seeds):

1. ``powerlaw_3485`` -- Chung-Lu graph on 3,485 vertices with expected
   weights from a truncated power law (exponent 2) and two calibrated hubs,
   undirected, deduplicated, int32 CSR. It stands in for the 3,485-word graph
   of "100 Days of GPU, Day 38" (median degree 3, max 1,255, second hub
   1,012), whose data file is not available. Seed 0.
2. ``er_2^20`` -- Erdos-Renyi style G(n, m): 2^20 vertices, 8,388,608 uniform
   endpoint pairs (average degree 16), self-loops and repeats dropped,
   symmetrised, int32 CSR. Seed 1.
3. ``rmat_22`` -- R-MAT scale 22, edge factor 16, (a, b, c, d) = (0.57, 0.19,
   0.19, 0.05), labels randomly permuted, symmetrised, self-loops and repeats
   dropped, int32 CSR. Seed 2.
4. ``grid_2048`` -- 2048 x 2048 4-neighbour lattice with each edge deleted
   independently with probability 0.1, int32 CSR, source the first corner of
   nonzero degree. Seed 3.
5. ``rmat_25`` -- R-MAT scale 25, edge factor 16, same recipe, int64 row_ptr
   and int32 col (about 4 GB). Seed 4.

Sources (except config 4's corner) are distinct vertices of nonzero degree
drawn uniformly from the config's seed on a stream of their own.
"""
from __future__ import annotations

import ctypes
import dataclasses
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "graphgen.c")
_LIB_PATH = os.path.join(_HERE, "libgraphgen.so")
_lock = threading.Lock()
_lib = None

# Stream ids inside one seed.
STREAM_EDGES = 1
STREAM_PERM = 2
STREAM_SOURCES = 3
STREAM_WEIGHTS = 4


def build(force: bool = False) -> str:
    """Compile ``graphgen.c`` (gcc -O3 -fopenmp) into ``libgraphgen.so``."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O3", "-fopenmp", "-Wall", "-shared",
                               "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32, vp, dbl = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_double)
            lib.gg_key.argtypes = [u64, u64]
            lib.gg_key.restype = u64
            lib.gg_draws.argtypes = [u64, u64, i64, vp]
            lib.gg_draws.restype = None
            lib.gg_rmat_edges.argtypes = [i32, i64, dbl, dbl, dbl, u64, vp, vp]
            lib.gg_rmat_edges.restype = None
            lib.gg_uniform_edges.argtypes = [i64, i64, u64, vp, vp]
            lib.gg_uniform_edges.restype = None
            lib.gg_permutation.argtypes = [i64, u64, vp]
            lib.gg_permutation.restype = None
            lib.gg_relabel.argtypes = [i64, vp, vp, vp]
            lib.gg_relabel.restype = None
            lib.gg_grid_edges.argtypes = [i64, i64, dbl, u64, vp, vp]
            lib.gg_grid_edges.restype = i64
            lib.gg_chung_lu_edges.argtypes = [i64, vp, u64, i64, vp, vp]
            lib.gg_chung_lu_edges.restype = i64
            lib.gg_build_csr.argtypes = [i64, i64, vp, vp, i32, i32, i32, vp, vp, i64]
            lib.gg_build_csr.restype = i64
            lib.gg_fingerprint.argtypes = [i64, vp, i64, vp]
            lib.gg_fingerprint.restype = u64
            lib.gg_pick_sources.argtypes = [i64, vp, i64, u64, i64, vp]
            lib.gg_pick_sources.restype = i64
            _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclasses.dataclass
class Graph:
    """A CSR graph: ``row_ptr`` (n+1, int32 or int64) and ``col`` (nnz, int32)."""
    name: str
    row_ptr: np.ndarray
    col: np.ndarray
    symmetric: bool = True
    sources: np.ndarray | None = None
    meta: dict = dataclasses.field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.row_ptr.shape[0] - 1)

    @property
    def nnz(self) -> int:
        return int(self.col.shape[0])

    @property
    def row_ptr_64(self) -> bool:
        return self.row_ptr.dtype == np.int64

    def degrees(self) -> np.ndarray:
        return np.diff(self.row_ptr.astype(np.int64))

    def fingerprint(self) -> str:
        rp = np.ascontiguousarray(self.row_ptr, dtype=np.int64)
        return "%016x" % _load().gg_fingerprint(self.n, _p(rp), self.nnz, _p(self.col))

    def stats(self) -> dict:
        deg = self.degrees()
        srt = np.sort(deg)[::-1]
        return {"n": self.n, "nnz": self.nnz, "max_degree": int(srt[0]) if self.n else 0,
                "second_degree": int(srt[1]) if self.n > 1 else 0,
                "median_degree": float(np.median(deg)) if self.n else 0.0,
                "mean_degree": float(deg.mean()) if self.n else 0.0,
                "isolated": int((deg == 0).sum()), "degree_one": int((deg == 1).sum())}


def key(seed: int, stream: int) -> int:
    return int(_load().gg_key(seed, stream))


def draws(k: int, first: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    _load().gg_draws(k, first, count, _p(out))
    return out


def from_edges(n: int, src, dst, symmetric: bool = True, drop_loops: bool = True,
               dedupe: bool = True, row_ptr_64: bool = False, name: str = "edges") -> Graph:
    """Build a CSR with sorted adjacency lists from an edge list."""
    src = np.ascontiguousarray(src, dtype=np.uint32)
    dst = np.ascontiguousarray(dst, dtype=np.uint32)
    m = int(src.shape[0])
    if dst.shape[0] != m:
        raise ValueError("src and dst differ in length")
    row_ptr = np.empty(n + 1, dtype=np.int64)
    cap = max(1, 2 * m if symmetric else m)
    col = np.empty(cap, dtype=np.int32)
    nnz = _load().gg_build_csr(n, m, _p(src), _p(dst), int(symmetric), int(drop_loops),
                               int(dedupe), _p(row_ptr), _p(col), cap)
    if nnz < 0:
        raise ValueError("gg_build_csr failed with code %d" % nnz)
    col = col[:nnz].copy() if nnz < cap else col
    if not row_ptr_64:
        if nnz >= 2**31:
            raise ValueError("int32 row_ptr cannot hold %d entries" % nnz)
        row_ptr = row_ptr.astype(np.int32)
    return Graph(name=name, row_ptr=row_ptr, col=col, symmetric=symmetric)


def from_csr(row_ptr, col, symmetric: bool, name: str = "csr") -> Graph:
    row_ptr = np.ascontiguousarray(row_ptr)
    if row_ptr.dtype not in (np.int32, np.int64):
        row_ptr = row_ptr.astype(np.int64)
    return Graph(name=name, row_ptr=row_ptr, col=np.ascontiguousarray(col, dtype=np.int32),
                 symmetric=symmetric)


def pick_sources(g: Graph, count: int, seed: int) -> np.ndarray:
    rp = np.ascontiguousarray(g.row_ptr, dtype=np.int64)
    out = np.empty(max(count, 1), dtype=np.int32)
    found = _load().gg_pick_sources(g.n, _p(rp), count, key(seed, STREAM_SOURCES),
                                    max(1000 * count, 10**6), _p(out))
    return out[:found].copy()


# ---------------------------------------------------------------- generators

def rmat(scale: int, edge_factor: int, seed: int, a=0.57, b=0.19, c=0.19,
         row_ptr_64: bool = False, name: str | None = None) -> Graph:
    n = 1 << scale
    m = edge_factor * n
    lib = _load()
    src = np.empty(m, dtype=np.uint32)
    dst = np.empty(m, dtype=np.uint32)
    lib.gg_rmat_edges(scale, m, a, b, c, key(seed, STREAM_EDGES), _p(src), _p(dst))
    perm = np.empty(n, dtype=np.uint32)
    lib.gg_permutation(n, key(seed, STREAM_PERM), _p(perm))
    lib.gg_relabel(m, _p(perm), _p(src), _p(dst))
    del perm
    g = from_edges(n, src, dst, symmetric=True, row_ptr_64=row_ptr_64,
                   name=name or "rmat_%d" % scale)
    g.meta.update(recipe="rmat", scale=scale, edge_factor=edge_factor, generated_edges=m,
                  seed=seed, abcd=[a, b, c, round(1 - a - b - c, 12)])
    return g


def uniform(n: int, m: int, seed: int, name: str | None = None) -> Graph:
    src = np.empty(m, dtype=np.uint32)
    dst = np.empty(m, dtype=np.uint32)
    _load().gg_uniform_edges(n, m, key(seed, STREAM_EDGES), _p(src), _p(dst))
    g = from_edges(n, src, dst, symmetric=True, name=name or "er_%d" % n)
    g.meta.update(recipe="uniform_pairs", generated_edges=m, seed=seed)
    return g


def grid(rows: int, cols: int, p_delete: float, seed: int, name: str | None = None) -> Graph:
    cap = rows * (cols - 1) + (rows - 1) * cols
    src = np.empty(max(cap, 1), dtype=np.uint32)
    dst = np.empty(max(cap, 1), dtype=np.uint32)
    kept = _load().gg_grid_edges(rows, cols, p_delete, key(seed, STREAM_EDGES), _p(src), _p(dst))
    g = from_edges(rows * cols, src[:kept], dst[:kept], symmetric=True,
                   name=name or "grid_%dx%d" % (rows, cols))
    g.meta.update(recipe="grid", rows=rows, cols=cols, p_delete=p_delete, seed=seed)
    return g


def chung_lu(weights, seed: int, name: str = "chung_lu") -> Graph:
    w = np.ascontiguousarray(weights, dtype=np.float64)
    n = int(w.shape[0])
    lib = _load()
    cap = 1 << 16
    while True:
        src = np.empty(cap, dtype=np.uint32)
        dst = np.empty(cap, dtype=np.uint32)
        kept = lib.gg_chung_lu_edges(n, _p(w), key(seed, STREAM_EDGES), cap, _p(src), _p(dst))
        if kept <= cap:
            break
        cap = int(kept)
    g = from_edges(n, src[:kept], dst[:kept], symmetric=True, name=name)
    g.meta.update(recipe="chung_lu", seed=seed)
    return g


# Config 1 weights: w = w_min / (1 - u)^(1/(gamma-1)) with gamma = 2, capped at
# W_CAP; the two largest are replaced by hub weights calibrated so that the
# realised hub degrees land near the page's 1,255 and 1,012.
POWERLAW_N = 3485
POWERLAW_W_MIN = 1.4
POWERLAW_W_CAP = 300.0
POWERLAW_HUBS = (3150.0, 2300.0)


def powerlaw_weights(seed: int) -> np.ndarray:
    u = draws(key(seed, STREAM_WEIGHTS), 0, POWERLAW_N).astype(np.float64)
    u = np.floor(u / 2048.0) * (1.0 / 9007199254740992.0)  # top 53 bits, as the C side
    w = POWERLAW_W_MIN / (1.0 - u)
    w = np.minimum(w, POWERLAW_W_CAP)
    top = np.argsort(-w, kind="stable")[:2]
    w[top[0]], w[top[1]] = POWERLAW_HUBS
    return w


def powerlaw_3485(seed: int = 0) -> Graph:
    g = chung_lu(powerlaw_weights(seed), seed, name="powerlaw_3485")
    g.meta.update(stand_in_for="Day 38 word graph (3,485 vertices)")
    return g


# ----------------------------------------------------------------- configs

CONFIGS = {
    1: dict(name="powerlaw_3485", seed=0, sources=64),
    2: dict(name="er_2^20", seed=1, sources=64),
    3: dict(name="rmat_22", seed=2, sources=64),
    4: dict(name="grid_2048", seed=3, sources=1),
    5: dict(name="rmat_25", seed=4, sources=16),
}


def _generate(cfg: int) -> Graph:
    seed = CONFIGS[cfg]["seed"]
    if cfg == 1:
        return powerlaw_3485(seed)
    if cfg == 2:
        return uniform(1 << 20, 16 * (1 << 20) // 2, seed, name="er_2^20")
    if cfg == 3:
        return rmat(22, 16, seed, name="rmat_22")
    if cfg == 4:
        return grid(2048, 2048, 0.1, seed, name="grid_2048")
    if cfg == 5:
        return rmat(25, 16, seed, row_ptr_64=True, name="rmat_25")
    raise ValueError("unknown config %r" % cfg)


def _cache_dir() -> str:
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return os.environ.get("BFS_GRAPH_CACHE", os.path.join(root, ".graph_cache"))


def _source_digest() -> str:
    h = hashlib.sha256()
    for path in (_SRC, os.path.abspath(__file__)):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def config(cfg: int, cache: bool = True) -> Graph:
    """Generate (or load from the on-disk cache) workload ``cfg`` in 1..5."""
    spec = CONFIGS[cfg]
    path = os.path.join(_cache_dir(), "cfg%d_%s.npz" % (cfg, _source_digest()))
    if cache and os.path.exists(path):
        try:
            with np.load(path, allow_pickle=False) as z:
                g = Graph(name=spec["name"], row_ptr=z["row_ptr"], col=z["col"],
                          symmetric=True, sources=z["sources"])
                g.meta = {"cached": True}
                return g
        except (OSError, ValueError, KeyError):
            pass
    g = _generate(cfg)
    if cfg == 4:
        corners = [0, 2047, 2048 * 2047, 2048 * 2048 - 1]
        deg = g.degrees()
        g.sources = np.array([next(c for c in corners if deg[c] > 0)], dtype=np.int32)
    else:
        g.sources = pick_sources(g, spec["sources"], spec["seed"])
    if cache:
        try:
            os.makedirs(_cache_dir(), exist_ok=True)
            tmp = path + ".%d.tmp.npz" % os.getpid()
            np.savez(tmp, row_ptr=g.row_ptr, col=g.col, sources=g.sources)
            os.replace(tmp, path)
        except OSError:
            pass
    return g


# ------------------------------------------------------------ small graphs

def path_graph(n: int) -> Graph:
    v = np.arange(max(n - 1, 0), dtype=np.uint32)
    return from_edges(n, v, v + 1, name="path_%d" % n)


def star_graph(n: int) -> Graph:
    leaves = np.arange(1, n, dtype=np.uint32)
    return from_edges(n, np.zeros_like(leaves), leaves, name="star_%d" % n)


def clique_graph(n: int) -> Graph:
    i, j = np.triu_indices(n, 1)
    return from_edges(n, i, j, name="clique_%d" % n)


def random_graph(n: int, p: float, seed: int, directed: bool = False,
                 loops: bool = False) -> Graph:
    """G(n, p) on all ordered (directed) or unordered pairs, counter-seeded."""
    r = draws(key(seed, STREAM_EDGES), 0, n * n).reshape(n, n)
    keep = (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0) < p
    if not directed:
        keep = np.triu(keep, 0 if loops else 1)
    if not loops:
        np.fill_diagonal(keep, False)
    i, j = np.nonzero(keep)
    return from_edges(n, i, j, symmetric=not directed, drop_loops=not loops,
                      name="gnp_%d_%g_%d%s" % (n, p, seed, "_dir" if directed else ""))
