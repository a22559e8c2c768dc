"""CPU oracle for level-synchronous BFS over CSR -- TEST INFRASTRUCTURE.

The oracle is a plain sequential C library (``bfs_oracle.c``) plus this thin
ctypes wrapper. It exists to check the CUDA path, and only the test suite,
the package smoke check and the benchmark's CPU-baseline leg may import it.
It shares no code with the CUDA library and does not import it.

What each function computes and which passage of the pages it follows is
written at the top of ``bfs_oracle.c``. In short:

* :func:`bfs` -- FIFO-queue BFS ("100 Days of GPU, Day 38", the host BFS;
  "The Frontier Model for Parallel BFS", section 22.1). Returns exact hop
  distances (-1 = unreached), the FIFO first-discoverer parent array
  (parent[source] = source) and the number of non-empty frontiers.
* :func:`bfs` with ``max_depth`` -- the same search stopped after the
  frontiers up to that depth (section 22.1's mid-search state).
* :func:`check_dist` -- the three-invariant certificate of exact distances.
* :func:`check_parent` -- BFS-tree validity (every parent is an in-neighbour
  one level up).
* :func:`level_sizes` -- per-level frontier sizes and the walked-edge count.
* :func:`walk_checksum` -- what the isolated neighbour walk of a frontier
  returns per slot ("100 Days of GPU, Day 38", "Measuring the mapping
  without measuring the launch").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bfs_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
EARG = -1
ENOMEM = -2


def build(force: bool = False) -> str:
    """Compile ``bfs_oracle.c`` into ``liboracle.so`` (plain gcc, -O2)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra",
                               "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_bfs_depth.argtypes = [i64, vp, i32, vp, i64, i64, vp, vp, vp]
            lib.oracle_bfs_depth.restype = i32
            lib.oracle_check_dist.argtypes = [i64, vp, i32, vp, i64, vp, vp]
            lib.oracle_check_dist.restype = i32
            lib.oracle_check_parent.argtypes = [i64, vp, i32, vp, i64, vp, vp, vp]
            lib.oracle_check_parent.restype = i32
            lib.oracle_level_sizes.argtypes = [i64, vp, i32, vp, vp, i64, vp, vp, vp]
            lib.oracle_level_sizes.restype = i32
            lib.oracle_walk_checksum.argtypes = [i64, vp, i32, vp, vp, i64, i64, vp]
            lib.oracle_walk_checksum.restype = i32
            _lib = lib
    return _lib


def _csr(row_ptr, col):
    row_ptr = np.ascontiguousarray(row_ptr)
    if row_ptr.dtype not in (np.int32, np.int64):
        row_ptr = row_ptr.astype(np.int64)
    col = np.ascontiguousarray(col, dtype=np.int32)
    n = row_ptr.shape[0] - 1
    return n, row_ptr, int(row_ptr.dtype == np.int64), col


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def bfs(row_ptr, col, source: int, max_depth: int = -1, want_parent: bool = True):
    """FIFO BFS. Returns ``(dist, parent, num_levels)``; parent is None if not wanted."""
    lib = _load()
    n, rp, rp64, col = _csr(row_ptr, col)
    dist = np.empty(n, dtype=np.int32)
    parent = np.empty(n, dtype=np.int32) if want_parent else None
    levels = ctypes.c_int64(0)
    rc = lib.oracle_bfs_depth(n, _ptr(rp), rp64, _ptr(col), int(source), int(max_depth),
                              _ptr(dist), _ptr(parent), ctypes.byref(levels))
    if rc != OK:
        raise ValueError("oracle_bfs failed with code %d" % rc)
    return dist, parent, int(levels.value)


def check_dist(row_ptr, col, source: int, dist):
    """Return ``(code, bad_vertex)``; code 0 means dist is the exact hop distance."""
    lib = _load()
    n, rp, rp64, col = _csr(row_ptr, col)
    dist = np.ascontiguousarray(dist, dtype=np.int32)
    bad = ctypes.c_int64(-1)
    rc = lib.oracle_check_dist(n, _ptr(rp), rp64, _ptr(col), int(source), _ptr(dist),
                               ctypes.byref(bad))
    return int(rc), int(bad.value)


def check_parent(row_ptr, col, source: int, dist, parent):
    """Return ``(code, bad_vertex)``; code 0 means parent is a valid BFS tree for dist."""
    lib = _load()
    n, rp, rp64, col = _csr(row_ptr, col)
    dist = np.ascontiguousarray(dist, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    bad = ctypes.c_int64(-1)
    rc = lib.oracle_check_parent(n, _ptr(rp), rp64, _ptr(col), int(source), _ptr(dist),
                                 _ptr(parent), ctypes.byref(bad))
    return int(rc), int(bad.value)


def level_sizes(row_ptr, dist, level_cap: int | None = None):
    """Return ``(sizes, num_levels, reached, edges_walked)`` for a distance array."""
    lib = _load()
    row_ptr = np.ascontiguousarray(row_ptr)
    if row_ptr.dtype not in (np.int32, np.int64):
        row_ptr = row_ptr.astype(np.int64)
    n = row_ptr.shape[0] - 1
    dist = np.ascontiguousarray(dist, dtype=np.int32)
    if level_cap is None:
        level_cap = int(dist.max()) + 1 if n > 0 else 0
    sizes = np.zeros(max(level_cap, 1), dtype=np.int64)
    nl, reached, edges = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib.oracle_level_sizes(n, _ptr(row_ptr), int(row_ptr.dtype == np.int64), _ptr(dist),
                                _ptr(sizes), int(level_cap), ctypes.byref(nl),
                                ctypes.byref(reached), ctypes.byref(edges))
    if rc != OK:
        raise ValueError("oracle_level_sizes failed with code %d" % rc)
    return sizes[:level_cap], int(nl.value), int(reached.value), int(edges.value)


def walk_checksum(row_ptr, col, frontier, repeats: int):
    """Per frontier slot: the wrapping 32-bit sum over r < repeats and the
    entries e of the slot's row of col[e] XOR r (uint32 array)."""
    lib = _load()
    n, rp, rp64, col = _csr(row_ptr, col)
    fr = np.ascontiguousarray(frontier, dtype=np.int32)
    out = np.zeros(fr.shape[0], dtype=np.uint32)
    rc = lib.oracle_walk_checksum(n, _ptr(rp), rp64, _ptr(col), _ptr(fr), int(fr.shape[0]),
                                  int(repeats), _ptr(out))
    if rc != OK:
        raise ValueError("oracle_walk_checksum failed with code %d" % rc)
    return out
