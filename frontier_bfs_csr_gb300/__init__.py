"""Level-synchronous frontier BFS over CSR on one GB300 (sm_103a).

This package is a thin ctypes binding over the C-ABI library
``libbfs_csr.so`` (declared in ``include/bfs_csr.h``). Every step of a search
runs in that library's CUDA kernels; this module only marshals arguments.
PyTorch supplies device memory and streams. There is no CPU fallback: if the
library has not been built (``python frontier_bfs_csr_gb300/build.py`` or
``__graft_entry__.build()``), importing the binding fails.

The functions below carry the C names. :class:`BfsCsr` wraps a handle for
the common case of torch tensors on the current device.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbfs_csr.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libbfs_csr.so is not built (expected at %s); run "
        "`python frontier_bfs_csr_gb300/build.py`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants
BFS_CSR_OK = 0
BFS_CSR_EINVAL = 1
BFS_CSR_ENOMEM = 2
BFS_CSR_ECUDA = 3
BFS_CSR_ETIMEOUT = 4
BFS_CSR_EUNSUPPORTED = 5
BFS_CSR_EDEVICE = 6

BFS_CSR_DIR_AUTO, BFS_CSR_DIR_PUSH, BFS_CSR_DIR_PULL = 0, 1, 2
BFS_CSR_ADV_AUTO, BFS_CSR_ADV_BINNED, BFS_CSR_ADV_MERGE_PATH, BFS_CSR_ADV_SINGLE_CTA = 0, 1, 2, 3
BFS_CSR_ADV_PADDED = 4
BFS_CSR_DISC_BITMAP, BFS_CSR_DISC_CAS, BFS_CSR_DISC_MIN = 0, 1, 2
BFS_CSR_FRONTIER_COMPACT, BFS_CSR_FRONTIER_PADDED_FILTER, BFS_CSR_FRONTIER_PADDED = 0, 1, 2
BFS_CSR_LOOP_PERSISTENT, BFS_CSR_LOOP_HOST, BFS_CSR_LOOP_GRAPH = 0, 1, 2
BFS_CSR_PARENT_AUTO, BFS_CSR_PARENT_END_PASS, BFS_CSR_PARENT_AT_DISCOVERY = 0, 1, 2
BFS_CSR_WALK_THREAD, BFS_CSR_WALK_WARP, BFS_CSR_WALK_BINNED, BFS_CSR_WALK_EDGE = 0, 1, 2, 3

EXPORTED = [
    "bfs_csr_default_options", "bfs_csr_workspace_bytes", "bfs_csr_create", "bfs_csr_run",
    "bfs_csr_run_init", "bfs_csr_run_levels",
    "bfs_csr_sync", "bfs_csr_level_stats", "bfs_csr_create_host", "bfs_csr_run_host",
    "bfs_csr_run_host_batch", "bfs_csr_destroy", "bfs_csr_status_string", "bfs_csr_last_cuda_error",
    "bfs_csr_run_noalloc", "bfs_csr_run_batch", "bfs_csr_walk",
]
BFS_CSR_NOALLOC_MAX_VERTICES = 1048576


class bfs_csr_options(ctypes.Structure):
    _fields_ = [
        ("direction", ctypes.c_int32),
        ("advance", ctypes.c_int32),
        ("discovery", ctypes.c_int32),
        ("loop_mode", ctypes.c_int32),
        ("small_max_degree", ctypes.c_int32),
        ("cta_min_degree", ctypes.c_int32),
        ("merge_path_min_frontier", ctypes.c_int32),
        ("binned_max_degree", ctypes.c_int32),
        ("pull_alpha", ctypes.c_double),
        ("max_depth", ctypes.c_int32),
        ("validate", ctypes.c_int32),
        ("block_threads", ctypes.c_int32),
        ("grid_blocks", ctypes.c_int32),
        ("barrier_timeout_ns", ctypes.c_int64),
        ("test_unreachable_barrier", ctypes.c_int32),
        ("push_beta", ctypes.c_int32),
        ("narrow_max_edges", ctypes.c_int32),
        ("lanes", ctypes.c_int32),
        ("parent_pass", ctypes.c_int32),
        ("frontier_output", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 2),
    ]


class bfs_csr_level_stat(ctypes.Structure):
    _fields_ = [
        ("level", ctypes.c_int32),
        ("direction", ctypes.c_int32),
        ("advance", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("frontier", ctypes.c_int64),
        ("frontier_edges", ctypes.c_int64),
        ("unvisited", ctypes.c_int64),
        ("max_degree", ctypes.c_int64),
        ("t_start_ns", ctypes.c_int64),
        ("t_work_ns", ctypes.c_int64),
    ]


_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_opt_p = ctypes.POINTER(bfs_csr_options)
_sig = {
    "bfs_csr_default_options": ([_opt_p], _i32),
    "bfs_csr_workspace_bytes": ([_i64, _i64, _i32, _opt_p, ctypes.POINTER(_sz)], _i32),
    "bfs_csr_create": ([ctypes.POINTER(_vp), _i64, _i64, _vp, _i32, _vp, _i32, _vp, _sz, _opt_p,
                        _vp], _i32),
    "bfs_csr_run": ([_vp, _i64, _vp, _vp, _vp, _vp], _i32),
    "bfs_csr_run_init": ([_vp, _i64, _vp, _vp, _vp], _i32),
    "bfs_csr_run_levels": ([_vp, _vp, _vp], _i32),
    "bfs_csr_sync": ([_vp, _vp, ctypes.POINTER(ctypes.c_int32)], _i32),
    "bfs_csr_level_stats": ([_vp, ctypes.POINTER(bfs_csr_level_stat), ctypes.c_int32,
                             ctypes.POINTER(ctypes.c_int32)], _i32),
    "bfs_csr_create_host": ([ctypes.POINTER(_vp), _i64, _i64, _vp, _i32, _vp, _i32, _opt_p, _vp],
                            _i32),
    "bfs_csr_run_host": ([_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "bfs_csr_run_host_batch": ([_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "bfs_csr_destroy": ([_vp], _i32),
    "bfs_csr_status_string": ([_i32], ctypes.c_char_p),
    "bfs_csr_last_cuda_error": ([_vp], _i32),
    "bfs_csr_run_noalloc": ([_i64, _i64, _vp, _vp, _i32, _i64, _vp, _vp, _vp,
                             ctypes.POINTER(ctypes.c_int32), _opt_p, _vp], _i32),
    "bfs_csr_run_batch": ([_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "bfs_csr_walk": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
}
for _name, (_args, _res) in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res
    globals()[_name] = _f


class BfsError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = bfs_csr_status_string(status).decode()
        super().__init__("%s: %s (status %d)" % (what, msg, status) if what else msg)


def _check(status: int, what: str, handle=None):
    if status != BFS_CSR_OK:
        err = BfsError(status, what)
        if handle is not None and status == BFS_CSR_ECUDA:
            err.cuda_error = bfs_csr_last_cuda_error(handle)
        raise err


def default_options(**overrides) -> bfs_csr_options:
    opt = bfs_csr_options()
    _check(bfs_csr_default_options(ctypes.byref(opt)), "bfs_csr_default_options")
    for k, v in overrides.items():
        if not hasattr(opt, k):
            raise AttributeError("bfs_csr_options has no field %r" % k)
        setattr(opt, k, v)
    return opt


def workspace_bytes(n: int, nnz: int, row_ptr_64: bool, options=None) -> int:
    out = _sz(0)
    opt = ctypes.byref(options) if options is not None else None
    _check(bfs_csr_workspace_bytes(n, nnz, int(row_ptr_64), opt, ctypes.byref(out)),
           "bfs_csr_workspace_bytes")
    return int(out.value)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class BfsCsr:
    """A search handle over a device CSR held in torch tensors.

    ``row_ptr`` (int32 or int64, n + 1) and ``col`` (int32, nnz) must be
    contiguous CUDA tensors that outlive the handle. The workspace is a torch
    uint8 tensor owned by this object.
    """

    def __init__(self, row_ptr, col, symmetric: bool = True, options=None, stream=None):
        import torch
        if not (row_ptr.is_cuda and col.is_cuda):
            raise ValueError("row_ptr and col must be CUDA tensors")
        if row_ptr.dtype not in (torch.int32, torch.int64) or col.dtype != torch.int32:
            raise ValueError("row_ptr must be int32/int64 and col int32")
        self.row_ptr = row_ptr.contiguous()
        self.col = col.contiguous()
        self.n = int(row_ptr.numel() - 1)
        self.nnz = int(col.numel())
        self.row_ptr_64 = row_ptr.dtype == torch.int64
        self.symmetric = bool(symmetric)
        self.options = options if options is not None else default_options()
        nbytes = workspace_bytes(self.n, self.nnz, self.row_ptr_64, self.options)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=row_ptr.device)
        h = _vp()
        status = bfs_csr_create(ctypes.byref(h), self.n, self.nnz, self.row_ptr.data_ptr(),
                                int(self.row_ptr_64),
                                self.col.data_ptr() if self.nnz else None,
                                int(self.symmetric), self.workspace.data_ptr(), nbytes,
                                ctypes.byref(self.options), _stream_ptr(stream))
        _check(status, "bfs_csr_create")
        self.handle = h

    def run(self, source: int, dist, parent=None, num_levels=None, stream=None) -> None:
        """Enqueue a search; results land in the given int32 CUDA tensors."""
        status = bfs_csr_run(self.handle, int(source), dist.data_ptr(),
                             parent.data_ptr() if parent is not None else None,
                             num_levels.data_ptr() if num_levels is not None else None,
                             _stream_ptr(stream))
        _check(status, "bfs_csr_run", self.handle)

    def run_init(self, source: int, dist, parent=None, stream=None) -> None:
        """First half of :meth:`run`: reset and seed (one kernel)."""
        status = bfs_csr_run_init(self.handle, int(source), dist.data_ptr(),
                                  parent.data_ptr() if parent is not None else None,
                                  _stream_ptr(stream))
        _check(status, "bfs_csr_run_init", self.handle)

    def run_levels(self, num_levels=None, stream=None) -> None:
        """Second half of :meth:`run`: the level loop."""
        status = bfs_csr_run_levels(self.handle,
                                    num_levels.data_ptr() if num_levels is not None else None,
                                    _stream_ptr(stream))
        _check(status, "bfs_csr_run_levels", self.handle)

    def sync(self, stream=None) -> int:
        levels = ctypes.c_int32(0)
        _check(bfs_csr_sync(self.handle, _stream_ptr(stream), ctypes.byref(levels)),
               "bfs_csr_sync", self.handle)
        return int(levels.value)

    def run_batch(self, sources, dist, parent=None, num_levels=None, stamps=None,
                  stream=None) -> None:
        """Search from every source (waits): row i of dist / parent (int32 CUDA
        tensors of len(sources) x n) gets source i's result, num_levels[i]
        (int32 CUDA tensor) its level count. The searches run on the handle's
        options.lanes lanes at once. stamps: int64 CUDA tensor of
        3 x len(sources) for the device timer (ns) at each search's init,
        level-loop start and level-loop end, or None."""
        import numpy as np
        src = np.ascontiguousarray(np.asarray(sources, dtype=np.int64))
        k = int(src.shape[0])
        for a in (dist, parent):
            if a is not None and (a.numel() != k * self.n or not a.is_contiguous()):
                raise ValueError("dist/parent must be contiguous len(sources) x n tensors")
        status = bfs_csr_run_batch(self.handle, k, src.ctypes.data, dist.data_ptr(),
                                   parent.data_ptr() if parent is not None else None,
                                   num_levels.data_ptr() if num_levels is not None else None,
                                   stamps.data_ptr() if stamps is not None else None,
                                   _stream_ptr(stream))
        _check(status, "bfs_csr_run_batch", self.handle)

    def walk(self, frontier, repeats: int, mapping: int, out, stream=None) -> None:
        """Enqueue the isolated neighbour walk of `frontier` (int32 CUDA
        tensor of vertex ids): out[i] (int32 or uint32 CUDA tensor, same
        length) gets the wrapping 32-bit sum over r < repeats and the entries
        e of frontier[i]'s row of col[e] XOR r."""
        size = int(frontier.numel())
        if out.numel() != size or not (frontier.is_contiguous() and out.is_contiguous()):
            raise ValueError("frontier and out must be contiguous and of the same length")
        status = bfs_csr_walk(self.handle, frontier.data_ptr() if size else None, size,
                              int(repeats), int(mapping), out.data_ptr() if size else None,
                              _stream_ptr(stream))
        _check(status, "bfs_csr_walk", self.handle)

    def search(self, source: int, want_parent: bool = True, stream=None):
        """Run one search and wait: returns (dist, parent or None, num_levels)."""
        import torch
        dev = self.row_ptr.device
        dist = torch.empty(self.n, dtype=torch.int32, device=dev)
        parent = torch.empty(self.n, dtype=torch.int32, device=dev) if want_parent else None
        self.run(source, dist, parent, stream=stream)
        levels = self.sync(stream)
        return dist, parent, levels

    def level_stats(self):
        cap = 1 << 16
        buf = (bfs_csr_level_stat * cap)()
        count = ctypes.c_int32(0)
        _check(bfs_csr_level_stats(self.handle, buf, cap, ctypes.byref(count)),
               "bfs_csr_level_stats")
        out = []
        for i in range(min(int(count.value), cap)):
            s = buf[i]
            out.append({"level": s.level, "direction": s.direction, "advance": s.advance,
                        "frontier": s.frontier, "frontier_edges": s.frontier_edges,
                        "unvisited": s.unvisited, "max_degree": s.max_degree,
                        "t_start_ns": s.t_start_ns, "t_work_ns": s.t_work_ns})
        return out

    def close(self) -> None:
        if getattr(self, "handle", None):
            bfs_csr_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BfsCsrHost:
    """A handle whose CSR and results live in host memory (numpy arrays).

    The library keeps device copies; :meth:`run` optionally re-uploads the
    CSR, searches, and copies dist/parent back before returning.
    """

    def __init__(self, row_ptr, col, symmetric: bool = True, options=None, stream=None):
        import numpy as np
        self.row_ptr = np.ascontiguousarray(row_ptr)
        if self.row_ptr.dtype not in (np.int32, np.int64):
            raise ValueError("row_ptr must be int32 or int64")
        self.col = np.ascontiguousarray(col, dtype=np.int32)
        self.n = int(self.row_ptr.shape[0] - 1)
        self.nnz = int(self.col.shape[0])
        self.row_ptr_64 = self.row_ptr.dtype == np.int64
        self.options = options if options is not None else default_options()
        h = _vp()
        status = bfs_csr_create_host(ctypes.byref(h), self.n, self.nnz,
                                     self.row_ptr.ctypes.data, int(self.row_ptr_64),
                                     self.col.ctypes.data if self.nnz else None, int(symmetric),
                                     ctypes.byref(self.options), _stream_ptr(stream))
        _check(status, "bfs_csr_create_host")
        self.handle = h

    def run(self, source: int, dist, parent=None, row_ptr=None, col=None, stream=None) -> int:
        levels = ctypes.c_int32(0)
        status = bfs_csr_run_host(self.handle, int(source),
                                  row_ptr.ctypes.data if row_ptr is not None else None,
                                  col.ctypes.data if col is not None else None,
                                  dist.ctypes.data,
                                  parent.ctypes.data if parent is not None else None,
                                  ctypes.addressof(levels), _stream_ptr(stream))
        _check(status, "bfs_csr_run_host", self.handle)
        return int(levels.value)

    def run_batch(self, sources, dist, parent=None, levels=None, row_ptr=None, col=None,
                  stream=None) -> None:
        """Search from every source; row i of dist (and parent) is source i's
        result. dist/parent: C-contiguous int32 arrays of len(sources) x n
        (pinned for asynchronous copies); levels: int32 array of len(sources)
        or None. row_ptr/col re-upload the CSR first, as in :meth:`run`."""
        import numpy as np
        src = np.ascontiguousarray(np.asarray(sources, dtype=np.int64))
        k = int(src.shape[0])
        for a in (dist, parent):
            if a is not None and (a.dtype != np.int32 or a.size != k * self.n or
                                  not a.flags["C_CONTIGUOUS"]):
                raise ValueError("dist/parent must be C-contiguous int32 of len(sources) x n")
        if levels is not None and (levels.dtype != np.int32 or levels.size != k):
            raise ValueError("levels must be int32 of len(sources)")
        status = bfs_csr_run_host_batch(self.handle, k, src.ctypes.data,
                                        row_ptr.ctypes.data if row_ptr is not None else None,
                                        col.ctypes.data if col is not None else None,
                                        dist.ctypes.data,
                                        parent.ctypes.data if parent is not None else None,
                                        levels.ctypes.data if levels is not None else None,
                                        _stream_ptr(stream))
        _check(status, "bfs_csr_run_host_batch", self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            bfs_csr_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
