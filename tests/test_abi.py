"""The C-ABI boundary without a GPU: the library loads, exports every function
the header declares, its structs match the header's layout, and the pure host
entry points (defaults, workspace sizing, status strings, argument checks)
behave as documented."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bfs_csr.h")


@pytest.fixture(scope="module")
def fbc():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import frontier_bfs_csr_gb300
    return frontier_bfs_csr_gb300


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bfs_csr_[a-z_0-9]+)\s*\(", text)))


def test_header_functions_exported(fbc):
    declared = _declared_functions()
    assert len(declared) >= 10
    lib = ctypes.CDLL(fbc.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(fbc.EXPORTED) == declared
    out = subprocess.run(["nm", "-D", "--defined-only", fbc.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for name in declared:
        assert re.search(r"\bT %s$" % name, out, flags=re.M), name


def _c_layout():
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "bfs_csr.h"
#define F(s, m) printf("%s.%s %zu\n", #s, #m, offsetof(s, m))
int main(void) {
  printf("sizeof_options %zu\n", sizeof(bfs_csr_options));
  printf("sizeof_stat %zu\n", sizeof(bfs_csr_level_stat));
  F(bfs_csr_options, direction); F(bfs_csr_options, advance); F(bfs_csr_options, discovery);
  F(bfs_csr_options, loop_mode); F(bfs_csr_options, small_max_degree);
  F(bfs_csr_options, cta_min_degree); F(bfs_csr_options, merge_path_min_frontier);
  F(bfs_csr_options, binned_max_degree); F(bfs_csr_options, pull_alpha);
  F(bfs_csr_options, max_depth); F(bfs_csr_options, validate); F(bfs_csr_options, block_threads);
  F(bfs_csr_options, grid_blocks); F(bfs_csr_options, barrier_timeout_ns);
  F(bfs_csr_options, test_unreachable_barrier); F(bfs_csr_options, push_beta);
  F(bfs_csr_options, narrow_max_edges); F(bfs_csr_options, lanes);
  F(bfs_csr_options, parent_pass); F(bfs_csr_options, frontier_output);
  F(bfs_csr_options, reserved);
  F(bfs_csr_level_stat, level); F(bfs_csr_level_stat, direction); F(bfs_csr_level_stat, advance);
  F(bfs_csr_level_stat, frontier); F(bfs_csr_level_stat, frontier_edges);
  F(bfs_csr_level_stat, unvisited); F(bfs_csr_level_stat, max_degree);
  F(bfs_csr_level_stat, t_start_ns); F(bfs_csr_level_stat, t_work_ns);
  return 0;
}
'''
    os.makedirs(os.path.join(ROOT, "_build"), exist_ok=True)
    with tempfile.TemporaryDirectory(dir=os.path.join(ROOT, "_build")) as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        with open(c, "w") as f:
            f.write(src)
        subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}


def test_struct_layouts_match_header(fbc):
    lay = _c_layout()
    assert ctypes.sizeof(fbc.bfs_csr_options) == lay["sizeof_options"]
    assert ctypes.sizeof(fbc.bfs_csr_level_stat) == lay["sizeof_stat"]
    for name, _ in fbc.bfs_csr_options._fields_:
        assert getattr(fbc.bfs_csr_options, name).offset == lay["bfs_csr_options." + name], name
    for name in ("level", "direction", "advance", "frontier", "frontier_edges", "unvisited",
                 "max_degree", "t_start_ns", "t_work_ns"):
        assert getattr(fbc.bfs_csr_level_stat, name).offset == lay["bfs_csr_level_stat." + name], name


def test_defaults(fbc):
    o = fbc.default_options()
    assert o.direction == fbc.BFS_CSR_DIR_AUTO and o.advance == fbc.BFS_CSR_ADV_AUTO
    assert o.discovery == fbc.BFS_CSR_DISC_BITMAP and o.loop_mode == fbc.BFS_CSR_LOOP_PERSISTENT
    assert (o.small_max_degree, o.cta_min_degree) == (32, 256)
    assert o.merge_path_min_frontier == 4096  # Gunrock paper's static hybrid threshold
    assert o.pull_alpha == 14.0 and o.push_beta == 24
    assert o.max_depth == -1 and o.validate == 1 and o.lanes == 1
    assert o.parent_pass == fbc.BFS_CSR_PARENT_AUTO
    assert o.barrier_timeout_ns > 0 and o.test_unreachable_barrier == 0


def test_workspace_sizing(fbc):
    small = fbc.workspace_bytes(1000, 5000, False)
    big = fbc.workspace_bytes(2000, 5000, False)
    wide = fbc.workspace_bytes(1000, 5000, True)
    assert 0 < small < big and small < wide
    # queues (2 x n int32) + offsets and row starts (4 x n x 4 or 8 bytes) dominate
    n = 1 << 20
    assert fbc.workspace_bytes(n, 16 * n, False) >= n * (8 + 16)
    assert fbc.workspace_bytes(n, 16 * n, True) >= n * (8 + 32)
    # the padded frontier modes add two arrays of nnz int32 per lane
    pad = fbc.workspace_bytes(n, 16 * n, False, fbc.default_options(frontier_output=2))
    assert pad - fbc.workspace_bytes(n, 16 * n, False) >= 2 * 16 * n * 4
    # every lane adds one search part; the graph part (probe array) is shared
    one = fbc.workspace_bytes(n, 16 * n, False, fbc.default_options(lanes=1))
    two = fbc.workspace_bytes(n, 16 * n, False, fbc.default_options(lanes=2))
    three = fbc.workspace_bytes(n, 16 * n, False, fbc.default_options(lanes=3))
    assert one < two < three and three - two == two - one and two - one < one
    assert fbc.workspace_bytes(n, 16 * n, False, fbc.default_options(lanes=0)) == one


def test_argument_checks_without_gpu(fbc):
    out = ctypes.c_size_t(0)
    assert fbc.bfs_csr_workspace_bytes(0, 0, 0, None, ctypes.byref(out)) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_workspace_bytes(1 << 31, 0, 0, None, ctypes.byref(out)) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_workspace_bytes(10, 1 << 31, 0, None, ctypes.byref(out)) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_workspace_bytes(10, -1, 0, None, ctypes.byref(out)) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_workspace_bytes(10, 1 << 31, 1, None, ctypes.byref(out)) == fbc.BFS_CSR_OK
    bad = fbc.default_options(direction=7)
    assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
        fbc.BFS_CSR_EINVAL
    bad = fbc.default_options(cta_min_degree=4, small_max_degree=8)
    assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
        fbc.BFS_CSR_EINVAL
    bad = fbc.default_options(block_threads=100)
    assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
        fbc.BFS_CSR_EINVAL
    for pp in (-1, 3):
        bad = fbc.default_options(parent_pass=pp)
        assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
            fbc.BFS_CSR_EINVAL
        bad = fbc.default_options(frontier_output=pp)
        assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
            fbc.BFS_CSR_EINVAL
        bad = fbc.default_options(discovery=pp)
        assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
            fbc.BFS_CSR_EINVAL
    for lanes in (-1, 9):
        bad = fbc.default_options(lanes=lanes)
        assert fbc.bfs_csr_workspace_bytes(10, 10, 0, ctypes.byref(bad), ctypes.byref(out)) == \
            fbc.BFS_CSR_EINVAL
    src = (ctypes.c_int64 * 1)(0)
    assert fbc.bfs_csr_run_batch(None, 1, src, None, None, None, None, None) == fbc.BFS_CSR_EINVAL
    h = ctypes.c_void_p()
    assert fbc.bfs_csr_create(None, 1, 0, None, 0, None, 1, None, 0, None, None) == \
        fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_create(ctypes.byref(h), 5, 3, None, 0, None, 1, None, 0, None, None) == \
        fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_run(None, 0, None, None, None, None) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_sync(None, None, None) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_destroy(None) == fbc.BFS_CSR_EINVAL
    assert fbc.bfs_csr_last_cuda_error(None) == 0


def test_status_strings(fbc):
    seen = set()
    for code in range(7):
        s = fbc.bfs_csr_status_string(code).decode()
        assert s and s not in seen
        seen.add(s)
    assert fbc.bfs_csr_status_string(99).decode() == "unknown status"
