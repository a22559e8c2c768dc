"""Host-side arithmetic of bench.py, on the CPU: the union of the searches'
level-loop intervals (the roofline's time base when searches overlap) and
the algorithmic byte model, against counts done by hand on tiny graphs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
import graphgen  # noqa: E402


def test_busy_time_is_the_union_of_intervals():
    assert bench.busy_time([]) == 0.0
    assert bench.busy_time([(0.0, 2.0)]) == 2.0
    assert bench.busy_time([(0.0, 2.0), (1.0, 3.0)]) == 3.0            # overlap
    assert bench.busy_time([(0.0, 1.0), (2.0, 3.0)]) == 2.0            # gap
    assert bench.busy_time([(2.0, 3.0), (0.0, 5.0), (1.0, 2.0)]) == 5.0  # nested, unsorted
    assert bench.busy_time([(0.0, 1.0), (1.0, 2.0)]) == 2.0            # touching


def _model(g, dist, dirs):
    rp = torch.from_numpy(g.row_ptr.astype(np.int64))
    col = torch.from_numpy(g.col)
    deg = torch.diff(rp)
    src_of_edge = torch.repeat_interleave(torch.arange(g.n, dtype=torch.int32), deg)
    stats = [{"direction": d} for d in dirs]
    return bench.algorithmic_bytes(torch, rp, col, deg, src_of_edge,
                                   torch.tensor(dist, dtype=torch.int32), stats, 4)


def test_byte_model_push_levels_by_hand():
    # path 0-1-2 from 0, int32 row_ptr (R = 4): per push level
    # (4+2R)|Q| + 4 m_F + 4 m_F + 2R|N| + 8|N| + 4|N| + (4+2R)|N'|
    g = graphgen.path_graph(3)
    total, per_level = _model(g, [0, 1, 2], [bench.DIR_PUSH] * 3)
    assert per_level == [12 + 4 + 4 + 8 + 8 + 4 + 12,    # F = {0}, m_F = 1, N = {1}
                         12 + 8 + 8 + 8 + 8 + 4 + 12,    # F = {1}, m_F = 2, N = {2}
                         12 + 4 + 4]                      # F = {2}, m_F = 1, N = {}
    assert total == sum(per_level)


def test_byte_model_pull_level_and_switches_by_hand():
    # star 0-{1,2,3} from leaf 1: push, pull, push; plus one isolated vertex 4
    g = graphgen.from_edges(5, [0, 0, 0], [1, 2, 3])
    total, per_level = _model(g, [1, 0, 2, 2, -1],
                              [bench.DIR_PUSH, bench.DIR_PULL, bench.DIR_PUSH])
    words = 1
    push0 = 12 + 4 + 4 + 8 + 8 + 4 + 12                  # F = {1}, N = {0}
    to_bitmap = 4 * words + 8 * 1                         # queue {0} -> bitmap
    # pull over U' = {2, 3}: each scans one entry (its only neighbour, 0, is in F)
    pull1 = 4 * words + 8 * 2 + 4 * 2 + 4 * 2 + 8 * 2 + 4 * words + 4 * 1
    to_queue = 4 * words + 8 * 2 + 12 * 2                 # bitmap {2, 3} -> queue
    push2 = 12 * 2 + 4 * 2 + 4 * 2                        # F = {2, 3}, N = {}
    assert per_level == [push0, to_bitmap + pull1, to_queue + push2]
    assert total == sum(per_level) + 4 * 1                # dist of the unreached vertex 4
