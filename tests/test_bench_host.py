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


def _counts(g, dist, dirs):
    rp = torch.from_numpy(g.row_ptr.astype(np.int64))
    col = torch.from_numpy(g.col)
    deg = torch.diff(rp)
    src_of_edge = torch.repeat_interleave(torch.arange(g.n, dtype=torch.int32), deg)
    stats = [{"direction": d, "advance": 0} for d in dirs]
    return bench.level_counts(torch, rp, col, deg, src_of_edge,
                              torch.tensor(dist, dtype=torch.int32), stats)


def test_byte_models_push_levels_by_hand():
    # path 0-1-2 from 0, int32 row_ptr (R = 4)
    g = graphgen.path_graph(3)
    counts = _counts(g, [0, 1, 2], [bench.DIR_PUSH] * 3)
    assert [(c["F"], c["mF"], c["N"]) for c in counts] == [(1, 1, 1), (1, 2, 1), (1, 1, 0)]
    # scope table, push: 4|F| + 2R|F| + 4 m_F (col) + 4 m_F (probe) + 8|N| + 4|N| + |N|/8
    assert [bench.survey_bytes(c, 3, 4) for c in counts] == [4 + 8 + 8 + 8 + 4,
                                                             4 + 8 + 16 + 8 + 4,
                                                             4 + 8 + 8]
    # the kernel: queue entries (4 + 2R) per vertex with edges, row offsets of
    # every winner 2R, queue entries written (4 + 2R)
    s_tot, k_tot, per = bench.search_bytes(counts, 3, 4, reached=3)
    assert per == [32, 40, 20] and s_tot == 92
    assert k_tot == (12 + 4 + 4 + 8 + 8 + 4 + 12) + (12 + 8 + 8 + 8 + 8 + 4 + 12) + (12 + 4 + 4)


def test_byte_models_pull_level_and_switches_by_hand():
    # star 0-{1,2,3} from leaf 1: push, pull, push; plus one isolated vertex 4
    g = graphgen.from_edges(5, [0, 0, 0], [1, 2, 3])
    counts = _counts(g, [1, 0, 2, 2, -1], [bench.DIR_PUSH, bench.DIR_PULL, bench.DIR_PUSH])
    # level 1 pulls over U = {2, 3} (vertex 4 has no edges): each finds its
    # only neighbour 0 after one entry
    assert (counts[1]["U"], counts[1]["c"], counts[1]["N"], counts[1]["tw"]) == (2, 2, 2, 1)
    n, words = 5, 1
    push0 = 4 + 8 + 8 + 8 + 4                              # F = {1}, m_F = 1, N = {0}
    pull1 = n // 8 + 8 * 2 + 8 * 2 + 8 * 2 + n // 8       # 2R|U| + 8c + 8|N|
    push2 = 4 * 2 + 8 * 2 + 8 * 2                          # F = {2, 3}, m_F = 2, N = {}
    s_tot, k_tot, per = bench.search_bytes(counts, n, 4, reached=4)
    assert per == [push0, pull1, push2] and s_tot == sum(per)
    k_push0 = 12 + 4 + 4 + 8 + 8 + 4 + 12
    to_bitmap = 4 * words + 8 * 1                          # queue {0} -> bitmap
    k_pull1 = 4 * words + 8 * 2 + 4 * 2 + 4 * 2 + 8 * 2 + 4 * words + 4 * 1
    to_queue = 4 * words + 8 * 2 + 12 * 2                  # bitmap {2, 3} -> queue
    k_push2 = 12 * 2 + 4 * 2 + 4 * 2
    assert k_tot == k_push0 + to_bitmap + k_pull1 + to_queue + k_push2 + 4 * 1


def test_pull_scan_counts_stop_at_the_first_frontier_neighbour():
    # edges 0-3, 3-5, 5-1, 5-2, 5-4, 1-6, 2-6; from 0 the distances are
    # 3:1, 5:2, {1, 2, 4}:3, 6:4. Vertex 5's row is [1, 2, 3, 4] and only 3
    # is at distance 1, so a bottom-up scan of 5 reads three entries.
    g = graphgen.from_edges(7, [0, 3, 5, 5, 5, 1, 2], [3, 5, 1, 2, 4, 6, 6])
    dist = [0, 3, 3, 1, 3, 2, 4]
    counts = _counts(g, dist, [bench.DIR_PUSH, bench.DIR_PULL, bench.DIR_PULL, bench.DIR_PULL,
                               bench.DIR_PUSH])
    assert g.col[g.row_ptr[5]:g.row_ptr[6]].tolist() == [1, 2, 3, 4]
    # level 1: U = {1, 2, 4, 5, 6}; 5 is found at its 3rd entry; 1 (row [5, 6]),
    # 2 (row [5, 6]), 4 (row [5]) and 6 (row [1, 2]) are scanned whole
    assert counts[1]["U"] == 5 and counts[1]["N"] == 1
    assert counts[1]["c"] == 3 + 2 + 2 + 1 + 2
    # level 2: U = {1, 2, 4, 6}; 1, 2, 4 find 5 at their first entry; 6 whole row
    assert counts[2]["c"] == 1 + 1 + 1 + 2


def test_lane_slots_against_the_day38_table(golden):
    """Lane slots as the Day 38 table counts them. Its levels of at most 32
    vertices run in one warp, so the thread mapping issues 32 x the largest
    degree there; the degree lists below are consistent with the table and
    text (level 4: ten vertices, 2,452 edges, degrees 1,255 and 1,012 and
    eight of at most 43; level 6: 1,579 vertices, 3,851 edges, largest 33)
    and reproduce its 40,160 thread and 2,656 warp slots for level 4 and
    its 50,560 warp slots for level 6."""
    t = golden("day38_level_table.json")
    for f, e, md, w, slots in zip(t["frontier"], t["edges"], t["max_degree"], t["warps"],
                                  t["lane_slots"]):
        if f <= 32:
            degrees = [md] + [1] * (f - 1)
            r = bench.lane_slots(degrees)
            assert r["warps"] == w == 1 and r["thread"] == slots == 32 * md
    lvl4 = [1255, 1012, 43, 43, 43, 12, 11, 11, 11, 11]
    assert len(lvl4) == 10 and sum(lvl4) == 2452
    r = bench.lane_slots(lvl4)
    assert (r["thread"], r["warp"], r["max_degree"]) == (40160, 2656, 1255)
    lvl6 = [33] + [3] * 662 + [2] * 916
    assert len(lvl6) == 1579 and sum(lvl6) == 3851
    assert bench.lane_slots(lvl6)["warp"] == 50560
    # hand counts: 33 entries of degree 1 and one of 40 take two thread warps
    r = bench.lane_slots([1] * 33 + [40])
    assert r["warps"] == 2 and r["thread"] == 32 * 1 + 32 * 40 and r["warp"] == 32 * 33 + 64
    assert bench.lane_slots([])["thread"] == 0
