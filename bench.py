#!/usr/bin/env python
"""Benchmark: BFS GTEPS on one GB300, fraction of the HBM roofline, and
per-level overhead.

A step is one pass of the whole search path over the workload's batch of
sources: one bfs_csr_run_batch call, which runs every source's search (init
kernel + persistent level loop) with `--lanes` searches in flight at once,
each on its share of the SMs. The default workload is the R-MAT scale-25
graph (2^25 vertices, edge factor 16, int64 row_ptr, int32 col, 16 seeded
sources), with the CSR resident in HBM before timing starts.

GTEPS counts, per search, the CSR entries of the reached vertices (the sum of
their out-degrees, "edges to walk" in the Day 38 level table); the same
count halved (undirected edges) is reported beside it.

Roofline: the algorithmic bytes of the level loops -- what each level's
chosen step must touch, replayed exactly from each search's own distances
and level directions (`survey_bytes`: queue, row offsets, col and one probe
word per scanned entry, dist + parent of the discovered vertices, the next
queue or bitmap) -- over the time during which at least one level loop ran
(device timer stamps the library records per search), against the measured
HBM copy bandwidth. The kernel's own bookkeeping beyond that (queue row
starts and degree prefixes, representation switches, the end-of-search dist
pass) is counted apart (`kernel_extra_bytes`).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica on its GPU
(the search does not shard) with its own slice of the sources.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BFS GTEPS on 1 GB300 and % of HBM roofline; per-level overhead (µs)"
DIR_PUSH, DIR_PULL = 1, 2

WORKLOADS = {
    5: "rmat_25: R-MAT scale 25, edge factor 16 (a,b,c,d = 0.57,0.19,0.19,0.05), permuted, "
       "symmetrised, deduplicated; int64 row_ptr, int32 col; 16 sources (seed 4)",
    3: "rmat_22: R-MAT scale 22, edge factor 16, int32 CSR; 64 sources (seed 2)",
    2: "er_2^20: uniform random graph, 2^20 vertices, average degree 16; 64 sources (seed 1)",
    4: "grid_2048: 2048x2048 lattice, edges deleted with p=0.1; corner source (seed 3)",
    1: "powerlaw_3485: Chung-Lu power-law graph, 3,485 vertices; 64 sources (seed 0)",
}

# The pages' own figures, quoted as context only (other hardware, other graph).
PAGES_CONTEXT = {
    "hardware": "Tesla T4 (sm_75, 40 SMs); 3,485-word graph, 31,812 CSR entries, 10 levels",
    "whole_bfs_ms": {"thread_per_vertex": 1.8091, "warp_per_vertex": 0.3340},
    "isolated_level_walk_x64_ms": {"level_4": [1.3724, 0.0881], "level_5": [1.0068, 0.0796],
                                   "level_6": [0.1172, 0.0485]},
    "lane_slots_thread_per_vertex": 251872, "useful_edges": 31758,
    "launches": "10 launches for 10 levels; 5-10 us per launch stated (PMPP ch. 15 notes)",
    "source": "100 Days of GPU, Day 38 'Results'; PMPP ch. 15 notes section 15.7",
}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def host_cores():
    try:
        aff = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        aff = None
    return {"online": os.cpu_count(), "affinity": aff}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, interval_ms: int = 50):
        self.cmd = ["nvidia-smi", "-i", str(device_index), "--query-gpu=" + self.QUERY,
                    "--format=csv,noheader,nounits", "-lms", str(interval_ms)]
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ byte models

def level_counts(torch, row_ptr64, col, deg, src_of_edge, dist, stats):
    """Exact per-level counts of one search, replayed on the device from its
    distances and the direction each level took.

    Per level k: F = |{v: dist v = k}|, Q = those with out-edges, mF = their
    out-degree sum, N = |{v: dist v = k + 1}| (the vertices level k
    discovers), Ne = those with out-edges, U = vertices of nonzero degree not
    reached by level k (unvisited at its start). Pull levels also get c = the
    CSR entries a bottom-up scan reads: for each vertex it finds, its row up
    to and including the first neighbour at distance k; for every other
    vertex of U, its whole row; and tw = 32-vertex words holding a find.
    """
    has_edges = deg > 0
    out = []
    ds = dd = None
    for k, st in enumerate(stats):
        in_k = dist == k
        nxt = dist == (k + 1)
        c = {"level": k, "direction": st["direction"], "advance": st["advance"],
             "F": int(in_k.sum().item()), "Q": int((in_k & has_edges).sum().item()),
             "mF": int(deg[in_k].sum().item()), "N": int(nxt.sum().item()),
             "Ne": int((nxt & has_edges).sum().item()),
             "U": int((((dist < 0) | (dist > k)) & has_edges).sum().item()), "c": 0, "tw": 0}
        if st["direction"] == DIR_PULL:
            if ds is None:
                ds = dist[src_of_edge.long()]
                dd = dist[col.long()]
            hit = (ds == k + 1) & (dd == k)
            pos = torch.nonzero(hit).squeeze(1)
            found = 0
            if pos.numel():
                owner = src_of_edge[pos].long()
                big = torch.full((dist.numel(),), np.iinfo(np.int64).max, dtype=torch.int64,
                                 device=dist.device)
                big.scatter_reduce_(0, owner, pos, reduce="amin")
                sel = nxt & has_edges
                found = int((big[sel] - row_ptr64[:-1][sel] + 1).sum().item())
                del big, owner
            rest = ((dist < 0) | (dist > k + 1)) & has_edges
            c["c"] = found + int(deg[rest].sum().item())
            if c["N"]:
                c["tw"] = int(torch.unique(torch.nonzero(nxt).squeeze(1) // 32).numel())
            del hit, pos
        out.append(c)
    return out


def survey_bytes(c, n: int, R: int) -> int:
    """Algorithmic bytes of one level: what the chosen step itself must touch.
    Top-down: the queue 4|F|, row offsets 2R|F|, col 4 m_F, one probe word per
    edge 4 m_F, dist + parent of the discovered vertices 8|N|, the next queue
    4|N| and bitmap |N|/8. Bottom-up: the visited bitmap n/8, row offsets
    2R|U|, col 4c and one frontier-bitmap word per scanned entry 4c, dist +
    parent 8|N|, the next-frontier bitmap n/8. Random single-word probes are
    counted at their word size."""
    if c["direction"] == DIR_PULL:
        return n // 8 + 2 * R * c["U"] + 8 * c["c"] + 8 * c["N"] + n // 8
    F, N = c["F"], c["N"]
    return 4 * F + 2 * R * F + 8 * c["mF"] + 8 * N + 4 * N + N // 8


def kernel_bytes(c, prev_dir: int, n: int, R: int) -> int:
    """The same level as this library's kernel touches it, single words at
    their size: a queue entry is (vertex, row start, degree prefix), so queue
    reads and writes are (4 + 2R) per vertex with out-edges and every winner's
    row offsets are read once (2R); a switch between the representations
    costs a bitmap pass (and the queue build reads row offsets); a pull level
    also rewrites the visited words that gained a vertex."""
    words = (n + 31) // 32
    F, Q, N, Ne = c["F"], c["Q"], c["N"], c["Ne"]
    b = 0
    if c["direction"] == DIR_PULL:
        if prev_dir == DIR_PUSH:
            b += 4 * words + 8 * Q
        b += 4 * words + 2 * R * c["U"] + 8 * c["c"] + 8 * N + 4 * words + 4 * c["tw"]
    else:
        if prev_dir == DIR_PULL:
            b += 4 * words + 2 * R * F + (4 + 2 * R) * Q
        b += (4 + 2 * R) * Q + 8 * c["mF"] + 2 * R * N + 8 * N + 4 * N + (4 + 2 * R) * Ne
    return b


def search_bytes(counts, n: int, R: int, reached: int):
    """(survey bytes, kernel bytes, survey bytes per level) of one search's
    level loop. The kernel also writes every unreached vertex's -1 at the
    end (4 (n - reached); the reached vertices' dist is counted at their
    discovery)."""
    prev = DIR_PUSH
    s_tot, k_tot, per = 0, 0, []
    for c in counts:
        sb = survey_bytes(c, n, R)
        per.append(sb)
        s_tot += sb
        k_tot += kernel_bytes(c, prev, n, R)
        prev = c["direction"]
    return s_tot, k_tot + 4 * (n - reached), per


def init_bytes_survey(n: int) -> int:
    """Init per the scope table: dist and parent filled (8n), two bitmaps
    cleared (n/4)."""
    return 8 * n + n // 4


def init_bytes_kernel(n: int, with_parent: bool = True) -> int:
    """This library's init kernel with bitmap discovery: one hop-code byte per
    vertex, parent (-1) unless the end-of-search pass writes parents, the
    visited bitmap written and the dead bitmap read."""
    words = (n + 31) // 32
    return (n + 15) // 16 * 16 + (4 * n if with_parent else 0) + 8 * words


def busy_time(intervals) -> float:
    """Length of the union of [start, end] intervals: the time during which
    at least one of them was running."""
    busy, cur_a, cur_b = 0.0, None, None
    for a, b in sorted(intervals):
        if cur_b is None or a > cur_b:
            if cur_b is not None:
                busy += cur_b - cur_a
            cur_a, cur_b = a, b
        else:
            cur_b = max(cur_b, b)
    if cur_b is not None:
        busy += cur_b - cur_a
    return float(busy)


def graph_tensors(torch, g, device):
    row_ptr = torch.from_numpy(g.row_ptr).to(device)
    col = torch.from_numpy(g.col).to(device)
    row64 = row_ptr.to(torch.int64)
    deg = torch.diff(row64)
    return row_ptr, col, row64, deg


# ------------------------------------------------------------------ distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(torch, ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(torch, ws, value: float, device) -> float:
    if ws == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(torch, ws, value: float, device) -> float:
    if ws == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def rank_sources(sources, rank: int, ws: int):
    """Replica split: rank r takes sources r, r + ws, ... (all of them if too few)."""
    mine = [int(s) for s in sources[rank::ws]]
    return mine if mine else [int(s) for s in sources]


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import torch

    import frontier_bfs_csr_gb300 as fbc
    import graphgen

    ws, rank, local = dist_env()
    if ws > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peak, peak_kind = measured_peaks()

    if rank == 0:
        g = graphgen.config(args.config)
    barrier(torch, ws)
    if rank != 0:
        g = graphgen.config(args.config)
    all_sources = g.sources[:args.sources] if args.sources > 0 else g.sources
    sources = rank_sources(all_sources, rank, ws)
    row_ptr, col, row64, deg = graph_tensors(torch, g, device)
    R = 8 if g.row_ptr_64 else 4
    bfs = fbc.BfsCsr(row_ptr, col, symmetric=True,
                     options=fbc.default_options(lanes=args.lanes))
    n = g.n
    k = len(sources)
    stream = torch.cuda.current_stream(device)

    # Untimed pass, one bfs_csr_run per source on the whole GPU: warms the
    # kernels and records, per source, the walked-edge count, the level
    # records, the replayed byte counts and the outputs (for the consistency
    # check of the timed batch).
    src_of_edge = torch.repeat_interleave(torch.arange(n, device=device, dtype=torch.int32), deg)
    ref_dist = torch.empty((k, n), dtype=torch.int32, device=device)
    ref_levels = []
    per_source = {}
    parent = torch.empty(n, dtype=torch.int32, device=device)
    for i, s in enumerate(sources):
        dist = ref_dist[i]
        bfs.run(s, dist, parent, stream=stream)
        levels = bfs.sync(stream)
        ref_levels.append(levels)
        reached_mask = dist >= 0
        reached = int(reached_mask.sum().item())
        edges = int(deg[reached_mask].sum().item())
        stats = bfs.level_stats()
        counts = level_counts(torch, row64, col, deg, src_of_edge, dist, stats)
        sb, kb, per = search_bytes(counts, n, R, reached)
        torch.cuda.empty_cache()
        per_source[s] = {"levels": levels, "edges": edges, "survey_bytes": sb, "kernel_bytes": kb,
                         "directions": "".join("P" if x["direction"] == DIR_PUSH else "U"
                                               for x in stats)}
        if i == 0:
            table = per_level_table(counts, per, stats, peak)
    del src_of_edge
    torch.cuda.empty_cache()

    # Timed step: one bfs_csr_run_batch over the batch of sources (the searches
    # run on `lanes` lanes at once); dist/parent rows per source.
    dist_b = torch.empty((k, n), dtype=torch.int32, device=device)
    parent_b = torch.empty((k, n), dtype=torch.int32, device=device)
    levels_b = torch.empty(k, dtype=torch.int32, device=device)
    for _ in range(max(args.warmup - 1, 0)):
        bfs.run_batch(sources, dist_b, parent_b, levels_b, stream=stream)

    # Timed region: K steps; every search records device timer stamps (init
    # start, level-loop start, level-loop end).
    stamps = torch.zeros((args.steps, 3 * k), dtype=torch.int64, device=device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    barrier(torch, ws)
    torch.cuda.synchronize(device)
    t0.record(stream)
    for i in range(args.steps):
        bfs.run_batch(sources, dist_b, parent_b, levels_b, stamps[i], stream=stream)
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier(torch, ws)
    clocks = sampler.stop()
    local_ms = t0.elapsed_time(t1)
    total_ms = max_over_ranks(torch, ws, local_ms, device)
    # Every row of the last timed step against the untimed single runs (the
    # CUDA path against itself: the oracle certifies the rows below).
    repeat_ok = bool(torch.equal(dist_b, ref_dist)) and \
        levels_b.cpu().tolist() == ref_levels
    del ref_dist
    torch.cuda.empty_cache()

    st = stamps.cpu().numpy().reshape(-1, 3).astype(np.float64) * 1e-6   # ms
    runs = st.shape[0]
    init_ms = (st[:, 1] - st[:, 0]).tolist()
    level_ms = (st[:, 2] - st[:, 1]).tolist()
    busy = busy_time(zip(st[:, 1], st[:, 2]))
    edges_local = sum(per_source[s]["edges"] for s in sources) * args.steps
    edges_all = sum_over_ranks(torch, ws, float(edges_local), device)
    value = edges_all / (total_ms * 1e-3) / 1e9

    lvl_bytes = sum(per_source[s]["survey_bytes"] for s in sources) * args.steps
    ker_bytes = sum(per_source[s]["kernel_bytes"] for s in sources) * args.steps
    achieved = lvl_bytes / (busy * 1e-3) / 1e9
    # parents are written by the end pass (and not filled at init) when the
    # parent array exceeds half of the L2
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    init_parent = 4 * n <= l2 // 2
    init_b = init_bytes_kernel(n, with_parent=init_parent) * runs
    init_gbs = init_b / (sum(init_ms) * 1e-3) / 1e9
    run_bytes = (lvl_bytes + init_bytes_survey(n) * runs) / args.steps

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "GTEPS", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.config], "n": n, "nnz": g.nnz,
                   "row_ptr": "int64" if g.row_ptr_64 else "int32",
                   "sources_per_step": len(sources), "parallelism": "replicas" if ws > 1 else "1gpu",
                   "lanes": args.lanes,
                   "concurrency": "bfs_csr_run_batch: %d searches in flight, each on 1/%d of "
                                  "the level kernel's CTAs" % (args.lanes, args.lanes),
                   "teps_numerator": "sum of out-degrees of reached vertices per search",
                   "l2": "inputs larger than L2 (CSR %.2f GB vs 129 MB L2)" % (
                       (g.row_ptr.nbytes + g.col.nbytes) / 1e9),
                   "csr_fingerprint": g.fingerprint()},
        "gteps_undirected": round(value / 2, 3),
        "per_search": {"levels_median": statistics.median(p["levels"] for p in per_source.values()),
                       "ms_median": round(statistics.median(
                           a + b for a, b in zip(init_ms, level_ms)), 4),
                       "directions": sorted(set(p["directions"] for p in per_source.values()))},
        "roofline": {"bound": "hbm", "kernel": "level_kernel",
                     "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": None,
                     "traffic_source": None,
                     "algorithmic_bytes_per_launch": int(lvl_bytes / runs),
                     "byte_model": "scope-table level bytes (bench.py survey_bytes), replayed "
                                   "from each search's distances and directions",
                     "kernel_extra_bytes_per_launch": int((ker_bytes - lvl_bytes) / runs),
                     "launch_ms_mean": round(sum(level_ms) / runs, 4),
                     "level_kernel_busy_ms": round(busy, 4),
                     "timing": "device timer stamps per search; achieved = algorithmic bytes "
                               "of every level-loop launch / time any level loop ran"},
        "run_roofline": {"bytes_per_step": int(run_bytes),
                         "achieved_gbs": round(run_bytes / (total_ms / args.steps * 1e-3) / 1e9, 1),
                         "frac": round(run_bytes / (total_ms / args.steps * 1e-3) / 1e9 / peak, 4),
                         "what": "init (8n + n/4) plus level bytes per step over the step time"},
        "per_level": table,
        "init_kernel": {"achieved_gbs": round(init_gbs, 1), "frac": round(init_gbs / peak, 4),
                        "bytes_per_launch": init_bytes_kernel(n, with_parent=init_parent),
                        "launch_ms_mean": round(sum(init_ms) / runs, 4)},
        "clocks": clocks,
        "gpu_launches": 2 * runs,
        "repeat_consistent": repeat_ok,
        "status_after_timing": "not certified (--no-cpu)",
    }
    traffic = read_traffic_summary(args.config)
    if traffic is not None:
        result["roofline"]["traffic"] = traffic
        result["roofline"]["traffic_source"] = ("committed ncu summary "
                                                "profiles/level_kernel_rmat25_traffic.txt "
                                                "(dram__bytes_read.sum + dram__bytes_write.sum "
                                                "per launch, same kernel source)")
    timed_rows = None
    if rank == 0 and not args.no_cpu:
        timed_rows = (list(sources), dist_b.cpu().numpy(), parent_b.cpu().numpy(),
                      levels_b.cpu().numpy())
    bfs.close()
    del dist_b, parent_b, stamps, bfs
    torch.cuda.empty_cache()

    config_rows = {}
    if rank == 0 and not args.no_configs:
        result["per_config"] = per_config(torch, fbc, graphgen, device, peak, config_rows,
                                          keep_rows=not args.no_cpu)
    if rank == 0 and not args.no_ablation:
        cases = [(2, None), (3, None)] + ([(5, g)] if args.config == 5 else [])
        result["ablation"] = ablation(torch, fbc, graphgen, device, cases)
    if rank == 0 and not args.no_overhead:
        result["per_level_overhead_us"] = per_level_overhead(torch, fbc, graphgen, device)
    if rank == 0 and not args.no_walk:
        result["walk"] = walk_section(torch, fbc, graphgen, device)
    if not args.no_e2e:
        result["e2e"] = run_e2e(torch, fbc, g, sources, args, device, ws)
    if rank == 0 and not args.no_cpu:
        base, cert = cpu_leg(g, timed_rows, config_rows, graphgen)
        result["cpu_baseline"] = base
        result["status_after_timing"] = cert["timed"]
        if "per_config" in result:
            for cfg, flag in cert["configs"].items():
                result["per_config"][cfg]["parity"] = flag
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def per_level_table(counts, per_bytes, stats, peak):
    """One search's levels: direction, advance, sizes, algorithmic bytes, the
    time from this level's start to the next one's (device stamps; the last
    level up to the end of its work), and the fraction of peak."""
    rows = []
    for i, (c, b) in enumerate(zip(counts, per_bytes)):
        t0 = stats[i]["t_start_ns"]
        t1 = stats[i + 1]["t_start_ns"] if i + 1 < len(stats) else stats[i]["t_work_ns"]
        us = max(t1 - t0, 1) / 1e3
        busy = max(stats[i]["t_work_ns"] - t0, 0) / 1e3
        gbs = b / (us * 1e-6) / 1e9
        rows.append({"level": c["level"], "dir": "push" if c["direction"] == DIR_PUSH else "pull",
                     "advance": {0: "-", 1: "binned", 2: "merge_path", 3: "single_cta"}.get(
                         c["advance"], str(c["advance"])),
                     "F": c["F"], "m_F": c["mF"], "U": c["U"], "N": c["N"], "c": c["c"],
                     "bytes": int(b), "us": round(us, 2), "busy_us": round(busy, 2),
                     "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)})
    return rows


def read_traffic_summary(cfg: int):
    """DRAM bytes per level-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source; otherwise None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "level_kernel_rmat25_traffic.txt")
    src = os.path.join(ROOT, "frontier_bfs_csr_gb300", "csrc", "bfs_device.cuh")
    if cfg != 5 or not os.path.exists(path):
        return None
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    fields = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256_16") != sha:
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def time_search(torch, bfs, s, dist, parent, stream, warm=3, reps=10):
    """Mean device time of bfs_csr_run (init + level loop) over `reps` runs
    after `warm` untimed ones (the Day 38 protocol), CUDA events."""
    for _ in range(warm):
        bfs.run(s, dist, parent, stream=stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        bfs.run(s, dist, parent, stream=stream)
    e1.record(stream)
    levels = bfs.sync(stream)
    return e0.elapsed_time(e1) / reps, levels


def per_config(torch, fbc, graphgen, device, peak, rows_out, keep_rows=True):
    """Configs 1-4: per source, the mean of 10 timed bfs_csr_run (after 3
    warm-ups); GTEPS as the median over sources and the aggregate (sum of
    edges over sum of times); the fraction of the HBM roofline of the whole
    run (init + levels, scope-table bytes) over its time. Each source's
    outputs are kept for the oracle's certification in the CPU leg."""
    out = {}
    stream = torch.cuda.current_stream(device)
    for cfg in (1, 2, 3, 4):
        g = graphgen.config(cfg)
        row_ptr, col, row64, deg = graph_tensors(torch, g, device)
        R = 8 if g.row_ptr_64 else 4
        srcs = [int(s) for s in g.sources]
        bfs = fbc.BfsCsr(row_ptr, col, symmetric=True)
        dist = torch.empty(g.n, dtype=torch.int32, device=device)
        parent = torch.empty_like(dist)
        soe = torch.repeat_interleave(torch.arange(g.n, device=device, dtype=torch.int32), deg)
        gteps, times, edges_l, bytes_l, levels_l = [], [], [], [], []
        dist_rows, par_rows, lev_rows = [], [], []
        overhead = None
        for s in srcs:
            ms, levels = time_search(torch, bfs, s, dist, parent, stream)
            reached_mask = dist >= 0
            reached = int(reached_mask.sum().item())
            edges = int(deg[reached_mask].sum().item())
            stats = bfs.level_stats()
            counts = level_counts(torch, row64, col, deg, soe, dist, stats)
            sb, _, _ = search_bytes(counts, g.n, R, reached)
            b_run = sb + init_bytes_survey(g.n)
            gteps.append(edges / (ms * 1e-3) / 1e9)
            times.append(ms)
            edges_l.append(edges)
            bytes_l.append(b_run)
            levels_l.append(levels)
            if cfg == 4:
                busy_ns = sum(max(x["t_work_ns"] - x["t_start_ns"], 0) for x in stats)
                overhead = {"t_run_us": round(ms * 1e3, 1), "levels": levels,
                            "busy_us": round(busy_ns / 1e3, 1),
                            "overhead_us_per_level": round((ms * 1e3 - busy_ns / 1e3) / levels, 3),
                            "definition": "(t_run - sum over levels of (last CTA's work end - "
                                          "level start)) / levels, persistent loop"}
            if keep_rows:
                dist_rows.append(dist.cpu().numpy())
                par_rows.append(parent.cpu().numpy())
                lev_rows.append(levels)
        bfs.close()
        del soe
        torch.cuda.empty_cache()
        agg = sum(edges_l) / (sum(times) * 1e-3) / 1e9
        frac = sum(bytes_l) / (sum(times) * 1e-3) / 1e9 / peak
        entry = {"workload": WORKLOADS[cfg], "n": g.n, "nnz": g.nnz, "sources": len(srcs),
                 "gteps_median": round(statistics.median(gteps), 4),
                 "gteps_aggregate": round(agg, 4),
                 "ms_per_search_median": round(statistics.median(times), 4),
                 "levels_median": statistics.median(levels_l),
                 "roofline_frac": round(frac, 4),
                 "timing": "bfs_csr_run (init + levels), CUDA events, 3 warm-ups + 10 timed "
                           "per source, one search at a time on the whole GPU",
                 "parity": "not certified (--no-cpu)"}
        if overhead is not None:
            entry["per_level_overhead"] = overhead
        out[str(cfg)] = entry
        if keep_rows:
            rows_out[str(cfg)] = (g, srcs, dist_rows, par_rows, lev_rows)
    return out


# name, options, (sources, timed repeats) when fewer than the default: the
# thread-mapped padded advance walks a hub's whole row on one thread.
ABLATION = [
    ("auto_dir+auto_adv(default)", dict(), None),
    ("push_only+auto_adv", dict(direction=1), None),
    ("pull_only", dict(direction=2), None),
    ("push_only+binned", dict(direction=1, advance=1), None),
    ("push_only+merge_path", dict(direction=1, advance=2), None),
    ("auto_dir+binned", dict(advance=1), None),
    ("auto_dir+merge_path", dict(advance=2), None),
    ("discovery_cas", dict(discovery=1), None),
    ("discovery_atomic_min", dict(discovery=2), None),
    ("atomic_min+padded+filter", dict(discovery=2, frontier_output=1), None),
    ("atomic_min+padded+filter+push_only", dict(discovery=2, frontier_output=1, direction=1), None),
    ("atomic_min+padded_no_filter(thread_mapped,push_only)", dict(discovery=2, frontier_output=2),
     (2, 1)),
    ("parent_end_pass", dict(parent_pass=1), None),
    ("parent_at_discovery", dict(parent_pass=2), None),
]


def ablation(torch, fbc, graphgen, device, cases, nsrc=16, reps=3):
    """Direction (push only, pull only, the automatic rule), push advance
    (degree-binned, merge path, and the automatic choice: the pages' static
    hybrid -- merge path from a 4,096-vertex frontier or an 8,192-degree hub
    -- plus the merge path for frontiers whose rows average 8 entries or
    more), discovery (bitmap
    atomicOr, atomicCAS, atomicMin on dist), the Gunrock-style padded frontier
    with and without its filter, and where parents are written, on the first
    16 sources of each config: one search at a time (lanes = 1), GTEPS of a
    bfs_csr_run_batch over the sources, median of `reps` timed batches after
    one warm-up. Each variant's distances are compared with the automatic
    variant's rows (the option matrix of the tests checks every variant
    against the oracle)."""
    out = {}
    stream = torch.cuda.current_stream(device)
    for cfg, g in cases:
        if g is None:
            g = graphgen.config(cfg)
        row_ptr, col, row64, deg = graph_tensors(torch, g, device)
        srcs = [int(s) for s in g.sources[:nsrc]]
        k = len(srcs)
        dist = torch.empty((k, g.n), dtype=torch.int32, device=device)
        ref = None
        res = {}
        edge_rows = None
        for name, over, limit in ABLATION:
            kv, rv = (min(k, limit[0]), limit[1]) if limit else (k, reps)
            bfs = fbc.BfsCsr(row_ptr, col, symmetric=True, options=fbc.default_options(**over))
            bfs.run_batch(srcs[:kv], dist[:kv], stream=stream)
            if edge_rows is None:
                edge_rows = [int(deg[dist[i] >= 0].sum().item()) for i in range(k)]
            ts = []
            for _ in range(rv):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                bfs.run_batch(srcs[:kv], dist[:kv], stream=stream)
                e1.record(stream)
                torch.cuda.synchronize(device)
                ts.append(e0.elapsed_time(e1))
            bfs.close()
            ms = statistics.median(ts)
            if ref is None:
                ref = dist.clone()
                same = True
            else:
                same = bool(torch.equal(dist[:kv], ref[:kv]))
            res[name] = {"gteps": round(sum(edge_rows[:kv]) / (ms * 1e-3) / 1e9, 2),
                         "ms_per_search": round(ms / kv, 4), "sources": kv, "timed": rv,
                         "same_dist_as_auto": same}
        auto = res["auto_dir+auto_adv(default)"]["gteps"]
        for name in res:
            res[name]["vs_auto"] = round(res[name]["gteps"] / auto, 3) if auto else None
        out[str(cfg)] = {"sources": k, "variants": res}
        del edge_rows
        del dist, ref, row_ptr, col, row64, deg
        torch.cuda.empty_cache()
    return out


def lane_slots(degrees):
    """Lane slots a level's neighbour walk issues ("100 Days of GPU, Day 38",
    the level table): with one thread per vertex each warp of 32 consecutive
    frontier entries runs as long as its longest row, so it issues 32 times
    its largest degree; with one warp per vertex each vertex takes
    ceil(degree / 32) passes of 32 lanes."""
    d = np.asarray(degrees, dtype=np.int64)
    warps = (d.size + 31) // 32
    pad = np.zeros(warps * 32, dtype=np.int64)
    pad[:d.size] = d
    thread = int(32 * pad.reshape(warps, 32).max(axis=1).sum()) if warps else 0
    warp = int(32 * ((d + 31) // 32).sum())
    return {"warps": int(warps), "thread": thread, "warp": warp, "edges": int(d.sum()),
            "max_degree": int(d.max()) if d.size else 0,
            "useful_thread": round(float(d.sum()) / thread, 4) if thread else None}


WALK_MAPPINGS = ("thread", "warp", "binned", "edge")


def walk_section(torch, fbc, graphgen, device, repeats=64, min_edges=1000):
    """The isolated neighbour walk of single levels (Day 38, "Measuring the
    mapping without measuring the launch") on the 3,485-vertex power-law
    graph from its most eccentric source (most levels, smallest id on ties;
    found by a GPU search from every vertex of nonzero degree): for every
    level with at least 1,000 edges, the frontier (vertex order) walked 64
    times by each mapping, 3 warm-ups + 10 timed launches (CUDA events, mean),
    the graph-derived lane slots, and the pages' T4 figures as context. The
    four mappings' checksums are compared with each other here; the tests
    compare them with the oracle's."""
    g = graphgen.config(1)
    row_ptr, col, row64, deg = graph_tensors(torch, g, device)
    bfs = fbc.BfsCsr(row_ptr, col, symmetric=True)
    dist = torch.empty(g.n, dtype=torch.int32, device=device)
    nl = torch.empty(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    best, best_levels = None, -1
    cand = torch.nonzero(deg > 0).squeeze(1).tolist()
    lev = torch.empty(len(cand), dtype=torch.int32, device=device)
    for i, s in enumerate(cand):
        bfs.run(s, dist, None, lev[i:i + 1], stream=stream)
    levels_all = lev.cpu().tolist()
    for s, L in zip(cand, levels_all):
        if L > best_levels:
            best, best_levels = s, L
    bfs.run(best, dist, None, nl, stream=stream)
    bfs.sync(stream)
    d_h = dist.cpu().numpy()
    deg_h = np.diff(g.row_ptr.astype(np.int64))
    rows, table = [], []
    for k in range(best_levels):
        frontier = np.nonzero(d_h == k)[0].astype(np.int32)
        slots = lane_slots(deg_h[frontier])
        table.append(dict(level=k, frontier=int(frontier.size), **slots))
        if slots["edges"] < min_edges:
            continue
        fr = torch.from_numpy(frontier).to(device)
        outs, ms = [], {}
        for m, name in enumerate(WALK_MAPPINGS):
            out = torch.empty(frontier.size, dtype=torch.int32, device=device)
            for _ in range(3):
                bfs.walk(fr, repeats, m, out, stream=stream)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(10):
                bfs.walk(fr, repeats, m, out, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize(device)
            ms[name] = round(e0.elapsed_time(e1) / 10, 5)
            outs.append(out.clone())
        same = all(bool(torch.equal(outs[0], o)) for o in outs[1:])
        rows.append({"level": k, "frontier": int(frontier.size), "edges": slots["edges"],
                     "max_degree": slots["max_degree"], "ms": ms,
                     "thread_over_warp": round(ms["thread"] / ms["warp"], 2),
                     "lane_slots": {"thread": slots["thread"], "warp": slots["warp"]},
                     "checksums_agree": same})
    bfs.close()
    return {"graph": WORKLOADS[1], "source": best, "levels": best_levels, "repeats": repeats,
            "timing": "bfs_csr_walk, 3 warm-ups + 10 timed launches, CUDA events, mean",
            "levels_timed": rows, "lane_slot_table": table,
            "lane_slots_whole_search": {"thread": sum(t["thread"] for t in table),
                                        "edges": sum(t["edges"] for t in table)},
            "pages_context": PAGES_CONTEXT}


def per_level_overhead(torch, fbc, graphgen, device):
    """Per-level cost on graphs made of narrow levels: the 2048x2048 grid from
    its corner and a 10,000-vertex path (one vertex per level), in the
    persistent loop, the CUDA-graph loop (one graph launch per search, a
    device-driven while node launching one level per iteration) and the host
    loop (one launch + one device->host read per level, the structure the
    Day 38 page measures). The plain figure is t_run per level; `*_sync` is
    (t_run - sum of level busy times) / levels, busy = last CTA's work end -
    level start from the level records."""
    out = {}
    cases = [("grid_2048", graphgen.config(4)), ("path_10000", graphgen.path_graph(10000))]
    for name, g in cases:
        rp = torch.from_numpy(g.row_ptr).to(device)
        cl = torch.from_numpy(g.col).to(device)
        s = int(g.sources[0]) if g.sources is not None else 0
        dist = torch.empty(g.n, dtype=torch.int32, device=device)
        row = {}
        for mode, loop in (("persistent", fbc.BFS_CSR_LOOP_PERSISTENT),
                           ("graph_loop", fbc.BFS_CSR_LOOP_GRAPH),
                           ("host_loop", fbc.BFS_CSR_LOOP_HOST)):
            b = fbc.BfsCsr(rp, cl, True, fbc.default_options(loop_mode=loop))
            b.run(s, dist)
            levels = b.sync()
            reps = 1 if loop == fbc.BFS_CSR_LOOP_HOST else 3
            best, best_busy = None, None
            for _ in range(reps):
                torch.cuda.synchronize(device)
                t = time.perf_counter()
                b.run(s, dist)
                b.sync()
                el = time.perf_counter() - t
                stats = b.level_stats()
                bz = sum(max(x["t_work_ns"] - x["t_start_ns"], 0) for x in stats) * 1e-9
                if best is None or el < best:
                    best, best_busy = el, bz
            b.close()
            row[mode] = round(best * 1e6 / levels, 3)
            row[mode + "_sync"] = round((best - best_busy) * 1e6 / levels, 3)
            row["levels"] = levels
        out[name] = row
    return out


def run_e2e(torch, fbc, g, sources, args, device, ws):
    """Host buffers through bfs_csr_run_host_batch: every step uploads the CSR
    from pinned memory, runs the batch of sources and copies every search's
    dist and parent back (the copy-back of one search overlaps the next)."""
    rp_pin = torch.from_numpy(g.row_ptr).pin_memory()
    col_pin = torch.from_numpy(g.col).pin_memory()
    rp_np, col_np = rp_pin.numpy(), col_pin.numpy()
    k = len(sources)
    dist_t = torch.empty((k, g.n), dtype=torch.int32).pin_memory()
    par_t = torch.empty((k, g.n), dtype=torch.int32).pin_memory()
    lev_t = torch.empty(k, dtype=torch.int32).pin_memory()
    dist_np, par_np, lev_np = dist_t.numpy(), par_t.numpy(), lev_t.numpy()
    h = fbc.BfsCsrHost(rp_np, col_np, True)
    steps = max(1, args.steps)
    deg = np.diff(g.row_ptr.astype(np.int64))
    h.run_batch(sources, dist_np, par_np, lev_np, row_ptr=rp_np, col=col_np)  # warm-up step
    edges_per_step = sum(int(deg[dist_np[i] >= 0].sum()) for i in range(k))
    torch.cuda.synchronize(device)
    t = time.perf_counter()
    for _ in range(steps):
        h.run_batch(sources, dist_np, par_np, lev_np, row_ptr=rp_np, col=col_np)
    elapsed = time.perf_counter() - t
    h.close()
    del dist_t, par_t
    elapsed = max_over_ranks(torch, ws, elapsed, device)
    edges = sum_over_ranks(torch, ws, float(edges_per_step * steps), device)
    h2d = int(g.row_ptr.nbytes + g.col.nbytes + 8 * k)
    d2h = int(k * (8 * g.n + 4))
    link = link_bandwidth(torch, device)
    return {"value": round(edges / elapsed / 1e9, 3), "unit": "GTEPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round(elapsed / steps * 1e3, 3),
            "api": "bfs_csr_create_host / bfs_csr_run_host_batch",
            "host_link": dict(link, copy_floor_ms=round(
                (h2d / link["h2d_gbs"] + d2h / link["d2h_gbs"]) / 1e6, 2))}


def link_bandwidth(torch, device, nbytes: int = 1 << 30, reps: int = 3):
    """Plain pinned-memory copies of one 1 GiB buffer each way (cudaMemcpyAsync
    through torch, CUDA events, best of reps), outside any timed region: the
    host link this box delivered, which bounds the end-to-end step."""
    hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    out = {}
    for name in ("h2d", "d2h"):
        best = float("inf")
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            if name == "h2d":
                dbuf.copy_(hbuf, non_blocking=True)
            else:
                hbuf.copy_(dbuf, non_blocking=True)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        out[name + "_gbs"] = round(nbytes / best / 1e6, 1)
    del hbuf, dbuf
    return out


# ------------------------------------------------------------------ CPU leg

def cpu_leg(g, timed_rows, config_rows, graphgen, budget_s: float = 20.0):
    """The oracle on the host, after every GPU measurement.

    (1) Baseline: the sequential FIFO BFS (C, one host thread) on a bounded
    sample of the timed workload, sources in order until ~budget_s seconds.
    (2) Certification of the GPU outputs: every row of the last timed step
    (and every per-config row) -- dist equal element by element to the
    oracle's where the baseline computed it, else accepted by the oracle's
    exact distance certificate; parent accepted by the oracle's tree check;
    the level count equal to max(dist) + 1. The checks run on several host
    threads at once (the oracle's ctypes calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    deg = np.diff(g.row_ptr.astype(np.int64))
    known = {}
    done, edges, elapsed = [], 0, 0.0
    srcs = timed_rows[0] if timed_rows is not None else [int(s) for s in g.sources]
    for s in srcs:
        t = time.perf_counter()
        d, _, _ = oracle.bfs(g.row_ptr, g.col, s, want_parent=True)
        elapsed += time.perf_counter() - t
        edges += int(deg[d >= 0].sum())
        done.append(s)
        known[s] = d
        if elapsed > budget_s:
            break
    cores = host_cores()
    base = {"value": round(edges / elapsed / 1e9, 4), "unit": "GTEPS", "cores": 1,
            "host_cores": cores["online"], "host_cores_affinity": cores["affinity"],
            "kind": "oracle",
            "sample": "%d of %d sources of the timed workload (a sample), %.1f s on one thread"
                      % (len(done), len(srcs), elapsed)}

    def certify(graph, s, d, p, lev, want=None):
        if want is not None:
            ok_d = bool(np.array_equal(d, want))
        else:
            ok_d = oracle.check_dist(graph.row_ptr, graph.col, s, d)[0] == 0
        ok_p = oracle.check_parent(graph.row_ptr, graph.col, s, d, p)[0] == 0
        return ok_d and ok_p and int(lev) == int(d.max()) + 1, want is not None

    workers = max(1, min(16, os.cpu_count() or 1))
    cert = {"timed": "not certified", "configs": {}}
    with ThreadPoolExecutor(max_workers=workers) as ex:
        if timed_rows is not None:
            srcs_t, dist_t, par_t, lev_t = timed_rows
            res = list(ex.map(lambda i: certify(g, srcs_t[i], dist_t[i], par_t[i], lev_t[i],
                                                known.get(srcs_t[i])), range(len(srcs_t))))
            good = sum(1 for ok, _ in res if ok)
            eq = sum(1 for _, e in res if e)
            cert["timed"] = ("oracle-certified: %d/%d rows of the last timed step (%d equal "
                             "element by element to the oracle's dist, the rest by its exact "
                             "distance certificate; every parent row tree-checked)"
                             % (good, len(res), eq)) if good == len(res) else \
                ("error: %d of %d rows of the last timed step failed the oracle's checks"
                 % (len(res) - good, len(res)))
        for cfg, (gc, s_c, d_c, p_c, l_c) in config_rows.items():
            res = list(ex.map(lambda i: certify(gc, s_c[i], d_c[i], p_c[i], l_c[i]),
                              range(len(s_c))))
            good = sum(1 for ok, _ in res if ok)
            cert["configs"][cfg] = ("oracle-certified %d/%d sources" % (good, len(res))
                                    if good == len(res) else
                                    "error: %d/%d sources failed" % (len(res) - good, len(res)))
    return base, cert


# ------------------------------------------------------------------ profiler cases

def run_profile_case(args):
    """Small cases for a profiler (ncu), nothing timed or printed but a line
    of what ran. 'levels': 3 warm-up searches, then --sources searches of
    --config (or only those at --source-index) in the host loop mode, so
    that every level is its own level_kernel launch. 'walk': the power-law graph's hub level (the level
    whose frontier holds the largest degree, most eccentric source) walked
    once by each mapping, 64 repeats."""
    import torch

    import frontier_bfs_csr_gb300 as fbc
    import graphgen
    device = torch.device("cuda", 0)
    if args.profile == "levels":
        if args.rmat_scale > 0:
            g = graphgen.rmat(args.rmat_scale, 16, 7)
            g.sources = graphgen.pick_sources(g, 24, 7)
        else:
            g = graphgen.config(args.config)
        row_ptr, col, _, _ = graph_tensors(torch, g, device)
        bfs = fbc.BfsCsr(row_ptr, col, True, fbc.default_options(loop_mode=fbc.BFS_CSR_LOOP_HOST))
        dist = torch.empty(g.n, dtype=torch.int32, device=device)
        parent = torch.empty_like(dist)
        nsrc = args.sources if args.sources > 0 else 1
        chosen = (g.sources[:nsrc] if not args.source_index else
                  [g.sources[int(i)] for i in args.source_index.split(",")])
        s0 = int(chosen[0])
        warm_levels = 0
        for _ in range(3):
            bfs.run(s0, dist, parent)
            warm_levels += bfs.sync()
        levels = []
        for s in chosen:
            bfs.run(int(s), dist, parent)
            levels.append(bfs.sync())
        bfs.close()
        print(json.dumps({"profile": "levels", "graph": g.name, "warmup_searches": 3,
                          "warmup_levels": warm_levels, "sources": [int(s) for s in chosen],
                          "levels_per_search": levels}))
        return
    g = graphgen.config(1)
    row_ptr, col, _, deg = graph_tensors(torch, g, device)
    bfs = fbc.BfsCsr(row_ptr, col, True)
    dist = torch.empty(g.n, dtype=torch.int32, device=device)
    lev = torch.empty(1, dtype=torch.int32, device=device)
    best, best_levels = None, -1
    for s in torch.nonzero(deg > 0).squeeze(1).tolist():
        bfs.run(s, dist, None, lev)
        L = int(lev.item())
        if L > best_levels:
            best, best_levels = s, L
    bfs.run(best, dist)
    bfs.sync()
    d = dist.cpu().numpy()
    dh = deg.cpu().numpy()
    hub_level = max(range(best_levels), key=lambda k: int(dh[d == k].max()))
    frontier = torch.from_numpy(np.nonzero(d == hub_level)[0].astype(np.int32)).to(device)
    out = torch.empty(frontier.numel(), dtype=torch.int32, device=device)
    for m in range(4):
        bfs.walk(frontier, 64, m, out)
    torch.cuda.synchronize(device)
    bfs.close()
    print(json.dumps({"profile": "walk", "source": best, "hub_level": hub_level,
                      "frontier": int(frontier.numel()),
                      "max_degree": int(dh[d == hub_level].max())}))


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as it stands, timed on the host: each step one FIFO BFS from
    the next source of the same workload (a bounded sample of a GPU step)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import graphgen
    import oracle
    g = graphgen.config(args.config)
    deg = np.diff(g.row_ptr.astype(np.int64))
    sources = [int(s) for s in (g.sources[:args.sources] if args.sources > 0 else g.sources)]
    for i in range(args.warmup):
        oracle.bfs(g.row_ptr, g.col, sources[i % len(sources)])
    edges, elapsed = 0, 0.0
    for i in range(args.steps):
        s = sources[(args.warmup + i) % len(sources)]
        t = time.perf_counter()
        d, _, _ = oracle.bfs(g.row_ptr, g.col, s)
        elapsed += time.perf_counter() - t
        edges += int(deg[d >= 0].sum())
    value = edges / elapsed / 1e9
    cores = host_cores()
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GTEPS", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOADS[args.config], "n": g.n, "nnz": g.nnz,
                       "sources_per_step": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": "GTEPS", "cores": 1,
                             "host_cores": cores["online"],
                             "host_cores_affinity": cores["affinity"],
                             "kind": "oracle",
                             "sample": "one source per step, %d steps" % args.steps},
            "e2e": {"value": round(value, 4), "unit": "GTEPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-overhead", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config GTEPS / roofline / parity of configs 1-4")
    ap.add_argument("--no-ablation", action="store_true",
                    help="skip the direction / advance ablation")
    ap.add_argument("--no-walk", action="store_true",
                    help="skip the isolated-level walk of the power-law graph")
    ap.add_argument("--profile", choices=["levels", "walk"], default=None,
                    help="run a small case for a profiler and exit (see run_profile_case)")
    ap.add_argument("--lanes", type=int, default=2,
                    help="searches bfs_csr_run_batch keeps in flight (1..8)")
    ap.add_argument("--sources", type=int, default=0,
                    help="use only the first S sources of the workload (0: all)")
    ap.add_argument("--rmat-scale", type=int, default=0,
                    help="--profile levels: an R-MAT graph of this scale (edge factor 16, "
                         "seed 7, 24 sources drawn with seed 7) instead of --config")
    ap.add_argument("--source-index", type=str, default="",
                    help="--profile levels: search only the workload's sources at these "
                         "indexes (comma-separated)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.profile is not None:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
