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

Roofline: the level loops' algorithmic bytes (the byte model in
`algorithmic_bytes`, replayed from each search's own distances and level
directions) over the time during which at least one level loop ran (from
device timer stamps the library records per search), against the measured
HBM copy bandwidth.

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


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


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


# ------------------------------------------------------------------ byte model

def algorithmic_bytes(torch, row_ptr, col, deg, src_of_edge, dist, stats, row_bytes):
    """Bytes the level kernel must touch, replayed from one search.

    row_ptr, col, deg, src_of_edge: device tensors of the graph (int64 row_ptr
    and degrees, int32 col and per-entry source). dist: the search's output.
    stats: its per-level records. Push level k (queue Q_k = frontier vertices
    with out-degree > 0, N_k = vertices at distance k + 1, N'_k those of them
    with edges): queue entries read (4 + 2R) |Q_k|, col 4 m_F, one visited word
    per edge 4 m_F, row offsets of each discovered vertex 2R |N_k|, dist and
    parent 8 |N_k|, its visited word 4 |N_k|, queue entries written (4 + 2R)
    |N'_k|. Pull level k (U'_k = unreached vertices of nonzero degree, c_k =
    entries scanned: up to and including the first neighbour at distance k for
    the vertices found, the whole row for the others): visited bitmap n/8,
    row offsets 2R |U'_k|, col 4 c_k, one frontier-bitmap word per scanned
    entry 4 c_k, dist and parent 8 |N_k|, next-frontier bitmap n/8, visited
    words with a discovery 4 per word. Representation switches: queue to bitmap
    n/8 + 8 |Q_k|; bitmap to queue n/8 + 2R |F_k| + (4 + 2R) |Q_k|. Output:
    the -1 of every unreached vertex's dist, 4 (n - reached), written by the
    level kernel when the search ends (the reached vertices' dist bytes are
    counted at their discovery above).
    """
    n = int(dist.numel())
    R = row_bytes
    words = (n + 31) // 32
    has_edges = deg > 0
    total = 0
    prev = DIR_PUSH
    per_level = []
    dist_src = None
    for k, st in enumerate(stats):
        in_k = dist == k
        nxt = dist == (k + 1)
        Fk = int(in_k.sum().item())
        Qk = int((in_k & has_edges).sum().item())
        Nk = int(nxt.sum().item())
        Nk_e = int((nxt & has_edges).sum().item())
        mF = int(deg[in_k].sum().item())
        b = 0
        if st["direction"] == DIR_PULL:
            if prev == DIR_PUSH:
                b += words * 4 + 8 * Qk
            unreached = ((dist < 0) | (dist > k)) & has_edges
            Uk = int(unreached.sum().item())
            if dist_src is None:
                dist_src = dist[src_of_edge.long()]
            dist_dst = dist[col.long()]
            hit = (dist_src == k + 1) & (dist_dst == k)
            pos = torch.nonzero(hit).squeeze(1)
            first = torch.full((n,), -1, dtype=torch.int64, device=dist.device)
            if pos.numel():
                owner = src_of_edge[pos].long()
                big = torch.full((n,), np.iinfo(np.int64).max, dtype=torch.int64,
                                 device=dist.device)
                big.scatter_reduce_(0, owner, pos, reduce="amin")
                found = nxt & has_edges
                first = torch.where(found, big - row_ptr[:-1], first)
            scanned_found = int((first[nxt] + 1).sum().item()) if Nk else 0
            not_found = unreached & ~nxt
            scanned_rest = int(deg[not_found].sum().item())
            c = scanned_found + scanned_rest
            touched_words = int(torch.unique(torch.nonzero(nxt).squeeze(1) // 32).numel()) if Nk else 0
            b += words * 4 + 2 * R * Uk + 4 * c + 4 * c + 8 * Nk + words * 4 + 4 * touched_words
        else:
            if prev == DIR_PULL:
                b += words * 4 + 2 * R * Fk + (4 + 2 * R) * Qk
            b += (4 + 2 * R) * Qk + 4 * mF + 4 * mF + 2 * R * Nk + 8 * Nk + 4 * Nk + (4 + 2 * R) * Nk_e
        per_level.append(b)
        total += b
        prev = st["direction"]
    total += 4 * int((dist < 0).sum().item())
    return total, per_level


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


def init_bytes(n: int, with_parent: bool = True) -> int:
    """The init kernel with bitmap discovery: one hop-code byte per vertex,
    parent (-1), the visited bitmap written and the dead bitmap read."""
    words = (n + 31) // 32
    return (n + 15) // 16 * 16 + (4 * n if with_parent else 0) + 8 * words


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
    row_ptr = torch.from_numpy(g.row_ptr).to(device)
    col = torch.from_numpy(g.col).to(device)
    R = 8 if g.row_ptr_64 else 4
    bfs = fbc.BfsCsr(row_ptr, col, symmetric=True,
                     options=fbc.default_options(lanes=args.lanes))
    n = g.n
    dist = torch.empty(n, dtype=torch.int32, device=device)
    parent = torch.empty(n, dtype=torch.int32, device=device)
    deg = torch.diff(row_ptr.to(torch.int64))
    stream = torch.cuda.current_stream(device)

    # Untimed pass over every source: warms the kernels and records, per
    # source, the walked-edge count, the level records and the byte model.
    src_of_edge = torch.repeat_interleave(torch.arange(n, device=device, dtype=torch.int32),
                                          deg)
    per_source = {}
    for s in sources:
        bfs.run(s, dist, parent, stream=stream)
        levels = bfs.sync(stream)
        reached = dist >= 0
        edges = int(deg[reached].sum().item())
        stats = bfs.level_stats()
        lb, per_level = algorithmic_bytes(torch, row_ptr.to(torch.int64), col, deg, src_of_edge,
                                          dist, stats, R)
        torch.cuda.empty_cache()
        per_source[s] = {"levels": levels, "edges": edges, "level_bytes": lb,
                         "directions": "".join("P" if x["direction"] == DIR_PUSH else "U"
                                               for x in stats),
                         "per_level_bytes": per_level}
    del src_of_edge
    # Timed step: one bfs_csr_run_batch over the batch of sources (the searches
    # run on `lanes` lanes at once); dist/parent rows per source.
    k = len(sources)
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
    # The last step's outputs against the untimed pass (same searches).
    status_ok = bool(torch.equal(dist_b[-1], dist)) if k else True

    st = stamps.cpu().numpy().reshape(-1, 3).astype(np.float64) * 1e-6   # ms
    runs = st.shape[0]
    init_ms = (st[:, 1] - st[:, 0]).tolist()
    level_ms = (st[:, 2] - st[:, 1]).tolist()
    busy = busy_time(zip(st[:, 1], st[:, 2]))
    edges_local = sum(per_source[s]["edges"] for s in sources) * args.steps
    edges_all = sum_over_ranks(torch, ws, float(edges_local), device)
    value = edges_all / (total_ms * 1e-3) / 1e9

    lvl_bytes = sum(per_source[s]["level_bytes"] for s in sources) * args.steps
    achieved = lvl_bytes / (busy * 1e-3) / 1e9
    init_b = init_bytes(n) * runs
    init_gbs = init_b / (sum(init_ms) * 1e-3) / 1e9

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
                     "algorithmic_bytes_per_launch": int(lvl_bytes / runs),
                     "launch_ms_mean": round(sum(level_ms) / runs, 4),
                     "level_kernel_busy_ms": round(busy, 4),
                     "timing": "device timer stamps per search; achieved = algorithmic bytes "
                               "of every level-loop launch / time any level loop ran"},
        "init_kernel": {"achieved_gbs": round(init_gbs, 1), "frac": round(init_gbs / peak, 4),
                        "bytes_per_launch": init_bytes(n), "launch_ms_mean": round(sum(init_ms) / runs, 4)},
        "clocks": clocks,
        "gpu_launches": 2 * runs,
        "status_after_timing": "ok" if status_ok else "error",
    }
    traffic = read_traffic_summary(args.config)
    if traffic is not None:
        result["roofline"]["traffic"] = traffic
    bfs.close()

    if rank == 0 and not args.no_overhead:
        result["per_level_overhead_us"] = per_level_overhead(torch, fbc, graphgen, device)
    if not args.no_e2e:
        result["e2e"] = run_e2e(torch, fbc, g, sources, args, device, ws)
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(g, sources)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


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


def per_level_overhead(torch, fbc, graphgen, device):
    """Time per level on graphs made of narrow levels: the 2048x2048 grid from
    its corner, and a 10,000-vertex path (one vertex per level), in the
    persistent loop and in the host loop (one launch + one device->host read
    per level, the structure the Day 38 page measures)."""
    out = {}
    cases = [("grid_2048", graphgen.config(4)), ("path_10000", graphgen.path_graph(10000))]
    for name, g in cases:
        rp = torch.from_numpy(g.row_ptr).to(device)
        cl = torch.from_numpy(g.col).to(device)
        s = int(g.sources[0]) if g.sources is not None else 0
        dist = torch.empty(g.n, dtype=torch.int32, device=device)
        row = {}
        for mode, loop in (("persistent", fbc.BFS_CSR_LOOP_PERSISTENT),
                           ("host_loop", fbc.BFS_CSR_LOOP_HOST)):
            b = fbc.BfsCsr(rp, cl, True, fbc.default_options(loop_mode=loop))
            b.run(s, dist)
            levels = b.sync()
            reps = 3 if loop == fbc.BFS_CSR_LOOP_PERSISTENT else 1
            times = []
            for _ in range(reps):
                torch.cuda.synchronize(device)
                t = time.perf_counter()
                b.run(s, dist)
                b.sync()
                times.append(time.perf_counter() - t)
            b.close()
            row[mode] = round(min(times) * 1e6 / levels, 3)
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
    elapsed = max_over_ranks(torch, ws, elapsed, device)
    edges = sum_over_ranks(torch, ws, float(edges_per_step * steps), device)
    return {"value": round(edges / elapsed / 1e9, 3), "unit": "GTEPS",
            "h2d_bytes_per_step": int(g.row_ptr.nbytes + g.col.nbytes + 8 * k),
            "d2h_bytes_per_step": int(k * (8 * g.n + 4)),
            "steps": steps, "ms_per_step": round(elapsed / steps * 1e3, 3),
            "api": "bfs_csr_create_host / bfs_csr_run_host_batch"}


def cpu_baseline(g, sources, budget_s: float = 20.0):
    """The oracle (sequential FIFO BFS in C, one host thread) on a bounded
    sample of the same workload: sources in order until ~budget_s seconds."""
    import oracle
    deg = np.diff(g.row_ptr.astype(np.int64))
    done, edges, elapsed = [], 0, 0.0
    for s in sources:
        t = time.perf_counter()
        d, _, _ = oracle.bfs(g.row_ptr, g.col, s, want_parent=True)
        elapsed += time.perf_counter() - t
        edges += int(deg[d >= 0].sum())
        done.append(s)
        if elapsed > budget_s:
            break
    return {"value": round(edges / elapsed / 1e9, 4), "unit": "GTEPS", "cores": 1,
            "kind": "oracle",
            "sample": "%d of %d sources of the timed workload, %.1f s" % (len(done), len(sources),
                                                                          elapsed)}


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
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GTEPS", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOADS[args.config], "n": g.n, "nnz": g.nnz,
                       "sources_per_step": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": "GTEPS", "cores": 1,
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
    ap.add_argument("--lanes", type=int, default=2,
                    help="searches bfs_csr_run_batch keeps in flight (1..8)")
    ap.add_argument("--sources", type=int, default=0,
                    help="use only the first S sources of the workload (0: all)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
