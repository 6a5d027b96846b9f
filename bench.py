#!/usr/bin/env python
"""Benchmark of the particle-to-grid deposit hot path on GB300.

Headline workload (one "step" = the whole current-deposit path on one batch):
  3D first-order (CIC) current deposit, periodic 256^3 grid, 16 particles per
  cell (268,435,456 particles), sort-time positions x_s, deposit positions
  x = x_s + v (0.1 % displaced by up to 3 cells), 8^3 tiles, 2-cell halo.
  step = tile counting sort (key, count, scan, permute) + tiled deposit
  (per-cell register accumulation over each tile segment, escape valve, one
  flush per node and tile).  Inputs stay resident in HBM; they are
  far larger than L2 (7.5 GB vs 129 MB), so no L2 flush is needed between steps.

Also measured in the same run (the other rows of the hot path, each on its own
workload): the 1D windowed CIC histogram, the 2D CIC deposit on 512^2, the 3D
quadratic deposit on the 192^3 density bump, and the ECSIM mass matrix on 64^3
(TF32 and BF16 tensor cores, and the CUDA-core baseline).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "particle deposits/sec (M/s) and achieved HBM GB/s vs peak on 1 GB300"
UNIT = "M deposits/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")


# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by kernel name.

    Each line: <kernel> <bytes_per_launch> <units_per_launch> <source-hash>.  An
    entry counts only while the kernel sources still hash to the recorded value.
    """
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    out = {}
    if not os.path.exists(p):
        return out
    with open(p) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) == 4 and line[3] == source_hash(line[0]):
                out[line[0]] = (float(line[1]), float(line[2]))
    return out


# Host -> device copies of the end-to-end leg run on this many streams.
UPLOAD_STREAMS = 4

# The source files each timed kernel is built from (all of them for a name not listed).
_COMMON = ["common.cuh", "checked.cuh", "profile.cuh"]
KERNEL_SOURCES = {
    "sort": ["tile_sort.cu", "tcgen05.cuh"] + _COMMON,
    "deposit_tiled": ["deposit_tiled.cuh", "deposit_quad3d.cuh", "deposit.cuh", "deposit.cu", "deposit_2d.cu",
                      "deposit_3d.cu"] + _COMMON,
    "deposit_zigzag": ["deposit_zigzag.cu", "deposit_tiled.cuh", "deposit.cuh"] + _COMMON,
    "mass": ["mass_matrix.cu", "mass_cic.cuh", "mass_cic_tc.cu", "mass_tsc.cu", "mass_tsc.cuh", "mass_tsc_tc.cu",
             "mass_common.cuh", "tcgen05.cuh"] + _COMMON,
    "cic1d": ["cic1d.cu"] + _COMMON,
}


def source_hash(kernel=None):
    """Hash of the sources a kernel is built from (prefix match on its timer name)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "particle_cell_grid_gb300", "csrc")
    files = None
    if kernel is not None:
        for key, fl in KERNEL_SOURCES.items():
            if kernel.startswith(key):
                files = fl
                break
    if files is None:
        files = [fn for fn in os.listdir(csrc) if fn.endswith((".cu", ".cuh"))]
    for fn in sorted(files):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:12]


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={CLOCK_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(", ") for r in self.file.read().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summarize(rows):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        busy = [r for r in rows if len(r) >= 10 and r[9].strip().isdigit() and int(r[9]) > 0] or rows
        for r in busy:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for k, nm in enumerate(names):
                if len(r) > 5 + k and "Active" in r[5 + k] and "Not" not in r[5 + k]:
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
class Dist:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            self.dist = dist

    def init(self, backend):
        if self.world > 1:
            import torch
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            self.dist.init_process_group(backend=backend)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x):
        if self.world == 1:
            return x
        import torch
        dev = "cuda" if self.dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


# ---------------------------------------------------------------------------
def time_steps(step, steps, warmup, dist, stream, pcg=None):
    """W untimed warm-up steps, then K steps between CUDA events on `stream`.

    With `pcg` given, the library's per-kernel event timing is on for exactly
    the K timed steps."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    if pcg is not None:
        pcg.profile_collect()   # drop anything recorded before
        pcg.profile_enable(True)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    if pcg is not None:
        pcg.profile_enable(False)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    return a.elapsed_time(b)  # ms


def roofline_entry(name, prof, bytes_per_launch, peak, traffic, units_per_launch):
    launches, total_ms = prof[name]
    avg_ms = total_ms / launches
    gbs = bytes_per_launch / (avg_ms * 1e-3) / 1e9
    tr = None
    if name in traffic:
        t_bytes, t_units = traffic[name]
        tr = t_bytes * (units_per_launch / t_units)  # scaled to a full launch when captured smaller
    return {"bound": "hbm", "kernel": name, "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "traffic": None if tr is None else round(tr),
            "algorithmic_bytes": int(bytes_per_launch), "avg_ms": round(avg_ms, 4), "launches": launches}


def current_workload(pcg, d, steps, warmup, dist, peaks, traffic, e2e_steps=0):
    """Time sort + tiled deposit on a current-deposit workload; returns a dict."""
    import torch
    grid, dim = d["grid"], len(d["grid"])
    n = d["n"]
    stream = torch.cuda.current_stream()
    dev = lambda a: torch.from_numpy(a).cuda()
    pos = [dev(p) for p in d["pos"]]
    vel = [dev(v) for v in d["vel"]]
    q = dev(d["q"])
    separate_keys = d["key_pos"] is not d["pos"]
    kp = [dev(k) for k in d["key_pos"]] if separate_keys else pos
    payload = pos + vel + [q]
    out = [torch.empty_like(p) for p in payload]
    nt = pcg.n_tiles(grid, d["tile"])
    offs = torch.empty(nt + 1, dtype=torch.int32, device="cuda")
    J = torch.empty((3,) + tuple(reversed(grid)), dtype=torch.float32, device="cuda")
    ws_s = torch.empty(max(pcg.tile_sort_workspace_size(grid, d["tile"], n, len(payload)), 256), dtype=torch.uint8,
                       device="cuda")
    ws_d = torch.empty(max(pcg.deposit_current_workspace_size(grid, d["tile"], n), 256), dtype=torch.uint8,
                       device="cuda")
    stats = pcg.new_stats()

    def step():
        pcg.tile_sort(grid, d["tile"], kp, payload, out=out, tile_offsets=offs, workspace=ws_s)
        pcg.deposit_current(grid, d["order"], out[:dim], out[dim:dim + 3], out[dim + 3], tile_offsets=offs,
                            tile=d["tile"], halo=d["halo"], J=J, stats=stats, workspace=ws_d)

    step()
    torch.cuda.synchronize()
    st = pcg.read_stats(stats)
    ms = time_steps(step, steps, warmup, dist, stream, pcg=pcg)
    timed = pcg.profile_collect()
    ms = dist.max(ms)
    res = {"n": n, "ms_per_step": ms / steps, "value": n * steps * dist.world / (ms * 1e-3) / 1e6,
           "escaped_per_step": st["n_escaped"], "invalid": st["n_invalid"], "profile": timed}
    # load balance: particles per tile (the sentinel bin of invalid particles excluded)
    tiles = np.diff(offs.cpu().numpy().astype(np.int64)[:nt + 1])[:nt]
    res["tile_load"] = {"max": int(tiles.max()), "mean": round(float(tiles.mean()), 1),
                        "max_over_mean": round(float(tiles.max() / max(tiles.mean(), 1e-30)), 2)}
    # stencil node updates the deposit performs per second: (order + 1)^dim x 3 components per particle
    dep = timed.get("deposit_tiled")
    if dep:
        upd = n * (d["order"] + 1) ** dim * 3
        res["stencil_updates_per_s"] = round(upd / (dep[1] / dep[0] * 1e-3), 1)
    # algorithmic bytes per launch of the main kernels
    kbytes = 4 * dim * (1 if separate_keys else 0)
    node_bytes = 12 * int(np.prod(grid))
    nf = dim + 4  # payload fields: positions, three velocity components, q
    alg = {
        "deposit_tiled": n * (4 * (dim + 4)) + node_bytes,
        "sort_scatter": n * (kbytes + 2 * 4 * nf),
        "sort_count": n * 4 * dim,
        # pass 1 reads key positions and payload, writes payload and the tile key;
        # pass 2 reads payload and key, writes payload; one pass: in and out once
        "sort_partition1": n * (kbytes + 4 * nf + 4 * (nf + 1)),
        "sort_partition2": n * (4 * (nf + 1) + 4 * nf),
        "sort_partition": n * (kbytes + 2 * 4 * nf),
    }
    kern = {}
    for name, b in alg.items():
        if name in timed:
            kern[name] = roofline_entry(name, timed, b, peaks["hbm_gbs"], traffic, n)
    res["kernels"] = kern
    # the whole sort (every sort launch of a step) on the bytes a sort must move:
    # key positions read once, the payload read once and written once
    sort_ms = sum(v[1] for k, v in timed.items() if k.startswith("sort_")) / max(steps, 1)
    if sort_ms > 0:
        sb = n * (kbytes + 2 * 4 * nf)
        gbs = sb / (sort_ms * 1e-3) / 1e9
        res["sort_roofline"] = {"bound": "hbm", "kernels": "all sort launches of one step", "ms": round(sort_ms, 4),
                                "algorithmic_bytes": int(sb), "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)}
    dom = max(timed.items(), key=lambda kv: kv[1][1])[0]
    res["dominant"] = dom
    res["gpu_launches"] = sum(v[0] for v in timed.values())

    if e2e_steps:
        # end to end through the public API: every step copies its inputs from
        # pinned host memory to the device and reads J back.  The copies of step
        # k + 1's inputs run on UPLOAD_STREAMS upload streams (the fields dealt
        # round-robin, so that several copy engines share the host link) into a
        # second set of device inputs while step k computes; J alternates between
        # two device buffers and each step's J is read back on its own stream, so
        # that the compute stream never queues behind a copy (it waits only for
        # its inputs and for the read-back of the J buffer it is about to reuse).
        h_in = [torch.from_numpy(a).pin_memory() for a in (list(d["key_pos"]) if separate_keys else [])
                + list(d["pos"]) + list(d["vel"]) + [d["q"]]]
        sets = [(kp if separate_keys else []) + payload]
        sets.append([torch.empty_like(t) for t in sets[0]])
        Jb = [J, torch.empty_like(J)]
        h_J = [torch.empty(J.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
        nk = dim if separate_keys else 0
        ups = [torch.cuda.Stream() for _ in range(UPLOAD_STREAMS)]  # uploads
        rs = torch.cuda.Stream()   # read-backs
        ready = [[torch.cuda.Event() for _ in ups] for _ in range(2)]  # inputs of set b on the device
        free = [torch.cuda.Event(), torch.cuda.Event()]    # set b consumed by its step
        done = [torch.cuda.Event(), torch.cuda.Event()]    # J buffer b written by its step
        read = [torch.cuda.Event(), torch.cuda.Event()]    # J buffer b read back

        def step_on(dset, Jt):
            kpp = dset[:nk] if separate_keys else dset[:dim]
            py = dset[nk:]
            pcg.tile_sort(grid, d["tile"], kpp, py, out=out, tile_offsets=offs, workspace=ws_s)
            pcg.deposit_current(grid, d["order"], out[:dim], out[dim:dim + 3], out[dim + 3], tile_offsets=offs,
                                tile=d["tile"], halo=d["halo"], J=Jt, stats=stats, workspace=ws_d)

        def upload(b, wait=None):
            for u, cs in enumerate(ups):
                if wait is not None:
                    cs.wait_event(wait)
                with torch.cuda.stream(cs):
                    for f in range(u, len(h_in), len(ups)):
                        sets[b][f].copy_(h_in[f], non_blocking=True)
                    ready[b][u].record(cs)

        def e2e_run(k_steps):
            for b in (0, 1):
                free[b].record(stream)
                read[b].record(stream)
            for cs in ups:
                cs.wait_stream(stream)
            rs.wait_stream(stream)
            upload(0)
            for k in range(k_steps):
                b = k & 1
                if k + 1 < k_steps:
                    upload(b ^ 1, wait=free[b ^ 1])
                for ev in ready[b]:
                    stream.wait_event(ev)
                stream.wait_event(read[b])
                step_on(sets[b], Jb[b])
                free[b].record(stream)
                done[b].record(stream)
                rs.wait_event(done[b])
                with torch.cuda.stream(rs):
                    h_J[b].copy_(Jb[b], non_blocking=True)
                    read[b].record(rs)
            stream.wait_stream(rs)

        e2e_run(2)  # warm-up
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        ea = torch.cuda.Event(enable_timing=True)
        eb = torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        e2e_run(e2e_steps)
        eb.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        ms_e = dist.max(ea.elapsed_time(eb))
        res["e2e"] = {"value": round(n * e2e_steps * dist.world / (ms_e * 1e-3) / 1e6, 3), "unit": UNIT,
                      "h2d_bytes_per_step": int(sum(h.numel() * 4 for h in h_in)),
                      "d2h_bytes_per_step": int(J.numel() * 4), "ms_per_step": round(ms_e / e2e_steps, 3),
                      "overlap": f"inputs of step k+1 uploaded on {UPLOAD_STREAMS} streams during step k; J "
                                 "double-buffered and read back on its own stream"}

        # the host link alone: the same pinned copies with nothing else running,
        # on one stream and on the upload streams
        def h2d_alone(streams):
            la = torch.cuda.Event(enable_timing=True)
            lb = torch.cuda.Event(enable_timing=True)
            la.record(streams[0])
            ends = []
            for u, cs in enumerate(streams):
                cs.wait_event(la)
                with torch.cuda.stream(cs):
                    for f in range(u, len(h_in), len(streams)):
                        sets[0][f].copy_(h_in[f], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                ends.append(ev)
            for ev in ends:
                streams[0].wait_event(ev)
            lb.record(streams[0])
            torch.cuda.synchronize()
            return round(res["e2e"]["h2d_bytes_per_step"] / (la.elapsed_time(lb) * 1e-3) / 1e9, 1)

        res["e2e"]["h2d_alone_gbs"] = h2d_alone(ups)
        res["e2e"]["h2d_alone_one_stream_gbs"] = h2d_alone(ups[:1])
        del h_in, h_J, sets, Jb
    del pos, vel, q, kp, payload, out, J, ws_s, ws_d
    torch.cuda.empty_cache()
    return res


def zigzag_workload(pcg, d, steps, warmup, dist, peaks, traffic):
    """Time sort (keyed on the previous positions) + tiled charge-conserving
    zigzag deposit on a 3D move workload; returns a dict."""
    import torch
    grid, n = d["grid"], d["n"]
    stream = torch.cuda.current_stream()
    dev = lambda a: torch.from_numpy(a).cuda()
    prev = [dev(a) for a in d["pos_prev"]]
    pos = [dev(a) for a in d["pos"]]
    q = dev(d["q"])
    payload = prev + pos + [q]
    out = [torch.empty_like(p) for p in payload]
    nt = pcg.n_tiles(grid, d["tile"])
    offs = torch.empty(nt + 1, dtype=torch.int32, device="cuda")
    J = torch.empty((3,) + tuple(reversed(grid)), dtype=torch.float32, device="cuda")
    ws_s = torch.empty(max(pcg.tile_sort_workspace_size(grid, d["tile"], n, len(payload)), 256), dtype=torch.uint8,
                       device="cuda")
    ws_d = torch.empty(max(pcg.deposit_current_workspace_size(grid, d["tile"], n), 256), dtype=torch.uint8,
                       device="cuda")
    stats = pcg.new_stats()

    def step():
        pcg.tile_sort(grid, d["tile"], prev, payload, out=out, tile_offsets=offs, workspace=ws_s)
        pcg.deposit_zigzag(grid, out[0:3], out[3:6], out[6], d["dt"], tile_offsets=offs, tile=d["tile"], J=J,
                           stats=stats, workspace=ws_d)

    step()
    torch.cuda.synchronize()
    st = pcg.read_stats(stats)
    ms = time_steps(step, steps, warmup, dist, stream, pcg=pcg)
    timed = pcg.profile_collect()
    ms = dist.max(ms)
    nf = 7  # payload fields: previous and current positions, q
    alg = {
        "deposit_zigzag": n * 4 * nf + 12 * int(np.prod(grid)),
        "sort_count": n * 12,
        "sort_partition1": n * (4 * nf + 4 * (nf + 1)),
        "sort_partition2": n * (4 * (nf + 1) + 4 * nf),
        "sort_partition": n * 2 * 4 * nf,
        "sort_scatter": n * 2 * 4 * nf,
    }
    kern = {name: roofline_entry(name, timed, b, peaks["hbm_gbs"], traffic, n)
            for name, b in alg.items() if name in timed}
    res = {"workload": f"zigzag3d {grid[0]}x{grid[1]}x{grid[2]} x {n // int(np.prod(grid))} ppc, "
                       "charge-conserving, sorted by previous position", "particles": n,
           "value": round(n * steps * dist.world / (ms * 1e-3) / 1e6, 1), "unit": UNIT,
           "ms_per_step": round(ms / steps, 4), "kernels": kern, "escaped_per_step": st["n_escaped"],
           "invalid": st["n_invalid"], "gpu_launches": sum(v[0] for v in timed.values())}
    del prev, pos, q, payload, out, J, ws_s, ws_d
    torch.cuda.empty_cache()
    return res


def host_cpu():
    """Host cores this process may use, all online cores, and the CPU model."""
    try:
        usable = len(os.sched_getaffinity(0))
    except Exception:
        usable = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"usable": usable, "nproc": os.cpu_count() or usable, "model": model or "unknown"}


def mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except Exception:
        pass
    return 8 << 30


def oracle_on_threads(d, ranges, threads):
    """The oracle's deposit over the particle ranges, one Python thread per range
    (ctypes releases the GIL during the call) and one private J each; the
    partial grids are summed.  Returns the summed J."""
    import concurrent.futures as cf
    import oracle

    def one(r):
        a, b = r
        return oracle.deposit_current(d["grid"], d["order"], [p[a:b] for p in d["pos"]],
                                      [v[a:b] for v in d["vel"]], d["q"][a:b])[0]

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(one, ranges))
    J = parts[0]
    for P in parts[1:]:
        J += P
    return J


def cpu_threads_for(d):
    """Threads for the all-core leg: every usable core, fewer when the private
    fp64 grids would take more than 40 % of the available host memory."""
    cpu = host_cpu()
    j_bytes = 3 * 8 * int(np.prod(d["grid"]))
    fit = max(1, int(0.4 * mem_available_bytes() // max(j_bytes, 1)))
    return min(cpu["usable"], fit), cpu


def cpu_baseline_current(d, target_s=8.0):
    """The fp64 oracle as it stands on bounded samples of the same workload:
    one thread, then the same calls spread over the host's cores."""
    import oracle
    n = d["n"]
    s0 = min(n, 500_000)
    t = time.perf_counter()
    oracle.deposit_current(d["grid"], d["order"], [p[:s0] for p in d["pos"]], [v[:s0] for v in d["vel"]],
                           d["q"][:s0])
    t0 = time.perf_counter() - t
    s = int(min(n, max(s0, s0 * target_s / max(t0, 1e-3))))
    t = time.perf_counter()
    oracle.deposit_current(d["grid"], d["order"], [p[:s] for p in d["pos"]], [v[:s] for v in d["vel"]],
                           d["q"][:s])
    dt1 = time.perf_counter() - t
    one = s / dt1 / 1e6
    threads, cpu = cpu_threads_for(d)
    sm = int(min(n, s * threads))
    bounds = np.linspace(0, sm, threads + 1).astype(np.int64)
    ranges = [(int(bounds[i]), int(bounds[i + 1])) for i in range(threads)]
    t = time.perf_counter()
    oracle_on_threads(d, ranges, threads)
    dtm = time.perf_counter() - t
    allc = sm / dtm / 1e6
    return {"value": round(allc, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "single_thread_value": round(one, 4), "host_cores": cpu["nproc"], "usable_cores": cpu["usable"],
            "cpu_model": cpu["model"],
            "sample": f"all-core leg: first {sm} of {n} particles (random order) of the same workload, full grid, "
                      f"fp64 C oracle on {threads} threads with one private J each, summed, {dtm:.1f} s; "
                      f"single-thread leg: first {s} particles, {dt1:.1f} s"}


def mass_workload(pcg, steps, warmup, dist, peaks, traffic, edge=64):
    import torch
    import synth
    d = synth.mass3d(grid=(edge, edge, edge))
    grid, n = d["grid"], d["n"]
    dev = lambda a: torch.from_numpy(a).cuda()
    dp = [dev(p) for p in d["pos"]]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    M = torch.empty(tuple(reversed(grid)) + (27, 3, 3), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    res = {"workload": f"mass3d {edge}^3 x 64 ppc (CIC, 27 offsets x 3x3 blocks)", "particles": n}
    alg_bytes = n * 28 + M.numel() * 4
    useful_flops = n * 8 * 8 * 9 * 2
    issued = {"tf32": n * 128 * 16 * 2, "bf16": n * 128 * 16 * 2, "simt": 0}
    tf32_peak = peaks["bf16_tflops"] / 2.0   # dense TF32 = half the bf16 rate (nominal 1.1 vs 2.25 PF)
    for prec in ("tf32", "bf16", "simt"):
        step = lambda: pcg.assemble_mass_matrix(grid, out[:3], out[3], out[4:7], offs, precision=prec, M=M)
        step()
        ms = time_steps(step, steps, warmup, dist, stream, pcg=pcg)
        timed = pcg.profile_collect()
        name = f"mass_matrix_{prec}"
        ent = roofline_entry(name, timed, alg_bytes, peaks["hbm_gbs"], traffic, n)
        kms = ent["avg_ms"]
        r = {"ms_per_call": round(ms / steps, 4), "kernel_ms": kms,
             "M_particles_per_s": round(n / (ms / steps * 1e-3) / 1e6, 1), "roofline": ent,
             "useful_tflops": round(useful_flops / (kms * 1e-3) / 1e12, 2)}
        if prec != "simt":
            pk = tf32_peak if prec == "tf32" else peaks["bf16_tflops"]
            r["issued_tflops"] = round(issued[prec] / (kms * 1e-3) / 1e12, 2)
            r["tensor_frac_issued"] = round(issued[prec] / (kms * 1e-3) / 1e12 / pk, 4)
            r["tensor_peak_tflops"] = pk
        res[prec] = r
    # the scalar (MPM) matrix of the same particles: one component, 27 floats per node
    Ms = torch.empty(tuple(reversed(grid)) + (27,), dtype=torch.float32, device="cuda")
    alg_s = n * 16 + Ms.numel() * 4
    sc = {"workload": f"scalar mass matrix, same particles ({edge}^3 x 64 ppc, 27 offsets)"}
    for prec in ("tf32", "bf16", "simt"):
        step = lambda: pcg.assemble_mass_matrix_scalar(grid, out[:3], out[3], offs, precision=prec, M=Ms)
        step()
        ms = time_steps(step, steps, warmup, dist, stream, pcg=pcg)
        timed = pcg.profile_collect()
        ent = roofline_entry(f"mass_scalar_{prec}", timed, alg_s, peaks["hbm_gbs"], traffic, n)
        sc[prec] = {"ms_per_call": round(ms / steps, 4), "kernel_ms": ent["avg_ms"],
                    "M_particles_per_s": round(n / (ms / steps * 1e-3) / 1e6, 1), "roofline": ent}
    res["scalar"] = sc
    del dp, out, offs, M, Ms
    torch.cuda.empty_cache()
    return res


def tsc_workload(pcg, steps, warmup, dist, peaks, traffic, edge=32):
    """Second-order (TSC) ECSIM mass matrix, 125 offsets x 3x3 per node: tcgen05
    TF32 and BF16, and the CUDA-core baseline."""
    import torch
    import synth
    d = synth.mass3d(grid=(edge, edge, edge))
    grid, n = d["grid"], d["n"]
    dev = lambda a: torch.from_numpy(a).cuda()
    dp = [dev(p) for p in d["pos"]]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    M = torch.empty(tuple(reversed(grid)) + (125, 3, 3), dtype=torch.float32, device="cuda")
    res = {"workload": f"mass3d TSC {edge}^3 x 64 ppc (125 offsets x 3x3 blocks)", "particles": n}
    useful = n * 27 * 27 * 9 * 2
    # issued tensor flops: per 64-particle chunk of a cell pair, 4 planes of M=128 x N=160 x K=64
    ncells = int(np.prod(grid))
    counts = np.diff(offs.cpu().numpy().astype(np.int64)[:ncells + 1])
    c2 = np.zeros(((grid[0] + 1) // 2) * 2 * grid[1] * grid[2], np.int64).reshape(grid[2], grid[1], -1)
    c2[:, :, :grid[0]] = counts.reshape(grid[2], grid[1], grid[0])
    pairs = c2.reshape(grid[2], grid[1], -1, 2)
    chunks = int(np.maximum((pairs[..., 0] + 31) // 32, (pairs[..., 1] + 31) // 32).sum())
    issued = chunks * 4 * 128 * 160 * 64 * 2
    tf32_peak = peaks["bf16_tflops"] / 2.0   # dense TF32 = half the bf16 rate (nominal 1.1 vs 2.25 PF)
    for prec in ("tf32", "bf16", "simt"):
        step = lambda: pcg.assemble_mass_matrix(grid, out[:3], out[3], out[4:7], offs, precision=prec, M=M, order=2)
        step()
        ms = time_steps(step, steps, warmup, dist, torch.cuda.current_stream(), pcg=pcg)
        timed = pcg.profile_collect()
        ent = roofline_entry(f"mass_tsc_{prec}", timed, n * 28 + M.numel() * 4, peaks["hbm_gbs"], traffic, n)
        r = {"ms_per_call": round(ms / steps, 4), "kernel_ms": ent["avg_ms"],
             "M_particles_per_s": round(n / (ms / steps * 1e-3) / 1e6, 1), "roofline": ent,
             "useful_tflops": round(useful / (ent["avg_ms"] * 1e-3) / 1e12, 2)}
        if prec != "simt":
            pk = tf32_peak if prec == "tf32" else peaks["bf16_tflops"]
            r["issued_tflops"] = round(issued / (ent["avg_ms"] * 1e-3) / 1e12, 2)
            r["tensor_frac_issued"] = round(issued / (ent["avg_ms"] * 1e-3) / 1e12 / pk, 4)
            r["tensor_peak_tflops"] = pk
        res[prec] = r
    del dp, out, offs, M
    torch.cuda.empty_cache()
    return res


def cic1d_workload(pcg, steps, warmup, dist):
    """The 1D windowed CIC histogram + loss, and its gradient dL/dx0, at the
    pages' N = 2000 and at N = 10^7 (the size their gradient timings use)."""
    import torch
    import synth
    dev = lambda a: torch.from_numpy(a).cuda()
    out = {"workload": "cic1d 1024 bins, T=50, h=0.005"}
    for n, k in ((2000, steps), (10_000_000, max(5, steps // 20))):
        d = synth.cic1d(n=n)
        x0, v, tg = dev(d["x0"]), dev(d["v"]), dev(d["target"])
        H = torch.empty(d["nbins"], dtype=torch.float32, device="cuda")
        L = torch.empty(1, dtype=torch.float64, device="cuda")
        g = torch.empty(n, dtype=torch.float64, device="cuda")
        args = (d["nsteps"], d["dt"], d["halfwidth"])
        fwd = lambda: pcg.deposit_cic1d(x0, v, tg, *args, H=H, loss=L)
        grad = lambda: pcg.deposit_cic1d_grad(x0, v, tg, *args, H=H, loss=L, dx0=g)
        for name, step in (("forward", fwd), ("forward+grad", grad)):
            us = time_steps(step, k, warmup, dist, torch.cuda.current_stream()) * 1e3 / k
            out[f"N={n} {name}"] = {"us_per_call": round(us, 2),
                                    "M_particle_steps_per_s": round(n * 50 / (us * 1e-6) / 1e6, 1)}
        del x0, v, tg, g
    out["note"] = ("N=2000: latency-bound, one cluster launch (+1 for the gradient); N=10^7: 80 MB of "
                   "input, resident in L2 between calls; ~4.5 screened steps per particle (those near its "
                   "window crossings), fp64 decisions on the ~5e6 selected pairs")
    return out


# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import particle_cell_grid_gb300 as pcg
    import synth

    dist = Dist(args.gpus)
    dist.init("nccl")
    torch.cuda.set_device(dist.local)
    pcg._lib.load()  # fails loudly without the library
    peaks, peak_src = load_peaks()
    traffic = load_traffic()

    g = args.grid
    d = synth.cic3d_drift(grid=(g, g, g))
    sampler = ClockSampler(dist.local)
    sampler.start()
    main = current_workload(pcg, d, args.steps, args.warmup, dist, peaks, traffic, e2e_steps=args.e2e_steps)
    clocks = ClockSampler.summarize(sampler.stop())
    cpu = cpu_baseline_current(d) if (dist.rank == 0 and dist.world == 1 and not args.no_cpu) else None
    del d

    # the roofline of the step's deposit kernel (the kernel the >= 50 % target is
    # about: particles read once + J written once); the sort is reported beside it
    roof = main["kernels"].get("deposit_tiled") or next(iter(main["kernels"].values()))
    line = {
        "metric": METRIC, "value": round(main["value"], 3), "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(main["ms_per_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64 generators of synth/)",
        "config": {"workload": f"cic3d_drift {g}^3 x 16 ppc, CIC current deposit (sort + tiled deposit)",
                   "grid": [g, g, g], "particles": main["n"], "order": 1, "tile": 8, "halo": 2,
                   "step": "pcg_tile_sort + pcg_deposit_current", "parallelism": "replicas" if dist.world > 1 else "1 GPU",
                   "l2": "inputs (7.5 GB) larger than L2 (129 MB); no flush"},
        "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")} |
                    {"kernel": roof["kernel"], "algorithmic_bytes": roof["algorithmic_bytes"],
                     "avg_ms": roof["avg_ms"], "peak_source": f"{peak_src} hbm_gbs (copy, burst)"},
        "roofline_sort": main.get("sort_roofline"),
        "dominant_kernel": main["dominant"],
        "kernels": main["kernels"],
        "profile_ms_per_step": {k: round(v[1] / args.steps, 4) for k, v in main["profile"].items()},
        "escaped_per_step": main["escaped_per_step"],
        "tile_load": main["tile_load"],
        "gpu_launches": main["gpu_launches"],
        "clocks": clocks,
    }
    if "e2e" in main:
        line["e2e"] = main["e2e"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if dist.world == 1 and not args.main_only:
        wl = {}
        ks, kw = max(3, args.steps // 10), max(3, args.warmup)
        wl["cic1d"] = cic1d_workload(pcg, 200, 5, dist)
        d2 = synth.cic2d()
        # the committed DRAM counters were taken on the cic3d_drift step: they
        # describe its launches only, so the other workloads report no traffic
        r2 = current_workload(pcg, d2, max(20, args.steps // 2), kw, dist, peaks, {})
        wl["cic2d_512"] = {"workload": "cic2d 512^2 x 8 ppc", "value": round(r2["value"], 1), "unit": UNIT,
                           "ms_per_step": round(r2["ms_per_step"], 4), "kernels": r2["kernels"]}
        del d2
        d4 = synth.quad3d_bump()
        r4 = current_workload(pcg, d4, ks, kw, dist, peaks, {})
        wl["quad3d_bump_192"] = {"workload": "quad3d_bump 192^3, mean 32 ppc, peak 320", "particles": r4["n"],
                                 "value": round(r4["value"], 1), "unit": UNIT,
                                 "ms_per_step": round(r4["ms_per_step"], 4), "kernels": r4["kernels"],
                                 "escaped_per_step": r4["escaped_per_step"], "tile_load": r4["tile_load"],
                                 "stencil_updates_per_s": r4.get("stencil_updates_per_s")}
        del d4
        wl["mass3d_64"] = mass_workload(pcg, ks, kw, dist, peaks, {})
        wl["mass3d_tsc_32"] = tsc_workload(pcg, ks, kw, dist, peaks, {})
        wl["mass3d_tsc_64"] = tsc_workload(pcg, 3, 3, dist, peaks, {}, edge=64)
        d5 = synth.zigzag3d()
        wl["zigzag3d_256"] = zigzag_workload(pcg, d5, ks, kw, dist, peaks, {})
        del d5
        line["workloads"] = wl
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def run_only(args):
    """One secondary workload alone (a profiling aid; not the benchmark line)."""
    import torch
    import particle_cell_grid_gb300 as pcg
    import synth
    dist = Dist(1)
    torch.cuda.set_device(0)
    pcg._lib.load()
    peaks, _ = load_peaks()
    traffic = {}  # the committed DRAM counters describe the cic3d_drift step only
    if args.only == "mass":
        out = mass_workload(pcg, args.steps, args.warmup, dist, peaks, traffic, edge=args.mass_grid)
    elif args.only == "cic1d":
        out = cic1d_workload(pcg, args.steps, args.warmup, dist)
    elif args.only == "tsc":
        out = tsc_workload(pcg, args.steps, args.warmup, dist, peaks, traffic, edge=args.mass_grid)
    elif args.only == "zigzag":
        out = zigzag_workload(pcg, synth.zigzag3d(grid=(args.zz_grid,) * 3), args.steps, args.warmup, dist, peaks,
                              traffic)
    else:
        if args.only == "quad":
            qg = args.quad_grid
            d = synth.quad3d_bump(grid=(qg, qg, qg), sigma_bump=16.0 * qg / 192)
        else:
            d = synth.cic2d()
        out = current_workload(pcg, d, args.steps, args.warmup, dist, peaks, traffic)
        out.pop("profile", None)
    print(json.dumps({"only": args.only, **out}), flush=True)


def run_reference(args):
    """The oracle as it stands on the host cores, on bounded samples of the same workload.

    Each step deposits a sample of consecutive particles of the (randomly
    ordered) workload, split over every usable core: one Python thread per core
    calls the oracle on its part into a private J (ctypes releases the GIL) and
    the parts are summed."""
    dist = Dist(args.gpus)
    if dist.rank != 0:
        return
    import oracle
    import synth
    d = synth.cic3d_drift()
    n = d["n"]
    total = args.steps + args.warmup
    threads, cpu = cpu_threads_for(d)
    s0 = 200_000
    t = time.perf_counter()
    oracle.deposit_current(d["grid"], 1, [p[:s0] for p in d["pos"]], [v[:s0] for v in d["vel"]], d["q"][:s0])
    rate = s0 / (time.perf_counter() - t)
    target_s = 90.0  # seconds for the whole --steps/--warmup run
    s = int(max(20_000 * threads, min(n, rate * threads * target_s / total)))

    def step(k):
        a0 = (k * s) % n
        b0 = min(n, a0 + s)
        bounds = np.linspace(a0, b0, threads + 1).astype(np.int64)
        oracle_on_threads(d, [(int(bounds[i]), int(bounds[i + 1])) for i in range(threads)], threads)
        return b0 - a0

    for k in range(args.warmup):
        step(k)
    t = time.perf_counter()
    done = sum(step(args.warmup + k) for k in range(args.steps))
    dt = time.perf_counter() - t
    value = done / dt / 1e6
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": "cic3d_drift 256^3 x 16 ppc, CIC current deposit", "grid": [256, 256, 256],
                       "particles": n, "sample_per_step": s},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "host_cores": cpu["nproc"], "usable_cores": cpu["usable"], "cpu_model": cpu["model"],
                             "sample": f"{s} consecutive particles per step of the {n}-particle workload "
                                       f"(random order), fp64 C oracle on {threads} threads, one private J each"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--grid", type=int, default=256, help="edge of the headline workload's grid (256 = full size)")
    ap.add_argument("--main-only", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--only", choices=["mass", "quad", "cic2d", "cic1d", "zigzag", "tsc"], default=None,
                    help="time one secondary workload alone and print its figures (for profiling)")
    ap.add_argument("--mass-grid", type=int, default=64, help="edge of the mass-matrix grid")
    ap.add_argument("--zz-grid", type=int, default=256, help="edge of the zigzag grid (--only zigzag)")
    ap.add_argument("--quad-grid", type=int, default=192,
                    help="edge of the quadratic bump grid (--only quad; the bump's width scales with it)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
