"""Benchmark: one step = the whole submanifold-conv hot path on one batch of
seeded synthetic voxels, through the C ABI:
    neighbour-map build (hash, probe, row-order sort, tile masks)
    -> forward, input gradient, weight and bias gradient (three streams after
       the map build, each call with its own conv workspace; --one-stream runs
       them one after the other).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                [--no-graph] [--one-stream] [--no-cpu-baseline]

Prints ONE JSON line (rank 0).  ``value`` = voxels/s over all ranks (each rank
runs its own independent replica of the workload: weak scaling, no data-path
collective).  Per-step device time comes from CUDA events on the launch
stream; L2 is flushed (256 MiB write) between steps, outside the events.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "submanifold conv3d fwd+bwd voxels/s & TFLOP/s (valid pairs), % of GB300 roofline"
DEFAULT_WORKLOAD = "b4_r64_spheres_c64_f16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


# ------------------------------------------------------------------ work model
def pass_work(N, P, cin, cout, s, splits):
    """Algorithmic FLOPs and gathered+written bytes per pass (valid pairs only)."""
    nbr_bytes = 4 * 28 * N  # nbr [N,27] + mask [N]
    w = 27 * cin * cout * s
    return {
        "fwd": (2.0 * P * cin * cout, P * cin * s + N * cout * s + nbr_bytes + w),
        "dgrad": (2.0 * P * cin * cout, P * cout * s + N * cin * s + nbr_bytes + w),
        "wgrad": (2.0 * P * cin * cout, P * cin * s + P * cout * s + 2 * splits * 27 * cin * cout * 4
                  + 27 * cin * cout * s + N * cout * s),
    }


def unique_bytes(N, cin, cout, s):
    """The stricter per-pass byte count: every input and output row once, plus the map
    (nbr + mask) and the weights; a pass that reuses its gathers from L2 can reach it."""
    return N * (cin + cout) * s + 4 * 28 * N + 27 * cin * cout * s


def nbrmap_bytes(N):
    # coords read twice (insert + Morton) + probe: coords + 27 table probes (~12 B) + nbr/mask write
    return 16 * N * 3 + 27 * 12 * N + 4 * 28 * N


# ------------------------------------------------------------------ ncu traffic
def source_digest(kernel: str) -> str:
    import hashlib
    f = {"k_gather_gemm_tc": "conv_tc.cu", "k_wgrad_tc": "wgrad_tc.cu"}[kernel]
    h = hashlib.sha256()
    for name in (f, "tc_ptx.cuh", "common.cuh"):
        h.update(open(os.path.join(ROOT, "voxel_gemm_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu summary
    profiles/traffic.json, or None if absent or taken on a different kernel source."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[workload][kernel]
    except Exception:
        return None
    return rec["dram_bytes_per_launch"] if rec.get("source_digest") == source_digest(kernel) else None


# ------------------------------------------------------------------ ranks
def max_over_ranks(value: float, world: int, device=None) -> float:
    """Slowest rank's value (the timed region ends when every replica is done)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_voxels_per_s(n_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own replica of n_per_rank voxels."""
    return world * n_per_rank / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.devnull if False else os.path.join("/tmp", f"vg_clocks_{os.getpid()}.csv"), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.out.name):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist
    from voxel_gemm_gb300 import ops, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = synth.WORKLOADS[args.workload]
    coords_np = synth.make_coords(wl)
    N = coords_np.shape[0]
    s = 4 if wl.dtype == "f32" else 2
    dt = synth.torch_dtype(wl.dtype)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        coords = torch.from_numpy(coords_np).to(dev)
        f, W, b, dY = synth.make_tensors(wl, N, device=dev)
        m = ops.NbrMap.alloc(N, wl.grid, wl.key_flag, device=dev)
        ws = ops.conv_workspace(N, wl.cin, wl.cout, dt, device=dev)
        out = torch.empty(N, wl.cout, dtype=dt, device=dev)
        dX = torch.empty(N, wl.cin, dtype=dt, device=dev)
        dW = torch.empty(27, wl.cin, wl.cout, dtype=dt, device=dev)
        db = torch.empty(wl.cout, dtype=dt, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    # The three convolution passes depend only on the map and the inputs, so after
    # the map build they run on three streams (each with its own conv workspace);
    # a pass's tail then overlaps the next one's start.  --one-stream issues them
    # one after the other on the timed stream instead.
    one_stream = args.one_stream
    with torch.cuda.stream(stream):
        ws_dx = ops.conv_workspace(N, wl.cin, wl.cout, dt, device=dev)
        ws_dw = ops.conv_workspace(N, wl.cin, wl.cout, dt, device=dev)
    s_dx = torch.cuda.Stream(device=dev)
    s_dw = torch.cuda.Stream(device=dev)

    def step():
        m.build(coords, stream)
        if one_stream:
            ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, stream=stream)
            ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, dW, db, ws, stream=stream)
            return
        s_dx.wait_stream(stream)
        s_dw.wait_stream(stream)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, stream=stream)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, None, None, ws_dx, stream=s_dx)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, None, dW, db, ws_dw, stream=s_dw)
        stream.wait_stream(s_dx)
        stream.wait_stream(s_dw)

    def timed(fn, k, ev_list):
        for _ in range(k):
            with torch.cuda.stream(stream):
                flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ev_list.append((e0, e1))

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    assert m.status(stream) == ops.VG_OK

    def graphed(fn):
        """Capture fn (stream-ordered C-ABI calls on `stream`) once; replay per step."""
        if args.no_graph:
            return fn
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        stream.synchronize()

        def replay():  # replay() launches on the current stream: make it the timed one
            with torch.cuda.stream(stream):
                g.replay()
        return replay

    eager_step = step
    step = graphed(eager_step)
    for _ in range(3):
        step()
    stream.synchronize()
    P = int(torch.stack([(m.mask >> k) & 1 for k in range(27)]).sum().item())

    # ---- timed region: exactly K steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank)
    sampler.start()
    evs = []
    t_wall0 = time.perf_counter()
    timed(step, args.steps, evs)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b_) for a, b_ in evs]
    tot_ms = max_over_ranks(sum(step_ms), world, dev)
    assert m.status(stream) == ops.VG_OK and ops.vg_conv_status(ws, stream) == ops.VG_OK
    if not one_stream:  # the other two workspaces are only used (and their error records set) then
        assert ops.vg_conv_status(ws_dx, stream) == ops.VG_OK and ops.vg_conv_status(ws_dw, stream) == ops.VG_OK
    ms_per_step = tot_ms / args.steps

    # ---- per-pass timings (same stream, same flush rule), for the roofline
    phases = {}
    kph = max(3, min(args.steps, 50))
    calls = {
        "nbrmap": lambda: m.build(coords, stream),
        "fwd": lambda: ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, stream=stream),
        "dgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, None, None, ws,
                                                stream=stream),
        "wgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, None, dW, db, ws,
                                                stream=stream),
    }
    for name, fn in calls.items():
        ev = []
        fn = graphed(fn)
        fn()
        timed(fn, kph, ev)
        torch.cuda.synchronize(dev)
        phases[name] = sum(a.elapsed_time(b_) for a, b_ in ev) / kph

    # ---- end to end through the public API with host buffers (pinned), copies inside the region
    h_coords = torch.from_numpy(coords_np).pin_memory()
    h_f, h_W, h_b, h_dY = (t.to("cpu").pin_memory() for t in (f, W, b, dY))
    h_out = torch.empty(out.shape, dtype=dt).pin_memory()
    h_dX = torch.empty(dX.shape, dtype=dt).pin_memory()
    h_dW = torch.empty(dW.shape, dtype=dt).pin_memory()
    h_db = torch.empty(db.shape, dtype=dt).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_coords, h_f, h_W, h_b, h_dY))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_dX, h_dW, h_db))

    # The copies run on two more streams (host-to-device and device-to-host) where
    # the data dependences allow: features and weights go up while the neighbour
    # map (which needs only the coordinates) is built, dY while the forward runs;
    # `out` comes back during the backward and dX during the weight gradient.  The
    # conv passes use the same streams as the device-only step.
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)

    def e2e_eager():
        ev_fwd_in, ev_bwd_in, ev_fwd, ev_dx = (torch.cuda.Event() for _ in range(4))
        with torch.cuda.stream(stream):
            coords.copy_(h_coords, non_blocking=True)
        up.wait_stream(stream)
        down.wait_stream(stream)
        with torch.cuda.stream(up):
            f.copy_(h_f, non_blocking=True)
            W.copy_(h_W, non_blocking=True)
            b.copy_(h_b, non_blocking=True)
            ev_fwd_in.record(up)
            dY.copy_(h_dY, non_blocking=True)
            ev_bwd_in.record(up)
        m.build(coords, stream)
        dx_stream = stream if one_stream else s_dx
        dw_stream = stream if one_stream else s_dw
        dx_ws = ws if one_stream else ws_dx
        dw_ws = ws if one_stream else ws_dw
        if not one_stream:
            s_dx.wait_stream(stream)
            s_dw.wait_stream(stream)
        stream.wait_event(ev_fwd_in)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, stream=stream)
        ev_fwd.record(stream)
        dx_stream.wait_event(ev_bwd_in)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, None, None, dx_ws, stream=dx_stream)
        ev_dx.record(dx_stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_fwd)
            h_out.copy_(out, non_blocking=True)
            down.wait_event(ev_dx)
            h_dX.copy_(dX, non_blocking=True)
        dw_stream.wait_event(ev_bwd_in)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, None, dW, db, dw_ws, stream=dw_stream)
        with torch.cuda.stream(dw_stream):
            h_dW.copy_(dW, non_blocking=True)
            h_db.copy_(db, non_blocking=True)
        for st in (up, down) if one_stream else (up, down, s_dx, s_dw):
            stream.wait_stream(st)

    e2e_step = graphed(e2e_eager)

    ke = max(3, min(args.steps, 100))
    for _ in range(2):
        e2e_step()
    stream.synchronize()
    ev = []
    timed(e2e_step, ke, ev)
    stream.synchronize()
    e2e_ms = sum(a.elapsed_time(b_) for a, b_ in ev) / ke

    # ---- roofline of the dominant kernel pass
    peaks = load_peaks()
    cplan = ops.vg_conv_describe(N, wl.cin, wl.cout, dt)
    nplan = ops.vg_nbrmap_describe(N, *wl.grid, wl.key_flag)
    splits = cplan["splits"]
    work = pass_work(N, P, wl.cin, wl.cout, s, splits)
    work["nbrmap"] = (0.0, float(nbrmap_bytes(N)))
    tc_peak = peaks["bf16_tflops"] * 1e12
    bw = peaks["hbm_gbs"] * 1e9
    rows = {}
    for name, (fl, by) in work.items():
        t = phases[name] * 1e-3
        bound = "tensor" if fl / tc_peak > by / bw else "hbm"
        if wl.dtype == "f32" and name != "nbrmap":
            bound = "hbm" if fl / tc_peak <= by / bw else "alu"
        rows[name] = {"ms": phases[name], "flops": fl, "bytes": by, "bound": bound,
                      "tflops": fl / t / 1e12, "gbs": by / t / 1e9,
                      "frac": (by / bw) / t if bound == "hbm" else (fl / tc_peak) / t}
        if name != "nbrmap":  # the same pass against the unique-byte roofline
            ub = unique_bytes(N, wl.cin, wl.cout, s)
            rows[name]["unique_bytes"] = ub
            rows[name]["frac_unique_roofline"] = max(fl / tc_peak, ub / bw) / t
    # dominant kernel: the slowest convolution pass (each pass is one GEMM kernel plus a
    # small weight repack / reduce); the map build is a chain of small kernels, reported in "passes"
    dom = max(("fwd", "dgrad", "wgrad"), key=lambda k: phases[k])
    d = rows[dom]
    kern = "k_wgrad_tc" if dom == "wgrad" else "k_gather_gemm_tc"
    roof = {"kernel": f"{kern} ({dom} pass)", "bound": d["bound"],
            "achieved": d["gbs"] if d["bound"] == "hbm" else d["tflops"],
            "peak": peaks["hbm_gbs"] if d["bound"] == "hbm" else peaks["bf16_tflops"],
            "unit": "GB/s" if d["bound"] == "hbm" else "TFLOP/s",
            "traffic": measured_traffic(wl.name, kern), "peak_source": peaks["source"] + " (burst)",
            "duration": "CUDA events around the whole pass call (repack + GEMM + reduce), an upper bound"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor":  # the same rate against the sustained (power-capped) matmul figure
        roof["frac_vs_sustained"] = roof["achieved"] / peaks["bf16_tflops_sustained"]
    t_roof = sum(max(fl / tc_peak, by / bw) for fl, by in work.values())
    total_fl = sum(fl for fl, _ in work.values())
    res = {
        "metric": METRIC, "value": aggregate_voxels_per_s(N, world, ms_per_step), "unit": "voxels/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "res": wl.res, "N": N, "P": P, "cin": wl.cin,
                   "cout": wl.cout, "step": "nbrmap build + fwd + dgrad + wgrad + dbias",
                   "l2": "flushed between steps (256 MiB write, outside the per-step events)",
                   "parallelism": f"replicas x{world}",
                   "launch": ("eager" if args.no_graph else "CUDA graph replay of the step's C-ABI calls")
                   + ("" if one_stream else "; fwd, dgrad and wgrad+db on three streams after the map build")},
        "tflops": world * total_fl / (ms_per_step * 1e-3) / 1e12,
        "roofline_step_frac": t_roof / (ms_per_step * 1e-3),
        "roofline": roof,
        "passes": rows,
        "e2e": {"value": world * N / (e2e_ms * 1e-3), "unit": "voxels/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * (nplan["launches"] + cplan["launches_fwd"] + cplan["launches_bwd"]),
        "gpu_launches_per_step": {"nbrmap": nplan["launches"], "fwd": cplan["launches_fwd"],
                                  "bwd": cplan["launches_bwd"]},
        "path": {"tensor_core": bool(cplan["tensor_core"]), "wgrad_splits": splits,
                 "hash_keys": 64 if nplan["key64"] else 32, "sort_passes": nplan["sort_passes"]},
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    return res


# ------------------------------------------------------------------ oracle arm (CPU)
def oracle_sample(wl, coords_np, budget_rows, seed=0, min_seconds=5.0):
    """Time the oracle on a bounded sample of the workload: the full neighbour map
    (scaled per voxel) and fwd + dgrad + wgrad over sampled rows, repeated over
    fresh row samples until at least `min_seconds` of conv work has run."""
    import numpy as np
    import oracle
    N = coords_np.shape[0]
    t0 = time.perf_counter()
    nbr, mask = oracle.nbrmap(coords_np, *wl.grid)
    t_map = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    R = min(N, budget_rows)
    rows_done, t_conv = 0, 0.0
    while t_conv < min_seconds or rows_done == 0:
        rows = np.sort(rng.choice(N, size=R, replace=False))
        sub = nbr[rows]
        valid = sub != oracle.NONE
        used = np.unique(sub[valid]).astype(np.int64)
        remap = np.full(sub.shape, oracle.NONE, dtype=np.uint32)
        remap[valid] = np.searchsorted(used, sub[valid].astype(np.int64)).astype(np.uint32)
        f = rng.standard_normal((used.size, wl.cin))
        W = rng.standard_normal((27, wl.cin, wl.cout)) * 0.05
        b = rng.standard_normal(wl.cout)
        g_used = rng.standard_normal((used.size, wl.cout))
        g_rows = rng.standard_normal((R, wl.cout))
        t1 = time.perf_counter()
        oracle.fwd(remap, f, W, b)
        oracle.dgrad_rows(remap, g_used, W)
        oracle.wgrad(remap, f, g_rows)
        t_conv += time.perf_counter() - t1
        rows_done += R
    per_voxel = t_map / N + t_conv / rows_done
    return 1.0 / per_voxel, {"rows": rows_done, "t_map_s": t_map, "t_conv_s": t_conv}


def run_reference(args):
    from voxel_gemm_gb300 import synth
    import oracle
    wl = synth.WORKLOADS[args.workload]
    coords_np = synth.make_coords(wl)
    budget = rows_budget(wl)
    for _ in range(args.warmup):
        oracle_sample(wl, coords_np, max(64, budget // 8), min_seconds=0.0)
    vals = []
    t0 = time.perf_counter()
    for k in range(args.steps):
        v, _ = oracle_sample(wl, coords_np, budget, seed=k, min_seconds=2.0)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    cores = oracle.num_threads()
    sample = (f"full neighbour map of N={coords_np.shape[0]} voxels, then fwd+dgrad+wgrad over "
              f"{min(budget, coords_np.shape[0])} seeded sampled rows per step; voxels/s = 1 / (map time per "
              f"voxel + conv time per sampled row)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "voxels/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "res": wl.res, "N": int(coords_np.shape[0]),
                       "cin": wl.cin, "cout": wl.cout},
            "cpu_baseline": {"value": value, "unit": "voxels/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def rows_budget(wl):
    # about 2-4 s of fp64 work per sample on a many-core host
    per_row = 3 * 10.6 * wl.cin * wl.cout
    return int(max(256, min(65536, 4e9 / per_row)))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each call eagerly instead of replaying a CUDA graph")
    ap.add_argument("--one-stream", action="store_true",
                    help="issue the step's conv passes one after the other on one stream")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            from voxel_gemm_gb300 import synth
            import oracle
            wl = synth.WORKLOADS[args.workload]
            coords_np = synth.make_coords(wl)
            v, info = oracle_sample(wl, coords_np, rows_budget(wl))
            res["cpu_baseline"] = {"value": v, "unit": "voxels/s", "cores": oracle.num_threads(),
                                   "kind": "oracle",
                                   "sample": f"full map of N={coords_np.shape[0]}, fwd+dgrad+wgrad over "
                                             f"{info['rows']} sampled rows ({info['t_map_s']:.2f}s map, "
                                             f"{info['t_conv_s']:.2f}s conv)"}
            # the same oracle on one host core, over a smaller row sample (about 3 s)
            cores = oracle.num_threads()
            oracle.set_num_threads(1)
            try:
                v1, info1 = oracle_sample(wl, coords_np, max(64, rows_budget(wl) // 8), min_seconds=3.0)
            finally:
                oracle.set_num_threads(cores)
            res["cpu_baseline"]["value_1core"] = v1
            res["cpu_baseline"]["sample_1core"] = f"{info1['rows']} sampled rows ({info1['t_conv_s']:.2f}s conv)"
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
