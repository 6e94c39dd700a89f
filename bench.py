"""Benchmark: one step = the whole submanifold-conv hot path on one batch of
seeded synthetic voxels, through the C ABI:
    neighbour-map build (column index or hash table, probe, row-order sort, tile masks)
    -> forward, input gradient, weight and bias gradient (three streams after
       the map build, each call with its own conv workspace; --one-stream runs
       them one after the other)
    -> with N > 1 ranks: the weight and bias gradients of all ranks summed in
       rank order (the data-parallel exchange step; every rank ends with the
       same bits).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                [--no-graph] [--one-stream] [--no-cpu-baseline] [--no-sweep]
python bench.py --ncu-step [--tf32] [--workload NAME] [--warmup W]   (a command for profilers)

Prints ONE JSON line (rank 0).  The headline workload (default: batch 1, 512^3
grid, Cin = Cout = 1024, bf16) gets the full record: step time, per-pass
roofline, end-to-end time with host buffers, clocks, CPU oracle baseline.
``sweep`` holds one shorter record per other workload (ms/step, per-pass ms
and roofline fractions).  ``value`` = voxels/s over all ranks: each rank runs
its own batch element(s) of the same shape (weak scaling, weights
replicated, gradients summed across ranks).  Per-step device time comes from
CUDA events on the launch stream; L2 is flushed (256 MiB write) between
steps, outside the events.
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
DEFAULT_WORKLOAD = "b1_r512_shapes_c1024_bf16"
SWEEP = ["b4_r64_spheres_c64_f16", "b2_r256_shapes_c128_bf16", "b1_r512_shapes_c256_bf16",
         "b1_r512_shapes_c512_bf16", "b1_r1024_shapes_c64_f16"]
INFER_WORKLOAD = "b1_r64_spheres_c256_bf16_infer"
REGULAR_WORKLOAD = "b1_r512_shapes_c256_bf16"
ORDER_WORKLOADS = ["b2_r256_shapes_c128_bf16", "b1_r512_shapes_c256_bf16", "b1_r1024_shapes_c64_f16"]
STEP = "nbrmap build + fwd + dgrad + wgrad + dbias"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 << 20


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
    """Algorithmic FLOPs and gathered+written bytes per pass (valid pairs only).
    The weight gradient's bytes include its split-K partial sums (written once,
    read once by the reduce); ``splitk_bytes`` gives that share separately."""
    nbr_bytes = 4 * 28 * N  # nbr [N,27] + mask [N]
    w = 27 * cin * cout * s
    return {
        "fwd": (2.0 * P * cin * cout, P * cin * s + N * cout * s + nbr_bytes + w),
        "dgrad": (2.0 * P * cin * cout, P * cout * s + N * cin * s + nbr_bytes + w),
        "wgrad": (2.0 * P * cin * cout, P * cin * s + P * cout * s + splitk_bytes(cin, cout, splits)
                  + 27 * cin * cout * s + N * cout * s),
    }


def splitk_bytes(cin, cout, splits):
    return 2 * splits * 27 * cin * cout * 4


def unique_bytes(N, cin, cout, s):
    """The stricter per-pass byte count: every input and output row once, plus the map
    (nbr + mask) and the weights; a pass that reuses its gathers from L2 can reach it."""
    return N * (cin + cout) * s + 4 * 28 * N + 27 * cin * cout * s


def nbrmap_bytes(N):
    # coords read twice (insert + Morton) + probe: coords + 27 table probes (~12 B) + nbr/mask write
    return 16 * N * 3 + 27 * 12 * N + 4 * 28 * N


def count_pairs(mask_u32) -> int:
    """P = number of valid (voxel, tap) pairs = total popcount of the tap masks."""
    import numpy as np
    m = np.asarray(mask_u32, dtype=np.uint32)
    return int(sum(int(((m >> k) & 1).sum()) for k in range(27)))


def workload_config(wl, N, P, world):
    """The workload description both arms print (identical dicts)."""
    s = 4 if wl.dtype == "f32" else 2
    in_bytes = N * (wl.cin + wl.cout) * s
    l2 = ("flushed between steps (256 MiB write, outside the per-step events); inputs "
          + ("larger than L2" if in_bytes > L2_BYTES else "smaller than L2")
          + f" ({in_bytes / 1e6:.1f} MB of features + grad_out)")
    return {"workload": wl.name, "B": wl.B, "res": wl.res, "N": int(N), "P": int(P), "cin": wl.cin,
            "cout": wl.cout, "dtype": wl.dtype, "global_batch": wl.B * world, "step": STEP, "l2": l2,
            "parallelism": "single GPU" if world == 1 else f"data-parallel x{world} (batch-sharded, "
                           "weights replicated, rank-ordered gradient sum)"}


# ------------------------------------------------------------------ ncu traffic
def source_digest(kernel: str) -> str:
    import hashlib
    f = {"k_gather_gemm_tc": "conv_tc.cu", "k_gather_gemm_pair": "conv_tc.cu", "k_wgrad_tc": "wgrad_tc.cu"}[kernel]
    h = hashlib.sha256()
    for name in (f, "tc_ptx.cuh", "common.cuh"):
        h.update(open(os.path.join(ROOT, "voxel_gemm_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def gather_kernel(n: int, cin: int, cout: int, sms: int) -> str:
    """The gather-GEMM kernel the library runs for the forward and input-gradient
    passes: k_gather_gemm_pair when both output widths are multiples of 256 and the
    pairs of 128-row tiles times the 256-column blocks give every SM a unit."""
    pairs = ((n + 127) // 128 + 1) // 2
    if all(c % 256 == 0 and pairs * (c // 256) >= sms for c in (cin, cout)):
        return "k_gather_gemm_pair"
    return "k_gather_gemm_tc"


def sms_of(dev) -> int:
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count


def measured_traffic(workload: str, kernel: str, P: int):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the committed
    ncu summary profiles/traffic.json (captured on a smaller case of the same kernel and
    channel count, scaled by valid pairs), or None if absent or taken on other sources."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["kernels"][workload][kernel]
    except Exception:
        return None
    if rec.get("source_digest") != source_digest(kernel):
        return None
    return rec["dram_bytes_per_pair"] * P


# ------------------------------------------------------------------ ranks
def max_over_ranks(value: float, world: int, device=None) -> float:
    """Slowest rank's value (the timed region ends when every rank is done)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_voxels_per_s(n_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch element(s) of n_per_rank voxels."""
    return world * n_per_rank / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"vg_clocks_{os.getpid()}_{gpu_index}.csv")
        self.mark = 0

    def start(self, wait_s=3.0):
        """Start nvidia-smi sampling every 100 ms and return once it has written a sample."""
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < wait_s and os.path.getsize(self.path) == 0:
            time.sleep(0.05)

    def begin_region(self):
        if self.proc is None:
            return
        self.out.flush()
        self.mark = os.path.getsize(self.path)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)  # let the sample that covers the end of the region land
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.path) as fh:
            fh.seek(self.mark)
            lines = fh.read().splitlines()
        os.unlink(self.path)
        rows = [[p.strip() for p in ln.split(",")] for ln in lines]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        num = lambda v: v.replace(".", "").isdigit()  # noqa: E731
        sm = [float(r[1]) for r in rows if num(r[1])]
        mx = [float(r[2]) for r in rows if num(r[2])]
        pw = [float(r[3]) for r in rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm
class Problem:
    """Device buffers of one workload on one rank (inputs, map, workspaces, outputs)."""

    def __init__(self, wl, rank, dev, stream):
        import torch
        from voxel_gemm_gb300 import ops, synth, shard
        self.wl = wl
        self.dev = dev
        self.stream = stream
        self.coords_np = shard.rank_coords(wl, rank)
        N = self.N = self.coords_np.shape[0]
        self.s = 4 if wl.dtype == "f32" else 2
        dt = self.dt = synth.torch_dtype(wl.dtype)
        with torch.cuda.stream(stream):
            self.coords = torch.from_numpy(self.coords_np).to(dev)
            self.f, self.W, self.b, self.dY = synth.make_tensors(wl, N, device=dev)
            if rank > 0:  # every rank's batch element has its own features; weights are replicated
                g = torch.Generator(device=dev)
                g.manual_seed(7919 * rank + wl.seed)
                self.f = torch.randn(N, wl.cin, generator=g, device=dev).to(dt)
                self.dY = torch.randn(N, wl.cout, generator=g, device=dev).to(dt)
            self.m = ops.NbrMap.alloc(N, wl.grid, wl.key_flag, device=dev)
            self.ws = [ops.conv_workspace(N, wl.cin, wl.cout, dt, device=dev) for _ in range(3)]
            self.out = torch.empty(N, wl.cout, dtype=dt, device=dev)
            self.dX = torch.empty(N, wl.cin, dtype=dt, device=dev)
            self.dW = torch.empty(27, wl.cin, wl.cout, dtype=dt, device=dev)
            self.db = torch.empty(wl.cout, dtype=dt, device=dev)
        self.s_dx = torch.cuda.Stream(device=dev)
        self.s_dw = torch.cuda.Stream(device=dev)


def run_workload(args, wl, rank, world, dev, flush, full):
    """Time K steps of workload `wl`; `full` adds the end-to-end and roofline records."""
    import torch
    from voxel_gemm_gb300 import ops, shard

    stream = torch.cuda.Stream(device=dev)
    pb = Problem(wl, rank, dev, stream)
    m, N = pb.m, pb.N
    one_stream = args.one_stream
    reducer = shard.GradientSum(world, pb.dW, pb.db, dev) if world > 1 else None

    def step():
        m.build(pb.coords, stream)
        if one_stream:
            ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, pb.f, pb.W, pb.b, pb.out, pb.ws[0], stream=stream)
            ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, pb.dX, pb.dW, pb.db, pb.ws[0],
                                   stream=stream)
        else:
            # the three passes depend only on the map and the inputs: after the map build
            # they run on three streams (each with its own conv workspace)
            pb.s_dx.wait_stream(stream)
            pb.s_dw.wait_stream(stream)
            ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, pb.f, pb.W, pb.b, pb.out, pb.ws[0], stream=stream)
            ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, pb.dX, None, None, pb.ws[1],
                                   stream=pb.s_dx)
            ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, None, pb.dW, pb.db, pb.ws[2],
                                   stream=pb.s_dw)
            stream.wait_stream(pb.s_dx)
            stream.wait_stream(pb.s_dw)
        if reducer is not None:  # data-parallel exchange: rank-ordered sum of dW and db
            reducer(stream)

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

    warmup = args.warmup if full else 3
    steps = args.steps if full else max(3, min(args.steps, 10))
    for _ in range(warmup):
        step()
    stream.synchronize()
    assert m.status(stream) == ops.VG_OK

    use_graph = not args.no_graph and world == 1  # collectives stay eager

    def graphed(fn):
        """Capture fn (stream-ordered C-ABI calls on `stream`) once; replay per step."""
        if not use_graph:
            return fn
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        stream.synchronize()

        def replay():  # replay() launches on the current stream: make it the timed one
            with torch.cuda.stream(stream):
                g.replay()
        return replay

    gstep = graphed(step)
    for _ in range(3):
        gstep()
    stream.synchronize()
    P = count_pairs(m.mask.cpu().numpy().view("uint32"))

    # ---- timed region: exactly K steps
    sampler = ClockSampler(dev.index) if full else None
    if sampler:
        sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.begin_region()
    evs = []
    t_wall0 = time.perf_counter()
    timed(gstep, steps, evs)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    tot_ms = max_over_ranks(sum(a.elapsed_time(b_) for a, b_ in evs), world, dev)
    assert m.status(stream) == ops.VG_OK
    for w_ in pb.ws:
        assert ops.vg_conv_status(w_, stream) == ops.VG_OK
    ms_per_step = tot_ms / steps

    # ---- per-pass timings (same stream, same flush rule), for the roofline
    phases = {}
    kph = max(3, min(steps, 20))
    calls = {
        "nbrmap": lambda: m.build(pb.coords, stream),
        "fwd": lambda: ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, pb.f, pb.W, pb.b, pb.out, pb.ws[0],
                                              stream=stream),
        "dgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, pb.dX, None, None,
                                                pb.ws[0], stream=stream),
        "wgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, None, pb.dW, pb.db,
                                                pb.ws[0], stream=stream),
    }
    for name, fn in calls.items():
        ev = []
        fn = graphed(fn)
        fn()
        timed(fn, kph, ev)
        torch.cuda.synchronize(dev)
        phases[name] = sum(a.elapsed_time(b_) for a, b_ in ev) / kph

    # ---- roofline per pass and of the dominant pass
    peaks = load_peaks()
    cplan = ops.vg_conv_describe(N, wl.cin, wl.cout, pb.dt)
    nplan = ops.vg_nbrmap_describe(N, *wl.grid, wl.key_flag)
    splits = cplan["splits"]
    work = pass_work(N, P, wl.cin, wl.cout, pb.s, splits)
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
            ub = unique_bytes(N, wl.cin, wl.cout, pb.s)
            rows[name]["unique_bytes"] = ub
            rows[name]["frac_unique_roofline"] = max(fl / tc_peak, ub / bw) / t
    sk = splitk_bytes(wl.cin, wl.cout, splits)
    rows["wgrad"]["splitk_bytes"] = sk
    if rows["wgrad"]["bound"] == "hbm":  # the same pass without the library's own split-K traffic
        rows["wgrad"]["frac_excl_splitk"] = ((work["wgrad"][1] - sk) / bw) / (phases["wgrad"] * 1e-3)
    # the dominant kernel: the one with the most device time per step (the gather GEMM
    # runs twice, forward and input gradient)
    # (at 256-column output blocks, with at least as many pairs of row tiles as SMs, the
    # gather GEMM runs as k_gather_gemm_pair: two tiles per unit sharing each weight tile)
    gk = gather_kernel(N, wl.cin, wl.cout, sms_of(dev))
    kernel_passes = {gk: ("fwd", "dgrad"), "k_wgrad_tc": ("wgrad",), "nbrmap": ("nbrmap",)}
    dom = max(kernel_passes, key=lambda k: sum(phases[q] for q in kernel_passes[k]))
    t_roof = sum(max(fl / tc_peak, by / bw) for fl, by in work.values())
    total_fl = sum(fl for fl, _ in work.values())
    tflops = world * total_fl / (ms_per_step * 1e-3) / 1e12
    rec = {"workload": wl.name, "N": N, "P": P, "ms_per_step": ms_per_step, "steps": steps,
           "value": aggregate_voxels_per_s(N, world, ms_per_step), "unit": "voxels/s", "tflops": tflops,
           "tflops_frac_of_bf16_peak": tflops / world / peaks["bf16_tflops"],
           "roofline_step_frac": t_roof / (ms_per_step * 1e-3), "dominant_kernel": dom,
           "passes": rows}
    if not full:
        return rec

    dps = kernel_passes[dom]
    fl_l = sum(work[q][0] for q in dps) / len(dps)  # per launch
    by_l = sum(work[q][1] for q in dps) / len(dps)
    t_l = sum(phases[q] for q in dps) / len(dps) * 1e-3  # mean launch duration
    bound = rows[dps[0]]["bound"]
    kname = {"nbrmap": "neighbour-map build (all its kernels)", gk: gk, "k_wgrad_tc": "k_wgrad_tc"}[dom]
    roof = {"kernel": f"{kname} ({' + '.join(dps)} pass{'es' if len(dps) > 1 else ''}, "
                      f"{sum(phases[q] for q in dps):.3f} ms per step)", "bound": bound,
            "achieved": by_l / t_l / 1e9 if bound == "hbm" else fl_l / t_l / 1e12,
            "peak": peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops"],
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "traffic": measured_traffic(wl.name, dom, P) if dom != "nbrmap" else None,
            "peak_source": peaks["source"] + " (burst)",
            "duration": "mean over the kernel's launches per step of the CUDA-event time of the whole pass "
                        "call (weight repack or split reduce included), an upper bound on the kernel's own time"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor":  # the same rate against the sustained (power-capped) matmul figure
        roof["frac_vs_sustained"] = roof["achieved"] / peaks["bf16_tflops_sustained"]
    if dom == "k_wgrad_tc" and "frac_excl_splitk" in rows["wgrad"]:
        roof["frac_excl_splitk"] = rows["wgrad"]["frac_excl_splitk"]

    # ---- end to end through the public API with host buffers (pinned), copies inside the region
    h_coords = torch.from_numpy(pb.coords_np).pin_memory()
    h_f, h_W, h_b, h_dY = (t.to("cpu").pin_memory() for t in (pb.f, pb.W, pb.b, pb.dY))
    h_out = torch.empty(pb.out.shape, dtype=pb.dt).pin_memory()
    h_dX = torch.empty(pb.dX.shape, dtype=pb.dt).pin_memory()
    h_dW = torch.empty(pb.dW.shape, dtype=pb.dt).pin_memory()
    h_db = torch.empty(pb.db.shape, dtype=pb.dt).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_coords, h_f, h_W, h_b, h_dY))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_dX, h_dW, h_db))
    # Copies run on two more streams where the data dependences allow.  Uploads go in
    # the order the passes can start: the coordinates (the map build needs nothing
    # else), the weights and bias, dY (the input gradient needs only dY and W), then
    # the features (the forward and the weight gradient need them).  Each result
    # comes back as soon as its pass ends: dX during the forward, out during the
    # weight gradient, dW and db last (57 MB at C = 1024, where dX and out are 1.2 GB
    # each).  The conv passes use the same streams as the device-only step.
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)

    def e2e_eager():
        ev_dy_in, ev_f_in, ev_fwd, ev_dx = (torch.cuda.Event() for _ in range(4))
        with torch.cuda.stream(stream):
            pb.coords.copy_(h_coords, non_blocking=True)
        up.wait_stream(stream)
        down.wait_stream(stream)
        with torch.cuda.stream(up):
            pb.W.copy_(h_W, non_blocking=True)
            pb.b.copy_(h_b, non_blocking=True)
            pb.dY.copy_(h_dY, non_blocking=True)
            ev_dy_in.record(up)
            pb.f.copy_(h_f, non_blocking=True)
            ev_f_in.record(up)
        m.build(pb.coords, stream)
        dx_stream = stream if one_stream else pb.s_dx
        dw_stream = stream if one_stream else pb.s_dw
        dx_ws, dw_ws = (pb.ws[0], pb.ws[0]) if one_stream else (pb.ws[1], pb.ws[2])
        if not one_stream:
            pb.s_dx.wait_stream(stream)
            pb.s_dw.wait_stream(stream)
        dx_stream.wait_event(ev_dy_in)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, pb.dX, None, None, dx_ws,
                               stream=dx_stream)
        ev_dx.record(dx_stream)
        stream.wait_event(ev_f_in)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, pb.f, pb.W, pb.b, pb.out, pb.ws[0], stream=stream)
        ev_fwd.record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_dx)
            h_dX.copy_(pb.dX, non_blocking=True)
            down.wait_event(ev_fwd)
            h_out.copy_(pb.out, non_blocking=True)
        dw_stream.wait_event(ev_fwd)  # after the forward, so that `out` comes back during it
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, pb.dY, pb.f, pb.W, None, pb.dW, pb.db, dw_ws,
                               stream=dw_stream)
        for st in (up, down) if one_stream else (up, down, pb.s_dx, pb.s_dw):
            stream.wait_stream(st)
        if reducer is not None:
            reducer(stream)
        with torch.cuda.stream(stream):
            h_dW.copy_(pb.dW, non_blocking=True)
            h_db.copy_(pb.db, non_blocking=True)

    e2e_step = graphed(e2e_eager)
    ke = max(3, min(args.steps, 100))
    for _ in range(2):
        e2e_step()
    stream.synchronize()
    ev = []
    timed(e2e_step, ke, ev)
    stream.synchronize()
    e2e_single_ms = max_over_ranks(sum(a.elapsed_time(b_) for a, b_ in ev) / ke, world, dev)

    # ---- end to end, pipelined as a training loop with input prefetch runs it: two
    # device slots (inputs, map, workspaces, outputs); step i's uploads go to slot i % 2
    # while step i - 1 computes, and step i's results come back while step i + 1
    # computes.  Every step still copies all of its inputs in and all of its results
    # out inside the timed region (K steps between one pair of events; the inputs are
    # larger than L2, so no flush between steps).
    pbs = [pb, Problem(wl, rank, dev, stream)]
    pbs[1].m.build(pbs[1].coords, stream)
    red2 = [reducer, shard.GradientSum(world, pbs[1].dW, pbs[1].db, dev) if world > 1 else None]
    stream.synchronize()

    def e2e_pipelined(k):
        done_compute, done_down = [None] * k, [None] * k
        for i in range(k):
            q = pbs[i % 2]
            mq = q.m
            ev_c, ev_dy, ev_f, ev_fwd, ev_dx, ev_end = (torch.cuda.Event() for _ in range(6))
            if i >= 2:  # the slot's previous step has read its inputs
                up.wait_event(done_compute[i - 2])
            with torch.cuda.stream(up):
                q.coords.copy_(h_coords, non_blocking=True)
                ev_c.record(up)
                q.W.copy_(h_W, non_blocking=True)
                q.b.copy_(h_b, non_blocking=True)
                q.dY.copy_(h_dY, non_blocking=True)
                ev_dy.record(up)
                q.f.copy_(h_f, non_blocking=True)
                ev_f.record(up)
            stream.wait_event(ev_c)
            if i >= 2:  # and its results have been copied out
                stream.wait_event(done_down[i - 2])
            mq.build(q.coords, stream)
            dxs = stream if one_stream else q.s_dx
            dws = stream if one_stream else q.s_dw
            dx_ws, dw_ws = (q.ws[0], q.ws[0]) if one_stream else (q.ws[1], q.ws[2])
            if not one_stream:
                q.s_dx.wait_stream(stream)
                q.s_dw.wait_stream(stream)
            dxs.wait_event(ev_dy)
            ops.vg_subm_conv3d_bwd(mq.ws, mq.nbr, mq.mask, q.dY, q.f, q.W, q.dX, None, None, dx_ws, stream=dxs)
            ev_dx.record(dxs)
            stream.wait_event(ev_f)
            ops.vg_subm_conv3d_fwd(mq.ws, mq.nbr, mq.mask, q.f, q.W, q.b, q.out, q.ws[0], stream=stream)
            ev_fwd.record(stream)
            dws.wait_event(ev_fwd)
            ops.vg_subm_conv3d_bwd(mq.ws, mq.nbr, mq.mask, q.dY, q.f, q.W, None, q.dW, q.db, dw_ws, stream=dws)
            if not one_stream:
                stream.wait_stream(q.s_dx)
                stream.wait_stream(q.s_dw)
            if red2[i % 2] is not None:
                red2[i % 2](stream)
            ev_end.record(stream)
            done_compute[i] = ev_end
            with torch.cuda.stream(down):
                down.wait_event(ev_dx)
                h_dX.copy_(q.dX, non_blocking=True)
                down.wait_event(ev_fwd)
                h_out.copy_(q.out, non_blocking=True)
                down.wait_event(ev_end)
                h_dW.copy_(q.dW, non_blocking=True)
                h_db.copy_(q.db, non_blocking=True)
                done_down[i] = torch.cuda.Event()
                done_down[i].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    e2e_pipelined(2)
    stream.synchronize()
    kp = max(4, min(args.steps, 100))
    up.wait_stream(stream)
    down.wait_stream(stream)
    e2e_sampler = ClockSampler(dev.index)  # the clocks while copies and compute overlap
    e2e_sampler.start()
    e2e_sampler.begin_region()
    e0p, e1p = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0p.record(stream)
    up.wait_stream(stream)
    e2e_pipelined(kp)
    e1p.record(stream)
    stream.synchronize()
    e2e_clocks = e2e_sampler.stop()
    e2e_ms = max_over_ranks(e0p.elapsed_time(e1p) / kp, world, dev)
    del pbs, red2

    nb_launch = nplan["launches"] + cplan["launches_fwd"] + cplan["launches_bwd"]
    rec.update({
        "roofline": roof, "clocks": clocks, "wall_s_timed_region": t_wall,
        "e2e": {"value": world * N / (e2e_ms * 1e-3), "unit": "voxels/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": kp, "schedule": "pipelined: step i's uploads while step i-1 computes, its downloads "
                                         "while step i+1 computes (two device slots; K steps between one "
                                         "pair of events)",
                "clocks": e2e_clocks,
                "single_step": {"value": world * N / (e2e_single_ms * 1e-3), "ms_per_step": e2e_single_ms,
                                "schedule": "one step at a time: uploads, passes and downloads overlapped "
                                            "within the step only (CUDA-graph replay, L2 flushed between steps)"}},
        "gpu_launches": steps * (nb_launch + (reducer.launches if reducer else 0)),
        "gpu_launches_per_step": {"nbrmap": nplan["launches"], "fwd": cplan["launches_fwd"],
                                  "bwd": cplan["launches_bwd"],
                                  "gradient_sum": reducer.launches if reducer else 0},
        "path": {"tensor_core": bool(cplan["tensor_core"]), "wgrad_splits": splits,
                 "map_index": nplan["index"],
                 "hash_keys": (64 if nplan["key64"] else 32) if nplan["index"] == "hash" else None,
                 "sort_passes": nplan["sort_passes"]},
        "launch": ("eager" if not use_graph else "CUDA graph replay of the step's C-ABI calls")
                  + ("" if one_stream else "; fwd, dgrad and wgrad+db on three streams after the map build"),
    })
    return rec


def run_inference(args, wl, dev, flush):
    """The small-N inference forward (few voxels, forward only): CUDA-event time of the
    forward call with the default plan (taps cut into groups when the (tile, channel
    block) units do not fill the SMs) and with VG_NO_SMALL_N_SPLIT, same inputs."""
    import torch
    from voxel_gemm_gb300 import ops, synth
    stream = torch.cuda.Stream(device=dev)
    coords_np = synth.make_coords(wl)
    N = coords_np.shape[0]
    dt = synth.torch_dtype(wl.dtype)
    s = 4 if wl.dtype == "f32" else 2
    with torch.cuda.stream(stream):
        coords = torch.from_numpy(coords_np).to(dev)
        f, W, b, _ = synth.make_tensors(wl, N, device=dev)
        m = ops.NbrMap.alloc(N, wl.grid, wl.key_flag, device=dev)
        out = torch.empty(N, wl.cout, dtype=dt, device=dev)
    m.build(coords, stream)
    assert m.status(stream) == ops.VG_OK
    P = count_pairs(m.mask.cpu().numpy().view("uint32"))
    rec = {"workload": wl.name, "N": N, "P": P, "pass": "fwd"}
    peaks = load_peaks()
    for tag, flags in (("split", 0), ("unsplit", ops.VG_NO_SMALL_N_SPLIT)):
        with torch.cuda.stream(stream):
            ws = ops.conv_workspace(N, wl.cin, wl.cout, dt, device=dev, flags=flags)
        call = lambda: ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, flags=flags,  # noqa: E731
                                              stream=stream)
        for _ in range(3):
            call()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        ts = []
        for _ in range(max(5, min(args.steps, 50))):
            with torch.cuda.stream(stream):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
            ts.append((e0, e1))
        stream.synchronize()
        assert ops.vg_conv_status(ws, stream) == ops.VG_OK
        ms = sum(a.elapsed_time(b_) for a, b_ in ts) / len(ts)
        plan = ops.vg_conv_describe(N, wl.cin, wl.cout, dt, flags)
        fl, by = pass_work(N, P, wl.cin, wl.cout, s, 1)["fwd"]
        rec[tag] = {"ms": ms, "launches": plan["launches_fwd"], "tflops": fl / (ms * 1e-3) / 1e12,
                    "frac_of_roofline": max(fl / (peaks["bf16_tflops"] * 1e12), by / (peaks["hbm_gbs"] * 1e9))
                    / (ms * 1e-3)}
    rec["speedup_split"] = rec["unsplit"]["ms"] / rec["split"]["ms"]
    return rec


def run_tf32(args, base, dev, flush):
    """fp32 features on a workload's voxels (Cin = Cout = 256): the three passes with
    VG_ALLOW_TF32 (tensor cores, TF32 inputs, fp32 accumulation) and without it (the
    exact fp32 FFMA path), CUDA-event time of each pass call."""
    import torch
    from voxel_gemm_gb300 import ops, synth
    stream = torch.cuda.Stream(device=dev)
    wl = synth.Workload(base.name + "_f32", base.B, base.res, base.shapes_per_sample, base.kinds, 256, 256, "f32",
                        base.seed, 2.0)
    coords_np = synth.make_coords(base)
    N = coords_np.shape[0]
    with torch.cuda.stream(stream):
        coords = torch.from_numpy(coords_np).to(dev)
        f, W, b, dY = synth.make_tensors(wl, N, device=dev)
        m = ops.NbrMap.alloc(N, base.grid, base.key_flag, device=dev)
        out = torch.empty(N, wl.cout, dtype=torch.float32, device=dev)
        dX = torch.empty(N, wl.cin, dtype=torch.float32, device=dev)
        dW = torch.empty_like(W)
        db = torch.empty_like(b)
    m.build(coords, stream)
    assert m.status(stream) == ops.VG_OK
    P = count_pairs(m.mask.cpu().numpy().view("uint32"))
    peaks = load_peaks()
    tf32_peak = peaks["bf16_tflops"] / 2  # dense TF32 rate: half the 16-bit rate (nominal ratio)
    rec = {"workload": wl.name, "N": N, "P": P, "cin": wl.cin, "cout": wl.cout,
           "tf32_peak_tflops": tf32_peak, "tf32_peak_source": peaks["source"] + " bf16 burst / 2"}
    for tag, flags in (("tf32", ops.VG_ALLOW_TF32), ("ffma", 0)):
        with torch.cuda.stream(stream):
            ws = ops.conv_workspace(N, wl.cin, wl.cout, torch.float32, device=dev, flags=flags)
        calls = {
            "fwd": lambda: ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, flags=flags, stream=stream),
            "dgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, None, None, ws, flags=flags,
                                                    stream=stream),
            "wgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, None, dW, db, ws, flags=flags,
                                                    stream=stream),
        }
        r = {}
        for name, call in calls.items():
            for _ in range(2):
                call()
            ts = []
            for _ in range(max(3, min(args.steps, 10))):
                with torch.cuda.stream(stream):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    call()
                    e1.record(stream)
                ts.append((e0, e1))
            stream.synchronize()
            ms = sum(a.elapsed_time(b_) for a, b_ in ts) / len(ts)
            fl = 2.0 * P * wl.cin * wl.cout
            r[name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12}
            if tag == "tf32":
                r[name]["frac_of_tf32_peak"] = r[name]["tflops"] / tf32_peak
        assert ops.vg_conv_status(ws, stream) == ops.VG_OK
        rec[tag] = r
        del ws
    rec["speedup_tf32"] = sum(v["ms"] for v in rec["ffma"].values()) / sum(v["ms"] for v in rec["tf32"].values())
    return rec


def run_row_orders(args, wl, dev, flush):
    """The two row orders of the neighbour map on one workload: Morton (the default)
    and Hilbert (VG_ORDER_HILBERT).  Per order: the useful fraction of the MMA rows
    (valid pairs / (rows x taps the tile masks make the GEMM process)), and the
    CUDA-event time of the map build, the forward and the weight-gradient call."""
    import numpy as np
    import torch
    from voxel_gemm_gb300 import ops, synth
    stream = torch.cuda.Stream(device=dev)
    coords_np = synth.make_coords(wl)
    N = coords_np.shape[0]
    dt = synth.torch_dtype(wl.dtype)
    with torch.cuda.stream(stream):
        coords = torch.from_numpy(coords_np).to(dev)
        f, W, b, dY = synth.make_tensors(wl, N, device=dev)
        out = torch.empty(N, wl.cout, dtype=dt, device=dev)
        dW = torch.empty(27, wl.cin, wl.cout, dtype=dt, device=dev)
        db = torch.empty(wl.cout, dtype=dt, device=dev)
        ws = ops.conv_workspace(N, wl.cin, wl.cout, dt, device=dev)
    rec = {"workload": wl.name, "N": N}
    for tag, flag in (("morton", 0), ("hilbert", ops.VG_ORDER_HILBERT)):
        m = ops.NbrMap.alloc(N, wl.grid, wl.key_flag | flag, device=dev)
        m.build(coords, stream)
        assert m.status(stream) == ops.VG_OK
        tm = m.tile_mask().cpu().numpy().view(np.uint32)
        pop_tiles = int(sum(int(((tm >> k) & 1).sum()) for k in range(27)))
        P = count_pairs(m.mask.cpu().numpy().view("uint32"))
        calls = {
            "nbrmap": lambda: m.build(coords, stream),
            "fwd": lambda: ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, stream=stream),
            "wgrad": lambda: ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, None, dW, db, ws, stream=stream),
        }
        r = {"useful_mma_row_fraction": P / (128.0 * pop_tiles)}
        for name, fn in calls.items():
            fn()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            ts = []
            for _ in range(max(3, min(args.steps, 10))):
                with torch.cuda.stream(stream):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                ts.append((e0, e1))
            stream.synchronize()
            r[name + "_ms"] = sum(a.elapsed_time(b_) for a, b_ in ts) / len(ts)
        assert ops.vg_conv_status(ws, stream) == ops.VG_OK
        rec[tag] = r
    return rec


def run_regular_conv(args, wl, dev, flush):
    """Strided (down-sampling) and transposed (up-sampling) sparse convolution on the
    workload's voxels: the map build, the strided forward, its backward (input,
    weight and bias gradient) and the transposed forward, each timed alone with CUDA
    events; FLOPs count valid (output, tap) pairs only."""
    import torch
    from voxel_gemm_gb300 import ops, synth
    stream = torch.cuda.Stream(device=dev)
    coords = torch.from_numpy(synth.make_coords(wl)).to(dev)
    dt = synth.torch_dtype(wl.dtype)
    peaks = load_peaks()
    recs = []
    for K, s_ in ((2, 2), (3, 2)):
        ev = []
        with torch.cuda.stream(stream):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
        m = ops.SparseMap(coords, wl.grid, K, s_, stream=stream)
        with torch.cuda.stream(stream):
            t1.record(stream)
        stream.synchronize()
        build_ms = t0.elapsed_time(t1)
        T = K ** 3
        g = torch.Generator(device=dev)
        g.manual_seed(17 + K)
        f = torch.randn(m.n_in, wl.cin, generator=g, device=dev).to(dt)
        W = (torch.randn(T, wl.cin, wl.cout, generator=g, device=dev) * (2.0 / (T * wl.cin)) ** 0.5).to(dt)
        b = torch.zeros(wl.cout, dtype=dt, device=dev)
        dY = torch.randn(m.n_out, wl.cout, generator=g, device=dev).to(dt)
        out = torch.empty(m.n_out, wl.cout, dtype=dt, device=dev)
        dX = torch.empty(m.n_in, wl.cin, dtype=dt, device=dev)
        dW = torch.empty_like(W)
        db = torch.empty_like(b)
        gc = torch.randn(m.n_out, wl.cin, generator=g, device=dev).to(dt)
        up_out = torch.empty(m.n_in, wl.cout, dtype=dt, device=dev)
        ws0 = m.workspace(0, wl.cin, wl.cout, dt)
        ws1 = m.workspace(1, wl.cin, wl.cout, dt)
        P = int((m.down().cpu().numpy().view("uint32") != 0xFFFFFFFF).sum())
        calls = {"strided_fwd": lambda: m.fwd(0, f, W, b, out, ws0, stream=stream),
                 "strided_bwd": lambda: m.bwd(0, dY, f, W, dX, dW, db, ws0, stream=stream),
                 "transposed_fwd": lambda: m.fwd(1, gc, W, b, up_out, ws1, stream=stream)}
        r = {"kernel": K, "stride": s_, "n_in": m.n_in, "n_out": m.n_out, "pairs": P, "map_build_ms": build_ms}
        for name, fn in calls.items():
            fn()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn()
            ts = []
            for _ in range(max(3, min(args.steps, 10))):
                with torch.cuda.stream(stream):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    gr.replay()
                    e1.record(stream)
                ts.append((e0, e1))
            stream.synchronize()
            ms = sum(a.elapsed_time(b_) for a, b_ in ts) / len(ts)
            fl = (2.0 if name != "strided_bwd" else 4.0) * P * wl.cin * wl.cout
            r[name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                       "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}
        assert ops.vg_conv_status(ws0, stream) == ops.VG_OK and ops.vg_conv_status(ws1, stream) == ops.VG_OK
        recs.append(r)
        del m, ws0, ws1
        torch.cuda.empty_cache()
    return {"workload": wl.name, "cases": recs}


def run_ours(args, rank, world, local_rank):
    import torch
    from voxel_gemm_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    wl = synth.WORKLOADS[args.workload]
    head = run_workload(args, wl, rank, world, dev, flush, full=True)
    torch.cuda.empty_cache()
    sweep = []
    # with N ranks only the headline runs: the other records are single-GPU measurements,
    # and a rank that failed one of them would leave the others waiting in a collective
    if not args.no_sweep and world == 1:
        for name in SWEEP:
            if name == wl.name:
                continue
            try:
                sweep.append(run_workload(args, synth.WORKLOADS[name], rank, world, dev, flush, full=False))
            except Exception as e:  # noqa: BLE001 - a failed sub-record must not hide the headline
                sweep.append({"workload": name, "error": f"{type(e).__name__}: {e}"})
            torch.cuda.empty_cache()
        try:
            infer = run_inference(args, synth.WORKLOADS[INFER_WORKLOAD], dev, flush)
        except Exception as e:  # noqa: BLE001
            infer = {"workload": INFER_WORKLOAD, "error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
        orders = []
        for name in ORDER_WORKLOADS:
            try:
                orders.append(run_row_orders(args, synth.WORKLOADS[name], dev, flush))
            except Exception as e:  # noqa: BLE001
                orders.append({"workload": name, "error": f"{type(e).__name__}: {e}"})
            torch.cuda.empty_cache()
        try:
            regular = run_regular_conv(args, synth.WORKLOADS[REGULAR_WORKLOAD], dev, flush)
        except Exception as e:  # noqa: BLE001
            regular = {"workload": REGULAR_WORKLOAD, "error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
        try:
            tf32 = run_tf32(args, synth.WORKLOADS[REGULAR_WORKLOAD], dev, flush)
        except Exception as e:  # noqa: BLE001
            tf32 = {"workload": REGULAR_WORKLOAD, "error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    else:
        infer = None
        orders = None
        regular = None
        tf32 = None

    res = {
        "metric": METRIC, "value": head["value"], "unit": "voxels/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic (seeded voxelised sphere/torus surfaces)",
        "config": workload_config(wl, head["N"], head["P"], world),
        "tflops": head["tflops"], "tflops_frac_of_bf16_peak": head["tflops_frac_of_bf16_peak"],
        "roofline_step_frac": head["roofline_step_frac"],
        "roofline": head["roofline"], "passes": head["passes"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"], "gpu_launches_per_step": head["gpu_launches_per_step"],
        "path": head["path"], "launch": head["launch"], "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
        "sweep": sweep,
        "inference_small_n": infer,
        "row_order_morton_vs_hilbert": orders,
        "regular_conv": regular,
        "tf32": tf32,
    }
    return res


# ------------------------------------------------------------------ oracle arm (CPU)
def oracle_sample(wl, coords_np, budget_rows, seed=0, min_seconds=5.0, nbrmap=None):
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
    if nbrmap is not None:
        nbrmap.append(mask)
    return 1.0 / per_voxel, {"rows": rows_done, "t_map_s": t_map, "t_conv_s": t_conv}


def run_reference(args, world):
    from voxel_gemm_gb300 import shard, synth
    import oracle
    wl = synth.WORKLOADS[args.workload]
    coords_np = shard.rank_coords(wl, 0)
    budget = rows_budget(wl)
    masks = []
    for _ in range(args.warmup):
        oracle_sample(wl, coords_np, max(64, budget // 8), min_seconds=0.0, nbrmap=masks)
    vals = []
    t0 = time.perf_counter()
    for k in range(args.steps):
        v, _ = oracle_sample(wl, coords_np, budget, seed=k, min_seconds=1.0, nbrmap=masks)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    cores = oracle.num_threads()
    N = int(coords_np.shape[0])
    P = count_pairs(masks[-1]) if masks else None
    sample = (f"full neighbour map of N={N} voxels, then fwd+dgrad+wgrad over "
              f"{min(budget, N)} seeded sampled rows per step; voxels/s = 1 / (map time per "
              f"voxel + conv time per sampled row)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "voxels/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded voxelised sphere/torus surfaces)",
            "config": workload_config(wl, N, P, world),
            "cpu_baseline": {"value": value, "unit": "voxels/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def rows_budget(wl):
    # about 1-2 s of fp64 work per sample on a many-core host
    per_row = 3 * 10.6 * wl.cin * wl.cout
    return int(max(256, min(65536, 2e9 / per_row)))


def run_ncu_step(args):
    """The command a profiler attaches to: --warmup eager steps, then one more, of the
    workload's map build + forward + input gradient + weight/bias gradient on one
    stream with one conv workspace (per step the kernels launch in that order).
    With --tf32: fp32 features at Cin = Cout = 256 on the workload's voxels, under
    VG_ALLOW_TF32 (the bench's TF32 record)."""
    import torch
    from voxel_gemm_gb300 import ops, synth
    wl = synth.WORKLOADS[args.workload]
    flags = 0
    if args.tf32:
        wl = synth.Workload(wl.name + "_f32", wl.B, wl.res, wl.shapes_per_sample, wl.kinds, 256, 256, "f32",
                            wl.seed, 2.0, key_flag=wl.key_flag)
        flags = ops.VG_ALLOW_TF32
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    coords = torch.from_numpy(synth.make_coords(wl)).to(dev)
    N = coords.shape[0]
    f, W, b, dY = synth.make_tensors(wl, N, device=dev)
    dt = f.dtype
    m = ops.NbrMap.alloc(N, wl.grid, wl.key_flag)
    ws = ops.conv_workspace(N, wl.cin, wl.cout, dt, flags=flags)
    out = torch.empty(N, wl.cout, dtype=dt, device=dev)
    dX = torch.empty(N, wl.cin, dtype=dt, device=dev)
    dW = torch.empty_like(W)
    db = torch.empty_like(b)
    for _ in range(args.warmup + 1):
        m.build(coords, s)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, flags=flags, stream=s)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, dW, db, ws, flags=flags, stream=s)
    s.synchronize()
    assert m.status(s) == ops.VG_OK and ops.vg_conv_status(ws, s) == ops.VG_OK
    print(json.dumps({"ncu_step": wl.name, "N": N}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-graph", action="store_true", help="launch each call eagerly instead of replaying a CUDA graph")
    ap.add_argument("--one-stream", action="store_true",
                    help="issue the step's conv passes one after the other on one stream")
    ap.add_argument("--ncu-step", action="store_true",
                    help="run --warmup + 1 eager steps on one stream and exit (for profilers)")
    ap.add_argument("--tf32", action="store_true",
                    help="with --ncu-step: fp32 features (C = 256) under VG_ALLOW_TF32")
    args = ap.parse_args()
    if args.ncu_step:
        run_ncu_step(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            from voxel_gemm_gb300 import shard, synth
            import oracle
            wl = synth.WORKLOADS[args.workload]
            coords_np = shard.rank_coords(wl, 0)
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
