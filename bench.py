"""Benchmark: the 25-point (radius 4, 8th-order) Laplacian sweep, fp32, on a 512^3 grid.

One step = one stencil_apply over the whole 512^3 grid (plan cached), inputs resident
in HBM.  The grid (512 MiB in, 512 MiB out) is larger than L2, so no flush is needed
between steps.  Also measured in the same run: the fused acoustic wave step on 640^3
("wave" key), the end-to-end host-buffer call ("e2e"), SM clocks during the timed
region, and the CPU oracle on the host cores ("cpu_baseline").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun) runs independent replicas, one per GPU: the path has no
exchange step at this size, so ranks never communicate on the data path; the value is
the total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from seismic_wave_propagation_gb300 import synth, traffic  # noqa: E402

METRIC = "GPoints/s and achieved HBM GB/s (% of GB300 peak), 25-pt R=4 fp32 at 512^3"
NX = NY = NZ = 512
R = 4
WAVE_N = 640
FALLBACK_HBM_GBS = 6800.0
E2E_WARMUP = 3
E2E_CALLS = 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The files that make up the device code (the kernels and their instantiation tables).
DEVICE_SOURCES = ("star_kernels.cuh", "kernel_table.h", "kernels_apply.cu", "kernels_wave.cu")


def kernel_source_hash() -> str:
    """Hash of the device code with comments and whitespace removed (the sources hold no
    string literal with a comment marker), so that comment edits keep recorded counters."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "seismic_wave_propagation_gb300", "csrc")
    for name in DEVICE_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(key: str, launch: dict | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel
    source and, for the launch-geometry keys the entry lists, on the geometry of `launch`."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[key]
        if e.get("kernel_source_hash") != kernel_source_hash():
            return None
        if launch is not None and any(e["launch"][k] != launch.get(k) for k in e.get("match", ())):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.gpu_id = gpu_id

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return dist, rank, local, world
    return None, 0, 0, 1


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def time_oracle(u: np.ndarray, c: np.ndarray, budget_s: float, min_reps: int = 1):
    """Oracle sweeps over z-slabs of the grid until ~budget_s; returns (points/s, sample, cores)."""
    import oracle
    oracle.build()
    nz = u.shape[0]
    c32 = c.astype(np.float32)
    # calibrate on a thin slab
    slab = u[: 2 * R + 8]
    t0 = time.perf_counter()
    oracle.apply(slab, c32, R)
    rate = traffic.interior_points(NX, NY, 2 * R + 8, R) / max(1e-9, time.perf_counter() - t0)
    planes = int(max(1, min(nz - 2 * R, rate * budget_s / ((NX - 2 * R) * (NY - 2 * R)))))
    sub = np.ascontiguousarray(u[: planes + 2 * R])
    pts = traffic.interior_points(NX, NY, planes + 2 * R, R)
    reps, t = 0, 0.0
    out = sub.copy()
    while reps < min_reps or t < budget_s * 0.5:
        t0 = time.perf_counter()
        oracle.apply(sub, c32, R, out=out)
        t += time.perf_counter() - t0
        reps += 1
        if t > budget_s:
            break
    sample = f"{reps} oracle sweep(s) of a {NX}x{NY}x{planes + 2 * R} slab of the 512^3 grid ({pts} interior points each)"
    return pts * reps / t, sample, oracle.num_threads()


def bench_config(world: int) -> dict:
    """The workload both arms time (the GPU line and the reference arm print this same dict)."""
    return {"workload": "star25_lap8_512", "nx": NX, "ny": NY, "nz": NZ, "radius": R,
            "coeffs": "8th-order Laplacian, h=1", "l2": "inputs (512 MiB) larger than L2; no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args, dist, rank, world):
    """Reference arm: the CPU oracle as it stands, on the host cores, same metric/config."""
    if rank != 0:
        return
    c = synth.laplacian8_coeffs()
    u = synth.uniform_field(NX, NY, NZ)
    import oracle
    oracle.build()
    per_step = min(args.cpu_budget, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(u, c, per_step)
    vals, samples = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, sample, cores = time_oracle(u, c, per_step)
        vals.append(v)
        samples.append(sample)
    wall = time.perf_counter() - t0
    gpts = statistics.median(vals) / 1e9
    line = {"metric": METRIC, "impl": "reference", "value": gpts, "unit": "GPoints/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": bench_config(world),
            "cpu_baseline": {"value": gpts, "unit": "GPoints/s", "cores": cores, "kind": "oracle",
                             "sample": samples[-1] if samples else ""},
            "e2e": {"value": gpts, "unit": "GPoints/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, dist, rank, local, world):
    import torch
    from seismic_wave_propagation_gb300 import StencilPlan

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peak, peak_kind = peaks()
    c = synth.laplacian8_coeffs()

    # ---- headline: 25-point sweep at 512^3 ---------------------------------------
    u = synth.uniform_field(NX, NY, NZ)
    d_in = torch.from_numpy(u.ravel()).to(dev)
    d_out = d_in.clone()
    plan = StencilPlan(NX, NY, NZ, R, c)
    info = plan.launch_info(0)
    s = stream.cuda_stream
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            plan.apply(d_in.data_ptr(), d_out.data_ptr(), s)
        plan.status(s)
        # One event pair around the timed region: events between the launches would add
        # their own gaps (measured 1.9 % per sweep).
        whole0, whole1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gpu_uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
        gpu_id = f"GPU-{gpu_uuid}" if gpu_uuid is not None and not str(gpu_uuid).startswith("GPU-") else (
            str(gpu_uuid) if gpu_uuid is not None else None)
        torch.cuda.synchronize(dev)
        barrier(dist)
        torch.cuda.synchronize(dev)
        with ClockSampler(gpu_id) as clk:
            time.sleep(0.25)
            whole0.record(stream)
            for _ in range(args.steps):
                plan.apply(d_in.data_ptr(), d_out.data_ptr(), s)
            whole1.record(stream)
            torch.cuda.synchronize(dev)
        barrier(dist)
        plan.status(s)
    total_ms = whole0.elapsed_time(whole1)
    avg_launch_s = total_ms / args.steps / 1e3  # every launch in the region is this kernel
    total_ms = max_over_ranks(dist, total_ms)
    interior = traffic.interior_points(NX, NY, NZ, R)
    pts_all = sum_over_ranks(dist, float(interior * args.steps))
    gpts = pts_all / (total_ms / 1e3) / 1e9
    algo_bytes = traffic.apply_bytes(NX, NY, NZ, R)
    achieved = algo_bytes / avg_launch_s / 1e9
    clocks = clk.summary()

    # ---- end to end through the host-buffer C-ABI call --------------------------------
    # Every call copies the step's input in from pinned host memory and its result out
    # (1 GiB of host transfers), pipelined over z-slabs inside the library.  Median of
    # E2E_CALLS timed calls after E2E_WARMUP untimed ones.
    h_in = torch.from_numpy(u.ravel()).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    in_np, out_np = h_in.numpy(), h_out.numpy()
    for _ in range(E2E_WARMUP):
        plan.apply_host(in_np, out_np, 1, s)
    torch.cuda.synchronize(dev)
    e2e_times, phases = [], []
    for _ in range(E2E_CALLS):
        t0 = time.perf_counter()
        plan.apply_host(in_np, out_np, 1, s)
        e2e_times.append(time.perf_counter() - t0)
        phases.append(plan.host_phases())
    e2e_s = statistics.median(e2e_times)
    e2e_s = max_over_ranks(dist, e2e_s)
    mid = sorted(range(len(e2e_times)), key=lambda i: e2e_times[i])[len(e2e_times) // 2]
    e2e = {"value": sum_over_ranks(dist, float(interior)) / e2e_s / 1e9, "unit": "GPoints/s",
           "h2d_bytes_per_step": 4 * NX * NY * NZ, "d2h_bytes_per_step": 4 * NX * NY * NZ,
           "ms_per_step": e2e_s * 1e3, "steps": E2E_CALLS, "warmup": E2E_WARMUP,
           "ms_min": min(e2e_times) * 1e3, "ms_max": max(e2e_times) * 1e3,
           "phases_of_median_call": phases[mid]}
    # The host link bounds this leg: time plain pinned copies of the same bytes, one way
    # at a time and both ways at once (as the pipelined call overlaps them), and report
    # the step's ceiling at the both-ways rate.
    d_in, d_src = torch.empty(h_in.numel(), device=dev), torch.empty(h_in.numel(), device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def h2d():
        with torch.cuda.stream(s_in):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            h_out.copy_(d_src, non_blocking=True)

    def both_ways():
        h2d()
        d2h()

    def median_s(fn, n=7):
        fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(n):
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            ts.append(time.perf_counter() - t0)
        return statistics.median(ts)
    link_s = median_s(both_ways)
    nbytes = 4 * NX * NY * NZ
    e2e["link"] = {"each_way_gbs": nbytes / link_s / 1e9, "ms": link_s * 1e3,
                   "h2d_alone_gbs": nbytes / median_s(h2d) / 1e9, "d2h_alone_gbs": nbytes / median_s(d2h) / 1e9,
                   "ceiling_value": float(interior) / link_s / 1e9,
                   "frac": (float(interior) / e2e_s) / (float(interior) / link_s),
                   "how": "pinned cudaMemcpyAsync of the step's bytes, H2D and D2H on two streams at once (median of 7)"}
    del d_in, d_src, h_in, h_out

    # ---- fused wave step at 640^3 ----------------------------------------------------
    wave = None
    if not args.skip_wave:
        n = WAVE_N
        up, uu, vv, ee = synth.wave_fields(n, n, n)
        f = [torch.from_numpy(a.ravel()).to(dev) for a in (up, uu, vv, ee)]
        nxt = f[0].clone()
        wplan = StencilPlan(n, n, n, R, c)
        a, b = f[0], f[1]
        wsteps = max(10, min(200, args.steps // 20))
        with torch.cuda.stream(stream):
            for _ in range(3):
                wplan.wave_step(a.data_ptr(), b.data_ptr(), nxt.data_ptr(), f[2].data_ptr(), f[3].data_ptr(), s)
                a, b, nxt = b, nxt, a
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            w0.record(stream)
            for _ in range(wsteps):
                wplan.wave_step(a.data_ptr(), b.data_ptr(), nxt.data_ptr(), f[2].data_ptr(), f[3].data_ptr(), s)
                a, b, nxt = b, nxt, a
            w1.record(stream)
            torch.cuda.synchronize(dev)
            wplan.status(s)
        wms = w0.elapsed_time(w1) / wsteps
        # The same step with the region split (eta read only in the 16-point sponge).
        with torch.cuda.stream(stream):
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            p0.record(stream)
            for _ in range(wsteps):
                wplan.wave_step_pml(a.data_ptr(), b.data_ptr(), nxt.data_ptr(), f[2].data_ptr(),
                                    f[3].data_ptr(), 16, s)
                a, b, nxt = b, nxt, a
            p1.record(stream)
            torch.cuda.synchronize(dev)
            wplan.status(s)
        pms = p0.elapsed_time(p1) / wsteps
        wbytes = traffic.wave_bytes(n, n, n, R)
        wint = traffic.interior_points(n, n, n, R)
        wave = {"workload": "wave25_640", "steps": wsteps, "ms_per_step": wms,
                "gpoints_per_s": wint / (wms / 1e3) / 1e9,
                "roofline": {"bound": "hbm", "achieved": wbytes / (wms / 1e3) / 1e9, "peak": peak,
                             "unit": "GB/s", "frac": wbytes / (wms / 1e3) / 1e9 / peak,
                             "traffic": profiled_traffic("wave25_640", wplan.launch_info(1))},
                "launch": wplan.launch_info(1),
                "pml16": {"ms_per_step": pms, "gpoints_per_s": wint / (pms / 1e3) / 1e9,
                          "wave_step_bytes_over_time_gbs": wbytes / (pms / 1e3) / 1e9}}
        wplan.close()
        del f, nxt, a, b
    plan.close()

    # ---- CPU oracle baseline (rank 0, N = 1 only) ---------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        v, sample, cores = time_oracle(u, c, args.cpu_budget)
        cpu = {"value": v / 1e9, "unit": "GPoints/s", "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": gpts, "unit": "GPoints/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": bench_config(world), "launch": info,
                "hbm_gbs": achieved, "hbm_frac_of_peak": achieved / peak,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "traffic": profiled_traffic("star25_512", info),
                             "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                             else "fallback 6.8 TB/s",
                             "algorithmic_bytes_per_launch": algo_bytes,
                             "avg_launch_ms": avg_launch_s * 1e3},
                "gpu_launches": args.steps,
                "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                           "reasons": clocks["reasons"], "samples": clocks["samples"]},
                "e2e": e2e, "cpu_baseline": cpu, "wave": wave}
        print(json.dumps(line), flush=True)


def run_profile_case(kind: str):
    """Three launches of the 512^3 case of one kernel (the 64^3 smoothing sweep for
    "direct64", on the direct-load kernel; the 25-point sweep of a 1152 x 1152 x 256 grid,
    whose planes take the 64 x 24 tile, for "sweep_wide"): the driver for ncu captures."""
    import torch
    from seismic_wave_propagation_gb300 import StencilPlan
    n = 64 if kind == "direct64" else NX
    dims = (1152, 1152, 256) if kind == "sweep_wide" else (n, n, n)
    r = 1 if kind in ("sweep7", "sweep7x2", "direct64") else R
    c = synth.average7_coeffs() if kind == "direct64" else synth.laplacian2_coeffs() if r == 1 else synth.laplacian8_coeffs()
    plan = StencilPlan(*dims, r, c)
    if kind == "direct64":
        plan.set_sweep_path("direct")
    if kind in ("sweep", "semi", "sweep7", "sweep7x2", "direct64", "sweep_wide"):
        u = torch.from_numpy(synth.uniform_field(*dims).ravel()).cuda()
        o = u.clone()
        fn = {"semi": plan.apply_semi, "sweep7x2": plan.apply2}.get(kind, plan.apply)
        for _ in range(3):
            fn(u, o)
    else:
        f = [torch.from_numpy(a.ravel()).cuda() for a in synth.wave_fields(n, n, n)]
        nxt = f[0].clone()
        for _ in range(3):
            if kind == "wave_inner":  # no band: the inner region's kernel covers all but one tile row
                plan.wave_step_pml(f[0], f[1], nxt, f[2], f[3], 0)
            else:
                plan.wave_step(f[0], f[1], nxt, f[2], f[3])
    torch.cuda.synchronize()
    plan.status()
    k = {"sweep": 0, "sweep7": 0, "direct64": 0, "sweep_wide": 0, "wave": 1, "wave_inner": 2, "semi": 3,
         "sweep7x2": 4}[kind]
    print(json.dumps({"profile_case": kind, "grid": list(dims), "launch": plan.launch_info(k)}))


def _time_loop(fn, steps, warmup, stream, warm_seconds=0.3):
    """Mean CUDA-event time of `fn` over `steps` calls, after at least `warmup` calls and at
    least `warm_seconds` of warm-up (the GPU may have idled through CPU work before)."""
    import torch
    t0 = time.perf_counter()
    done = 0
    while done < warmup or time.perf_counter() - t0 < warm_seconds:
        fn()
        done += 1
        if done % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _first_step_parity(torch, plan, w, c, stream, samples=40000):
    """The workload's first sweep or step from its initial fields, checked against the
    oracle at sampled interior points: the largest error as a fraction of the tolerance
    (1e-5 * sum|c| * max|u| per sweep; 2e-5 * (2 + 0.2 * sum|c|) * max|u| for a step)."""
    import oracle
    oracle.build()
    nx, ny, nz, r = w["nx"], w["ny"], w["nz"], w["radius"]
    rng = np.random.default_rng(11)
    idx = (rng.integers(r, nx - r, samples) + nx * (rng.integers(r, ny - r, samples)
                                                  + ny * rng.integers(r, nz - r, samples))).astype(np.int64)
    c32 = c.astype(np.float32)
    with torch.cuda.stream(stream):
        if w["init"] == "wave":
            f = synth.wave_fields(nx, ny, nz)
            d = [torch.from_numpy(a.ravel()).cuda() for a in f]
            nxt = d[0].clone()
            plan.wave_step(d[0], d[1], nxt, d[2], d[3], stream)
            plan.status(stream)
            got = nxt.cpu().numpy()[idx]
            want = oracle.wave_points(f[0], f[1], f[2], f[3], c32, r, idx)
            tol = 2e-5 * (2 + 0.2 * float(np.sum(np.abs(c32)))) * float(np.max(np.abs(f[1])))
        else:
            u0 = synth.sinusoid_field(nx, ny, nz) if w["init"] == "sinusoids" else synth.uniform_field(nx, ny, nz)
            d = torch.from_numpy(u0.ravel()).cuda()
            o = d.clone()
            plan.apply(d, o, stream)
            plan.status(stream)
            got = o.cpu().numpy()[idx]
            want = oracle.apply_points(u0, c32, r, idx)
            tol = 1e-5 * float(np.sum(np.abs(c32))) * float(np.max(np.abs(u0)))
    return float(np.max(np.abs(got.astype(np.float64) - want))) / tol


def run_extra_rows(torch, stream, peak):
    """The next rows beside the workloads: the wave step on the 7-point eta damping (its
    one-off damping pass and a step on the result), the region-split step, and the 512^3
    25-point sweep held as z-slabs with its ghost exchange (one GPU)."""
    from seismic_wave_propagation_gb300 import StencilPlan, StencilSlabs
    out = {}
    n = 640
    c = synth.laplacian8_coeffs()
    plan = StencilPlan(n, n, n, R, c)
    f = [torch.from_numpy(a.ravel()).cuda() for a in synth.wave_fields(n, n, n)]
    eff = torch.empty_like(f[3])
    nxt = f[0].clone()
    with torch.cuda.stream(stream):
        ms_eta = _time_loop(lambda: plan.eta_stencil(f[3], eff, 0.5, 1.0 / 12.0, stream), 20, 3, stream)
        ms_plain = _time_loop(lambda: plan.wave_step(f[0], f[1], nxt, f[2], f[3], stream), 30, 3, stream)
        ms_eff = _time_loop(lambda: plan.wave_step(f[0], f[1], nxt, f[2], eff, stream), 30, 3, stream)
        ms_pml = _time_loop(lambda: plan.wave_step_pml(f[0], f[1], nxt, f[2], f[3], 16, stream), 30, 3, stream)
        plan.status(stream)
    wb = traffic.wave_bytes(n, n, n, R)
    out["wave 640^3, pointwise eta"] = json.dumps({"ms": round(ms_plain, 4), "frac_of_peak": round(wb / (ms_plain / 1e3) / 1e9 / peak, 3)})
    out["wave 640^3, 7-point eta damping (N3)"] = json.dumps({
        "damping_pass_ms_once": round(ms_eta, 4),
        "damping_pass_frac_of_peak": round(traffic.apply_bytes(n, n, n, 1) / (ms_eta / 1e3) / 1e9 / peak, 3),
        "step_ms": round(ms_eff, 4), "step_frac_of_peak": round(wb / (ms_eff / 1e3) / 1e9 / peak, 3)})
    out["wave 640^3, region split, 16-point band (N1)"] = json.dumps({"ms": round(ms_pml, 4)})
    plan.close()
    del f, eff, nxt
    m = 512
    u0 = synth.uniform_field(m, m, m)
    whole = StencilPlan(m, m, m, R, c)
    a = torch.from_numpy(u0.ravel()).cuda()
    b = a.clone()
    with torch.cuda.stream(stream):
        ms_whole = _time_loop(lambda: whole.apply(a, b, stream), 100, 10, stream)
        whole.status(stream)
    whole.close()
    del a, b
    row = {"whole_grid_ms": round(ms_whole, 4)}
    for P in (2, 4, 8):
        sl = StencilSlabs(m, m, m, R, c, P)
        xs = []
        for k in range(P):
            e = sl.extent(k)
            xs.append(torch.from_numpy(np.ascontiguousarray(u0[e["begin"]:e["end"]]).ravel()).cuda())
        ys = [x.clone() for x in xs]
        with torch.cuda.stream(stream):
            ms = _time_loop(lambda: sl.apply(xs, ys, stream), 100, 10, stream)
            ms_x = _time_loop(lambda: sl.exchange(xs, stream), 100, 10, stream)
            sl.status(stream)
        row[f"{P}_slabs_ms"] = round(ms, 4)
        row[f"{P}_slabs_exchange_alone_ms"] = round(ms_x, 4)
        sl.close()
        del xs, ys
    out["sweep 512^3 as z-slabs on one GPU (N4)"] = json.dumps(row)
    torch.cuda.empty_cache()
    return out


def run_report_configs(args):
    """Time all five workloads as their configs define them (sweeps/steps loops), plus the
    CPU oracle on a bounded sample of each; one JSON line per workload and a markdown table."""
    import torch
    from seismic_wave_propagation_gb300 import StencilPlan
    peak, _ = peaks()
    stream = torch.cuda.Stream()
    out = []
    for name, w in synth.WORKLOADS.items():
        nx, ny, nz, r = w["nx"], w["ny"], w["nz"], w["radius"]
        c = synth.coeffs_for(w["coeffs"])
        plan = StencilPlan(nx, ny, nz, r, c)
        interior = traffic.interior_points(nx, ny, nz, r)
        with torch.cuda.stream(stream):
            if w["init"] == "wave":
                f = [torch.from_numpy(a.ravel()).cuda() for a in synth.wave_fields(nx, ny, nz)]
                bufs = [f[0], f[1], f[0].clone()]
                v, e = f[2], f[3]

                def loop():  # the workload's step loop, one graph launch
                    plan.wave_steps(bufs[0], bufs[1], bufs[2], v, e, w["steps"], -1, True, stream)
                units, per = w["steps"], traffic.wave_bytes(nx, ny, nz, r)
            else:
                u0 = synth.sinusoid_field(nx, ny, nz) if w["init"] == "sinusoids" else synth.uniform_field(nx, ny, nz)
                a = torch.from_numpy(u0.ravel()).cuda()
                bufs = [a, a.clone()]
                nsw = w["sweeps"]

                def loop():  # the workload's ping-pong sweeps, one graph launch (one sweep: one launch)
                    if nsw == 1:
                        plan.apply(bufs[0], bufs[1], stream)
                    else:
                        plan.sweeps(bufs[0], bufs[1], nsw, True, stream)
                units, per = nsw, traffic.apply_bytes(nx, ny, nz, r)
            reps = max(1, min(101, int(2000 // max(1, units))))
            ms = _time_loop(loop, reps, 3, stream)
            chained = None
            if w["init"] != "wave" and units == 1 and nx * ny * nz <= 1 << 20:
                # a single sweep of a small grid is launch-bound: also report its time when
                # sweeps are chained back to back in one graph
                chained = _time_loop(lambda: plan.sweeps(bufs[0], bufs[1], 1000, True, stream), 5, 2, stream) / 1000
            plan.status(stream)
        ms_unit = ms / units
        key = {"star25_lap8_512": ("star25_512", 0), "wave25_640": ("wave25_640", 1)}.get(name)
        dram = profiled_traffic(key[0], plan.launch_info(key[1])) if key else None
        line = {"workload": name, "grid": [nx, ny, nz], "radius": r, "units": units,
                "ms_per_sweep_or_step": ms_unit, "gpoints_per_s": interior / (ms_unit / 1e3) / 1e9,
                "hbm_gbs": per / (ms_unit / 1e3) / 1e9, "frac_of_peak": per / (ms_unit / 1e3) / 1e9 / peak,
                "compulsory_bytes_per_point": per / interior,
                "dram_bytes_per_point_ncu": dram / interior if dram else None,
                "parity_max_err_over_tol": None, "timed_loops": reps}
        if w["init"] != "wave":
            line["sweep_path"] = plan.sweep_path
        if chained is not None:
            line["ms_per_sweep_chained_1000_in_one_graph"] = chained
        if not args.skip_cpu:
            # The CPU-oracle leg: the workload's first sweep or step checked against the
            # oracle at sampled points, then the oracle timed on a bounded sample.
            line["parity_max_err_over_tol"] = _first_step_parity(torch, plan, w, c, stream)
            import oracle
            oracle.build()
            cc = c.astype(np.float32)
            planes = max(2 * r + 1, min(nz, 2 * r + max(1, int(4e7 // max(1, nx * ny)))))
            if w["init"] == "wave":
                sub = [np.ascontiguousarray(x[:planes]) for x in synth.wave_fields(nx, ny, planes)]
                t0 = time.perf_counter()
                oracle.wave_step(sub[0], sub[1], sub[2], sub[3], cc, r)
            else:
                sub = np.ascontiguousarray(synth.uniform_field(nx, ny, planes))
                t0 = time.perf_counter()
                oracle.apply(sub, cc, r)
            dt = time.perf_counter() - t0
            line["cpu_oracle_gpoints_per_s"] = traffic.interior_points(nx, ny, planes, r) / dt / 1e9
            line["cpu_cores"] = oracle.num_threads()
        print(json.dumps(line), flush=True)
        out.append(line)
        plan.close()
        del bufs
        torch.cuda.empty_cache()
    # The two sweep kernels side by side: the transposed z filter (stencil_apply) and the
    # semi-stencil form (stencil_apply_semi), single launches at 512^3 (inputs > L2).
    n = 512
    u = torch.from_numpy(synth.uniform_field(n, n, n).ravel()).cuda()
    o = u.clone()
    cmp = []
    for r in (1, 4):
        plan = StencilPlan(n, n, n, r, synth.laplacian8_coeffs() if r == 4 else synth.laplacian2_coeffs())
        per = traffic.apply_bytes(n, n, n, r)
        row = {"comparison": f"sweep R={r} {n}^3"}
        with torch.cuda.stream(stream):
            for label, fn in (("transposed", plan.apply), ("semi", plan.apply_semi)):
                ms = _time_loop(lambda: fn(u, o, stream), 200, 10, stream)
                row[label] = {"ms": ms, "hbm_gbs": per / (ms / 1e3) / 1e9, "frac_of_peak": per / (ms / 1e3) / 1e9 / peak}
            plan.status(stream)
        print(json.dumps(row), flush=True)
        cmp.append(row)
        plan.close()
    extra = run_extra_rows(torch, stream, peak)
    print("| workload | GPoints/s | HBM GB/s | % of measured peak | ms per sweep/step | B/pt DRAM (ncu) / compulsory "
          "| parity max err/tol | CPU oracle GPoints/s |")
    print("|---|---|---|---|---|---|---|---|")
    for l in out:
        dram = "—" if l["dram_bytes_per_point_ncu"] is None else f"{l['dram_bytes_per_point_ncu']:.2f}"
        par = "—" if l["parity_max_err_over_tol"] is None else f"{l['parity_max_err_over_tol']:.3f}"
        print(f"| {l['workload']} | {l['gpoints_per_s']:.1f} | {l['hbm_gbs']:.0f} | {100 * l['frac_of_peak']:.1f} | "
              f"{l['ms_per_sweep_or_step']:.4f} | {dram} / {l['compulsory_bytes_per_point']:.2f} | {par} | "
              f"{l.get('cpu_oracle_gpoints_per_s', float('nan')):.2f} |")
    print("| row | measurement |")
    print("|---|---|")
    for k, v in extra.items():
        print(f"| {k} | {v} |")
    print("| sweep kernel | transposed z filter: ms, % of peak | semi-stencil: ms, % of peak |")
    print("|---|---|---|")
    for row in cmp:
        t, m = row["transposed"], row["semi"]
        print(f"| {row['comparison']} | {t['ms']:.4f}, {100 * t['frac_of_peak']:.1f} | {m['ms']:.4f}, {100 * m['frac_of_peak']:.1f} |")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of CPU oracle work")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-wave", action="store_true")
    ap.add_argument("--profile", choices=["sweep", "sweep7", "sweep7x2", "wave", "wave_inner", "semi", "direct64",
                                          "sweep_wide"],
                    help="run 3 launches of the 512^3 case (ncu driver); sweep7 is the 7-point Laplacian, "
                         "sweep7x2 its two-sweep pass, wave_inner the band step with no band (no-eta kernel), "
                         "direct64 the 64^3 smoothing sweep on the direct-load kernel, sweep_wide the 25-point "
                         "sweep of 1152 x 1152 x 256 (64 x 24 tiles)")
    ap.add_argument("--report-configs", action="store_true", help="time all five workloads")
    args = ap.parse_args()
    if args.profile or args.report_configs:
        from seismic_wave_propagation_gb300 import build as b
        b.build()
        if args.profile:
            run_profile_case(args.profile)
        else:
            run_report_configs(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist, rank, local, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, dist, rank, world)
    else:
        from seismic_wave_propagation_gb300 import build as b
        b.build()
        run_ours(args, dist, rank, local, world)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
