"""Benchmark of the deterministic sum / scatter-add / scan library on one GPU
(replicas on N GPUs under torchrun).

One step = one call of the operation on one batch of the workload's
synthetic input, inputs resident in HBM.  The headline workload is the
indexed scatter-add: n = 2^24 f32 N(0,1) values into 1,024 uniform bins
(hist -> offsets -> stable scatter -> segmented tree).  The JSON line also
carries, measured in the same run, every other operation on its own workload
("ops"), the dominant kernel's roofline, the end-to-end number through host
buffers, the nondeterministic atomic / look-back baselines, and the CPU oracle
timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl det|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deterministic_floating_point_gb300 import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# workloads: name -> builder returning a dict with
#   step()          one call of the operation (device inputs resident)
#   elems           elements per step (the Gelem/s unit)
#   algo_bytes      algorithmic bytes per step of the dominant kernel and per step
#   dominant        name of the dominant kernel
#   e2e(...)        callables for the host-buffer end-to-end path
#   oracle_sample() CPU oracle on a bounded sample -> (elements, seconds)


def _np_dt(name):
    return {"f32": np.float32, "f64": np.float64}[name]


def _timed_oracle(fn, budget_s=3.0):
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return reps, time.perf_counter() - t0


def build_workload(name, torch, det, dev):
    """Device-resident inputs and the step closures of one workload."""
    tdt = {"f32": torch.float32, "f64": torch.float64}
    dt = "f64" if name.endswith("f64") else "f32"
    code = 0 if dt == "f32" else 1
    npdt = _np_dt(dt)

    if name.startswith("sum"):
        n = workloads.SUM_N if name.startswith("sum_small") else 1 << 28
        x_np = workloads.sum_input(n=n, dtype=npdt)
        x = torch.from_numpy(x_np).to(dev)
        out = torch.empty(1, dtype=tdt[dt], device=dev)
        ws = det.workspace(det.lib().det_sum_workspace_bytes(n, code), dev)
        s = x_np.itemsize
        host_x = torch.from_numpy(x_np).pin_memory()
        host_out = torch.empty(1, dtype=tdt[dt]).pin_memory()

        def step():
            det.det_sum(x, out, workspace=ws)

        def e2e_step():
            x.copy_(host_x, non_blocking=True)
            det.det_sum(x, out, workspace=ws)
            host_out.copy_(out, non_blocking=True)

        def oracle_sample():
            import oracle
            m = min(n, 1 << 26)
            reps, secs = _timed_oracle(lambda: oracle.det_sum(x_np[:m]))
            return m * reps, secs, f"{reps} x det_sum of the first {m} elements, 1 thread"

        return dict(step=step, elems=n, algo_bytes=n * s, step_bytes=n * s, dominant="det_sum",
                    dtype=dt, e2e_step=e2e_step, h2d=n * s, d2h=s, oracle_sample=oracle_sample,
                    config={"workload": f"det_sum n={n} uniform[0,12) {dt} seed 0", "n": n,
                            "l2": "flushed between timed steps"})

    if name.startswith("scan") or name.startswith("segscan"):
        seg = name.startswith("segscan")
        n = workloads.SCAN_SMALL_N if "small" in name else workloads.SCAN_N
        x_np = workloads.scan_input(n=n, dtype=npdt)
        x = torch.from_numpy(x_np).to(dev)
        y = torch.empty_like(x)
        s = x_np.itemsize
        host_x = torch.from_numpy(x_np).pin_memory()
        host_y = torch.empty_like(host_x).pin_memory()
        if seg:
            off_np = workloads.segment_offsets(n)
            off = torch.from_numpy(off_np).to(dev)
            ws = det.workspace(det.lib().det_segmented_scan_workspace_bytes(n, off.numel() - 1, code), dev)

            def step():
                det.det_segmented_scan(x, off, y, workspace=ws)
        else:
            ws = det.workspace(det.lib().det_scan_workspace_bytes(n, code), dev)

            def step():
                det.det_scan(x, y, workspace=ws)

        def e2e_step():
            x.copy_(host_x, non_blocking=True)
            step()
            host_y.copy_(y, non_blocking=True)

        def oracle_sample():
            import oracle
            m = min(n, 1 << 24)
            if seg:
                o = workloads.segment_offsets(m)
                reps, secs = _timed_oracle(lambda: oracle.det_segmented_scan(x_np[:m], o))
            else:
                reps, secs = _timed_oracle(lambda: oracle.det_scan(x_np[:m]))
            return m * reps, secs, f"{reps} x {'segmented ' if seg else ''}scan of the first {m} elements, 1 thread"

        kern = "det_segmented_scan" if seg else "det_scan"
        extra = " segments geometric(mean 4096)" if seg else ""
        return dict(step=step, elems=n, algo_bytes=2 * n * s, step_bytes=2 * n * s, dominant=kern,
                    dtype=dt, e2e_step=e2e_step, h2d=n * s, d2h=n * s, oracle_sample=oracle_sample,
                    config={"workload": f"{kern} forward inclusive n={n} lognormal(0,1) {dt} seed 4{extra}",
                            "n": n, "l2": "inputs and outputs larger than L2; L2 flushed between timed steps"})

    if name.startswith("scatter") or name.startswith("skew"):
        skew = name.startswith("skew")
        if skew:
            values_np, bins_np, out0_np = workloads.skewed_scatter_input(dtype=npdt)
            wdesc = (f"det_scatter_add n={values_np.size} N(0,1) {dt}, Zipf(1.1) bins over {out0_np.size}, "
                     f"5% out of range, seed 3")
        else:
            bin0 = "bin0" in name
            values_np, bins_np, out0_np = workloads.scatter_input(dtype=npdt, all_in_bin0=bin0)
            wdesc = (f"det_scatter_add n={values_np.size} N(0,1) {dt}, "
                     + ("all records in bin 0" if bin0 else f"{out0_np.size} uniform bins") + ", seed 2")
        n, m = values_np.size, out0_np.size
        v = torch.from_numpy(values_np).to(dev)
        b = torch.from_numpy(bins_np).to(dev)
        out = torch.from_numpy(out0_np).to(dev)
        ws = det.workspace(det.lib().det_scatter_add_workspace_bytes(n, m, code), dev)
        s = values_np.itemsize
        host_v = torch.from_numpy(values_np).pin_memory()
        host_b = torch.from_numpy(bins_np).pin_memory()
        host_out = torch.empty_like(out, device="cpu").pin_memory()
        passes = 1 if m <= 1024 else 2

        def step():
            det.det_scatter_add(out, b, v, workspace=ws)

        def e2e_step():
            v.copy_(host_v, non_blocking=True)
            b.copy_(host_b, non_blocking=True)
            det.det_scatter_add(out, b, v, workspace=ws)
            host_out.copy_(out, non_blocking=True)

        def oracle_sample():
            import oracle
            k = min(n, 1 << 22)
            reps, secs = _timed_oracle(lambda: oracle.det_scatter_add(out0_np, bins_np[:k], values_np[:k]))
            return k * reps, secs, f"{reps} x det_scatter_add of the first {k} records, 1 thread"

        # one sort pass reads key + value and writes value (+ key between passes)
        pass_bytes = n * (4 + s + s + (4 if passes > 1 else 0))
        if passes == 1:
            step_bytes = n * (4 + (4 + s) + s + s) + 2 * m * s        # hist, pass, tree, out
        else:
            step_bytes = n * (4 + 2 * (4 + s) + 2 * (4 + s) + 4 + s) + 2 * m * s
        return dict(step=step, elems=n, algo_bytes=pass_bytes, step_bytes=step_bytes, dominant="det_sort_pass",
                    dtype=dt, e2e_step=e2e_step, h2d=n * (4 + s), d2h=m * s, oracle_sample=oracle_sample,
                    config={"workload": wdesc, "n": n, "bins": m, "sort_passes": passes,
                            "l2": "L2 flushed between timed steps"})

    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------


def time_steps(torch, wl, steps, flush, timer_cls=None):
    """Per-step CUDA-event times (ms) with an L2 flush before each step."""
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    kernel_ms = []
    for i in range(steps):
        flush.zero_()
        if timer_cls is not None:
            with timer_cls(64) as kt:
                evs[i][0].record(stream)
                wl["step"]()
                evs[i][1].record(stream)
            kernel_ms.append(kt)
        else:
            evs[i][0].record(stream)
            wl["step"]()
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    kernels = []
    for kt in kernel_ms:
        kernels.append(kt.kernels())
    return times, kernels


def traffic_for(kernel, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on this workload with the current source of the kernel's file."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload, {}).get(kernel)
        if not e:
            return None
        src = os.path.join(ROOT, e["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return e["dram_bytes_per_launch"] if h == e["source_sha"] else None
    except Exception:
        return None


def run_det(args, torch, rank, world):
    from deterministic_floating_point_gb300 import det
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peak, peak_kind = load_peaks()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    wl = build_workload(args.workload, torch, det, dev)
    for _ in range(args.warmup):
        wl["step"]()
    torch.cuda.synchronize()

    launches0 = det.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        times, kernels = time_steps(torch, wl, args.steps, flush, det.KernelTimer)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
    launches = det.launch_count() - launches0
    total_ms = sum(times)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = world * wl["elems"] * args.steps / (total_ms * 1e-3) / 1e9

    # dominant kernel: average launch duration over the timed steps
    per_kernel = {}
    for step_k in kernels:
        for name, ms in step_k:
            per_kernel.setdefault(name, []).append(ms)
    dom = wl["dominant"]
    dom_ms = statistics.mean(per_kernel[dom]) if dom in per_kernel else None
    achieved = wl["algo_bytes"] / (dom_ms * 1e-3) / 1e9 if dom_ms else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": (achieved / peak) if achieved else None,
                "traffic": traffic_for(dom, args.workload), "kernel": dom,
                "kernel_ms": dom_ms, "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                "algo_bytes_per_launch": wl["algo_bytes"],
                "kernel_share": {k: round(sum(v) / total_ms, 4) for k, v in per_kernel.items()}}

    # end to end through host buffers (pinned), same metric
    for _ in range(2):
        wl["e2e_step"]()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        wl["e2e_step"]()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e = {"value": wl["elems"] / (e2e_ms * 1e-3) / 1e9, "unit": "Gelem/s",
           "h2d_bytes_per_step": wl["h2d"], "d2h_bytes_per_step": wl["d2h"], "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        elems, secs, what = wl["oracle_sample"]()
        cpu = {"value": elems / secs / 1e9, "unit": "Gelem/s", "cores": 1, "kind": "oracle",
               "sample": what}

    line = {"metric": "Gelem/s and achieved HBM GB/s (% of GB300 HBM peak) for det sum/scatter/scan",
            "value": value, "unit": "Gelem/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl["dtype"], "data": "synthetic", "config": dict(wl["config"], parallelism=f"replicas{world}"),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk.summary(), "step_ms_min": min(times), "step_ms_median": statistics.median(times),
            "algo_gbs_per_step": wl["step_bytes"] / (ms_per_step * 1e-3) / 1e9}
    return line


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle  # noqa: F401
    wl = build_workload(args.workload, None, None, None) if False else None
    _ = wl
    # The reference arm is the CPU oracle, timed as it stands on the host cores.
    name = args.workload
    t_all = []
    elems = None
    what = None
    for i in range(args.warmup + args.steps):
        e, s, what = ref_sample(name)
        if i >= args.warmup:
            t_all.append(s)
            elems = e
    secs = sum(t_all) / len(t_all)
    v = elems / secs / 1e9
    return {"impl": "reference", "metric": "Gelem/s and achieved HBM GB/s (% of GB300 HBM peak) for det sum/scatter/scan",
            "value": v, "unit": "Gelem/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ref_dtype(name), "data": "synthetic", "config": {"workload": name, "sample": what},
            "cpu_baseline": {"value": v, "unit": "Gelem/s", "cores": 1, "kind": "oracle", "sample": what},
            "e2e": {"value": v, "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def ref_dtype(name):
    return "f64" if name.endswith("f64") else "f32"


def ref_sample(name):
    """One bounded oracle step of the workload: (elements, seconds, description)."""
    import oracle
    npdt = _np_dt(ref_dtype(name))
    if name.startswith("sum"):
        n = 1 << 24
        x = workloads.sum_input(n=n, dtype=npdt)
        t0 = time.perf_counter()
        oracle.det_sum(x)
        return n, time.perf_counter() - t0, f"det_sum of {n} elements"
    if name.startswith("scatter") or name.startswith("skew"):
        k = 1 << 22
        if name.startswith("skew"):
            values, bins, out0 = workloads.skewed_scatter_input(n=k, dtype=npdt)
        else:
            values, bins, out0 = workloads.scatter_input(n=k, dtype=npdt, all_in_bin0="bin0" in name)
        t0 = time.perf_counter()
        oracle.det_scatter_add(out0, bins, values)
        return k, time.perf_counter() - t0, f"{name}: det_scatter_add of {k} records"
    if name.startswith("scan") or name.startswith("segscan"):
        n = 1 << 22
        x = workloads.scan_input(n=n, dtype=npdt)
        t0 = time.perf_counter()
        if name.startswith("segscan"):
            oracle.det_segmented_scan(x, workloads.segment_offsets(n))
        else:
            oracle.det_scan(x)
        return n, time.perf_counter() - t0, f"{name} of {n} elements"
    raise SystemExit(f"unknown workload {name}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="det", choices=["det", "reference"])
    ap.add_argument("--workload", default="scatter")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    line = run_det(args, torch, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
