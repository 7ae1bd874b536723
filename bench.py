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
# GB300's FP64 rate: 1.25 TFLOP/s nominal, an FMA counted as two operations,
# i.e. 0.625 T adds/s -- two FP64 lanes per SM per clock on 152 SMs at 2,070 MHz.
FP64_ADDS_PER_S = 152 * 2 * 2.07e9
FP64_MEASURED = {}     # {"rate": adds/s from the add-only probe, measured once per run}
BLOCK_THREADS = 0      # --block-threads: launch shape of the library calls (never changes the bits)
N_OVERRIDE = 0         # --n: element count of the sum and scan workloads (smaller cases for profiler captures)


def max_over_ranks(torch, value, device, world):
    """The largest of the ranks' values, on every rank (a job takes as long as
    its slowest rank).  One rank: the value itself."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, elems, steps, total_ms):
    """Gelem/s of the whole job: each of the `world` ranks processes `elems`
    elements per step, `steps` steps in `total_ms` (the slowest rank's time)."""
    return world * elems * steps / (total_ms * 1e-3) / 1e9


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


def fingerprint(torch, *tensors):
    """Fingerprint of result bits: SHA-256 of small results; for large ones,
    SHA-256 of per-block weighted sums of the bit patterns (integer
    arithmetic, so any changed element changes some block sum)."""
    import hashlib as _h
    hs = _h.sha256()
    for t in tensors:
        nbytes = t.numel() * t.element_size()
        if nbytes <= (64 << 20):
            hs.update(t.detach().cpu().numpy().tobytes())
            continue
        bits = t.detach().reshape(-1).view(torch.int64 if t.element_size() == 8 else torch.int32)
        k = 8192
        pad = (-bits.numel()) % k
        if pad:
            bits = torch.cat([bits, bits.new_zeros(pad)])
        blocks = bits.view(-1, k)
        w = torch.arange(1, 2 * k, 2, device=t.device, dtype=bits.dtype)
        hs.update(blocks.sum(dim=1, dtype=torch.int64).cpu().numpy().tobytes())
        hs.update((blocks * w).sum(dim=1, dtype=torch.int64).cpu().numpy().tobytes())
    return hs.hexdigest()


def build_workload(name, torch, det, dev):
    """Device-resident inputs and the step closures of one workload."""
    tdt = {"f32": torch.float32, "f64": torch.float64}
    dt = "f64" if name.endswith("f64") else "f32"
    code = 0 if dt == "f32" else 1
    npdt = _np_dt(dt)

    if name.startswith("sum"):
        n = N_OVERRIDE or (workloads.SUM_N if name.startswith("sum_small") else 1 << 28)
        x_np = workloads.sum_input(n=n, dtype=npdt)
        x = torch.from_numpy(x_np).to(dev)
        out = torch.empty(1, dtype=tdt[dt], device=dev)
        ws = det.workspace(det.lib().det_sum_workspace_bytes(n, code), dev)
        s = x_np.itemsize
        host_x = torch.from_numpy(x_np).pin_memory()
        host_out = torch.empty(1, dtype=tdt[dt]).pin_memory()

        def step():
            det.det_sum(x, out, workspace=ws, block_threads=BLOCK_THREADS)

        def e2e_step():
            x.copy_(host_x, non_blocking=True)
            det.det_sum(x, out, workspace=ws)
            host_out.copy_(out, non_blocking=True)

        def oracle_sample():
            import oracle
            m = min(n, 1 << 26)
            reps, secs = _timed_oracle(lambda: oracle.det_sum(x_np[:m]))
            return m * reps, secs, f"{reps} x det_sum of the first {m} elements, 1 thread"

        return dict(state={"x": x, "out": out}, step=step, elems=n, algo_bytes=n * s, step_bytes=n * s,
                    adds=(n - 1) if dt == "f64" else None,
                    dominant="det_sum",
                    dtype=dt, e2e_step=e2e_step, h2d=n * s, d2h=s, oracle_sample=oracle_sample,
                    config={"workload": f"det_sum n={n} uniform[0,12) {dt} seed 0", "n": n,
                            "l2": "flushed between timed steps"})

    if (name.startswith("scan") or name.startswith("segscan")) and name != "scan_i32":
        seg = name.startswith("segscan")
        restart = name.startswith("segscan_restart")
        sflags = (1 if "excl" in name else 0) | (2 if "rev" in name else 0)
        n = N_OVERRIDE or (workloads.SCAN_SMALL_N if "small" in name else workloads.SCAN_N)
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

            gflags = sflags | (det.SCAN_SEGMENT_RESTART if restart else 0)

            def step():
                det.det_segmented_scan(x, off, y, flags=gflags, workspace=ws, block_threads=BLOCK_THREADS)
        else:
            ws = det.workspace(det.lib().det_scan_workspace_bytes(n, code), dev)

            def step():
                det.det_scan(x, y, flags=sflags, workspace=ws, block_threads=BLOCK_THREADS)

        def e2e_step():
            x.copy_(host_x, non_blocking=True)
            step()
            host_y.copy_(y, non_blocking=True)

        def oracle_sample():
            import oracle
            m = min(n, 1 << 24)
            if seg:
                o = workloads.segment_offsets(m)
                reps, secs = _timed_oracle(
                    lambda: oracle.det_segmented_scan(x_np[:m], o, sflags | (4 if restart else 0)))
            else:
                reps, secs = _timed_oracle(lambda: oracle.det_scan(x_np[:m], sflags))
            return m * reps, secs, f"{reps} x {'segmented ' if seg else ''}scan of the first {m} elements, 1 thread"

        kern = ("det_segmented_scan_restart" if restart else "det_segmented_scan") if seg else "det_scan"
        extra = (" segments geometric(mean 4096)" + (", each scanned alone" if restart else "")) if seg else ""
        return dict(state={"x": x, "y": y}, step=step, elems=n, algo_bytes=2 * n * s, step_bytes=2 * n * s,
                    adds=(2 * n) if dt == "f64" else None,
                    dominant=kern,
                    dtype=dt, e2e_step=e2e_step, h2d=n * s, d2h=n * s, oracle_sample=oracle_sample,
                    config={"workload": f"{kern} {('reverse' if sflags & 2 else 'forward')} "
                                        f"{('exclusive' if sflags & 1 else 'inclusive')} n={n} lognormal(0,1) {dt} "
                                        f"seed 4{extra}", "flags": sflags,
                            "n": n, "l2": "inputs and outputs larger than L2; L2 flushed between timed steps"})

    if name in ("scatter_sub", "scatter_min", "scatter_max"):
        op = name.split("_")[1]
        values_np, bins_np, out0_np = workloads.scatter_input(dtype=npdt)
        n, m = values_np.size, out0_np.size
        v = torch.from_numpy(values_np).to(dev)
        b = torch.from_numpy(bins_np).to(dev)
        out = torch.from_numpy(out0_np).to(dev)
        s = values_np.itemsize
        fn = {"sub": det.det_scatter_sub, "min": det.det_scatter_min, "max": det.det_scatter_max}[op]
        nbytes = (det.lib().det_scatter_add_workspace_bytes(n, m, code) if op == "sub"
                  else det.lib().det_scatter_minmax_workspace_bytes(m, code))
        ws = det.workspace(nbytes, dev)
        host_v = torch.from_numpy(values_np).pin_memory()
        host_b = torch.from_numpy(bins_np).pin_memory()
        host_out = torch.empty_like(out, device="cpu").pin_memory()

        def step():
            fn(out, b, v, workspace=ws, block_threads=BLOCK_THREADS)

        def e2e_step():
            v.copy_(host_v, non_blocking=True)
            b.copy_(host_b, non_blocking=True)
            fn(out, b, v, workspace=ws)
            host_out.copy_(out, non_blocking=True)

        def oracle_sample():
            import oracle
            k = min(n, 1 << 22)
            f = {"sub": oracle.det_scatter_sub, "min": oracle.det_scatter_min, "max": oracle.det_scatter_max}[op]
            reps, secs = _timed_oracle(lambda: f(out0_np, bins_np[:k], values_np[:k]))
            return k * reps, secs, f"{reps} x det_scatter_{op} of the first {k} records, 1 thread"

        if op == "sub":   # the scatter-add path: a sort pass dominates
            dom, algo = "det_sort_pass", n * (4 + s + s)
            step_bytes = n * (4 + (4 + s) + s + s) + 2 * m * s
        else:             # one pass over the records, keys in shared memory
            dom, algo = "det_minmax_scatter", n * (4 + s)
            step_bytes = n * (4 + s) + 2 * m * s
        return dict(state={"out": out, "out0": torch.from_numpy(out0_np).to(dev), "b": b, "v": v}, step=step,
                    elems=n, algo_bytes=algo, step_bytes=step_bytes, dominant=dom,
                    dtype=dt, e2e_step=e2e_step, h2d=n * (4 + s), d2h=m * s, oracle_sample=oracle_sample,
                    config={"workload": f"det_scatter_{op} n={n} N(0,1) {dt}, {m} uniform bins, seed 2", "n": n,
                            "bins": m, "l2": "L2 flushed between timed steps"})

    if name == "scatter_vec3":
        values_np, bins_np, out0_np = workloads.vec_scatter_input(dtype=npdt)
        n, W = values_np.shape
        m = out0_np.shape[0]
        v = torch.from_numpy(values_np).to(dev)
        b = torch.from_numpy(bins_np).to(dev)
        out = torch.from_numpy(out0_np).to(dev)
        s = values_np.itemsize
        ws = det.workspace(det.lib().det_scatter_add_vec_workspace_bytes(n, m, W, code), dev)
        host_v = torch.from_numpy(values_np).pin_memory()
        host_b = torch.from_numpy(bins_np).pin_memory()
        host_out = torch.empty_like(out, device="cpu").pin_memory()

        def step():
            det.det_scatter_add_vec(out, b, v, workspace=ws, block_threads=BLOCK_THREADS)

        def e2e_step():
            v.copy_(host_v, non_blocking=True)
            b.copy_(host_b, non_blocking=True)
            det.det_scatter_add_vec(out, b, v, workspace=ws)
            host_out.copy_(out, non_blocking=True)

        def oracle_sample():
            import oracle
            k = min(n, 1 << 21)
            reps, secs = _timed_oracle(lambda: oracle.det_scatter_add_rows(out0_np, bins_np[:k], values_np[:k]))
            return k * W * reps, secs, f"{reps} x vec{W} scatter of the first {k} records, 1 thread"

        # count (key in), pass (key and whole record in, W components out), W trees (W components in):
        # the one-pass sort of records of at most 16 bytes carries the records itself
        step_bytes = n * (4 + 4 + 2 * W * s + W * s) + 2 * m * W * s
        return dict(state={"out": out, "out0": torch.from_numpy(out0_np).to(dev), "b": b, "v": v}, step=step,
                    elems=n * W, algo_bytes=n * (4 + 2 * W * s), step_bytes=step_bytes, dominant="det_sort_pass",
                    dtype=dt, e2e_step=e2e_step, h2d=n * (4 + W * s), d2h=m * W * s, oracle_sample=oracle_sample,
                    config={"workload": f"det_scatter_add_vec n={n} vec{W} N(0,1) {dt}, {m} uniform bins, seed 6",
                            "n": n, "width": W, "bins": m, "l2": "L2 flushed between timed steps"})

    if name == "gather_grad":
        # the pages' backward example at the row workload's sizes: out = table[idx] forward,
        # table.grad[idx] += grad_out backward (det_gather_rows, then det_scatter_add_rows)
        from deterministic_floating_point_gb300 import autograd
        gout_np, idx_np, table_np = workloads.rows_input(dtype=npdt)
        M, W = gout_np.shape
        R = table_np.shape[0]
        table = torch.from_numpy(table_np).to(dev).requires_grad_(True)
        idx = torch.from_numpy(idx_np).to(dev)
        gout = torch.from_numpy(gout_np).to(dev)
        s = gout_np.itemsize
        host_g = torch.from_numpy(gout_np).pin_memory()
        host_grad = torch.empty_like(table, device="cpu").pin_memory()

        def step():
            table.grad = None
            autograd.gather(table, idx).backward(gout)

        def e2e_step():
            gout.copy_(host_g, non_blocking=True)
            step()
            host_grad.copy_(table.grad, non_blocking=True)

        def oracle_sample():
            import oracle
            k = 1 << 17
            z = np.zeros_like(table_np)

            def f():
                oracle.det_gather_rows(table_np, idx_np[:k])
                oracle.det_scatter_add_rows(z, idx_np[:k], gout_np[:k])
            reps, secs = _timed_oracle(f)
            return k * W * reps, secs, f"{reps} x gather + adjoint scatter of the first {k} rows, 1 thread"

        # forward: read table rows, write out; backward: read grad_out, table.grad in/out, sorted ids
        bwd_bytes = M * W * s + 2 * R * W * s + 4 * M
        return dict(state={"table": table, "idx": idx, "gout": gout}, step=step, elems=M * W, algo_bytes=bwd_bytes,
                    step_bytes=2 * M * W * s + bwd_bytes, dominant="det_rows", dtype=dt, e2e_step=e2e_step,
                    h2d=M * W * s, d2h=R * W * s, oracle_sample=oracle_sample,
                    config={"workload": f"autograd gather of {M} rows x {W} {dt} from a {R}-row table + backward "
                                        "(rows workload inputs, seed 5)", "rows": M, "table_rows": R, "row_len": W,
                            "l2": "L2 flushed between timed steps"})

    if name == "scan_i32":
        n = N_OVERRIDE or workloads.SCAN_N
        # count -> exclusive scan -> write: 0/1 flags of the scan workload's values
        x_np = (workloads.scan_input(n=n, dtype=np.float32) > 1.0).astype(np.int32)
        x = torch.from_numpy(x_np).to(dev)
        y = torch.empty_like(x)
        tot = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = det.workspace(det.lib().det_scan_i32_workspace_bytes(n), dev)
        host_x = torch.from_numpy(x_np).pin_memory()
        host_y = torch.empty_like(host_x).pin_memory()

        def step():
            det.det_scan_i32(x, y, exclusive=True, total_out=tot, workspace=ws, block_threads=BLOCK_THREADS)

        def e2e_step():
            x.copy_(host_x, non_blocking=True)
            step()
            host_y.copy_(y, non_blocking=True)

        def oracle_sample():
            import oracle
            k = min(n, 1 << 24)
            reps, secs = _timed_oracle(lambda: oracle.det_scan_i32(x_np[:k], exclusive=True))
            return k * reps, secs, f"{reps} x exclusive int32 scan of the first {k} flags, 1 thread"

        return dict(state={"x": x, "y": y}, step=step, elems=n, algo_bytes=8 * n, step_bytes=8 * n,
                    dominant="det_iscan_tiles", dtype="i32", e2e_step=e2e_step, h2d=4 * n, d2h=4 * n,
                    oracle_sample=oracle_sample,
                    config={"workload": f"det_scan_i32 exclusive n={n} flags (lognormal(0,1) seed 4 > 1)", "n": n,
                            "l2": "inputs and outputs larger than L2; L2 flushed between timed steps"})

    if name.startswith("slot_alloc"):
        multi = name == "slot_alloc_multi"
        if multi:   # 2^24 reservations spread over 1,024 counters (the scatter bins)
            _, idx_np, _ = workloads.scatter_input(dtype=np.float32)
            C = workloads.SCATTER_BINS
            wdesc = f"det_slot_alloc n={idx_np.size} one slot each, {C} uniform counters, seed 2"
        else:       # the pages' counter benchmark: slot = atomic_add(count, 0, 1), 1,048,576 writes
            idx_np = np.zeros(1 << 20, np.int32)
            C = 1
            wdesc = f"det_slot_alloc n={idx_np.size} one slot each, one counter (count.zero_() before)"
        n = idx_np.size
        idx = torch.from_numpy(idx_np).to(dev)
        ctr = torch.zeros(C, dtype=torch.int32, device=dev)
        slots = torch.empty(n, dtype=torch.int32, device=dev)
        ws = det.workspace(det.lib().det_slot_alloc_workspace_bytes(n, C), dev)
        host_idx = torch.from_numpy(idx_np).pin_memory()
        host_slots = torch.empty_like(host_idx).pin_memory()

        def step():
            det.det_slot_alloc(ctr, idx, slot_out=slots, workspace=ws, block_threads=BLOCK_THREADS)

        def e2e_step():
            idx.copy_(host_idx, non_blocking=True)
            step()
            host_slots.copy_(slots, non_blocking=True)

        def oracle_sample():
            import oracle
            k = min(n, 1 << 22)
            reps, secs = _timed_oracle(lambda: oracle.det_slot_alloc(np.zeros(C, np.int32), idx_np[:k]))
            return k * reps, secs, f"{reps} x det_slot_alloc of the first {k} reservations, 1 thread"

        dom = "det_sort_pass" if multi else "det_iscan_tiles"
        algo = n * (4 + 4) if not multi else n * (4 + 4)   # index in, slot / sorted index out
        return dict(state={"ctr": ctr, "idx": idx, "slots": slots, "C": C}, step=step, elems=n, algo_bytes=algo,
                    step_bytes=n * 8, dominant=dom, dtype="i32", e2e_step=e2e_step, h2d=4 * n, d2h=4 * n,
                    oracle_sample=oracle_sample,
                    config={"workload": wdesc, "n": n, "counters": C, "l2": "L2 flushed between timed steps"})

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
            det.det_scatter_add(out, b, v, workspace=ws, block_threads=BLOCK_THREADS)

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
        return dict(state={"out": out, "out0": torch.from_numpy(out0_np).to(dev), "b": b, "v": v}, step=step,
                    elems=n, algo_bytes=pass_bytes, step_bytes=step_bytes, dominant="det_sort_pass",
                    dtype=dt, e2e_step=e2e_step, h2d=n * (4 + s), d2h=m * s, oracle_sample=oracle_sample,
                    config={"workload": wdesc, "n": n, "bins": m, "sort_passes": passes,
                            "l2": "L2 flushed between timed steps"})

    if name.startswith("rows"):
        ordered = name.startswith("rows_ordered")
        src_np, idx_np, dst0_np = workloads.rows_input(dtype=npdt)
        M, W = src_np.shape
        R = dst0_np.shape[0]
        src = torch.from_numpy(src_np).to(dev)
        idx = torch.from_numpy(idx_np).to(dev)
        dst = torch.from_numpy(dst0_np).to(dev)
        prev = torch.empty_like(src)
        ws = det.workspace(det.lib().det_scatter_add_rows_workspace_bytes(M, R, W, code), dev)
        s = src_np.itemsize
        host_src = torch.from_numpy(src_np).pin_memory()
        host_idx = torch.from_numpy(idx_np).pin_memory()
        host_prev = torch.empty_like(host_src).pin_memory()

        def step():
            det.det_scatter_add_rows(dst, idx, src, prev_out=prev, workspace=ws, block_threads=BLOCK_THREADS,
                                     ordered=ordered)

        def e2e_step():
            src.copy_(host_src, non_blocking=True)
            idx.copy_(host_idx, non_blocking=True)
            det.det_scatter_add_rows(dst, idx, src, prev_out=prev, workspace=ws, ordered=ordered)
            host_prev.copy_(prev, non_blocking=True)

        def oracle_sample():
            import oracle
            k = 1 << 17
            f = oracle.det_scatter_add_rows_ordered if ordered else oracle.det_scatter_add_rows
            reps, secs = _timed_oracle(lambda: f(dst0_np, idx_np[:k], src_np[:k]))
            return k * W * reps, secs, f"{reps} x row scatter of the first {k} source rows, 1 thread"

        rows_bytes = 2 * M * W * s + 2 * R * W * s + 4 * M    # src in, prev out, dst in/out, sorted ids
        return dict(state={"dst": dst, "dst0": torch.from_numpy(dst0_np).to(dev), "idx": idx, "src": src,
                           "prev": prev}, step=step, elems=M * W, algo_bytes=rows_bytes,
                    step_bytes=rows_bytes + 12 * M,
                    dominant="det_rows_ordered" if ordered else "det_rows", dtype=dt, e2e_step=e2e_step,
                    h2d=M * W * s + 4 * M, d2h=M * W * s, oracle_sample=oracle_sample,
                    config={"workload": f"det_scatter_add_rows{'_ordered' if ordered else ''} src {M}x{W} N(0,1) "
                                        f"{dt}, rows uniform over {R}, prev returned, seed 5",
                            "src_rows": M, "dst_rows": R, "row_len": W,
                            "l2": "inputs larger than L2; L2 flushed between timed steps"})

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


def add_checks(name, wl, torch, det, dev):
    """Attach closures for determinism counting: det_once() and base_once()
    run the deterministic call / its nondeterministic baseline from the same
    initial state and return a fingerprint of the result bits."""
    st = wl["state"]
    if name.startswith("sum"):
        x, out = st["x"], st["out"]
        bout = torch.empty_like(out)
        wl["det_once"] = lambda: (wl["step"](), fingerprint(torch, out))[1]
        wl["base_once"] = lambda: (det.atomic_sum(x, bout), fingerprint(torch, bout))[1]
        wl["base_step"] = lambda: det.atomic_sum(x, bout)
        wl["base_name"] = "atomic_sum"
    elif name in ("scatter_sub", "scatter_min", "scatter_max"):
        out, out0, b, v = st["out"], st["out0"], st["b"], st["v"]

        def d1():
            out.copy_(out0)
            wl["step"]()
            return fingerprint(torch, out)
        wl["det_once"] = d1
        if name == "scatter_sub":   # the atomic form: atomicAdd of the negated values
            nv = -v

            def b1():
                out.copy_(out0)
                det.atomic_scatter_add(out, b, nv)
                return fingerprint(torch, out)
            wl["base_once"] = b1
            wl["base_step"] = lambda: det.atomic_scatter_add(out, b, nv)
            wl["base_name"] = "atomic_scatter_add of -values"
    elif name == "gather_grad":
        table = st["table"]
        wl["det_once"] = lambda: (wl["step"](), fingerprint(torch, table.grad))[1]
    elif name == "scan_i32":
        y = st["y"]
        wl["det_once"] = lambda: (wl["step"](), fingerprint(torch, y))[1]
    elif name.startswith("slot_alloc"):
        ctr, idx, slots = st["ctr"], st["idx"], st["slots"]
        bslots = torch.empty_like(slots)

        def d1():
            ctr.zero_()
            wl["step"]()
            return fingerprint(torch, slots, ctr)

        def b1():
            ctr.zero_()
            det.atomic_slot_alloc(ctr, idx, bslots)
            return fingerprint(torch, bslots, ctr)
        wl["det_once"], wl["base_once"] = d1, b1
        wl["base_step"] = lambda: det.atomic_slot_alloc(ctr, idx, bslots)
        wl["base_name"] = "atomic_slot_alloc (atomicAdd slots)"
    elif name == "scatter_vec3":
        out, out0 = st["out"], st["out0"]

        def d1():
            out.copy_(out0)
            wl["step"]()
            return fingerprint(torch, out)
        wl["det_once"] = d1
    elif name.startswith("scatter") or name.startswith("skew"):
        out, out0, b, v = st["out"], st["out0"], st["b"], st["v"]

        def d1():
            out.copy_(out0)
            wl["step"]()
            return fingerprint(torch, out)

        def b1():
            out.copy_(out0)
            det.atomic_scatter_add(out, b, v)
            return fingerprint(torch, out)
        wl["det_once"], wl["base_once"] = d1, b1
        wl["base_step"] = lambda: det.atomic_scatter_add(out, b, v)
        wl["base_name"] = "atomic_scatter_add"
    elif name.startswith("rows"):
        dst, dst0, idx, src, prev = st["dst"], st["dst0"], st["idx"], st["src"], st["prev"]

        def d1():
            dst.copy_(dst0)
            wl["step"]()
            return fingerprint(torch, dst, prev)

        def b1():
            dst.copy_(dst0)
            det.atomic_scatter_add_rows(dst, idx, src, prev_out=prev)
            return fingerprint(torch, dst, prev)
        wl["det_once"], wl["base_once"] = d1, b1
        wl["base_step"] = lambda: det.atomic_scatter_add_rows(dst, idx, src, prev_out=prev)
        wl["base_name"] = "atomic_scatter_add_rows"
    elif name.startswith("scan") or name.startswith("segscan"):
        x, y = st["x"], st["y"]
        yb = torch.empty_like(y)
        bws = det.workspace(det.lib().det_dlb_scan_workspace_bytes(x.numel(), 0 if x.dtype == torch.float32 else 1),
                            dev)
        wl["det_once"] = lambda: (wl["step"](), fingerprint(torch, y))[1]
        if name.startswith("scan"):
            wl["base_once"] = lambda: (det.dlb_scan(x, yb, bws), fingerprint(torch, yb))[1]
            wl["base_step"] = lambda: det.dlb_scan(x, yb, bws)
            wl["base_name"] = "dlb_scan (unmodified look-back)"
    return wl


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


# Every configuration of the hot path at each dtype it names (a workload name
# ending in _f64 is the f64 arm, any other the f32 arm), then the next rows.
OPS = ["sum", "sum_f64", "sum_small", "sum_small_f64",
       "scatter", "scatter_f64", "scatter_bin0", "scatter_bin0_f64",
       "skew", "skew_f64",
       "scan", "scan_f64", "scan_excl", "scan_rev", "scan_rev_excl", "scan_rev_excl_f64",
       "scan_small", "scan_small_f64", "segscan", "segscan_f64",
       "rows", "rows_f64",
       "scatter_sub", "scatter_min", "scatter_max", "scan_i32", "slot_alloc", "slot_alloc_multi", "scatter_vec3",
       "rows_ordered", "gather_grad", "segscan_restart", "segscan_restart_f64"]


def measure_op(name, torch, det, dev, flush, steps, runs, peak):
    """One workload: device time per step, dominant-kernel roofline, the
    baseline's time, and distinct result fingerprints over repeated runs."""
    wl = add_checks(name, build_workload(name, torch, det, dev), torch, det, dev)
    for _ in range(3):
        wl["step"]()
    torch.cuda.synchronize()
    times, _ = time_steps(torch, wl, steps, flush, None)                    # the call, no per-kernel hooks
    ktimes, kernels = time_steps(torch, wl, steps, flush, det.KernelTimer)  # the kernels, separately
    per_kernel = {}
    for step_k in kernels:
        for kname, ms in step_k:
            per_kernel.setdefault(kname, []).append(ms)
    dom = wl["dominant"]
    dom_ms = statistics.mean(per_kernel[dom]) if dom in per_kernel else None
    ms = statistics.mean(times)
    res = {"workload": wl["config"]["workload"], "dtype": wl["dtype"], "Gelem_s": wl["elems"] / (ms * 1e-3) / 1e9,
           "ms_per_step": ms, "step_GB_s": wl["step_bytes"] / (ms * 1e-3) / 1e9,
           "kernel": dom, "kernel_ms": dom_ms,
           "kernel_GB_s": (wl["algo_bytes"] / (dom_ms * 1e-3) / 1e9) if dom_ms else None,
           "kernel_frac_of_peak": (wl["algo_bytes"] / (dom_ms * 1e-3) / 1e9 / peak) if dom_ms else None,
           "kernel_share": {k: round(sum(v) / sum(ktimes), 4) for k, v in per_kernel.items()}}
    if wl.get("adds") and dom_ms:
        res["kernel_Gadd_s"] = wl["adds"] / (dom_ms * 1e-3) / 1e9
        res["kernel_frac_of_fp64_add_peak"] = wl["adds"] / (dom_ms * 1e-3) / FP64_ADDS_PER_S
        if FP64_MEASURED.get("rate"):
            res["kernel_frac_of_measured_fp64_add_rate"] = wl["adds"] / (dom_ms * 1e-3) / FP64_MEASURED["rate"]
    res["distinct_results_det"] = len({wl["det_once"]() for _ in range(runs)})
    if "base_once" in wl:
        for _ in range(2):
            wl["base_step"]()
        torch.cuda.synchronize()
        bt = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            wl["base_step"]()
            e1.record()
            bt.append((e0, e1))
        torch.cuda.synchronize()
        bms = statistics.mean(a.elapsed_time(b) for a, b in bt)
        res["baseline"] = {"name": wl["base_name"], "ms_per_step": bms,
                           "Gelem_s": wl["elems"] / (bms * 1e-3) / 1e9,
                           "det_over_baseline_time": ms / bms,
                           "distinct_results": len({wl["base_once"]() for _ in range(runs)})}
    del wl
    torch.cuda.empty_cache()
    return res


def measure_add_rate(torch, det, dev, dtype):
    """The device's add rate in `dtype` (adds/s): the add-only probe launch,
    timed with CUDA events on the current stream, best of 5."""
    sink = torch.zeros(1, dtype=dtype, device=dev)
    stream = torch.cuda.current_stream()
    best = 0.0
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        adds = det.add_rate_probe(dtype, 4096, sink)
        e1.record(stream)
        e1.synchronize()
        best = max(best, adds / (e0.elapsed_time(e1) * 1e-3))
    return best


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
        # the headline steps run without the per-kernel event hooks (they add
        # host work to every launch); a second, separate pass times the kernels
        times, _ = time_steps(torch, wl, args.steps, flush, None)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
    launches = det.launch_count() - launches0
    ktimes, kernels = time_steps(torch, wl, args.steps, flush, det.KernelTimer)
    total_ms = max_over_ranks(torch, sum(times), dev, world)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, wl["elems"], args.steps, total_ms)
    step_bytes = wl["step_bytes"]

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
                "kernel_share": {k: round(sum(v) / sum(ktimes), 4) for k, v in per_kernel.items()}}
    adds = wl.get("adds")
    if adds and dom_ms and adds / FP64_ADDS_PER_S > wl["algo_bytes"] / (peak * 1e9):
        # the FP64 add rate, not HBM, bounds this kernel: report against it
        hbm = {k: roofline[k] for k in ("achieved", "peak", "unit", "frac", "peak_kind")}
        a = adds / (dom_ms * 1e-3) / 1e9
        measured = measure_add_rate(torch, det, dev, torch.float64)
        roofline.update({"bound": "alu", "achieved": a, "peak": FP64_ADDS_PER_S / 1e9, "unit": "Gadd/s",
                         "frac": a * 1e9 / FP64_ADDS_PER_S,
                         "peak_kind": "nominal FP64 add rate (1.25 TFLOP/s, FMA = 2: 152 SMs x 2 adds x 2.07 GHz)",
                         "measured_peak": measured / 1e9, "frac_of_measured": a * 1e9 / measured,
                         "algo_adds_per_launch": adds, "hbm": hbm})

    # end to end through host buffers (pinned), same metric
    # (whole job: every rank's steps, timed from a common barrier, the slowest rank's time)
    for _ in range(2):
        wl["e2e_step"]()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        wl["e2e_step"]()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_total = max_over_ranks(torch, e0.elapsed_time(e1), dev, world)
    e2e = {"value": whole_job_rate(world, wl["elems"], args.steps, e2e_total), "unit": "Gelem/s",
           "h2d_bytes_per_step": wl["h2d"], "d2h_bytes_per_step": wl["d2h"], "ms_per_step": e2e_total / args.steps}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        elems, secs, what = wl["oracle_sample"]()
        cpu = dict({"value": elems / secs / 1e9, "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                    "sample": what}, **host_cpu())

    dtype, config = wl["dtype"], dict(wl["config"], parallelism=f"replicas{world}")
    ops = {}
    if args.ops and rank == 0:
        FP64_MEASURED["rate"] = measure_add_rate(torch, det, dev, torch.float64)
        FP64_MEASURED["f32_rate"] = measure_add_rate(torch, det, dev, torch.float32)
        # the headline workload's own determinism count and baseline, then
        # every other workload of the hot path, measured the same way
        add_checks(args.workload, wl, torch, det, dev)
        head = {"distinct_results_det": len({wl["det_once"]() for _ in range(args.runs)})}
        if "base_once" in wl:
            head["baseline"] = {"name": wl["base_name"],
                                "distinct_results": len({wl["base_once"]() for _ in range(args.runs)})}
        ops[args.workload] = head
        del wl
        torch.cuda.empty_cache()
        for name in OPS:
            if name != args.workload:
                ops[name] = measure_op(name, torch, det, dev, flush, max(3, min(args.steps, 5)), args.runs, peak)

    line = {"metric": "Gelem/s and achieved HBM GB/s (% of GB300 HBM peak) for det sum/scatter/scan",
            "value": value, "unit": "Gelem/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype, "data": "synthetic", "config": config,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk.summary(), "step_ms_min": min(times), "step_ms_median": statistics.median(times),
            "algo_gbs_per_step": step_bytes / (ms_per_step * 1e-3) / 1e9, "ops": ops}
    if FP64_MEASURED:
        line["add_rate_probe_Gadd_s"] = {"f64": FP64_MEASURED["rate"] / 1e9, "f32": FP64_MEASURED["f32_rate"] / 1e9,
                                         "f64_nominal": FP64_ADDS_PER_S / 1e9}
    return line


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle  # noqa: F401
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
            "cpu_baseline": dict({"value": v, "unit": "Gelem/s", "cores": 1, "kind": "oracle", "sample": what},
                                 **host_cpu()),
            "e2e": {"value": v, "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def host_cpu():
    """The host the oracle ran on: logical CPU count and model name."""
    info = {"nproc": os.cpu_count()}
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu part")):
                    model = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    info["cpu_model"] = model
    return info


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
    if name.startswith("rows"):
        k = 1 << 16
        src, idx, dst0 = workloads.rows_input(src_rows=k, dtype=npdt)
        t0 = time.perf_counter()
        oracle.det_scatter_add_rows(dst0, idx, src)
        return k * src.shape[1], time.perf_counter() - t0, f"det_scatter_add_rows of {k} source rows x 64"
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
        fl = (1 if "excl" in name else 0) | (2 if "rev" in name else 0)
        if name.startswith("segscan"):
            oracle.det_segmented_scan(x, workloads.segment_offsets(n), fl | (4 if "restart" in name else 0))
        else:
            oracle.det_scan(x, fl)
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
    ap.add_argument("--block-threads", type=int, default=0)
    ap.add_argument("--n", type=int, default=0,
                    help="element count of the sum and scan workloads (default: the configured size)")
    ap.add_argument("--no-ops", dest="ops", action="store_false",
                    help="skip the other workloads measured beside the headline one")
    ap.add_argument("--runs", type=int, default=10, help="repeated runs for the distinct-result counts")
    args = ap.parse_args()
    global BLOCK_THREADS, N_OVERRIDE
    BLOCK_THREADS = args.block_threads
    N_OVERRIDE = args.n
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
