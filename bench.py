"""Benchmark of the isotonic fit on one GB300 (or N replicas under torchrun).

Default workload: one row of 10,000,000 float32 values, y = linspace(0, 3, n)
+ N(0, 1) (seed 0), unit weights, non-decreasing fit.  One step is one call of
iso_fit over that row (chunk hulls, segment-list merge tree, expansion).  The
input (40 MB) and the fit (40 MB) fit in L2, so L2 is flushed (a 256 MB write)
before every timed step, outside the timed interval; each step is timed with
CUDA events on the launching stream.

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle instead
(the reference arm), on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "isotonic fit elements/s (1x10^7 row; batched rows) and HBM GB/s vs GB300 peak"
UNIT = "elements/s"
WORKLOAD = "row1e7"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cross_rank_max(x, device):
    """The largest x over the ranks of the default process group (x itself
    with no group): the job's step time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(elements_per_rank, world, ms_max):
    """Whole-job throughput: every rank processed its own copy of the
    workload (weak scaling) in at most ms_max per step."""
    return world * elements_per_rank / (ms_max * 1e-3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


WORKLOAD_TEXT = {
    "row1e7": "1 row x 10,000,000 fp32, y = linspace(0,3,n) + N(0,1) (seed 0), unit weights, "
              "non-decreasing fit",
    "row65k": "1 row x 65,536 fp32, y = linspace(0,3,n) + N(0,1) (seed 0), unit weights, "
              "non-decreasing fit",
    "batch4096x1024": "4,096 rows x 1,024 fp32, y = linspace(0,3,n) + N(0,1) (seed 0), unit "
                      "weights, non-decreasing fit",
    "dense16x4m": "16 rows x 4,194,304 fp32, y = sort(U(0,1)) + 1e-7 i (fp64, then fp32), "
                  "w ~ U(0.5, 2), non-decreasing fit",
    "softrank1024x8192": "1,024 rows x 8,192 fp32 soft-rank rows (theta ~ N(0,1) sorted "
                         "decreasing, eps = 1), unit weights, non-increasing fit",
}


def workload_desc(W):
    return {
        "workload": WORKLOAD_TEXT[W.name],
        "name": W.name, "rows": W.rows, "n": W.n, "weighted": W.weighted,
        "increasing": W.increasing,
        "l2": "flushed before every timed step (256 MB write outside the timed interval)",
    }


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() in ("active", "1", "0x1"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# traffic figure from the committed ncu summary, valid only for the current source
# ---------------------------------------------------------------------------
def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "convex_hull_pava_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload, kernel):
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload, {}).get(kernel)
        if e and e.get("source_hash") == kernel_source_hash():
            return float(e["bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def time_oracle(W, budget_s=10.0, max_reps=200):
    import oracle
    import numpy as np
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.pava(W.y, W.w, W.increasing)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    per = el / reps
    return {"value": W.elements / per, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} full passes of the fp64 PAVA oracle over the {W.rows}x{W.n} "
                      f"workload, one thread, {el:.1f} s"}


def host_cpu():
    """os.cpu_count() and the CPU's model as /proc/cpuinfo names it."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
        for key in ("model name", "Model", "Hardware"):
            hit = [l.split(":", 1)[1].strip() for l in info if l.startswith(key)]
            if hit:
                model = hit[0]
                break
        else:
            imp = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")]
            part = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")]
            if imp and part:
                model = f"implementer {imp[0]}, part {part[0]}"
    except OSError:
        pass
    return {"cpu_count": os.cpu_count(), "cpu_model": model}


def _oracle_rows_worker(shm_y, shm_w, shape, increasing, a, b):
    import numpy as np
    from multiprocessing import shared_memory
    import oracle
    sy = shared_memory.SharedMemory(name=shm_y)
    y = np.ndarray(shape, dtype=np.float32, buffer=sy.buf)
    w = None
    if shm_w:
        sw = shared_memory.SharedMemory(name=shm_w)
        w = np.ndarray(shape, dtype=np.float32, buffer=sw.buf)
    t0 = time.perf_counter()
    oracle.pava(y[a:b], None if w is None else w[a:b], increasing)
    dt = time.perf_counter() - t0
    sy.close()
    if shm_w:
        sw.close()
    return dt


def time_oracle_all_cores(W, pool, cores):
    """The oracle over every row of a batched workload, one row per task across
    the host's cores (rows read from shared memory), after one untimed pass."""
    import numpy as np
    from multiprocessing import shared_memory
    need = W.y.nbytes + (0 if W.w is None else W.w.nbytes)
    try:
        st = os.statvfs("/dev/shm")
        free = st.f_bavail * st.f_frsize
    except OSError:
        free = 0
    if free < 2 * need:
        return {"unavailable": f"/dev/shm has {free} bytes free, {need} needed"}
    sy = shared_memory.SharedMemory(create=True, size=W.y.nbytes)
    np.ndarray(W.y.shape, dtype=np.float32, buffer=sy.buf)[...] = W.y
    sw = None
    if W.w is not None:
        sw = shared_memory.SharedMemory(create=True, size=W.w.nbytes)
        np.ndarray(W.w.shape, dtype=np.float32, buffer=sw.buf)[...] = W.w
    try:
        per = max(1, W.rows // (4 * cores))
        tasks = [(sy.name, sw.name if sw else "", W.y.shape, W.increasing, a, min(a + per, W.rows))
                 for a in range(0, W.rows, per)]
        pool.starmap(_oracle_rows_worker, tasks)
        reps, t0 = 0, time.perf_counter()
        while True:
            pool.starmap(_oracle_rows_worker, tasks)
            reps += 1
            el = time.perf_counter() - t0
            if el >= 2.0 or reps >= 50:
                break
        el /= reps
    finally:
        sy.close(); sy.unlink()
        if sw:
            sw.close(); sw.unlink()
    return {"value": W.elements / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"all {W.rows} rows of {W.n}, {len(tasks)} tasks of up to {per} rows over "
                      f"{cores} processes, mean of {reps} passes after an untimed one "
                      f"({el:.3f} s per pass)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from convex_hull_pava_gb300 import workloads as wl
    W = wl.make(getattr(args, "workload", WORKLOAD))
    import oracle
    oracle.build()
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.pava(W.y, W.w, W.increasing)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    per = sum(times) / len(times)
    val = W.elements / per
    cb = {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
          "sample": f"{len(times)} timed full passes over the {W.rows}x{W.n} workload, one thread"}
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(W), "cpu_baseline": cb,
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def copy_control(name, make, dev, flush, stream):
    """Median per-stage times (CUDA events around each kernel) of iso_fit and of
    the materialised-copy control on one workload."""
    import numpy as np
    import torch
    import convex_hull_pava_gb300 as chp
    yh, wh, inc = make()
    y = torch.from_numpy(np.atleast_2d(yh)).to(dev)
    w = None if wh is None else torch.from_numpy(np.atleast_2d(wh)).to(dev)
    rows, n = y.shape
    o = torch.empty_like(y)
    b = torch.empty(y.shape, dtype=torch.uint8, device=dev)
    wa = torch.empty(max(chp.iso_fit_workspace_bytes(rows, n, w is not None), 1), dtype=torch.uint8, device=dev)
    wc = torch.empty(max(chp.iso_fit_copy_control_workspace_bytes(rows, n, w is not None), 1),
                     dtype=torch.uint8, device=dev)
    out = {}
    for tag, f in (("segment_lists", lambda: chp.iso_fit(y, w, inc, out=o, blocks=b, workspace=wa, stream=stream)),
                   ("control", lambda: chp.iso_fit_copy_control(y, w, inc, out=o, blocks=b, workspace=wc,
                                                                stream=stream))):
        f()
        chp.profile_enable(True)
        stages, tot = {}, []
        for _ in range(7):
            flush.zero_()
            f()
            r = chp.profile_read()
            for nm, ms in r:
                stages.setdefault(nm, []).append(ms)
            tot.append(sum(ms for _, ms in r))
        chp.profile_enable(False)
        st = {k: float(np.median(v)) for k, v in stages.items()}
        merge = sum(v for k, v in st.items() if k.startswith(("merge_", "ctl_")))
        out[tag] = {"ms": float(np.median(tot)), "merge_stage_ms": merge, "stages_ms": st}
    out["whole_ratio"] = out["control"]["ms"] / out["segment_lists"]["ms"]
    out["merge_stage_ratio"] = out["control"]["merge_stage_ms"] / out["segment_lists"]["merge_stage_ms"]
    del y, w, o, b, wa, wc
    return name, out


def run_gpu(args):
    import numpy as np
    import torch
    import convex_hull_pava_gb300 as chp
    from convex_hull_pava_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, peak_kind = peaks()

    W = wl.make(getattr(args, "workload", WORKLOAD))
    y = torch.from_numpy(W.y).to(dev)
    w = None if W.w is None else torch.from_numpy(W.w).to(dev)
    out = torch.empty_like(y)
    blocks = torch.empty(y.shape, dtype=torch.uint8, device=dev)
    status = torch.empty(W.rows, dtype=torch.int32, device=dev)
    ws = torch.empty(max(chp.iso_fit_workspace_bytes(W.rows, W.n, w is not None), 1),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(want_blocks=False):
        chp.iso_fit(y, w, W.increasing, out=out, blocks=blocks if want_blocks else None,
                    want_blocks=want_blocks, row_status=status, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    # ---- timed region: K product calls (no per-kernel events), L2 flushed
    # before each, each step timed by CUDA events on the launching stream ----
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()
        step_ms.append(a.elapsed_time(b))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()

    # ---- per-kernel split: the same calls again, in a separate pass, with CUDA
    # events around every kernel (iso_profile_enable); the library's kernels
    # launched per call are counted here ----
    chp.profile_enable(True)
    kern, prof_ms, per_call = {}, [], 0
    for _ in range(min(args.steps, 100)):
        flush.zero_()
        step()
        r = chp.profile_read()
        per_call = len(r)
        prof_ms.append(sum(ms for _, ms in r))
        for name, ms in r:
            kern.setdefault(name, []).append(ms)
    torch.cuda.synchronize()
    chp.profile_enable(False)
    launches = per_call * args.steps

    ms_step = cross_rank_max(float(np.mean(step_ms)), dev)
    value = job_value(W.elements, world, ms_step)

    # dominant kernel and its roofline: algorithmic bytes of that kernel per launch
    kavg = {k: float(np.mean(v)) for k, v in kern.items()}
    dom = max(kavg, key=kavg.get)
    alg_bytes = {
        # read y (and w); the chunk hull reads the input once
        "chunk_hull": W.elements * (8 if W.weighted else 4),
        # write the fit
        "expand": W.elements * 4,
        # descriptor lists only; no per-element traffic
        "merge_groups": 0,
        "merge_top": 0,
    }
    ab = alg_bytes.get(dom, W.elements * (12 if W.weighted else 8))
    achieved = ab / (kavg[dom] * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": committed_traffic(W.name, dom),
            "peak_kind": peak_kind, "algorithmic_bytes_per_launch": ab,
            "kernel_ms": kavg,
            "kernel_split": f"separate pass of {len(prof_ms)} calls with per-kernel CUDA events "
                            f"(sum of kernels {float(np.mean(prof_ms)):.4f} ms per call); the "
                            f"timed steps run without them"}
    fit_bytes = W.elements * (12 if W.weighted else 8)
    whole = fit_bytes / (ms_step * 1e-3) / 1e9

    # ---- end to end through the public API with pinned host buffers: the
    # input y is in pinned host memory and the fit goes to pinned host memory.
    # Three ways through the same call: (1) the host buffers passed straight to
    # iso_fit, whose kernels read y and write the fit over the host link
    # (NVLink-C2C); (2) explicit copies to and from device buffers around each
    # call, one call at a time; (3) the same copies for a stream of independent
    # problems, the next problem's input copied in while this one is fitted and
    # copied out (two device slots, copies on their own streams).  One call
    # cannot start writing its fit before all of y has arrived (every output
    # depends on every input), so (1) and (2) pay the link's read and write
    # times in turn; (3) overlaps the two directions.  e2e reports the fastest;
    # all are in the line, with the link's own copy rates. ----
    yh = torch.from_numpy(W.y).pin_memory()
    wh = None if W.w is None else torch.from_numpy(W.w).pin_memory()
    oh = torch.empty(W.y.shape, dtype=torch.float32).pin_memory()

    def e2e_time(one):
        ts = []
        for i in range(max(3, args.steps // 4) + 2):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            one()
            b.record(stream)
            b.synchronize()
            if i >= 2:
                ts.append(a.elapsed_time(b))
        return float(np.mean(ts))

    def in_place():
        chp.iso_fit(yh, wh, W.increasing, out=oh, want_blocks=False, workspace=ws, stream=stream)

    def with_copies():
        yd = yh.to(dev, non_blocking=True)
        wd = None if wh is None else wh.to(dev, non_blocking=True)
        z, _, _ = chp.iso_fit(yd, wd, W.increasing, want_blocks=False, workspace=ws, stream=stream)
        oh.copy_(z, non_blocking=True)

    # (3): host buffers rotate over four sets (more bytes than L2 holds), so
    # no problem's input can still be cached from an earlier one
    nrot = 4
    yhs = [yh] + [torch.from_numpy(W.y).pin_memory() for _ in range(nrot - 1)]
    whs = None if wh is None else [wh] + [torch.from_numpy(W.w).pin_memory() for _ in range(nrot - 1)]
    ohs = [oh] + [torch.empty(W.y.shape, dtype=torch.float32).pin_memory() for _ in range(nrot - 1)]
    yds = [torch.empty(W.y.shape, dtype=torch.float32, device=dev) for _ in range(2)]
    wds = None if wh is None else [torch.empty(W.w.shape, dtype=torch.float32, device=dev) for _ in range(2)]
    ods = [torch.empty(W.y.shape, dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_fit = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(nsteps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        s_in.wait_event(a)
        s_out.wait_event(a)
        for i in range(nsteps):
            k, h = i % 2, i % nrot
            if i >= 2:
                s_in.wait_event(ev_fit[k])        # slot k's input read by its last fit
            with torch.cuda.stream(s_in):
                yds[k].copy_(yhs[h], non_blocking=True)
                if wds is not None:
                    wds[k].copy_(whs[h], non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_out[k])      # slot k's fit copied out
            chp.iso_fit(yds[k], None if wds is None else wds[k], W.increasing, out=ods[k],
                        want_blocks=False, workspace=ws, stream=stream)
            ev_fit[k].record(stream)
            s_out.wait_event(ev_fit[k])
            with torch.cuda.stream(s_out):
                ohs[h].copy_(ods[k], non_blocking=True)
                ev_out[k].record(s_out)
        stream.wait_event(ev_out[0])
        if nsteps > 1:
            stream.wait_event(ev_out[1])
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / nsteps

    npipe = max(10, args.steps // 4)
    pipelined(npipe)
    e2e_modes = {"host_buffers_in_place": e2e_time(in_place), "explicit_copies": e2e_time(with_copies)}
    pipe_runs = [pipelined(npipe) for _ in range(3)]     # three runs of npipe problems: the median
    e2e_modes["pipelined_copies"] = float(np.median(pipe_runs))

    # the host link's own rates on the same bytes: one direction at a time and
    # both at once (copy engines, pinned memory)
    def link_rates():
        def t(fn, reps=10):
            fn()
            torch.cuda.synchronize(dev)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            b.synchronize()
            return a.elapsed_time(b) / reps

        def both():
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_in):
                yds[0].copy_(yhs[1], non_blocking=True)
            with torch.cuda.stream(s_out):
                ohs[1].copy_(ods[0], non_blocking=True)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)

        nb = W.elements * 4
        h2d = t(lambda: yds[0].copy_(yhs[1], non_blocking=True))
        d2h = t(lambda: ohs[1].copy_(ods[0], non_blocking=True))
        bi = t(both)
        # a step moves y (and w) in and the fit out: the floors at these rates
        b_in, b_out = W.elements * (8 if W.weighted else 4), W.elements * 4
        return {"bytes": nb, "h2d_gbs": nb / h2d / 1e6, "d2h_gbs": nb / d2h / 1e6,
                "both_directions_gbs": 2 * nb / bi / 1e6,
                "one_call_floor_ms": h2d * b_in / nb + d2h * b_out / nb,
                "overlapped_floor_ms": bi * (b_in + b_out) / (2 * nb)}

    link = link_rates()

    # bridge-search depth of one call (untimed; the library's debugging counters)
    def bridge_counts(call):
        chp.bridge_stats_mode(1)
        try:
            call()
            return chp.bridge_stats_read()
        finally:
            chp.bridge_stats_mode(0)

    bridge = bridge_counts(step) if W.n > 8192 else None
    e2e_mode = min(e2e_modes, key=e2e_modes.get)
    e2e_val = job_value(W.elements, world, cross_rank_max(e2e_modes[e2e_mode], dev))
    e2e_all = {k: job_value(W.elements, world, cross_rank_max(v, dev)) for k, v in e2e_modes.items()}

    # ---- the other named workloads (parity-test configurations), for context ----
    also = {}
    pool = None
    if not args.quick and rank == 0 and world == 1 and not args.no_cpu:
        import multiprocessing as mproc
        cores = os.cpu_count() or 1
        pool = mproc.get_context("spawn").Pool(cores)
    if not args.quick:
        for name in ("batch4096x1024", "dense16x4m", "softrank1024x8192", "row65k"):
            V = wl.make(name)
            yv = torch.from_numpy(V.y).to(dev)
            wv = None if V.w is None else torch.from_numpy(V.w).to(dev)
            ov = torch.empty_like(yv)
            bv = torch.empty(yv.shape, dtype=torch.uint8, device=dev)
            wsv = torch.empty(max(chp.iso_fit_workspace_bytes(V.rows, V.n, wv is not None), 1),
                              dtype=torch.uint8, device=dev)
            def fv():
                chp.iso_fit(yv, wv, V.increasing, out=ov, blocks=bv, workspace=wsv, stream=stream)
            ts = []
            for i in range(13):
                flush.zero_()
                a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
                a.record(stream); fv(); b.record(stream); b.synchronize()
                if i >= 3:
                    ts.append(a.elapsed_time(b))
            t = float(np.median(ts)) * 1e-3
            by = V.elements * (12 if V.weighted else 8)
            rec = {"elements_per_s": V.elements / t, "ms": t * 1e3, "gbs": by / t / 1e9,
                   "frac": by / t / 1e9 / hbm_peak, "bytes": by}
            if V.grad is not None:
                gv = torch.from_numpy(V.grad).to(dev)
                dv = torch.empty_like(gv)
                wsb = torch.empty(max(chp.iso_backward_workspace_bytes(V.rows, V.n, wv is not None), 1),
                                  dtype=torch.uint8, device=dev)
                ts = []
                for i in range(13):
                    flush.zero_()
                    a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    chp.iso_backward(gv, bv, wv, out=dv, workspace=wsb, stream=stream)
                    b.record(stream); b.synchronize()
                    if i >= 3:
                        ts.append(a.elapsed_time(b))
                tb = float(np.median(ts)) * 1e-3
                bb = V.elements * (9 if wv is None else 13)
                rec["backward"] = {"elements_per_s": V.elements / tb, "ms": tb * 1e3,
                                   "gbs": bb / tb / 1e9, "frac": bb / tb / 1e9 / hbm_peak}
            if pool is not None and V.rows > 1:
                rec["cpu_all_cores"] = time_oracle_all_cores(V, pool, os.cpu_count() or 1)
            if V.n > 8192:
                rec["bridge_search"] = bridge_counts(fv)
            also[name] = rec
            del yv, wv, ov, bv, wsv
        # the soft rank end to end (sort, non-increasing fit, gather; backward
        # through the block averaging), 1,024 rows x 8,192 N(0,1) values
        from convex_hull_pava_gb300.soft_rank import soft_rank
        xs = torch.from_numpy(wl.normal((1024, 8192), 31)).to(dev)
        gs = torch.from_numpy(wl.normal((1024, 8192), 32)).to(dev)
        sr = {}
        for tag, eps in (("eps_1", 1.0), ("eps_1_over_n", 1.0 / 8192)):
            ts = []
            for i in range(13):
                flush.zero_()
                x = xs.clone().requires_grad_(True)
                a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                soft_rank(x, eps).backward(gs)
                b.record(stream); b.synchronize()
                if i >= 3:
                    ts.append(a.elapsed_time(b))
            t = float(np.median(ts)) * 1e-3
            sr[tag] = {"ms_fwd_bwd": t * 1e3, "elements_per_s": xs.numel() / t}
        also["soft_rank_1024x8192"] = sr
        # a ragged batch of calibration curves: 65,536 segments of 1 to 8,192
        # points (log-uniform) and 8 of about 2^20, weighted, end to end
        lens = wl.ragged_lengths(65_536, 8192, seed=0, long_segments=8, long_len=1 << 20)
        yr_h, wr_h, off_h = wl.ragged_calibration(lens, seed=0)
        yr = torch.from_numpy(yr_h).to(dev)
        wr = torch.from_numpy(wr_h).to(dev)
        offr = torch.from_numpy(off_h).to(dev)
        orr = torch.empty_like(yr)
        br = torch.empty(yr.shape, dtype=torch.uint8, device=dev)
        wsr = torch.empty(chp.iso_fit_ragged_workspace_bytes(lens.size, yr.numel(), int(lens.max()), True),
                          dtype=torch.uint8, device=dev)
        ts = []
        for i in range(13):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            chp.iso_fit_ragged(yr, offr, wr, True, max_len=int(lens.max()), out=orr, blocks=br,
                               workspace=wsr, stream=stream)
            b.record(stream); b.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        t = float(np.median(ts)) * 1e-3
        by = yr.numel() * 13 + off_h.nbytes
        also["ragged_calibration_65536"] = {
            "segments": int(lens.size), "elements": int(yr.numel()),
            "elements_per_s": yr.numel() / t, "ms": t * 1e3, "gbs": by / t / 1e9,
            "frac": by / t / 1e9 / hbm_peak, "bytes": by}
        del yr, wr, offr, orr, br, wsr
        # the paper's Table 1 shapes (decreasing unweighted fits of noisy ramps),
        # with the paper's H100 time beside ours (other hardware: context only)
        t1 = {}
        for rows, n, h100 in ((100, 10**3, 0.07), (10**6, 16, 0.28), (10**4, 10**3, 0.35),
                              (10**3, 10**4, 0.37), (1, 10**6, 0.21), (1, 10**7, 0.56),
                              (1, 10**8, 2.74)):
            yv = torch.from_numpy(wl.noisy_ramp(rows, n, 0)).to(dev)
            ov = torch.empty_like(yv)
            wsv = torch.empty(max(chp.iso_fit_workspace_bytes(rows, n, False), 1), dtype=torch.uint8,
                              device=dev)
            ts = []
            for i in range(13):
                flush.zero_()
                a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                chp.iso_fit(yv, None, False, out=ov, want_blocks=False, workspace=wsv, stream=stream)
                b.record(stream); b.synchronize()
                if i >= 3:
                    ts.append(a.elapsed_time(b))
            t = float(np.median(ts))
            t1[f"{rows}x{n}"] = {"ms": t, "paper_h100_ms": h100, "elements_per_s": rows * n / t * 1e3}
            del yv, ov, wsv
        also["paper_table1_decreasing"] = t1
        # the materialised-copy control against the segment lists: whole call and
        # merge stage (segment lists: the two merge kernels; control: its setup,
        # levels and root list)
        ctl_cases = [("row1e7", lambda: (W.y, W.w, W.increasing))]
        ctl_cases.append(("dense16x4m", lambda: (lambda V: (V.y, V.w, V.increasing))(wl.make("dense16x4m"))))
        if args.control_table:
            for fam, n in (("increasing", 10**7), ("increasing", 10**8), ("cliff", 10**8),
                           ("noise", 10**7), ("noise", 10**8)):
                ctl_cases.append((f"{fam}_{n:.0e}", lambda fam=fam, n=n: (wl.family(fam, 1, n, 0), None, True)))
        also["copy_control"] = {k: v for k, v in (copy_control(name, mk, dev, flush, stream)
                                                 for name, mk in ctl_cases)}

    if pool is not None:
        pool.close()
        pool.join()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = time_oracle(W, budget_s=args.cpu_seconds)
        cpu["host"] = host_cpu()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "config": workload_desc(W),
            "hbm_gbs_whole_call": whole, "hbm_frac_whole_call": whole / hbm_peak,
            "roofline": roof, "cpu_baseline": cpu, "bridge_search": bridge,
            "e2e": {"value": e2e_val, "unit": UNIT,
                    "h2d_bytes_per_step": W.elements * (8 if W.weighted else 4),
                    "d2h_bytes_per_step": W.elements * 4, "mode": e2e_mode, "modes": e2e_all,
                    "pipelined_problems": npipe,
                    "pipelined_ms_per_problem_runs": pipe_runs,
                    "l2": "single calls flush L2 before each; the pipelined problems rotate over "
                          f"{nrot} host input buffers ({nrot * W.elements * 4 >> 20} MiB)",
                    "host_link": link},
            "gpu_launches": launches, "clocks": clocks, "also": also,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def wl_names():
    sys.path.insert(0, ROOT)
    from convex_hull_pava_gb300 import workloads as wl
    return wl.CONFIG_NAMES


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default=WORKLOAD, choices=wl_names(),
                    help="the workload of the timed steps, for profiling (the metric is quoted "
                         "on the default)")
    ap.add_argument("--control-table", action="store_true",
                    help="also time the materialised-copy control on increasing, cliff and noise "
                         "rows of 10^7 and 10^8 elements")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
