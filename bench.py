"""Benchmark of the DiT norm/modulation hot path (one JSON line on rank 0).

Headline workload (one step): the video-DiT per-token modulation block at Wan
scale, the largest single-GPU configuration,
  ln_modulate:            out1 = LN(x) * (1 + scale) + shift        x [1, 32760, 5120]
  rmsnorm_tanh_residual:  out2 = r + tanh(g) * RMSNorm(x) * w       g, r [1, 32760, 5120]
with per-token scale/shift [1, 32760, 5120], w [5120], eps 1e-6, bfloat16,
lossless variant, every call through the C ABI of libmbx.so.  Inputs are
synthetic (seeded N(0,1) activations, N(0,0.1) modulation, 1+N(0,0.05) weight).

Secondary workload (keys under "image_dit"): the image-DiT block norm path at
Qwen-Image scale, ln_modulate on x [2, 4352, 3072] with per-sample
scale/shift [2, 3072], then residual_gate_add x' + gate * y.

L2 policy: every headline step streams 2.68 GB, far more than L2 (129 MB),
and two buffer sets alternate; the image-DiT step rotates three 267 MB sets,
so no step reads a tensor the previous ~530 MB of traffic touched.

Metric: achieved HBM GB/s = algorithmic bytes (every input read once, every
output written once) / device time, from CUDA events on the launching stream.
Multi-GPU (torchrun): each rank runs its own copy of the workload (rows are
independent: no collective on the data path); the barrier and the max over
ranks of the timed region are the only communication.

--impl reference times the CPU oracle (oracle/, plain C) on a bounded sample
of the same workload, on this host's cores.
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

METRIC = "achieved HBM GB/s (% of GB300 peak) and µs/call for LN+AdaLN modulate"

# headline: video-DiT per-token modulation, [1, 32760, 5120]
VS, VD = 32760, 5120
V_T = VS * VD * 2                                    # one [1,32760,5120] bf16 tensor
V_LN_BYTES = 4 * V_T                                 # read x, scale, shift; write out1
V_TANH_BYTES = 4 * V_T + 2 * VD                      # read x, g, r, w; write out2
V_STEP_BYTES = V_LN_BYTES + V_TANH_BYTES
WORKLOAD = ("video-DiT per-token modulation: ln_modulate x[1,32760,5120] with per-token "
            "scale/shift [1,32760,5120] (eps 1e-6), then rmsnorm_tanh_residual "
            "out = r + tanh(g)*RMSNorm(x)*w with g, r [1,32760,5120], w [5120] (eps 1e-6), "
            "bf16, lossless")
L2_NOTE = ("2 alternating buffer sets of 2.35 GB; each step streams 2.68 GB "
           "(inputs larger than L2, no re-read)")

# secondary: image-DiT block norm path, [2, 4352, 3072]
IB, IS, ID = 2, 4352, 3072
I_T = IB * IS * ID * 2                               # one [2,4352,3072] bf16 tensor
I_LN_BYTES = 2 * I_T + 2 * IB * ID * 2               # read x, write out, scale + shift
I_RGA_BYTES = 3 * I_T + IB * ID * 2                  # read x', y, write out, gate
I_STEP_BYTES = I_LN_BYTES + I_RGA_BYTES
I_WORKLOAD = ("image-DiT block norm path: ln_modulate x[2,4352,3072] (per-sample scale/shift "
              "[2,3072], eps 1e-6) then residual_gate_add x'[2,4352,3072] + gate[2,3072]*y, "
              "bf16, lossless")
I_L2_NOTE = "3 rotating buffer sets of 267 MB (inputs larger than L2 per step, no re-read)"

# kernel sources behind each timed operation (the key of the DRAM traffic table)
_KERNEL_FILES = {
    "ln_modulate": ["ln_pipe.cuh", "ln_modulate.cu"],
    "rmsnorm_tanh_residual": ["rmsnorm.cu", "tanh_bf16_table.inc"],
    "residual_gate_add": ["residual.cu"],
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_sha(op: str) -> str:
    k = os.path.join(ROOT, "modulation_bit_exact_gb300", "csrc", "kernels")
    files = ["numerics.cuh", "rowops.cuh", "launch.h"] + _KERNEL_FILES[op]
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(k, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(op: str, workload: str):
    """Per-launch DRAM bytes (read + write) of `op` on `workload` from the
    committed ncu summary, if it was taken on the current kernel source (else
    None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_sha(op)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if (len(parts) >= 4 and not line.startswith("#") and parts[0] == op and parts[1] == workload
                    and parts[3] == sha):
                return int(parts[2])
    return None


class Clocks:
    """nvidia-smi sampling (every 100 ms) around the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}




# ---------------------------------------------------------------------- CPU oracle


def _video_sample(rows: int = 256):
    """The headline workload's recipe on `rows` tokens (CPU): bf16 bit patterns
    x, scale, shift, g, r [rows, 5120] and w [5120]."""
    import numpy as np
    import torch

    import synth
    d = synth.video_dit_block(seq=rows)
    u = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1, VD)
    return (u(d["x"]), u(d["scale"]), u(d["shift"]), u(d["gate"]), u(d["residual"]),
            u(d["weight"]).reshape(-1))


def _oracle_step_rows(arrays, r0: int, n: int):
    """Both operations of the headline step on rows [r0, r0 + n) of the sample."""
    import oracle
    X, SC, SH, G, R, W = arrays
    oracle.ln_modulate(X[r0:r0 + n], SC[r0:r0 + n], SH[r0:r0 + n], 1e-6)
    oracle.rmsnorm_tanh_residual(X[r0:r0 + n], G[r0:r0 + n], R[r0:r0 + n], W, 1e-6)


ROW_BYTES = V_STEP_BYTES / VS  # algorithmic bytes of one token row of the step


def oracle_rate(budget_s: float, rows_per_call: int = 16):
    """GB/s of the CPU oracle, one thread, on row samples of the headline
    workload (both operations), over about budget_s seconds; returns
    (GB/s, rows done, seconds)."""
    import oracle
    arrays = _video_sample()
    oracle.lib()
    nblk = arrays[0].shape[0] // rows_per_call
    done, t0 = 0, time.perf_counter()
    while True:
        _oracle_step_rows(arrays, (done // rows_per_call % nblk) * rows_per_call, rows_per_call)
        done += rows_per_call
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done * ROW_BYTES / el / 1e9, done, el


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's `value` (the job time of a weak-scaling run
    is the slowest rank's); `value` itself when there is one process."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _oracle_share(job):
    """One host process's share of the all-cores oracle baseline: rows
    [lo, hi) of the sample, both operations, for about `budget` seconds."""
    arrays, lo, hi, budget, rows_per_call = job
    import oracle
    oracle.lib()
    done, t0 = 0, time.perf_counter()
    n = max(1, (hi - lo) // rows_per_call)
    while True:
        _oracle_step_rows(arrays, lo + (done // rows_per_call % n) * rows_per_call, rows_per_call)
        done += rows_per_call
        el = time.perf_counter() - t0
        if el >= budget:
            return done, el


def oracle_rate_all_cores(budget_s: float, rows_per_call: int = 4):
    """The same oracle, one process per host core (a spawned pool: safe after
    CUDA is initialised), each on a static share of the sample rows; returns
    (GB/s, rows done, seconds, processes)."""
    import multiprocessing as mp
    arrays = _video_sample()
    n = os.cpu_count() or 1
    rows = arrays[0].shape[0]
    share = max(rows_per_call, rows // n // rows_per_call * rows_per_call)
    jobs = [(arrays, (i * share) % rows, min(rows, (i * share) % rows + share), budget_s, rows_per_call)
            for i in range(n)]
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_share, jobs)
    done = sum(r[0] for r in res)
    el = max(r[1] for r in res)
    return done * ROW_BYTES / el / 1e9, done, el, n


_REF_DATA = None


def _ref_init(arrays):
    global _REF_DATA
    _REF_DATA = arrays
    import oracle
    oracle.lib()


def _ref_rows(job):
    """Both operations of the headline step on rows [r0, r0 + rows) (one process)."""
    r0, rows = job
    _oracle_step_rows(_REF_DATA, r0, rows)
    return rows


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on this host's cores
    (one spawned process per core, each on a static share of the step's rows)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import multiprocessing as mp

    import oracle
    arrays = _video_sample()
    oracle.lib()
    n = os.cpu_count() or 1
    sample_rows = arrays[0].shape[0]
    # size a step so that warmup + steps take about 60 s in all
    t0 = time.perf_counter()
    _oracle_step_rows(arrays, 0, 4)
    per_row = (time.perf_counter() - t0) / 4
    per_proc = int(max(1, min(sample_rows, 60.0 / max(1, args.steps + args.warmup) / max(per_row, 1e-9))))
    rows = per_proc * n

    with mp.get_context("spawn").Pool(n, initializer=_ref_init, initargs=(arrays,)) as pool:
        def step(i):
            jobs = [(((i * n + k) * per_proc) % (sample_rows - per_proc + 1), per_proc) for k in range(n)]
            pool.map(_ref_rows, jobs)

        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(i)
        el = time.perf_counter() - t0
    gbs = rows * ROW_BYTES * args.steps / el / 1e9
    sample = (f"{rows} token rows of the step per step (both operations; the full step is "
              f"{VS} rows of [1,32760,5120]), {n} processes, one per host core, {per_proc} rows each")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- GPU arm


def _video_sets(mbx, dev, rank, n=2):
    """Buffer sets of the headline step, created on the device."""
    import torch

    import synth
    sets = []
    for i in range(n):
        d = synth.video_dit_block(seed=4 + 100 * i + 1000 * rank, device=dev)
        s = dict(x=d["x"], scale=d["scale"], shift=d["shift"], out1=torch.empty_like(d["x"]),
                 g=d["gate"], r=d["residual"], w=d["weight"], out2=torch.empty_like(d["x"]))
        sets.append((s, {k: mbx._view(t) for k, t in s.items()}))
    return sets


def _image_sets(mbx, dev, rank, n=3):
    """Buffer sets of the image-DiT step, created on the device."""
    import torch

    import synth
    sets = []
    for i in range(n):
        d = synth.image_dit_block(seed=2 + 100 * i + 1000 * rank, device=dev)
        d2 = synth.image_dit_block(seed=3 + 100 * i + 1000 * rank, device=dev)
        s = dict(x=d["x"], scale=d["scale"], shift=d["shift"], out1=torch.empty_like(d["x"]),
                 xb=d2["x"], gate=d["gate"], y=d["y"], out2=torch.empty_like(d["x"]))
        sets.append((s, {k: mbx._view(t) for k, t in s.items()}))
    return sets


def _time_loops(stream, K, step, calls):
    """K steps with events at the two ends only (an event between the calls
    would stop each from overlapping its launch with the previous one's
    drain), then each call alone K times back to back, events at the ends.
    Returns (step ms total, [call ms total], status)."""
    import torch
    st = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        st |= step(i)
    e1.record(stream)
    per_call = []
    for fn in calls:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(K):
            st |= fn(i)
        b.record(stream)
        per_call.append((a, b))
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), [a.elapsed_time(b) for a, b in per_call], st


def run_gpu(args):
    import ctypes

    import torch

    import modulation_bit_exact_gb300 as mbx

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    L = mbx.lib()
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    eps = ctypes.c_float(1e-6)
    ref = ctypes.byref

    vsets = _video_sets(mbx, dev, rank)
    isets = _image_sets(mbx, dev, rank)
    torch.cuda.synchronize(dev)

    def v_ln(i):
        v = vsets[i % 2][1]
        return L.mbx_ln_modulate(ref(v["out1"]), ref(v["x"]), ref(v["scale"]), ref(v["shift"]), eps, 0, sptr)

    def v_tanh(i):
        v = vsets[i % 2][1]
        return L.mbx_rmsnorm_tanh_residual(ref(v["out2"]), ref(v["x"]), ref(v["g"]), ref(v["r"]), ref(v["w"]),
                                           eps, 0, sptr)

    def i_ln(i):
        v = isets[i % 3][1]
        return L.mbx_ln_modulate(ref(v["out1"]), ref(v["x"]), ref(v["scale"]), ref(v["shift"]), eps, 0, sptr)

    def i_rga(i):
        v = isets[i % 3][1]
        return L.mbx_residual_gate_add(ref(v["out2"]), ref(v["xb"]), ref(v["gate"]), ref(v["y"]), 0, sptr)

    v_step = lambda i: v_ln(i) | v_tanh(i)
    i_step = lambda i: i_ln(i) | i_rga(i)

    for i in range(args.warmup):
        if v_step(i) | i_step(i):
            raise RuntimeError("launch failed")
    torch.cuda.synchronize(dev)

    K = args.steps
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    if not gpu_uuid.startswith("GPU-"):
        gpu_uuid = "GPU-" + gpu_uuid
    clocks = Clocks(gpu_uuid)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with clocks:
        v_ms, (v_ln_ms, v_tanh_ms), st_v = _time_loops(stream, K, v_step, (v_ln, v_tanh))
        i_ms, (i_ln_ms, i_rga_ms), st_i = _time_loops(stream, K, i_step, (i_ln, i_rga))
    if st_v | st_i:
        raise RuntimeError("launch failed")
    if dist:
        dist.barrier()
    v_ms = max_over_ranks(v_ms, dist, dev)
    i_ms = max_over_ranks(i_ms, dist, dev)

    # End to end on the headline step: every step copies its inputs in from
    # pinned host memory, runs both calls through the C ABI and copies its
    # outputs back to pinned host memory.  Copies in, compute and copies out
    # run on three streams with two device buffer sets, so step i+1's inputs
    # travel while step i computes and step i-1's outputs return (the way a
    # serving loop overlaps them); events order each set's reuse.  Every rank
    # measures its own replica; the slowest is reported.
    names_in = ("x", "scale", "shift", "g", "r", "w")
    names_out = ("out1", "out2")
    host = {k: torch.empty(vsets[0][0][k].shape, dtype=torch.bfloat16, pin_memory=True)
            for k in names_in + names_out}
    for k in names_in:
        host[k].copy_(vsets[0][0][k])
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    cptr = ctypes.c_void_p(s_cmp.cuda_stream)
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    for e in ev_in + ev_cmp + ev_out:
        e.record(stream)
    torch.cuda.synchronize(dev)
    n_e2e = 4

    def e2e_step(i):
        b = i % 2
        t, v = vsets[b]
        s_in.wait_event(ev_cmp[b])  # the calls that last read this set are done
        with torch.cuda.stream(s_in):
            for k in names_in:
                t[k].copy_(host[k], non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        s_cmp.wait_event(ev_out[b])  # this set's outputs have been copied out
        st = L.mbx_ln_modulate(ref(v["out1"]), ref(v["x"]), ref(v["scale"]), ref(v["shift"]), eps, 0, cptr)
        st |= L.mbx_rmsnorm_tanh_residual(ref(v["out2"]), ref(v["x"]), ref(v["g"]), ref(v["r"]), ref(v["w"]),
                                          eps, 0, cptr)
        if st != 0:
            raise RuntimeError("launch failed")
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            for k in names_out:
                host[k].copy_(t[k], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    # three runs, the median reported: the host link is shared with the
    # machine's other GPUs and a single run can catch their traffic
    runs = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_out)  # after the last copy out, which follows every earlier step
        torch.cuda.synchronize(dev)
        runs.append(e0.elapsed_time(e1) / n_e2e)
    e2e_ms = max_over_ranks(sorted(runs)[1], dist, dev)
    h2d = sum(host[k].numel() * 2 for k in names_in)
    d2h = sum(host[k].numel() * 2 for k in names_out)
    e2e = {"value": round(V_STEP_BYTES * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_ms, 4), "steps": n_e2e,
           "runs_ms_per_step": [round(r, 4) for r in runs], "of_runs": "median of 3",
           "overlap": "copies in, compute, copies out on three streams, two device buffer sets"}
    del host

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = peaks()

    def kern(name, ms, nbytes, workload):
        us = ms / K * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us_per_call": round(us, 3), "bytes": nbytes, "gbs": round(gbs, 1),
                "frac": round(gbs / peak, 4), "frac_of_8tbs_spec": round(gbs / 8000.0, 4),
                "traffic": dram_traffic(name, workload)}

    v_kern = {"ln_modulate": kern("ln_modulate", v_ln_ms, V_LN_BYTES, "video"),
              "rmsnorm_tanh_residual": kern("rmsnorm_tanh_residual", v_tanh_ms, V_TANH_BYTES, "video")}
    i_kern = {"ln_modulate": kern("ln_modulate", i_ln_ms, I_LN_BYTES, "image"),
              "residual_gate_add": kern("residual_gate_add", i_rga_ms, I_RGA_BYTES, "image")}
    dom = max(v_kern, key=lambda k: v_kern[k]["us_per_call"])
    roof = {"bound": "hbm", "achieved": v_kern[dom]["gbs"], "peak": peak, "unit": "GB/s",
            "frac": v_kern[dom]["frac"], "traffic": v_kern[dom]["traffic"], "kernel": dom,
            "bytes_per_launch": v_kern[dom]["bytes"],
            "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, null unless "
                            "captured on the current kernel source",
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s"}
    cpu = None
    if world == 1:  # the oracle on this host's cores, timed at N = 1 only
        cpu_gbs, cpu_rows, cpu_s = oracle_rate(args.cpu_seconds)
        all_gbs, all_rows, all_s, all_n = oracle_rate_all_cores(args.cpu_seconds)
        cpu = {"value": round(all_gbs, 4), "unit": "GB/s", "cores": all_n, "kind": "oracle",
               "sample": f"{all_rows} token rows of the headline step (both operations, [rows,5120]) "
                         f"in {all_s:.1f} s, {all_n} processes, one per host core, each on a static "
                         f"share of a 256-row sample; single thread: {cpu_gbs:.4f} GB/s "
                         f"({cpu_rows} rows in {cpu_s:.1f} s)",
               "value_1_thread": round(cpu_gbs, 4)}
    value = V_STEP_BYTES * K * world / (v_ms * 1e-3) / 1e9
    i_value = I_STEP_BYTES * K * world / (i_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(v_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": L2_NOTE, "variant": "lossless",
                   "parallelism": f"replicas x{world} (row-independent, no data-path collective)"},
        "ln_modulate_us_per_call": v_kern["ln_modulate"]["us_per_call"],
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "frac_of_8tbs_spec": round(value / world / 8000.0, 4),
        "kernels": v_kern,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "image_dit": {
            "workload": I_WORKLOAD, "l2": I_L2_NOTE, "value": round(i_value, 2), "unit": "GB/s",
            "ms_per_step": round(i_ms / K, 5), "frac_of_hbm_peak": round(i_value / world / peak, 4),
            "ln_modulate_us_per_call": i_kern["ln_modulate"]["us_per_call"], "kernels": i_kern},
        "gpu_launches": 8 * K * world,
        "kernel_timing": {"how": "per workload: K steps with events at the ends, then each call alone, "
                                 "K launches back to back, events at the ends",
                          "launches": 8 * K * world},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------- suite


def run_suite(args):
    """Every operation x variant on the configurations' shapes, one JSON line
    per case: device time per call (CUDA events, median of 5 repeats of a
    rotating loop over buffer sets whose total exceeds L2, with the fastest
    and slowest repeat as us_min / us_max; for calls under 64 MB also the
    device time per call through a CUDA graph, us_device, which leaves out
    host submission), GB/s of the algorithmic bytes and the fraction of the
    measured HBM peak."""
    import torch

    import modulation_bit_exact_gb300 as mbx
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, _ = peaks()
    L2 = 129 * 2 ** 20
    want_ops = set(args.ops.split(",")) if getattr(args, "ops", None) else None

    spread = {}  # min and max of the five repeats of the last case timed

    def time_graph(sets, fn, calls=64):
        """Device time per call without host submission: `calls` launches
        over the rotating sets captured in one CUDA graph, replayed five
        times (median).  None if capture is refused."""
        try:
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                for i in range(len(sets)):
                    fn(sets[i])
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                for i in range(calls):
                    fn(sets[i % len(sets)])
            g.replay()
            torch.cuda.synchronize(dev)
            ts = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(b) / calls * 1e3)
            del g
            return round(sorted(ts)[2], 2)
        except Exception:
            torch.cuda.synchronize(dev)
            return None

    def time_cases(make, nbytes, fn):
        per_set = max(1, nbytes)
        nsets = max(2, min(8, int(3 * L2 // per_set) + 1))
        sets = [make(i) for i in range(nsets)]
        # small calls: the device time through a CUDA graph as well
        spread["device"] = time_graph(sets, fn) if nbytes < 64 * 2 ** 20 else None
        for i in range(3 * nsets):
            fn(sets[i % nsets])
        torch.cuda.synchronize(dev)
        reps = max(10, min(200, int(2e9 // per_set)))
        times = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(reps):
                fn(sets[i % nsets])
            b.record()
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b) / reps * 1e3)
        times.sort()
        spread.update(lo=round(times[0], 2), hi=round(times[-1], 2))
        return times[2]

    def row_case(name, B, S, D, tok):
        rows = B * S
        mrows = rows if tok else B

        def make(i):
            g = torch.Generator(device=dev).manual_seed(1000 + i)
            r = lambda *sh, std=1.0, mean=0.0: (torch.randn(*sh, generator=g, device=dev) * std + mean).to(torch.bfloat16)
            return dict(x=r(rows, D), y=r(rows, D), res=r(rows, D), g=r(mrows, D) if tok else r(mrows, D, std=0.1),
                        sc=r(mrows, D, std=0.1), sh=r(mrows, D, std=0.1), w=r(D, std=0.05, mean=1.0),
                        b=r(1, D, std=0.5), out=torch.empty(rows, D, dtype=torch.bfloat16, device=dev),
                        out2=torch.empty(rows, D, dtype=torch.bfloat16, device=dev),
                        q=torch.empty(rows, D, dtype=torch.uint8, device=dev),
                        s8=torch.full((1,), 0.02, dtype=torch.float32, device=dev),
                        q4=torch.empty(rows, D // 2, dtype=torch.uint8, device=dev),
                        sf4=torch.zeros(mbx.nvfp4_sf_shape(rows, D), dtype=torch.uint8, device=dev),
                        g4=torch.full((1,), 60.0, dtype=torch.float32, device=dev))
        T = rows * D * 2
        M = mrows * D * 2
        ops = {
            "ln_modulate": (2 * T + 2 * M, lambda s, v: mbx.ln_modulate(s["x"], s["sc"], s["sh"], variant=v, out=s["out"])),
            "rmsnorm_scale": (2 * T + M + D * 2, lambda s, v: mbx.rmsnorm_scale(s["x"], s["w"], s["sc"], variant=v, out=s["out"])),
            "rmsnorm_tanh_residual": (3 * T + M + D * 2, lambda s, v: mbx.rmsnorm_tanh_residual(s["x"], s["g"], s["res"], s["w"], variant=v, out=s["out"])),
            "residual_gate_add": (3 * T + M, lambda s, v: mbx.residual_gate_add(s["x"], s["g"], s["y"], variant=v, out=s["out"])),
            "gated_residual_ln_modulate": (4 * T + 3 * M + D * 2, lambda s, v: mbx.gated_residual_ln_modulate(
                s["res"], s["g"], s["y"], s["sc"], s["sh"], bias=s["b"], variant=v, out=s["out"], residual_out=s["out2"])),
            "ln_modulate_fp8": (2 * T + 2 * M + T // 2, lambda s, v: mbx.ln_modulate_fp8(
                s["x"], s["sc"], s["sh"], s["s8"], variant=v, out=s["out"], out_fp8=s["q"])),
            "gated_residual_ln_modulate_fp8": (4 * T + 3 * M + D * 2 + T // 2, lambda s, v: mbx.gated_residual_ln_modulate_fp8(
                s["res"], s["g"], s["y"], s["sc"], s["sh"], s["s8"], bias=s["b"], variant=v, out=s["out"],
                residual_out=s["out2"], out_fp8=s["q"])),
            "ln_modulate_nvfp4": (2 * T + 2 * M + T // 4 + T // 32, lambda s, v: mbx.ln_modulate_nvfp4(
                s["x"], s["sc"], s["sh"], s["g4"], variant=v, out=s["out"], out_fp4=s["q4"], out_sf=s["sf4"])),
            "gated_residual_ln_modulate_nvfp4": (4 * T + 3 * M + D * 2 + T // 4 + T // 32,
                                                 lambda s, v: mbx.gated_residual_ln_modulate_nvfp4(
                s["res"], s["g"], s["y"], s["sc"], s["sh"], s["g4"], bias=s["b"], variant=v, out=s["out"],
                residual_out=s["out2"], out_fp4=s["q4"], out_sf=s["sf4"])),
        }
        for op, (nb, fn) in ops.items():
            if want_ops and op not in want_ops:
                continue
            for v in ("lossless", "high"):
                us = time_cases(make, nb, lambda st: fn(st, v))
                gbs = nb / (us * 1e-6) / 1e9
                print(json.dumps({"case": name, "shape": [rows, D], "modulation": "per-token" if tok else "per-sample",
                                  "op": op, "variant": v, "us_per_call": round(us, 2), "us_min": spread["lo"],
                                  "us_max": spread["hi"], "us_device": spread["device"], "bytes": nb,
                                  "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}), flush=True)

    def qkv_case(name, B, s_txt, gh, gw, H):
        hd = 128

        def make(i):
            return synth.qkv_epilogue_case(seed=2000 + i, device=dev, batch=B, s_txt=s_txt, grid_h=gh, grid_w=gw, heads=H)
        nb = 2 * B * (s_txt + gh * gw) * 3 * H * hd * 2
        for v in ("lossless", "high"):
            fn = lambda q: mbx.qk_norm_rope_qkv_epilogue(q["txt"], q["img"], B, H, hd, q["wq_txt"], q["wk_txt"],
                                                         q["wq_img"], q["wk_img"], q["cos_txt"], q["sin_txt"],
                                                         q["cos_img"], q["sin_img"], variant=v)
            us = time_cases(make, nb, fn)
            gbs = nb / (us * 1e-6) / 1e9
            print(json.dumps({"case": name, "shape": [B, s_txt, gh * gw, H, hd], "op": "qk_norm_rope_qkv_epilogue",
                              "variant": v, "us_per_call": round(us, 2), "us_min": spread["lo"],
                              "us_max": spread["hi"], "bytes": nb, "gbs": round(gbs, 1),
                              "frac_of_peak": round(gbs / peak, 4)}), flush=True)

    def table_case(name, rows, D, tab_dt=torch.float32, emb_dt=torch.bfloat16):
        def make(i):
            g = torch.Generator(device=dev).manual_seed(3000 + i)
            return dict(t=(torch.randn(6, D, generator=g, device=dev) / D ** 0.5).to(tab_dt),
                        e=torch.randn(rows, 6 * D, generator=g, device=dev).to(emb_dt),
                        o=torch.empty(6, rows, D, dtype=torch.float32, device=dev))
        esz = 2 if emb_dt == torch.bfloat16 else 4
        nb = rows * 6 * D * (esz + 4) + 6 * D * (2 if tab_dt == torch.bfloat16 else 4)
        us = time_cases(make, nb, lambda st: mbx.modulation_table_add(st["t"], st["e"], out=st["o"]))
        gbs = nb / (us * 1e-6) / 1e9
        print(json.dumps({"case": name, "shape": [rows, 6, D], "op": "modulation_table_add",
                          "variant": "exact", "us_per_call": round(us, 2), "us_min": spread["lo"],
                          "us_max": spread["hi"], "bytes": nb, "gbs": round(gbs, 1),
                          "frac_of_peak": round(gbs / peak, 4)}), flush=True)

    only = getattr(args, "only", None)
    if only:
        if "table" in only:
            table_case("Wan2.2-TI2V table [1,109120,6,3072] bf16 temb", 31 * 44 * 80, 3072)
            table_case("video table [1,32760,6,5120] bf16 temb", 32760, 5120)
            table_case("video table [1,32760,6,5120] f32 temb", 32760, 5120, emb_dt=torch.float32)
        if "tiny" in only:
            row_case("tiny [2,256,512]", 2, 256, 512, False)
            row_case("sweep [77,3072]", 1, 77, 3072, False)
        if "image" in only:
            row_case("image-DiT [2,4352,3072]", 2, 4352, 3072, False)
        if "video" in only:
            row_case("video-DiT [1,32760,5120] per-token", 1, 32760, 5120, True)
        if "qkv" in only:
            qkv_case("QKV epilogue [2,256+64x64,24x128]", 2, 256, 64, 64, 24)
        if "sweep" in only.split(","):
            for D in (1024, 3072, 4096, 8192):
                row_case(f"sweep [65536,{D}]", 1, 65536, D, False)
        if "sweep2" in only.split(","):
            for D in (2048, 5120, 6144):
                row_case(f"sweep [65536,{D}]", 1, 65536, D, False)
        if "sweep4k" in only.split(","):
            for D in (1024, 3072, 4096, 8192):
                row_case(f"sweep [4096,{D}]", 1, 4096, D, False)
        if "sweepmid" in only.split(","):
            for T in (16384, 32768):
                for D in (2048, 3072, 4096):
                    row_case(f"sweep [{T},{D}]", 1, T, D, False)
        return 0
    row_case("tiny [2,256,512]", 2, 256, 512, False)
    row_case("sweep [77,3072]", 1, 77, 3072, False)
    row_case("image-DiT [2,4352,3072]", 2, 4352, 3072, False)
    qkv_case("QKV epilogue [2,256+64x64,24x128]", 2, 256, 64, 64, 24)
    row_case("video-DiT [1,32760,5120] per-token", 1, 32760, 5120, True)
    for D in (1024, 4096, 8192):
        for T in (4096, 65536):
            row_case(f"sweep [{T},{D}]", 1, T, D, False)
    table_case("Wan2.2-TI2V table [1,109120,6,3072] bf16 temb", 31 * 44 * 80, 3072)
    table_case("video table [1,32760,6,5120] bf16 temb", 32760, 5120)
    return 0


# ---------------------------------------------------------------- profiler drivers


def run_profile_calls(args):
    """Launch a fixed set of calls `--steps` times, untimed, for a profiler to
    capture (the commands in profiles/ run these)."""
    import torch

    import modulation_bit_exact_gb300 as mbx
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    r = lambda *sh, std=1.0: (torch.randn(*sh, generator=g, device=dev) * std).to(torch.bfloat16)
    calls = []
    if args.profile_calls == "ln":  # ln_modulate on x [4,4352,3072]: 107 MB in, 107 MB out
        d = synth.image_dit_block(batch=4, device=dev)
        calls.append(lambda: mbx.ln_modulate(d["x"], d["scale"], d["shift"]))
    elif args.profile_calls == "image":  # the bench kernels plus the fused gated LN, [8704, 3072]
        x, y, res = r(8704, 3072), r(8704, 3072), r(8704, 3072)
        sc, sh, gt = (r(2, 3072, std=0.1) for _ in range(3))
        b = r(1, 3072, std=0.5)
        out, out2 = torch.empty_like(x), torch.empty_like(x)
        calls += [lambda: mbx.ln_modulate(x, sc, sh, out=out),
                  lambda: mbx.residual_gate_add(x, gt, y, out=out),
                  lambda: mbx.gated_residual_ln_modulate(res, gt, y, sc, sh, bias=b, out=out, residual_out=out2)]
    elif args.profile_calls == "next":  # QKV epilogue, gated LN, FP8 LN, modulation table
        q = synth.qkv_epilogue_case(device=dev)
        res, upd = r(8704, 3072), r(8704, 3072)
        gt, sc, sh = (r(2, 3072, std=0.1) for _ in range(3))
        b = r(1, 3072, std=0.5)
        out, out2 = torch.empty_like(res), torch.empty_like(res)
        q8 = torch.empty(8704, 3072, dtype=torch.uint8, device=dev)
        s8 = torch.tensor([0.02], device=dev)
        table = torch.randn(6, 3072, generator=g, device=dev)
        temb = r(4096, 6 * 3072)
        tout = torch.empty(6, 4096, 3072, device=dev)
        calls += [lambda: mbx.qk_norm_rope_qkv_epilogue(q["txt"], q["img"], 2, 24, 128, q["wq_txt"], q["wk_txt"],
                                                        q["wq_img"], q["wk_img"], q["cos_txt"], q["sin_txt"],
                                                        q["cos_img"], q["sin_img"]),
                  lambda: mbx.gated_residual_ln_modulate(res, gt, upd, sc, sh, bias=b, out=out, residual_out=out2),
                  lambda: mbx.ln_modulate_fp8(res, sc, sh, s8, out=out, out_fp8=q8),
                  lambda: mbx.modulation_table_add(table, temb, out=tout)]
    elif args.profile_calls == "video":  # the headline step, one buffer set: 2.35 GB on the device
        d = synth.video_dit_block(device=dev)
        out1, out2 = torch.empty_like(d["x"]), torch.empty_like(d["x"])
        calls += [lambda: mbx.ln_modulate(d["x"], d["scale"], d["shift"], out=out1),
                  lambda: mbx.rmsnorm_tanh_residual(d["x"], d["gate"], d["residual"], d["weight"], out=out2)]
    elif args.profile_calls == "rms":  # both RMSNorm ops at image-DiT size, per-sample modulation
        x, res, gtok = r(8704, 3072), r(8704, 3072), r(8704, 3072)
        sc = r(2, 3072, std=0.1)
        w = (torch.randn(3072, generator=g, device=dev) * 0.05 + 1).to(torch.bfloat16)
        out = torch.empty_like(x)
        calls += [lambda: mbx.rmsnorm_scale(x, w, sc, out=out),
                  lambda: mbx.rmsnorm_tanh_residual(x, gtok, res, w, out=out)]
    elif args.profile_calls == "nvfp4":  # the NVFP4 producers at image-DiT size
        x, res, upd = r(8704, 3072), r(8704, 3072), r(8704, 3072)
        gt, sc, sh = (r(2, 3072, std=0.1) for _ in range(3))
        b = r(1, 3072, std=0.5)
        out, out2 = torch.empty_like(x), torch.empty_like(x)
        q4 = torch.empty(8704, 1536, dtype=torch.uint8, device=dev)
        sf4 = torch.zeros(mbx.nvfp4_sf_shape(8704, 3072), dtype=torch.uint8, device=dev)
        g4 = torch.full((1,), 60.0, dtype=torch.float32, device=dev)
        calls += [lambda: mbx.ln_modulate_nvfp4(x, sc, sh, g4, out=out, out_fp4=q4, out_sf=sf4),
                  lambda: mbx.gated_residual_ln_modulate_nvfp4(res, gt, upd, sc, sh, g4, bias=b, out=out,
                                                               residual_out=out2, out_fp4=q4, out_sf=sf4)]
    for _ in range(args.steps):
        for c in calls:
            c()
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_calls": args.profile_calls, "rounds": args.steps, "calls_per_round": len(calls)}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="mbx", choices=["mbx", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    help="with --suite: run only the named groups (tiny, image, video, qkv, sweep, sweep2, sweep4k, sweepmid, table)")
    ap.add_argument("--ops", default=None, help="with --suite: run only the named operations (comma list)")
    ap.add_argument("--suite", action="store_true",
                    help="time every operation and variant on the configurations' shapes "
                         "(one JSON line per case) instead of the benchmark step")
    ap.add_argument("--profile-calls", default=None, choices=["ln", "image", "next", "video", "rms", "nvfp4"],
                    help="launch a fixed set of calls --steps times, untimed, for a profiler")
    args = ap.parse_args()
    if args.profile_calls:
        return run_profile_calls(args)
    if args.suite:
        return run_suite(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
