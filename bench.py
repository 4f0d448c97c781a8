"""Benchmark of the Q4_0 x f32 hot path on GB300 (one JSON line on stdout).

One step = one pass of the M = 1 decode GEMVs of the 32-layer decoder sweep
(hidden 4096, GQA: per layer q, o 4096 -> 4096; k, v 4096 -> 1024; gate, up
4096 -> 14336; down 14336 -> 4096): 224 GEMVs streaming 3.93 GB of Q4_0
weights, through libqm's C ABI as one call of qm_gemv_q4_0_list (two
launches of the persistent list kernel, 128 and 96 independent problems, as
the library splits a list; within a layer q, k
and v read one input vector and gate and up another, as in a decoder).
Inputs are synthetic (seeded generators in ``synth``); the weights are 30
times the L2, so no step finds them there.

value = Q4_0 weight bytes streamed per step / device time per step (GB/s), the
GEMV weight-stream rate of the metric, timed with CUDA events over --steps
steps after --warmup steps.  ``roofline`` is the step's one launch against
the measured HBM copy rate.  ``e2e`` repeats the step with host operands: the
128 activation vectors copied host -> device and all 224 outputs device -> host
inside the timed region, the copies of neighbouring steps overlapping a
step's kernel on separate streams.

Every other workload is reported in the same line: ``roofline.per_config``
holds the GEMV and dequant rows (M=1 at K=N=4096 back to back, config 1's
M=8 up and down GEMVs, the dequant of the 14336 x 4096 weight, the decoder
sweep as 224 launches at M=1 and M=8, stacked, through the list GEMV three
ways, and through the act-quant GEMV and its list) as weight GB/s against HBM,
and ``prefill`` the GEMM rows (M=32 and M=256 at 4096 x 4096, M=1024 at both
FFN shapes, the decoder sweep at M=512) as TFLOP/s against the tensor-core
bound.  ``q8_0`` holds the Q8_0 quantize and dequant, ``host_us_per_call``
the host time of the C-ABI calls.

``cpu_baseline`` times the oracle (fp64 C) on this host on a bounded column
sample of the step (the first columns of each of layer 0's seven
projections): one thread, and all cores through OpenMP.  ``--impl
reference`` runs that oracle as the reference arm, each step a bounded column
sample of the same workload, on the same metric.
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

import synth  # noqa: E402

METRIC = "Q4_0 GEMV weight GB/s (% of HBM peak); prefill TFLOP/s (% of roofline)"
WORKLOAD = "q4_0_gemv_decoder_sweep_m1_32_layers"
FALLBACK_HBM_GBS = 6800.0
REPLICAS = 4  # config 1's GEMVs: 4 x 66 MB of weights (plus activations) > 129 MB of L2
SWEEP_LAYERS = 32
STEP_REPLICAS = 3  # activation and output buffers of the step (the weights are shared)
WARMUP_S = 0.3     # minimum seconds of warm-up load before timing


def bench_config(world: int) -> dict:
    """The workload description both arms print (identical dicts)."""
    return {"workload": WORKLOAD, "M": 1, "layers": SWEEP_LAYERS,
            "projections": "q, o 4096->4096; k, v 4096->1024; gate, up 4096->14336; down 14336->4096",
            "inputs": "per layer 4 activation vectors: q, k, v share one, gate and up one, o and down their own",
            "gemvs_per_step": 7 * SWEEP_LAYERS, "seed": 5,
            "api": "qm_gemv_q4_0_list: one call per step, 224 independent GEMVs (the library runs them "
                   "as two persistent launches of at most 128 problems)",
            "l2": "3.93 GB of weights per step, 30x the L2",
            "parallelism": f"replicas x{world}",
            "value_definition": "Q4_0 weight bytes streamed per step / step time"}


# ------------------------------------------------------------------ helpers

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
KERNEL_SOURCES = {"dequant_q4_0": "dequant.cu", "gemv_q4_0_tc": "gemv_tc.cu",
                  "gemm_q4_0_tc": "gemm_tc.cu", "gemv_q4_0_list": "gemv_list.cu"}


def source_digest(kernel: str) -> str:
    import hashlib
    path = os.path.join(ROOT, "bit_block_quantized_qm_gb300", "csrc", KERNEL_SOURCES[kernel])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary, or
    None when there is none for this kernel and workload, or when the
    kernel's source changed after the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    digest = source_digest(kernel)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            fields = dict(kv.split("=", 1) for kv in line.split())
            if (fields.get("kernel") == kernel and fields.get("workload") == workload and
                    fields.get("source_sha256_16") == digest):
                return int(fields["dram_bytes_per_launch"])
    return None


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks: a step is as slow as the slowest rank.
    With one rank (dist None) x itself."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: int, world: int, ms_step: float) -> float:
    """Whole-job throughput: the bytes every rank streamed in one step over
    the (slowest rank's) step time."""
    return bytes_per_rank * world / (ms_step * 1e-3) / 1e9


DECODER_PROJS = tuple(p for (p, _, _) in synth.DECODER_LAYER)
# The projection (index within a layer) whose input vector each one reads.
SHARED_INPUT = {"q": 0, "k": 0, "v": 0, "o": 3, "gate": 4, "up": 4, "down": 6}


def sweep_cases():
    """The step's 224 GEMVs (M = 1), layer by layer."""
    return synth.workload(4, layers=SWEEP_LAYERS, sweep_m=(1,))


def sweep_operands(qm, torch, dev, cases, replicas: int):
    """Device operands of the decoder sweep's GEMVs: the weights (resident,
    shared by the replicas), and per replica one buffer of the layers'
    activation vectors (q, k and v read one, gate and up another, o and down
    their own), one buffer of all outputs and the list of problems over them.
    Returns (weights, host activations, output floats, replicas)."""
    weights = [torch.from_numpy(c.weights()).to(dev) for c in cases]
    src = [7 * (i // 7) + SHARED_INPUT[DECODER_PROJS[i % 7]] for i in range(len(cases))]
    inputs = sorted(set(src))
    a_start = dict(zip(inputs, np.cumsum([0] + [cases[j].K for j in inputs])))
    a_off = [a_start[j] for j in src]
    c_off = np.cumsum([0] + [c.N for c in cases])
    a_host = np.concatenate([cases[j].acts().ravel() for j in inputs])
    reps = []
    for _ in range(replicas):
        A = torch.from_numpy(a_host).to(dev, copy=True)
        C = torch.empty(int(c_off[-1]), dtype=torch.float32, device=dev)
        arr = qm.gemv_problem_array([
            (A.data_ptr() + 4 * int(a_off[i]), weights[i].data_ptr(), C.data_ptr() + 4 * int(c_off[i]),
             c.N, c.K, -1) for i, c in enumerate(cases)])
        reps.append({"A": A, "C": C, "problems": arr})
    if dev.type == "cuda":
        torch.cuda.synchronize()
    return weights, a_host, int(c_off[-1]), reps


def step_cases():
    cases = synth.workload(1)
    up = next(c for c in cases if c.name == "gemv_m8_k4096_n14336")
    down = next(c for c in cases if c.name == "gemv_m8_k14336_n4096")
    deq = next(c for c in cases if c.op == "dequant")
    return up, down, deq


def gemv_bytes(c) -> int:
    """Algorithmic bytes of a matmul: the weight stream once, A read, C written."""
    return c.weight_bytes + c.M * c.K * 4 + c.M * c.N * 4


def dequant_bytes(c) -> int:
    n = c.N * c.K
    return c.weight_bytes + n * 4


class ClockSampler:
    """nvidia-smi samples (timestamped) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index, self.period_ms = index, period_ms
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        source = "timed_region"
        if len(inside) < 3:
            inside = [p for (t, p) in self.samples if t0 - 1.0 <= t <= t1 + 1.0]
            source = "timed_region_pm_1s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max((num(p[2]) or 0.0) for p in inside),
                "reasons": reasons, "samples": len(inside), "source": source}


# ------------------------------------------------------------ reference arm

def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """The CPU oracle on a bounded sample of one step: the first `cols` output
    columns (the rows of W they stream) of each of layer 0's seven
    projections, with `cols` sized so that the sample takes about `budget_s`
    seconds.  Every layer has the same shapes and weight distribution, so a
    column of layer 0 costs what any layer's does.  The metric is a rate,
    weight bytes streamed per second, so the sample's own bytes over its own
    time need no scaling.  With parallel=True the oracle is the OpenMP build
    of the same source (entries shared over every core)."""

    def __init__(self, budget_s: float, parallel: bool):
        import oracle
        self.parallel = parallel
        if parallel:
            os.environ.setdefault("OMP_NUM_THREADS", str(host_cores()))
            self.threads = int(os.environ["OMP_NUM_THREADS"])
            self.o = oracle.load_parallel()
        else:
            self.threads = 1
            self.o = oracle.load()
        self.cases = synth.workload(4, layers=1, sweep_m=(1,))
        self.data = {c.name: (c.acts(), c.weights()) for c in self.cases}
        # Calibrate seconds per column per unit of K.
        c = self.cases[0]
        n0 = 4 * self.threads
        self._run(c, n0)
        t0 = time.perf_counter()
        self._run(c, n0)
        per_col_k = (time.perf_counter() - t0) / (n0 * c.K)
        share = budget_s / len(self.cases)
        self.cols = {x.name: int(max(1, min(x.N, share / (per_col_k * x.K)))) for x in self.cases}

    def _run(self, c, n):
        A, blob = self.data[c.name]
        mi, ni = np.repeat(np.arange(c.M), n), np.tile(np.arange(n), c.M)
        self.o.matmul_q4_0_entries(A, blob, c.N, c.K, mi, ni)

    def run(self) -> float:
        """One sampled step; its wall time in seconds."""
        t0 = time.perf_counter()
        for c in self.cases:
            self._run(c, self.cols[c.name])
        return time.perf_counter() - t0

    @property
    def weight_bytes(self) -> int:
        """Q4_0 bytes of the sampled columns (each column is one row of W)."""
        return sum(self.cols[c.name] * (c.K // 32) * 18 for c in self.cases)

    def describe(self) -> str:
        per = ", ".join(f"{c.tags[1][1]} {self.cols[c.name]}/{c.N}" for c in self.cases)
        return (f"{'OpenMP, ' + str(self.threads) + ' threads' if self.parallel else 'one thread'}: "
                f"the first columns of each of layer 0's seven M=1 projections per step "
                f"({per}; {self.weight_bytes} weight bytes); value = sampled weight bytes / "
                f"sample time")


def run_reference(args, rank: int, world: int) -> None:
    """The CPU oracle as the reference arm, each step a bounded sample of the
    step's workload, timed whole (no extrapolation)."""
    if rank != 0:
        return
    budget = min(4.0, max(0.05, 100.0 / (args.steps + args.warmup)))
    st = OracleSample(budget, parallel=True)
    for _ in range(args.warmup):
        st.run()
    times = [st.run() for _ in range(args.steps)]
    step_s = statistics.mean(times)
    value = st.weight_bytes / step_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": st.threads, "kind": "oracle",
                         "sample": st.describe()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "sample_note": "ms_per_step is the measured time of the sampled step, not extrapolated",
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_leg() -> dict:
    """The oracle timed on this host on a column sample of the step: one
    thread (~8 s) and all cores with OpenMP (~8 s)."""
    out = {}
    for parallel in (False, True):
        st = OracleSample(8.0, parallel)
        t = st.run()
        out["parallel" if parallel else "single"] = {
            "value": st.weight_bytes / t / 1e9, "unit": "GB/s", "cores": st.threads,
            "seconds": t, "sample": st.describe()}
    par = out["parallel"]
    return {"value": par["value"], "unit": "GB/s", "cores": par["cores"], "kind": "oracle",
            "sample": par["sample"], "host_cores": host_cores(),
            "single_thread": out["single"]}


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import bit_block_quantized_qm_gb300 as qm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    qm.load_library()
    peaks = measured_peaks()
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)

    # The step's operands.  The 224 weights are resident (loaded once, as a
    # model's are) and read only; each step's inputs are the layers'
    # activation vectors, its result the 224 output vectors, each held in one
    # contiguous buffer per replica so that a step moves them with one copy
    # each way.  Within a layer q, k and v read one vector (the attention
    # input), gate and up another (the FFN input), o and down their own.
    cases = sweep_cases()
    weights, a_host, c_total, reps = sweep_operands(qm, torch, dev, cases, STEP_REPLICAS)
    wbytes = sum(c.weight_bytes for c in cases)
    alg_bytes = sum(gemv_bytes(c) for c in cases)

    def step(rp, ev=None):
        if ev is not None:
            ev[0].record(stream)
        rc = qm.qm_gemv_q4_0_list_ptr(rp["problems"], 1, 0, sh)
        if rc != qm.QM_OK:
            raise RuntimeError(f"decoder sweep list: {qm.qm_status_string(rc)}")
        if ev is not None:
            ev[1].record(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # Warm-up: the --warmup steps, then more until the GPU has run for at
    # least WARMUP_S seconds (the SM clock ramps up under load).
    t_warm = time.time()
    i = 0
    while i < args.warmup or time.time() - t_warm < WARMUP_S:
        step(reps[i % STEP_REPLICAS])
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if qm.qm_device_status(clear=True) != qm.QM_OK:
        raise RuntimeError("device error word set during warm-up")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = qm.qm_launch_count()
    barrier()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(reps[i % STEP_REPLICAS])
    end.record(stream)
    barrier()
    t_wall1 = time.time()
    launches = qm.qm_launch_count() - launches0
    total_ms = start.elapsed_time(end)
    # Keep the GPU busy long enough for the clock sampler to see it under load.
    if t_wall1 - t_wall0 < 1.0:
        t_soak0 = time.time()
        i = 0
        while time.time() - t_soak0 < 1.5:
            step(reps[i % STEP_REPLICAS])
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        t_wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    if qm.qm_device_status(clear=True) != qm.QM_OK:
        raise RuntimeError("device error word set during the timed region")

    ms_step = max_over_ranks(total_ms / args.steps, dist, dev)
    value = job_gbs(wbytes, world, ms_step)

    # The kernel alone: events on the launching stream around each call of a
    # second pass (a call is two launches of the list kernel, back to back;
    # the gap between two steps is the difference from ms_step).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(reps[i % STEP_REPLICAS], evs[i])
    torch.cuda.synchronize()
    call_ms = [ev[0].elapsed_time(ev[1]) for ev in evs]
    launch_ms = statistics.mean(call_ms)

    # ---------------------------------------------------------------- e2e
    # Each step copies its activations in from pinned host memory, runs, and
    # copies its outputs back, as a decode loop would: inputs on one copy
    # stream, the kernel on the main stream, outputs on a second copy stream,
    # so that step i + 1's inputs and step i - 1's outputs move while step i
    # computes.  A replica's buffers are refilled only after its previous
    # step's outputs have been read back.
    a_pinned = torch.from_numpy(a_host).pin_memory()
    c_pinned = torch.empty(c_total, dtype=torch.float32).pin_memory()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    freed = [None] * STEP_REPLICAS

    def e2e_step(i):
        r = i % STEP_REPLICAS
        rp = reps[r]
        with torch.cuda.stream(s_in):
            if freed[r] is not None:
                s_in.wait_event(freed[r])
            rp["A"].copy_(a_pinned, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        stream.wait_event(ev_in)
        step(rp)
        ev_c = torch.cuda.Event()
        ev_c.record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c)
            c_pinned.copy_(rp["C"], non_blocking=True)
            ev_out = torch.cuda.Event()
            ev_out.record(s_out)
        freed[r] = ev_out

    h2d = a_pinned.numel() * 4
    d2h = c_pinned.numel() * 4
    e2e_steps = max(3, min(args.steps, 100))
    for i in range(2 * STEP_REPLICAS):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    e2e_value = job_gbs(wbytes, world, e2e_ms)
    # Outputs read back against a fresh device result of the same list.
    torch.cuda.synchronize()
    e2e_readback_ok = bool(torch.equal(c_pinned, reps[(e2e_steps - 1) % STEP_REPLICAS]["C"].cpu()))
    del a_pinned, c_pinned

    # ------------------------------------------------------------ roofline
    hbm = peaks["hbm_gbs"]
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm",
                "kernel": "gemv_q4_0_list (persistent list GEMV, mma.sync bf16 split, f32 accumulation)",
                "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": measured_traffic("gemv_q4_0_list", WORKLOAD),
                "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": alg_bytes,
                "algorithmic_bytes_definition": "sum over the 224 GEMVs of N*K*0.5625 weight + K*4 A + N*4 C",
                "launch_unit": "one qm_gemv_q4_0_list call: two launches of the list kernel (128 and 96 "
                               "problems); achieved and traffic are per call",
                "launch_ms": launch_ms,
                "launch_ms_median": statistics.median(call_ms), "launch_ms_min": min(call_ms),
                "calls_timed": len(call_ms),
                "weight_gbs_per_launch": wbytes / (launch_ms * 1e-3) / 1e9,
                "per_config": {}}

    prefill = None
    q8 = None
    host_cost = None
    if not args.no_sweep:
        legs = configs_leg(qm, dev, peaks, clocks, cases, weights)
        roofline["per_config"].update(legs["gemv"])
        prefill = legs["prefill"]
        q8 = legs["q8_0"]
        host_cost = legs["host"]
    del weights, reps

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": bench_config(world),
        "hbm_frac": value / hbm,
        "roofline": roofline,
        "prefill": prefill,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "readback_matches_device": e2e_readback_ok,
                "inputs": "the 128 activation vectors (4 per layer) in, the 224 output vectors out; the "
                          "3.93 GB of weights resident (loaded once before timing)",
                "overlap": "inputs, kernel and outputs on three streams; step i+1's inputs "
                           "and step i-1's outputs move while step i computes"},
        "gpu_launches": launches,
        "host_us_per_call": host_cost,
        "q8_0": q8,
        "clocks": clocks,
        "hbm_peak_gbs": hbm, "peak_source": peaks["source"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_leg()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def graph_ms(torch, fn, passes: int = 5) -> float:
    """Capture fn() (launches on the current stream) into a CUDA graph after two
    eager warm-up calls, replay it, and return the best per-replay time (ms)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(passes):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return best


MMAS_PER_PRODUCT = 4  # the tensor-core GEMM takes all four bf16 piece products


def timed_loop(torch, fn, calls: int, warm: int = 3) -> float:
    """Mean ms per call of fn(i) over `calls` calls (events around the loop,
    none in between), after `warm` untimed calls."""
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(calls):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls


def configs_leg(qm, dev, peaks, clocks, cases, weights) -> dict:
    """Every other workload, each on its own synthetic inputs (`cases` and
    `weights`: the decoder sweep's 224 GEMVs and their resident weights):

    GEMV / dequant rows (weight GB/s against HBM):
      cfg0: GEMV M=1, K=N=4096 (9.44 MB), 16 weight replicas back to back in
            a CUDA graph (the replicas exceed L2);
      cfg1: GEMV M=8 up (K=4096, N=14336) and down (K=14336, N=4096), 4
            rotating replicas, each launch timed with events around it;
      cfg1_dequant: dequant of the 14336 x 4096 weight, 4 rotating replicas;
      cfg4 M=1 / M=8: the 32-layer decoder sweep (q, k, v, o, gate, up, down;
            hidden 4096, GQA; 3.93 GB of weights, all resident), a CUDA graph
            of its 224 launches, as a decode loop replays it; also with q|k|v
            and gate|up stacked by rows (128 launches).  Activations: one
            synthetic A per (M, K), shared by the layers (no attention or
            activation functions between the projections).
    GEMM rows (TFLOP/s against the tensor-core bound, bf16 peak / 4 MMAs per
    product, and against the FP32 FMA peak):
      cfg2: M=32 and M=256 at K=N=4096 (A with 1% outliers), 16 weight replicas;
      cfg3: M=1024 at (K=4096, N=14336) and (K=14336, N=4096), 2 replicas;
      cfg4 M=512: the decoder sweep, eager launches.
    """
    import torch
    hbm = peaks["hbm_gbs"]
    bf16 = peaks["bf16_tflops"]
    tc_bound = bf16 / MMAS_PER_PRODUCT
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    fp32_peak = sm_count * 128 * 2 * sm_max * 1e6 / 1e12
    sh = lambda: int(torch.cuda.current_stream().cuda_stream)  # noqa: E731
    gemv, prefill = {}, {}

    def mm(A, W, C, M, N, K, what):
        rc = qm.qm_matmul_q4_0_ptr(A.data_ptr(), W.data_ptr(), C.data_ptr(), M, N, K, sh())
        if rc != qm.QM_OK:
            raise RuntimeError(f"{what}: {qm.qm_status_string(rc)}")

    def gemv_row(workload, kernel, wbytes, ms, launches=1):
        gbs = wbytes / (ms * 1e-3) / 1e9
        return {"workload": workload, "kernel": kernel, "ms": ms, "weight_gbs": gbs,
                "frac": gbs / hbm, "bound": "hbm", "launches": launches}

    def gemm_row(workload, flops, ms):
        tf = flops / (ms * 1e-3) / 1e12
        return {"workload": workload, "kernel": "gemm_q4_0_tc", "ms": ms, "tflops": tf,
                "frac": tf / tc_bound, "bound": "tensor", "peak": tc_bound,
                "vs_fp32_fma_peak": tf / fp32_peak}

    # cfg0: back-to-back M = 1 GEMVs at K = N = 4096.
    c0 = synth.workload(0)[0]
    w0 = [torch.from_numpy(c0.weights()).to(dev) for _ in range(16)]
    a0 = torch.from_numpy(c0.acts()).to(dev)
    o0 = torch.empty((1, c0.N), dtype=torch.float32, device=dev)

    def m1_fn():
        for w in w0:
            mm(a0, w, o0, 1, c0.N, c0.K, "cfg0")
    ms0 = graph_ms(torch, m1_fn) / len(w0)
    gemv["cfg0_gemv_m1_k4096_n4096"] = gemv_row(
        "GEMV M=1, K=N=4096, 16 replicas back to back in a CUDA graph", "gemv_q4_0_tc",
        c0.weight_bytes, ms0)

    # The same GEMVs with the activations quantized to Q8_0 first (the
    # act-quant fused GEMV, qm_matmul_q4_0_q8act): a different product, timed
    # on the same weights.
    def q8act(A, W, C, M, N, K, what):
        rc = qm.qm_matmul_q4_0_q8act_ptr(A.data_ptr(), W.data_ptr(), C.data_ptr(), M, N, K, sh())
        if rc != qm.QM_OK:
            raise RuntimeError(f"{what}: {qm.qm_status_string(rc)}")

    def m1_q8_fn():
        for w in w0:
            q8act(a0, w, o0, 1, c0.N, c0.K, "cfg0 q8act")
    ms0q = graph_ms(torch, m1_q8_fn) / len(w0)
    gemv["cfg0_q8act_m1_k4096_n4096"] = gemv_row(
        "GEMV M=1, K=N=4096 with the activations quantized to Q8_0 in the kernel "
        "(qm_matmul_q4_0_q8act), 16 replicas back to back in a CUDA graph", "gemv_q4_0_tc<q8>",
        c0.weight_bytes, ms0q)
    del w0

    # cfg1: the M = 8 decode-batch GEMVs, each launch between two events.
    for key, c in zip(("cfg1_gemv_up", "cfg1_gemv_down"), step_cases()[:2]):
        ws = [torch.from_numpy(c.weights()).to(dev) for _ in range(REPLICAS)]
        A = torch.from_numpy(c.acts()).to(dev)
        C = torch.empty((c.M, c.N), dtype=torch.float32, device=dev)
        for i in range(2 * REPLICAS):
            mm(A, ws[i % REPLICAS], C, c.M, c.N, c.K, c.name)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(40)]
        for i, ev in enumerate(evs):
            ev[0].record()
            mm(A, ws[i % REPLICAS], C, c.M, c.N, c.K, c.name)
            ev[1].record()
        torch.cuda.synchronize()
        ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs)
        row = gemv_row(f"{c.name}: M=8 decode batch, {REPLICAS} rotating weight replicas, "
                       "events around each launch", "gemv_q4_0_tc", c.weight_bytes, ms)
        row["alg_gbs"] = gemv_bytes(c) / (ms * 1e-3) / 1e9
        row["algorithmic_bytes_per_launch"] = gemv_bytes(c)
        row["traffic"] = measured_traffic("gemv_q4_0_tc", c.name)
        gemv[key] = row
        del ws, A, C

    # cfg1 dequant.
    deq = step_cases()[2]
    nb = deq.weight_bytes // 18
    dw = [torch.from_numpy(deq.weights()).to(dev) for _ in range(REPLICAS)]
    dout = [torch.empty(nb * 32, dtype=torch.float32, device=dev) for _ in range(REPLICAS)]

    def deq_fn(i):
        rc = qm.qm_dequant_q4_0_ptr(dw[i % REPLICAS].data_ptr(), nb, dout[i % REPLICAS].data_ptr(), sh())
        if rc != qm.QM_OK:
            raise RuntimeError(f"dequant: {qm.qm_status_string(rc)}")
    ms = timed_loop(torch, deq_fn, 20)
    row = gemv_row("dequant_q4_0 of the 14336 x 4096 weight, 4 rotating replicas",
                   "dequant_q4_0_fast", deq.weight_bytes, ms)
    row["alg_gbs"] = dequant_bytes(deq) / (ms * 1e-3) / 1e9
    row["frac"] = row["alg_gbs"] / hbm
    row["algorithmic_bytes_per_launch"] = dequant_bytes(deq)
    row["traffic"] = measured_traffic("dequant_q4_0", deq.name)
    gemv["cfg1_dequant"] = row
    del dw, dout

    # cfg2 and cfg3: prefill GEMMs.
    for c in synth.workload(2) + synth.workload(3):
        reps = 16 if c.weight_bytes < 16 << 20 else 2
        ws = [torch.from_numpy(c.weights()).to(dev) for _ in range(reps)]
        A = torch.from_numpy(c.acts()).to(dev)
        C = torch.empty((c.M, c.N), dtype=torch.float32, device=dev)
        calls = 32 if c.M < 1024 else 6

        def fn(i, ws=ws, A=A, C=C, c=c):
            mm(A, ws[i % len(ws)], C, c.M, c.N, c.K, c.name)
        ms = timed_loop(torch, fn, calls)
        key = ("cfg2_" if c.M < 1024 else "cfg3_") + c.name
        prefill[key] = gemm_row(f"{c.name} ({reps} weight replicas)", 2.0 * c.M * c.N * c.K, ms)
        del ws, A, C

    # cfg4: the 32-layer decoder sweep.
    wbytes = sum(c.weight_bytes for c in cases)
    layer_shapes = [(c.N, c.K) for c in cases[:7]]

    def acts(M):
        return {K: torch.from_numpy(synth.activations(M, K, 5, key=(2, M, K))).to(dev)
                for K in (4096, 14336)}

    def sweep_fn(M, A, outs):
        def fn():
            for i, c in enumerate(cases):
                mm(A[c.K], weights[i], outs[i % 7], M, c.N, c.K, f"sweep {c.name} M={M}")
        return fn

    # The sweep through the act-quant fused GEMV (qm_matmul_q4_0_q8act).
    for M in (1, 8):
        A = acts(M)
        outs = [torch.empty((M, N), dtype=torch.float32, device=dev) for (N, K) in layer_shapes]

        def q8_sweep(M=M, A=A, outs=outs):
            for i, c in enumerate(cases):
                q8act(A[c.K], weights[i], outs[i % 7], M, c.N, c.K, f"q8act sweep {c.name} M={M}")
        ms = graph_ms(torch, q8_sweep)
        gemv[f"cfg4_sweep_m{M}_q8act"] = gemv_row(
            f"32-layer decoder sweep at M={M} with the activations quantized to Q8_0 in the kernel "
            f"(qm_matmul_q4_0_q8act): CUDA graph of {len(cases)} launches", "gemv_q4_0_tc<q8>",
            wbytes, ms, len(cases))

    for M in (1, 8):
        A = acts(M)
        outs = [torch.empty((M, N), dtype=torch.float32, device=dev) for (N, K) in layer_shapes]
        ms = graph_ms(torch, sweep_fn(M, A, outs))
        gemv[f"cfg4_sweep_m{M}"] = gemv_row(
            f"32-layer decoder sweep at M={M}: CUDA graph of {len(cases)} GEMV launches, "
            "3.93 GB of weights per pass", "gemv_q4_0_tc", wbytes, ms, len(cases))

    # M = 1 through the list GEMV (qm_gemv_q4_0_list, one persistent launch
    # per list), every problem with its own output:
    #   * per_group: 4 lists per layer, [q, k, v], [o], [gate, up], [down], as an
    #     engine with attention and activation kernels in between launches them;
    #   * one_list: all 224 GEMVs of the sweep in one list, independent;
    #   * chained: the same list with the decoder's ordering (q, k, v wait for the
    #     previous layer's down; o for v; gate and up for o; down for up): every
    #     activation read waits for those problems to finish on every SM, as a
    #     chain of dependent projections would (the activations themselves stay
    #     the shared synthetic ones, so values do not grow through 224 products).
    A1 = acts(1)
    louts = [torch.empty((1, c.N), dtype=torch.float32, device=dev) for c in cases]
    ctr = torch.zeros(len(cases), dtype=torch.int32, device=dev)
    # Within a layer: the index of the last problem each projection waits for
    # (None: the previous layer's down).
    proj_wait = {"q": None, "k": None, "v": None, "o": 2, "gate": 3, "up": 3, "down": 5}

    def list_problems(chained):
        out = []
        for i, c in enumerate(cases):
            wf = -1
            if chained:
                layer, p = divmod(i, 7)
                rel = proj_wait[DECODER_PROJS[p]]
                wf = 7 * layer + rel if rel is not None else 7 * layer - 1
            out.append((A1[c.K].data_ptr(), weights[i].data_ptr(), louts[i].data_ptr(), c.N, c.K, wf))
        return out

    def run_lists(lists, with_ctr):
        s = sh()
        for lst in lists:
            rc = qm.qm_gemv_q4_0_list_ptr(lst, 1, ctr.data_ptr() if with_ctr else 0, s)
            if rc != qm.QM_OK:
                raise RuntimeError(f"gemv list: {qm.qm_status_string(rc)}")

    groups = []
    for layer in range(32):
        b = 7 * layer
        ps = list_problems(False)[b:b + 7]
        groups += [ps[0:3], ps[3:4], ps[4:6], ps[6:7]]
    variants = (("per_group", groups, False, len(groups)),
                ("one_list", [list_problems(False)], False, 1),
                ("chained", [list_problems(True)], True, 1))
    for name, lists, with_ctr, nl in variants:
        ms = graph_ms(torch, lambda lists=lists, with_ctr=with_ctr: run_lists(lists, with_ctr))
        gemv[f"cfg4_sweep_m1_list_{name}"] = gemv_row(
            f"32-layer decoder sweep at M=1 through qm_gemv_q4_0_list ({name}): CUDA graph of "
            f"{nl} list launches", "gemv_q4_0_list", wbytes, ms, nl)

    # The act-quant product through its list (qm_gemv_q4_0_q8act_list): one
    # list of all 224 independent GEMVs, and the chained one.
    def run_q8_lists(lists, with_ctr):
        s = sh()
        for lst in lists:
            rc = qm.qm_gemv_q4_0_list_ptr(lst, 1, ctr.data_ptr() if with_ctr else 0, s, q8act=True)
            if rc != qm.QM_OK:
                raise RuntimeError(f"q8act gemv list: {qm.qm_status_string(rc)}")
    for name, lists, with_ctr, nl in variants[1:]:
        ms = graph_ms(torch, lambda lists=lists, with_ctr=with_ctr: run_q8_lists(lists, with_ctr))
        gemv[f"cfg4_sweep_m1_q8act_list_{name}"] = gemv_row(
            f"32-layer decoder sweep at M=1 with the activations quantized to Q8_0 in the kernel, "
            f"through qm_gemv_q4_0_q8act_list ({name}): CUDA graph of {nl} list launches",
            "gemv_q4_0_list<q8>", wbytes, ms, nl)
    del louts

    # The same weights with q|k|v and gate|up stacked by rows (one row-major
    # block stream each, as an engine with fused projections stores them).
    fused = []
    for layer in range(32):
        w = weights[7 * layer:7 * layer + 7]
        fused += [torch.cat([w[0], w[1], w[2]]), w[3], torch.cat([w[4], w[5]]), w[6]]
    fused_shapes = [(4096 + 1024 + 1024, 4096), (4096, 4096), (2 * 14336, 4096), (4096, 14336)]
    for M in (1, 8):
        A = acts(M)
        outs = [torch.empty((M, N), dtype=torch.float32, device=dev) for (N, K) in fused_shapes]

        def fused_fn(M=M, A=A, outs=outs):
            for i, wf in enumerate(fused):
                N, K = fused_shapes[i % 4]
                mm(A[K], wf, outs[i % 4], M, N, K, f"stacked sweep M={M}")
        ms = graph_ms(torch, fused_fn)
        gemv[f"cfg4_sweep_m{M}_stacked"] = gemv_row(
            f"the decoder sweep at M={M} with q|k|v and gate|up stacked by rows: CUDA graph of "
            f"{len(fused)} GEMV launches", "gemv_q4_0_tc", wbytes, ms, len(fused))
    del fused

    # The sweep at M = 512, eager launches.
    A = acts(512)
    outs = [torch.empty((512, N), dtype=torch.float32, device=dev) for (N, K) in layer_shapes]
    fn = sweep_fn(512, A, outs)
    ms = timed_loop(torch, lambda i: fn(), 3, warm=1)
    flops = sum(2.0 * 512 * c.N * c.K for c in cases)
    prefill["cfg4_sweep_m512"] = gemm_row("32-layer decoder sweep at M=512 (7.15 TFLOP per pass), "
                                          "eager launches", flops, ms)
    prefill["bound_note"] = (f"tensor-core bound = measured bf16 dense peak {bf16} TFLOP/s / "
                             f"{MMAS_PER_PRODUCT} bf16 MMAs per useful product; FP32 FMA peak "
                             f"{fp32_peak:.1f} TFLOP/s at {sm_max} MHz")
    del A, outs, fn
    torch.cuda.empty_cache()
    return {"gemv": gemv, "prefill": prefill, "q8_0": q8_0_leg(qm, dev, peaks),
            "host": host_cost_leg(qm, dev)}


def host_cost_leg(qm, dev) -> dict:
    """Host time per call, eager: 200 calls enqueued back to back (the GPU
    queue never fills), wall clock around the enqueue loop only.  Includes
    the ctypes call from Python; ``ctypes_floor`` is a call of qm_version
    through the same binding."""
    import torch
    sh = int(torch.cuda.current_stream().cuda_stream)

    def per_call(fn, n=200):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        return (t1 - t0) / n * 1e6

    lib = qm.load_library()
    out = {"unit": "us per call", "ctypes_floor": per_call(lambda: lib.qm_version(), 2000)}
    for name, (M, N, K) in (("gemv_m1_k4096_n4096", (1, 4096, 4096)), ("gemv_m8_k4096_n14336", (8, 14336, 4096)),
                            ("gemm_m512_k4096_n4096", (512, 4096, 4096))):
        w = torch.from_numpy(synth.q4_0_weights(N, K, 1)).to(dev)
        a = torch.from_numpy(synth.activations(M, K, 2)).to(dev)
        c = torch.empty((M, N), dtype=torch.float32, device=dev)

        def call(a=a, w=w, c=c, M=M, N=N, K=K):
            rc = qm.qm_matmul_q4_0_ptr(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, sh)
            if rc != qm.QM_OK:
                raise RuntimeError(qm.qm_status_string(rc))
        out["qm_matmul_q4_0_" + name] = per_call(call, 200 if M < 512 else 50)
        del w, a, c
    cases = synth.workload(4, layers=1, sweep_m=(1,))
    ws = [torch.from_numpy(c.weights()).to(dev) for c in cases]
    acts = {K: torch.from_numpy(synth.activations(1, K, 5)).to(dev) for K in (4096, 14336)}
    outs = [torch.empty((1, c.N), dtype=torch.float32, device=dev) for c in cases]
    problems = [(acts[c.K].data_ptr(), w.data_ptr(), o.data_ptr(), c.N, c.K, -1)
                for c, w, o in zip(cases, ws, outs)]

    def list_call():
        rc = qm.qm_gemv_q4_0_list_ptr(problems, 1, 0, sh)
        if rc != qm.QM_OK:
            raise RuntimeError(qm.qm_status_string(rc))
    out["qm_gemv_q4_0_list_one_layer_7_problems"] = per_call(list_call, 100)
    return out


def q8_0_leg(qm, dev, peaks) -> dict:
    """Q8_0 quantize and dequant of a 14336 x 4096 tensor (58.7 M elements),
    4 rotating replicas (> L2), CUDA events over 20 calls each after warm-up.
    Algorithmic bytes per call (the page's cost model): n * 4 + n * 1.0625."""
    import torch
    n = 14336 * 4096
    reps = 4
    g = synth.rng(6, (0,))
    x_host = g.standard_normal(n).astype(np.float32)
    xs = [torch.from_numpy(x_host).to(dev) for _ in range(reps)]
    qs = [torch.empty(n // 32 * 34, dtype=torch.uint8, device=dev) for _ in range(reps)]
    ys = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(reps)]
    sh = int(torch.cuda.current_stream().cuda_stream)

    def timed(fn, calls=20):
        for i in range(4):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(calls):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / calls

    def quant(i):
        rc = qm.qm_quantize_q8_0_ptr(xs[i % reps].data_ptr(), n, qs[i % reps].data_ptr(), sh)
        if rc != qm.QM_OK:
            raise RuntimeError(f"quantize_q8_0: {qm.qm_status_string(rc)}")

    def deq(i):
        rc = qm.qm_dequant_q8_0_ptr(qs[i % reps].data_ptr(), n // 32, ys[i % reps].data_ptr(), sh)
        if rc != qm.QM_OK:
            raise RuntimeError(f"dequant_q8_0: {qm.qm_status_string(rc)}")

    nbytes = n * 4 + n // 32 * 34
    hbm = peaks["hbm_gbs"]
    out = {"workload": "Q8_0 quantize and dequant of 14336 x 4096 f32 (58.7 M elements), "
                       "4 rotating replicas",
           "algorithmic_bytes_per_call": nbytes}
    for name, fn in (("quantize", quant), ("dequant", deq)):
        ms = timed(fn)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "gbs": gbs, "hbm_frac": gbs / hbm}
    del xs, qs, ys
    torch.cuda.empty_cache()
    return out


def profile_case(args) -> None:
    """Run one operation a few times on cuda:0 and exit, for profiler captures
    (``--profile-case gemm --M .. --N .. --K .. [--algo QM_ALGO_*]``, any M;
    ``--profile-case q8act --M .. --N .. --K ..``, M <= 8; ``--profile-case
    list --layers L``: the bench step's list for L layers (the decoder
    sweep's shapes, weights and activation vectors) through
    qm_gemv_q4_0_list (``--q8act``: qm_gemv_q4_0_q8act_list);
    ``--profile-case dequant``: dequant_q4_0 of the 14336 x 4096 weight; or
    ``--profile-case q8_0``).
    Prints a one-line note, not a bench line."""
    import torch
    import bit_block_quantized_qm_gb300 as qm
    qm.load_library()
    dev = torch.device("cuda", 0)
    sh = int(torch.cuda.current_stream().cuda_stream)
    if args.profile_case in ("gemm", "q8act"):
        M, N, K = args.M, args.N, args.K
        blob = synth.q4_0_weights(N, K, 1)
        A = synth.activations(M, K, 2)
        w = torch.from_numpy(blob).to(dev)
        a = torch.from_numpy(A).to(dev)
        c = torch.empty((M, N), dtype=torch.float32, device=dev)
        for _ in range(args.calls):
            if args.profile_case == "gemm":
                rc = qm.qm_matmul_q4_0_algo_ptr(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K,
                                                args.algo, sh)
            else:
                rc = qm.qm_matmul_q4_0_q8act_ptr(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, sh)
            if rc != qm.QM_OK:
                raise RuntimeError(qm.qm_status_string(rc))
    elif args.profile_case == "list":
        cases = synth.workload(4, layers=args.layers, sweep_m=(1,))
        _, _, _, reps = sweep_operands(qm, torch, dev, cases, 1)
        for _ in range(args.calls):
            rc = qm.qm_gemv_q4_0_list_ptr(reps[0]["problems"], 1, 0, sh, q8act=args.q8act)
            if rc != qm.QM_OK:
                raise RuntimeError(qm.qm_status_string(rc))
    elif args.profile_case == "dequant":
        deq = step_cases()[2]
        nb = deq.weight_bytes // 18
        w = torch.from_numpy(deq.weights()).to(dev)
        out = torch.empty(nb * 32, dtype=torch.float32, device=dev)
        for _ in range(args.calls):
            rc = qm.qm_dequant_q4_0_ptr(w.data_ptr(), nb, out.data_ptr(), sh)
            if rc != qm.QM_OK:
                raise RuntimeError(qm.qm_status_string(rc))
    else:
        n = 14336 * 4096
        x = torch.from_numpy(synth.rng(6, (0,)).standard_normal(n).astype(np.float32)).to(dev)
        q = torch.empty(n // 32 * 34, dtype=torch.uint8, device=dev)
        y = torch.empty(n, dtype=torch.float32, device=dev)
        for _ in range(args.calls):
            for rc in (qm.qm_quantize_q8_0_ptr(x.data_ptr(), n, q.data_ptr(), sh),
                       qm.qm_dequant_q8_0_ptr(q.data_ptr(), n // 32, y.data_ptr(), sh)):
                if rc != qm.QM_OK:
                    raise RuntimeError(qm.qm_status_string(rc))
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "calls": args.calls}), flush=True)


def main(argv=None) -> None:
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip the CPU oracle timing (for profiler runs)")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the M=1 GEMV, decoder-sweep and prefill reports (profiler runs)")
    p.add_argument("--profile-case", choices=("gemm", "q8act", "list", "q8_0", "dequant"), default=None,
                   help="run one operation a few times and exit (profiler captures)")
    p.add_argument("--M", type=int, default=512)
    p.add_argument("--N", type=int, default=4096)
    p.add_argument("--K", type=int, default=4096)
    p.add_argument("--calls", type=int, default=3)
    p.add_argument("--layers", type=int, default=8, help="decoder layers for --profile-case list")
    p.add_argument("--q8act", action="store_true",
                   help="--profile-case list through qm_gemv_q4_0_q8act_list (the act-quant product)")
    p.add_argument("--algo", type=int, default=0,
                   help="QM_ALGO_* value for --profile-case gemm (0: automatic choice)")
    args = p.parse_args(argv)
    if args.profile_case:
        profile_case(args)
        return
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
