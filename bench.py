"""Benchmark of the Q4_0 x f32 hot path on GB300 (one JSON line on stdout).

One step = one pass of the whole hot path over the decode-batch workload:
  * GEMV M=8, K=4096,  N=14336 (FFN up projection),
  * GEMV M=8, K=14336, N=4096  (FFN down projection),
  * dequant_q4_0 of the 14336 x 4096 weight to f32,
each through libqm's C ABI (qm_matmul_q4_0 / qm_dequant_q4_0) on one stream.
Inputs are synthetic (seeded generators in ``synth``).  Every step uses a
different replica of all operands, and the replicas together exceed the L2
several times, so no step finds its inputs in L2.

value = Q4_0 weight bytes streamed per step / device time per step (GB/s),
timed with CUDA events over --steps steps after --warmup steps.  ``e2e``
repeats the step with host operands: pinned host -> device copies of every
input and device -> host copies of every output inside the timed region, the
copies of neighbouring steps overlapping a step's kernels on separate streams.

Beside the step, the line reports (keys ``m1_gemv``, ``decode_sweep``,
``prefill``, ``q8_0``): back-to-back M=1 GEMVs at K=N=4096, the 32-layer
decoder sweep at M=1 and M=8 replayed from a CUDA graph (weight GB/s against
HBM), the same sweep at M=512 (TFLOP/s against the tensor-core bound of the
3-MMA split), and the Q8_0 quantize and dequant of a 14336 x 4096 tensor (GB/s
against HBM).

``--impl reference`` times the CPU oracle instead (on a bounded sample of the
same step, extrapolated per column), on the same metric.
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
WORKLOAD = "q4_0_decode_batch_m8_ffn_up_down_plus_dequant"
FALLBACK_HBM_GBS = 6800.0
REPLICAS = 4  # 4 x (99 MB read + 235 MB written) >> 129 MB of L2


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
                  "gemm_q4_0_tc": "gemm_tc.cu"}


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

class OracleStep:
    """The CPU oracle on one step of the workload, bounded to a time budget:
    it computes the first `cols` output columns (all M rows) of each GEMV and
    the first `blocks` blocks of the dequant, and scales each part's time by
    (total / computed).  With a large enough budget the sample is the whole
    step.  Single-threaded."""

    def __init__(self, budget_s: float):
        import oracle
        self.o = oracle.load()
        self.up, self.down, self.deq = step_cases()
        self.data = {c.name: (c.acts(), c.weights()) for c in (self.up, self.down)}
        self.deq_blob = self.deq.weights()
        # calibrate seconds per multiply-add on a small slice
        A, blob = self.data[self.up.name]
        mi, ni = np.repeat(np.arange(8), 16), np.tile(np.arange(16), 8)
        self.o.matmul_q4_0_entries(A, blob, self.up.N, self.up.K, mi, ni)
        t0 = time.perf_counter()
        self.o.matmul_q4_0_entries(A, blob, self.up.N, self.up.K, mi, ni)
        per_mac = (time.perf_counter() - t0) / (8 * 16 * self.up.K)
        share = budget_s * 0.48
        self.cols = {c.name: int(max(1, min(c.N, share / (per_mac * c.M * c.K))))
                     for c in (self.up, self.down)}
        nb = self.deq.weight_bytes // 18
        self.blocks = int(max(32, min(nb, budget_s * 0.04 / 1.5e-9 / 32)))

    def run(self):
        t = {}
        for c in (self.up, self.down):
            A, blob = self.data[c.name]
            n = self.cols[c.name]
            mi, ni = np.repeat(np.arange(c.M), n), np.tile(np.arange(n), c.M)
            t0 = time.perf_counter()
            self.o.matmul_q4_0_entries(A, blob, c.N, c.K, mi, ni)
            t[c.name] = (time.perf_counter() - t0) * c.N / n
        nb = self.deq.weight_bytes // 18
        blob = self.deq_blob[: self.blocks * 18]
        t0 = time.perf_counter()
        self.o.dequant_q4_0(blob)
        t["dequant"] = (time.perf_counter() - t0) * nb / self.blocks
        return sum(t.values()), t

    def describe(self) -> str:
        nb = self.deq.weight_bytes // 18
        return (f"per step, one thread: all {self.up.M} rows x first {self.cols[self.up.name]} "
                f"of {self.up.N} columns of the up GEMV, x first {self.cols[self.down.name]} of "
                f"{self.down.N} of the down GEMV, and the first {self.blocks} of {nb} blocks of "
                f"the dequant; each part's time scaled by total/computed")

    @property
    def weight_bytes(self) -> int:
        return self.up.weight_bytes + self.down.weight_bytes + self.deq.weight_bytes


def run_reference(args, rank: int, world: int) -> None:
    """The CPU oracle on the same step (bounded sample, extrapolated)."""
    if rank != 0:
        return
    budget = min(12.0, max(0.05, 75.0 / (args.steps + args.warmup)))
    st = OracleStep(budget)
    for _ in range(args.warmup):
        st.run()
    times, parts = [], []
    for _ in range(args.steps):
        s, p = st.run()
        times.append(s)
        parts.append(p)
    step_s = statistics.mean(times)
    value = st.weight_bytes / step_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 8, "shapes": "K=4096,N=14336; K=14336,N=4096; "
                   "dequant 14336x4096", "seeds": [1, 2]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": st.describe()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "parts_s": {k: statistics.mean(p[k] for p in parts) for k in parts[0]},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_leg() -> dict:
    """The oracle timed on this host (1 thread) on a ~12 s sample of the step."""
    st = OracleStep(12.0)
    total, parts = st.run()
    return {"value": st.weight_bytes / total / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": st.describe(), "seconds_per_step": total,
            "parts_s": parts}


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

    up, down, deq = step_cases()
    host = {"up_A": up.acts(), "up_W": up.weights(), "down_A": down.acts(),
            "down_W": down.weights(), "deq_W": deq.weights()}
    n_blocks = deq.weight_bytes // 18
    reps = []
    for r in range(REPLICAS):
        reps.append({
            "up_A": torch.from_numpy(host["up_A"]).to(dev),
            "up_W": torch.from_numpy(host["up_W"]).to(dev),
            "up_C": torch.empty((up.M, up.N), dtype=torch.float32, device=dev),
            "down_A": torch.from_numpy(host["down_A"]).to(dev),
            "down_W": torch.from_numpy(host["down_W"]).to(dev),
            "down_C": torch.empty((down.M, down.N), dtype=torch.float32, device=dev),
            "deq_W": torch.from_numpy(host["deq_W"]).to(dev),
            "deq_out": torch.empty(n_blocks * 32, dtype=torch.float32, device=dev),
        })
    torch.cuda.synchronize()

    def call(rc, what):
        if rc != qm.QM_OK:
            raise RuntimeError(f"{what}: {qm.qm_status_string(rc)}")

    def step(rp, ev=None):
        if ev is not None:
            ev[0].record(stream)
        call(qm.qm_matmul_q4_0_ptr(rp["up_A"].data_ptr(), rp["up_W"].data_ptr(),
                                   rp["up_C"].data_ptr(), up.M, up.N, up.K, sh), "up")
        if ev is not None:
            ev[1].record(stream)
        call(qm.qm_matmul_q4_0_ptr(rp["down_A"].data_ptr(), rp["down_W"].data_ptr(),
                                   rp["down_C"].data_ptr(), down.M, down.N, down.K, sh), "down")
        if ev is not None:
            ev[2].record(stream)
        call(qm.qm_dequant_q4_0_ptr(rp["deq_W"].data_ptr(), n_blocks, rp["deq_out"].data_ptr(),
                                    sh), "dequant")
        if ev is not None:
            ev[3].record(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step(reps[i % REPLICAS])
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
        step(reps[i % REPLICAS])
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
            step(reps[i % REPLICAS])
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

    # Per-kernel split, from a separate pass with events between the kernels
    # (an event between two kernels also ends their programmatic overlap, so
    # these times are slightly longer than their share of the timed step).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(reps[i % REPLICAS], evs[i])
    torch.cuda.synchronize()
    per_op = {"gemv_up": [], "gemv_down": [], "dequant": []}
    for ev in evs:
        per_op["gemv_up"].append(ev[0].elapsed_time(ev[1]))
        per_op["gemv_down"].append(ev[1].elapsed_time(ev[2]))
        per_op["dequant"].append(ev[2].elapsed_time(ev[3]))
    avg = {k: statistics.mean(v) for k, v in per_op.items()}

    wbytes = up.weight_bytes + down.weight_bytes + deq.weight_bytes
    value = job_gbs(wbytes, world, ms_step)

    # ---------------------------------------------------------------- e2e
    pinned = {k: torch.from_numpy(v.view(np.uint8).ravel() if v.dtype != np.uint8 else v)
              .pin_memory() for k, v in host.items()}
    out_host = {"up_C": torch.empty(up.M * up.N * 4, dtype=torch.uint8).pin_memory(),
                "down_C": torch.empty(down.M * down.N * 4, dtype=torch.uint8).pin_memory(),
                "deq_out": torch.empty(n_blocks * 128, dtype=torch.uint8).pin_memory()}

    # Each step copies its inputs in, runs, and copies its outputs back, as a
    # serving loop would: inputs on one copy stream, the kernels on the main
    # stream, outputs on a second copy stream, so that step i + 1's inputs and
    # step i - 1's outputs move (in opposite directions) while step i
    # computes.  A replica's buffers are refilled only after its previous
    # step's outputs have been read back.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    freed = [None] * REPLICAS

    def e2e_step(i):
        r = i % REPLICAS
        rp = reps[r]
        with torch.cuda.stream(s_in):
            if freed[r] is not None:
                s_in.wait_event(freed[r])
            for k in host:
                rp[k].view(torch.uint8).view(-1).copy_(pinned[k], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        stream.wait_event(ev_in)
        step(rp)
        ev_c = torch.cuda.Event()
        ev_c.record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c)
            for k in out_host:
                out_host[k].copy_(rp[k].view(torch.uint8).view(-1), non_blocking=True)
            ev_out = torch.cuda.Event()
            ev_out.record(s_out)
        freed[r] = ev_out

    h2d = sum(v.nbytes for v in host.values())
    d2h = sum(int(v.numel()) for v in out_host.values())
    e2e_steps = max(3, min(args.steps, 50))
    for i in range(2 * REPLICAS):
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

    # ------------------------------------------------------------ roofline
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = clocks.get("sm_mhz") or 0.0
    sm_max = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    fp32_peak_max = sm_count * 128 * 2 * sm_max * 1e6 / 1e12
    fp32_peak_live = sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12 if sm_mhz else None
    hbm = peaks["hbm_gbs"]
    paths = {}
    for key, c in (("gemv_up", up), ("gemv_down", down)):
        ms = avg[key]
        flops = 2.0 * c.M * c.N * c.K
        paths[key] = {
            "kernel": "gemv_q4_0_tc (mma.sync bf16 split, f32 accumulation)",
            "ms": ms, "weight_gbs": c.weight_bytes / (ms * 1e-3) / 1e9,
            "alg_gbs": gemv_bytes(c) / (ms * 1e-3) / 1e9,
            "hbm_frac": gemv_bytes(c) / (ms * 1e-3) / 1e9 / hbm,
            "tflops": flops / (ms * 1e-3) / 1e12,
            "bound_time_ms": gemv_bytes(c) / (hbm * 1e9) * 1e3,
        }
    paths["dequant"] = {"ms": avg["dequant"],
                        "alg_gbs": dequant_bytes(deq) / (avg["dequant"] * 1e-3) / 1e9,
                        "hbm_frac": dequant_bytes(deq) / (avg["dequant"] * 1e-3) / 1e9 / hbm}
    dominant = max(avg, key=avg.get)
    if dominant == "dequant":
        achieved = paths["dequant"]["alg_gbs"]
        roofline = {"bound": "hbm", "kernel": "dequant_q4_0", "achieved": achieved,
                    "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": measured_traffic("dequant_q4_0", deq.name),
                    "peak_source": peaks["source"],
                    "algorithmic_bytes_per_launch": dequant_bytes(deq)}
    else:
        c = up if dominant == "gemv_up" else down
        achieved = paths[dominant]["alg_gbs"]
        roofline = {"bound": "hbm", "kernel": "gemv_q4_0_tc (" + dominant + ")",
                    "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": measured_traffic("gemv_q4_0_tc", c.name),
                    "peak_source": peaks["source"],
                    "algorithmic_bytes_per_launch": gemv_bytes(c)}

    sweep = None
    if not args.no_sweep:
        sweep = sweep_leg(qm, dev, peaks, fp32_peak_max, fp32_peak_live)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 8,
                   "shapes": "K=4096,N=14336; K=14336,N=4096; dequant 14336x4096",
                   "seeds": [1, 2], "l2": f"{REPLICAS} rotating operand replicas (> L2)",
                   "parallelism": f"replicas x{world}",
                   "value_definition": "Q4_0 weight bytes streamed per step / step time"},
        "roofline": roofline,
        "paths": paths,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "overlap": "inputs, kernels and outputs on three streams; step i+1's inputs "
                           "and step i-1's outputs move while step i computes"},
        "gpu_launches": launches,
        "m1_gemv": sweep["m1_gemv"] if sweep else None,
        "decode_sweep": sweep["decode"] if sweep else None,
        "prefill": sweep["prefill"] if sweep else None,
        "q8_0": sweep["q8_0"] if sweep else None,
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


def sweep_leg(qm, dev, peaks, fp32_peak_max, fp32_peak_live) -> dict:
    """The decoder sweep (32 layers of q, k, v, o, gate, up, down; hidden 4096,
    grouped-query attention) at M = 1, 8 and 512 through qm_matmul_q4_0, plus
    back-to-back M = 1 GEMVs at K = N = 4096.  Weights: all 32 layers resident
    (3.93 GB, far beyond L2).  Activations: one synthetic A per (M, K), shared
    by the layers (the projections are not chained: no attention and no
    activation functions).  M = 1 and 8 replay a CUDA graph of the 224 launches
    (what a decode loop does); M = 512 is launched eagerly."""
    import torch
    hbm = peaks["hbm_gbs"]
    cases = synth.workload(4, layers=32, sweep_m=(1,))
    weights = [torch.from_numpy(c.weights()).to(dev) for c in cases]
    wbytes = sum(c.weight_bytes for c in cases)
    layer_shapes = [(c.N, c.K) for c in cases[:7]]
    sh = lambda: int(torch.cuda.current_stream().cuda_stream)  # noqa: E731

    def sweep_fn(M, A, outs):
        def fn():
            s = sh()
            for i, c in enumerate(cases):
                o = outs[i % 7]
                rc = qm.qm_matmul_q4_0_ptr(A[c.K].data_ptr(), weights[i].data_ptr(),
                                           o.data_ptr(), M, c.N, c.K, s)
                if rc != qm.QM_OK:
                    raise RuntimeError(f"sweep {c.name} M={M}: {qm.qm_status_string(rc)}")
        return fn

    def acts(M):
        return {K: torch.from_numpy(synth.activations(M, K, 5, key=(2, M, K))).to(dev)
                for K in (4096, 14336)}

    decode = {}
    for M in (1, 8):
        A = acts(M)
        outs = [torch.empty((M, N), dtype=torch.float32, device=dev) for (N, K) in layer_shapes]
        ms = graph_ms(torch, sweep_fn(M, A, outs))
        decode[f"m{M}"] = {"ms_per_pass": ms, "weight_gbs": wbytes / (ms * 1e-3) / 1e9,
                           "hbm_frac": wbytes / (ms * 1e-3) / 1e9 / hbm,
                           "launches_per_pass": len(cases)}
    decode["workload"] = ("32-layer decoder sweep (q,k,v,o,gate,up,down; hidden 4096, GQA), "
                          "3.93 GB of Q4_0 weights per pass, CUDA graph of 224 GEMV launches")

    # The same weights with q|k|v and gate|up stacked by rows (one row-major
    # block stream each, as an engine with fused projections stores them):
    # 4 GEMVs per layer, 128 launches per pass.
    fused, fused_shapes = [], []
    for layer in range(32):
        w = weights[7 * layer:7 * layer + 7]
        fused += [torch.cat([w[0], w[1], w[2]]), w[3], torch.cat([w[4], w[5]]), w[6]]
    fused_shapes = [(4096 + 1024 + 1024, 4096), (4096, 4096), (2 * 14336, 4096), (4096, 14336)]
    for M in (1, 8):
        A = acts(M)
        outs = [torch.empty((M, N), dtype=torch.float32, device=dev) for (N, K) in fused_shapes]

        def fused_fn(M=M, A=A, outs=outs):
            s = sh()
            for i, wf in enumerate(fused):
                N, K = fused_shapes[i % 4]
                rc = qm.qm_matmul_q4_0_ptr(A[K].data_ptr(), wf.data_ptr(), outs[i % 4].data_ptr(),
                                           M, N, K, s)
                if rc != qm.QM_OK:
                    raise RuntimeError(f"fused sweep M={M}: {qm.qm_status_string(rc)}")
        ms = graph_ms(torch, fused_fn)
        decode[f"m{M}_fused_layout"] = {"ms_per_pass": ms, "weight_gbs": wbytes / (ms * 1e-3) / 1e9,
                                        "hbm_frac": wbytes / (ms * 1e-3) / 1e9 / hbm,
                                        "launches_per_pass": len(fused)}
    del fused

    # Back-to-back M = 1 GEMVs at K = N = 4096 (16 weight replicas > L2).
    c0 = synth.workload(0)[0]
    w0 = [torch.from_numpy(c0.weights()).to(dev) for _ in range(16)]
    a0 = torch.from_numpy(c0.acts()).to(dev)
    o0 = torch.empty((1, c0.N), dtype=torch.float32, device=dev)

    def m1_fn():
        s = sh()
        for w in w0:
            rc = qm.qm_matmul_q4_0_ptr(a0.data_ptr(), w.data_ptr(), o0.data_ptr(), 1, c0.N, c0.K, s)
            if rc != qm.QM_OK:
                raise RuntimeError(f"m1 gemv: {qm.qm_status_string(rc)}")
    ms0 = graph_ms(torch, m1_fn) / len(w0)
    m1 = {"workload": "GEMV M=1, K=N=4096 (9.44 MB of weights), 16 replicas back to back "
                      "in a CUDA graph",
          "us_per_gemv": ms0 * 1e3, "weight_gbs": c0.weight_bytes / (ms0 * 1e-3) / 1e9,
          "hbm_frac": c0.weight_bytes / (ms0 * 1e-3) / 1e9 / hbm}
    del w0

    # Prefill: the same sweep at M = 512, eager launches.
    A = acts(512)
    outs = [torch.empty((512, N), dtype=torch.float32, device=dev) for (N, K) in layer_shapes]
    fn = sweep_fn(512, A, outs)
    fn()
    torch.cuda.synchronize()
    passes = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(passes):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / passes
    flops = sum(2.0 * 512 * c.N * c.K for c in cases)
    tflops = flops / (ms * 1e-3) / 1e12
    bf16 = peaks["bf16_tflops"]
    prefill = {
        "workload": "32-layer decoder sweep at M=512 (7.15 TFLOP per pass), eager launches",
        "kernel": "gemm_q4_0_tc (tcgen05, A split into bf16 hi+lo, W exact as two bf16 "
                  "pieces, 3 MMAs per product, f32 accumulation in TMEM)",
        "ms_per_pass": ms, "tflops": tflops,
        "roofline": {
            "bound": "tensor", "achieved": tflops, "peak": bf16 / 3.0, "unit": "TFLOP/s",
            "frac": tflops / (bf16 / 3.0),
            "peak_note": "measured bf16 dense peak / 3 MMAs per useful product",
            "mma_tflops_issued": 3.0 * tflops, "bf16_peak_tflops": bf16,
            "fp32_fma_peak_tflops_max_clock": fp32_peak_max,
            "vs_fp32_fma_peak_max_clock": tflops / fp32_peak_max,
            "fp32_fma_peak_tflops_live_clock": fp32_peak_live}}
    del weights
    torch.cuda.empty_cache()
    return {"decode": decode, "m1_gemv": m1, "prefill": prefill, "q8_0": q8_0_leg(qm, dev, peaks)}


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
    (``--profile-case gemm --M .. --N .. --K .. [--algo QM_ALGO_*]``, any M,
    or ``--profile-case q8_0``).
    Prints a one-line note, not a bench line."""
    import torch
    import bit_block_quantized_qm_gb300 as qm
    qm.load_library()
    dev = torch.device("cuda", 0)
    sh = int(torch.cuda.current_stream().cuda_stream)
    if args.profile_case == "gemm":
        M, N, K = args.M, args.N, args.K
        blob = synth.q4_0_weights(N, K, 1)
        A = synth.activations(M, K, 2)
        w = torch.from_numpy(blob).to(dev)
        a = torch.from_numpy(A).to(dev)
        c = torch.empty((M, N), dtype=torch.float32, device=dev)
        for _ in range(args.calls):
            rc = qm.qm_matmul_q4_0_algo_ptr(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K,
                                            args.algo, sh)
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
    p.add_argument("--profile-case", choices=("gemm", "q8_0"), default=None,
                   help="run one operation a few times and exit (profiler captures)")
    p.add_argument("--M", type=int, default=512)
    p.add_argument("--N", type=int, default=4096)
    p.add_argument("--K", type=int, default=4096)
    p.add_argument("--calls", type=int, default=3)
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
