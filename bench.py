#!/usr/bin/env python
"""Benchmark of the hot path: FP16 TN GEMM at M=N=K=4096 and the M=1 GEMV
(N=4096, K=14336), both through the C ABI of libtmagemm.so.

One step = one gemm_f16 launch (4096^3) + one gemv_f16 launch (4096 x 14336).
Inputs are resident in HBM before timing; each kernel rotates through enough
distinct input sets (> 2x L2) that every launch reads its operands from HBM.
Per-kernel times come from CUDA events on the launching stream.

Prints ONE JSON line (rank 0).  `value` is the GEMM's TFLOP/s over all ranks;
the GEMV's GB/s is in `gemv`.  `--impl reference` times the CPU oracle instead
(the only reference that exists for this path) on a bounded sample.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP16 GEMM TFLOP/s at 4096³ (% of dense peak); M=1 GEMV HBM GB/s"
GEMM_M = GEMM_N = GEMM_K = 4096
GEMV_N, GEMV_K = 4096, 14336
WORKLOAD = ("gemm_f16 TN D=A*B^T M=N=K=4096, A,B ~ U[-1,1] fp16, fp32 accumulate, fp16 out; "
            "+ gemv_f16 y=x*W^T N=4096 K=14336, x,W ~ N(0,0.02) fp16")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The sources each committed DRAM-traffic capture depends on (by key prefix).
KERNEL_SOURCES = {
    "gemm_tn_f16_kernel": ["tma_pipelined_tensor_tn_gb300/csrc/gemm_tn.cu",
                           "tma_pipelined_tensor_tn_gb300/csrc/ptx.cuh",
                           "tma_pipelined_tensor_tn_gb300/csrc/tile_sched.cuh"],
    "gemv_pieces_kernel": ["tma_pipelined_tensor_tn_gb300/csrc/gemv.cu",
                           "tma_pipelined_tensor_tn_gb300/csrc/ptx.cuh"],
}


def gemm_flops(M=GEMM_M, N=GEMM_N, K=GEMM_K):
    return 2.0 * M * N * K


def gemm_bytes(M=GEMM_M, N=GEMM_N, K=GEMM_K):
    return 2.0 * (M * K + N * K + M * N)


def gemv_bytes(N=GEMV_N, K=GEMV_K):
    """Algorithmic bytes: W (N*K) + x (K) + y (N) fp16 elements, each once."""
    return 2.0 * (N * K + K + N)


def max_over_ranks(values, device=None):
    """Element-wise max of `values` over all ranks of the default process group
    (the values unchanged when there is none).  Used for the timed region:
    the job takes as long as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_value(units_per_step, steps, world, total_seconds):
    """Throughput of the whole job: the units every rank processed over the
    slowest rank's time (replicas: each rank runs the full workload)."""
    return world * steps * units_per_step / total_seconds


def _code_only(text):
    """C/C++ source without comments and whitespace: a capture stays valid
    across comment edits, not across code changes."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_hash(kernel):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(key):
    """DRAM bytes per launch from a committed ncu summary, if the kernel sources
    have not changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(key)
    kernel = key.split("@")[0]
    if not e or kernel not in KERNEL_SOURCES or e.get("sources_hash") != sources_hash(kernel):
        return None
    return e.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    """Samples SM clock, power and clock-event reasons during the timed region.

    Reads NVML through ctypes (about every millisecond) and falls back to
    ``nvidia-smi -lms 100`` when NVML cannot be loaded.  Read-only.
    """
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []          # (t, sm_mhz, max_mhz, power_w, reasons_mask)
        self.stop_evt = threading.Event()
        self.thread = None
        self.source = None
        self.note = None
        self.window = None

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            u = getattr(torch.cuda.get_device_properties(self.dev), "uuid", None)
            if u is not None:
                uuid = ("GPU-" + str(u)).encode()
        except Exception:
            uuid = None
        if uuid is None or nv.nvmlDeviceGetHandleByUUID(uuid, ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.dev.index or 0), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        return nv, h

    def _run_nvml(self, nv, h):
        import ctypes
        clk, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self.stop_evt.is_set():
            t = time.perf_counter()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                p = pw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                r = rs.value if get_reasons(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((t, float(clk.value), float(mx.value), p, int(r)))
            time.sleep(0.001)

    def _run_smi(self):
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
        proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev.index or 0}", f"--query-gpu={fields}",
                                 "--format=csv,noheader,nounits", "-lms", "100"],
                                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        bits = (0x8, 0x40, 0x20, 0x4)
        try:
            for line in proc.stdout:
                if self.stop_evt.is_set():
                    break
                parts = [x.strip() for x in line.split(",")]
                try:
                    mask = sum(b for b, v in zip(bits, parts[3:7]) if v.lower().startswith("active"))
                    self.samples.append((time.perf_counter(), float(parts[0]), float(parts[1]),
                                         float(parts[2]), mask))
                except (ValueError, IndexError):
                    continue
        finally:
            proc.terminate()

    def start(self):
        try:
            nv, h = self._nvml_handle()
            self.source = "nvml"
            self.thread = threading.Thread(target=self._run_nvml, args=(nv, h), daemon=True)
        except OSError as e:
            self.note = f"nvml unavailable ({e}); nvidia-smi at 100 ms"
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._run_smi, daemon=True)
        self.thread.start()

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        time.sleep(0.05)
        self.stop_evt.set()
        if self.thread is not None:
            self.thread.join(timeout=5)
        t0, t1 = self.window or (float("-inf"), float("inf"))
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if len(inside) >= 3 else self.samples
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": self.note or "no samples"}
        mask = 0
        for s in used:
            mask |= s[4]
        out = {"sm_mhz": statistics.median(s[1] for s in used),
               "sm_max_mhz": max(s[2] for s in used),
               "sm_mhz_min": min(s[1] for s in used),
               "power_w_max": max((s[3] for s in used if s[3] is not None), default=None),
               "samples": len(used), "samples_in_timed_region": len(inside),
               "source": self.source,
               "reasons": sorted(n for b, n in self.REASONS.items() if mask & b)}
        if self.note:
            out["note"] = self.note
        return out


# ------------------------------------------------------------- CPU oracle ----

def oracle_gemm_sample(rows, A_np, B_np, threads=0):
    """Oracle on the first `rows` rows of the 4096^3 GEMM; returns (s, threads)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.gemm_f16(A_np[:rows], B_np, threads=threads)
    dt = time.perf_counter() - t0
    return dt, oracle.max_threads() if threads <= 0 else threads


def cpu_baseline(target_s=12.0):
    """Time the oracle, as it stands, on a bounded sample of the 4096^3 GEMM."""
    import oracle
    from tma_pipelined_tensor_tn_gb300 import inputs
    A, B = inputs.gemm_inputs(GEMM_M, GEMM_N, GEMM_K, seed=0)
    A_np, B_np = A.numpy(), B.numpy()
    dt, cores = oracle_gemm_sample(8, A_np, B_np)            # calibrate
    rows = int(max(8, min(GEMM_M, 8 * target_s / max(dt, 1e-3))))
    dt, cores = oracle_gemm_sample(rows, A_np, B_np)
    tflops = gemm_flops(rows, GEMM_N, GEMM_K) / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of 4096 rows of D for the 4096^3 GEMM "
                      f"({rows}x4096x4096 FP64 MACs, {dt:.1f} s)"}


def cpu_model():
    """The host CPU's model name, from /proc/cpuinfo or lscpu (empty if neither)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return ""


def oracle_per_config():
    """The oracle's wall time on each workload configuration: 256^3 and the
    GEMV in full on one core and on all cores, the ragged 4000x3000x4160 GEMM
    in full on all cores, and 8192^3 on its first 256 rows (scaled to the
    whole GEMM), with the core count and CPU model."""
    import oracle
    from tma_pipelined_tensor_tn_gb300 import inputs
    oracle.build()
    out = {"cores": oracle.max_threads(), "cpu_model": cpu_model()}

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    A, B = inputs.gemm_inputs(256, 256, 256, seed=0)
    a, b = A.numpy(), B.numpy()
    for th, key in ((1, "gemm_256_1core_s"), (0, "gemm_256_all_cores_s")):
        out[key] = timed(lambda: oracle.gemm_f16(a, b, threads=th))
    x, W = inputs.gemv_inputs(GEMV_N, GEMV_K, seed=0)
    xv, wv = x.numpy(), W.numpy()
    for th, key in ((1, "gemv_1core_s"), (0, "gemv_all_cores_s")):
        out[key] = timed(lambda: oracle.gemv_f16(xv, wv, threads=th))
    A, B = inputs.gemm_inputs(4000, 3000, 4160, seed=0)
    a, b = A.numpy(), B.numpy()
    out["gemm_ragged_all_cores_s"] = timed(lambda: oracle.gemm_f16(a, b))
    A, B = inputs.gemm_inputs(8192, 8192, 8192, seed=0)
    a, b = A.numpy()[:256], B.numpy()
    out["gemm_8192_all_cores_s_scaled"] = timed(lambda: oracle.gemm_f16(a, b)) * 8192 / 256
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample."""
    if rank != 0:
        return 0
    import oracle
    from tma_pipelined_tensor_tn_gb300 import inputs
    oracle.build()
    A, B = inputs.gemm_inputs(GEMM_M, GEMM_N, GEMM_K, seed=0)
    A_np, B_np = A.numpy(), B.numpy()
    x, W = inputs.gemv_inputs(GEMV_N, GEMV_K, seed=0)
    x_np, W_np = x.numpy(), W.numpy()
    # size a step at about 1.5 s of oracle work
    dt, cores = oracle_gemm_sample(8, A_np, B_np)
    rows = int(max(8, min(GEMM_M, 8 * 1.5 / max(dt, 1e-3))))
    for _ in range(args.warmup):
        oracle.gemm_f16(A_np[:rows], B_np)
    gemm_t = gemv_t = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.gemm_f16(A_np[:rows], B_np)
        t1 = time.perf_counter()
        oracle.gemv_f16(x_np, W_np)
        t2 = time.perf_counter()
        gemm_t += t1 - t0
        gemv_t += t2 - t1
    value = args.steps * gemm_flops(rows, GEMM_N, GEMM_K) / gemm_t / 1e12
    gemv_gbs = args.steps * gemv_bytes() / gemv_t / 1e9
    sample = (f"each step: rows 0..{rows - 1} of D for the 4096^3 GEMM ({rows}x4096x4096 FP64 MACs) "
              f"+ the full 4096x14336 GEMV")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * (gemm_t + gemv_t) / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "reference": "CPU oracle (FP64, plain loops)",
                   "sample_rows": rows},
        "gemv": {"value": gemv_gbs, "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- ours ----

def run_ours(args, rank, world, local_rank):
    import torch
    import tma_pipelined_tensor_tn_gb300 as tg
    from tma_pipelined_tensor_tn_gb300 import inputs

    tg.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 129 * 1024 * 1024
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # ---- resident inputs, rotated so that every launch misses L2 ----
    A, B = inputs.gemm_inputs(GEMM_M, GEMM_N, GEMM_K, seed=rank)
    x, W = inputs.gemv_inputs(GEMV_N, GEMV_K, seed=rank)
    r_gemm = inputs.l2_rotation_count(int(gemm_bytes()), l2)
    r_gemv = inputs.l2_rotation_count(int(gemv_bytes()), l2)
    dA, dB = A.to(dev), B.to(dev)
    gemm_sets = [(dA, dB, torch.empty((GEMM_M, GEMM_N), dtype=torch.float16, device=dev))]
    for _ in range(r_gemm - 1):
        gemm_sets.append((dA.clone(), dB.clone(),
                          torch.empty((GEMM_M, GEMM_N), dtype=torch.float16, device=dev)))
    dx, dW = x.to(dev), W.to(dev)
    gemv_sets = [(dx, dW, torch.empty((GEMV_N,), dtype=torch.float16, device=dev))]
    for _ in range(r_gemv - 1):
        gemv_sets.append((dx.clone(), dW.clone(), torch.empty((GEMV_N,), dtype=torch.float16, device=dev)))
    torch.cuda.synchronize(dev)

    def step(i):
        a, b, d = gemm_sets[i % r_gemm]
        s1 = tg.gemm_f16(GEMM_M, GEMM_N, GEMM_K, a.data_ptr(), b.data_ptr(), d.data_ptr(), sh)
        return s1

    def step_gemv(i):
        xv, wv, yv = gemv_sets[i % r_gemv]
        return tg.gemv_f16(GEMV_N, GEMV_K, xv.data_ptr(), wv.data_ptr(), yv.data_ptr(), sh)

    for i in range(args.warmup):
        assert step(i) == 0 and step_gemv(i) == 0
    tg.check(stream)

    # Timed region: K GEMM launches back to back, then K GEMV launches, each
    # batch between one pair of CUDA events on the launching stream (event
    # pairs around every single launch would add their own overhead to these
    # 20-100 us kernels).
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.05)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    launches = 0
    evs[0].record(stream)
    for i in range(args.steps):
        s1 = step(i)
        launches += 1
        if s1:
            raise RuntimeError(f"gemm launch failed: {tg.strerror(s1)}")
    evs[1].record(stream)
    for i in range(args.steps):
        s2 = step_gemv(i)
        launches += 1
        if s2:
            raise RuntimeError(f"gemv launch failed: {tg.strerror(s2)}")
    evs[2].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t1 = time.perf_counter()
    wall = t1 - t0
    clocks.mark(t0, t1)
    clk = clocks.stop()
    tg.check(stream)

    times = [evs[0].elapsed_time(evs[1]), evs[1].elapsed_time(evs[2]), wall]
    gemm_total_ms, gemv_total_ms, wall = max_over_ranks(times, device=dev)

    # ---- end to end through the C ABI: host buffers, copies inside the region ----
    # The library's host-buffer executor (tmagemm_host_pipeline_*): every step
    # copies its A and B from pinned host memory, runs gemm_f16 and copies D
    # back to pinned host memory; the three phases run on their own streams so
    # step i+1's inputs travel while step i computes.  Timed on the host clock
    # from the call to the return of synchronize (what a caller waits).
    # Up to 32 steps: the first step's upload and the last one's download do
    # not overlap anything, so short runs understate the steady state.
    from tma_pipelined_tensor_tn_gb300.pipeline import HostGemmPipeline
    e2e_steps = max(4, min(args.steps, 32))
    pipe = HostGemmPipeline(GEMM_M, GEMM_N, GEMM_K, torch.float16, depth=2, device=dev)
    hA = A.pin_memory()
    hB = B.pin_memory()
    hDs = [torch.empty((GEMM_M, GEMM_N), dtype=torch.float16).pin_memory() for _ in range(2)]
    pipe.run([hA] * 2, [hB] * 2, hDs)        # warm-up of the copy path
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    pipe.run([hA] * e2e_steps, [hB] * e2e_steps, [hDs[i % 2] for i in range(e2e_steps)])
    pipe.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3
    pipe.close()
    e2e_ms = max_over_ranks([e2e_ms], device=dev)[0]
    tg.check(stream)

    extras = measure_extras(tg, dev, stream, l2)
    extras.update(measure_distributions(tg, dev, stream, l2))
    extras["gemm_4096_plan"] = tg.tmagemm_gemm_plan(GEMM_M, GEMM_N, GEMM_K, 0)

    peaks, peak_src = load_peaks()
    gemm_avg_s = gemm_total_ms / 1e3 / args.steps
    gemv_avg_s = gemv_total_ms / 1e3 / args.steps
    value = whole_job_value(gemm_flops(), args.steps, world, gemm_total_ms / 1e3) / 1e12
    achieved = gemm_flops() / gemm_avg_s / 1e12
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    gemv_gbs = gemv_bytes() / gemv_avg_s / 1e9
    peak_h = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": (gemm_total_ms + gemv_total_ms) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemm": [GEMM_M, GEMM_N, GEMM_K],
                   "gemv": [GEMV_N, GEMV_K],
                   "l2": f"inputs larger than L2: {r_gemm} rotating GEMM sets and {r_gemv} "
                         f"rotating GEMV sets ({l2 // 2**20} MiB L2)",
                   "parallelism": f"replicas x{world}", "seed": "rank"},
        "gemm": {"value": achieved, "unit": "TFLOP/s", "us_per_launch": gemm_avg_s * 1e6,
                 "pct_of_dense_peak": 100.0 * achieved / peak_t},
        "gemv": {"value": gemv_gbs, "unit": "GB/s", "us_per_launch": gemv_avg_s * 1e6,
                 "pct_of_hbm_peak": 100.0 * gemv_gbs / peak_h},
        "roofline": {"bound": "tensor", "kernel": "gemm_tn_f16_kernel", "achieved": achieved,
                     "peak": peak_t, "unit": "TFLOP/s", "frac": achieved / peak_t,
                     "traffic": load_traffic("gemm_tn_f16_kernel@gemm_4096"),
                     "peak_source": f"{peak_src} bf16_tflops (burst; fp16 dense = bf16 dense)",
                     "flops_per_launch": gemm_flops()},
        "roofline_gemv": {"bound": "hbm", "kernel": "gemv_pieces_kernel", "achieved": gemv_gbs,
                          "peak": peak_h, "unit": "GB/s", "frac": gemv_gbs / peak_h,
                          "traffic": load_traffic("gemv_pieces_kernel@gemv_4096x14336"),
                          "peak_source": f"{peak_src} hbm_gbs",
                          "bytes_per_launch": gemv_bytes()},
        "e2e": {"value": e2e_steps * gemm_flops() / (e2e_ms / 1e3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": pipe.h2d_bytes_per_step(),
                "d2h_bytes_per_step": pipe.d2h_bytes_per_step(),
                "steps": e2e_steps,
                "what": "tmagemm_host_pipeline (C ABI): per step pinned host A,B -> device, "
                        "gemm_f16, D -> pinned host; copies and GEMMs of neighbouring steps "
                        "overlap on three streams (2 device slots); host clock"},
        "gpu_launches": launches,
        "extras": extras,
        "wall_s_timed_region": wall,
        "clocks": clk,
        "device": props.name,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
        line["cpu_baseline"]["per_config"] = oracle_per_config()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def _time_launches(fn, reps, stream):
    """Average device time of `fn` over `reps` back-to-back launches (events on `stream`)."""
    import torch
    for _ in range(3):
        fn(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


# Spin cycles queued ahead of a per-launch distribution: about 10 ms at GB300
# clocks, longer than the host needs to enqueue 100 launches and their events.
HOLD_CYCLES = 20_000_000


def _launch_distribution(fn, reps, stream):
    """Per-launch device times of `fn` (an event pair around every launch,
    which also keeps consecutive launches from overlapping): min, median and
    90th percentile in microseconds.  A spin kernel queued first holds the
    stream until every launch and event is enqueued, so the time the host
    takes to issue a launch (Python, ctypes, tensor-map encoding) never falls
    between an event and its kernel."""
    import torch
    for _ in range(3):
        fn(0)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HOLD_CYCLES)
    for i, (e0, e1) in enumerate(evs):
        e0.record(stream)
        fn(i)
        e1.record(stream)
    torch.cuda.synchronize()
    t = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)
    return {"min_us": t[0], "median_us": statistics.median(t),
            "p90_us": t[min(len(t) - 1, int(0.9 * len(t)))], "launches": reps}


def measure_distributions(tg, dev, stream, l2):
    """Per-launch statistics of the two headline kernels over 100 launches
    each: the 4096^3 GEMM and the GEMV on inputs rotated past L2 (cold), and
    the GEMV once more on one weight set that stays in L2 between launches
    (warm, labelled as such)."""
    import torch
    from tma_pipelined_tensor_tn_gb300 import inputs
    sh = stream.cuda_stream
    out = {}
    A, B = inputs.gemm_inputs(GEMM_M, GEMM_N, GEMM_K, seed=0)
    n_g = inputs.l2_rotation_count(2 * (GEMM_M * GEMM_K + GEMM_N * GEMM_K), l2)
    gsets = [(A.to(dev), B.to(dev))]
    gsets += [(gsets[0][0].clone(), gsets[0][1].clone()) for _ in range(n_g - 1)]
    D = torch.empty((GEMM_M, GEMM_N), dtype=torch.float16, device=dev)

    def gemm(i):
        a, b = gsets[i % n_g]
        assert tg.gemm_f16(GEMM_M, GEMM_N, GEMM_K, a.data_ptr(), b.data_ptr(), D.data_ptr(), sh) == 0

    dist = _launch_distribution(gemm, 100, stream)
    dist["tflops_at_median"] = gemm_flops() / dist["median_us"] / 1e6
    out["gemm_4096_per_launch"] = dist
    del gsets
    x, W = inputs.gemv_inputs(GEMV_N, GEMV_K, seed=0)
    n_v = inputs.l2_rotation_count(gemv_bytes(), l2)
    vsets = [(x.to(dev), W.to(dev))]
    vsets += [(vsets[0][0].clone(), vsets[0][1].clone()) for _ in range(n_v - 1)]
    y = torch.empty((GEMV_N,), dtype=torch.float16, device=dev)

    def gemv(i, sets=vsets):
        xv, wv = sets[i % len(sets)]
        assert tg.gemv_f16(GEMV_N, GEMV_K, xv.data_ptr(), wv.data_ptr(), y.data_ptr(), sh) == 0

    dist = _launch_distribution(gemv, 100, stream)
    dist["gbs_at_median"] = gemv_bytes() / dist["median_us"] / 1e3
    out["gemv_4096x14336_per_launch_cold"] = dist
    # The same without programmatic dependent launch: each launch waits for
    # the end of the event before it, with no early scheduling at all.
    assert tg.tmagemm_set_pdl(0) == 0
    try:
        dist = _launch_distribution(gemv, 100, stream)
    finally:
        tg.tmagemm_set_pdl(1)
    dist["gbs_at_median"] = gemv_bytes() / dist["median_us"] / 1e3
    dist["note"] = "plain launches (no programmatic dependent launch)"
    out["gemv_4096x14336_per_launch_cold_plain"] = dist
    dist = _launch_distribution(lambda i: gemv(i, vsets[:1]), 100, stream)
    dist["gbs_at_median"] = gemv_bytes() / dist["median_us"] / 1e3
    dist["note"] = "warm L2: the same 117 MB weight set every launch"
    out["gemv_4096x14336_per_launch_warm_l2"] = dist
    tg.check(stream)
    return out


def measure_extras(tg, dev, stream, l2):
    """Rows beyond the headline path, each against the plain kernel on the same
    shape: split-K GEMM on a shape with few output tiles and a long K."""
    import torch
    from tma_pipelined_tensor_tn_gb300 import inputs
    sh = stream.cuda_stream
    out = {}
    M, N, K = 1024, 1024, 16384
    A, B = inputs.gemm_inputs(M, N, K, seed=7)
    sets = inputs.l2_rotation_count(2 * (M * K + N * K), l2)
    ops = [(A.to(dev), B.to(dev)) if i == 0 else None for i in range(sets)]
    for i in range(1, sets):
        ops[i] = (ops[0][0].clone(), ops[0][1].clone())
    D = torch.empty((M, N), dtype=torch.float16, device=dev)
    need = tg.gemm_f16_splitk_workspace_size(M, N, K, 0)
    ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    plan = tg.tmagemm_gemm_plan(M, N, K, torch.cuda.get_device_properties(dev).multi_processor_count, 0)

    def plain(i):
        a, b = ops[i % sets]
        assert tg.gemm_f16(M, N, K, a.data_ptr(), b.data_ptr(), D.data_ptr(), sh) == 0

    def split(i):
        a, b = ops[i % sets]
        assert tg.gemm_f16_splitk(M, N, K, a.data_ptr(), b.data_ptr(), D.data_ptr(), 0,
                                  ws.data_ptr(), need, sh) == 0

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    auto_plan = tg.tmagemm_gemm_plan(M, N, K, sms, 1, sms // 2)
    t_auto = _time_launches(plain, 50, stream)          # gemm_f16: cluster split-K
    t_split = _time_launches(split, 50, stream)         # gemm_f16_splitk: FP32 workspace
    assert tg.tmagemm_set_cluster_split(1) == 0
    try:
        t_plain = _time_launches(plain, 50, stream)     # gemm_f16 on the tile kernel alone
    finally:
        tg.tmagemm_set_cluster_split(0)
    tg.check(stream)
    fl = gemm_flops(M, N, K)
    out["splitk_1024x1024x16384"] = {
        "gemm_f16_us": t_auto, "gemm_f16_tflops": fl / t_auto / 1e6,
        "gemm_f16_cluster_split": auto_plan["cluster_k"],
        "splitk_workspace_us": t_split, "splitk_workspace_tflops": fl / t_split / 1e6,
        "splitk_workspace_parts": plan["splits"], "workspace_bytes": need,
        "tile_kernel_only_us": t_plain, "tile_kernel_only_tflops": fl / t_plain / 1e6,
        "note": "gemm_f16 splits K over clusters and reduces in distributed shared memory; "
                "gemm_f16_splitk writes FP32 partials and reduces in a second kernel"}

    # bf16 forms of the two headline kernels, same shapes and rotation rules.
    Mh = Nh = Kh = 4096
    Ab, Bb = inputs.gemm_inputs(Mh, Nh, Kh, seed=8)
    Ab, Bb = Ab.to(torch.bfloat16), Bb.to(torch.bfloat16)
    rs = inputs.l2_rotation_count(int(gemm_bytes()), l2)
    bsets = [(Ab.to(dev), Bb.to(dev))]
    for _ in range(rs - 1):
        bsets.append((bsets[0][0].clone(), bsets[0][1].clone()))
    Dh = torch.empty((Mh, Nh), dtype=torch.bfloat16, device=dev)

    def gemm_b(i):
        a, b = bsets[i % rs]
        assert tg.gemm_bf16(Mh, Nh, Kh, a.data_ptr(), b.data_ptr(), Dh.data_ptr(), sh) == 0

    t_gb = _time_launches(gemm_b, 100, stream)
    xg, Wg = inputs.gemv_inputs(GEMV_N, GEMV_K, seed=9)
    rv = inputs.l2_rotation_count(int(gemv_bytes()), l2)
    vsets = [(xg.to(torch.bfloat16).to(dev), Wg.to(torch.bfloat16).to(dev))]
    for _ in range(rv - 1):
        vsets.append((vsets[0][0].clone(), vsets[0][1].clone()))
    yb = torch.empty((GEMV_N,), dtype=torch.bfloat16, device=dev)

    def gemv_b(i):
        xv, wv = vsets[i % rv]
        assert tg.gemv_bf16(GEMV_N, GEMV_K, xv.data_ptr(), wv.data_ptr(), yb.data_ptr(), sh) == 0

    t_vb = _time_launches(gemv_b, 100, stream)
    tg.check(stream)
    out["bf16_gemm_4096"] = {"us": t_gb, "tflops": gemm_flops() / t_gb / 1e6}
    out["bf16_gemv_4096x14336"] = {"us": t_vb, "gbs": gemv_bytes() / t_vb / 1e3}

    # Skinny decode GEMMs at the GEMV's weight shape: M tokens x (4096 x 14336).
    for Ms in (8, 16, 32, 64):
        Xs = (torch.randn((Ms, GEMV_K), generator=torch.Generator().manual_seed(Ms)) * 0.02).half()
        xsets = [Xs.to(dev)] * rv
        Ds = torch.empty((Ms, GEMV_N), dtype=torch.float16, device=dev)
        wsets = [(vsets[i][1].view(torch.float16)) for i in range(rv)]
        need_s = tg.gemm_f16_small_m_workspace_size(Ms, GEMV_N, GEMV_K)
        ws_s = torch.empty((max(need_s, 16),), dtype=torch.uint8, device=dev)

        def small(i, Ms=Ms, Ds=Ds, ws_s=ws_s, need_s=need_s):
            assert tg.gemm_f16_small_m(Ms, GEMV_N, GEMV_K, xsets[i % rv].data_ptr(),
                                       wsets[i % rv].data_ptr(), Ds.data_ptr(), ws_s.data_ptr(),
                                       need_s, sh) == 0

        t_s = _time_launches(small, 100, stream)
        tg.check(stream)
        Dc = torch.empty_like(Ds)

        def small_cublas(i, Dc=Dc):   # context only: cuBLAS on the same inputs
            torch.matmul(xsets[i % rv], wsets[i % rv].T, out=Dc)

        t_c = _time_launches(small_cublas, 100, stream)
        by = 2.0 * (GEMV_N * GEMV_K + Ms * GEMV_K + Ms * GEMV_N)
        out[f"small_m{Ms}_4096x14336"] = {"us": t_s, "gbs": by / t_s / 1e3,
                                          "tflops": 2.0 * Ms * GEMV_N * GEMV_K / t_s / 1e6,
                                          "kernel": ("mma.sync register fragments" if Ms <= 16
                                                     else "tcgen05 tile kernel, cluster split-K"),
                                          "cublas_us": t_c}

    # Grouped GEMM: 8 experts, 8192 routed tokens (skewed counts), N=4096, K=2048,
    # against one dense GEMM over the same 8192 rows.
    G, T, Ng, Kg = 8, 8192, 4096, 2048
    rng = torch.Generator().manual_seed(11)
    counts = GROUPED_COUNTS
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    Ag = (torch.rand((T, Kg), generator=rng) * 2 - 1).half().to(dev)
    Bg = (torch.rand((G, Ng, Kg), generator=rng) * 2 - 1).half().to(dev)
    Dg = torch.empty((T, Ng), dtype=torch.float16, device=dev)

    def grouped(i):
        assert tg.gemm_f16_grouped(G, offs, Ng, Kg, Ag.data_ptr(), Bg.data_ptr(), Dg.data_ptr(),
                                   sh) == 0

    def dense(i):
        assert tg.gemm_f16(T, Ng, Kg, Ag.data_ptr(), Bg.data_ptr(), Dg.data_ptr(), sh) == 0

    t_g = _time_launches(grouped, 50, stream)
    t_d = _time_launches(dense, 50, stream)
    tg.check(stream)
    fl = 2.0 * T * Ng * Kg
    # The parity workloads beyond the headline, for their TFLOP/s: 256^3
    # (launch-bound: direct calls and 100 calls replayed from one CUDA graph),
    # the ragged 4000x3000x4160 shape, and 8192^3 (5 launches).
    for name, (Mw, Nw, Kw, reps) in {"gemm_ragged_4000x3000x4160": (4000, 3000, 4160, 50),
                                     "gemm_8192": (8192, 8192, 8192, 5),
                                     "gemm_256": (256, 256, 256, 200)}.items():
        Aw, Bw = inputs.gemm_inputs(Mw, Nw, Kw, seed=12)
        aw, bw = Aw.to(dev), Bw.to(dev)
        dw = torch.empty((Mw, Nw), dtype=torch.float16, device=dev)
        fn = (lambda i, aw=aw, bw=bw, dw=dw, Mw=Mw, Nw=Nw, Kw=Kw:
              tg.gemm_f16(Mw, Nw, Kw, aw.data_ptr(), bw.data_ptr(), dw.data_ptr(), sh))
        t_w = _time_launches(lambda i: fn(i) == 0 or None, reps, stream)
        entry = {"us": t_w, "tflops": gemm_flops(Mw, Nw, Kw) / t_w / 1e6}
        pw = tg.tmagemm_gemm_plan(Mw, Nw, Kw, 0)
        entry["plan"] = {"BN": pw["BN"], "pair": pw["pair"], "tiles": pw["tiles"],
                         "units": pw["units"], "cluster_k": pw["cluster_k"],
                         **tg.tmagemm_gemm_tail_plan(Mw, Nw, Kw, 0)}
        if name == "gemm_256":
            gs = torch.cuda.Stream(dev)
            gs.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(100):
                    tg.gemm_f16(Mw, Nw, Kw, aw.data_ptr(), bw.data_ptr(), dw.data_ptr(),
                                gs.cuda_stream)
            graph.replay()
            torch.cuda.synchronize(dev)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(5):
                graph.replay()
            g1.record(stream)
            torch.cuda.synchronize(dev)
            t_graph = g0.elapsed_time(g1) * 1e3 / 500
            entry.update({"us_in_graph": t_graph,
                          "tflops_in_graph": gemm_flops(Mw, Nw, Kw) / t_graph / 1e6})
        tg.check(stream)
        out[name] = entry

    # Context, not a target: torch.matmul (cuBLAS) on the same shapes and
    # rotating fp16 inputs, so the GEMM can be compared on this machine.
    for name, (Mc, Nc, Kc, reps) in {"cublas_fp16_4096": (4096, 4096, 4096, 50),
                                     "cublas_fp16_8192": (8192, 8192, 8192, 5)}.items():
        csets = [inputs.gemm_inputs(Mc, Nc, Kc, seed=20 + j) for j in range(3 if Mc < 8192 else 1)]
        csets = [(a.to(dev), b.to(dev)) for a, b in csets]
        dc = torch.empty((Mc, Nc), dtype=torch.float16, device=dev)

        def cublas(i, csets=csets, dc=dc):
            a, b = csets[i % len(csets)]
            torch.matmul(a, b.T, out=dc)

        t_c = _time_launches(cublas, reps, stream)
        out[name] = {"us": t_c, "tflops": gemm_flops(Mc, Nc, Kc) / t_c / 1e6,
                     "what": "torch.matmul(A, B.T, out=D), cuBLAS, for comparison only"}
        del csets

    out["grouped_8x(8192_tokens)x4096x2048"] = {
        "us": t_g, "tflops": fl / t_g / 1e6, "dense_same_rows_us": t_d,
        "dense_tflops": fl / t_d / 1e6, "group_rows": [int(c) for c in counts]}
    return out


# Rows routed to each of 8 experts out of 8192 tokens: a fixed skewed split
# (one draw of a Dirichlet(0.7) routing, stored so every run times the same shapes).
GROUPED_COUNTS = [1697, 2233, 321, 376, 105, 1822, 706, 932]

CASES = ("gemm4096", "gemv", "splitk", "small_m8", "small_m16", "small_m32", "small_m64", "grouped",
         "bf16_gemm", "bf16_gemv",
         "gemm8192", "gemm_ragged", "gemm256", "decode128_8192")


def run_case(args, name):
    """One workload alone (for profilers): `warmup` launches, then `steps`
    launches between one pair of CUDA events; prints a short JSON line."""
    import torch
    import tma_pipelined_tensor_tn_gb300 as tg
    from tma_pipelined_tensor_tn_gb300 import inputs
    tg.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    if name in ("gemm4096", "bf16_gemm", "gemm8192", "splitk", "gemm_ragged", "gemm256",
                "decode128_8192"):
        M, N, K = {"gemm4096": (4096,) * 3, "bf16_gemm": (4096,) * 3, "gemm8192": (8192,) * 3,
                   "splitk": (1024, 1024, 16384), "gemm_ragged": (4000, 3000, 4160),
                   "gemm256": (256,) * 3, "decode128_8192": (128, 8192, 8192)}[name]
        A, B = inputs.gemm_inputs(M, N, K, seed=0)
        if name == "bf16_gemm":
            A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
        a, b = A.to(dev), B.to(dev)
        d = torch.empty((M, N), dtype=a.dtype, device=dev)
        need = tg.gemm_f16_splitk_workspace_size(M, N, K, 0) if name == "splitk" else 0
        ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
        fl = 2.0 * M * N * K
        if name == "splitk":
            fn = lambda: tg.gemm_f16_splitk(M, N, K, a.data_ptr(), b.data_ptr(), d.data_ptr(), 0,
                                            ws.data_ptr(), need, sh)
        elif name == "bf16_gemm":
            fn = lambda: tg.gemm_bf16(M, N, K, a.data_ptr(), b.data_ptr(), d.data_ptr(), sh)
        else:
            fn = lambda: tg.gemm_f16(M, N, K, a.data_ptr(), b.data_ptr(), d.data_ptr(), sh)
        unit = ("TFLOP/s", fl / 1e12)
    elif name in ("gemv", "bf16_gemv", "small_m8", "small_m16", "small_m32", "small_m64"):
        # Weight sets rotated past L2: consecutive launches read HBM.
        x, W = inputs.gemv_inputs(GEMV_N, GEMV_K, seed=0)
        if name == "bf16_gemv":
            x, W = x.to(torch.bfloat16), W.to(torch.bfloat16)
        l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 << 20)
        nw = inputs.l2_rotation_count(int(gemv_bytes()), l2)
        ws_rot = [W.to(dev)]
        ws_rot += [ws_rot[0].clone() for _ in range(nw - 1)]
        turn = [0]

        def w_next():
            turn[0] += 1
            return ws_rot[turn[0] % nw].data_ptr()

        if name.startswith("small_m"):
            Ms = int(name[7:])
            X = (torch.randn((Ms, GEMV_K), generator=torch.Generator().manual_seed(1)) * 0.02).half()
            xv = X.to(dev)
            y = torch.empty((Ms, GEMV_N), dtype=torch.float16, device=dev)
            need = tg.gemm_f16_small_m_workspace_size(Ms, GEMV_N, GEMV_K)
            ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
            fn = lambda: tg.gemm_f16_small_m(Ms, GEMV_N, GEMV_K, xv.data_ptr(), w_next(),
                                             y.data_ptr(), ws.data_ptr(), need, sh)
            by = 2.0 * (GEMV_N * GEMV_K + Ms * GEMV_K + Ms * GEMV_N)
        else:
            xv = x.to(dev)
            y = torch.empty((GEMV_N,), dtype=x.dtype, device=dev)
            g = tg.gemv_bf16 if name == "bf16_gemv" else tg.gemv_f16
            fn = lambda: g(GEMV_N, GEMV_K, xv.data_ptr(), w_next(), y.data_ptr(), sh)
            by = gemv_bytes()
        unit = ("GB/s", by / 1e9)
    elif name == "grouped":
        G, T, Ng, Kg = 8, 8192, 4096, 2048
        counts = GROUPED_COUNTS
        offs = [0]
        for c in counts:
            offs.append(offs[-1] + c)
        rng = torch.Generator().manual_seed(11)
        a = (torch.rand((T, Kg), generator=rng) * 2 - 1).half().to(dev)
        b = (torch.rand((G, Ng, Kg), generator=rng) * 2 - 1).half().to(dev)
        d = torch.empty((T, Ng), dtype=torch.float16, device=dev)
        fn = lambda: tg.gemm_f16_grouped(G, offs, Ng, Kg, a.data_ptr(), b.data_ptr(), d.data_ptr(), sh)
        unit = ("TFLOP/s", 2.0 * T * Ng * Kg / 1e12)
    else:
        raise SystemExit(f"unknown case {name}")
    for _ in range(args.warmup):
        assert fn() == 0
    tg.check(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        assert fn() == 0
    e1.record(stream)
    torch.cuda.synchronize(dev)
    tg.check(stream)
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    print(json.dumps({"case": name, "us_per_launch": us, "value": unit[1] / (us * 1e-6),
                      "unit": unit[0], "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="time one workload alone (for profiling); prints a short line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.case:
        return run_case(args, args.case)
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
