#!/usr/bin/env python3
"""Benchmark: fused NF4-QLoRA linear layer, forward + backward, on B300.

One step = one forward (qlora_linear_fwd) and one backward (qlora_linear_bwd)
of the projection workload over one batch of synthetic tokens, inputs already
resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
                  [--no-extra] [--no-cpu-baseline]

The default workload is the largest single-GPU one: 16384 tokens through a
4096 -> 14336 projection at rank 64 (the top of the token sweep).  Besides the
headline line the same run measures the other projection workloads (key
"extra") with shorter timed regions.

N > 1 is launched by torchrun: each rank runs its own independent replica of
the workload on its own GPU (no collective on the data path; "scaling": "weak").
`--impl reference` times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused QLoRA linear fwd+bwd TFLOP/s & tokens/s; % of BF16 TC / HBM roofline"
DEFAULT_CONFIG = "sweep_m16384"
# Workloads measured beside the headline one (shorter timed regions each).
EXTRA_CONFIGS = ("llama3_8b_q_proj", "llama3_8b_mlp_up", "llama3_8b_mlp_down", "qwen14b_attn", "qwen14b_mlp",
                 "sweep_m1", "sweep_m16", "sweep_m128", "sweep_m1024")
# A timed region shorter than this runs at burst clocks: its roofline takes the
# burst bf16 peak; longer regions take the sustained (power-capped) one.
BURST_REGION_S = 1.0


def shape_of(name):
    from rank_adapter_linear_nf4_b300 import synthetic
    return synthetic.SHAPES[name]


def fwd_only(sh) -> bool:
    """Small-token workloads (M < 128) are forward passes: weight-streaming, HBM-bound."""
    return sh.M < 128


def step_flops(sh) -> float:
    """Algorithmic flops of one step: forward + backward (no dW: the base is
    frozen), or the forward alone for the small-token workloads."""
    M, K, N, r = sh.M, sh.d_in, sh.d_out, sh.r
    fwd = 2 * M * K * N + 2 * M * r * (K + N)
    bwd = 2 * M * K * N + 4 * M * r * (K + N)
    return float(fwd if fwd_only(sh) else fwd + bwd)


def step_bytes(sh) -> float:
    """Algorithmic HBM bytes of one step: the NF4 weight (codes + fp32 absmax)
    once per pass, the bf16 activations read and written, the low-rank factors
    and the small fp32 outputs."""
    M, K, N, r = sh.M, sh.d_in, sh.d_out, sh.r
    w = 0.5625 * K * N
    fwd = w + 2.0 * M * K + 2.0 * M * N + 2.0 * r * (K + N) + 4.0 * M * r
    if fwd_only(sh):
        return fwd
    bwd = w + 2.0 * M * N * 2 + 2.0 * M * K * 2 + 2.0 * r * (K + N) + 4.0 * M * r + 4.0 * r * (K + N)
    return fwd + bwd


# The source files each measured kernel is built from (a stored traffic figure
# counts only while they are unchanged).
KERNEL_SOURCES = {
    "lora_main_fwd": ("lora_kernels.cu", "nf4_lut.cuh", "ptx.cuh", "kernels.h"),
    "lora_main_dX": ("lora_kernels.cu", "nf4_lut.cuh", "ptx.cuh", "kernels.h"),
    "lora_stream_fwd": ("lora_stream.cu", "nf4_lut.cuh", "ptx.cuh", "kernels.h"),
}


def sources_hash(kernel: str) -> str:
    """Hash of the CUDA sources `kernel` is built from."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "rank_adapter_linear_nf4_b300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or tuple(sorted(os.listdir(csrc)))
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/traffic.json, if captured from these sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(f"{kernel}@{workload}")
    if not e or e.get("sources") != sources_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def kernel_work(sh, kind):
    """Algorithmic (flops, bytes) of one launch of a kernel of the layer."""
    M, K, N, r = sh.M, sh.d_in, sh.d_out, sh.r
    w_bytes = 0.5625 * K * N
    if kind == "lora_main_fwd":
        return 2.0 * M * K * N + 2.0 * M * r * N, w_bytes + 2.0 * M * K + 2.0 * M * N + 2.0 * M * r + 2.0 * r * N
    if kind == "lora_main_dX":
        return 2.0 * M * K * N + 2.0 * M * r * K, w_bytes + 2.0 * M * N + 2.0 * M * K + 2.0 * M * r + 2.0 * r * K
    if kind == "lora_stream_fwd":
        return (2.0 * M * K * N + 2.0 * M * r * N,
                w_bytes + 2.0 * M * K + 2.0 * M * N + 2.0 * r * N + 2.0 * M * r)
    if kind == "lora_rows_T":
        return 2.0 * M * K * r, 2.0 * M * K + 2.0 * K * r + 6.0 * M * r
    if kind == "lora_rows_G":
        return 2.0 * M * N * r, 2.0 * M * N + 2.0 * N * r + 8.0 * M * r
    if kind == "lora_red_dA_dB":
        return 2.0 * M * r * (K + N), 2.0 * M * (K + N) + 4.0 * M * r + 4.0 * r * (K + N)
    return 0.0, 0.0


def workload_desc(sh) -> str:
    kind = "rank-stabilised " if sh.rank_stabilised else ""
    return (f"{sh.name}: M={sh.M} tokens, d_in={sh.d_in} -> d_out={sh.d_out}, r={sh.r}, "
            f"{kind}s={sh.s:g}, NF4 blocksize 64, {'fwd' if fwd_only(sh) else 'fwd+bwd'}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sust": p["bf16_tflops_sustained"],
                "src": "measured"}
    return {"hbm": 6400.0, "bf16": 1800.0, "bf16_sust": 1400.0, "src": "fallback"}


def power_capped(clocks) -> bool:
    """The clock record of a region shows the power cap holding the SM clock down."""
    if not clocks or not clocks.get("samples"):
        return False
    med, top = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    return bool(med and top and med < 0.95 * top and capped)


def tensor_peak(peaks, region_s, clocks=None):
    """The bf16 peak a region is judged against, and its name: the burst figure
    for a short region at full clock, the sustained one (measured under the
    power cap) for a region of a second or more or one whose clock record shows
    the power cap holding the clock down."""
    if region_s < BURST_REGION_S and not power_capped(clocks):
        return peaks["bf16"], f"bf16 dense burst ({peaks['src']}; timed region {region_s * 1e3:.0f} ms < 1 s)"
    why = (f"timed region {region_s:.1f} s" if region_s >= BURST_REGION_S else
           f"timed region {region_s * 1e3:.0f} ms at a median SM clock of {clocks.get('sm_mhz')} MHz under sw_power_cap")
    return peaks["bf16_sust"], f"bf16 dense sustained ({peaks['src']}; {why})"


# ---------------------------------------------------------------- clocks (NVML)

class _Nvml:
    """The few read-only NVML queries the sampler needs, through pynvml when it
    is importable, else straight from the driver's libnvidia-ml with ctypes."""

    CLOCK_SM = 1

    def __init__(self, torch_dev: int):
        import torch
        uuid = str(torch.cuda.get_device_properties(torch_dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        try:
            import pynvml
            pynvml.nvmlInit()
            self.py = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            self.source = "pynvml"
            return
        except Exception:
            self.py = None
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self.source = "libnvidia-ml (ctypes)"
        fn = None
        for name in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
            if hasattr(lib, name):
                fn = getattr(lib, name)
                break
        self._reasons_fn = fn

    def sm_mhz(self) -> int:
        if self.py:
            return int(self.py.nvmlDeviceGetClockInfo(self.h, self.py.NVML_CLOCK_SM))
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo")
        return int(v.value)

    def max_sm_mhz(self) -> int:
        if self.py:
            return int(self.py.nvmlDeviceGetMaxClockInfo(self.h, self.py.NVML_CLOCK_SM))
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo")
        return int(v.value)

    def power_w(self) -> float:
        if self.py:
            return self.py.nvmlDeviceGetPowerUsage(self.h) / 1000.0
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetPowerUsage")
        return v.value / 1000.0

    def reasons(self) -> int:
        if self.py:
            for fn in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
                if hasattr(self.py, fn):
                    return int(getattr(self.py, fn)(self.h))
            return 0
        if self._reasons_fn is None:
            return 0
        v = ctypes.c_ulonglong()
        if self._reasons_fn(self.h, ctypes.byref(v)) != 0:
            return 0
        return int(v.value)


class ClockSampler:
    """Samples the SM clock, power and clock-event reasons every ~2 ms in a
    thread from before the warm-up to the end of the run; each timed region
    keeps the samples taken inside it (host time stamps)."""

    REASONS = [("gpu_idle", 0x1), ("applications_clocks", 0x2), ("sw_power_cap", 0x4),
               ("hw_slowdown", 0x8), ("sync_boost", 0x10), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake", 0x80)]

    def __init__(self, torch_dev: int, period_s: float = 0.002):
        self.samples = []
        self.err = ""
        self.period = period_s
        self.nv = None
        try:
            self.nv = _Nvml(torch_dev)
            self.max_mhz = self.nv.max_sm_mhz()
        except Exception as e:
            self.err = f"NVML unavailable: {e!r}"[:200]
            self.max_mhz = None

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append((time.perf_counter(), self.nv.sm_mhz(), self.nv.power_w(), self.nv.reasons()))
            except Exception:
                pass
            time.sleep(self.period)

    def start(self):
        if self.nv is None:
            return
        self._stop = threading.Event()
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        if self.nv is not None:
            self._stop.set()
            self._t.join()

    def summary(self, t0: float, t1: float):
        """Clocks seen in the host-time window [t0, t1]."""
        if self.nv is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": self.err}
        s = [x for x in self.samples if t0 <= x[0] <= t1]
        mask = 0
        for x in s:
            mask |= x[3]
        reasons = [n for n, b in self.REASONS if mask & b and n != "gpu_idle"]
        out = {"sm_mhz": statistics.median([x[1] for x in s]) if s else None,
               "sm_min_mhz": min(x[1] for x in s) if s else None,
               "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(s),
               "power_w_median": statistics.median([x[2] for x in s]) if s else None,
               "window_ms": (t1 - t0) * 1e3, "period_ms": self.period * 1e3, "source": self.nv.source}
        return out


# ---------------------------------------------------------------- oracle timing (CPU)

class OracleRunner:
    """The oracle on the first `tokens` tokens of the workload: one step is
    NF4 dequantisation of the full weight + forward + backward (fp64)."""

    # quantised weights by (d_in, d_out, r): workloads of one weight shape share one
    _weights = {}

    def __init__(self, sh, tokens: int):
        from oracle import qlora_oracle as O
        from rank_adapter_linear_nf4_b300 import synthetic
        self.O, self.sh = O, sh
        X, dY = synthetic.activations(tokens, sh.d_in, sh.d_out, seed=0)
        f = lambda t: t.float().numpy()
        self.X, self.dY = f(X), f(dY)
        key = (sh.d_in, sh.d_out, sh.r)
        if key not in OracleRunner._weights:
            W, A, B = synthetic.weights(sh.d_in, sh.d_out, sh.r, seed=1)
            OracleRunner._weights[key] = (f(A), f(B)) + tuple(O.quantize_nf4(f(W)))
        self.A, self.B, self.packed, self.absmax = OracleRunner._weights[key]
        self.fwd_only = fwd_only(sh)

    @staticmethod
    def blas_threads() -> int:
        try:
            from threadpoolctl import threadpool_info
            return max([int(i.get("num_threads", 1)) for i in threadpool_info()] or [1])
        except Exception:
            return os.cpu_count() or 1

    def step(self):
        O, sh = self.O, self.sh
        Wd = O.dequantize_nf4(self.packed, self.absmax, sh.d_out, sh.d_in)
        _, T = O.lora_forward(self.X, Wd, self.A, self.B, sh.s)
        if not self.fwd_only:
            O.lora_backward(self.X, self.dY, Wd, self.A, self.B, sh.s, T=T)

    def time_calls(self, min_seconds: float, max_calls: int = 1000):
        times = []
        t_all = time.perf_counter()
        while len(times) < max_calls:
            t0 = time.perf_counter()
            self.step()
            times.append(time.perf_counter() - t0)
            if time.perf_counter() - t_all >= min_seconds:
                break
        return statistics.median(times), len(times)


def sample_shape(sh, tokens):
    from rank_adapter_linear_nf4_b300.synthetic import LayerShape
    return LayerShape(sh.name, tokens, sh.d_in, sh.d_out, sh.r, sh.alpha, sh.rank_stabilised)


def cpu_baseline(sh, min_seconds=10.0):
    """The oracle on the host cores, all BLAS threads, then one thread, each on a
    bounded sample of the workload's tokens (the full weight every step)."""
    tokens = min(sh.M, 256)
    runner = OracleRunner(sh, tokens)
    threads = runner.blas_threads()
    per_call, calls = runner.time_calls(min_seconds)
    flops = step_flops(sample_shape(sh, tokens))
    out = {"value": flops / per_call / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "tokens_per_s": tokens / per_call,
           "sample": f"{tokens} of {sh.M} tokens of the same workload (NF4 dequantise of the full "
                     f"weight + fp64 forward{'' if fwd_only(sh) else ' + backward'}), median of {calls} calls, "
                     f"{per_call * 1e3:.1f} ms per call, {threads} BLAS threads"}
    out["single_thread"] = single_thread_baseline(sh, min_seconds / 2)
    out["full_runs"] = cpu_full_runs()
    return out


# Workloads small enough for the oracle to run whole (every token) in seconds.
CPU_FULL_CONFIGS = ("tiny", "sweep_m1", "sweep_m16", "sweep_m128")


def cpu_full_runs(min_seconds=1.5):
    """The oracle on whole small workloads, all BLAS threads: per workload the
    median time of one step (NF4 dequantise of the full weight + fp64 forward,
    and backward from 128 tokens on) and its rate."""
    out = {}
    for name in CPU_FULL_CONFIGS:
        sh = shape_of(name)
        runner = OracleRunner(sh, sh.M)
        per_call, calls = runner.time_calls(min_seconds)
        out[name] = {"ms_per_step": per_call * 1e3, "value": step_flops(sh) / per_call / 1e12, "unit": "TFLOP/s",
                     "tokens_per_s": sh.M / per_call, "calls": calls,
                     "step": "fwd" if fwd_only(sh) else "fwd+bwd"}
    return out


SINGLE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def single_thread_baseline(sh, min_seconds):
    """The oracle on one core: a child process with every BLAS thread count set
    to 1 before numpy loads (32 tokens of the workload)."""
    import subprocess
    env = dict(os.environ, **{k: "1" for k in SINGLE_THREAD_ENV})
    env.pop("RANK", None)
    cmd = [sys.executable, os.path.abspath(__file__), "--single-thread-probe", "--config", sh.name,
           "--cpu-seconds", str(min_seconds)]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        return json.loads(res.stdout.strip().splitlines()[-1])
    except Exception as e:   # report, do not fail the run
        return {"error": f"{type(e).__name__}: {e}"[:200]}


def run_single_thread_probe(args):
    sh = shape_of(args.config)
    tokens = min(sh.M, 32)
    runner = OracleRunner(sh, tokens)
    per_call, calls = runner.time_calls(args.cpu_seconds)
    flops = step_flops(sample_shape(sh, tokens))
    print(json.dumps({"value": flops / per_call / 1e12, "unit": "TFLOP/s", "cores": 1,
                      "tokens_per_s": tokens / per_call,
                      "sample": f"{tokens} tokens, median of {calls} calls, {per_call * 1e3:.1f} ms per call, "
                                f"BLAS threads 1 ({', '.join(SINGLE_THREAD_ENV)})"}))
    return 0


# ---------------------------------------------------------------- multi-rank helpers

def max_over_ranks(ms: float, world: int, device) -> float:
    """The job's time: the slowest rank's (all ranks get it).  One rank: unchanged."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_rank_step: float, ms_step: float, world: int) -> float:
    """Whole-job rate: the work every rank did per step over the (max-over-ranks) step time."""
    return work_per_rank_step * world / (ms_step * 1e-3)


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    sh = shape_of(args.config)
    tokens = min(sh.M, 128)
    runner = OracleRunner(sh, tokens)
    threads = runner.blas_threads()
    for _ in range(args.warmup):
        runner.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        runner.step()
    elapsed = time.perf_counter() - t0
    per_step = elapsed / max(1, args.steps)
    sample = sample_shape(sh, tokens)
    value = step_flops(sample) / per_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(sh), "sample_tokens_per_step": tokens},
        "tokens_per_s": tokens / per_step,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {tokens} of {sh.M} tokens (dequantise + fp64 fwd"
                                   f"{'' if fwd_only(sh) else ' + bwd'})"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

class Workload:
    """Resident inputs of one workload on the device, rotated over enough
    copies that no step finds its inputs in L2 (the copies sit at different
    addresses; L2 is physically indexed, so a copy is as cold as new data)."""

    def __init__(self, sh, dev, rank: int, l2: int):
        import torch
        from rank_adapter_linear_nf4_b300 import qlora, synthetic
        self.sh = sh
        M, K, N, r = sh.M, sh.d_in, sh.d_out, sh.r
        self.only_fwd = fwd_only(sh)
        read = 2 * M * K + 0.5625 * K * N + (0 if self.only_fwd else 2 * M * N)
        written = 2 * M * N + (0 if self.only_fwd else 2 * M * K)
        self.set_bytes = read + written
        self.n_sets = max(2, math.ceil(2.0 * l2 / self.set_bytes))
        self.l2 = l2
        self.ws = torch.empty(max(16, qlora.qlora_workspace_bytes(M, K, N, r)), dtype=torch.uint8, device=dev)
        inp = synthetic.layer_inputs(sh, seed=2 + 2 * rank)
        X, dY, W, A, B = (inp[k].to(dev) for k in ("X", "dY", "W", "A", "B"))
        packed, absmax = qlora.qlora_quantize_nf4(W)
        del W
        self.sets = []
        for i in range(self.n_sets):
            c = (lambda t: t) if i == 0 else (lambda t: t.clone())
            self.sets.append(dict(X=c(X), dY=None if self.only_fwd else c(dY), packed=c(packed),
                                  absmax=c(absmax), A=c(A), B=c(B),
                                  Y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                                  XA=torch.empty(M, r, dtype=torch.float32, device=dev),
                                  dX=None if self.only_fwd else torch.empty(M, K, dtype=torch.bfloat16, device=dev),
                                  dA=torch.empty(K, r, dtype=torch.float32, device=dev),
                                  dB=torch.empty(r, N, dtype=torch.float32, device=dev)))
        self.dY0 = dY
        torch.cuda.synchronize()

    def step(self, i):
        from rank_adapter_linear_nf4_b300 import qlora
        sh, t = self.sh, self.sets[i % self.n_sets]
        qlora.qlora_linear_fwd(t["X"], t["packed"], t["absmax"], t["A"], t["B"], sh.s,
                               Y=t["Y"], XA=t["XA"], workspace=self.ws)
        if not self.only_fwd:
            qlora.qlora_linear_bwd(t["X"], t["dY"], t["packed"], t["absmax"], t["A"], t["B"], sh.s,
                                   t["XA"], dX=t["dX"], dA=t["dA"], dB=t["dB"], workspace=self.ws)

    def l2_note(self):
        return (f"inputs rotated over {self.n_sets} resident copies of {self.set_bytes / 1e6:.0f} MB "
                f"(> 2x the {self.l2 / 1e6:.0f} MB L2)")


def make_timer(stream, world, dev, barrier):
    import torch

    def timed(fn, steps):
        """(max-over-ranks ms, host start, host end) of `steps` calls of fn."""
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier()
        h0 = time.perf_counter()
        start.record(stream)
        for i in range(steps):
            fn(i)
        end.record(stream)
        torch.cuda.synchronize()
        h1 = time.perf_counter()
        barrier()
        return max_over_ranks(start.elapsed_time(end), world, dev), h0, h1
    return timed


# Idle time before the per-kernel region, so that it starts from the same power
# state as the timed region before it (a second burst right after the first runs
# under the power cap).
COOL_DOWN_S = 1.0


def per_kernel_profile(wl, steps, timed, sampler):
    """The same steps with every library launch bracketed by CUDA events on its
    stream: per kind, launches, total ms, average us, share; and the clocks of
    that region."""
    from rank_adapter_linear_nf4_b300 import qlora
    time.sleep(COOL_DOWN_S)
    qlora.qlora_profile_enable(True)
    qlora.qlora_profile_collect()
    prof_ms, h0, h1 = timed(wl.step, steps)
    kernels = qlora.qlora_profile_collect()
    qlora.qlora_profile_enable(False)
    total = sum(v[0] for v in kernels.values())
    per = {k: {"launches": n, "total_ms": round(t, 4), "avg_us": round(t / n * 1e3, 2),
               "share": round(t / total, 4)}
           for k, (t, n) in sorted(kernels.items(), key=lambda kv: -kv[1][0])}
    return per, prof_ms / steps, sampler.summary(h0, h1)


def kernel_roofline(sh, name, avg_us, peaks, region_s, clocks=None):
    """Achieved rate of one launch of `name` against its roofline (tensor for
    the main GEMMs of large-token workloads, HBM otherwise)."""
    kf, kb = kernel_work(sh, name)
    t = avg_us * 1e-6
    tpk, tkind = tensor_peak(peaks, region_s, clocks)
    ridge = tpk * 1e12 / (peaks["hbm"] * 1e9)
    tensor = {"achieved": kf / t / 1e12, "unit": "TFLOP/s", "peak": tpk, "frac": kf / t / 1e12 / tpk,
              "peak_kind": tkind, "frac_of_sustained": kf / t / 1e12 / peaks["bf16_sust"],
              "frac_of_burst": kf / t / 1e12 / peaks["bf16"]}
    hbm = {"achieved": kb / t / 1e9, "unit": "GB/s", "peak": peaks["hbm"], "frac": kb / t / 1e9 / peaks["hbm"],
           "peak_kind": f"HBM copy ({peaks['src']})"}
    bound = "tensor" if kb > 0 and kf / kb >= ridge else "hbm"
    main = tensor if bound == "tensor" else hbm
    out = {"bound": bound, "achieved": main["achieved"], "peak": main["peak"], "unit": main["unit"],
           "frac": main["frac"], "kernel": name, "peak_kind": main["peak_kind"],
           "flops_per_launch": kf, "algorithmic_bytes_per_launch": kb, "avg_launch_us": avg_us,
           "arithmetic_intensity": kf / kb if kb else None}
    if bound == "tensor":
        out["frac_of_sustained"] = tensor["frac_of_sustained"]
        out["frac_of_burst"] = tensor["frac_of_burst"]
        out["hbm_frac"] = hbm["frac"]
    else:
        out["tensor_frac"] = tensor["frac"]
    return out


def dominant_layer_kernel(kernels):
    """The layer's heaviest GEMM-type kernel (main fused kernels, or the token-stream forward)."""
    for k in kernels:   # sorted by total time
        if k in ("lora_main_fwd", "lora_main_dX", "lora_stream_fwd"):
            return k
    return next(iter(kernels))


def measure_extra(sh, dev, rank, l2, peaks, timed, sampler, target_s=0.15, warmup=5):
    """One workload beside the headline: step time, per-kernel profile, rooflines."""
    import torch
    wl = Workload(sh, dev, rank, l2)
    for i in range(warmup):
        wl.step(i)
    est_ms, _, _ = timed(wl.step, 3)
    steps = int(max(10, min(2000, target_s / (est_ms / 3 * 1e-3))))
    total_ms, h0, h1 = timed(wl.step, steps)
    ms = total_ms / steps
    kernels, prof_ms, prof_clocks = per_kernel_profile(wl, steps, timed, sampler)
    flops, nbytes = step_flops(sh), step_bytes(sh)
    region_s = total_ms * 1e-3
    step_clocks = sampler.summary(h0, h1)
    tpk, tkind = tensor_peak(peaks, region_s, step_clocks)
    dom = dominant_layer_kernel(kernels)
    res = {"workload": workload_desc(sh), "steps": steps, "ms_per_step": ms,
           "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "tokens_per_s": sh.M / (ms * 1e-3),
           "step_frac_of_bf16": flops / (ms * 1e-3) / 1e12 / tpk, "step_peak_kind": tkind,
           "step_hbm_gbs": nbytes / (ms * 1e-3) / 1e9, "step_frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm"],
           "dominant": kernel_roofline(sh, dom, kernels[dom]["avg_us"], peaks, region_s, prof_clocks),
           "kernels": kernels, "profiled_ms_per_step": prof_ms, "clocks": step_clocks,
           "profiled_clocks": prof_clocks,
           "l2": wl.l2_note()}
    del wl
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    from rank_adapter_linear_nf4_b300 import qlora

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    sh = shape_of(args.config)
    peaks = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.current_stream(dev)
    timed = make_timer(stream, world, dev, barrier)

    sampler = ClockSampler(local)
    sampler.start()
    wl = Workload(sh, dev, rank, l2)

    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()

    # ---- official timed region
    launches0 = qlora.qlora_launch_count()
    total_ms, h0, h1 = timed(wl.step, args.steps)
    clocks = sampler.summary(h0, h1)
    launches = qlora.qlora_launch_count() - launches0
    if qlora.qlora_device_status(clear=True) != 0:
        raise RuntimeError("device status word reports an error during the timed region")

    ms_step = total_ms / args.steps
    region_s = total_ms * 1e-3
    flops = step_flops(sh)
    tflops_rank = flops / (ms_step * 1e-3) / 1e12
    value = job_rate(flops, ms_step, world) / 1e12
    tokens_per_s = job_rate(sh.M, ms_step, world)

    if args.only_steps:   # for profilers: the warm-up and the timed steps, nothing else
        sampler.stop()
        if rank == 0:
            print(json.dumps({"workload": workload_desc(sh), "ms_per_step": ms_step, "value": value,
                              "unit": "TFLOP/s", "steps": args.steps, "note": "--only-steps"}))
        if world > 1:
            dist.destroy_process_group()
        return 0

    # ---- same region again with every library launch bracketed by CUDA events
    per_kernel, prof_ms, prof_clocks = per_kernel_profile(wl, args.steps, timed, sampler)
    roof_kind = dominant_layer_kernel(per_kernel)
    roofline = kernel_roofline(sh, roof_kind, per_kernel[roof_kind]["avg_us"], peaks, region_s, prof_clocks)
    roofline["traffic"] = stored_traffic(roof_kind, sh.name)
    roofline["traffic_note"] = ("dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed ncu "
                                "capture of these kernel sources" if roofline["traffic"] is not None else
                                "no ncu capture of the current kernel sources for this workload")

    # ---- the same steps captured once in a CUDA graph and replayed: launch-amortised
    # time, reported beside (not instead of) the stream-launched value
    graph = graph_timing(wl.step, wl.n_sets, flops, world, timed)

    # ---- end to end: pinned host buffers, copies inside the timed region
    e2e = e2e_timing(wl, args, timed, flops, world)

    codec = codec_rooflines(sh, wl.sets, dev, peaks)

    extra = {}
    blocks = {}
    if not args.no_extra:
        del wl
        torch.cuda.empty_cache()
        try:
            blocks = measure_blocks(dev, timed, peaks)
        except Exception as e:   # report, do not fail the run
            blocks = {"error": f"{type(e).__name__}: {e}"[:300]}
        for name in EXTRA_CONFIGS:
            if name == sh.name:
                continue
            try:
                extra[name] = measure_extra(shape_of(name), dev, rank, l2, peaks, timed, sampler)
            except Exception as e:   # report, do not fail the run
                extra[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    sampler.stop()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    tpk, tkind = tensor_peak(peaks, region_s, clocks)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(sh), "l2": e2e.pop("l2_note"),
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": tokens_per_s,
        "frac_of_bf16_peak_whole_step": {"frac": tflops_rank / tpk, "peak_kind": tkind,
                                         "sustained": tflops_rank / peaks["bf16_sust"],
                                         "burst": tflops_rank / peaks["bf16"]},
        "roofline": roofline,
        "kernels": per_kernel,
        "profiled_ms_per_step": prof_ms,
        "profiled_clocks": prof_clocks,
        "gpu_launches": launches,
        "hbm_kernels": codec,
        "blocks": blocks,
        "cuda_graph": graph,
        "clocks": clocks,
        "e2e": e2e,
        "extra": extra,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sh, min_seconds=args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def e2e_timing(wl, args, timed, flops, world):
    """Forward + backward through the public API from pinned host inputs to host
    outputs, the copies inside the timed region, pipelined as a caller streaming
    host data would: two sets of device buffers, uploads on one stream and
    downloads on another, so that step i+1's upload and step i-1's download run
    beside step i's kernels (and beside each other: the link carries both
    directions at once).  Every step still uploads its X and dY and reads back
    its Y, dX, dA and dB."""
    import torch
    from rank_adapter_linear_nf4_b300 import qlora
    sh, t0 = wl.sh, wl.sets[0]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    hX = t0["X"].cpu().pin_memory()
    hdY = None if wl.only_fwd else wl.dY0.cpu().pin_memory()
    sets = []
    for _ in range(2):
        d = {"X": torch.empty_like(t0["X"]), "Y": torch.empty_like(t0["Y"]), "XA": torch.empty_like(t0["XA"]),
             "hY": torch.empty_like(t0["Y"], device="cpu").pin_memory()}
        for k in ("x_ready", "dy_ready", "fwd_done", "bwd_done", "out_done"):
            d[k] = torch.cuda.Event()
        if not wl.only_fwd:
            d.update({"dY": torch.empty_like(wl.dY0), "dX": torch.empty_like(t0["dX"]),
                      "dA": torch.empty_like(t0["dA"]), "dB": torch.empty_like(t0["dB"]),
                      "hdX": torch.empty_like(t0["dX"], device="cpu").pin_memory(),
                      "hdA": torch.empty_like(t0["dA"], device="cpu").pin_memory(),
                      "hdB": torch.empty_like(t0["dB"], device="cpu").pin_memory()})
        sets.append(d)
    steps = max(3, min(args.steps, 200))

    def e2e_step(i):
        d = sets[i % 2]
        if i == 0:
            s_in.wait_stream(comp)   # nothing before the region's start
        # upload: this set's inputs were last read by step i-2's kernels
        if i >= 2:
            s_in.wait_event(d["bwd_done"])
        with torch.cuda.stream(s_in):
            d["X"].copy_(hX, non_blocking=True)
            d["x_ready"].record(s_in)
            if not wl.only_fwd:
                d["dY"].copy_(hdY, non_blocking=True)
                d["dy_ready"].record(s_in)
        # kernels: this set's outputs were last read back by step i-2's download
        comp.wait_event(d["x_ready"])
        if i >= 2:
            comp.wait_event(d["out_done"])
        qlora.qlora_linear_fwd(d["X"], t0["packed"], t0["absmax"], t0["A"], t0["B"], sh.s,
                               Y=d["Y"], XA=d["XA"], workspace=wl.ws)
        d["fwd_done"].record(comp)
        if not wl.only_fwd:
            comp.wait_event(d["dy_ready"])
            qlora.qlora_linear_bwd(d["X"], d["dY"], t0["packed"], t0["absmax"], t0["A"], t0["B"], sh.s,
                                   d["XA"], dX=d["dX"], dA=d["dA"], dB=d["dB"], workspace=wl.ws)
        d["bwd_done"].record(comp)
        # download: Y as soon as the forward is done, the gradients after the backward
        with torch.cuda.stream(s_out):
            s_out.wait_event(d["fwd_done"])
            d["hY"].copy_(d["Y"], non_blocking=True)
            if not wl.only_fwd:
                s_out.wait_event(d["bwd_done"])
                d["hdX"].copy_(d["dX"], non_blocking=True)
                d["hdA"].copy_(d["dA"], non_blocking=True)
                d["hdB"].copy_(d["dB"], non_blocking=True)
            d["out_done"].record(s_out)
        if i == steps - 1:
            comp.wait_stream(s_out)   # the region ends after the last download
            comp.wait_stream(s_in)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    ms = timed(e2e_step, steps)[0] / steps
    h2d = hX.numel() * 2 + (0 if wl.only_fwd else hdY.numel() * 2)
    d2h = t0["Y"].numel() * 2 + (0 if wl.only_fwd else t0["dX"].numel() * 2 + t0["dA"].numel() * 4 +
                                 t0["dB"].numel() * 4)
    return {"value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "pipeline": "two buffer sets; uploads and downloads on their own streams",
            "l2_note": wl.l2_note()}


def graph_timing(step, n_sets, flops, world, timed, replays=20):
    """Steps captured in one CUDA graph (a whole number of input-set rotations) and
    replayed; ms per step over the replays."""
    import torch
    per_graph = n_sets * max(1, 16 // n_sets)
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(per_graph):   # warm the allocator on the capture stream
                step(i)
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(g):
            for i in range(per_graph):
                step(i)
        g.replay()
        torch.cuda.synchronize()
        ms = timed(lambda i: g.replay(), replays)[0] / (replays * per_graph)
    except Exception as e:   # report, do not fail the run
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    return {"ms_per_step": ms, "value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "steps_per_graph": per_graph, "replays": replays}


def measure_blocks(dev, timed, peaks, reps=10):
    """Rows f3 and f1 as whole calls, each beside its plain form:
    * the SwiGLU MLP block of Llama-3-8B (8192 tokens, 4096 -> 14336 -> 4096,
      rank 64 on gate, up and down), forward + backward, with the gate fused
      into the layers' epilogues against the block with the separate gate kernels;
    * q/k/v of Llama-3-8B (4096 tokens, 4096 -> 4096 + 1024 + 1024, rank 64 each)
      as one grouped layer call against three layer calls, forward + backward.
    Inputs are larger than L2; each form is timed over `reps` back-to-back runs."""
    import torch
    from rank_adapter_linear_nf4_b300 import mlp, multi, qlora, synthetic
    out = {}
    M, dm, dff, r = 8192, 4096, 14336, 64
    s = 16.0 / r
    X, dY = (t.to(dev) for t in synthetic.activations(M, dm, dm, seed=41))
    Wg, Ag, Bg = (t.to(dev) for t in synthetic.weights(dm, dff, r, seed=42))
    Wu, Au, Bu = (t.to(dev) for t in synthetic.weights(dm, dff, r, seed=43))
    Wd, Ad, Bd = (t.to(dev) for t in synthetic.weights(dff, dm, r, seed=44))
    pd, ad = qlora.qlora_quantize_nf4(Wd)
    down = mlp.Layer(pd, ad, Ad, Bd)
    pi, ai = qlora.qlora_quantize_nf4(mlp.interleave_weights(Wg, Wu))
    Ai, Bi = mlp.interleave_adapters(Ag, Bg, Au, Bu)
    gu_fused = mlp.Layer(pi, ai, Ai, Bi)
    ps, as_ = qlora.qlora_quantize_nf4(torch.cat([Wg, Wu], dim=0).contiguous())
    As, Bs = multi.stack_adapters([Ag, Au], [Bg, Bu])
    gu_plain = mlp.Layer(ps, as_, As, Bs)
    del Wg, Wu, Wd

    def fused(i):
        Y, saved = mlp.swiglu_mlp_fwd(X, gu_fused, down, s)
        mlp.swiglu_mlp_bwd(X, dY, saved, gu_fused, down, s)

    def plain(i):
        Y, saved = mlp.swiglu_mlp_fwd_unfused(X, gu_plain, down, s)
        mlp.swiglu_mlp_bwd_unfused(X, dY, saved, gu_plain, down, s)

    flops = (step_flops(synthetic.LayerShape("gu", M, dm, 2 * dff, 2 * r, 16.0)) +
             step_flops(synthetic.LayerShape("d", M, dff, dm, r, 16.0)))
    res = {"workload": f"SwiGLU MLP block, {M} tokens, {dm} -> {dff} -> {dm}, rank {r} (gate/up layer 2 x {r})"}
    for name, fn in (("fused", fused), ("separate_gate", plain)):
        for i in range(2):
            fn(i)
        ms = timed(fn, reps)[0] / reps
        res[name] = {"ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12}
    res["saved_ms"] = res["separate_gate"]["ms_per_step"] - res["fused"]["ms_per_step"]
    out["swiglu_mlp_block"] = res
    del X, dY, down, gu_fused, gu_plain
    torch.cuda.empty_cache()

    M, K, outs, r = 4096, 4096, (4096, 1024, 1024), 64
    s = 16.0 / r
    X, _ = synthetic.activations(M, K, 8, seed=51)
    X = X.to(dev)
    layers = [tuple(t.to(dev) for t in synthetic.weights(K, n, r, seed=52 + i)) for i, n in enumerate(outs)]
    g = torch.Generator(device=dev).manual_seed(53)
    dY = torch.randn(M, sum(outs), device=dev, generator=g).to(torch.bfloat16)
    Ws, As, Bs = [w for w, _, _ in layers], [a for _, a, _ in layers], [b for _, _, b in layers]
    p = multi.packing(Ws, As)
    A_cat, B_cat = multi.stack_adapters(As, Bs, p)
    pk, am = qlora.qlora_quantize_nf4(multi.stack_weights(Ws))
    sep = [(qlora.qlora_quantize_nf4(w), a, b) for w, a, b in layers]
    dYs = [dY[:, sl].contiguous() for sl in p.out_slices()]

    def grouped(i):
        _, _, T = multi.multi_linear_fwd(X, pk, am, A_cat, B_cat, s, p)
        multi.multi_linear_bwd(X, dY, pk, am, A_cat, B_cat, s, T, p)

    def separate(i):
        for ((pq, aq), a, b), dy in zip(sep, dYs):
            _, T = qlora.qlora_linear_fwd(X, pq, aq, a, b, s)
            qlora.qlora_linear_bwd(X, dy, pq, aq, a, b, s, T)

    flops = sum(step_flops(synthetic.LayerShape("p", M, K, n, r, 16.0)) for n in outs)
    res = {"workload": f"q/k/v, {M} tokens, {K} -> {' + '.join(map(str, outs))}, rank {r} each",
           "layout": "grouped" if p.grouped else "dense"}
    for name, fn in (("one_call", grouped), ("three_calls", separate)):
        for i in range(2):
            fn(i)
        ms = timed(fn, reps)[0] / reps
        res[name] = {"ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12}
    res["note"] = "three_calls leaves the three dX to be summed; one_call returns their sum"
    out["stacked_qkv"] = res
    torch.cuda.empty_cache()
    return out


def codec_rooflines(sh, sets, dev, peaks, reps=20):
    """The HBM-bound kernels beside the layer, each timed alone with CUDA events,
    alternating two inputs (> L2 together): NF4 quantise and dequantise of this
    workload's weight (rows a1, a2), the merged weight bf16(W_deq + s.(A.B)^T)
    (the merge export), and the SwiGLU gate and its backward at [M, d_out]
    (the gate between a stacked gate/up layer of this width and a down layer)."""
    import torch
    from rank_adapter_linear_nf4_b300 import qlora
    n = sh.d_in * sh.d_out
    Ws = [qlora.qlora_dequant_nf4(t["packed"], t["absmax"], sh.d_out, sh.d_in) for t in sets[:2]]
    outs = [torch.empty_like(w) for w in Ws]
    pk = [torch.empty_like(t["packed"]) for t in sets[:2]]
    am = [torch.empty_like(t["absmax"]) for t in sets[:2]]
    g = torch.Generator(device=dev).manual_seed(5)
    m_rows = max(sh.M, 1024)
    gus = [torch.randn(m_rows, 2 * sh.d_out, device=dev, generator=g).to(torch.bfloat16) for _ in range(2)]
    dhs = [torch.randn(m_rows, sh.d_out, device=dev, generator=g).to(torch.bfloat16) for _ in range(2)]
    hs = [torch.empty_like(d) for d in dhs]
    dgus = [torch.empty_like(x) for x in gus]
    m_ff = m_rows * sh.d_out
    res = {}
    for name, fn, nbytes, elems in (
            ("nf4_quantize", lambda i: qlora.qlora_quantize_nf4(Ws[i % 2], packed=pk[i % 2], absmax=am[i % 2]),
             2.0 * n + 0.5 * n + n / 16.0, n),
            ("nf4_dequant", lambda i: qlora.qlora_dequant_nf4(sets[i % 2]["packed"], sets[i % 2]["absmax"],
                                                              sh.d_out, sh.d_in, out=outs[i % 2]),
             0.5 * n + n / 16.0 + 2.0 * n, n),
            ("lora_merge", lambda i: qlora.qlora_merge_nf4(sets[i % 2]["packed"], sets[i % 2]["absmax"],
                                                           sets[i % 2]["A"], sets[i % 2]["B"], sh.s, sh.d_out,
                                                           sh.d_in, out=outs[i % 2]),
             0.5 * n + n / 16.0 + 2.0 * n + 2.0 * sh.r * (sh.d_in + sh.d_out), n),
            ("swiglu_fwd", lambda i: qlora.qlora_swiglu_fwd(gus[i % 2], out=hs[i % 2]), 6.0 * m_ff, m_ff),
            ("swiglu_bwd", lambda i: qlora.qlora_swiglu_bwd(gus[i % 2], dhs[i % 2], out=dgus[i % 2]),
             10.0 * m_ff, m_ff)):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        # per-launch CUDA events recorded by the library around each kernel on its
        # stream: device time of the kernel alone, without host call overhead
        qlora.qlora_profile_enable(True)
        qlora.qlora_profile_collect()
        for i in range(reps):
            fn(i)
        prof = qlora.qlora_profile_collect()
        qlora.qlora_profile_enable(False)
        ms, cnt = prof[name]
        us = ms / cnt * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm"], "avg_launch_us": us,
                     "algorithmic_bytes_per_launch": nbytes, "elements": elems}
    del Ws, outs, pk, am, gus, dhs, hs, dgus
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="measure the headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--single-thread-probe", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--only-steps", action="store_true",
                    help="run the warm-up and the timed steps only (for profiler launch lists and captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.single_thread_probe:
        return run_single_thread_probe(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
