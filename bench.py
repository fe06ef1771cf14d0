#!/usr/bin/env python3
"""Benchmark: fused NF4-QLoRA linear layer, forward + backward, on B300.

One step = one forward (qlora_linear_fwd) and one backward (qlora_linear_bwd)
of the projection workload over one batch of synthetic tokens, inputs already
resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

N > 1 is launched by torchrun: each rank runs its own independent replica of
the workload on its own GPU (no collective on the data path; "scaling": "weak").
`--impl reference` times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
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
DEFAULT_CONFIG = "llama3_8b_q_proj"


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


def sources_hash() -> str:
    """Hash of the CUDA sources: a stored ncu traffic figure counts only for these."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "rank_adapter_linear_nf4_b300", "csrc")
    for fn in sorted(os.listdir(csrc)):
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
    if not e or e.get("sources") != sources_hash():
        return None
    return e.get("dram_bytes_per_launch")


def kernel_work(sh, kind):
    """Algorithmic (flops, bytes) of one launch of a main fused kernel."""
    M, K, N, r = sh.M, sh.d_in, sh.d_out, sh.r
    w_bytes = 0.5625 * K * N
    if kind == "lora_main_fwd":
        return 2.0 * M * K * N + 2.0 * M * r * N, w_bytes + 2.0 * M * K + 2.0 * M * N + 2.0 * M * r + 2.0 * r * N
    return 2.0 * M * K * N + 2.0 * M * r * K, w_bytes + 2.0 * M * N + 2.0 * M * K + 2.0 * M * r + 2.0 * r * K


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


# ---------------------------------------------------------------- clocks (NVML)

class ClockSampler:
    """Samples SM clock, power and clock-event reasons during the timed region:
    NVML every ~10 ms in a thread, else `nvidia-smi -lms 100` in the background."""

    REASONS = [("gpu_idle", 0x1), ("applications_clocks", 0x2), ("sw_power_cap", 0x4),
               ("hw_slowdown", 0x8), ("sync_boost", 0x10), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake", 0x80)]
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active"]

    def __init__(self, torch_dev: int):
        self.mode = None
        self.samples = []
        self.err = ""
        try:
            import pynvml
            import torch
            pynvml.nvmlInit()
            self.nv = pynvml
            try:
                uuid = str(torch.cuda.get_device_properties(torch_dev).uuid)
                self.h = pynvml.nvmlDeviceGetHandleByUUID(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
            except Exception:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[torch_dev]) if vis and vis.split(",")[0].isdigit() else torch_dev
                self.h = pynvml.nvmlDeviceGetHandleByIndex(idx)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err = f"NVML: {e!r}"
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "smi"
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                self.smi_index = vis.split(",")[torch_dev] if vis else str(torch_dev)

    def _reasons(self):
        nv = self.nv
        for fn in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
            if hasattr(nv, fn):
                return int(getattr(nv, fn)(self.h))
        return 0

    def _run(self):
        while not self._stop.is_set():
            try:
                sm = self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM)
                pw = self.nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0
                self.samples.append((sm, pw, self._reasons()))
            except Exception:
                pass
            time.sleep(0.01)

    def start(self):
        if self.mode == "nvml":
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        elif self.mode == "smi":
            import subprocess
            self._p = subprocess.Popen(
                ["nvidia-smi", "-i", self.smi_index, "--query-gpu=" + ",".join(self.SMI_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

    def stop(self):
        if self.mode == "nvml":
            self._stop.set()
            self._t.join()
        elif self.mode == "smi":
            self._p.terminate()
            out, _ = self._p.communicate(timeout=10)
            self.max_mhz = None
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.max_mhz = float(f[1])
                    self.samples.append((float(f[0]), float(f[2]), int(f[3], 16)))
                except (ValueError, IndexError):
                    pass
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no clock source: " + self.err}
        s = self.samples
        mask = 0
        for _, _, r in s:
            mask |= r
        reasons = [n for n, b in self.REASONS if mask & b and n != "gpu_idle"]
        out = {"sm_mhz": statistics.median([x[0] for x in s]) if s else None,
               "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(s),
               "power_w_median": statistics.median([x[1] for x in s]) if s else None,
               "source": self.mode}
        if self.err:
            out["note"] = self.err
        return out


# ---------------------------------------------------------------- oracle timing (CPU)

class OracleRunner:
    """The oracle on the first `tokens` tokens of the workload: one step is
    NF4 dequantisation of the full weight + forward + backward (fp64)."""

    def __init__(self, sh, tokens: int):
        from oracle import qlora_oracle as O
        from rank_adapter_linear_nf4_b300 import synthetic
        self.O, self.sh = O, sh
        X, dY = synthetic.activations(tokens, sh.d_in, sh.d_out, seed=0)
        W, A, B = synthetic.weights(sh.d_in, sh.d_out, sh.r, seed=1)
        f = lambda t: t.float().numpy()
        self.X, self.dY, self.A, self.B = f(X), f(dY), f(A), f(B)
        self.packed, self.absmax = O.quantize_nf4(f(W))
        try:
            from threadpoolctl import threadpool_info
            self.threads = max([int(i.get("num_threads", 1)) for i in threadpool_info()] or [1])
        except Exception:
            self.threads = os.cpu_count() or 1

    def step(self):
        O, sh = self.O, self.sh
        Wd = O.dequantize_nf4(self.packed, self.absmax, sh.d_out, sh.d_in)
        _, T = O.lora_forward(self.X, Wd, self.A, self.B, sh.s)
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
    tokens = min(sh.M, 256)
    runner = OracleRunner(sh, tokens)
    per_call, calls = runner.time_calls(min_seconds)
    flops = step_flops(sample_shape(sh, tokens))
    return {"value": flops / per_call / 1e12, "unit": "TFLOP/s", "cores": runner.threads, "kind": "oracle",
            "tokens_per_s": tokens / per_call,
            "sample": f"{tokens} of {sh.M} tokens of the same workload (NF4 dequantise of the full "
                      f"weight + fp64 forward + backward), median of {calls} calls, "
                      f"{per_call * 1e3:.1f} ms per call"}


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
    threads = runner.threads
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
                         "sample": f"each step: {tokens} of {sh.M} tokens (dequantise + fp64 fwd + bwd)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist
    from rank_adapter_linear_nf4_b300 import qlora, synthetic

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

    # ---- resident input sets, rotated so that no step finds its inputs in L2
    M, K, N, r = sh.M, sh.d_in, sh.d_out, sh.r
    set_bytes = 2 * M * K + 2 * M * N + 0.5625 * K * N + 2 * M * K + 2 * M * N
    n_sets = max(2, math.ceil(2.0 * l2 / set_bytes))
    sets = []
    ws = torch.empty(max(16, qlora.qlora_workspace_bytes(M, K, N, r)), dtype=torch.uint8, device=dev)
    for i in range(n_sets):
        inp = synthetic.layer_inputs(sh, seed=2 * i + 2 * rank * n_sets)
        X, dY, W, A, B = (inp[k].to(dev) for k in ("X", "dY", "W", "A", "B"))
        packed, absmax = qlora.qlora_quantize_nf4(W)
        del W
        sets.append(dict(X=X, dY=dY, packed=packed, absmax=absmax, A=A, B=B,
                         Y=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                         XA=torch.empty(M, r, dtype=torch.float32, device=dev),
                         dX=torch.empty(M, K, dtype=torch.bfloat16, device=dev),
                         dA=torch.empty(K, r, dtype=torch.float32, device=dev),
                         dB=torch.empty(r, N, dtype=torch.float32, device=dev)))
    torch.cuda.synchronize()

    only_fwd = fwd_only(sh)

    def step(i):
        t = sets[i % n_sets]
        qlora.qlora_linear_fwd(t["X"], t["packed"], t["absmax"], t["A"], t["B"], sh.s,
                               Y=t["Y"], XA=t["XA"], workspace=ws)
        if not only_fwd:
            qlora.qlora_linear_bwd(t["X"], t["dY"], t["packed"], t["absmax"], t["A"], t["B"], sh.s,
                                   t["XA"], dX=t["dX"], dA=t["dA"], dB=t["dB"], workspace=ws)

    def timed(fn, steps):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier()
        start.record(stream)
        for i in range(steps):
            fn(i)
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(start.elapsed_time(end), world, dev)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # ---- official timed region
    sampler = ClockSampler(local)
    launches0 = qlora.qlora_launch_count()
    sampler.start()
    total_ms = timed(step, args.steps)
    clocks = sampler.stop()
    launches = qlora.qlora_launch_count() - launches0
    if qlora.qlora_device_status(clear=True) != 0:
        raise RuntimeError("device status word reports an error during the timed region")

    ms_step = total_ms / args.steps
    flops = step_flops(sh)
    tflops_rank = flops / (ms_step * 1e-3) / 1e12
    value = job_rate(flops, ms_step, world) / 1e12
    tokens_per_s = job_rate(M, ms_step, world)

    # ---- same region again with every library launch bracketed by CUDA events
    qlora.qlora_profile_enable(True)
    qlora.qlora_profile_collect()
    prof_total_ms = timed(step, args.steps)
    kernels = qlora.qlora_profile_collect()
    qlora.qlora_profile_enable(False)
    dom = max(kernels.items(), key=lambda kv: kv[1][0])[0]
    main_kinds = [k for k in ("lora_main_fwd", "lora_main_dX") if k in kernels]
    roof_kind = dom if dom in ("lora_main_fwd", "lora_main_dX") else (main_kinds[0] if main_kinds else dom)
    k_ms, k_n = kernels[roof_kind]
    k_avg_s = k_ms / k_n * 1e-3
    kf, kb = kernel_work(sh, roof_kind)
    ridge = peaks["bf16_sust"] * 1e12 / (peaks["hbm"] * 1e9)
    if kf / kb >= ridge:
        achieved = kf / k_avg_s / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_sust"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_sust"], "traffic": None,
                    "kernel": roof_kind, "peak_kind": f"bf16 dense sustained ({peaks['src']})",
                    "frac_of_burst_peak": achieved / peaks["bf16"]}
    else:
        achieved = kb / k_avg_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm"], "traffic": None, "kernel": roof_kind,
                    "peak_kind": f"HBM copy ({peaks['src']})"}
    roofline["flops_per_launch"] = kf
    roofline["algorithmic_bytes_per_launch"] = kb
    roofline["avg_launch_us"] = k_avg_s * 1e6
    roofline["traffic"] = stored_traffic(roof_kind, sh.name)
    roofline["traffic_note"] = ("dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed ncu "
                                "capture of these kernel sources" if roofline["traffic"] is not None else
                                "no ncu capture of the current kernel sources")
    per_kernel = {k: {"launches": n, "total_ms": round(t, 4), "avg_us": round(t / n * 1e3, 2),
                      "share": round(t / sum(v[0] for v in kernels.values()), 4)}
                  for k, (t, n) in sorted(kernels.items(), key=lambda kv: -kv[1][0])}

    # ---- the same steps captured once in a CUDA graph and replayed: launch-amortised
    # time, reported beside (not instead of) the stream-launched value
    graph = graph_timing(step, n_sets, flops, world, timed)

    # ---- end to end: pinned host buffers, copies inside the timed region
    t0 = sets[0]
    hX = t0["X"].cpu().pin_memory()
    hdY = t0["dY"].cpu().pin_memory()
    hY = torch.empty_like(t0["Y"], device="cpu").pin_memory()
    hdX = torch.empty_like(t0["dX"], device="cpu").pin_memory()
    hdA = torch.empty_like(t0["dA"], device="cpu").pin_memory()
    hdB = torch.empty_like(t0["dB"], device="cpu").pin_memory()
    dX_in, dY_in = torch.empty_like(t0["X"]), torch.empty_like(t0["dY"])

    def e2e_step(i):
        dX_in.copy_(hX, non_blocking=True)
        if not only_fwd:
            dY_in.copy_(hdY, non_blocking=True)
        qlora.qlora_linear_fwd(dX_in, t0["packed"], t0["absmax"], t0["A"], t0["B"], sh.s,
                               Y=t0["Y"], XA=t0["XA"], workspace=ws)
        hY.copy_(t0["Y"], non_blocking=True)
        if not only_fwd:
            qlora.qlora_linear_bwd(dX_in, dY_in, t0["packed"], t0["absmax"], t0["A"], t0["B"], sh.s,
                                   t0["XA"], dX=t0["dX"], dA=t0["dA"], dB=t0["dB"], workspace=ws)
            hdX.copy_(t0["dX"], non_blocking=True)
            hdA.copy_(t0["dA"], non_blocking=True)
            hdB.copy_(t0["dB"], non_blocking=True)

    e2e_step(0)
    e2e_steps = max(3, min(args.steps, 200))
    e2e_ms = timed(e2e_step, e2e_steps) / e2e_steps
    h2d = hX.numel() * 2 + (0 if only_fwd else hdY.numel() * 2)
    d2h = hY.numel() * 2 + (0 if only_fwd else hdX.numel() * 2 + hdA.numel() * 4 + hdB.numel() * 4)

    codec = codec_rooflines(sh, sets, dev, peaks, stream)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(sh),
                   "l2": f"inputs rotated over {n_sets} resident sets of {set_bytes / 1e6:.0f} MB "
                         f"(> 2x the {l2 / 1e6:.0f} MB L2)",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": tokens_per_s,
        "frac_of_bf16_peak_whole_step": {"sustained": tflops_rank / peaks["bf16_sust"],
                                         "burst": tflops_rank / peaks["bf16"]},
        "roofline": roofline,
        "kernels": per_kernel,
        "profiled_ms_per_step": prof_total_ms / args.steps,
        "gpu_launches": launches,
        "hbm_kernels": codec,
        "cuda_graph": graph,
        "clocks": clocks,
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sh, min_seconds=args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


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
        ms = timed(lambda i: g.replay(), replays) / (replays * per_graph)
    except Exception as e:   # report, do not fail the run
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    return {"ms_per_step": ms, "value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "steps_per_graph": per_graph, "replays": replays}


def codec_rooflines(sh, sets, dev, peaks, stream, reps=20):
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
    gus = [torch.randn(sh.M, 2 * sh.d_out, device=dev, generator=g).to(torch.bfloat16) for _ in range(2)]
    dhs = [torch.randn(sh.M, sh.d_out, device=dev, generator=g).to(torch.bfloat16) for _ in range(2)]
    hs = [torch.empty_like(d) for d in dhs]
    dgus = [torch.empty_like(x) for x in gus]
    m_ff = sh.M * sh.d_out
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
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
