"""The bench's measurement arithmetic on CPU: the step's algorithmic flops are
the sum over the kernels one step launches (so a dominant kernel's fraction
and the step's fraction rest on the same counts), and the bf16 peak a region
is judged against follows the clock regime it ran in."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_logic_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


SHAPES = ["tiny", "llama3_8b_q_proj", "llama3_8b_mlp_up", "qwen14b_attn", "sweep_m1", "sweep_m16", "sweep_m128",
          "sweep_m16384"]


@pytest.mark.parametrize("name", SHAPES)
def test_step_flops_are_the_kernels_flops(bench, name):
    sh = bench.shape_of(name)
    if bench.fwd_only(sh):
        # one forward: the weight stream (or main kernel) and the rank-r pre-pass T = X.A
        kinds = ("lora_stream_fwd", "lora_rows_T")
    else:
        kinds = ("lora_main_fwd", "lora_main_dX", "lora_rows_T", "lora_rows_G", "lora_red_dA_dB")
    total = sum(bench.kernel_work(sh, k)[0] for k in kinds)
    assert total == pytest.approx(bench.step_flops(sh), rel=1e-12)


def test_step_flops_closed_form(bench):
    # forward 2MKN + 2Mr(K+N); backward 2MKN (dX) + 2Mr(K+N) (G, then dX's low-rank
    # stages) + 2Mr(K+N) (dA and dB); M = 16384, 4096 -> 14336, r = 64
    M, K, N, r = 16384, 4096, 14336, 64
    assert bench.step_flops(bench.shape_of("sweep_m16384")) == 4.0 * M * K * N + 6.0 * M * r * (K + N)


def test_forward_only_below_128_tokens(bench):
    assert bench.fwd_only(bench.shape_of("sweep_m16"))
    assert not bench.fwd_only(bench.shape_of("sweep_m128"))


PEAKS = {"bf16": 1811.4, "bf16_sust": 1393.8, "hbm": 6497.4, "src": "measured"}


def _clocks(mhz, reasons, samples=50, top=2032):
    return {"sm_mhz": mhz, "sm_max_mhz": top, "reasons": reasons, "samples": samples}


def test_short_region_at_full_clock_takes_the_burst_peak(bench):
    peak, kind = bench.tensor_peak(PEAKS, 0.06, _clocks(2032, []))
    assert peak == 1811.4 and "burst" in kind


def test_long_region_takes_the_sustained_peak(bench):
    peak, kind = bench.tensor_peak(PEAKS, 1.5, _clocks(2032, []))
    assert peak == 1393.8 and "sustained" in kind


def test_power_capped_short_region_takes_the_sustained_peak(bench):
    peak, kind = bench.tensor_peak(PEAKS, 0.7, _clocks(1582, ["sw_power_cap"]))
    assert peak == 1393.8 and "sw_power_cap" in kind


def test_cap_reason_without_a_slower_clock_is_not_a_cap(bench):
    # the reason flag alone, with the median clock at its maximum
    assert not bench.power_capped(_clocks(2032, ["sw_power_cap"]))
    # a slow clock without the reason is not attributed to the cap either
    assert not bench.power_capped(_clocks(1500, []))
    # no samples: nothing is known, the region is judged by its length
    assert not bench.power_capped(_clocks(1500, ["sw_power_cap"], samples=0))
    peak, _ = bench.tensor_peak(PEAKS, 0.7, None)
    assert peak == 1811.4


def test_job_rate_counts_every_rank(bench):
    # 100 units per rank-step, 10 ms per step, 4 ranks: 40,000 units/s
    assert bench.job_rate(100.0, 10.0, 4) == pytest.approx(40000.0)
