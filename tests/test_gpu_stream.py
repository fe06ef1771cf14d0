"""The forward for 1..16 tokens (the NF4 weight-stream kernel) against the oracle.

Same bar as the other layer tests: per output tensor, max|gpu - oracle| <=
1e-2 * max|oracle|, every element compared.  The kernel splits its items (16
weight rows x 256 input features) evenly over CTAs and warps, in units of 16
rows x 1024 features; the cases walk units split between two warps or CTAs,
row groups summed over many slices (long d_in), a last slice shorter than
1024, ragged last row groups (d_out % 16 != 0), ranks 1..128 and token counts
on both sides of 8.  d_in % 256 != 0 goes to the main kernel.
Low-rank-dominant cases (zero base weight, B ~ N(0, 1)) check that term on its
own, since with the standard scales it is only a few percent of Y.
"""
import pytest
import torch

from rank_adapter_linear_nf4_b300 import synthetic
from tests.parity_utils import check_layer, run_gpu

pytestmark = pytest.mark.gpu


def _inputs(M, K, N, r, seed=0, b_std=0.01):
    X, dY = synthetic.activations(M, K, N, seed)
    W, A, B = synthetic.weights(K, N, r, seed + 1, b_std=b_std)
    return {"X": X, "dY": dY, "W": W, "A": A, "B": B}


CASES = [
    # (M, d_in, d_out, r, s); an item is 16 weight rows x 256 input features
    (1, 256, 256, 16, 1.0),         # 16 units of one item
    (3, 256, 64, 8, 2.0),           # a single CTA
    (8, 4096, 64, 16, 1.0),         # four slices per row group
    (9, 512, 136, 24, 0.5),         # two token groups with 9 tokens; last group 8 rows; units split
    (16, 512, 14336, 128, 0.25),    # 896 row groups; rank 128
    (5, 14336, 256, 64, 0.25),      # long contraction: 14 slices per row group
    (16, 4096, 4096, 16, 1.0),      # the q_proj layer at 16 tokens
    (12, 512, 200, 65, 1.25),       # rank padded to 128, A padded (r % 8 != 0), last group 8 rows
    (2, 256, 8, 1, 3.0),            # one 8-row group (8 rows past d_out), rank 1
    (4, 1024, 64 * 148 + 8, 16, 0.5),   # 593 row groups, the last one 8 rows
    (7, 1280, 14336, 32, 0.5),      # a last slice of 256 features
    (16, 320, 96, 48, 1.0),         # d_in % 256 != 0: the main kernel
    (1, 192, 40, 4, 2.0),           # d_in % 256 != 0: the main kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M{}_K{}_N{}_r{}".format(*c[:4]))
def test_stream_forward_full(case):
    M, K, N, r, s = case
    check_layer(_inputs(M, K, N, r, seed=M + N + K), s, bwd=False)


@pytest.mark.parametrize("case", [(1, 256, 256, 16, 1.0), (16, 512, 136, 100, 0.75), (7, 4096, 192, 64, 0.5)],
                         ids=lambda c: "M{}_K{}_N{}_r{}".format(*c[:4]))
def test_stream_lowrank_dominant(case):
    M, K, N, r, s = case
    inp = _inputs(M, K, N, r, seed=11, b_std=1.0)
    inp["W"] = torch.zeros_like(inp["W"])
    check_layer(inp, s, bwd=False)


def test_stream_with_backward():
    """Forward through the stream kernel, backward through the main kernels."""
    check_layer(_inputs(16, 512, 384, 16, seed=5), 0.5)


def test_stream_kernel_is_the_one_launched():
    from rank_adapter_linear_nf4_b300 import qlora
    dev = torch.device("cuda", 0)
    # 1..16 tokens with d_in % 256 == 0 take the stream kernel, the rest the main kernel
    for M, K, want, other in ((16, 256, "lora_stream_fwd", "lora_main_fwd"), (17, 256, "lora_main_fwd", "lora_stream_fwd"),
                              (4, 320, "lora_main_fwd", "lora_stream_fwd")):
        inp = _inputs(M, K, 256, 16, seed=M)
        X, W, A, B = (inp[k].to(dev) for k in ("X", "W", "A", "B"))
        packed, absmax = qlora.qlora_quantize_nf4(W)
        torch.cuda.synchronize()
        qlora.qlora_profile_enable(True)
        qlora.qlora_profile_collect()
        qlora.qlora_linear_fwd(X, packed, absmax, A, B, 1.0)
        prof = qlora.qlora_profile_collect()
        qlora.qlora_profile_enable(False)
        assert prof.get(want, (0.0, 0))[1] == 1, (M, prof)
        assert prof.get(other, (0.0, 0))[1] == 0, (M, prof)


def test_stream_repeat_is_bitwise_identical():
    """Row groups are summed by whichever warp completes them last, in slice and
    part order: repeated calls give the same bits."""
    inp = _inputs(16, 4096, 14336, 64, seed=2)
    a = run_gpu(inp, 0.25, bwd=False)
    for _ in range(3):
        b = run_gpu(inp, 0.25, bwd=False)
        assert torch.equal(a["Y"], b["Y"])
