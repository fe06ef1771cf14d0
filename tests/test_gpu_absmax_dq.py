"""The block absmax stored in 8 bits (row f4) on the GPU against the oracle.

Bit-exact: the stored bytes and group scales, and the expanded absmax, against
oracle.quantize_absmax_dq / dequantize_absmax_dq (both take the decisions in
fp32 with IEEE division and round-to-nearest-even).  Then the layer run on the
expanded absmax against the oracle's layer on the oracle's expansion, at the
layer tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import synthetic
from tests.parity_utils import TOL, assert_close, np32

pytestmark = pytest.mark.gpu


def _round_trip(a_np):
    from rank_adapter_linear_nf4_b300 import qlora
    a = torch.from_numpy(np.ascontiguousarray(a_np, dtype=np.float32)).cuda()
    q8, sc = qlora.qlora_quantize_absmax_dq(a)
    back = qlora.qlora_dequant_absmax_dq(q8, sc)
    torch.cuda.synchronize()
    q_ref, sc_ref = O.quantize_absmax_dq(a_np)
    assert np.array_equal(q8.cpu().numpy(), q_ref)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(back.cpu().numpy().view(np.uint32), O.dequantize_absmax_dq(q_ref, sc_ref).view(np.uint32))


@pytest.mark.parametrize("n", [1, 255, 256, 257, 700, 65536 + 37])
def test_absmax_dq_bitexact_random(n):
    g = np.random.default_rng(n)
    a = (np.abs(g.normal(size=n)) * np.exp(g.uniform(-6, 6, size=n))).astype(np.float32)
    if n > 600:
        a[256:512] = 0.0                     # an all-zero group
    _round_trip(a)


def test_absmax_dq_bitexact_weight_absmax():
    """The absmax of a full-size weight (the MLP projection), as quantised."""
    from rank_adapter_linear_nf4_b300 import qlora
    sh = synthetic.SHAPES["llama3_8b_mlp_up"]
    W, _, _ = synthetic.weights(sh.d_in, sh.d_out, sh.r, seed=7)
    _, absmax = qlora.qlora_quantize_nf4(W.cuda())
    _round_trip(absmax.cpu().numpy())


def test_absmax_dq_representable_scales():
    g = np.random.default_rng(3)
    k = g.integers(0, 256, size=512)
    k[5] = k[300] = 255
    a = (k * 2.0 ** -9).astype(np.float32)
    _round_trip(a)


@pytest.mark.parametrize("case", [(96, 512, 384, 16, 1.0), (8, 1024, 512, 64, 0.5)],
                         ids=lambda c: "M{}_K{}_N{}_r{}".format(*c[:4]))
def test_layer_on_8bit_absmax(case):
    from rank_adapter_linear_nf4_b300 import qlora
    M, K, N, r, s = case
    X, dY = synthetic.activations(M, K, N, seed=M)
    W, A, B = synthetic.weights(K, N, r, seed=M + 1)
    dev = torch.device("cuda", 0)
    packed, absmax = qlora.qlora_quantize_nf4(W.to(dev))
    q8, sc = qlora.qlora_quantize_absmax_dq(absmax)
    absmax2 = qlora.qlora_dequant_absmax_dq(q8, sc)          # the scale the layer runs on
    Xd, dYd, Ad, Bd = X.to(dev), dY.to(dev), A.to(dev), B.to(dev)
    Y, T = qlora.qlora_linear_fwd(Xd, packed, absmax2, Ad, Bd, s)
    dX, dA, dB = qlora.qlora_linear_bwd(Xd, dYd, packed, absmax2, Ad, Bd, s, T)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0
    p_np = packed.cpu().numpy()
    q_ref, sc_ref = O.quantize_absmax_dq(absmax.cpu().numpy())
    Wd = O.dequantize_nf4(p_np, O.dequantize_absmax_dq(q_ref, sc_ref), N, K)
    Y_ref, T_ref = O.lora_forward(np32(X), Wd, np32(A), np32(B), s)
    dX_ref, dA_ref, dB_ref = O.lora_backward(np32(X), np32(dY), Wd, np32(A), np32(B), s)
    assert_close("Y", np32(Y), Y_ref, TOL)
    assert_close("dX", np32(dX), dX_ref, TOL)
    assert_close("dA", dA.cpu().numpy(), dA_ref, TOL)
    assert_close("dB", dB.cpu().numpy(), dB_ref, TOL)
    # the 8-bit scale moves the weight by at most half a step of its group's scale
    Wd_fp32 = O.dequantize_nf4(p_np, absmax.cpu().numpy(), N, K)
    assert np.max(np.abs(Wd - Wd_fp32)) <= np.max(sc_ref) * 0.5 * 1.01 + np.max(np.abs(Wd_fp32)) * 2.0 ** -7
