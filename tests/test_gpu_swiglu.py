"""SwiGLU gate and the SwiGLU MLP block on the GPU against the oracle.

The gate is elementwise: every output is checked against the fp64 oracle to
one bf16 ulp (the kernel computes in fp32 and rounds once), besides the layer
bar max|gpu - oracle| <= 1e-2 max|oracle|.  The block (stacked gate/up layer,
gate, down layer, and the backward through all three) is checked at the layer
bar against the oracle's composition, whose intermediates are stored in bf16
as the block stores them.
"""
import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import mlp, multi, synthetic
from tests.parity_utils import TOL, assert_close, np32

pytestmark = pytest.mark.gpu


def _ulp_close(name, got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    bound = np.abs(ref) * 2.0 ** -7 + 1e-30
    bad = int(np.count_nonzero(err > bound))
    assert bad == 0, f"{name}: {bad} elements off by more than one bf16 ulp"
    assert_close(name, got, ref, TOL)


@pytest.mark.parametrize("M,d_ff,scale", [(1, 8, 1.0), (37, 2816, 2.0), (256, 14336, 4.0), (5, 64, 30.0)])
def test_swiglu_gate(M, d_ff, scale):
    from rank_adapter_linear_nf4_b300 import qlora
    g = torch.Generator().manual_seed(M + d_ff)
    gu = (torch.randn(M, 2 * d_ff, generator=g) * scale).to(torch.bfloat16)
    dh = torch.randn(M, d_ff, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    h = qlora.qlora_swiglu_fwd(gu.to(dev))
    dgu = qlora.qlora_swiglu_bwd(gu.to(dev), dh.to(dev))
    torch.cuda.synchronize()
    _ulp_close("h", np32(h), O.swiglu_forward(np32(gu)))
    _ulp_close("dgu", np32(dgu), O.swiglu_backward(np32(gu), np32(dh)))


def test_swiglu_empty():
    from rank_adapter_linear_nf4_b300 import qlora
    dev = torch.device("cuda", 0)
    gu = torch.empty(0, 128, dtype=torch.bfloat16, device=dev)
    assert qlora.qlora_swiglu_fwd(gu).shape == (0, 64)
    assert qlora.qlora_swiglu_bwd(gu, torch.empty(0, 64, dtype=torch.bfloat16, device=dev)).shape == (0, 128)


@pytest.mark.parametrize("M,d_model,d_ff,r,s", [(192, 512, 1408, 32, 0.5), (8, 1024, 2816, 64, 0.25)])
def test_swiglu_mlp_block(M, d_model, d_ff, r, s):
    """gate/up (ranks r + r) -> SwiGLU -> down (rank r), forward and backward."""
    from rank_adapter_linear_nf4_b300 import qlora
    X, _ = synthetic.activations(M, d_model, d_model, 21)
    Wg, Ag, Bg = synthetic.weights(d_model, d_ff, r, 22)
    Wu, Au, Bu = synthetic.weights(d_model, d_ff, r, 23)
    Wd, Ad, Bd = synthetic.weights(d_ff, d_model, r, 24)
    dY = torch.randn(M, d_model, generator=torch.Generator().manual_seed(25)).to(torch.bfloat16)
    A_gu, B_gu = multi.stack_adapters([Ag, Au], [Bg, Bu])
    W_gu = multi.stack_weights([Wg, Wu])
    dev = torch.device("cuda", 0)
    pk_gu, am_gu = qlora.qlora_quantize_nf4(W_gu.to(dev))
    pk_d, am_d = qlora.qlora_quantize_nf4(Wd.to(dev))
    gate_up = mlp.Layer(pk_gu, am_gu, A_gu.to(dev), B_gu.to(dev))
    down = mlp.Layer(pk_d, am_d, Ad.to(dev), Bd.to(dev))
    Xd = X.to(dev)
    Y, saved = mlp.swiglu_mlp_fwd(Xd, gate_up, down, s)
    dX, (dA_gu, dB_gu), (dA_d, dB_d) = mlp.swiglu_mlp_bwd(Xd, dY.to(dev), saved, gate_up, down, s)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0

    q, a = O.quantize_nf4(np32(W_gu))
    Wd_gu = O.dequantize_nf4(q, a, 2 * d_ff, d_model)
    q, a = O.quantize_nf4(np32(Wd))
    Wd_d = O.dequantize_nf4(q, a, d_model, d_ff)
    args = (Wd_gu, np32(A_gu), np32(B_gu), Wd_d, np32(Ad), np32(Bd), s)
    Y_ref, saved_ref = O.swiglu_mlp_forward(np32(X), *args)
    dX_ref, (dA_gu_ref, dB_gu_ref), (dA_d_ref, dB_d_ref) = O.swiglu_mlp_backward(np32(X), np32(dY), saved_ref, *args)
    assert_close("Y", np32(Y), Y_ref)
    assert_close("dX", np32(dX), dX_ref)
    assert_close("dA_d", dA_d.cpu().numpy(), dA_d_ref)
    assert_close("dB_d", dB_d.cpu().numpy(), dB_d_ref)
    p = multi.packing([Wg, Wu], [Ag, Au])
    dA_gu_i, dB_gu_i = multi.split_grads(dA_gu, dB_gu, p)
    dA_ref_i, dB_ref_i = multi.split_grads(torch.from_numpy(dA_gu_ref), torch.from_numpy(dB_gu_ref), p)
    for i in range(2):
        assert_close(f"dA_gu{i}", dA_gu_i[i].cpu().numpy(), dA_ref_i[i].numpy())
        assert_close(f"dB_gu{i}", dB_gu_i[i].cpu().numpy(), dB_ref_i[i].numpy())
