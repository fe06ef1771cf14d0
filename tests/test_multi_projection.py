"""Several projections of one input as one stacked layer (q/k/v, gate/up).

CPU tests pin the identity the stacking relies on, with the oracle alone:
quantising the stacked weight gives the stacked codes bit for bit, and the
stacked layer's outputs and gradients equal the separate layers' (dX as
their sum).  GPU tests run the stacked layer through the library and compare
each projection with its own oracle, at the layer tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import multi, synthetic
from tests.parity_utils import TOL, assert_close, np32


def _projections(M, K, d_outs, ranks, seed):
    X, _ = synthetic.activations(M, K, sum(d_outs), seed)
    Ws, As, Bs = [], [], []
    for i, (n, r) in enumerate(zip(d_outs, ranks)):
        W, A, B = synthetic.weights(K, n, r, seed + 1 + i)
        Ws.append(W)
        As.append(A)
        Bs.append(B)
    g = torch.Generator().manual_seed(seed + 99)
    dY = torch.randn(M, sum(d_outs), generator=g).to(torch.bfloat16)
    return X, dY, Ws, As, Bs


def test_packing_layout():
    X, dY, Ws, As, Bs = _projections(4, 128, (64, 32, 32), (8, 4, 4), 0)
    p = multi.packing(Ws, As)
    assert p.d_out == 128 and p.r == 16
    A_cat, B_cat = multi.stack_adapters(As, Bs)
    assert A_cat.shape == (128, 16) and B_cat.shape == (16, 128)
    for i, (rs, os) in enumerate(zip(p.rank_slices(), p.out_slices())):
        assert torch.equal(A_cat[:, rs], As[i])
        assert torch.equal(B_cat[rs, os], Bs[i])
        off = B_cat[rs].clone()
        off[:, os] = 0
        assert float(off.abs().max()) == 0.0          # block-diagonal
    with pytest.raises(ValueError):
        multi.packing(Ws, [torch.zeros(128, 96)] * 3)   # 288 > 256


def test_grouped_packing_layout():
    """Equal ranks of 64: each projection's ranks at 64 * i, B_cat block-diagonal;
    small ranks keep the dense layout unless the grouped one is asked for."""
    _, _, Ws, As, Bs = _projections(4, 128, (256, 128, 128), (64, 64, 64), 0)
    p = multi.packing(Ws, As)
    assert p.grouped and p.group_rank == 64 and p.r == 192
    A_cat, B_cat = multi.stack_adapters(As, Bs, p)
    assert A_cat.shape == (128, 192) and B_cat.shape == (192, 512)
    for i, (rs, os) in enumerate(zip(p.rank_slices(), p.out_slices())):
        assert rs == slice(64 * i, 64 * i + 64)
        assert torch.equal(A_cat[:, rs], As[i]) and torch.equal(B_cat[rs, os], Bs[i])
    _, _, Ws, As, Bs = _projections(4, 128, (256, 128, 96), (16, 8, 16), 0)
    assert not multi.packing(Ws, As).grouped                     # 3 x 64 columns against 40
    p = multi.packing(Ws, As, grouped=True)
    assert p.group_rank == 64 and p.r == 192
    A_cat, B_cat = multi.stack_adapters(As, Bs, p)
    for i, (rs, os) in enumerate(zip(p.rank_slices(), p.out_slices())):
        assert rs == slice(64 * i, 64 * i + p.ranks[i])
        pad = A_cat[:, 64 * i + p.ranks[i]:64 * (i + 1)]
        assert float(pad.abs().max()) == 0.0 if pad.numel() else True
        assert torch.equal(B_cat[rs, os], Bs[i])
    with pytest.raises(ValueError):
        multi.packing(*_projections(4, 128, (96, 128), (8, 8), 0)[2:4], grouped=True)   # 96 % 128 != 0


def test_stacked_quantisation_is_the_stack_of_quantisations():
    _, _, Ws, As, _ = _projections(1, 256, (128, 64, 64), (4, 4, 4), 1)
    parts = [O.quantize_nf4(np32(W)) for W in Ws]
    packed, absmax = O.quantize_nf4(np32(multi.stack_weights(Ws)))
    assert np.array_equal(packed, np.concatenate([q for q, _ in parts]))
    assert np.array_equal(absmax.view(np.uint32), np.concatenate([a for _, a in parts]).view(np.uint32))


@pytest.mark.parametrize("d_outs,grouped", [((64, 32, 32), False), ((128, 128, 64), True)])
def test_stacked_layer_equals_separate_layers_in_the_oracle(d_outs, grouped):
    M, K, ranks, s = 6, 128, (8, 4, 4), 0.5
    X, dY, Ws, As, Bs = _projections(M, K, d_outs, ranks, 2)
    p = multi.packing(Ws, As, grouped=grouped)
    A_cat, B_cat = multi.stack_adapters(As, Bs, p)
    W_cat = multi.stack_weights(Ws)
    q, a = O.quantize_nf4(np32(W_cat))
    Wd_cat = O.dequantize_nf4(q, a, p.d_out, K)
    Xn, dYn = np32(X), np32(dY)
    Y_cat, T_cat = O.lora_forward(Xn, Wd_cat, np32(A_cat), np32(B_cat), s)
    dX_cat, dA_cat, dB_cat = O.lora_backward(Xn, dYn, Wd_cat, np32(A_cat), np32(B_cat), s)
    dX_sum = np.zeros_like(dX_cat)
    for i, (rs, os) in enumerate(zip(p.rank_slices(), p.out_slices())):
        qi, ai = O.quantize_nf4(np32(Ws[i]))
        Wdi = O.dequantize_nf4(qi, ai, d_outs[i], K)
        Yi, Ti = O.lora_forward(Xn, Wdi, np32(As[i]), np32(Bs[i]), s)
        dXi, dAi, dBi = O.lora_backward(Xn, dYn[:, os], Wdi, np32(As[i]), np32(Bs[i]), s)
        np.testing.assert_allclose(Y_cat[:, os], Yi, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(T_cat[:, rs], Ti, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dA_cat[:, rs], dAi, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dB_cat[rs, os], dBi, rtol=1e-12, atol=1e-12)
        dX_sum += dXi
    np.testing.assert_allclose(dX_cat, dX_sum, rtol=1e-10, atol=1e-10)


CASES = [
    # (M, d_in, d_outs, ranks, s, grouped: None = the packing's choice)
    (256, 1024, (1024, 256, 256), (16, 16, 16), 1.0, None),   # q/k/v with grouped-query k, v (dense)
    (8, 1024, (1024, 256, 256), (16, 16, 16), 1.0, None),     # the same with 8 tokens (token-stream forward)
    (192, 512, (1408, 1408), (64, 64), 0.25, False),          # gate/up, dense, sum of ranks 128
    (256, 1024, (1024, 256, 256), (64, 64, 64), 0.25, None),  # q/k/v at rank 64: grouped, 192 rank columns
    (8, 1024, (1024, 256, 256), (64, 64, 64), 0.25, None),    # the same with 8 tokens
    (192, 512, (1408, 1408), (64, 64), 0.25, None),           # gate/up at rank 64: grouped
    (130, 512, (512, 256, 200), (16, 8, 24), 0.5, True),      # grouped with padded ranks, ragged last group
    (8, 512, (1408, 1408), (64, 64), 0.25, True),             # grouped, 8 tokens: the token-stream forward
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "M{}_K{}_N{}_r{}{}".format(
    c[0], c[1], "+".join(map(str, c[2])), "+".join(map(str, c[3])), "_grouped" if c[5] else ""))
def test_stacked_layer_on_gpu(case):
    from rank_adapter_linear_nf4_b300 import qlora
    M, K, d_outs, ranks, s, grouped = case
    X, dY, Ws, As, Bs = _projections(M, K, d_outs, ranks, 3)
    p = multi.packing(Ws, As, grouped=grouped)
    dev = torch.device("cuda", 0)
    A_cat, B_cat = (t.to(dev) for t in multi.stack_adapters(As, Bs, p))
    W_cat = multi.stack_weights(Ws).to(dev)
    packed, absmax = qlora.qlora_quantize_nf4(W_cat)
    # the stacked codes are the separate projections' codes
    for W, os in zip(Ws, p.out_slices()):
        pk, am = qlora.qlora_quantize_nf4(W.to(dev))
        assert torch.equal(pk, packed[os.start * K // 2:os.stop * K // 2])
        assert torch.equal(am, absmax[os.start * K // 64:os.stop * K // 64])
    Xd, dYd = X.to(dev), dY.to(dev)
    Ys, Y_cat, T = multi.multi_linear_fwd(Xd, packed, absmax, A_cat, B_cat, s, p)
    if p.grouped:
        dX, dA_cat, dB_cat = qlora.qlora_linear_bwd_grouped(Xd, dYd, packed, absmax, A_cat, B_cat, s, T, p.d_outs,
                                                            p.group_rank)
        dA, dB = multi.split_grads(dA_cat, dB_cat, p)
    else:
        dX, dA, dB = multi.multi_linear_bwd(Xd, dYd, packed, absmax, A_cat, B_cat, s, T, p)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0
    Xn, dYn = np32(X), np32(dY)
    dX_ref = np.zeros((M, K))
    for i, os in enumerate(p.out_slices()):
        qi, ai = O.quantize_nf4(np32(Ws[i]))
        Wdi = O.dequantize_nf4(qi, ai, d_outs[i], K)
        Yi, _ = O.lora_forward(Xn, Wdi, np32(As[i]), np32(Bs[i]), s)
        dXi, dAi, dBi = O.lora_backward(Xn, dYn[:, os], Wdi, np32(As[i]), np32(Bs[i]), s)
        assert_close(f"Y{i}", np32(Ys[i]), Yi, TOL)
        assert_close(f"dA{i}", dA[i].cpu().numpy(), dAi, TOL)
        assert_close(f"dB{i}", dB[i].cpu().numpy(), dBi, TOL)
        dX_ref += dXi
    assert_close("dX", np32(dX), dX_ref, TOL)
    if p.grouped:
        # dB is computed in the diagonal blocks only: the rest keeps the zeros it started with,
        # so the low-rank work is sum_i group_rank * d_out_i, not r * d_out
        off = dB_cat.clone()
        for g, os in enumerate(p.out_slices()):
            off[g * p.group_rank:(g + 1) * p.group_rank, os] = 0
        assert float(off.abs().max()) == 0.0
