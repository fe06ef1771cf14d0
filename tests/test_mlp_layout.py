"""Host-side layout of the fused SwiGLU block: the interleaved order of the
gate/up layer's rows (64-row chunks, gate then up) and its inverse."""
import torch

from rank_adapter_linear_nf4_b300 import mlp


def test_interleave_roundtrip():
    d_ff = 192
    gu = torch.arange(2 * d_ff, dtype=torch.float32).reshape(1, -1)
    W_g = torch.arange(d_ff, dtype=torch.float32).reshape(-1, 1)
    W_u = W_g + 1000
    W_int = mlp.interleave_weights(W_g, W_u)
    assert W_int[:64, 0].tolist() == list(range(64))
    assert W_int[64:128, 0].tolist() == [1000 + i for i in range(64)]
    assert W_int[128:192, 0].tolist() == list(range(64, 128))
    assert torch.equal(mlp.deinterleave(gu[:, mlp.gate_up_order(d_ff)]), gu)


def test_interleaved_adapters_place_each_rank_block_in_its_columns():
    d_ff, r = 128, 3
    Bg = torch.full((r, d_ff), 1.0)
    Bu = torch.full((r, d_ff), 2.0)
    A = torch.zeros(8, r)
    A_cat, B_int = mlp.interleave_adapters(A, Bg, A, Bu)
    assert A_cat.shape == (8, 2 * r) and B_int.shape == (2 * r, 2 * d_ff)
    B = mlp.deinterleave(B_int)
    assert torch.all(B[:r, :d_ff] == 1.0) and torch.all(B[:r, d_ff:] == 0.0)
    assert torch.all(B[r:, d_ff:] == 2.0) and torch.all(B[r:, :d_ff] == 0.0)
    # gate feature f sits in column 128 * (f // 64) + f % 64 of the interleaved layout
    assert torch.all(B_int[:r, 64:128] == 0.0) and torch.all(B_int[:r, 0:64] == 1.0)
