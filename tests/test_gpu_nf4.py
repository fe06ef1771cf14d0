"""NF4 quantise / dequantise on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import synthetic

pytestmark = pytest.mark.gpu


def _quant_gpu(W):
    from rank_adapter_linear_nf4_b300 import qlora
    packed, absmax = qlora.qlora_quantize_nf4(W.cuda())
    Wd = qlora.qlora_dequant_nf4(packed, absmax, W.shape[0], W.shape[1])
    torch.cuda.synchronize()
    return packed.cpu().numpy(), absmax.cpu().numpy(), Wd.cpu()


def _check_weight(W):
    packed, absmax, Wd = _quant_gpu(W)
    Wn = W.float().numpy()
    p_ref, a_ref = O.quantize_nf4(Wn)
    assert np.array_equal(packed, p_ref)
    assert np.array_equal(absmax.view(np.uint32), a_ref.view(np.uint32))
    d_ref = O.dequantize_nf4(p_ref, a_ref, W.shape[0], W.shape[1])
    assert np.array_equal(Wd.float().numpy().view(np.uint32), d_ref.view(np.uint32))


@pytest.mark.parametrize("shape", [(256, 256), (40, 576), (1, 64), (136, 320), (4096, 4096)])
def test_quantize_dequant_bitexact_random(shape):
    n_out, n_in = shape
    W, _, _ = synthetic.weights(n_in, n_out, 8, seed=n_out + n_in)
    _check_weight(W)


@pytest.mark.parametrize("name", ["llama3_8b_mlp_up", "qwen14b_mlp"])
def test_quantize_dequant_bitexact_full_size(name):
    sh = synthetic.SHAPES[name]
    W, _, _ = synthetic.weights(sh.d_in, sh.d_out, sh.r, seed=1)
    _check_weight(W)


def test_codebook_points_and_zero_blocks():
    g = np.random.default_rng(5)
    n_out, n_in = 64, 512
    nb = n_out * n_in // 64
    q = g.integers(0, 16, size=(nb, 64)).astype(np.uint8)
    q[np.arange(nb), g.integers(0, 64, size=nb)] = 15
    a = torch.tensor(np.exp2(g.uniform(-12, 6, size=nb)), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    vals = (O.NF4_CODE[q] * a[:, None]).astype(np.float32)
    vals[::7] = 0.0                                  # every 7th block all zero
    W = torch.from_numpy(vals.reshape(n_out, n_in)).to(torch.bfloat16)
    packed, absmax, Wd = _quant_gpu(W)
    nz = np.ones(nb, dtype=bool)
    nz[::7] = False
    assert np.array_equal(O.unpack_codes(packed).reshape(nb, 64)[nz], q[nz])
    assert np.all(O.unpack_codes(packed).reshape(nb, 64)[~nz] == 7)
    assert np.array_equal(absmax[nz], a[nz]) and np.all(absmax[~nz] == 0)
    assert np.array_equal(Wd.float().numpy().view(np.uint32), W.float().numpy().view(np.uint32))


def test_dequant_arbitrary_codes():
    from rank_adapter_linear_nf4_b300 import qlora
    g = np.random.default_rng(9)
    n_out, n_in = 96, 448
    packed = g.integers(0, 256, size=n_out * n_in // 2, dtype=np.uint8)
    absmax = g.uniform(0, 50, size=n_out * n_in // 64).astype(np.float32)
    absmax[::5] = 0
    Wd = qlora.qlora_dequant_nf4(torch.from_numpy(packed).cuda(), torch.from_numpy(absmax).cuda(),
                                 n_out, n_in)
    ref = O.dequantize_nf4(packed, absmax, n_out, n_in)
    assert np.array_equal(Wd.cpu().float().numpy().view(np.uint32), ref.view(np.uint32))
