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


def _all_bf16_upto(m_bits: int) -> np.ndarray:
    """Every bf16 bit pattern w with |w| <= the positive bf16 m_bits (both signs)."""
    pos = np.arange(0, m_bits + 1, dtype=np.uint32).astype(np.uint16)
    return np.concatenate([pos, pos | np.uint16(0x8000)])


@pytest.mark.parametrize("m_bits", [0x3F80, 0x3C23, 0x4121, 0x3E9B, 0x0080, 0x0005, 0x7E00, 0x7F7F])
def test_quantize_every_weight_of_an_absmax(m_bits):
    """Brute force over the code decision: for one absmax m, every bf16 weight
    |w| <= m (tens of thousands of values, so every value next to a decision
    threshold is among them) is quantised in blocks that all hold m, and each
    code is compared with the oracle's.  The m values cover ordinary scales, the
    smallest normal and a subnormal bf16, and scales near the top of the range."""
    vals = _all_bf16_upto(m_bits)
    per = 63
    nb = -(-vals.size // per)
    nb = -(-nb // 64) * 64                               # whole rows of 64 blocks
    blocks = np.zeros((nb, 64), dtype=np.uint16)
    blocks[:, 0] = m_bits                                 # absmax of every block is m
    flat = np.zeros(nb * per, dtype=np.uint16)
    flat[:vals.size] = vals
    blocks[:, 1:] = flat.reshape(nb, per)
    W = torch.from_numpy(blocks.view(np.int16).reshape(nb // 64, 64 * 64)).view(torch.bfloat16)
    _check_weight(W)


# (absmax, weight) bf16 pairs whose quotient lies within 2^-21 of a decision
# threshold (found by scanning every absmax in [1, 2) and every weight; scaling
# both by a power of two keeps the quotient): the closest calls the code
# decision has to make
_NEAR_PAIRS = [(0x3F83, 0x3ECC), (0x3FA1, 0x3D4D), (0x3FA2, 0xBD6C), (0x3FF3, 0xBDB1)]


def test_quantize_weights_next_to_thresholds():
    rows = []
    for m_bits, w_bits in _NEAR_PAIRS:
        for k in (-100, -20, -7, 0, 5, 60, 120):       # both scaled by 2^k
            blk = np.full(64, (w_bits & 0x7FFF) + (k << 7) | (w_bits & 0x8000), dtype=np.uint16)
            blk[0] = m_bits + (k << 7)
            blk[1::2] ^= 0x8000                          # both signs
            rows.append(blk)
    blocks = np.stack(rows)
    blocks = np.concatenate([blocks, np.zeros((64 - len(blocks) % 64, 64), dtype=np.uint16)])
    W = torch.from_numpy(blocks.view(np.int16).reshape(-1, 64 * 64)).view(torch.bfloat16)
    _check_weight(W)
