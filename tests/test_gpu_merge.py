"""The merged 16-bit weight (qlora_merge_nf4) on the GPU against the oracle.

Bar: the oracle rounds the exact fp64 value W_deq + s.(A.B)^T once to bf16; the
kernel accumulates A.B in fp32 and rounds fma(s, AB, W_deq) to bf16.  At least
99.9 % of the elements are bit-identical (the fp32 accumulation moves a value
across a bf16 rounding boundary only when it lands very close to one), and
every element is within one bf16 step of the oracle plus the fp32 rounding of
its operands, 2^-20 * (|W_deq| + |s| * (|A| . |B|)^T) -- where W_deq and the
adapter term nearly cancel, that absolute term is what bounds the difference.
"""
import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import synthetic

pytestmark = pytest.mark.gpu

CASES = [
    # (d_out, d_in, r, s).  r % 8 == 0 takes the persistent kernel (A^T, B^T by TMA,
    # a run of tiles per CTA); other ranks the one-tile-per-CTA kernel.
    (256, 256, 8, 2.0),        # fewer tiles than SMs
    (136, 320, 12, 1.5),       # ragged tiles in both directions, r % 8 != 0
    (136, 320, 16, 1.5),       # the same raggedness on the persistent kernel
    (1000, 1280, 24, 0.5),     # last row block 104 rows, rank 24 (B^T rows past r are zero)
    (384, 512, 128, 0.125),
    (1024, 4096, 64, 0.25),
    (4096, 4096, 16, 1.0),     # the q_proj weight: runs of ~7 tiles crossing row blocks
    (8200, 4096, 64, 0.25),    # 65 row blocks, the last 8 rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N{}_K{}_r{}".format(*c[:3]))
def test_merge_matches_oracle(case):
    from rank_adapter_linear_nf4_b300 import qlora
    N, K, r, s = case
    dev = torch.device("cuda", 0)
    W, A, B = synthetic.weights(K, N, r, seed=N + r, b_std=0.05)
    packed, absmax = qlora.qlora_quantize_nf4(W.to(dev))
    out = qlora.qlora_merge_nf4(packed, absmax, A.to(dev), B.to(dev), s, N, K)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0
    got = out.float().cpu().numpy()
    p_np = packed.cpu().numpy()
    a_np = absmax.cpu().numpy()
    Wd = O.dequantize_nf4(p_np, a_np, N, K)
    ref = O.merged_weight_bf16(Wd, A.float().numpy(), B.float().numpy(), s)
    same = O.bf16_bits(got) == O.bf16_bits(ref)
    assert same.mean() >= 0.999, same.mean()
    mag = np.abs(Wd).astype(np.float64) + abs(s) * (np.abs(A.float().numpy()).astype(np.float64)
                                                     @ np.abs(B.float().numpy()).astype(np.float64)).T
    bound = np.abs(ref) * 2.0 ** -7 + mag * 2.0 ** -20
    assert np.all(np.abs(got.astype(np.float64) - ref) <= bound)


def test_merge_zero_adapter_is_dequant():
    """B = 0: the merged weight is qlora_dequant_nf4's output, bit for bit."""
    from rank_adapter_linear_nf4_b300 import qlora
    dev = torch.device("cuda", 0)
    W, A, B = synthetic.weights(512, 384, 32, seed=5)
    packed, absmax = qlora.qlora_quantize_nf4(W.to(dev))
    out = qlora.qlora_merge_nf4(packed, absmax, A.to(dev), torch.zeros_like(B).to(dev), 3.0, 384, 512)
    deq = qlora.qlora_dequant_nf4(packed, absmax, 384, 512)
    torch.cuda.synchronize()
    assert torch.equal(out, deq)
