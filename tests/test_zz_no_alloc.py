"""The allocation-free forward (qlora_linear_fwd_noalloc) against the ordinary one
and against the oracle.

The no-workspace entry point exists for callers that cannot hand the layer a
scratch buffer (another allocator owns the device memory, or nothing may be
allocated after start-up).  Its scratch is a fixed array inside the library
that every call reuses, so these checks call it twice in a row on the same
stream and compare both results with qlora_linear_fwd, through the C ABI, and
with the CPU oracle on sampled rows.  This file is collected last on purpose;
it also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import synthetic
from tests.parity_utils import TOL, np32, oracle_weight, rel_max_err

pytestmark = pytest.mark.gpu

QLORA_OK = 0
QLORA_ERR_WORKSPACE = 7


def _lib():
    from rank_adapter_linear_nf4_b300 import qlora
    return qlora.load_library()


def _noalloc_call(lib, X, packed, absmax, A, B, s, Y, XA):
    M, d_in = X.shape
    r, d_out = B.shape
    stream = torch.cuda.current_stream(X.device).cuda_stream
    return lib.qlora_linear_fwd_noalloc(
        X.data_ptr(), M, d_in, d_out, packed.data_ptr(), absmax.data_ptr(), A.data_ptr(),
        B.data_ptr(), r, ctypes.c_float(s), Y.data_ptr(), XA.data_ptr(), stream)


@pytest.mark.parametrize("case", [(300, 320, 136, 12, 1.5),      # r % 8 != 0: padded A in the array
                                  (4096, 4096, 4096, 16, 1.0),    # the q_proj projection
                                  (16, 4096, 4096, 16, 1.0)],     # 16 tokens: panels shared by CTAs, their
                                                                  # counters and partials in the array
                         ids=["ragged_r12", "q_proj", "tokens16_split_panels"])
def test_noalloc_forward_matches_workspace_forward_twice(case):
    from rank_adapter_linear_nf4_b300 import qlora
    M, K, N, r, s = case
    dev = torch.device("cuda", 0)
    lib = _lib()
    X, _ = synthetic.activations(M, K, N, seed=21)
    W, A, B = synthetic.weights(K, N, r, seed=22)
    X, W, A, B = X.to(dev), W.to(dev), A.to(dev), B.to(dev)
    packed, absmax = qlora.qlora_quantize_nf4(W)
    Y_ref, XA_ref = qlora.qlora_linear_fwd(X, packed, absmax, A, B, s)
    # the oracle on sampled rows (all rows for the small cases)
    rows = synthetic.sample_rows(M, n=64, block=32) if M > 512 else None
    _, _, Wd = oracle_weight(W.cpu())
    Y_o, T_o = O.lora_forward(np32(X), Wd, np32(A), np32(B), s, rows=rows)
    sel = slice(None) if rows is None else rows
    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        XA = torch.full((M, r), float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc_call(lib, X, packed, absmax, A, B, s, Y, XA) == QLORA_OK
        torch.cuda.synchronize()
        assert qlora.qlora_device_status(clear=True) == 0
        for name, got, ref, orc in (("Y", Y, Y_ref, Y_o), ("XA", XA, XA_ref, T_o)):
            g = got.float().cpu().numpy()
            r_ = ref.float().cpu().numpy()
            assert np.all(np.isfinite(g)), (call, name)
            assert rel_max_err(g, r_) <= TOL, (call, name)
            assert rel_max_err(g[sel], orc) <= TOL, (call, name, "oracle")


def test_noalloc_rejects_shapes_beyond_its_array():
    lib = _lib()
    fake = 0x10000   # never dereferenced: the size check fails first
    status = lib.qlora_linear_fwd_noalloc(fake, 1 << 20, 4096, 4096, fake, fake, fake, fake, 64,
                                          ctypes.c_float(1.0), fake, fake, None)
    assert status == QLORA_ERR_WORKSPACE
