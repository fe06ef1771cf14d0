"""The error path of the bounded device waits, without a GPU fault.

Every wait in the library's kernels gives up after about one second, records
QLORA_ERR_TIMEOUT in the device status word and lets the kernel wind down.
The test hook qlora_debug_stall_main_launches(n) makes the next n launches of
the fused main kernel load no token operand, so none of its stages completes
and its waits run out (nothing else is changed: no trap, no bad address, no
unbounded loop).  The checks: the status word reports the timeout, the
context stays usable, and the next ordinary call matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O
from rank_adapter_linear_nf4_b300 import synthetic
from tests.parity_utils import TOL, np32, oracle_weight, rel_max_err

pytestmark = pytest.mark.gpu

QLORA_ERR_TIMEOUT = 6


def test_stalled_main_kernel_reports_timeout_then_recovers():
    from rank_adapter_linear_nf4_b300 import qlora
    dev = torch.device("cuda", 0)
    M, K, N, r, s = 64, 256, 384, 8, 2.0      # more than 16 tokens: the fused main kernel
    X, _ = synthetic.activations(M, K, N, seed=31)
    W, A, B = synthetic.weights(K, N, r, seed=32)
    Xd, Wd_, Ad, Bd = X.to(dev), W.to(dev), A.to(dev), B.to(dev)
    packed, absmax = qlora.qlora_quantize_nf4(Wd_)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0

    qlora.qlora_debug_stall_main_launches(1)
    try:
        t0 = time.perf_counter()
        qlora.qlora_linear_fwd(Xd, packed, absmax, Ad, Bd, s)
        code = qlora.qlora_device_status(clear=True)      # synchronises
        waited = time.perf_counter() - t0
    finally:
        qlora.qlora_debug_stall_main_launches(0)
    assert code == QLORA_ERR_TIMEOUT
    assert 0.5 < waited < 30.0, waited                   # the wait ran out after about a second

    # the context is intact and the next call is the ordinary one
    Y, XA = qlora.qlora_linear_fwd(Xd, packed, absmax, Ad, Bd, s)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0
    _, _, Wdq = oracle_weight(W)
    Y_ref, T_ref = O.lora_forward(np32(X), Wdq, np32(A), np32(B), s)
    assert rel_max_err(np32(Y), Y_ref) <= TOL
    assert rel_max_err(XA.cpu().numpy(), T_ref) <= TOL



@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_stalled_pair_kernel_reports_timeout_then_recovers(direction):
    """The same for the main kernel's CTA-pair form (256-token tiles, at least
    256 output features): both CTAs of every pair wind down after the stalled
    waits, and the next call is the ordinary one."""
    from rank_adapter_linear_nf4_b300 import qlora
    dev = torch.device("cuda", 0)
    M, K, N, r, s = 512, 384, 512, 8, 2.0     # 256-token tiles; Y and dX both have >= 256 features
    X, dY = synthetic.activations(M, K, N, seed=41)
    W, A, B = synthetic.weights(K, N, r, seed=42)
    Xd, dYd, Wd_, Ad, Bd = X.to(dev), dY.to(dev), W.to(dev), A.to(dev), B.to(dev)
    packed, absmax = qlora.qlora_quantize_nf4(Wd_)
    Y, XA = qlora.qlora_linear_fwd(Xd, packed, absmax, Ad, Bd, s)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0

    qlora.qlora_debug_stall_main_launches(1)
    try:
        t0 = time.perf_counter()
        if direction == "fwd":
            qlora.qlora_linear_fwd(Xd, packed, absmax, Ad, Bd, s)
        else:
            qlora.qlora_linear_bwd(Xd, dYd, packed, absmax, Ad, Bd, s, XA)
        code = qlora.qlora_device_status(clear=True)
        waited = time.perf_counter() - t0
    finally:
        qlora.qlora_debug_stall_main_launches(0)
    assert code == QLORA_ERR_TIMEOUT
    assert 0.5 < waited < 30.0, waited

    _, _, Wdq = oracle_weight(W)
    if direction == "fwd":
        Y, XA = qlora.qlora_linear_fwd(Xd, packed, absmax, Ad, Bd, s)
        torch.cuda.synchronize()
        assert qlora.qlora_device_status(clear=True) == 0
        Y_ref, _ = O.lora_forward(np32(X), Wdq, np32(A), np32(B), s)
        assert rel_max_err(np32(Y), Y_ref) <= TOL
    else:
        dX, dA_, dB_ = qlora.qlora_linear_bwd(Xd, dYd, packed, absmax, Ad, Bd, s, XA)
        torch.cuda.synchronize()
        assert qlora.qlora_device_status(clear=True) == 0
        dX_ref, dA_ref, dB_ref = O.lora_backward(np32(X), np32(dY), Wdq, np32(A), np32(B), s)
        assert rel_max_err(np32(dX), dX_ref) <= TOL
        assert rel_max_err(dA_.cpu().numpy(), dA_ref) <= TOL
        assert rel_max_err(dB_.cpu().numpy(), dB_ref) <= TOL
