"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/qlora.h declares, validates arguments before touching
the device, and carries the same NF4 table as the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import qlora_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from rank_adapter_linear_nf4_b300 import build, qlora
    build.build()
    return qlora.load_library()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(qlora_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("qlora_quantize_nf4", "qlora_dequant_nf4", "qlora_linear_fwd",
                     "qlora_linear_bwd", "qlora_workspace_bytes", "qlora_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_codebook_equals_oracle(lib):
    from rank_adapter_linear_nf4_b300 import qlora
    assert np.array_equal(np.float32(qlora.qlora_nf4_codebook()), O.NF4_CODE)


def test_status_strings(lib):
    from rank_adapter_linear_nf4_b300 import qlora
    for code, name in qlora.STATUS_NAMES.items():
        assert qlora.qlora_status_string(code).startswith(name)


def test_workspace_bytes(lib):
    from rank_adapter_linear_nf4_b300 import qlora
    assert qlora.qlora_workspace_bytes(64, 256, 256, 8) > 0
    # padded A + two [M, rp] bf16 buffers, rp = 64
    assert qlora.qlora_workspace_bytes(4096, 4096, 4096, 16) >= (4096 + 2 * 4096) * 64 * 2
    assert qlora.qlora_workspace_bytes(64, 100, 256, 8) == 0      # d_in % 64
    assert qlora.qlora_workspace_bytes(64, 256, 252, 8) == 0      # d_out % 8
    assert qlora.qlora_workspace_bytes(64, 256, 256, 0) == 0
    assert qlora.qlora_workspace_bytes(64, 256, 256, 257) == 0
    assert qlora.qlora_workspace_bytes(64, 256, 256, 256) > 0


FAKE = 0x10000      # 16-byte aligned, never dereferenced: validation fails first
MISALIGNED = 0x10008


def _fwd(lib, X=FAKE, M=64, K=256, N=256, P=FAKE, S=FAKE, A=FAKE, B=FAKE, r=8, Y=FAKE, XA=FAKE,
         ws=FAKE, ws_bytes=1 << 30):
    return lib.qlora_linear_fwd(X, M, K, N, P, S, A, B, r, 2.0, Y, XA, ws, ws_bytes, None)


def test_forward_argument_validation(lib):
    assert _fwd(lib, K=100) == 4
    assert _fwd(lib, N=260 - 2) == 4
    assert _fwd(lib, r=0) == 4 and _fwd(lib, r=257) == 4
    assert _fwd(lib, M=-1) == 2 and _fwd(lib, K=0) == 2
    assert _fwd(lib, X=None) == 1 and _fwd(lib, P=None) == 1 and _fwd(lib, XA=None) == 1
    assert _fwd(lib, X=MISALIGNED) == 3 and _fwd(lib, Y=MISALIGNED) == 3
    assert _fwd(lib, ws=None) == 7 or _fwd(lib, ws=None) == 3
    assert _fwd(lib, ws_bytes=16) == 7
    assert _fwd(lib, M=0, X=None, Y=None, XA=None) == 0   # empty input launches nothing


def test_backward_argument_validation(lib):
    def bwd(X=FAKE, dY=FAKE, M=64, dX=FAKE, dA=FAKE, dB=FAKE, ws_bytes=1 << 30, K=256):
        return lib.qlora_linear_bwd(X, dY, M, K, 256, FAKE, FAKE, FAKE, FAKE, 8, 2.0, FAKE,
                                    dX, dA, dB, FAKE, ws_bytes, None)
    assert bwd(dA=None) == 1 and bwd(dB=None) == 1 and bwd(dY=None) == 1
    assert bwd(dX=MISALIGNED) == 3
    assert bwd(ws_bytes=0) == 7
    assert bwd(K=320 + 1) == 4


def test_codec_argument_validation(lib):
    assert lib.qlora_quantize_nf4(FAKE, 4, 100, FAKE, FAKE, None) == 4
    assert lib.qlora_quantize_nf4(FAKE, 0, 64, FAKE, FAKE, None) == 2
    assert lib.qlora_quantize_nf4(None, 4, 64, FAKE, FAKE, None) == 1
    assert lib.qlora_dequant_nf4(FAKE, MISALIGNED, 4, 64, FAKE, None) == 3


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from rank_adapter_linear_nf4_b300 import qlora
    with pytest.raises(ValueError):
        qlora.qlora_quantize_nf4(torch.zeros(4, 64, dtype=torch.bfloat16))


def test_merge_argument_validation(lib):
    def merge(N=256, K=256, r=8, P=FAKE, S=FAKE, A=FAKE, B=FAKE, out=FAKE):
        return lib.qlora_merge_nf4(P, S, N, K, A, B, r, 1.0, out, None)
    assert merge(r=0) == 4 and merge(r=129) == 4
    assert merge(K=100) == 4 and merge(N=252) == 4
    assert merge(N=0) == 2
    assert merge(A=None) == 1 and merge(out=None) == 1
    assert merge(out=MISALIGNED) == 3


def test_swiglu_argument_validation(lib):
    def fwd(M=4, d_ff=64, gu=FAKE, h=FAKE):
        return lib.qlora_swiglu_fwd(gu, M, d_ff, h, None)

    def bwd(M=4, d_ff=64, gu=FAKE, dh=FAKE, dgu=FAKE):
        return lib.qlora_swiglu_bwd(gu, dh, M, d_ff, dgu, None)
    assert fwd(d_ff=12) == 4 and bwd(d_ff=12) == 4
    assert fwd(d_ff=0) == 2 and fwd(M=-1) == 2 and bwd(d_ff=0) == 2
    assert fwd(gu=None) == 1 and bwd(dh=None) == 1 and bwd(dgu=None) == 1
    assert fwd(h=MISALIGNED) == 3 and bwd(gu=MISALIGNED) == 3
    assert fwd(M=0, gu=None, h=None) == 0 and bwd(M=0, gu=None, dh=None, dgu=None) == 0


def test_stall_hook_is_off_by_default_and_rejects_negative(lib):
    from rank_adapter_linear_nf4_b300 import qlora
    assert lib.qlora_debug_stall_main_launches(-1) == 2     # QLORA_ERR_SHAPE, nothing armed
    assert lib.qlora_debug_stall_main_launches(0) == 0


def test_absmax_dq_argument_validation(lib):
    assert lib.qlora_quantize_absmax_dq(FAKE, 0, FAKE, FAKE, None) == 2
    assert lib.qlora_quantize_absmax_dq(None, 8, FAKE, FAKE, None) == 1
    assert lib.qlora_quantize_absmax_dq(FAKE, 8, MISALIGNED, FAKE, None) == 3
    assert lib.qlora_dequant_absmax_dq(FAKE, FAKE, -1, FAKE, None) == 2
    assert lib.qlora_dequant_absmax_dq(FAKE, None, 8, FAKE, None) == 1
    assert lib.qlora_dequant_absmax_dq(FAKE, FAKE, 8, MISALIGNED, None) == 3


def test_grouped_argument_validation(lib):
    import ctypes
    groups = (ctypes.c_int64 * 3)(256, 128, 128)

    def fwd(n=3, g=groups, width=64, M=16, K=256):
        return lib.qlora_linear_fwd_grouped(FAKE, M, K, n, g, width, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, FAKE,
                                            FAKE, 1 << 30, None)
    assert fwd(g=None) == 1
    assert fwd(n=0) == 4 and fwd(n=9) == 4
    assert fwd(width=32) == 4                                # a multiple of 64
    assert fwd(width=128) == 4                               # 3 x 128 > 256
    assert fwd(g=(ctypes.c_int64 * 3)(200, 128, 128)) == 4   # a group but the last not a multiple of 128
    assert fwd(g=(ctypes.c_int64 * 3)(256, 0, 128)) == 2
    assert fwd(K=100) == 4
