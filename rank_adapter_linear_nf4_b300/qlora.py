"""Thin Python binding of the C ABI in ``include/qlora.h``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libqlora_b300.so``.  Tensors are torch CUDA tensors (torch is
used for device memory and streams); calls are queued on the current torch
stream of the tensors' device.  There is no CPU fallback: if the library is
not built, or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

QLORA_OK = 0
STATUS_NAMES = {
    0: "QLORA_OK", 1: "QLORA_ERR_NULL", 2: "QLORA_ERR_SHAPE", 3: "QLORA_ERR_ALIGN",
    4: "QLORA_ERR_UNSUPPORTED", 5: "QLORA_ERR_CUDA", 6: "QLORA_ERR_TIMEOUT",
    7: "QLORA_ERR_WORKSPACE",
    8: "QLORA_ERR_INTERNAL",
}

_c_void_p, _i64, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "qlora_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qlora_last_cuda_error": (ctypes.c_int, []),
    "qlora_nf4_codebook": (None, [ctypes.POINTER(ctypes.c_float)]),
    "qlora_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "qlora_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "qlora_profile_collect": (ctypes.c_int, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float),
                                             ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "qlora_launch_count": (ctypes.c_int64, []),
    "qlora_debug_stall_main_launches": (ctypes.c_int, [ctypes.c_int]),
    "qlora_quantize_nf4": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "qlora_dequant_nf4": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p]),
    "qlora_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32]),
    "qlora_quantize_absmax_dq": (ctypes.c_int, [_c_void_p, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "qlora_dequant_absmax_dq": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "qlora_linear_fwd": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p,
                                        _c_void_p, _c_void_p, _i32, _f32, _c_void_p, _c_void_p,
                                        _c_void_p, _sz, _c_void_p]),
    "qlora_linear_fwd_noalloc": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p,
                                                _c_void_p, _c_void_p, _i32, _f32, _c_void_p, _c_void_p,
                                                _c_void_p]),
    "qlora_merge_nf4": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p, _i32, _f32,
                                       _c_void_p, _c_void_p]),
    "qlora_swiglu_fwd": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p]),
    "qlora_swiglu_bwd": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p]),
    "qlora_linear_fwd_swiglu": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                                               _c_void_p, _i32, _f32, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                               _sz, _c_void_p]),
    "qlora_linear_bwd_swiglu": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p,
                                               _c_void_p, _c_void_p, _i32, _f32, _c_void_p, _c_void_p, _c_void_p,
                                               _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "qlora_swiglu_mlp_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, _i32]),
    "qlora_swiglu_mlp_fwd": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _f32,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _f32,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                            _c_void_p, _sz, _c_void_p]),
    "qlora_swiglu_mlp_bwd": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _i64,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _f32,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _f32,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                            _c_void_p, _sz, _c_void_p]),
    "qlora_linear_bwd": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p, _i32, _f32, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p, _c_void_p, _sz,
                                        _c_void_p]),
    "qlora_linear_fwd_grouped": (ctypes.c_int, [_c_void_p, _i64, _i64, _i32, ctypes.POINTER(_i64), _i32,
                                                _c_void_p, _c_void_p, _c_void_p, _c_void_p, _f32, _c_void_p,
                                                _c_void_p, _c_void_p, _sz, _c_void_p]),
    "qlora_linear_bwd_grouped": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _i32, ctypes.POINTER(_i64),
                                                _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _f32,
                                                _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _sz,
                                                _c_void_p]),
}

_lib = None


class QloraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == 5 and _lib is not None:
            detail = f" (cudaError {_lib.qlora_last_cuda_error()})"
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}{detail}")


def load_library(path: str = LIB_PATH):
    """Loads the native library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with rank_adapter_linear_nf4_b300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != QLORA_OK:
        raise QloraError(fn, status)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def qlora_status_string(status: int) -> str:
    return load_library().qlora_status_string(status).decode()


def qlora_nf4_codebook() -> list[float]:
    buf = (ctypes.c_float * 16)()
    load_library().qlora_nf4_codebook(buf)
    return list(buf)


def qlora_device_status(clear: bool = True) -> int:
    """Synchronises the device and returns (optionally clears) the status word."""
    code = ctypes.c_int(0)
    _check("qlora_device_status", load_library().qlora_device_status(ctypes.byref(code), int(clear)))
    return code.value


def qlora_profile_enable(enable: bool = True) -> None:
    """Bracket every library kernel launch with CUDA events (launch accounting)."""
    _check("qlora_profile_enable", load_library().qlora_profile_enable(int(enable)))


def qlora_profile_collect() -> dict:
    """Per kernel kind since the last collect: {name: (total_ms, launches)}."""
    n_max = 16
    names = (ctypes.c_char_p * n_max)()
    ms = (ctypes.c_float * n_max)()
    cnt = (ctypes.c_int * n_max)()
    n = load_library().qlora_profile_collect(names, ms, cnt, n_max)
    if n < 0:
        raise QloraError("qlora_profile_collect", 5)
    return {names[i].decode(): (float(ms[i]), int(cnt[i])) for i in range(n)}


def qlora_launch_count() -> int:
    return int(load_library().qlora_launch_count())


def qlora_debug_stall_main_launches(launches: int) -> None:
    """Test hook: the next `launches` launches of the fused main kernel load no
    token operand, so their bounded waits run out and report QLORA_ERR_TIMEOUT."""
    _check("qlora_debug_stall_main_launches", load_library().qlora_debug_stall_main_launches(int(launches)))


def qlora_workspace_bytes(M: int, d_in: int, d_out: int, r: int) -> int:
    return int(load_library().qlora_workspace_bytes(M, d_in, d_out, r))


def qlora_quantize_nf4(W: torch.Tensor, packed: torch.Tensor | None = None,
                       absmax: torch.Tensor | None = None):
    """W [n_out, n_in] bf16 -> (packed uint8 [n_out*n_in/2], absmax fp32 [n_out*n_in/64])."""
    lib = load_library()
    n_out, n_in = W.shape
    if packed is None:
        packed = torch.empty(n_out * n_in // 2, dtype=torch.uint8, device=W.device)
    if absmax is None:
        absmax = torch.empty(n_out * n_in // 64, dtype=torch.float32, device=W.device)
    _check("qlora_quantize_nf4", lib.qlora_quantize_nf4(
        _dev(W, "W", torch.bfloat16), n_out, n_in, _dev(packed, "packed", torch.uint8),
        _dev(absmax, "absmax", torch.float32), _stream(W)))
    return packed, absmax


def qlora_dequant_nf4(packed: torch.Tensor, absmax: torch.Tensor, n_out: int, n_in: int,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    lib = load_library()
    if out is None:
        out = torch.empty(n_out, n_in, dtype=torch.bfloat16, device=packed.device)
    _check("qlora_dequant_nf4", lib.qlora_dequant_nf4(
        _dev(packed, "packed", torch.uint8), _dev(absmax, "absmax", torch.float32), n_out, n_in,
        _dev(out, "out", torch.bfloat16), _stream(packed)))
    return out


def qlora_merge_nf4(packed: torch.Tensor, absmax: torch.Tensor, A: torch.Tensor, B: torch.Tensor, s: float,
                    d_out: int, d_in: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """Merged weight bf16(W_deq + s . (A . B)^T), [d_out, d_in] bf16."""
    lib = load_library()
    r = B.shape[0]
    if A.shape != (d_in, r) or B.shape != (r, d_out):
        raise ValueError(f"A must be [{d_in}, r] and B [r, {d_out}], got {tuple(A.shape)}, {tuple(B.shape)}")
    if out is None:
        out = torch.empty(d_out, d_in, dtype=torch.bfloat16, device=packed.device)
    _check("qlora_merge_nf4", lib.qlora_merge_nf4(
        _dev(packed, "packed", torch.uint8), _dev(absmax, "absmax", torch.float32), d_out, d_in,
        _dev(A, "A", torch.bfloat16), _dev(B, "B", torch.bfloat16), r, float(s),
        _dev(out, "out", torch.bfloat16), _stream(packed)))
    return out


def qlora_swiglu_fwd(gu: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """h = silu(g) * u from the stacked gate/up output gu [M, 2*d_ff] -> [M, d_ff] bf16."""
    lib = load_library()
    M, two = gu.shape
    d_ff = two // 2
    if out is None:
        out = torch.empty(M, d_ff, dtype=torch.bfloat16, device=gu.device)
    _check("qlora_swiglu_fwd", lib.qlora_swiglu_fwd(
        _dev(gu, "gu", torch.bfloat16), M, d_ff, _dev(out, "h", torch.bfloat16), _stream(gu)))
    return out


def qlora_swiglu_bwd(gu: torch.Tensor, dh: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """[d/dg | d/du] of h = silu(g) * u, in the layout of gu [M, 2*d_ff] bf16."""
    lib = load_library()
    M, two = gu.shape
    d_ff = two // 2
    if dh.shape != (M, d_ff):
        raise ValueError(f"dh must be [{M}, {d_ff}], got {tuple(dh.shape)}")
    if out is None:
        out = torch.empty(M, 2 * d_ff, dtype=torch.bfloat16, device=gu.device)
    _check("qlora_swiglu_bwd", lib.qlora_swiglu_bwd(
        _dev(gu, "gu", torch.bfloat16), _dev(dh, "dh", torch.bfloat16), M, d_ff,
        _dev(out, "dgu", torch.bfloat16), _stream(gu)))
    return out


def qlora_quantize_absmax_dq(absmax: torch.Tensor):
    """The block absmax in 8 bits: (q8 uint8 [n], scale2 fp32 [ceil(n / 256)])."""
    lib = load_library()
    n = absmax.numel()
    q8 = torch.empty(n, dtype=torch.uint8, device=absmax.device)
    scale2 = torch.empty(-(-n // 256), dtype=torch.float32, device=absmax.device)
    _check("qlora_quantize_absmax_dq", lib.qlora_quantize_absmax_dq(
        _dev(absmax, "absmax", torch.float32), n, _dev(q8, "q8", torch.uint8), _dev(scale2, "scale2", torch.float32),
        _stream(absmax)))
    return q8, scale2


def qlora_dequant_absmax_dq(q8: torch.Tensor, scale2: torch.Tensor, *, absmax: torch.Tensor | None = None):
    """The fp32 block absmax the layer calls take, from its 8-bit storage."""
    lib = load_library()
    n = q8.numel()
    if absmax is None:
        absmax = torch.empty(n, dtype=torch.float32, device=q8.device)
    _check("qlora_dequant_absmax_dq", lib.qlora_dequant_absmax_dq(
        _dev(q8, "q8", torch.uint8), _dev(scale2, "scale2", torch.float32), n, _dev(absmax, "absmax", torch.float32),
        _stream(q8)))
    return absmax


def _workspace(M, d_in, d_out, r, device, workspace):
    need = qlora_workspace_bytes(M, d_in, d_out, r)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return workspace, need


def qlora_linear_fwd(X: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor,
                     A: torch.Tensor, B: torch.Tensor, s: float, *,
                     Y: torch.Tensor | None = None, XA: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None):
    """Y = X . W_deq^T + s . (X . A) . B.  Returns (Y bf16 [M, d_out], XA fp32 [M, r])."""
    lib = load_library()
    M, d_in = X.shape
    r, d_out = B.shape
    if A.shape != (d_in, r):
        raise ValueError(f"A must be [{d_in}, {r}], got {tuple(A.shape)}")
    if Y is None:
        Y = torch.empty(M, d_out, dtype=torch.bfloat16, device=X.device)
    if XA is None:
        XA = torch.empty(M, r, dtype=torch.float32, device=X.device)
    workspace, _ = _workspace(M, d_in, d_out, r, X.device, workspace)
    _check("qlora_linear_fwd", lib.qlora_linear_fwd(
        _dev(X, "X", torch.bfloat16), M, d_in, d_out, _dev(packed, "packed", torch.uint8),
        _dev(absmax, "absmax", torch.float32), _dev(A, "A", torch.bfloat16),
        _dev(B, "B", torch.bfloat16), r, float(s), _dev(Y, "Y", torch.bfloat16),
        _dev(XA, "XA", torch.float32), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(X)))
    return Y, XA


def qlora_linear_fwd_noalloc(X: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor,
                             A: torch.Tensor, B: torch.Tensor, s: float, *,
                             Y: torch.Tensor | None = None, XA: torch.Tensor | None = None):
    """The forward without a workspace: its scratch is a fixed array inside the
    library (for callers that cannot allocate one).  Returns (Y, XA)."""
    lib = load_library()
    M, d_in = X.shape
    r, d_out = B.shape
    if A.shape != (d_in, r):
        raise ValueError(f"A must be [{d_in}, {r}], got {tuple(A.shape)}")
    if Y is None:
        Y = torch.empty(M, d_out, dtype=torch.bfloat16, device=X.device)
    if XA is None:
        XA = torch.empty(M, r, dtype=torch.float32, device=X.device)
    _check("qlora_linear_fwd_noalloc", lib.qlora_linear_fwd_noalloc(
        _dev(X, "X", torch.bfloat16), M, d_in, d_out, _dev(packed, "packed", torch.uint8),
        _dev(absmax, "absmax", torch.float32), _dev(A, "A", torch.bfloat16),
        _dev(B, "B", torch.bfloat16), r, float(s), _dev(Y, "Y", torch.bfloat16),
        _dev(XA, "XA", torch.float32), _stream(X)))
    return Y, XA


def qlora_linear_bwd(X: torch.Tensor, dY: torch.Tensor, packed: torch.Tensor,
                     absmax: torch.Tensor, A: torch.Tensor, B: torch.Tensor, s: float,
                     XA: torch.Tensor, *, need_dX: bool = True,
                     dX: torch.Tensor | None = None, dA: torch.Tensor | None = None,
                     dB: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Hand-written backward.  Returns (dX bf16 [M, d_in] or None, dA fp32 [d_in, r], dB fp32 [r, d_out])."""
    lib = load_library()
    M, d_in = X.shape
    r, d_out = B.shape
    if dY.shape != (M, d_out):
        raise ValueError(f"dY must be [{M}, {d_out}], got {tuple(dY.shape)}")
    if need_dX and dX is None:
        dX = torch.empty(M, d_in, dtype=torch.bfloat16, device=X.device)
    if dA is None:
        dA = torch.empty(d_in, r, dtype=torch.float32, device=X.device)
    if dB is None:
        dB = torch.empty(r, d_out, dtype=torch.float32, device=X.device)
    workspace, _ = _workspace(M, d_in, d_out, r, X.device, workspace)
    dx_ptr = _dev(dX, "dX", torch.bfloat16) if dX is not None else None
    _check("qlora_linear_bwd", lib.qlora_linear_bwd(
        _dev(X, "X", torch.bfloat16), _dev(dY, "dY", torch.bfloat16), M, d_in, d_out,
        _dev(packed, "packed", torch.uint8), _dev(absmax, "absmax", torch.float32),
        _dev(A, "A", torch.bfloat16), _dev(B, "B", torch.bfloat16), r, float(s),
        _dev(XA, "XA", torch.float32), dx_ptr, _dev(dA, "dA", torch.float32),
        _dev(dB, "dB", torch.float32), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(X)))
    return dX, dA, dB


def _group_array(group_d_out):
    arr = (_i64 * len(group_d_out))(*[int(n) for n in group_d_out])
    return arr, sum(int(n) for n in group_d_out)


def qlora_linear_fwd_grouped(X: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor, A: torch.Tensor,
                             B: torch.Tensor, s: float, group_d_out, group_rank: int, *,
                             Y: torch.Tensor | None = None, XA: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None):
    """Stacked projections with block-diagonal low-rank blocks (group g: output
    features of group_d_out[g], rank columns [g*group_rank, (g+1)*group_rank)).
    Returns (Y bf16 [M, d_out], XA fp32 [M, r])."""
    lib = load_library()
    M, d_in = X.shape
    groups, d_out = _group_array(group_d_out)
    r = len(group_d_out) * int(group_rank)
    if A.shape != (d_in, r) or B.shape != (r, d_out):
        raise ValueError(f"A must be [{d_in}, {r}] and B [{r}, {d_out}]")
    if Y is None:
        Y = torch.empty(M, d_out, dtype=torch.bfloat16, device=X.device)
    if XA is None:
        XA = torch.empty(M, r, dtype=torch.float32, device=X.device)
    workspace, _ = _workspace(M, d_in, d_out, r, X.device, workspace)
    _check("qlora_linear_fwd_grouped", lib.qlora_linear_fwd_grouped(
        _dev(X, "X", torch.bfloat16), M, d_in, len(group_d_out), groups, int(group_rank),
        _dev(packed, "packed", torch.uint8), _dev(absmax, "absmax", torch.float32), _dev(A, "A", torch.bfloat16),
        _dev(B, "B", torch.bfloat16), float(s), _dev(Y, "Y", torch.bfloat16), _dev(XA, "XA", torch.float32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(X)))
    return Y, XA


def qlora_linear_bwd_grouped(X: torch.Tensor, dY: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor,
                             A: torch.Tensor, B: torch.Tensor, s: float, XA: torch.Tensor, group_d_out,
                             group_rank: int, *, need_dX: bool = True, workspace: torch.Tensor | None = None):
    """Backward of qlora_linear_fwd_grouped.  Returns (dX or None, dA [d_in, r],
    dB [r, d_out]); dB holds the diagonal blocks (zeros elsewhere)."""
    lib = load_library()
    M, d_in = X.shape
    groups, d_out = _group_array(group_d_out)
    r = len(group_d_out) * int(group_rank)
    if dY.shape != (M, d_out):
        raise ValueError(f"dY must be [{M}, {d_out}], got {tuple(dY.shape)}")
    dX = torch.empty(M, d_in, dtype=torch.bfloat16, device=X.device) if need_dX else None
    dA = torch.empty(d_in, r, dtype=torch.float32, device=X.device)
    dB = torch.zeros(r, d_out, dtype=torch.float32, device=X.device)
    workspace, _ = _workspace(M, d_in, d_out, r, X.device, workspace)
    dx_ptr = _dev(dX, "dX", torch.bfloat16) if dX is not None else None
    _check("qlora_linear_bwd_grouped", lib.qlora_linear_bwd_grouped(
        _dev(X, "X", torch.bfloat16), _dev(dY, "dY", torch.bfloat16), M, d_in, len(group_d_out), groups,
        int(group_rank), _dev(packed, "packed", torch.uint8), _dev(absmax, "absmax", torch.float32),
        _dev(A, "A", torch.bfloat16), _dev(B, "B", torch.bfloat16), float(s), _dev(XA, "XA", torch.float32),
        dx_ptr, _dev(dA, "dA", torch.float32), _dev(dB, "dB", torch.float32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(X)))
    return dX, dA, dB


def qlora_linear_fwd_swiglu(X: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor, A: torch.Tensor,
                            B: torch.Tensor, s: float, *, gu: torch.Tensor | None = None,
                            h: torch.Tensor | None = None, XA: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None):
    """The interleaved gate/up layer with the SwiGLU gate in its epilogue.
    Returns (gu [M, 2*d_ff], h [M, d_ff], XA [M, r])."""
    lib = load_library()
    M, d_in = X.shape
    r, two_ff = B.shape
    d_ff = two_ff // 2
    if A.shape != (d_in, r):
        raise ValueError(f"A must be [{d_in}, {r}], got {tuple(A.shape)}")
    if gu is None:
        gu = torch.empty(M, two_ff, dtype=torch.bfloat16, device=X.device)
    if h is None:
        h = torch.empty(M, d_ff, dtype=torch.bfloat16, device=X.device)
    if XA is None:
        XA = torch.empty(M, r, dtype=torch.float32, device=X.device)
    workspace, _ = _workspace(M, d_in, two_ff, r, X.device, workspace)
    _check("qlora_linear_fwd_swiglu", lib.qlora_linear_fwd_swiglu(
        _dev(X, "X", torch.bfloat16), M, d_in, d_ff, _dev(packed, "packed", torch.uint8),
        _dev(absmax, "absmax", torch.float32), _dev(A, "A", torch.bfloat16), _dev(B, "B", torch.bfloat16), r,
        float(s), _dev(gu, "gu", torch.bfloat16), _dev(h, "h", torch.bfloat16), _dev(XA, "XA", torch.float32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(X)))
    return gu, h, XA


def qlora_linear_bwd_swiglu(h: torch.Tensor, dY: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor,
                            A: torch.Tensor, B: torch.Tensor, s: float, XA: torch.Tensor, gu: torch.Tensor, *,
                            dgu: torch.Tensor | None = None, dA: torch.Tensor | None = None,
                            dB: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """The down layer's backward with the gate's backward in its epilogue.
    Returns (dgu [M, 2*d_ff] interleaved like gu, dA, dB)."""
    lib = load_library()
    M, d_ff = h.shape
    r, d_out = B.shape
    if dY.shape != (M, d_out) or gu.shape != (M, 2 * d_ff):
        raise ValueError("dY must be [M, d_out] and gu [M, 2*d_ff]")
    if dgu is None:
        dgu = torch.empty(M, 2 * d_ff, dtype=torch.bfloat16, device=h.device)
    if dA is None:
        dA = torch.empty(d_ff, r, dtype=torch.float32, device=h.device)
    if dB is None:
        dB = torch.empty(r, d_out, dtype=torch.float32, device=h.device)
    workspace, _ = _workspace(M, d_ff, d_out, r, h.device, workspace)
    _check("qlora_linear_bwd_swiglu", lib.qlora_linear_bwd_swiglu(
        _dev(h, "h", torch.bfloat16), _dev(dY, "dY", torch.bfloat16), M, d_ff, d_out,
        _dev(packed, "packed", torch.uint8), _dev(absmax, "absmax", torch.float32), _dev(A, "A", torch.bfloat16),
        _dev(B, "B", torch.bfloat16), r, float(s), _dev(XA, "XA", torch.float32), _dev(gu, "gu", torch.bfloat16),
        _dev(dgu, "dgu", torch.bfloat16), _dev(dA, "dA", torch.float32), _dev(dB, "dB", torch.float32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(h)))
    return dgu, dA, dB


def qlora_swiglu_mlp_workspace_bytes(M: int, d_model: int, d_ff: int, r_gu: int, r_d: int) -> int:
    return int(load_library().qlora_swiglu_mlp_workspace_bytes(M, d_model, d_ff, r_gu, r_d))


def qlora_swiglu_mlp_fwd(X, gu_layer, d_layer, s_gu: float, s_d: float, *, workspace=None):
    """The fused SwiGLU block forward; gu_layer / d_layer are (packed, absmax, A, B).
    Returns (Y, saved) with saved = (gu, h, T_gu, T_d)."""
    lib = load_library()
    M, d_model = X.shape
    pg, ag, Ag, Bg = gu_layer
    pd, ad, Ad, Bd = d_layer
    r_gu, r_d = Bg.shape[0], Bd.shape[0]
    d_ff = Bg.shape[1] // 2
    dev = X.device
    Y = torch.empty(M, d_model, dtype=torch.bfloat16, device=dev)
    gu = torch.empty(M, 2 * d_ff, dtype=torch.bfloat16, device=dev)
    h = torch.empty(M, d_ff, dtype=torch.bfloat16, device=dev)
    T_gu = torch.empty(M, r_gu, dtype=torch.float32, device=dev)
    T_d = torch.empty(M, r_d, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, qlora_swiglu_mlp_workspace_bytes(M, d_model, d_ff, r_gu, r_d)),
                                dtype=torch.uint8, device=dev)
    _check("qlora_swiglu_mlp_fwd", lib.qlora_swiglu_mlp_fwd(
        _dev(X, "X", torch.bfloat16), M, d_model, d_ff,
        _dev(pg, "gu_packed", torch.uint8), _dev(ag, "gu_absmax", torch.float32), _dev(Ag, "A_gu", torch.bfloat16),
        _dev(Bg, "B_gu", torch.bfloat16), r_gu, float(s_gu),
        _dev(pd, "d_packed", torch.uint8), _dev(ad, "d_absmax", torch.float32), _dev(Ad, "A_d", torch.bfloat16),
        _dev(Bd, "B_d", torch.bfloat16), r_d, float(s_d),
        _dev(Y, "Y", torch.bfloat16), _dev(gu, "gu", torch.bfloat16), _dev(h, "h", torch.bfloat16),
        _dev(T_gu, "T_gu", torch.float32), _dev(T_d, "T_d", torch.float32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(X)))
    return Y, (gu, h, T_gu, T_d)


def qlora_swiglu_mlp_bwd(X, dY, saved, gu_layer, d_layer, s_gu: float, s_d: float, *, need_dX: bool = True,
                         workspace=None):
    """The fused SwiGLU block backward.  Returns dX, (dA_gu, dB_gu), (dA_d, dB_d)."""
    lib = load_library()
    M, d_model = X.shape
    gu, h, T_gu, T_d = saved
    pg, ag, Ag, Bg = gu_layer
    pd, ad, Ad, Bd = d_layer
    r_gu, r_d = Bg.shape[0], Bd.shape[0]
    d_ff = Bg.shape[1] // 2
    dev = X.device
    dgu = torch.empty(M, 2 * d_ff, dtype=torch.bfloat16, device=dev)
    dX = torch.empty(M, d_model, dtype=torch.bfloat16, device=dev) if need_dX else None
    dA_gu = torch.empty(d_model, r_gu, dtype=torch.float32, device=dev)
    dB_gu = torch.empty(r_gu, 2 * d_ff, dtype=torch.float32, device=dev)
    dA_d = torch.empty(d_ff, r_d, dtype=torch.float32, device=dev)
    dB_d = torch.empty(r_d, d_model, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, qlora_swiglu_mlp_workspace_bytes(M, d_model, d_ff, r_gu, r_d)),
                                dtype=torch.uint8, device=dev)
    _check("qlora_swiglu_mlp_bwd", lib.qlora_swiglu_mlp_bwd(
        _dev(X, "X", torch.bfloat16), _dev(dY, "dY", torch.bfloat16), M, d_model, d_ff,
        _dev(pg, "gu_packed", torch.uint8), _dev(ag, "gu_absmax", torch.float32), _dev(Ag, "A_gu", torch.bfloat16),
        _dev(Bg, "B_gu", torch.bfloat16), r_gu, float(s_gu),
        _dev(pd, "d_packed", torch.uint8), _dev(ad, "d_absmax", torch.float32), _dev(Ad, "A_d", torch.bfloat16),
        _dev(Bd, "B_d", torch.bfloat16), r_d, float(s_d),
        _dev(gu, "gu", torch.bfloat16), _dev(h, "h", torch.bfloat16), _dev(T_gu, "T_gu", torch.float32),
        _dev(T_d, "T_d", torch.float32), _dev(dgu, "dgu", torch.bfloat16),
        _dev(dX, "dX", torch.bfloat16) if dX is not None else None, _dev(dA_gu, "dA_gu", torch.float32),
        _dev(dB_gu, "dB_gu", torch.float32), _dev(dA_d, "dA_d", torch.float32), _dev(dB_d, "dB_d", torch.float32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(X)))
    return dX, (dA_gu, dB_gu), (dA_d, dB_d)
