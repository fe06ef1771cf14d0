"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import qlora_oracle as O

# Acceptance bound for floating-point outputs: per output tensor,
# max|gpu - oracle| <= TOL * max|oracle|  (bf16 inputs, fp32 accumulation).
TOL = 1e-2


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").float().numpy()


def rel_max_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    gpu = np.asarray(gpu, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    if scale == 0.0:
        return 0.0 if err == 0.0 else float("inf")
    return err / scale


def assert_close(name: str, gpu, ref, tol: float = TOL):
    e = rel_max_err(gpu, ref)
    assert e <= tol, f"{name}: max|gpu-oracle| / max|oracle| = {e:.3e} > {tol:.0e}"
    return e


def run_gpu(inp: dict, s: float, bwd: bool = True, need_dX: bool = True):
    """Quantise W, run forward (and backward) on cuda:0; returns CPU tensors."""
    from rank_adapter_linear_nf4_b300 import qlora
    dev = torch.device("cuda", 0)
    X, dY, W, A, B = (inp[k].to(dev) for k in ("X", "dY", "W", "A", "B"))
    packed, absmax = qlora.qlora_quantize_nf4(W)
    Y, XA = qlora.qlora_linear_fwd(X, packed, absmax, A, B, s)
    out = {"packed": packed, "absmax": absmax, "Y": Y, "XA": XA}
    if bwd:
        dX, dA, dB = qlora.qlora_linear_bwd(X, dY, packed, absmax, A, B, s, XA, need_dX=need_dX)
        out.update(dX=dX, dA=dA, dB=dB)
    torch.cuda.synchronize()
    assert qlora.qlora_device_status(clear=True) == 0
    return {k: (v.cpu() if v is not None else None) for k, v in out.items()}


def oracle_weight(W: torch.Tensor):
    Wn = np32(W)
    packed, absmax = O.quantize_nf4(Wn)
    Wd = O.dequantize_nf4(packed, absmax, Wn.shape[0], Wn.shape[1])
    return packed, absmax, Wd


def check_layer(inp: dict, s: float, rows=None, bwd: bool = True, need_dX: bool = True,
                tol: float = TOL) -> dict:
    """Runs both sides and asserts parity; returns the achieved relative errors."""
    g = run_gpu(inp, s, bwd=bwd, need_dX=need_dX)
    packed, absmax, Wd = oracle_weight(inp["W"])
    assert np.array_equal(g["packed"].numpy(), packed), "NF4 codes differ"
    assert np.array_equal(g["absmax"].numpy().view(np.uint32), absmax.view(np.uint32)), "absmax differs"
    X, dY, A, B = (np32(inp[k]) for k in ("X", "dY", "A", "B"))
    errs = {}
    Y_ref, T_ref = O.lora_forward(X, Wd, A, B, s, rows=rows)
    sel = slice(None) if rows is None else rows
    errs["Y"] = assert_close("Y", np32(g["Y"])[sel], Y_ref, tol)
    errs["XA"] = assert_close("XA", g["XA"].numpy()[sel], T_ref, tol)
    if bwd:
        dX_ref, dA_ref, dB_ref = O.lora_backward(X, dY, Wd, A, B, s, dx_rows=rows)
        if need_dX:
            errs["dX"] = assert_close("dX", np32(g["dX"])[sel], dX_ref, tol)
        errs["dA"] = assert_close("dA", g["dA"].numpy(), dA_ref, tol)
        errs["dB"] = assert_close("dB", g["dB"].numpy(), dB_ref, tol)
    return errs
