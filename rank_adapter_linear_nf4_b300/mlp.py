"""The SwiGLU MLP block of two LoRA-adapted NF4 layers, as library calls:

    gu = gate_up(X)            one stacked layer, output columns [gate | up]
    h  = silu(gate) * up       qlora_swiglu_fwd
    Y  = down(h)

and the backward in reverse (down's backward gives dh, qlora_swiglu_bwd turns
it into the stacked layer's dY, whose backward gives dX).  The pages fuse the
MLP into their forward ("Unsloth性能实测：比传统方法快2倍真的吗？", section 2.2).
Every step runs in the library's kernels; this module only sequences the calls
and keeps the activations the backward needs (gu, h and the two saved T).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import qlora


@dataclass
class Layer:
    """One NF4 LoRA layer: codes, absmax (qlora_quantize_nf4), A [d_in, r], B [r, d_out]."""
    packed: torch.Tensor
    absmax: torch.Tensor
    A: torch.Tensor
    B: torch.Tensor


def swiglu_mlp_fwd(X: torch.Tensor, gate_up: Layer, down: Layer, s: float):
    """Y [M, d_model] and the saved tensors (gu, T_gu, h, T_d)."""
    gu, T_gu = qlora.qlora_linear_fwd(X, gate_up.packed, gate_up.absmax, gate_up.A, gate_up.B, s)
    h = qlora.qlora_swiglu_fwd(gu)
    Y, T_d = qlora.qlora_linear_fwd(h, down.packed, down.absmax, down.A, down.B, s)
    return Y, (gu, T_gu, h, T_d)


def swiglu_mlp_bwd(X: torch.Tensor, dY: torch.Tensor, saved, gate_up: Layer, down: Layer, s: float):
    """dX and the adapters' gradients ((dA_gu, dB_gu), (dA_d, dB_d))."""
    gu, T_gu, h, T_d = saved
    dh, dA_d, dB_d = qlora.qlora_linear_bwd(h, dY, down.packed, down.absmax, down.A, down.B, s, T_d)
    dgu = qlora.qlora_swiglu_bwd(gu, dh)
    dX, dA_gu, dB_gu = qlora.qlora_linear_bwd(X, dgu, gate_up.packed, gate_up.absmax, gate_up.A, gate_up.B, s,
                                              T_gu)
    return dX, (dA_gu, dB_gu), (dA_d, dB_d)
