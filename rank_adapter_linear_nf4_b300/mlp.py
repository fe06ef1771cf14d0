"""The SwiGLU MLP block of two LoRA-adapted NF4 layers, as library calls:

    gu = gate_up(X)            one stacked layer of the gate and up projections
    h  = silu(gate) * up
    Y  = down(h)

and the backward in reverse.  The pages fuse the MLP into their forward
("Unsloth性能实测：比传统方法快2倍真的吗？", section 2.2).

Two forms, the same arithmetic (gu, h, dh and dgu rounded to bf16 at the same
points):

* fused (``swiglu_mlp_fwd`` / ``swiglu_mlp_bwd``): the gate/up layer's rows are
  interleaved in 64-row chunks ([gate 0..63 | up 0..63 | gate 64..127 | ...]),
  so its epilogue computes h beside gu, and the down layer's backward epilogue
  turns dh into dgu without storing dh: one call each way
  (qlora_swiglu_mlp_fwd / _bwd), no separate gate pass;
* unfused (``swiglu_mlp_fwd_unfused`` / ``_bwd_unfused``): stacked [gate | up]
  layer, qlora_swiglu_fwd / _bwd between the layers.

Every step runs in the library's kernels; this module only arranges memory
(the interleaved packing, one-time) and sequences calls.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import qlora

CHUNK = 64   # rows of the gate/up interleave


@dataclass
class Layer:
    """One NF4 LoRA layer: codes, absmax (qlora_quantize_nf4), A [d_in, r], B [r, d_out]."""
    packed: torch.Tensor
    absmax: torch.Tensor
    A: torch.Tensor
    B: torch.Tensor

    def args(self):
        return self.packed, self.absmax, self.A, self.B


# ---------------------------------------------------------------- interleaved layout

def gate_up_order(d_ff: int) -> torch.Tensor:
    """Row (or column) order of the interleaved gate/up layer: position i of the
    interleaved layout holds row order[i] of the [gate | up] stacking."""
    if d_ff % CHUNK != 0:
        raise ValueError(f"d_ff must be a multiple of {CHUNK}")
    c = torch.arange(d_ff // CHUNK).repeat_interleave(CHUNK) * CHUNK
    j = torch.arange(d_ff) % CHUNK
    out = torch.empty(2 * d_ff, dtype=torch.long)
    pos = (c * 2) + j
    out[pos] = torch.arange(d_ff)              # gate features
    out[pos + CHUNK] = torch.arange(d_ff) + d_ff   # up features
    return out


def interleave_weights(W_gate: torch.Tensor, W_up: torch.Tensor) -> torch.Tensor:
    """[2*d_ff, d_in] bf16: the interleaved gate/up weight, to quantise once."""
    order = gate_up_order(W_gate.shape[0]).to(W_gate.device)
    return torch.cat([W_gate, W_up], dim=0)[order].contiguous()


def interleave_adapters(A_gate, B_gate, A_up, B_up):
    """A_cat = [A_gate | A_up] [d_in, r_g + r_u] and B_cat [r_g + r_u, 2*d_ff] with
    B_gate in the gate columns of its rows, B_up in the up columns of its rows."""
    d_ff = B_gate.shape[1]
    A_cat = torch.cat([A_gate, A_up], dim=1).contiguous()
    rg, ru = B_gate.shape[0], B_up.shape[0]
    B_stack = torch.zeros(rg + ru, 2 * d_ff, dtype=B_gate.dtype, device=B_gate.device)
    B_stack[:rg, :d_ff] = B_gate
    B_stack[rg:, d_ff:] = B_up
    order = gate_up_order(d_ff).to(B_gate.device)
    return A_cat, B_stack[:, order].contiguous()


def deinterleave(gu: torch.Tensor) -> torch.Tensor:
    """[..., 2*d_ff] interleaved -> [..., 2*d_ff] as [gate | up]."""
    d_ff = gu.shape[-1] // 2
    order = gate_up_order(d_ff).to(gu.device)
    out = torch.empty_like(gu)
    out[..., order] = gu
    return out


def split_adapter_grads(dA_cat, dB_cat, r_gate: int):
    """(dA_gate, dB_gate), (dA_up, dB_up) from the interleaved layer's gradients."""
    d_ff = dB_cat.shape[1] // 2
    dB = deinterleave(dB_cat)
    return ((dA_cat[:, :r_gate], dB[:r_gate, :d_ff]), (dA_cat[:, r_gate:], dB[r_gate:, d_ff:]))


# ---------------------------------------------------------------- fused block

def swiglu_mlp_fwd(X: torch.Tensor, gate_up: Layer, down: Layer, s_gu: float, s_d: float | None = None):
    """Y [M, d_model] and the saved tensors (gu, h, T_gu, T_d); gate_up interleaved."""
    return qlora.qlora_swiglu_mlp_fwd(X, gate_up.args(), down.args(), s_gu, s_gu if s_d is None else s_d)


def swiglu_mlp_bwd(X: torch.Tensor, dY: torch.Tensor, saved, gate_up: Layer, down: Layer, s_gu: float,
                   s_d: float | None = None):
    """dX and the adapters' gradients ((dA_gu, dB_gu), (dA_d, dB_d)); dB_gu interleaved."""
    return qlora.qlora_swiglu_mlp_bwd(X, dY, saved, gate_up.args(), down.args(), s_gu, s_gu if s_d is None else s_d)


# ---------------------------------------------------------------- unfused block

def swiglu_mlp_fwd_unfused(X: torch.Tensor, gate_up: Layer, down: Layer, s: float):
    """Y [M, d_model] and the saved tensors (gu, T_gu, h, T_d); gate_up stacked [gate | up]."""
    gu, T_gu = qlora.qlora_linear_fwd(X, gate_up.packed, gate_up.absmax, gate_up.A, gate_up.B, s)
    h = qlora.qlora_swiglu_fwd(gu)
    Y, T_d = qlora.qlora_linear_fwd(h, down.packed, down.absmax, down.A, down.B, s)
    return Y, (gu, T_gu, h, T_d)


def swiglu_mlp_bwd_unfused(X: torch.Tensor, dY: torch.Tensor, saved, gate_up: Layer, down: Layer, s: float):
    """dX and the adapters' gradients ((dA_gu, dB_gu), (dA_d, dB_d))."""
    gu, T_gu, h, T_d = saved
    dh, dA_d, dB_d = qlora.qlora_linear_bwd(h, dY, down.packed, down.absmax, down.A, down.B, s, T_d)
    dgu = qlora.qlora_swiglu_bwd(gu, dh)
    dX, dA_gu, dB_gu = qlora.qlora_linear_bwd(X, dgu, gate_up.packed, gate_up.absmax, gate_up.A, gate_up.B, s,
                                              T_gu)
    return dX, (dA_gu, dB_gu), (dA_d, dB_d)
