"""Several LoRA-adapted NF4 projections of the same input as one layer call.

The pages apply the adapter to several projections of one activation: q/k/v/o
and gate/up/down as `target_modules` ("UnSloth加速原理：CUDA内核融合与内存优化",
section 内核融合).  Projections that read the same X and share the scale s are
one wider layer:

* the frozen weights stack along d_out.  NF4 blocks are 64 consecutive
  elements of a row (d_in % 64 == 0), so quantising the stacked weight gives
  the stacked codes and absmax of the separate weights, bit for bit;
* the A matrices stack along the rank, A_cat = [A_1 | A_2 | ...] (d_in x sum r);
* B becomes block-diagonal, B_cat = diag(B_1, B_2, ...) (sum r x sum d_out).

Then one forward computes [Y_1 | Y_2 | ...] with a single read of X and a
single T = X.A_cat, and one backward gives dX = sum_i dX_i (what the separate
layers' input gradients add up to), dA_cat = [dA_1 | dA_2 | ...], and the
diagonal blocks of dB_cat are the dB_i (the off-diagonal blocks are the
gradients of the structural zeros and are ignored).  sum r must stay within
the layer's rank limit (128).

This module only arranges memory (one-time packing, views into the outputs);
every step of the layer runs in the library's kernels through `qlora`.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import qlora

MAX_RANK = 128


@dataclass(frozen=True)
class Packing:
    """Row / rank offsets of the projections inside the stacked layer."""
    d_outs: tuple[int, ...]
    ranks: tuple[int, ...]

    @property
    def d_out(self) -> int:
        return sum(self.d_outs)

    @property
    def r(self) -> int:
        return sum(self.ranks)

    def out_slices(self) -> list[slice]:
        o, out = 0, []
        for n in self.d_outs:
            out.append(slice(o, o + n))
            o += n
        return out

    def rank_slices(self) -> list[slice]:
        o, out = 0, []
        for r in self.ranks:
            out.append(slice(o, o + r))
            o += r
        return out


def packing(Ws, As) -> Packing:
    """Offsets for weights W_i [d_out_i, d_in] and adapters A_i [d_in, r_i]."""
    if not Ws or len(Ws) != len(As):
        raise ValueError("one A per weight, at least one projection")
    d_in = Ws[0].shape[1]
    for W, A in zip(Ws, As):
        if W.shape[1] != d_in or A.shape[0] != d_in:
            raise ValueError("every projection reads the same d_in")
    p = Packing(tuple(int(W.shape[0]) for W in Ws), tuple(int(A.shape[1]) for A in As))
    if p.r > MAX_RANK:
        raise ValueError(f"sum of ranks {p.r} exceeds {MAX_RANK}")
    return p


def stack_weights(Ws) -> torch.Tensor:
    """[sum d_out, d_in]: the frozen weights, to quantise once with qlora_quantize_nf4."""
    return torch.cat(list(Ws), dim=0).contiguous()


def stack_adapters(As, Bs) -> tuple[torch.Tensor, torch.Tensor]:
    """A_cat [d_in, sum r] and the block-diagonal B_cat [sum r, sum d_out]."""
    A_cat = torch.cat(list(As), dim=1).contiguous()
    r_tot = A_cat.shape[1]
    n_tot = sum(B.shape[1] for B in Bs)
    B_cat = torch.zeros(r_tot, n_tot, dtype=Bs[0].dtype, device=Bs[0].device)
    r0 = n0 = 0
    for B in Bs:
        B_cat[r0:r0 + B.shape[0], n0:n0 + B.shape[1]] = B
        r0 += B.shape[0]
        n0 += B.shape[1]
    return A_cat, B_cat


def split_outputs(Y_cat: torch.Tensor, p: Packing) -> list[torch.Tensor]:
    """Views Y_i [M, d_out_i] into the stacked output (or dY_i into a stacked dY buffer)."""
    return [Y_cat[:, sl] for sl in p.out_slices()]


def split_grads(dA_cat: torch.Tensor, dB_cat: torch.Tensor, p: Packing):
    """Views dA_i [d_in, r_i] and dB_i [r_i, d_out_i] (the diagonal blocks)."""
    dA = [dA_cat[:, rs] for rs in p.rank_slices()]
    dB = [dB_cat[rs, os] for rs, os in zip(p.rank_slices(), p.out_slices())]
    return dA, dB


def multi_linear_fwd(X, packed_cat, absmax_cat, A_cat, B_cat, s, p: Packing):
    """All projections of X in one layer call: (views Y_i, stacked Y, saved T)."""
    Y_cat, T = qlora.qlora_linear_fwd(X, packed_cat, absmax_cat, A_cat, B_cat, s)
    return split_outputs(Y_cat, p), Y_cat, T


def multi_linear_bwd(X, dY_cat, packed_cat, absmax_cat, A_cat, B_cat, s, T, p: Packing):
    """dX (summed over the projections), and the views dA_i, dB_i."""
    dX, dA_cat, dB_cat = qlora.qlora_linear_bwd(X, dY_cat, packed_cat, absmax_cat, A_cat, B_cat, s, T)
    dA, dB = split_grads(dA_cat, dB_cat, p)
    return dX, dA, dB
