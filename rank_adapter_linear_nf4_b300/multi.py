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
the layer's rank limit (256).

Two layouts of the low-rank part:

* dense: A_cat columns and B_cat rows packed end to end (sum r); the layer
  treats B_cat as one dense matrix, so every output tile's low-rank stages and
  dB run over all sum r ranks;
* grouped: every projection's ranks padded to one width (a multiple of 64) and
  placed at i * width; the layer (qlora_linear_fwd_grouped / _bwd_grouped)
  then adds to each output tile only its own projection's block and computes
  only the diagonal blocks of dB.  Needs at most 8 projections, every d_out
  but the last a multiple of 128 and n * width <= 256.

`packing` takes the grouped layout when it is possible and needs no more
low-rank columns than the dense one (equal ranks that are multiples of 64, such
as q/k/v or gate/up at rank 64), else the dense one.

This module only arranges memory (one-time packing, views into the outputs);
every step of the layer runs in the library's kernels through `qlora`.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import qlora

MAX_RANK = 256


MAX_GROUPS = 8


def _padded_rank(r: int) -> int:
    """The layer's padded rank width (64, 128 or 256 columns)."""
    return 64 if r <= 64 else 128 if r <= 128 else 256


@dataclass(frozen=True)
class Packing:
    """Row / rank offsets of the projections inside the stacked layer.
    group_rank > 0: the grouped layout (each projection's ranks at i * group_rank)."""
    d_outs: tuple[int, ...]
    ranks: tuple[int, ...]
    group_rank: int = 0

    @property
    def d_out(self) -> int:
        return sum(self.d_outs)

    @property
    def r(self) -> int:
        """Columns of A_cat (rows of B_cat)."""
        return len(self.ranks) * self.group_rank if self.group_rank else sum(self.ranks)

    @property
    def grouped(self) -> bool:
        return self.group_rank > 0

    def out_slices(self) -> list[slice]:
        o, out = 0, []
        for n in self.d_outs:
            out.append(slice(o, o + n))
            o += n
        return out

    def rank_slices(self) -> list[slice]:
        if self.grouped:
            return [slice(i * self.group_rank, i * self.group_rank + r) for i, r in enumerate(self.ranks)]
        o, out = 0, []
        for r in self.ranks:
            out.append(slice(o, o + r))
            o += r
        return out


def packing(Ws, As, grouped: bool | None = None) -> Packing:
    """Offsets for weights W_i [d_out_i, d_in] and adapters A_i [d_in, r_i].
    grouped: None picks the layout (see the module notes), True / False forces it."""
    if not Ws or len(Ws) != len(As):
        raise ValueError("one A per weight, at least one projection")
    d_in = Ws[0].shape[1]
    for W, A in zip(Ws, As):
        if W.shape[1] != d_in or A.shape[0] != d_in:
            raise ValueError("every projection reads the same d_in")
    d_outs = tuple(int(W.shape[0]) for W in Ws)
    ranks = tuple(int(A.shape[1]) for A in As)
    width = 64 * -(-max(ranks) // 64)
    can_group = (len(ranks) <= MAX_GROUPS and len(ranks) * width <= MAX_RANK
                 and all(n % 128 == 0 for n in d_outs[:-1]))
    if grouped is None:
        grouped = can_group and _padded_rank(len(ranks) * width) <= _padded_rank(sum(ranks))
    elif grouped and not can_group:
        raise ValueError("the grouped layout needs <= 8 projections, d_out % 128 == 0 but for the last, "
                         f"and n * width <= {MAX_RANK}")
    p = Packing(d_outs, ranks, width if grouped else 0)
    if p.r > MAX_RANK:
        raise ValueError(f"sum of ranks {p.r} exceeds {MAX_RANK}")
    return p


def stack_weights(Ws) -> torch.Tensor:
    """[sum d_out, d_in]: the frozen weights, to quantise once with qlora_quantize_nf4."""
    return torch.cat(list(Ws), dim=0).contiguous()


def stack_adapters(As, Bs, p: Packing | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """A_cat [d_in, p.r] and the block-diagonal B_cat [p.r, sum d_out], in the
    layout of p (dense when p is None), zero outside the projections' blocks."""
    d_in = As[0].shape[0]
    n_tot = sum(B.shape[1] for B in Bs)
    if p is None:
        p = Packing(tuple(int(B.shape[1]) for B in Bs), tuple(int(A.shape[1]) for A in As))
    A_cat = torch.zeros(d_in, p.r, dtype=As[0].dtype, device=As[0].device)
    B_cat = torch.zeros(p.r, n_tot, dtype=Bs[0].dtype, device=Bs[0].device)
    for A, B, rs, os in zip(As, Bs, p.rank_slices(), p.out_slices()):
        A_cat[:, rs] = A
        B_cat[rs, os] = B
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
    if p.grouped:
        Y_cat, T = qlora.qlora_linear_fwd_grouped(X, packed_cat, absmax_cat, A_cat, B_cat, s, p.d_outs,
                                                  p.group_rank)
    else:
        Y_cat, T = qlora.qlora_linear_fwd(X, packed_cat, absmax_cat, A_cat, B_cat, s)
    return split_outputs(Y_cat, p), Y_cat, T


def multi_linear_bwd(X, dY_cat, packed_cat, absmax_cat, A_cat, B_cat, s, T, p: Packing):
    """dX (summed over the projections), and the views dA_i, dB_i."""
    if p.grouped:
        dX, dA_cat, dB_cat = qlora.qlora_linear_bwd_grouped(X, dY_cat, packed_cat, absmax_cat, A_cat, B_cat, s, T,
                                                            p.d_outs, p.group_rank)
    else:
        dX, dA_cat, dB_cat = qlora.qlora_linear_bwd(X, dY_cat, packed_cat, absmax_cat, A_cat, B_cat, s, T)
    dA, dB = split_grads(dA_cat, dB_cat, p)
    return dX, dA, dB
