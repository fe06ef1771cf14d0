"""Seeded synthetic inputs for the NF4-QLoRA linear layer.

This module draws random numbers and rounds them to bf16; it holds none of the
layer's arithmetic.  The CUDA path, the oracle and the benchmark all take their
inputs from here, so both sides of every comparison see identical bytes.

Recipe (the pages fine-tune on SFT datasets that are not available here; these
shapes and distributions stand in for them):
  * X and dY ~ N(0, 1), drawn in fp32, rounded to bf16;
  * base weight W [d_out, d_in] ~ N(0, 0.02^2) (0.02 is the standard
    deviation), drawn in fp32, rounded to bf16, then NF4-quantised by the
    library under test;
  * A [d_in, r] ~ U(-1/sqrt(d_in), 1/sqrt(d_in)), B [r, d_out] ~ N(0, 0.01^2),
    both rounded to bf16.
Seeds: ``seed`` drives X and dY, ``seed + 1`` drives W, A and B.
"""
from __future__ import annotations

from dataclasses import dataclass
import math

import numpy as np
import torch


@dataclass(frozen=True)
class LayerShape:
    """One projection workload: M tokens, d_in -> d_out, rank r, LoRA alpha."""
    name: str
    M: int
    d_in: int
    d_out: int
    r: int
    alpha: float
    rank_stabilised: bool = False

    @property
    def s(self) -> float:
        d = math.sqrt(self.r) if self.rank_stabilised else float(self.r)
        return float(self.alpha) / d


# Transformer projection shapes used for parity cases and the benchmark.
SHAPES = {
    "tiny": LayerShape("tiny", 64, 256, 256, 8, 16.0),
    "llama3_8b_q_proj": LayerShape("llama3_8b_q_proj", 4096, 4096, 4096, 16, 16.0),
    "llama3_8b_mlp_up": LayerShape("llama3_8b_mlp_up", 8192, 4096, 14336, 64, 16.0),
    "llama3_8b_mlp_down": LayerShape("llama3_8b_mlp_down", 8192, 14336, 4096, 64, 16.0),
    "qwen14b_attn": LayerShape("qwen14b_attn", 8192, 5120, 5120, 16, 32.0, True),
    "qwen14b_mlp": LayerShape("qwen14b_mlp", 8192, 5120, 13824, 16, 32.0, True),
}
for _m in (1, 16, 128, 1024, 16384):
    SHAPES[f"sweep_m{_m}"] = LayerShape(f"sweep_m{_m}", _m, 4096, 14336, 64, 16.0)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def activations(M: int, d_in: int, d_out: int, seed: int = 0):
    """X [M, d_in] and dY [M, d_out], bf16, ~N(0, 1)."""
    g = np.random.default_rng(seed)
    X = _bf16(g.standard_normal((M, d_in), dtype=np.float32))
    dY = _bf16(g.standard_normal((M, d_out), dtype=np.float32))
    return X, dY


def weights(d_in: int, d_out: int, r: int, seed: int = 1,
            w_std: float = 0.02, b_std: float = 0.01):
    """W [d_out, d_in], A [d_in, r], B [r, d_out], all bf16."""
    g = np.random.default_rng(seed)
    W = _bf16(g.standard_normal((d_out, d_in), dtype=np.float32) * np.float32(w_std))
    lim = 1.0 / math.sqrt(d_in)
    A = _bf16(g.uniform(-lim, lim, size=(d_in, r)).astype(np.float32))
    B = _bf16(g.standard_normal((r, d_out), dtype=np.float32) * np.float32(b_std))
    return W, A, B


def layer_inputs(shape: LayerShape, seed: int = 0):
    """All inputs of one workload as CPU bf16 tensors: dict X, dY, W, A, B."""
    X, dY = activations(shape.M, shape.d_in, shape.d_out, seed)
    W, A, B = weights(shape.d_in, shape.d_out, shape.r, seed + 1)
    return {"X": X, "dY": dY, "W": W, "A": A, "B": B}


def sample_rows(M: int, n: int = 256, block: int = 128, seed: int = 7) -> np.ndarray:
    """Sorted row indices: n seeded-random rows plus the first and last row block."""
    g = np.random.default_rng(seed)
    rows = set(range(min(block, M)))
    rows |= set(range(max(0, M - block), M))
    rows |= set(int(i) for i in g.choice(M, size=min(n, M), replace=False))
    return np.array(sorted(rows), dtype=np.int64)
