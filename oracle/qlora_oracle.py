"""Plain CPU oracle for the fused NF4-QLoRA linear layer (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code, table or helper with the
CUDA library; it keeps its own copy of the NF4 codebook.

What it computes, with the passage each step follows:

* The layer: a frozen base weight W stored in 4-bit NF4, plus a trainable
  low-rank pair A (d_in x r) and B (r x d_out), scale s, no dropout, no bias:
  ``Y = X . dequant(W)^T + s . (X . A) . B``.
  Pages: "UnSloth加速原理：CUDA内核融合与内存优化", section "内核融合" (the
  Linear -> LoRA_A -> LoRA_B -> Add chain fused into one kernel, and the
  ``get_peft_model(..., lora_dropout=0, bias="none")`` / ``load_in_4bit``
  example), and its section "LoRA张量的紧凑布局" (A in R^{d_in x r},
  B in R^{r x d_out}).  The ReLU that page puts between LoRA_A and LoRA_B is
  not part of LoRA and is not computed (the LoRA product is linear).
* The hand-written backward (dX, dA, dB; no gradient for the frozen base):
  page "解锁 AI 潜能：Unsloth 的算法奥秘与实现全解析", section "Triton 编写的高效内核"
  (gradients computed by hand), and page "Unsloth性能实测：比传统方法快2倍真的吗？",
  section 3.2 "框架层：手动反向传播引擎" (LoRA gradients injected directly).
* The scale: s = alpha / r, or alpha / sqrt(r) for the rank-stabilised variant,
  page "Unsloth更新日志解读：新功能带来的实际收益", section 2.1 "--use_rslora".
  The oracle takes s itself.
* NF4 storage: the pages name NF4 only (page "UnSloth加速原理", section "内核融合",
  ``load_in_4bit=True``; page "Unsloth更新日志解读", section 1.1, NF4-resident
  weights).  The concrete format is the plainest reading: the 16-level NF4 code
  table published with QLoRA (Dettmers et al., 2023, "QLoRA: Efficient
  Finetuning of Quantized LLMs", Appendix E), blocks of 64 consecutive elements
  of the row-major weight, one fp32 absmax per block, two codes per byte with
  the first element in the high nibble.  Optionally (row f4) the absmax itself
  is stored in 8 bits per block with one fp32 scale per 256 blocks
  (``quantize_absmax_dq``); the NF4 dequantisation then uses the stored value.

Precision: the NF4 code decision is taken in fp32 (correctly rounded division
w / absmax, then an exact comparison against the midpoints between adjacent
codes, evaluated in double where they are exact); dequantisation is one fp32
multiply rounded to nearest-even bf16.  Those steps decide integers or bits and
are fixed by the format.  The contractions are evaluated in fp64 from the
bf16-valued inputs, so the oracle is the exact result up to fp64 rounding.
"""
from __future__ import annotations

import numpy as np

# NF4 code table, ascending; QLoRA (Dettmers et al., 2023), Appendix E.
# Seven negative levels, zero, eight positive levels; c[0] = -1, c[7] = 0, c[15] = 1.
NF4_CODE = np.array(
    [
        -1.0,
        -0.6961928009986877,
        -0.5250730514526367,
        -0.39491748809814453,
        -0.28444138169288635,
        -0.18477343022823334,
        -0.09105003625154495,
        0.0,
        0.07958029955625534,
        0.16093020141124725,
        0.24611230194568634,
        0.33791524171829224,
        0.44070982933044434,
        0.5626170039176941,
        0.7229568362236023,
        1.0,
    ],
    dtype=np.float32,
)

BLOCK = 64          # elements per absmax block (flattened row-major)
ZERO_CODE = 7       # index of 0.0 in NF4_CODE


def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32.

    bf16 keeps the upper 16 bits of the IEEE binary32 pattern.  Rounding to
    nearest-even adds 0x7FFF plus the lowest kept bit before truncating.
    Finite inputs only.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if not np.all(np.isfinite(f)):
        raise ValueError("bf16_round: non-finite input")
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).reshape(f.shape)


def bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("bf16_bits: value is not bf16-representable")
    return (u >> np.uint32(16)).astype(np.uint16)


def code_midpoints() -> np.ndarray:
    """The 15 decision boundaries (c[i] + c[i+1]) / 2, in double (exact there)."""
    c = NF4_CODE.astype(np.float64)
    return (c[:-1] + c[1:]) / 2.0


def nearest_code(x32) -> np.ndarray:
    """Index of the nearest NF4 level to each fp32 value x (ties -> lower index).

    q = number of midpoints strictly below x.  An x exactly on a midpoint is not
    above it, so it keeps the lower index.
    """
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    mids = code_midpoints()
    q = np.zeros(x.shape, dtype=np.int64)
    for m in mids:               # 15 comparisons, one per boundary
        q += (x > m).astype(np.int64)
    return q.astype(np.uint8)


def quantize_nf4(W) -> tuple[np.ndarray, np.ndarray]:
    """NF4-quantise a bf16-valued weight W [n_out, n_in] (given as float32).

    Returns (packed uint8 [n_out*n_in/2], absmax float32 [n_out*n_in/64]).
    Per block b of 64 consecutive elements of the row-major flattening:
    absmax_b = max |w| (exact in fp32); if absmax_b == 0 every code is the zero
    level; else x = fl32(w / absmax_b) and q = nearest_code(x).  Byte j holds
    code 2j in its high nibble and code 2j+1 in its low nibble.
    """
    W = np.asarray(W, dtype=np.float32)
    if W.ndim != 2:
        raise ValueError("W must be 2-D [n_out, n_in]")
    if W.size % BLOCK != 0:
        raise ValueError("element count must be a multiple of 64")
    if not np.all(np.isfinite(W)):
        raise ValueError("non-finite weights are not supported")
    flat = W.reshape(-1, BLOCK)
    absmax = np.max(np.abs(flat), axis=1).astype(np.float32)
    q = np.full(flat.shape, ZERO_CODE, dtype=np.uint8)
    nz = absmax > 0
    if np.any(nz):
        x = (flat[nz] / absmax[nz][:, None]).astype(np.float32)   # IEEE fp32 division
        q[nz] = nearest_code(x)
    q = q.reshape(-1)
    packed = ((q[0::2] << 4) | q[1::2]).astype(np.uint8)
    return packed, absmax


def unpack_codes(packed) -> np.ndarray:
    """Codes in element order from the packed stream (high nibble first)."""
    p = np.asarray(packed, dtype=np.uint8)
    q = np.empty(p.size * 2, dtype=np.uint8)
    q[0::2] = p >> 4
    q[1::2] = p & 0x0F
    return q


def dequantize_nf4(packed, absmax, n_out: int, n_in: int) -> np.ndarray:
    """W_deq [n_out, n_in] as bf16-exact float32: bf16_rn(fl32(c[q] * absmax_b))."""
    q = unpack_codes(packed)
    if q.size != n_out * n_in:
        raise ValueError("packed size does not match the shape")
    a = np.asarray(absmax, dtype=np.float32)
    scale = np.repeat(a, BLOCK)
    prod = (NF4_CODE[q] * scale).astype(np.float32)      # one fp32 multiply
    return bf16_round(prod).reshape(n_out, n_in)


# ---------------------------------------------------------------- row f4: the absmax stored in 8 bits

DQ_GROUP = 256      # block absmax values per second-level group


def quantize_absmax_dq(absmax) -> tuple[np.ndarray, np.ndarray]:
    """Second-level ("double") quantisation of the block absmax (row f4).

    The pages name NF4 only (page "UnSloth加速原理：CUDA内核融合与内存优化", section
    "内核融合", ``load_in_4bit``); QLoRA (Dettmers et al., 2023, section 3,
    "Double Quantization") stores the fp32 block constants themselves in 8 bits,
    in groups of 256.  The plainest well-defined version is taken: per group g of
    256 consecutive absmax values (the last group may be shorter), with c_g the
    largest of them,
        scale2_g = fl32(c_g / 255)           (0 when c_g == 0)
        q8_i     = the integer nearest fl32(a_i / scale2_g), ties to even,
                   limited to [0, 255]       (0 when scale2_g == 0)
    so each block's scale costs one byte plus a 256th of an fp32.
    Returns (q8 uint8 [n], scale2 float32 [ceil(n / 256)]).
    """
    a = np.asarray(absmax, dtype=np.float32).reshape(-1)
    n = a.size
    n_groups = -(-n // DQ_GROUP)
    scale2 = np.zeros(n_groups, dtype=np.float32)
    q8 = np.zeros(n, dtype=np.uint8)
    for g in range(n_groups):
        seg = a[g * DQ_GROUP:(g + 1) * DQ_GROUP]
        c = np.float32(seg.max())
        if c == 0.0:
            continue
        sc = np.float32(c / np.float32(255.0))                 # IEEE fp32 division
        scale2[g] = sc
        x = (seg / sc).astype(np.float32)                      # IEEE fp32 division
        q8[g * DQ_GROUP:(g + 1) * DQ_GROUP] = np.clip(np.rint(x), 0, 255).astype(np.uint8)
    return q8, scale2


def dequantize_absmax_dq(q8, scale2) -> np.ndarray:
    """The stored absmax: a'_i = fl32(q8_i * scale2_g), the block scale the NF4
    dequantisation then uses in place of the fp32 absmax."""
    q = np.asarray(q8, dtype=np.uint8).reshape(-1)
    sc = np.repeat(np.asarray(scale2, dtype=np.float32), DQ_GROUP)[:q.size]
    return (q.astype(np.float32) * sc).astype(np.float32)


def _f64(x):
    """fp64 view of an input: bf16/fp32 values widen exactly; fp64 stays as is
    (the finite-difference pins perturb inputs in fp64)."""
    a = np.asarray(x)
    if a.dtype == np.float64:
        return a
    return a.astype(np.float32).astype(np.float64)


def lora_forward(X, W_deq, A, B, s: float, rows=None):
    """Forward pass: returns (Y, T) in fp64.

    T = X . A            (M x r; the activation saved for the backward)
    Y = X . W_deq^T + s . T . B
    ``rows`` restricts both outputs to those rows of X (each row of the layer
    is independent of the others, so this is the same result row by row).
    """
    X = _f64(X)
    if rows is not None:
        X = X[np.asarray(rows)]
    Wd, A64, B64 = _f64(W_deq), _f64(A), _f64(B)
    T = X @ A64
    Y = X @ Wd.T + float(s) * (T @ B64)
    return Y, T


def lora_backward(X, dY, W_deq, A, B, s: float, T=None, dx_rows=None):
    """Hand-written backward: returns (dX, dA, dB) in fp64.

    G  = dY . B^T                  (M x r)
    dX = dY . W_deq + s . G . A^T  (the base weight's forward operand was W_deq^T)
    dA = s . X^T . G
    dB = s . T^T . dY,  T = X . A
    W is frozen: there is no dW.  ``dx_rows`` restricts dX to those rows
    (dA and dB always reduce over every row).  ``T`` may be passed to reuse
    the forward's saved activation.
    """
    X64, dY64 = _f64(X), _f64(dY)
    Wd, A64, B64 = _f64(W_deq), _f64(A), _f64(B)
    s = float(s)
    if T is None:
        T = X64 @ A64
    else:
        T = np.asarray(T, dtype=np.float64)
    G = dY64 @ B64.T
    dA = s * (X64.T @ G)
    dB = s * (T.T @ dY64)
    if dx_rows is None:
        dX = dY64 @ Wd + s * (G @ A64.T)
    else:
        r_ = np.asarray(dx_rows)
        dX = dY64[r_] @ Wd + s * (G[r_] @ A64.T)
    return dX, dA, dB


def merged_weight(W_deq, A, B, s: float) -> np.ndarray:
    """Merged dense weight W_deq + s . (A . B)^T in fp64 (the 16-bit export).

    Page "这不是“魔法”是把Unsloth的底层优化逻辑榨干了用", section 4
    (``save_pretrained_merged(..., "merged_16bit")``): the adapter folded
    into the base weight.
    """
    return _f64(W_deq) + float(s) * (_f64(A) @ _f64(B)).T


def merged_weight_bf16(W_deq, A, B, s: float) -> np.ndarray:
    """The 16-bit export: merged_weight rounded to bf16 (nearest, ties to even).

    Same page and section as merged_weight (the "merged_16bit" save).
    """
    return bf16_round(merged_weight(W_deq, A, B, s))


def lora_scale(alpha: float, r: int, rank_stabilised: bool = False) -> float:
    """s = alpha / r, or alpha / sqrt(r) for the rank-stabilised variant."""
    return float(alpha) / (float(np.sqrt(r)) if rank_stabilised else float(r))


def swiglu_forward(gu) -> np.ndarray:
    """h = silu(g) * u in fp64, g the first and u the second half of the columns.

    silu(x) = x / (1 + exp(-x)).  The SwiGLU gate of the MLP block between the
    stacked gate/up projection and the down projection; the pages fuse the
    MLP into their forward (page "Unsloth性能实测：比传统方法快2倍真的吗？",
    section 2.2) and name SwiGLU among the fused transformer operators (page
    "UnSloth加速原理：CUDA内核融合与内存优化", section "在ms-swift中的角色").
    """
    gu = _f64(gu)
    d_ff = gu.shape[1] // 2
    g, u = gu[:, :d_ff], gu[:, d_ff:]
    return g / (1.0 + np.exp(-g)) * u


def swiglu_backward(gu, dh) -> np.ndarray:
    """[dL/dg | dL/du] of h = silu(g) * u, in the layout of gu, fp64.

    dL/du = dh * silu(g); dL/dg = dh * u * sigma(g) * (1 + g * (1 - sigma(g))),
    the derivative of x * sigma(x) written out.  Same passages as swiglu_forward.
    """
    gu, dh = _f64(gu), _f64(dh)
    d_ff = gu.shape[1] // 2
    g, u = gu[:, :d_ff], gu[:, d_ff:]
    sg = 1.0 / (1.0 + np.exp(-g))
    return np.concatenate([dh * u * sg * (1.0 + g * (1.0 - sg)), dh * g * sg], axis=1)


def _stored(x, store_bf16: bool):
    return bf16_round(x) if store_bf16 else _f64(x)


def swiglu_mlp_forward(X, Wd_gu, A_gu, B_gu, Wd_d, A_d, B_d, s: float, store_bf16: bool = True):
    """The SwiGLU MLP block of two LoRA layers: Y = down(swiglu(gate_up(X))).

    gate_up is one layer whose output columns are [gate | up] (the stacked
    projection).  With ``store_bf16`` its output and h are rounded to bf16
    between the layers, as the block stores them; without it they stay fp64
    (the exact composition, which the finite-difference pin uses).  Returns Y
    and the saved tensors (gu, T_gu, h, T_d).
    """
    gu, T_gu = lora_forward(X, Wd_gu, A_gu, B_gu, s)
    gu = _stored(gu, store_bf16)
    h = _stored(swiglu_forward(gu), store_bf16)
    Y, T_d = lora_forward(h, Wd_d, A_d, B_d, s)
    return Y, (gu, T_gu, h, T_d)


def swiglu_mlp_backward(X, dY, saved, Wd_gu, A_gu, B_gu, Wd_d, A_d, B_d, s: float, store_bf16: bool = True):
    """Gradients of the block: dX, (dA_gu, dB_gu), (dA_d, dB_d).

    dh comes out of the down layer's backward and dgu out of the gate's; with
    ``store_bf16`` both are rounded to bf16 between the steps, as the block
    stores them, otherwise they stay fp64.
    """
    gu, T_gu, h, T_d = saved
    dh, dA_d, dB_d = lora_backward(h, dY, Wd_d, A_d, B_d, s, T=T_d)
    dh = _stored(dh, store_bf16)
    dgu = _stored(swiglu_backward(gu, dh), store_bf16)
    dX, dA_gu, dB_gu = lora_backward(X, dgu, Wd_gu, A_gu, B_gu, s, T=T_gu)
    return dX, (dA_gu, dB_gu), (dA_d, dB_d)
