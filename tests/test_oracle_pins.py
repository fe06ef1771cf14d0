"""Pins for the CPU oracle: each test checks it against something other than
itself -- the published NF4 table, a library rounding routine, closed forms,
identities the layer must satisfy, and finite differences."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import qlora_oracle as O


def _read_numbers(path):
    vals = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return vals


def _torch_bf16(x32):
    """Library rounding: torch's fp32 -> bf16 conversion (nearest-even)."""
    return torch.from_numpy(np.asarray(x32, dtype=np.float32)).to(torch.bfloat16).float().numpy()


# ----------------------------------------------------------------- codebook

def test_codebook_is_published_table(golden_dir):
    tab = np.array(_read_numbers(os.path.join(golden_dir, "nf4_codebook.txt")), dtype=np.float64)
    assert tab.shape == (16,)
    assert np.array_equal(O.NF4_CODE.astype(np.float64), tab)


def test_codebook_structure():
    c = O.NF4_CODE.astype(np.float64)
    assert np.all(np.diff(c) > 0)
    assert c[0] == -1.0 and c[15] == 1.0 and c[O.ZERO_CODE] == 0.0
    assert int(np.sum(c < 0)) == 7 and int(np.sum(c > 0)) == 8


def test_codebook_normal_quantile_construction():
    """NF4 levels are normal quantiles (QLoRA section 3): 8 positive levels from
    quantiles on [delta, 0.5), 7 negative ones mirrored, plus an exact zero,
    normalised to [-1, 1]; delta is the mean of 1-1/(2*15) and 1-1/(2*16)."""
    from scipy.stats import norm
    delta = 0.5 * ((1 - 1 / 30) + (1 - 1 / 32))
    pos = norm.ppf(np.linspace(delta, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(delta, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, [0.0], neg]))
    v = v / np.max(np.abs(v))
    assert np.max(np.abs(v - O.NF4_CODE.astype(np.float64))) <= 1e-6


# ----------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_library():
    g = np.random.default_rng(3)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        g.standard_normal(20000).astype(np.float32) * np.float32(100.0),
        g.uniform(-1, 1, 20000).astype(np.float32),
    ])
    # exact ties: low half exactly 0x8000, with even and odd kept parts
    hi = g.integers(0x3000, 0x4800, size=4000, dtype=np.uint32)
    ties = ((hi << 16) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, -0.0, 1.0, -1.0])])
    assert np.array_equal(O.bf16_round(x).view(np.uint32), _torch_bf16(x).view(np.uint32))


# ----------------------------------------------------------------- code decision

def test_nearest_code_brute_force():
    g = np.random.default_rng(5)
    x = g.uniform(-1, 1, 50000).astype(np.float32)
    x = np.concatenate([x, O.NF4_CODE, np.float32([0.0])])
    c = O.NF4_CODE.astype(np.float64)
    d = np.abs(x.astype(np.float64)[:, None] - c[None, :])
    brute = np.argmin(d, axis=1)   # first minimum -> lower index on a tie
    assert np.array_equal(O.nearest_code(x).astype(np.int64), brute)


def test_nearest_code_ties_go_low():
    c = O.NF4_CODE
    # midpoints next to zero are c/2, exact in fp32
    m78 = np.float32(c[8] / np.float32(2))
    m67 = np.float32(c[6] / np.float32(2))
    up = lambda v: np.nextafter(v, np.float32(np.inf))
    dn = lambda v: np.nextafter(v, np.float32(-np.inf))
    xs = np.float32([m78, up(m78), dn(m78), m67, up(m67), dn(m67)])
    assert list(O.nearest_code(xs)) == [7, 8, 7, 6, 7, 6]


# ----------------------------------------------------------------- quantise / dequantise

def _codebook_weight(n_out, n_in, seed):
    """W whose every element is bf16(c[q] * a_block) with a planted +-a per block."""
    g = np.random.default_rng(seed)
    nb = n_out * n_in // 64
    q = g.integers(0, 16, size=(nb, 64)).astype(np.uint8)
    pos = g.integers(0, 64, size=nb)
    q[np.arange(nb), pos] = np.where(g.integers(0, 2, size=nb) == 1, 15, 0)
    a = _torch_bf16(np.exp2(g.uniform(-10, 4, size=nb)).astype(np.float32))
    W = _torch_bf16((O.NF4_CODE[q] * a[:, None]).astype(np.float32))
    return W.reshape(n_out, n_in), q.reshape(-1), a


@pytest.mark.parametrize("shape", [(1, 64), (3, 128), (16, 256), (40, 576)])
def test_quantize_round_trip_on_codebook_points(shape):
    n_out, n_in = shape
    W, q, a = _codebook_weight(n_out, n_in, seed=n_out * 131 + n_in)
    packed, absmax = O.quantize_nf4(W)
    assert np.array_equal(absmax, a)
    assert np.array_equal(O.unpack_codes(packed), q)
    Wd = O.dequantize_nf4(packed, absmax, n_out, n_in)
    assert np.array_equal(Wd.view(np.uint32), W.view(np.uint32))


def test_zero_block():
    W = np.zeros((2, 128), dtype=np.float32)
    W[1, 64:] = _torch_bf16(np.float32([0.5]))[0]
    packed, absmax = O.quantize_nf4(W)
    assert absmax[0] == 0 and absmax[1] == 0 and absmax[2] == 0 and absmax[3] == 0.5
    assert np.all(packed[:96] == 0x77)
    assert np.all(O.dequantize_nf4(packed, absmax, 2, 128)[0] == 0.0)


def test_pack_golden_example(golden_dir):
    spec = {}
    with open(os.path.join(golden_dir, "nf4_pack_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                spec[k] = v
    n_out, n_in = int(spec["n_out"][0]), int(spec["n_in"][0])
    W = np.zeros(n_out * n_in, dtype=np.float32)
    w = np.float32([float(v) for v in spec["w"]])
    W[: w.size] = w
    packed, absmax = O.quantize_nf4(W.reshape(n_out, n_in))
    assert list(absmax) == [float(v) for v in spec["absmax"]]
    prefix = bytes.fromhex(spec["packed_prefix_hex"][0])
    fill = bytes.fromhex(spec["packed_fill_hex"][0])[0]
    assert bytes(packed[: len(prefix)]) == prefix
    assert np.all(packed[len(prefix):] == fill)
    codes = [int(v) for v in spec["codes"]]
    assert list(O.unpack_codes(packed)[: len(codes)]) == codes


def test_dequant_is_one_fp32_multiply_then_library_rounding():
    g = np.random.default_rng(11)
    n_out, n_in = 8, 192
    packed = g.integers(0, 256, size=n_out * n_in // 2, dtype=np.uint8)
    absmax = g.uniform(1e-3, 3.0, size=n_out * n_in // 64).astype(np.float32)
    Wd = O.dequantize_nf4(packed, absmax, n_out, n_in)
    hi = (packed >> 4).astype(np.int64)
    lo = (packed & 15).astype(np.int64)
    codes = np.stack([hi, lo], axis=1).reshape(-1)
    scale = np.repeat(absmax, 64)
    prod = np.array([np.float32(O.NF4_CODE[k]) * np.float32(s) for k, s in zip(codes, scale)],
                    dtype=np.float32)
    assert np.array_equal(Wd.reshape(-1).view(np.uint32), _torch_bf16(prod).view(np.uint32))


def test_quantize_matches_brute_force_on_random_weights():
    g = np.random.default_rng(13)
    W = _torch_bf16(g.standard_normal((6, 320)).astype(np.float32) * np.float32(0.02))
    packed, absmax = O.quantize_nf4(W)
    flat = W.reshape(-1, 64)
    c = O.NF4_CODE.astype(np.float64)
    for b in range(flat.shape[0]):
        amax = max(abs(float(v)) for v in flat[b])
        assert absmax[b] == np.float32(amax)
        for i in range(64):
            x = float(np.float32(flat[b, i]) / np.float32(amax))
            best = min(range(16), key=lambda k: (abs(x - c[k]), k))
            assert O.unpack_codes(packed)[b * 64 + i] == best


# ----------------------------------------------------------------- forward

def _small_problem(M, K, N, r, seed):
    g = np.random.default_rng(seed)
    X = _torch_bf16(g.standard_normal((M, K)).astype(np.float32))
    W = _torch_bf16(g.standard_normal((N, K)).astype(np.float32) * np.float32(0.02))
    A = _torch_bf16(g.uniform(-0.1, 0.1, (K, r)).astype(np.float32))
    B = _torch_bf16(g.standard_normal((r, N)).astype(np.float32) * np.float32(0.05))
    packed, absmax = O.quantize_nf4(W)
    Wd = O.dequantize_nf4(packed, absmax, N, K)
    return X, Wd, A, B


def test_forward_one_hot_closed_form():
    """X = one-hot rows picks a COLUMN of W_deq (W is [d_out, d_in]) and a row of A."""
    K, N, r, s = 128, 192, 5, 1.75
    _, Wd, A, B = _small_problem(4, K, N, r, seed=17)
    ks = [0, 3, 77, 127]
    X = np.zeros((len(ks), K), dtype=np.float32)
    for i, k in enumerate(ks):
        X[i, k] = 1.0
    Y, T = O.lora_forward(X, Wd, A, B, s)
    for i, k in enumerate(ks):
        for n in range(0, N, 37):
            lora = sum(float(A[k, j]) * float(B[j, n]) for j in range(r))
            assert Y[i, n] == pytest.approx(float(Wd[n, k]) + s * lora, rel=1e-12, abs=1e-15)
        for j in range(r):
            assert T[i, j] == float(A[k, j])


def test_forward_lora_zero_reduces_to_base_gemm():
    X, Wd, A, B = _small_problem(16, 128, 64, 4, seed=19)
    Y0, _ = O.lora_forward(X, Wd, A, np.zeros_like(B), 3.0)
    ref = torch.from_numpy(X.astype(np.float64)) @ torch.from_numpy(Wd.astype(np.float64)).T
    assert np.allclose(Y0, ref.numpy(), rtol=1e-12, atol=1e-12)
    Y1, _ = O.lora_forward(X, Wd, np.zeros_like(A), B, 3.0)
    assert np.allclose(Y1, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_forward_merged_weight_identity():
    X, Wd, A, B = _small_problem(12, 192, 128, 8, seed=23)
    s = 0.625
    Y, _ = O.lora_forward(X, Wd, A, B, s)
    Wm = O.merged_weight(Wd, A, B, s)
    assert Wm.shape == Wd.shape
    assert np.allclose(Y, X.astype(np.float64) @ Wm.T, rtol=1e-11, atol=1e-12)


def test_forward_linear_in_s_and_row_independent():
    X, Wd, A, B = _small_problem(10, 64, 64, 3, seed=29)
    Y0, _ = O.lora_forward(X, Wd, A, B, 0.0)
    Y1, _ = O.lora_forward(X, Wd, A, B, 1.0)
    Y3, _ = O.lora_forward(X, Wd, A, B, 3.0)
    assert np.allclose(Y3, Y0 + 3.0 * (Y1 - Y0), rtol=1e-11, atol=1e-12)
    rows = [1, 4, 9]
    Yr, Tr = O.lora_forward(X, Wd, A, B, 3.0, rows=rows)
    _, T = O.lora_forward(X, Wd, A, B, 3.0)
    assert np.array_equal(Yr, Y3[rows]) and np.array_equal(Tr, T[rows])


# ----------------------------------------------------------------- backward

def _fd_problem():
    g = np.random.default_rng(31)
    M, K, N, r = 4, 64, 64, 4
    X = g.standard_normal((M, K))
    Wd = g.standard_normal((N, K)) * 0.02
    A = g.standard_normal((K, r)) * 0.1
    B = g.standard_normal((r, N)) * 0.1
    R = g.standard_normal((M, N))
    return X, Wd, A, B, R


def _loss(X, Wd, A, B, R, s):
    Y, _ = O.lora_forward(X, Wd, A, B, s)
    return float(np.sum(Y * R))


@pytest.mark.parametrize("s", [0.5, 2.0])
def test_backward_central_finite_differences(s):
    """L = <Y, R>: dL/dX, dL/dA, dL/dB by central differences in fp64 against the
    hand-written backward with dY = R."""
    X, Wd, A, B, R = _fd_problem()
    dX, dA, dB = O.lora_backward(X, R, Wd, A, B, s)
    h = 1e-4
    g = np.random.default_rng(37)
    for name, P, grad in (("X", X, dX), ("A", A, dA), ("B", B, dB)):
        for _ in range(12):
            idx = tuple(int(g.integers(0, n)) for n in P.shape)
            Pp, Pm = P.copy(), P.copy()
            Pp[idx] += h
            Pm[idx] -= h
            args_p = {"X": X, "A": A, "B": B}
            args_m = dict(args_p)
            args_p[name], args_m[name] = Pp, Pm
            lp = _loss(args_p["X"], Wd, args_p["A"], args_p["B"], R, s)
            lm = _loss(args_m["X"], Wd, args_m["A"], args_m["B"], R, s)
            fd = (lp - lm) / (2 * h)
            assert fd == pytest.approx(grad[idx], rel=1e-6, abs=1e-9), (name, idx)


def test_backward_special_cases():
    X, Wd, A, B, R = _fd_problem()
    s = 1.5
    dX, dA, dB = O.lora_backward(X, R, Wd, A, np.zeros_like(B), s)
    assert np.all(dA == 0.0)
    assert np.allclose(dX, R @ Wd, rtol=1e-12, atol=1e-14)
    dX, dA, dB = O.lora_backward(X, R, Wd, np.zeros_like(A), B, s)
    assert np.all(dB == 0.0)


def test_backward_uses_saved_activation_and_rows():
    X, Wd, A, B, R = _fd_problem()
    s = 0.75
    _, T = O.lora_forward(X, Wd, A, B, s)
    full = O.lora_backward(X, R, Wd, A, B, s)
    saved = O.lora_backward(X, R, Wd, A, B, s, T=T, dx_rows=[0, 3])
    assert np.allclose(saved[0], full[0][[0, 3]], rtol=0, atol=1e-15)
    assert np.allclose(saved[1], full[1], rtol=0, atol=1e-15)
    assert np.allclose(saved[2], full[2], rtol=0, atol=1e-15)


def test_scale():
    assert O.lora_scale(16, 16) == 1.0
    assert O.lora_scale(16, 64) == 0.25
    assert O.lora_scale(16, 8) == 2.0
    assert O.lora_scale(32, 16, rank_stabilised=True) == 8.0
    assert O.lora_scale(16, 64, rank_stabilised=True) == pytest.approx(2.0)
    assert math.isclose(O.lora_scale(10, 3, True), 10 / math.sqrt(3))


def test_merged_export_with_zero_adapter_is_the_dequantised_weight():
    """B = 0: the 16-bit export is the bf16 dequantised weight itself, bit for bit."""
    rng = np.random.default_rng(31)
    W = O.bf16_round(rng.normal(0.0, 0.02, size=(24, 128)).astype(np.float32))
    packed, absmax = O.quantize_nf4(W)
    Wd = O.dequantize_nf4(packed, absmax, 24, 128)
    A = O.bf16_round(rng.uniform(-0.1, 0.1, size=(128, 8)).astype(np.float32))
    B = np.zeros((8, 24), dtype=np.float32)
    out = O.merged_weight_bf16(Wd, A, B, 2.0)
    assert np.array_equal(O.bf16_bits(out), O.bf16_bits(Wd))


def test_merged_export_with_one_hot_adapter_moves_one_column():
    """A = e_k0 (a single 1 in rank 0), B row 0 = v: only column k0 changes, to
    bf16(W[:, k0] + s*v), a sum of two exact values rounded once."""
    rng = np.random.default_rng(32)
    Wd = O.bf16_round(rng.normal(0.0, 0.02, size=(16, 64)).astype(np.float32))
    A = np.zeros((64, 4), dtype=np.float32)
    A[37, 0] = 1.0
    v = O.bf16_round(rng.normal(0.0, 0.01, size=16).astype(np.float32))
    B = np.zeros((4, 16), dtype=np.float32)
    B[0] = v
    out = O.merged_weight_bf16(Wd, A, B, 0.5)
    others = np.ones(64, dtype=bool)
    others[37] = False
    assert np.array_equal(out[:, others], Wd[:, others])
    expect = O.bf16_round((Wd[:, 37].astype(np.float64) + 0.5 * v.astype(np.float64)))
    assert np.array_equal(O.bf16_bits(out[:, 37]), O.bf16_bits(expect))


# ---- SwiGLU gate of the MLP block ------------------------------------------

def test_swiglu_forward_against_library_sigmoid():
    """h = g * sigma(g) * u with scipy's expit as sigma, and closed-form values."""
    from scipy.special import expit
    rng = np.random.default_rng(7)
    gu = rng.normal(0.0, 3.0, size=(5, 16))
    g, u = gu[:, :8], gu[:, 8:]
    np.testing.assert_allclose(O.swiglu_forward(gu), g * expit(g) * u, rtol=1e-14, atol=1e-300)
    one = np.array([[0.0, 1.0, 40.0, -40.0, 1.0, 1.0, 1.0, 1.0]])
    h = O.swiglu_forward(one)[0]
    assert h[0] == 0.0                                        # silu(0) = 0
    assert abs(h[1] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15     # silu(1) = sigma(1)
    assert abs(h[2] - 40.0) < 1e-12 and abs(h[3]) < 1e-15     # saturation at both ends


def test_swiglu_gate_is_the_first_half():
    gu = np.array([[2.0, 3.0]])
    assert O.swiglu_forward(gu)[0, 0] == 2.0 / (1.0 + np.exp(-2.0)) * 3.0
    assert O.swiglu_forward(gu[:, ::-1])[0, 0] == 3.0 / (1.0 + np.exp(-3.0)) * 2.0


def test_swiglu_backward_matches_finite_differences():
    rng = np.random.default_rng(8)
    gu = rng.normal(0.0, 2.0, size=(3, 12))
    dh = rng.normal(0.0, 1.0, size=(3, 6))
    grad = O.swiglu_backward(gu, dh)
    eps = 1e-6
    num = np.zeros_like(gu)
    for idx in np.ndindex(gu.shape):
        p, m = gu.copy(), gu.copy()
        p[idx] += eps
        m[idx] -= eps
        num[idx] = np.sum((O.swiglu_forward(p) - O.swiglu_forward(m)) * dh) / (2 * eps)
    np.testing.assert_allclose(grad, num, rtol=1e-7, atol=1e-9)


def test_swiglu_mlp_block_backward_matches_finite_differences():
    """The whole block (gate/up layer, gate, down layer) with fp64 intermediates:
    the gradients of L = <Y, R> by central differences in X, A and B of both layers."""
    rng = np.random.default_rng(9)
    M, dm, dff, r, s = 3, 8, 6, 2, 0.7
    X = rng.normal(size=(M, dm))
    Wgu = rng.normal(size=(2 * dff, dm)) * 0.5
    Wd = rng.normal(size=(dm, dff)) * 0.5
    Agu, Bgu = rng.normal(size=(dm, r)), rng.normal(size=(r, 2 * dff))
    Ad, Bd = rng.normal(size=(dff, r)), rng.normal(size=(r, dm))
    R = rng.normal(size=(M, dm))

    def loss(X_, Agu_, Bgu_, Ad_, Bd_):
        Y, _ = O.swiglu_mlp_forward(X_, Wgu, Agu_, Bgu_, Wd, Ad_, Bd_, s, store_bf16=False)
        return float(np.sum(Y * R))

    Y, saved = O.swiglu_mlp_forward(X, Wgu, Agu, Bgu, Wd, Ad, Bd, s, store_bf16=False)
    dX, (dAgu, dBgu), (dAd, dBd) = O.swiglu_mlp_backward(X, R, saved, Wgu, Agu, Bgu, Wd, Ad, Bd, s,
                                                         store_bf16=False)
    args = [X, Agu, Bgu, Ad, Bd]
    for k, grad in enumerate([dX, dAgu, dBgu, dAd, dBd]):
        num = np.zeros_like(args[k])
        for idx in np.ndindex(args[k].shape):
            p = [a.copy() for a in args]
            m = [a.copy() for a in args]
            p[k][idx] += 1e-6
            m[k][idx] -= 1e-6
            num[idx] = (loss(*p) - loss(*m)) / 2e-6
        # central-difference noise is ~1e-7 here; a wrong term or sign is off by O(1)
        np.testing.assert_allclose(grad, num, rtol=1e-5, atol=1e-7)


def test_swiglu_mlp_block_forward_one_hot():
    """One-hot token and exact NF4 weights (entries in {-a, 0, a}, one at +-a per
    block): Y picks one column of the down weight times silu(g) * u of one
    feature, with g, u read off the stacked weight; silu by scipy's expit."""
    from scipy.special import expit
    dm, dff, k = 64, 8, 5
    Wgu = np.zeros((2 * dff, dm), dtype=np.float32)
    Wgu[3, k], Wgu[dff + 3, k] = 0.5, -0.25            # g_3 = 0.5, u_3 = -0.25; every other feature 0
    Wd = np.zeros((dm, dff), dtype=np.float32)
    Wd[7, 3] = 2.0                                     # Y[:, 7] = 2 h_3
    for W in (Wgu, Wd):
        q, a = O.quantize_nf4(W)
        assert np.array_equal(O.dequantize_nf4(q, a, *W.shape), W)   # exact NF4 points
    X = np.zeros((1, dm), dtype=np.float32)
    X[0, k] = 1.0
    Z = np.zeros
    Y, _ = O.swiglu_mlp_forward(X, Wgu, Z((dm, 1)), Z((1, 2 * dff)), Wd, Z((dff, 1)), Z((1, dm)), 1.0,
                                store_bf16=False)
    want = np.zeros((1, dm))
    want[0, 7] = 2.0 * 0.5 * expit(0.5) * -0.25
    np.testing.assert_allclose(Y, want, rtol=1e-14, atol=1e-300)


# ---------------------------------------------------------------- row f4: 8-bit absmax

def test_absmax_dq_exact_on_representable_scales():
    """A group whose largest absmax is 255 * 2^e has scale2 = 2^e exactly, so
    every k * 2^e (k in 0..255) is stored as k and comes back exactly."""
    g = np.random.default_rng(21)
    for e in (-20, -3, 0, 7):
        k = g.integers(0, 256, size=256)
        k[17] = 255
        a = (k.astype(np.float64) * 2.0 ** e).astype(np.float32)
        q, sc = O.quantize_absmax_dq(a)
        assert sc[0] == np.float32(2.0 ** e)
        assert np.array_equal(q.astype(np.int64), k)
        assert np.array_equal(O.dequantize_absmax_dq(q, sc), a)


def test_absmax_dq_brute_force_nearest_code():
    """Each stored byte is the code whose value k * scale2 is nearest a_i among all
    256 (searched exhaustively in fp64; a tie between two codes goes to the even
    one), over a ragged last group, and the largest absmax of a group is 255."""
    g = np.random.default_rng(22)
    a = (np.abs(g.normal(size=700)) * np.exp(g.uniform(-4, 4, size=700))).astype(np.float32)
    q, sc = O.quantize_absmax_dq(a)
    assert sc.size == 3 and q.size == 700
    for i in range(a.size):
        s_g = np.float64(sc[i // 256])
        x = np.float64(np.float32(np.float32(a[i]) / np.float32(s_g)))   # the quotient in fp32
        d = np.abs(x - np.arange(256, dtype=np.float64))
        best = np.flatnonzero(d == d.min())
        want = best[0] if best.size == 1 else best[best % 2 == 0][0]
        assert q[i] == want, i
    for grp in range(3):
        seg = a[grp * 256:(grp + 1) * 256]
        assert q[grp * 256 + int(np.argmax(seg))] == 255


def test_absmax_dq_error_bound_and_zero_groups():
    """|a' - a| is at most half a step of the group's scale (plus fp32 rounding),
    and an all-zero group stores zeros with scale 0."""
    g = np.random.default_rng(23)
    a = np.abs(g.normal(size=1024)).astype(np.float32)
    a[256:512] = 0.0
    q, sc = O.quantize_absmax_dq(a)
    r = O.dequantize_absmax_dq(q, sc)
    assert sc[1] == 0.0 and not np.any(q[256:512]) and not np.any(r[256:512])
    step = np.repeat(sc.astype(np.float64), 256)
    assert np.all(np.abs(r.astype(np.float64) - a) <= 0.5 * step * (1 + 2.0 ** -20) + 2.0 ** -24 * a)
