"""The argument behind the NF4 quantise kernel's division-free code decision.

The kernel forms x' = fl(w * fl(1/m)) instead of the format's fl32(w / m)
whenever fl(1/m) is a normal float.  Scaling w and m by the same power of two
scales both quotients exactly (a quotient below 2^-126 gives the zero code
either way), so the decision only depends on pairs with m in [1, 2).  Checked
here on the CPU with numpy's correctly rounded float32 arithmetic: for every
bf16 m in [1, 2) and every bf16 |w| <= m the two quotients give the same code
(exhaustive), and random pairs across the whole exponent range agree too.  The
GPU tests compare the kernel itself with the oracle.
"""
import numpy as np

from oracle import qlora_oracle as O


def _codes(x32):
    return O.nearest_code(x32)


def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def test_reciprocal_quotient_gives_the_same_code_exhaustive():
    for m_bits in range(0x3F80, 0x4000):
        wb = np.arange(0, m_bits + 1, dtype=np.uint32)
        wb = np.concatenate([wb, wb | 0x8000])
        w = _bf16(wb)
        m = _bf16(m_bits)
        x_fast = w * (np.float32(1) / m)
        x_ieee = w / m
        assert x_fast.dtype == np.float32 and x_ieee.dtype == np.float32
        assert np.array_equal(_codes(x_fast), _codes(x_ieee)), hex(m_bits)


def test_reciprocal_quotient_gives_the_same_code_any_exponent():
    g = np.random.default_rng(11)
    n = 400_000
    m_bits = g.integers(0x0080, 0x7E80, size=n, dtype=np.uint32)      # 1/m a normal float
    m = _bf16(m_bits)
    frac = g.uniform(-1.0, 1.0, size=n).astype(np.float32)
    w = _bf16((((frac * m).view(np.uint32)) >> 16))                   # a bf16 with |w| <= m
    keep = np.abs(w) <= m
    w, m = w[keep], m[keep]
    with np.errstate(under="ignore"):
        x_fast = w * (np.float32(1) / m)
        x_ieee = w / m
    assert np.array_equal(_codes(x_fast), _codes(x_ieee))
