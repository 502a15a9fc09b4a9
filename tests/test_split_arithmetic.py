"""The arithmetic of the fp32-accurate tensor-core products (okls_tc3.cu),
checked on the CPU with an emulation of bf16 round-to-nearest-even:

* an fp32 value x splits into three bf16 terms b1 = bf16(x), b2 = bf16(x - b1),
  b3 = bf16(x - b1 - b2), each difference exact in fp32, and b1 + b2 + b3 = x
  exactly (|b2| <= 2^-8 |x|, |b3| <= 2^-17 |x|: three 8-bit terms with signed
  rounding cover fp32's 24-bit significand);
* the product of two split values keeps six terms (b1 c1; b1 c2, b2 c1 at up
  to 2^-8 of the leading one; b1 c3, b3 c1, b2 c2 at up to 2^-15), each exact
  in fp32, and misses x c by the two dropped cross terms b2 c3 + b3 c2 and
  b3 c3: at most 2^-24 + 2^-34 of |x c|, fp32's unit roundoff;
* a value that bf16 holds exactly (the identity's 0 and 1, a bf16 gradient)
  splits into itself and two zeros, so its products are exact.
(Products and terms inside fp32's normal range.)
"""

import numpy as np


def bf16_rn(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def split3(x: np.ndarray):
    x = np.asarray(x, dtype=np.float32)
    b1 = bf16_rn(x)
    r1 = (x - b1).astype(np.float32)
    b2 = bf16_rn(r1)
    r2 = (r1 - b2).astype(np.float32)
    b3 = bf16_rn(r2)
    return b1, b2, b3, r1, r2


def _samples(n=200000, seed=0):
    """fp32 values over 2^-20 .. 2^20: the products and their smallest kept
    terms (2^-18 of the leading one) stay in fp32's normal range, where the
    exactness claims hold (an operand's data spans far less)."""
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, n)
    expo = rng.integers(-20, 20, n)
    sign = rng.choice([-1.0, 1.0], n)
    return (sign * mant * np.exp2(expo)).astype(np.float32)


def test_split_differences_are_exact_and_three_terms_hold_x():
    x = _samples()
    b1, b2, b3, r1, r2 = split3(x)
    x64 = x.astype(np.float64)
    # the differences formed in fp32 are the exact differences
    assert np.array_equal(r1.astype(np.float64), x64 - b1.astype(np.float64))
    assert np.array_equal(r2.astype(np.float64), r1.astype(np.float64) - b2.astype(np.float64))
    # each term is a bf16 value
    for b in (b1, b2, b3):
        assert np.array_equal(bf16_rn(b), b)
    assert np.array_equal(b1.astype(np.float64) + b2 + b3, x64)
    assert np.all(np.abs(b2) <= 2.0 ** -8 * np.abs(x)) and np.all(np.abs(b3) <= 2.0 ** -17 * np.abs(x))


def test_six_term_product_error_bound():
    x = _samples(seed=1)
    c = _samples(seed=2)
    a1, a2, a3, _, _ = (t.astype(np.float64) for t in split3(x))
    c1, c2, c3, _, _ = (t.astype(np.float64) for t in split3(c))
    terms = [a1 * c1, a1 * c2, a2 * c1, a1 * c3, a3 * c1, a2 * c2]
    # each product of two bf16 values has at most 16 significant bits: exact in fp32
    for t in terms:
        assert np.array_equal(t.astype(np.float32).astype(np.float64), t)
    exact = x.astype(np.float64) * c.astype(np.float64)
    approx = sum(terms)
    rel = np.abs(approx - exact) / np.abs(exact)
    assert np.all(rel <= 2.0 ** -24 + 2.0 ** -34), float(rel.max())
    # what is dropped is exactly the three smallest cross terms
    a1x, a2x, a3x, c1x, c2x, c3x = a1, a2, a3, c1, c2, c3
    assert np.allclose(exact - approx, a2x * c3x + a3x * c2x + a3x * c3x, rtol=1e-12, atol=0.0)
    # and the kept terms fall off as the split says: 2^-8 and 2^-15 of the leading one
    lead = np.abs(terms[0])
    assert np.all(np.abs(terms[1]) + np.abs(terms[2]) <= 2.0 ** -7 * lead * (1 + 2.0 ** -7))
    assert np.all(np.abs(terms[3]) + np.abs(terms[4]) + np.abs(terms[5]) <= 2.0 ** -15 * lead * (1 + 2.0 ** -7))


def test_bf16_values_split_exactly():
    rng = np.random.default_rng(3)
    g = bf16_rn(rng.standard_normal(10000).astype(np.float32))
    for v in (g, np.array([0.0, 1.0, -1.0, 0.5], dtype=np.float32)):
        b1, b2, b3, _, _ = split3(v)
        assert np.array_equal(b1, v) and not b2.any() and not b3.any()
    # the identity's products reproduce the other operand: 1 x (c1 + c2 + c3) = c
    c = _samples(seed=4)
    c1, c2, c3, _, _ = split3(c)
    assert np.array_equal(c1.astype(np.float64) + c2 + c3, c.astype(np.float64))
