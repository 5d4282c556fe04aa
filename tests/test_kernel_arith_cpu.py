"""Host-side proofs of the arithmetic shortcuts the quantising kernels rely on (no GPU).

The group step of the asymmetric quantiser is fl32((hi - lo) / 15). The kernels form it without
a division: q0 = fl32(d * r15) with r15 = fl32(1/15), the remainder e = d - 15 q0 (exact, one
FMA), and q1 = fl32(q0 + e * r15) (one FMA), Markstein's correction step. Whether that equals
the correctly rounded quotient depends only on d's significand (scaling d by 2^j scales every
quantity by 2^j while the results stay normal), so checking all 2^23 significands of one binade
with exact integer arithmetic proves it for every d whose quotient is a normal float.
"""

from fractions import Fraction

import numpy as np


def _rn_shift(num, sh):
    """round(num / 2^sh) to nearest, ties to even, for non-negative int64 arrays."""
    k = num >> sh
    rem = num - (k << sh)
    half = np.int64(1) << (sh - 1)
    return k + ((rem > half) | ((rem == half) & ((k & 1) == 1)))


def _rn32(fr: Fraction) -> Fraction:
    """A positive rational rounded to fp32's 24-bit significand (normal range), ties to even."""
    e = fr.numerator.bit_length() - fr.denominator.bit_length()
    while Fraction(2) ** e > fr:
        e -= 1
    while Fraction(2) ** (e + 1) <= fr:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    k = fr / ulp
    f = k.numerator // k.denominator
    rem = k - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f * ulp


def test_division_by_15_with_one_correction_is_correctly_rounded():
    r15 = np.float32(1) / np.float32(15)
    assert float(r15).hex() == "0x1.1111120000000p-4"            # the kernel's constant
    R = int(float(r15) * 2.0 ** 27)                                # r15 = R 2^-27, R < 2^24
    assert R * 2.0 ** -27 == float(r15) and 2 ** 23 <= R < 2 ** 24
    X = np.arange(2 ** 23, 2 ** 24, dtype=np.int64)                # d = X 2^-23 in [1, 2)
    P = X * R                                                      # d r15 = P 2^-50, exact
    nb = np.floor(np.log2(P.astype(np.float64))).astype(np.int64)
    nb = np.where((np.int64(1) << (nb + 1)) <= P, nb + 1, nb)
    nb = np.where((np.int64(1) << nb) > P, nb - 1, nb)
    sh = nb - 23
    Q0 = _rn_shift(P, sh)                                          # q0 = Q0 2^(sh - 50)
    carry = Q0 >= (np.int64(1) << 24)
    Q0 = np.where(carry, Q0 >> 1, Q0)
    sh = np.where(carry, sh + 1, sh)
    E = (X << 27) - 15 * (Q0 << sh)                                # e = E 2^-50, exact
    C = E * R                                                      # e r15 = C 2^-77
    lsb = sh + 27                                                  # q0's ulp = 2^lsb units
    k = C >> lsb
    rem = C - (k << lsb)
    half = np.int64(1) << (lsb - 1)
    Q1 = Q0 + k + ((rem > half) | ((rem == half) & (((Q0 + k) & 1) == 1)))
    num = X << (27 - sh)                                           # d / 15 in q0's ulps = num / 15
    kq = num // 15
    rq = num - kq * 15
    Qc = kq + ((2 * rq > 15) | ((2 * rq == 15) & ((kq & 1) == 1)))
    # the correction changes the answer where the plain product is wrong ...
    assert np.count_nonzero(Q0 != Qc) > 10 ** 6
    # ... and is right for every significand (a quotient that lands on a binade edge is checked
    # with exact rationals instead of the fixed-ulp integers)
    edge = (Q1 >= (1 << 24)) | (Q1 < (1 << 23)) | (Qc >= (1 << 24))
    assert np.count_nonzero(edge) < 100
    assert np.array_equal(Q1[~edge], Qc[~edge])
    rf = Fraction(float(r15))
    for i in np.nonzero(edge)[0]:
        d = Fraction(int(X[i]), 2 ** 23)
        q0 = _rn32(d * rf)
        assert _rn32(q0 + (d - 15 * q0) * rf) == _rn32(d / 15)
