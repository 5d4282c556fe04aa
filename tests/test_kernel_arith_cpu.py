"""Host-side proofs of the arithmetic shortcuts the kernels rely on (no GPU): the division-free
group step of the quantiser, and the integer form of the decode GEMV (byte planes and DP4A order,
exactness of the 16-bit block fixed point).

The group step of the asymmetric quantiser is fl32((hi - lo) / n) with n = 2^N - 1 levels (15,
7 or 3 for 4-, 3- and 2-bit codes). The kernels form it without a division: q0 = fl32(d * r)
with r = fl32(1/n), the remainder e = d - n q0 (exact, one FMA), and q1 = fl32(q0 + e * r) (one
FMA), Markstein's correction step. Whether that equals the correctly rounded quotient depends
only on d's significand (scaling d by 2^j scales every quantity by 2^j while the results stay
normal), so checking all 2^23 significands of one binade with exact integer arithmetic proves
it for every d whose quotient is a normal float.
"""

import pytest

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


KERNEL_RECIPROCALS = {15: "0x1.1111120000000p-4", 7: "0x1.24924a0000000p-3",
                      3: "0x1.5555560000000p-2"}


@pytest.mark.parametrize("n", [15, 7, 3])
def test_division_by_levels_with_one_correction_is_correctly_rounded(n):
    r = np.float32(1) / np.float32(n)
    assert float(r).hex() == KERNEL_RECIPROCALS[n]                  # the kernel's constant
    _, er = np.frexp(float(r))                                     # r in [2^(er-1), 2^er)
    sr = 24 - int(er)                                              # r = R 2^-sr, R < 2^24
    R = int(float(r) * 2.0 ** sr)
    assert R * 2.0 ** -sr == float(r) and 2 ** 23 <= R < 2 ** 24
    u = 23 + sr                                                    # unit 2^-u for d r and e
    X = np.arange(2 ** 23, 2 ** 24, dtype=np.int64)                # d = X 2^-23 in [1, 2)
    P = X * R                                                      # d r = P 2^-u, exact
    nb = np.floor(np.log2(P.astype(np.float64))).astype(np.int64)
    nb = np.where((np.int64(1) << (nb + 1)) <= P, nb + 1, nb)
    nb = np.where((np.int64(1) << nb) > P, nb - 1, nb)
    sh = nb - 23
    Q0 = _rn_shift(P, sh)                                          # q0 = Q0 2^(sh - u)
    carry = Q0 >= (np.int64(1) << 24)
    Q0 = np.where(carry, Q0 >> 1, Q0)
    sh = np.where(carry, sh + 1, sh)
    E = (X << sr) - n * (Q0 << sh)                                 # e = E 2^-u, exact
    C = E * R                                                      # e r = C 2^-(u + sr)
    lsb = sh + sr                                                  # q0's ulp = 2^lsb units
    k = C >> lsb
    rem = C - (k << lsb)
    half = np.int64(1) << (lsb - 1)
    Q1 = Q0 + k + ((rem > half) | ((rem == half) & (((Q0 + k) & 1) == 1)))
    num = X << (sr - sh)                                           # d / n in q0's ulps = num / n
    kq = num // n
    rq = num - kq * n
    Qc = kq + ((2 * rq > n) | ((2 * rq == n) & ((kq & 1) == 1)))
    # the correction changes the answer where the plain product is wrong ...
    assert np.count_nonzero(Q0 != Qc) > 10 ** 6
    # ... and is right for every significand (a quotient that lands on a binade edge is checked
    # with exact rationals instead of the fixed-ulp integers)
    edge = (Q1 >= (1 << 24)) | (Q1 < (1 << 23)) | (Qc >= (1 << 24))
    assert np.count_nonzero(edge) < 100
    assert np.array_equal(Q1[~edge], Qc[~edge])
    rf = Fraction(float(r))
    for i in np.nonzero(edge)[0]:
        d = Fraction(int(X[i]), 2 ** 23)
        q0 = _rn32(d * rf)
        assert _rn32(q0 + (d - n * q0) * rf) == _rn32(d / n)


# ---------------------------------------------------------------- decode GEMV integer form

def _byte_perm(x, y, s):
    """PTX prmt (default mode): byte i of the result is byte (s >> 4i) & 7 of {y, x}."""
    b = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    return sum(b[(s >> (4 * i)) & 7] << (8 * i) for i in range(4))


def _planes(xi8):
    """The four byte planes of one packed word (channels 8w .. 8w+7), as the kernel builds them."""
    u = [int(v) & 0xFFFFFFFF for v in xi8]
    le = _byte_perm(_byte_perm(u[0], u[2], 0x0040), _byte_perm(u[4], u[6], 0x0040), 0x5410)
    lo = _byte_perm(_byte_perm(u[1], u[3], 0x0040), _byte_perm(u[5], u[7], 0x0040), 0x5410)
    he = _byte_perm(_byte_perm(u[0], u[2], 0x0051), _byte_perm(u[4], u[6], 0x0051), 0x5410)
    ho = _byte_perm(_byte_perm(u[1], u[3], 0x0051), _byte_perm(u[5], u[7], 0x0051), 0x5410)
    return le, lo, he, ho


def _dp4a(a, b, c, b_signed):
    sb = [((b >> (8 * i)) & 0xFF) for i in range(4)]
    if b_signed:
        sb = [v - 256 if v >= 128 else v for v in sb]
    return c + sum(((a >> (8 * i)) & 0xFF) * sb[i] for i in range(4))


def test_gemv_byte_planes_give_the_exact_integer_dot():
    """Codes of one 32-channel item (nibble i of word w is channel 8w + i) split into even and
    odd nibble bytes, activations x_int in [-2^15, 2^15) split into the planes above: four DP4A
    per word give sum q x_int, and hi * 256 + lo - z * sum x_int is sum (q - z) x_int exactly."""
    rng = np.random.Generator(np.random.PCG64(5))
    for _ in range(300):
        xi = rng.integers(-32767, 32768, 32)
        q = rng.integers(0, 16, 32)
        z = int(rng.integers(0, 16))
        lo = hi = 0
        for w in range(4):
            word = sum(int(q[8 * w + i]) << (4 * i) for i in range(8))
            ev, od = word & 0x0F0F0F0F, (word >> 4) & 0x0F0F0F0F
            le, lo_p, he, ho = _planes(xi[8 * w: 8 * w + 8])
            lo = _dp4a(od, lo_p, _dp4a(ev, le, lo, False), False)
            hi = _dp4a(od, ho, _dp4a(ev, he, hi, True), True)
        assert hi * 256 + lo - z * int(xi.sum()) == int(((q - z) * xi).sum())


def test_fixed_point_is_exact_within_five_binades_of_the_block_max():
    """x~ = x_int 2^(e - 15) with max|x~| < 2^e: every fp16 x~ with |x~| >= 2^(e - 5) times
    2^(15 - e) is an integer (its 11-bit significand ends at or above 2^(e - 15)), so only
    smaller activations are rounded; and |x_int| stays below 2^15."""
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)   # finite >= 0
    h = h[h > 0]
    for e in range(-10, 17):
        blk = h[h < 2.0 ** e]
        big = blk[blk >= 2.0 ** (e - 5)]
        scaled = big * 2.0 ** (15 - e)
        assert np.all(scaled == np.rint(scaled)) and np.all(scaled < 2 ** 15)


# ---------------------------------------------------------------- residual code decisions

def _rn32_signed(fr: Fraction) -> Fraction:
    if fr == 0:
        return Fraction(0)
    return _rn32(fr) if fr > 0 else -_rn32(-fr)


def _rint_even(fr: Fraction) -> int:
    f = fr.numerator // fr.denominator
    rem = fr - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def test_residual_shifted_domain_codes_equal_the_quotient_rule():
    """rint(fl32(w' / step)) without a division, both ways the kernels take it (r = fl32(1/step),
    kM = 1.5 2^23): the residual forms u = fl32(w' r + kM) in one FMA and checks
    fl32(w' r + (kM - u)); the pack kernel does the same against C = kM + z for the group's zero
    point z (an integer, so the code comes out as u - kM); the plain form rounds t = fl32(w' r)
    with two adds against kM and checks |t - rint(t)|. The margin is 1/2 - 2^-17; past it every
    form takes the IEEE quotient. In exact arithmetic, on quotients concentrated near the
    rounding boundaries, all give the defined integer."""
    kM = Fraction(3 * 2 ** 22)
    margin = Fraction(1, 2) - Fraction(1, 2 ** 17)
    rng = np.random.Generator(np.random.PCG64(9))
    n_edge = n_fast_wrong = 0
    for i in range(4000):
        step = _rn32_signed(Fraction(float(np.float32(np.exp(rng.uniform(-9, 3))))))
        k = int(rng.integers(-15, 16))
        if i % 2:
            q = Fraction(k) + Fraction(1, 2) + Fraction(int(rng.integers(-2 ** 12, 2 ** 12)), 2 ** 28)
        else:
            q = Fraction(float(rng.uniform(-15.4, 15.4)))
        wp = _rn32_signed(q * step)                      # a representable w' near that quotient
        want = _rint_even(_rn32_signed(wp / step))
        r = _rn32_signed(1 / step)
        u = _rn32_signed(wp * r + kM)
        e = _rn32_signed(wp * r + (kM - u))
        n_fast_wrong += int(u - kM) != want
        if abs(e) >= margin:
            n_edge += 1
            got = _rint_even(_rn32_signed(wp / step))
        else:
            got = int(u - kM)
        assert got == want, (float(wp), float(step))
        z = int(rng.integers(0, 16))                    # the pack kernel's shifted form
        c = kM + z
        up = _rn32_signed(wp * r + c)
        ep = _rn32_signed(wp * r + (c - up))
        got_shift = _rint_even(_rn32_signed(wp / step)) if abs(ep) >= margin else int(up - c)
        assert got_shift == want, (float(wp), float(step), z)
        t = _rn32_signed(wp * r)                        # the plain form
        rt = _rn32_signed(_rn32_signed(t + kM) - kM)
        got_pack = _rint_even(_rn32_signed(wp / step)) if abs(_rn32_signed(t - rt)) >= margin \
            else int(rt)
        assert got_pack == want, (float(wp), float(step))
    # the near-boundary branch was exercised, and the samples reach quotients where the fast
    # path alone would pick the wrong integer
    assert n_edge > 0 and n_fast_wrong > 0


def _clamp(v, lo, hi):
    return max(lo, min(hi, v))


@pytest.mark.parametrize("bits,symmetric", [(4, False), (4, True), (3, False), (2, True)])
def test_clip_near_tie_test_on_the_clamped_code(bits, symmetric):
    """The clipping search decides its codes with the fast rounding nq = -rint(w' rcp) and falls
    back to IEEE division only where min |g^2 - 1/4| <= 2^-16, g = w' rcp + clamp(nq): the
    remainder against the CLAMPED code. The rounding rule (rint_quotient) leaves the fast integer
    and the IEEE one different only where the fast remainder f = w' rcp + nq has |f| >= 1/2 -
    2^-17, and then by one step toward f's side. Checked here in exact rationals, over every
    clamp range the quantisers use, codes up to four steps past either end and remainders
    across [-1/2, 1/2] concentrated at both ends: wherever the other rounding would give a
    different CLAMPED code the test fires, and it never fires for weights two or more steps
    beyond the range (such as a group's largest magnitude under ratio 0.6, exactly 12.5 steps
    out, which the unclamped test would send down the slow path)."""
    half = 2 ** (bits - 1)
    if symmetric:   # code - zero in [-2^(N-1), 2^(N-1) - 1]: -(code - zero) in [1 - half, half]
        ranges = [(1 - half, half)]
    else:           # codes 0 .. 2^N - 1, zero point z in that range
        qmax = 2 ** bits - 1
        ranges = [(z - qmax, z) for z in range(qmax + 1)]
    eps = Fraction(1, 2 ** 17)
    fs = [Fraction(1, 2) - eps * k / 4 for k in range(0, 9)] + [Fraction(1, 4), Fraction(0)]
    fs = fs + [-f for f in fs]
    thresh = Fraction(1, 2 ** 16)
    for nlo, nhi in ranges:
        for nq in range(nlo - 4, nhi + 5):
            nc = _clamp(nq, nlo, nhi)
            for f in fs:
                x = -nq + f                      # w' rcp, with nq = -rint(x) the fast decision
                g = x + nc
                fires = abs(g * g - Fraction(1, 4)) <= thresh
                if abs(f) >= Fraction(1, 2) - eps:
                    # the IEEE rounding may take the neighbour on f's side
                    nq_other = nq - 1 if f > 0 else nq + 1
                    if _clamp(nq_other, nlo, nhi) != nc:
                        assert fires, (nlo, nhi, nq, f)
                if nq >= nhi + 2 or nq <= nlo - 2:
                    assert not fires, (nlo, nhi, nq, f)
