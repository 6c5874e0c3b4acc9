"""The E4M3 quantising append's division, checked in exact arithmetic on the CPU.

`append_e4m3_kernel` (decode_context_mla_gb300/csrc/relayout.cu) forms each quotient x / scale
as Markstein's correction of a reciprocal product: y = RN(1 / scale), q = RN(x y),
r = RN(x - scale q) and qc = RN(q + r y) (two FMAs); where qc lies within one binary32 step of
a point at which rounding to E4M3 changes direction, it takes the IEEE division instead.  Here
every step is evaluated exactly with rationals and rounded to binary32 by hand, and two claims
are checked on random pairs of the shapes the kernel meets (bf16 values over the row's scale
amax / 448) and on constructed hard cases (quotients at E4M3 midpoints and next to binary32
midpoints): qc is RN(x / scale) or a neighbour of it, and the E4M3 code the kernel stores is
the one the correctly rounded quotient gives.  A planted mistake (no correction step, no
guard) must be caught.
"""
import random
from fractions import Fraction

import numpy as np

import oracle as O


def rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value (ties to even), subnormals included."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1                                   # now 2^e <= a < 2^(e + 1)
    e = max(e, -126)                             # subnormals share the last exponent
    unit = Fraction(2) ** (e - 23)
    m = a / unit
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    assert fl <= 2 ** 24 and e <= 127
    return s * fl * unit


def step32(v: Fraction) -> Fraction:
    """The binary32 spacing at v (v a normal binary32 value)."""
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    return Fraction(2) ** (max(e, -126) - 23)


def near_e4m3_midpoint(v: Fraction) -> bool:
    """The kernel's test, on the binary32 bits of v."""
    u = int(np.float32(float(v)).view(np.uint32)) & 0x7FFFFFFF
    e = (u >> 23) - 127
    if e < -10:
        return False
    drop = 20 if e >= -6 else 14 - e
    sig = (u & 0x7FFFFF) | 0x800000
    low, half = sig & ((1 << drop) - 1), 1 << (drop - 1)
    return low + 1 >= half and low <= half + 1


def kernel_quotient(a: Fraction, b: Fraction, mistake=False):
    """(qc, the value the kernel converts) for x = a, scale = b."""
    y = rn32(1 / b)
    q = rn32(a * y)
    if mistake:
        return q, q
    r = rn32(a - b * q)
    qc = rn32(q + r * y)
    return qc, (rn32(a / b) if near_e4m3_midpoint(qc) else qc)


def code(v: Fraction) -> int:
    c = min(max(float(v), -448.0), 448.0)
    return int(O.round_to_e4m3(np.array([c]))[0])


def bf16(v: float) -> Fraction:
    b = np.float32(v).view(np.uint32) & np.uint32(0xFFFF0000)
    return Fraction(float(np.uint32(b).view(np.float32)))


def cases(seed=7, rows=60, per_row=60):
    rng = random.Random(seed)
    for _ in range(rows):
        xs = [bf16(rng.gauss(0, 1) * 2.0 ** rng.randint(-40, 40)) for _ in range(per_row)]
        amax = max(abs(x) for x in xs)
        if amax == 0:
            continue
        scale = rn32(amax / 448)
        if scale < Fraction(2) ** -126:          # a subnormal scale takes the IEEE division
            continue
        for x in xs:
            yield x, scale
    # quotients exactly at E4M3 midpoints (and one binary32 step either side), over scales
    # that are not powers of two
    mids = [Fraction(17, 16), Fraction(19, 16), Fraction(17, 8), Fraction(9, 32), Fraction(13),
            Fraction(104), Fraction(432), Fraction(3, 1024), Fraction(5, 1024), Fraction(1, 1024)]
    for s in (Fraction(3), Fraction(5), Fraction(7, 8), Fraction(11, 64), Fraction(13, 4096)):
        for m in mids:
            for d in (-1, 0, 1):
                v = m + d * step32(m)
                x = rn32(v * s)
                yield x, s
                yield -x, s
    # quotients next to binary32 midpoints: x = RN((k + 1/2) step * s) for odd-ish scales
    for _ in range(2000):
        s = rn32(Fraction(rng.randint(2 ** 23, 2 ** 24 - 1), 2 ** rng.randint(20, 40)))
        k = rng.randint(2 ** 23, 2 ** 24 - 1)
        m = (k + Fraction(1, 2)) * Fraction(2) ** rng.randint(-30, -15)
        yield rn32(m * s), s


def test_quotient_is_faithful_and_the_code_is_the_correctly_rounded_one():
    n = 0
    for a, b in cases():
        exact = rn32(a / b)
        qc, used = kernel_quotient(a, b)
        assert abs(qc - exact) <= step32(exact), (a, b)
        assert code(used) == code(exact), (a, b)
        n += 1
    assert n > 5000


def test_model_catches_a_missing_correction():
    assert any(code(kernel_quotient(a, b, mistake=True)[1]) != code(rn32(a / b)) for a, b in cases())
