"""The channel mean's definition rounds twice, mu = fp32(fp64(S) * 2^-24 / Nk);
the GPU kernels instead round once, to the fp32 nearest S / Nk (integer long
division, no fp64).  This pins the fact that the two are equal whenever
|S| < 2^53 and Nk < 2^24 (the oracle asserts the first; the library limits
the second), on random and on adversarial cases: quotients within a few
units of an fp32 rounding midpoint, in every magnitude range."""
from fractions import Fraction

import numpy as np


def rn24_exact(A: int, N: int) -> np.float32:
    """The fp32 nearest A / N (ties to even), from exact rational arithmetic."""
    q = Fraction(A, N)
    if q == 0:
        return np.float32(0.0)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    k = q / ulp
    fl = k.numerator // k.denominator
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return np.float32(float(fl * ulp))


def via_fp64(A: int, N: int) -> np.float32:
    return np.float32(np.float64(A) / np.float64(N))


def test_single_rounding_equals_fp64_route():
    rng = np.random.default_rng(5)
    cases = []
    for _ in range(4000):
        N = int(rng.integers(1, 2 ** 24))
        A = int(rng.integers(0, 2 ** 53))
        cases.append((A, N))
    # quotients next to fp32 midpoints b = (2k+1) 2^(e-24): A = N b + d
    for e in range(-20, 53):
        for _ in range(60):
            N = int(rng.integers(1, 2 ** 24)) if rng.random() < 0.5 else int(rng.integers(1, 64))
            k = int(rng.integers(2 ** 23, 2 ** 24))
            b = Fraction(2 * k + 1) * Fraction(2) ** (e - 24)
            base = N * b
            for d in (-2, -1, 0, 1, 2):
                A = int(base) + d if base.denominator == 1 else int(base) + d
                if 0 < A < 2 ** 53:
                    cases.append((A, N))
    for A, N in cases:
        assert rn24_exact(A, N) == via_fp64(A, N), (A, N)
