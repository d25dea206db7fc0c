"""The integer and floating-point rewrites the correlation kernels make of the
coefficient (The CUDA Handbook, chapter 15: the per-shift sums of Listing 15-5
combined with the box sums of section 15.8), checked exactly on the CPU.  No
kernel runs here; each test restates one rewrite with numpy's wrapping
integers or emulated float32 roundings and holds it to the exact int64 value
at the extremes that decide it.

- Centered products (the Toeplitz and transform kernels accumulate
  C = sum (I - 128)(T - 128)):  SumIT = C + 128 SumI + 128 SumT - 16384 N,
  exact in wrapping 32-bit arithmetic because SumIT < 2^32.
- 32-bit coefficient terms (the dp4a kernel for N <= 363 pixels):
  N SumIT - SumI SumT and N SumI2 - SumI^2 are N^2 times a covariance or a
  variance of values in 0..255, so at most N^2 * 127.5^2 < 2^31 in
  magnitude; wrapping 32-bit products give them exactly.  At N = 364 the
  bound is passed.
- The bank kernel's four-operation fp32 numerator (one exact group, at most
  258 pixels): p2 = fl(SumI SumT), e2 = fma(SumI, SumT, -p2) (its exact
  error), num = fl(fma(N, SumIT, -p2) - e2), within a few units in the last
  place of the exact numerator, so the coefficient is within 1e-6.
- The bounds behind the kernels' integer and fp32 widths (the largest width
  and group size checked one step past the limit too) and the transform
  kernel's prime and roots of unity.
"""
import numpy as np
import pytest

U32 = np.uint32


def window_sums(I, T):
    I = I.astype(np.int64)
    T = T.astype(np.int64)
    return int(I.sum()), int((I * I).sum()), int((I * T).sum()), int(T.sum())


def extreme_windows(rng, N):
    """Windows and templates that put the covariance and the variance at or
    near their bounds: half 0 / half 255 patterns, constant blocks, and
    random pixels."""
    half = np.zeros(N, np.uint8)
    half[: N // 2] = 255
    out = [(half, half), (half, 255 - half), (np.full(N, 255, np.uint8), np.full(N, 255, np.uint8)),
           (np.zeros(N, np.uint8), np.full(N, 255, np.uint8))]
    for _ in range(20):
        out.append((rng.integers(0, 256, N).astype(np.uint8), rng.integers(0, 256, N).astype(np.uint8)))
    return out


@pytest.mark.parametrize("N", [1, 2, 16, 256, 363, 4096, 30000])
def test_centered_products_give_sum_it_in_wrapping_32_bits(N):
    rng = np.random.default_rng(N)
    for I, T in extreme_windows(rng, N):
        sI, _, sIT, sT = window_sums(I, T)
        C = int(((I.astype(np.int64) - 128) * (T.astype(np.int64) - 128)).sum())
        assert C + 128 * sI + 128 * sT - 16384 * N == sIT
        # the kernels' form: C as a 32-bit word, cT = 128 SumT - 16384 N
        with np.errstate(over="ignore"):
            cT = U32(128) * U32(sT) - U32(16384) * U32(N)
            got = U32(C & 0xFFFFFFFF) + U32(128) * U32(sI) + cT
        assert int(got) == sIT


@pytest.mark.parametrize("N", [1, 2, 3, 100, 256, 362, 363])
def test_32_bit_coefficient_terms_are_exact_up_to_363_pixels(N):
    rng = np.random.default_rng(1000 + N)
    for I, T in extreme_windows(rng, N):
        sI, sI2, sIT, sT = window_sums(I, T)
        num, vI = N * sIT - sI * sT, N * sI2 - sI * sI
        with np.errstate(over="ignore"):
            num32 = (U32(N) * U32(sIT) - U32(sI) * U32(sT)).astype(np.int32)
            vI32 = U32(N) * U32(sI2) - U32(sI) * U32(sI)
        assert int(num32) == num
        assert int(vI32) == vI
        assert abs(num) <= N * N * 127.5 ** 2 < 2 ** 31


def test_the_32_bit_bound_is_passed_at_364_pixels():
    N = 364
    half = np.zeros(N, np.uint8)
    half[: N // 2] = 255
    sI, sI2, sIT, sT = window_sums(half, half)
    num, vI = N * sIT - sI * sT, N * sI2 - sI * sI
    assert num == vI == N * N * 127.5 ** 2
    assert num >= 2 ** 31                        # no longer a positive int32
    with np.errstate(over="ignore"):
        num32 = (U32(N) * U32(sIT) - U32(sI) * U32(sT)).astype(np.int32)
    assert int(num32) != num


def f32(x):
    return np.float32(x)


def fma32(a, b, c):
    """fma in float32: a*b + c formed exactly in float64 (all operands here
    are integers and the product and the sum stay below 2^53, so both are
    exact there), then rounded once."""
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def bank_numerator(N, sI, sT, sIT):
    Nf, sIf, sTf, sitf = f32(N), f32(sI), f32(sT), f32(sIT)
    p2 = f32(sIf * sTf)
    e2 = fma32(sIf, sTf, -p2)
    return f32(fma32(Nf, sitf, -p2) - e2)


@pytest.mark.parametrize("wT,hT", [(16, 16), (1, 1), (3, 5), (16, 8), (2, 129), (258, 1), (8, 32)])
def test_bank_fp32_numerator_and_coefficient(wT, hT):
    N = wT * hT
    assert N * 255 * 255 < 2 ** 24                  # one exact fp32 group
    rng = np.random.default_rng(N * 7 + wT)
    cases = extreme_windows(rng, N)
    # near-zero numerators with large SumI * SumT: a window and a template
    # that differ by one pixel step around a bright level
    base = np.full(N, 200, np.uint8)
    bumped = base.copy()
    bumped[0] = 201
    cases += [(base, bumped), (bumped, base), (bumped, bumped)]
    for I, T in cases:
        sI, sI2, sIT, sT = window_sums(I, T)
        assert sIT < 2 ** 24 and sI < 2 ** 24 and sT < 2 ** 24
        num = N * sIT - sI * sT
        got = float(bank_numerator(N, sI, sT, sIT))
        # two roundings of values at most |num| + ulp(SumI * SumT) / 2
        bound = 2.0 ** -23 * abs(num) + 2.0 ** -47 * sI * sT + 1e-30
        assert abs(got - num) <= bound, (I[:4], T[:4], got, num)
        vI, vT = N * sI2 - sI * sI, N * int((T.astype(np.int64) ** 2).sum()) - sT * sT
        if vI > 0 and vT > 0:
            r_exact = num / np.sqrt(float(vI) * float(vT))
            r_f32 = np.float32(got) * np.float32(1.0 / np.sqrt(np.float64(vI))) * \
                np.float32(1.0 / np.sqrt(np.float64(vT)))
            assert abs(float(r_f32) - r_exact) <= 1e-6


def is_prime(n):
    if n < 2:
        return False
    d = 2
    while d * d <= n:
        if n % d == 0:
            return False
        d += 1
    return True


def test_exactness_bounds_the_kernels_rely_on():
    # table builder: a row's running sums in uint32 up to W = 66051 (the
    # largest width whose row of 255s squares to less than 2^32); the
    # look-back row words pack SumI in 25 bits and SumI2 in 32
    assert 66051 * 255 ** 2 < 2 ** 32 <= 66052 * 255 ** 2
    assert 66051 * 255 < 2 ** 25
    # look-back words hold a table value in 57 bits: the largest Q entry of
    # an image below 2^31 pixels
    assert (2 ** 31 - 1) * 255 ** 2 < 2 ** 57
    # dp4a numerator: SumIT in uint32 for templates up to 66051 pixels
    assert 66051 * 255 ** 2 < 2 ** 32
    # bank kernel: fp32 accumulation exact while a group has at most 258
    # pixels (every partial sum an integer below 2^24)
    assert 258 * 255 ** 2 < 2 ** 24 <= 259 * 255 ** 2
    # Toeplitz kernel: centered products |(I-128)(T-128)| <= 2^14, groups of
    # at most 1024 products stay within 2^24, where fp32 holds every integer
    assert 128 * 128 == 2 ** 14 and 1024 * 2 ** 14 == 2 ** 24
    assert float(np.float32(2 ** 24)) == 2 ** 24 and float(np.float32(2 ** 24 - 1)) == 2 ** 24 - 1
    # transform kernel: p = 119 * 2^23 + 1 is prime, 3 generates its
    # multiplicative group (so 256th roots of unity exist), and a centered
    # correlation of up to 30000 pixels is recovered from its residue
    p = 998244353
    assert p == 119 * 2 ** 23 + 1 and is_prime(p)
    assert all(pow(3, (p - 1) // q, p) != 1 for q in (2, 7, 17))     # p - 1 = 2^23 * 7 * 17
    w256 = pow(3, (p - 1) // 256, p)
    assert pow(w256, 256, p) == 1 and pow(w256, 128, p) == p - 1
    assert 2 * 2 ** 14 * 30000 < p
    assert 4 * p < 2 ** 32                                             # lazy residues in [0, 4p)
