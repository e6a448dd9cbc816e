"""The arithmetic of the INT4 x FP8 kernel's zero point, checked on the host.

The kernel applies a group's zero point on the tensor cores:
    z 2^-9 * xs = sum_j (sign(I) u_j 2^a_j) * (z 2^b_j),  I = 512 xs,
where xs is the group's sum of e4m3 activation codes (a multiple of 2^-9 below
2^16 in magnitude), u_j are the base-16 digits of |I| (seven of them) and
a_j + b_j = 4j - 18. The identity needs both factors of every term to be e4m3
numbers, exactly, for every digit and every zero point, and the seven digits to
cover every I the activations can produce. Both are checked here with the e4m3
format as the FP8 oracle defines it (float8_e4m3fn: bias 7, subnormals m 2^-9,
largest finite 448). The exponents are the kernel's (w4a8_kernel.cu,
f8_digit_a / f8_digit_b), restated.
"""
import numpy as np

from oracle import fp8_oracle as f8

DIGITS = 7


def digit_a(j):
    return 4 * j - 9 if j < 4 else 4


def digit_b(j):
    return 4 * j - 18 - digit_a(j)


def is_e4m3(v):
    v = np.asarray(v, dtype=np.float64)
    return np.array_equal(f8.e4m3_decode(f8.e4m3_round(v)), v)


def test_every_factor_is_an_e4m3_number():
    u = np.arange(16, dtype=np.float64)
    for j in range(DIGITS):
        assert digit_a(j) + digit_b(j) == 4 * j - 18
        for sign in (1.0, -1.0):
            assert is_e4m3(sign * u * 2.0 ** digit_a(j)), j
            assert is_e4m3(-sign * u * 2.0 ** digit_b(j)), j


def test_largest_group_sum_fits_seven_digits():
    # 128 codes of magnitude 448 (the largest e4m3 number): I = 512 * 448 * 128
    largest = 512 * 448 * 128
    assert largest < 16 ** DIGITS
    # every code is a multiple of 2^-9, so I is an integer
    codes = f8.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = codes[np.isfinite(codes)]
    assert np.all(np.equal(np.mod(finite * 512, 1), 0))


def zero_point_term(I, z):
    """sum_j (sign(I) u_j 2^a_j) * (-z 2^b_j), each product and the sum exact in fp64."""
    u = abs(int(I))
    sign = -1.0 if I < 0 else 1.0
    total = 0.0
    for j in range(DIGITS):
        a = sign * ((u >> (4 * j)) & 0xF) * 2.0 ** digit_a(j)
        b = -float(z) * 2.0 ** digit_b(j)
        total += a * b
    return total


def test_digits_reproduce_the_zero_point_exactly():
    rng = np.random.default_rng(7)
    largest = 512 * 448 * 128
    values = [0, 1, -1, 15, 16, -255, 4095, 65536, largest, -largest, largest - 1]
    values += [int(v) for v in rng.integers(-largest, largest + 1, size=2000)]
    for I in values:
        for z in range(16):
            # -z 2^-9 xs = -z 2^-18 I, exact in fp64 (at most 29 significant bits)
            assert zero_point_term(I, z) == -z * 2.0 ** -18 * I, (I, z)


def test_a_dropped_digit_is_caught():
    # a planted mistake: six digits instead of seven loses the top one
    I = 512 * 448 * 128
    u = abs(I)
    six = sum(((u >> (4 * j)) & 0xF) * 16 ** j for j in range(6))
    assert six != u
