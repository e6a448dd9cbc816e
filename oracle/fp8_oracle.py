"""CPU oracle for the INT4-weight x FP8-activation form of the layer: what the
tcgen05 kind::f8f6f4 kernel (w4a8_gemm) must compute.

TEST INFRASTRUCTURE ONLY, like the rest of `oracle/`: only the test suite, the
smoke check and the benchmark's CPU arm may import it; it shares no code with
the CUDA path.

What the pages say ("量化层加载:AWQ / GPTQ / Marlin / fp8", 边界与失败): when
Marlin's activation type is float8_e4m3fn, the 4-bit weights go through a
preprocessing op and the scales are multiplied by 512. The same page lists the
fp8 activation schemes of its Fp8Config (per-tensor / per-block, static /
dynamic). Everything else below is a reading, written out as the definition:

  * e4m3 ("float8_e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 holds the subnormals m * 2^-9; no infinities; the codes
    S.1111.111 are NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
  * Weights: v = q - z (an integer in [-15, 15]) is stored as the e4m3 number
    v * 2^-9, which is exact (|v| <= 7 subnormal, 8..15 the smallest binade),
    and the scale becomes 512 * s, so (v * 2^-9) * (512 * s) = (q - z) * s = W
    exactly: the "scales x 512".
  * Activations: dynamic per-tensor scaling, s_x = max|x| / 448 (1 when x is
    all zero), x8 = e4m3(x / s_x) rounded to nearest even and saturated at 448.
    The pages leave the precision of this step open; since it decides integer
    codes, it is taken in the kernel's precision: s_x = RN_fp32(max|x| / 448)
    and x / s_x as one fp32 division rounded to nearest (max|x| is exact in
    fp32, being an fp16 / bf16 value), then rounded to e4m3.
  * y[m, n] = s_x * sum_k x8[m, k] * W[k, n], in fp64 here.
"""
from __future__ import annotations

import numpy as np

from . import w4a16_oracle as core

E4M3_MAX = 448.0
E4M3_BIAS = 7


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 codes (uint8) -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = (1.0 + man / 8.0) * np.exp2(exp - E4M3_BIAS)
    subnormal = (man / 8.0) * np.exp2(1 - E4M3_BIAS)
    v = sign * np.where(exp == 0, subnormal, normal)
    return np.where((exp == 0xF) & (man == 0x7), np.nan, v)


def _finite_grid():
    """All finite non-negative e4m3 values, ascending, with their codes."""
    codes = np.arange(0x7F, dtype=np.uint8)  # 0x00 .. 0x7E
    return e4m3_decode(codes), codes


def e4m3_round(values) -> np.ndarray:
    """float64 -> nearest e4m3 code; ties to the even code (mantissa LSB 0);
    magnitudes above 448 saturate to 448. NaN input is not accepted."""
    v = np.asarray(values, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN has no e4m3 rounding here")
    grid, codes = _finite_grid()
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(grid, a, side="left")            # first grid value >= a
    hi = np.minimum(hi, len(grid) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    exact = grid[hi] == a
    pick_hi = np.where(exact, True,
                       np.where(d_hi < d_lo, True,
                                np.where(d_hi > d_lo, False, (codes[hi] & 1) == 0)))
    mag = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    neg = (v < 0) & (mag != 0)
    return np.where(neg, mag | 0x80, mag).astype(np.uint8)


def int4_diff_to_e4m3(v) -> np.ndarray:
    """v = q - z in [-15, 15] -> the e4m3 code of v * 2^-9 (exact)."""
    v = np.asarray(v, dtype=np.int64)
    if (np.abs(v) > 15).any():
        raise ValueError("q - z lies in [-15, 15]")
    return e4m3_round(v.astype(np.float64) * 2.0 ** -9)


def quantize_act_per_tensor(x: np.ndarray):
    """Dynamic per-tensor fp8 activations: (codes, s_x) with s_x = max|x|/448,
    both divisions in fp32 rounded to nearest (x holds fp16 / bf16 values, exact
    in fp32); s_x is returned as the fp32 value (in a float64)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    s_x = amax / np.float32(E4M3_MAX) if amax > 0 else np.float32(1.0)
    q = (x32 / s_x).astype(np.float64)
    return e4m3_round(q), float(s_x)


def reference_y_w4a8(x_bits, qweight, qzeros, scales_bits, group: int, dtype: str,
                     fmt: str = "awq") -> np.ndarray:
    """fp64 y of the INT4 x FP8 form: x (half bits of `dtype`) quantised per
    tensor to e4m3, W from the checkpoint words as in the W4A16 oracle, and the
    weights taken through their e4m3 form v * 2^-9 with the scales times 512."""
    q, z, s = core.layer_codes(qweight, qzeros, scales_bits, dtype, fmt)
    K, N = q.shape
    gk = core.group_of_rows(K, group)
    v = q.astype(np.int64) - z[gk].astype(np.int64)
    w8 = e4m3_decode(int4_diff_to_e4m3(v))                 # v * 2^-9
    W = w8 * (512.0 * s[gk])
    codes, s_x = quantize_act_per_tensor(core.half_bits_to_f64(x_bits, dtype))
    return s_x * core.gemm(e4m3_decode(codes), W)
