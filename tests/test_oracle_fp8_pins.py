"""Pins for the INT4 x FP8 oracle (oracle/fp8_oracle.py) against the e4m3
format's published facts, torch's own float8_e4m3fn conversion, structural
invariants and reductions to the W4A16 oracle. The last tests plant mistakes in
copies of its functions and check that a pin catches them."""
import numpy as np
import pytest

import oracle
import synth
from oracle import fp8_oracle as f8

ALL = np.arange(256, dtype=np.uint8)


def check_decode(decode):
    v = decode(ALL)
    # the format's fixed points: 1.0, the smallest subnormal and normal, the
    # largest finite value, and the two NaN codes
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert set(np.flatnonzero(np.isnan(v)).tolist()) == {0x7F, 0xFF}
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # codes ascend with value
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign bit only flips the sign
    # spacing: 2^-9 through the subnormals and the first binade, then doubling per binade
    gaps = np.diff(pos)
    for e in range(16):
        lo, hi = 8 * e, min(8 * e + 8, 0x7E)  # the gaps after each code of binade e
        step = 2.0 ** (max(e, 1) - 10)
        assert np.all(gaps[lo:hi] == step), e


def test_e4m3_decode_facts():
    check_decode(f8.e4m3_decode)


def test_e4m3_decode_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    t = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = f8.e4m3_decode(ALL)
    fin = ~np.isnan(t)
    assert np.array_equal(np.isnan(mine), ~fin)
    assert np.array_equal(mine[fin], t[fin])


def check_round(round_fn):
    grid = f8.e4m3_decode(ALL[:0x7F])
    # every finite value rounds to itself (either sign)
    assert np.array_equal(f8.e4m3_decode(round_fn(grid)), grid)
    assert np.array_equal(f8.e4m3_decode(round_fn(-grid[1:])), -grid[1:])
    # midpoints go to the neighbour with the even code; just off them, to the nearer
    mids = (grid[:-1] + grid[1:]) / 2
    got = round_fn(mids).astype(np.int64)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))
    eps = np.diff(grid) * 1e-3
    assert np.array_equal(round_fn(mids - eps).astype(np.int64), lo)
    assert np.array_equal(round_fn(mids + eps).astype(np.int64), lo + 1)
    # saturation at the largest finite value
    assert f8.e4m3_decode(round_fn(np.array([449.0, 1e6, -1e6]))).tolist() == [448.0, 448.0, -448.0]


def test_e4m3_round():
    check_round(f8.e4m3_round)


def test_e4m3_round_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    x = np.random.default_rng(61).standard_normal(20000) * np.exp2(
        np.random.default_rng(62).integers(-12, 8, 20000))
    x = x[np.abs(x) <= 440.0]
    x32 = x.astype(np.float32)  # torch converts from fp32; compare on the fp32 values
    t = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = f8.e4m3_round(x32.astype(np.float64))
    # both round to nearest even; compare values (torch may keep -0)
    assert np.array_equal(f8.e4m3_decode(mine), f8.e4m3_decode(t))


def test_activation_quantisation_in_fp32_matches_torch():
    """The per-tensor quantisation takes its decisions in fp32: s_x is the fp32
    quotient max|x| / 448 and every code is the e4m3 rounding of the fp32
    quotient x / s_x, as torch computes them (fp32 tensors, float8_e4m3fn)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    xb = synth.make_custom_x(67, 16, 512, "bf16")
    codes, s_x = f8.quantize_act_per_tensor(oracle.half_bits_to_f64(xb, "bf16"))
    xt = torch.from_numpy(synth.bits_to_f32(xb, "bf16"))
    st = xt.abs().max() / torch.tensor(448.0, dtype=torch.float32)
    assert np.float32(s_x) == st.item()
    q = xt / st
    keep = (q.abs() < 448.0).numpy()  # torch does not saturate; compare inside the range
    t = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f8.e4m3_decode(codes)[keep], f8.e4m3_decode(t)[keep])
    # the decision differs from an fp64 one somewhere on a large enough input
    # only through the quotients' rounding: both lie within one e4m3 step
    q64 = oracle.half_bits_to_f64(xb, "bf16") / (np.max(np.abs(oracle.half_bits_to_f64(xb, "bf16"))) / 448.0)
    assert np.max(np.abs(f8.e4m3_decode(codes) - f8.e4m3_decode(f8.e4m3_round(q64)))) <= 32.0


def test_int4_weights_in_e4m3_are_exact():
    """(q - z) * 2^-9 is exact in e4m3 for every difference of two 4-bit codes,
    and with the scale times 512 it gives W = (q - z) * s exactly."""
    v = np.arange(-15, 16)
    w8 = f8.e4m3_decode(f8.int4_diff_to_e4m3(v))
    assert np.array_equal(w8, v * 2.0 ** -9)
    s = np.array([0.0123, 3.5, 1e-3])
    assert np.array_equal(w8[:, None] * (512.0 * s)[None, :], v[:, None] * s[None, :])
    with pytest.raises(ValueError):
        f8.int4_diff_to_e4m3(np.array([16]))


def _grid_x(rng, M, K, j, dtype):
    """x on the e4m3 grid times 2^j, with max |x| = 448 * 2^j: per-tensor
    quantisation of it is exact."""
    grid = f8.e4m3_decode(ALL[:0x7F])
    idx = rng.integers(0, 0x7F, (M, K))
    sign = rng.choice([-1.0, 1.0], (M, K))
    x = sign * grid[idx] * 2.0 ** j
    x[0, 0] = 448.0 * 2.0 ** j
    return synth.f32_to_bits(x.astype(np.float32), dtype)


def check_reduces_to_w4a16(ref_fn):
    for dtype, j in (("bf16", -8), ("fp16", -9), ("bf16", 0)):
        L = synth.make_custom_layer([63, j + 16], 256, 48, group=128, dtype=dtype)
        x = _grid_x(np.random.default_rng([64, -j]), 3, 256, j, dtype)
        assert np.array_equal(
            ref_fn(x, L.qweight, L.qzeros, L.scales, 128, dtype),
            oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, dtype, "awq"))


def test_w4a8_reduces_to_w4a16_on_exact_inputs():
    check_reduces_to_w4a16(f8.reference_y_w4a8)


def test_w4a8_error_bound_and_scale_invariance():
    """On random x the only difference from the W4A16 result is the rounding
    of x: |y8 - y16| <= sum_k |x - x8| |W|, with |x - x8| at most half an e4m3
    step. Scaling x by a power of two scales y by the same power exactly."""
    K, N = 512, 64
    L = synth.make_custom_layer(65, K, N, group=128, dtype="bf16")
    x = synth.make_custom_x(66, 4, K, "bf16")
    y8 = f8.reference_y_w4a8(x, L.qweight, L.qzeros, L.scales, 128, "bf16")
    y16 = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "bf16", "awq")
    q, z, s = oracle.layer_codes(L.qweight, L.qzeros, L.scales, "bf16", "awq")
    W = np.abs(oracle.dequant(q, z, s, oracle.group_of_rows(K, 128)).astype(np.float64))
    xv = oracle.half_bits_to_f64(x, "bf16")
    s_x = np.max(np.abs(xv)) / 448.0
    half_step = np.maximum(np.abs(xv) * 2.0 ** -4, s_x * 2.0 ** -10)
    bound = half_step @ W
    assert np.all(np.abs(y8 - y16) <= bound * (1 + 1e-9) + 1e-12)
    assert np.max(np.abs(y8 - y16)) > 0  # the rounding is really there
    x2 = synth.f32_to_bits((xv * 4.0).astype(np.float32), "bf16")
    assert np.array_equal(f8.reference_y_w4a8(x2, L.qweight, L.qzeros, L.scales, 128, "bf16"),
                          4.0 * y8)


# --------------------------------------------------------------------------- #
# Planted mistakes                                                              #
# --------------------------------------------------------------------------- #
def _decode_bias8(codes):
    return f8.e4m3_decode(codes) / 2.0  # planted: exponent bias 8 instead of 7


def _round_truncate(values):
    v = np.asarray(values, dtype=np.float64)
    grid = f8.e4m3_decode(ALL[:0x7F])
    a = np.minimum(np.abs(v), 448.0)
    mag = (np.searchsorted(grid, a, side="right") - 1).astype(np.uint8)  # planted: toward zero
    return np.where(v < 0, mag | 0x80, mag).astype(np.uint8)


def _ref_without_512(x_bits, qweight, qzeros, scales_bits, group, dtype):
    return f8.reference_y_w4a8(x_bits, qweight, qzeros, scales_bits, group, dtype) / 512.0


def test_mutant_decode_bias_is_caught():
    with pytest.raises(AssertionError):
        check_decode(_decode_bias8)


def test_mutant_truncating_round_is_caught():
    with pytest.raises(AssertionError):
        check_round(_round_truncate)


def test_mutant_missing_scale_factor_is_caught():
    with pytest.raises(AssertionError):
        check_reduces_to_w4a16(_ref_without_512)
