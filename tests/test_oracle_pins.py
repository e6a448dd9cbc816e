"""Pins for the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: the constants
and shapes the pages print (tests/golden/), the independent checkpoint writer in
`synth`, closed forms, invariants, and exact rational brute force on tiny inputs.
The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU) and check that these pins catch them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden_kv, read_golden_unpack

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------- #
# Constants and shapes the pages print                                          #
# --------------------------------------------------------------------------- #
def test_printed_constants():
    g = read_golden_kv("awq_format_constants.txt")
    assert list(oracle.REVERSE_AWQ_PACK_ORDER) == g["reverse_awq_pack_order"]
    assert oracle.PACK_FACTOR == g["pack_factor"][0] == 32 // 4
    assert list(oracle.SUPPORTED_GROUPS) == g["supported_groups"]


def check_golden_unpack(mod=oracle):
    for kind, word, codes in read_golden_unpack("unpack_examples.txt"):
        w = np.array([[np.uint32(word).view(np.int32)]])
        if kind == "awq":
            got = mod.unpack_awq(w)[0].tolist()
        else:
            got = mod.unpack_rows_std(w)[:, 0].tolist()
            got2 = mod.unpack_cols_std(w)[0].tolist()
            assert got2 == codes, (kind, hex(word), got2, codes)
        assert got == codes, (kind, hex(word), got, codes)


def test_golden_unpack_examples():
    check_golden_unpack()


def test_standard_bit_positions():
    # [AWQ] §5.1: the standard order puts index i at bit 4i.
    g = read_golden_kv("awq_format_constants.txt")
    for i, bit in enumerate(g["standard_bit_of_index"]):
        codes = np.zeros((8, 1), dtype=np.uint8)
        codes[i, 0] = 1
        assert int(oracle.pack_rows_std(codes)[0, 0]) == 1 << bit
        codes_c = np.zeros((1, 8), dtype=np.uint8)
        codes_c[0, i] = 1
        assert int(oracle.pack_cols_std(codes_c)[0, 0]) == 1 << bit


def test_tiny_shapes_match_printed():
    g = read_golden_kv("awq_format_constants.txt")
    L = synth.make_workload_layer(0, 0)
    assert list(L.qweight.shape) == g["tiny_qweight_shape"]
    assert list(L.qzeros.shape) == g["tiny_qzeros_shape"]
    assert list(L.scales.shape) == g["tiny_scales_shape"]
    qw_std, z_std = oracle.repack_awq_to_std(L.qweight, L.qzeros)
    assert list(qw_std.shape) == g["tiny_std_qweight_shape"]
    assert z_std.shape == L.qzeros.shape


# --------------------------------------------------------------------------- #
# Unpack: exhaustive single nibble, and round trips through the writer          #
# --------------------------------------------------------------------------- #
def check_awq_single_nibble(mod=oracle):
    for p in range(8):
        for v in range(16):
            w = np.array([[np.uint32(v << (4 * p)).view(np.int32)]])
            got = mod.unpack_awq(w)[0]
            expect = np.zeros(8, dtype=np.uint8)
            # column j holds nibble REV[j]; REV is the printed constant
            j = read_golden_kv("awq_format_constants.txt")["reverse_awq_pack_order"].index(p)
            expect[j] = v
            assert np.array_equal(got, expect), (p, v, got)


def test_awq_single_nibble_exhaustive():
    check_awq_single_nibble()


def test_unpack_inverts_writer_awq():
    L = synth.make_custom_layer(1, 512, 512, group=128, keep_codes=True)
    assert np.array_equal(oracle.unpack_awq(L.qweight), L.q)
    assert np.array_equal(oracle.unpack_awq(L.qzeros), L.z)


def test_unpack_inverts_writer_gptq():
    L = synth.make_custom_layer(2, 512, 256, group=64, fmt="gptq", act_order=True,
                                dtype="fp16", keep_codes=True)
    assert np.array_equal(oracle.unpack_rows_std(L.qweight), L.q)
    assert np.array_equal(oracle.unpack_cols_std(L.qzeros), L.z)


def test_random_word_round_trip():
    rng = np.random.default_rng(7)
    words = rng.integers(0, 2**32, size=(1000, 125), dtype=np.uint64).astype(np.uint32).view(np.int32)
    # AWQ: unpack, then repack with the writer's packer (an independent implementation)
    assert np.array_equal(synth._pack_awq(oracle.unpack_awq(words)), words)
    assert np.array_equal(oracle.pack_cols_std(oracle.unpack_cols_std(words)), words)
    assert np.array_equal(oracle.pack_rows_std(oracle.unpack_rows_std(words)), words)
    # the GPTQ writer's row packer inverts the oracle's row unpack
    assert np.array_equal(synth._pack_rows_std(oracle.unpack_rows_std(words)), words)


# --------------------------------------------------------------------------- #
# AWQ -> standard repack                                                        #
# --------------------------------------------------------------------------- #
def check_repack_matches_gptq_writer(mod=oracle):
    """Same codes written once as AWQ and once as GPTQ (two writer code paths)."""
    L = synth.make_custom_layer(3, 256, 128, group=64, keep_codes=True)
    qw_std, z_std = mod.repack_awq_to_std(L.qweight, L.qzeros)
    assert np.array_equal(qw_std, synth._pack_rows_std(L.q))
    assert np.array_equal(z_std, synth._pack_cols_std(L.z))


def test_repack_matches_gptq_writer():
    check_repack_matches_gptq_writer()


def test_repack_tiny_brute_force():
    # One bit at a time: the code at AWQ (k, n) must land at std row k//8, column n,
    # bits 4*(k%8) — checked on every position of a 16 x 16 layer.
    K, N = 16, 16
    for k in range(K):
        for n in range(N):
            codes = np.zeros((K, N), dtype=np.uint8)
            codes[k, n] = 0b1011
            qw_std, _ = oracle.repack_awq_to_std(synth._pack_awq(codes),
                                                  np.zeros((1, N // 8), np.int32))
            expect = np.zeros((K // 8, N), dtype=np.uint32)
            expect[k // 8, n] = 0b1011 << (4 * (k % 8))
            assert np.array_equal(qw_std.view(np.uint32), expect)


# --------------------------------------------------------------------------- #
# Tile layout (own format: bijection, round trip, scalar vs vectorised)         #
# --------------------------------------------------------------------------- #
def test_tile_pos_is_bijection():
    # 128 x 256: two whole column groups, so every word holds codes
    K, N = 128, 256
    seen = set()
    for k in range(K):
        for n in range(N):
            seen.add(oracle.tile_pos(k, n, K, N))
    assert len(seen) == K * N
    assert {w for w, _ in seen} == set(range(oracle.tile_words(K, N)))


def test_tile_padding_is_zero_and_injective():
    # 128 x 48: three of a group's eight tiles carry codes, the rest is zero padding
    K, N = 128, 48
    assert oracle.tile_words(K, N) == K * 128 // 8
    seen = {oracle.tile_pos(k, n, K, N) for k in range(K) for n in range(N)}
    assert len(seen) == K * N
    codes = np.full((K, N), 15, dtype=np.uint8)
    words = oracle.tile_pack(codes).view(np.uint32)
    used = {w for w, _ in seen}
    for w in range(len(words)):
        assert (words[w] != 0) == (w in used)


def test_tile_group_order():
    # atom (kb, nt) = ((nt // 8) * (K / 64) + kb) * 8 + nt % 8: the eight tiles of
    # a column group at one k-atom are adjacent, then the next k-atom follows
    K, N = 192, 272
    A = K // 64
    for kb in range(A):
        for nt in range(N // 16):
            w, _ = oracle.tile_pos(64 * kb, 16 * nt, K, N)
            assert w == (((nt // 8) * A + kb) * 8 + nt % 8) * 128
    assert oracle.tile_pos(64, 0, K, N)[0] == 8 * 128
    assert oracle.tile_pos(0, 16, K, N)[0] == 128
    assert oracle.tile_pos(0, 128, K, N)[0] == A * 8 * 128


def test_tile_pack_matches_tile_pos():
    K, N = 128, 32
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    words = oracle.tile_pack(codes).view(np.uint32)
    for k in range(K):
        for n in range(N):
            w, p = oracle.tile_pos(k, n, K, N)
            assert (int(words[w]) >> (4 * p)) & 0xF == codes[k, n]


def test_tile_round_trip():
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 16, size=(640, 272), dtype=np.uint8)
    assert np.array_equal(oracle.tile_unpack(oracle.tile_pack(codes), 640, 272), codes)


def test_tile_first_word_layout():
    # Word 0 of atom 0: column 0, rows 0..7, row r at nibble TILE_NIBBLE_ROW.index(r).
    codes = np.zeros((64, 16), dtype=np.uint8)
    codes[:8, 0] = np.arange(1, 9)
    w0 = int(oracle.tile_pack(codes).view(np.uint32)[0])
    assert [(w0 >> (4 * p)) & 0xF for p in range(8)] == [1, 3, 5, 7, 2, 4, 6, 8]
    # Word 1 of atom 0 holds column 8, word 2 rows 32..39 of column 0.
    codes[:] = 0
    codes[0, 8] = 9
    codes[32, 0] = 5
    w = oracle.tile_pack(codes).view(np.uint32)
    assert int(w[1]) & 0xF == 9 and int(w[2]) & 0xF == 5


# --------------------------------------------------------------------------- #
# Act-order permutation                                                         #
# --------------------------------------------------------------------------- #
def test_act_order_perm_brute_force():
    rng = np.random.default_rng(5)
    for K, g in ((256, 32), (512, 128), (96, 32)):
        gi = synth.act_order_gidx(rng, K, g)
        perm = oracle.act_order_perm(gi)
        brute = [k for _, k in sorted((int(gi[k]), k) for k in range(K))]
        assert perm.tolist() == brute
        assert oracle.gidx_is_regular(gi, g)
        # sorted rows give group j // g
        assert np.array_equal(gi[perm], np.arange(K) // g)


def test_gidx_regularity_detects_bad_counts():
    gi = np.repeat(np.arange(4), 32).astype(np.int32)
    assert oracle.gidx_is_regular(gi, 32)
    gi[0] = 1
    assert not oracle.gidx_is_regular(gi, 32)
    gi[0] = 7
    assert not oracle.gidx_is_regular(gi, 32)


# --------------------------------------------------------------------------- #
# Dequantisation                                                                #
# --------------------------------------------------------------------------- #
def test_dequant_closed_forms():
    K, N, g = 256, 16, 128
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    gk = oracle.group_of_rows(K, g)
    # q == z -> 0
    z = q[::g].copy()
    zz = np.repeat(z, g, axis=0)
    q_eq = zz.copy()
    # scales are half-precision values (the storage dtype), so (q - z) * s is exact
    s = rng.uniform(0.001, 0.1, size=(K // g, N)).astype(np.float16).astype(np.float64)
    assert np.all(oracle.dequant(q_eq, z, s, gk) == 0)
    # z == 0, s == 1 -> q
    W = oracle.dequant(q, np.zeros((K // g, N), np.uint8), np.ones((K // g, N)), gk)
    assert np.array_equal(W, q.astype(np.float32))
    # q=15, z=0 -> +15 s ; q=0, z=15 -> -15 s
    z15 = np.full((K // g, N), 15, np.uint8)
    W = oracle.dequant(np.zeros((K, N), np.uint8), z15, s, gk)
    assert np.array_equal(W.astype(np.float64), -15 * s[gk])
    W = oracle.dequant(np.full((K, N), 15, np.uint8), np.zeros_like(z15), s, gk)
    assert np.array_equal(W.astype(np.float64), 15 * s[gk])


def check_dequant_vs_writer(mod=oracle):
    """|W - w| <= s/2 wherever the writer's code was not clamped."""
    for dtype in ("fp16", "bf16"):
        L = synth.make_custom_layer(21, 512, 256, group=128, dtype=dtype, keep_codes=True,
                                    keep_float=True)
        q, z, s = mod.layer_codes(L.qweight, L.qzeros, L.scales, dtype, "awq")
        gk = mod.group_of_rows(512, 128)
        W = mod.dequant(q, z, s, gk).astype(np.float64)
        unclamped = (L.q > 0) & (L.q < 15)
        err = np.abs(W - L.w.astype(np.float64))
        bound = s[gk] * 0.5 * (1 + 1e-6)
        assert np.all(err[unclamped] <= bound[unclamped])
        # clamped codes are still within s/2 + the clamp distance; the bulk is unclamped
        assert unclamped.mean() > 0.95


def test_dequant_vs_writer():
    check_dequant_vs_writer()


def test_symmetric_checkpoint():
    """A symmetric checkpoint (no qzeros) reads as zero point 8 everywhere:
    code 8 dequantises to 0, codes 0 / 15 to -8 s / +7 s, and the whole-layer
    reference equals that of the same checkpoint with an explicit all-8 qzeros
    (packed by the writer) for both formats; the writer's symmetric codes stay
    within s/2 of the float weights wherever they are not clamped."""
    K, N, g = 256, 64, 128
    for fmt in ("awq", "gptq"):
        L = synth.make_custom_layer([22, fmt == "awq"], K, N, group=g, dtype="bf16", fmt=fmt,
                                    symmetric=True, keep_codes=True, keep_float=True)
        assert L.qzeros is None
        q, z, s = oracle.layer_codes(L.qweight, None, L.scales, "bf16", fmt)
        assert z.shape == (K // g, N) and np.all(z == 8)
        gk = oracle.group_of_rows(K, g)
        W = oracle.dequant(q, z, s, gk).astype(np.float64)
        assert np.array_equal(W[q == 8], np.zeros(int((q == 8).sum())))
        assert np.array_equal(W[q == 0], -8 * s[gk][q == 0])
        assert np.array_equal(W[q == 15], 7 * s[gk][q == 15])
        unclamped = (L.q > 0) & (L.q < 15)
        assert unclamped.mean() > 0.95
        assert np.all(np.abs(W - L.w)[unclamped] <= (s[gk] * 0.5 * (1 + 1e-6))[unclamped])
        eights = np.full((K // g, N), 8, np.uint8)
        qz = synth._pack_awq(eights) if fmt == "awq" else synth._pack_cols_std(eights)
        x = synth.make_custom_x([23], 3, K, "bf16")
        assert np.array_equal(oracle.reference_y(x, L.qweight, None, L.scales, g, "bf16", fmt),
                              oracle.reference_y(x, L.qweight, qz, L.scales, g, "bf16", fmt))


def test_reference_bias_closed_forms():
    """With x = 0 the reference is the bias itself; a zero bias changes nothing;
    the bias shifts every row by the same vector (on a column subset too)."""
    K, N = 256, 48
    L = synth.make_custom_layer([26], K, N, group=128, dtype="fp16")
    b = synth.f32_to_bits(np.random.default_rng(27).standard_normal(N).astype(np.float32), "fp16")
    bf = oracle.half_bits_to_f64(b, "fp16")
    zero_x = synth.f32_to_bits(np.zeros((2, K), np.float32), "fp16")
    assert np.array_equal(oracle.reference_y(zero_x, L.qweight, L.qzeros, L.scales, 128, "fp16",
                                             "awq", bias_bits=b), np.tile(bf, (2, 1)))
    x = synth.make_custom_x([28], 3, K, "fp16")
    plain = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "fp16", "awq")
    zb = synth.f32_to_bits(np.zeros(N, np.float32), "fp16")
    assert np.array_equal(oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "fp16", "awq",
                                             bias_bits=zb), plain)
    cols = np.array([3, 17, 40])
    with_b = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "fp16", "awq",
                                cols=cols, bias_bits=b)
    assert np.allclose(with_b - plain[:, cols], bf[cols][None, :], rtol=0, atol=1e-12)


def test_dequant_is_exact_in_fp32():
    # (q - z) * s for every q, z and many scales: fp32 result equals the exact rational.
    rng = np.random.default_rng(4)
    for dtype in ("fp16", "bf16"):
        sbits = rng.integers(0x0400 if dtype == "fp16" else 0x3800, 0x5800 if dtype == "fp16" else 0x4300,
                             size=64, dtype=np.uint16)
        s = oracle.half_bits_to_f64(sbits, dtype)
        for qq in range(16):
            for zz in range(16):
                v = oracle.dequant(np.full((1, 64), qq, np.uint8), np.full((1, 64), zz, np.uint8),
                                   s[None, :], np.zeros(1, np.int64))[0]
                for i in range(64):
                    assert Fraction(float(v[i])) == (qq - zz) * Fraction(float(s[i]))


def test_group_sizes_and_per_channel():
    K = 256
    assert np.array_equal(oracle.group_of_rows(K, 32), np.arange(K) // 32)
    assert np.array_equal(oracle.group_of_rows(K, -1), np.zeros(K))
    gi = np.arange(K)[::-1] // 64
    assert np.array_equal(oracle.group_of_rows(K, 64, gi), gi)


# --------------------------------------------------------------------------- #
# GEMM                                                                          #
# --------------------------------------------------------------------------- #
def check_gemm_exact_rational(mod=oracle):
    """Oracle y vs an exact rational sum computed from the writer's codes."""
    for (M, K, N, dtype, fmt, ao) in ((1, 128, 8, "fp16", "awq", False),
                                      (3, 256, 16, "bf16", "awq", False),
                                      (2, 256, 8, "fp16", "gptq", True)):
        L = synth.make_custom_layer([9, M, K, N], K, N, group=128 if not ao else 64,
                                    dtype=dtype, fmt=fmt, act_order=ao, keep_codes=True)
        x = synth.make_custom_x([10, M], M, K, dtype)
        y = mod.reference_y(x, L.qweight, L.qzeros, L.scales, L.group, dtype, fmt, g_idx=L.g_idx)
        xv = synth.bits_to_f32(x, dtype)
        sv = synth.bits_to_f32(L.scales, dtype)
        gk = (L.g_idx if ao else np.arange(K) // L.group)
        for m in range(M):
            for n in range(N):
                acc = Fraction(0)
                for k in range(K):
                    g = int(gk[k])
                    acc += Fraction(float(xv[m, k])) * (int(L.q[k, n]) - int(L.z[g, n])) * \
                        Fraction(float(sv[g, n]))
                assert abs(Fraction(float(y[m, n])) - acc) <= abs(acc) * Fraction(1, 2**50) + \
                    Fraction(1, 2**80), (m, n, float(y[m, n]), float(acc))


def test_gemm_exact_rational():
    check_gemm_exact_rational()


MOE_CASES = (
    # dtype, K, N, group, row offsets (E + 1)
    ("fp16", 128, 8, 64, [0, 2, 2, 5]),   # an expert without rows between two with rows
    ("bf16", 128, 16, 32, [0, 0, 3]),     # the first expert without rows
)


def _moe_case(dtype, K, N, group, off):
    E = len(off) - 1
    layers = [synth.make_custom_layer([51, e, K, N], K, N, group=group, dtype=dtype,
                                      keep_codes=True) for e in range(E)]
    x = synth.make_custom_x([52, K], off[-1], K, dtype)
    return layers, x


def check_moe_exact_rational(moe_fn):
    """The grouped reference vs exact rational sums from the writer's codes, each
    row's expert found by scanning the offsets."""
    for dtype, K, N, group, off in MOE_CASES:
        layers, x = _moe_case(dtype, K, N, group, off)
        y = moe_fn(x, [(L.qweight, L.qzeros, L.scales) for L in layers], off, group, dtype, "awq")
        assert y.shape == (off[-1], N)
        xv = synth.bits_to_f32(x, dtype)
        for m in range(off[-1]):
            e = next(i for i in range(len(layers)) if off[i] <= m < off[i + 1])
            L = layers[e]
            sv = synth.bits_to_f32(L.scales, dtype)
            for n in range(N):
                acc = Fraction(0)
                for k in range(K):
                    g = k // group
                    acc += Fraction(float(xv[m, k])) * (int(L.q[k, n]) - int(L.z[g, n])) * \
                        Fraction(float(sv[g, n]))
                assert abs(Fraction(float(y[m, n])) - acc) <= abs(acc) * Fraction(1, 2**50) + \
                    Fraction(1, 2**80), (m, n, e)


def test_moe_reference_exact_rational():
    check_moe_exact_rational(oracle.moe_reference_y)


def test_moe_reference_single_expert_is_plain_gemm():
    """One expert owning every row: the grouped GEMM is the plain one."""
    L = synth.make_custom_layer(53, 256, 48, group=128, dtype="bf16")
    x = synth.make_custom_x(54, 7, 256, "bf16")
    assert np.array_equal(
        oracle.moe_reference_y(x, [(L.qweight, L.qzeros, L.scales)], [0, 7], 128, "bf16", "awq"),
        oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "bf16", "awq"))


def test_moe_reference_rejects_bad_offsets():
    L = synth.make_custom_layer(55, 128, 8, group=64, dtype="fp16")
    x = synth.make_custom_x(56, 4, 128, "fp16")
    ex = [(L.qweight, L.qzeros, L.scales)] * 2
    for off in ([1, 2, 4], [0, 3, 2], [0, 2, 3], [0, 4]):
        with pytest.raises(ValueError):
            oracle.moe_reference_y(x, ex, off, 64, "fp16", "awq")


def test_gemm_one_hot_rows():
    L = synth.make_custom_layer(31, 256, 64, group=128, dtype="bf16")
    q, z, s = oracle.layer_codes(L.qweight, L.qzeros, L.scales, "bf16", "awq")
    W = oracle.dequant(q, z, s, oracle.group_of_rows(256, 128))
    for k in (0, 1, 127, 128, 255):
        x = np.zeros((1, 256), np.uint16)
        x[0, k] = 0x3F80  # bf16 1.0
        y = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "bf16", "awq")
        assert np.array_equal(y[0], W[k].astype(np.float64))


def test_act_order_identity_grouping_matches_plain():
    L = synth.make_custom_layer(41, 256, 64, group=64, dtype="fp16", fmt="gptq")
    x = synth.make_custom_x(42, 3, 256, "fp16")
    y_plain = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 64, "fp16", "gptq")
    gi = (np.arange(256) // 64).astype(np.int32)
    y_gidx = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 64, "fp16", "gptq", g_idx=gi)
    assert np.array_equal(y_plain, y_gidx)


def test_act_order_permutation_invariance():
    L = synth.make_custom_layer(43, 512, 32, group=128, dtype="fp16", fmt="gptq", act_order=True)
    x = synth.make_custom_x(44, 2, 512, "fp16")
    y = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 128, "fp16", "gptq", g_idx=L.g_idx)
    perm = oracle.act_order_perm(L.g_idx)
    q = oracle.unpack_rows_std(L.qweight)
    q_sorted = q[perm]
    y_sorted = oracle.reference_y(x[:, perm], oracle.pack_rows_std(q_sorted), L.qzeros, L.scales,
                                  128, "fp16", "gptq", g_idx=L.g_idx[perm])
    assert np.allclose(y, y_sorted, rtol=1e-12, atol=1e-12)
    # With rows sorted, the group of row j is j // group.
    y_plain = oracle.reference_y(x[:, perm], oracle.pack_rows_std(q_sorted), L.qzeros, L.scales,
                                 128, "fp16", "gptq")
    assert np.allclose(y, y_plain, rtol=1e-12, atol=1e-12)


def test_reference_sampled_matches_full():
    L = synth.make_custom_layer(45, 256, 96, group=32, dtype="bf16")
    x = synth.make_custom_x(46, 5, 256, "bf16")
    y = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 32, "bf16", "awq")
    rows, cols = [0, 3, 4], [1, 50, 95]
    ys = oracle.reference_y(x, L.qweight, L.qzeros, L.scales, 32, "bf16", "awq", rows=rows,
                            cols=cols, col_chunk=2)
    assert np.array_equal(ys, y[np.ix_(rows, cols)])


def test_rounding_helpers():
    # bf16: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0)
    v = np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-9), 3.0, 0.0])
    r = oracle.round_f64_to_half_value(v, "bf16")
    assert r.tolist() == [1.0, 1 + 2**-6, -1.0, 3.0, 0.0]
    r16 = oracle.round_f64_to_half_value(np.array([1 + 2**-11, 1 + 3 * 2**-11]), "fp16")
    assert r16.tolist() == [1.0, 1 + 2**-9]
    bits = oracle.round_f64_to_half_bits(np.array([1.0, -2.0, 1 + 2**-7]), "bf16")
    assert bits.tolist() == [0x3F80, 0xC000, 0x3F81]
    assert oracle.half_bits_to_f64(np.array([0x3C00, 0xC000], np.uint16), "fp16").tolist() == [1.0, -2.0]


def test_rel_err_definition():
    assert oracle.rel_err(np.array([1.0, 2.0]), np.array([1.0, 4.0])) == 0.5
    assert oracle.rel_err(np.zeros(3), np.zeros(3)) == 0.0


# --------------------------------------------------------------------------- #
# Mutation tests: a planted mistake in the oracle must fail a pin                #
# --------------------------------------------------------------------------- #
class _Mutant:
    """A copy of the oracle's namespace with one function or constant replaced."""

    def __init__(self, **repl):
        for k in dir(oracle.core):
            if not k.startswith("__"):
                setattr(self, k, getattr(oracle.core, k))
        self._repl = repl
        for k, v in repl.items():
            setattr(self, k, v)


def _mutant_unpack_identity_order(words):
    u = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    R, C = u.shape
    out = np.empty((R, C, 8), dtype=np.uint8)
    for j in range(8):
        out[:, :, j] = (u >> (4 * j)) & 0xF  # planted: standard order instead of AWQ's
    return out.reshape(R, C * 8)


def _mutant_dequant_sign(q, z, s, g_of_k, cols=None):
    diff = z[g_of_k].astype(np.int64) - q.astype(np.int64)  # planted: z - q
    return (diff * s[g_of_k]).astype(np.float32)


def _mutant_dequant_no_zero(q, z, s, g_of_k, cols=None):
    return (q.astype(np.float64) * s[g_of_k]).astype(np.float32)  # planted: dropped zero


def _mutant_dequant_wrong_group(q, z, s, g_of_k, cols=None):
    g = np.minimum(g_of_k + 1, z.shape[0] - 1)  # planted: off-by-one group
    return ((q.astype(np.int64) - z[g]) * s[g]).astype(np.float32)


def _mutant_pack_rows_reversed(codes):
    K, N = codes.shape
    c = np.asarray(codes).astype(np.int64).reshape(K // 8, 8, N)
    acc = np.zeros((K // 8, N), dtype=np.int64)
    for i in range(8):
        acc += c[:, 7 - i, :] << (4 * i)  # planted: reversed nibble order
    return acc.astype(np.uint32).view(np.int32)


def test_mutant_identity_order_is_caught():
    m = _Mutant(unpack_awq=_mutant_unpack_identity_order)
    with pytest.raises(AssertionError):
        check_golden_unpack(m)
    with pytest.raises(AssertionError):
        check_awq_single_nibble(m)


@pytest.mark.parametrize("bad", [_mutant_dequant_sign, _mutant_dequant_no_zero,
                                 _mutant_dequant_wrong_group])
def test_mutant_dequant_is_caught(bad):
    m = _Mutant(dequant=bad)
    with pytest.raises(AssertionError):
        check_dequant_vs_writer(m)


def test_mutant_repack_order_is_caught():
    def repack(qweight, qzeros):
        return _mutant_pack_rows_reversed(oracle.unpack_awq(qweight)), \
            oracle.pack_cols_std(oracle.unpack_awq(qzeros))
    with pytest.raises(AssertionError):
        check_repack_matches_gptq_writer(_Mutant(repack_awq_to_std=repack))


def test_mutant_transposed_gemm_is_caught():
    def bad_gemm(x, W):
        Wt = np.asarray(W, np.float64)
        # planted: wrong operand order / reversed K
        return np.asarray(x, np.float64)[:, ::-1] @ Wt
    with pytest.raises(AssertionError):
        check_gemm_exact_rational(_Mutant(gemm=bad_gemm, reference_y=_rebind_reference(bad_gemm)))


def _rebind_reference(gemm_fn):
    def reference_y(x_bits, qweight, qzeros, scales_bits, group, dtype, fmt, g_idx=None,
                    rows=None, cols=None, col_chunk=4096):
        q, z, s = oracle.layer_codes(qweight, qzeros, scales_bits, dtype, fmt)
        K, N = q.shape
        x = oracle.half_bits_to_f64(x_bits, dtype)
        gk = oracle.group_of_rows(K, group, g_idx)
        return gemm_fn(x, oracle.dequant(q, z, s, gk))
    return reference_y


def _mutant_moe_next_expert(x_bits, experts, offsets, group, dtype, fmt):
    """Planted: each range multiplied by the following expert's weights."""
    y = np.zeros((len(x_bits), oracle.half_bits_to_f64(experts[0][2], dtype).shape[1]))
    for e in range(len(experts)):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            qw, qz, sc = experts[min(e + 1, len(experts) - 1)]
            y[r0:r1] = oracle.reference_y(x_bits[r0:r1], qw, qz, sc, group, dtype, fmt)
    return y


def _mutant_moe_shifted_ranges(x_bits, experts, offsets, group, dtype, fmt):
    """Planted: expert e takes rows [off[e] + 1, off[e+1] + 1) (an off-by-one)."""
    T = len(x_bits)
    y = np.zeros((T, oracle.half_bits_to_f64(experts[0][2], dtype).shape[1]))
    for e, (qw, qz, sc) in enumerate(experts):
        r0, r1 = min(int(offsets[e]) + 1, T), min(int(offsets[e + 1]) + 1, T)
        if r1 > r0:
            y[r0:r1] = oracle.reference_y(x_bits[r0:r1], qw, qz, sc, group, dtype, fmt)
    return y


@pytest.mark.parametrize("bad", [_mutant_moe_next_expert, _mutant_moe_shifted_ranges])
def test_mutant_moe_is_caught(bad):
    with pytest.raises(AssertionError):
        check_moe_exact_rational(bad)
