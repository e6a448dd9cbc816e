"""Both small-M kernels against the oracle, on the layer variants each must handle.

w4a16_gemm runs M <= 16 calls on one of two kernels: layers with at most 96 KB
of packed weights per SM (the small shapes of test_gpu_parity.py) on the
streaming kernel, larger ones on the clustered split-K kernel. The layers here
are above that size, so every variant (group 32 / 64 / 128 / all of K, fp16 and
bf16, bias, act-order with and without the staged x, an odd tile count) also
runs on the clustered kernel. Both kernels use exact operands, so the result is
within one output ulp of the exact fp64 value; it is checked on a sample of
columns that includes the first and last column groups.
"""
import numpy as np
import pytest

import oracle
import synth
from libutil import ensure_built, half_from_dev, half_to_dev, to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-3


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    import int4_weight_only_repack_gb300 as mod
    return mod


def ulp_error(y_bits, y_ref, dtype):
    y = oracle.half_bits_to_f64(y_bits, dtype)
    mant = 11 if dtype == "fp16" else 8
    e = np.floor(np.log2(np.maximum(np.abs(y_ref), 1e-30)))
    if dtype == "fp16":
        e = np.maximum(e, -14)
    ulp = 2.0 ** (e - (mant - 1))
    return float(np.max(np.abs(y - y_ref) / (ulp + 1e-5 * np.max(np.abs(y_ref)))))


def sample_cols(N, rng):
    cols = np.concatenate([np.arange(0, 48), np.arange(N - 48, N),
                           rng.choice(np.arange(48, N - 48), 256, replace=False)])
    return np.unique(cols)


CASES = [
    # K, N, group, dtype, fmt, act_order, bias, Ms
    (4096, 8192, 128, "bf16", "awq", False, True, (1, 5, 16)),
    (4096, 8192, 64, "fp16", "awq", False, False, (3, 16)),
    (4096, 8192, 32, "bf16", "awq", False, False, (2, 9)),
    (4096, 8192, -1, "bf16", "awq", False, True, (1, 16)),
    (4096, 8208, 128, "bf16", "awq", False, False, (1, 16)),
    (5120, 6144, 128, "fp16", "gptq", True, False, (1, 16)),
]


@pytest.mark.parametrize("K,N,group,dtype,fmt,act_order,bias,Ms", CASES)
def test_clustered_kernel_variants(w4, K, N, group, dtype, fmt, act_order, bias, Ms):
    import torch
    assert K * N / 2 / torch.cuda.get_device_properties(0).multi_processor_count > 96 * 1024
    g = K if group == -1 else group
    L = synth.make_custom_layer([140, K, N, g], K, N, group=g, dtype=dtype, fmt=fmt,
                                act_order=act_order)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    sc = half_to_dev(L.scales, dtype)
    if fmt == "awq":
        layer = w4.repack_awq(to_dev(L.qweight), to_dev(L.qzeros), sc, K, N, group, tdt)
    else:
        layer = w4.repack_gptq(to_dev(L.qweight), to_dev(L.qzeros), sc, to_dev(L.g_idx), K, N,
                               group, tdt)
    torch.cuda.synchronize()
    b = None
    bias_t = None
    if bias:
        b = synth.f32_to_bits(np.random.default_rng(141).standard_normal(N).astype(np.float32),
                              dtype)
        bias_t = half_to_dev(b, dtype)
    cols = sample_cols(N, np.random.default_rng([142, K, N]))
    for M in Ms:
        xb = synth.make_custom_x([143, K, M], M, K, dtype)
        x = half_to_dev(xb, dtype)
        y = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        w4.linear(x, layer, y=y, bias=bias_t)
        torch.cuda.synchronize()
        got = half_from_dev(y)
        assert np.all(np.isfinite(oracle.half_bits_to_f64(got, dtype))), M
        y_ref = oracle.reference_y(xb, L.qweight, L.qzeros, L.scales, group, dtype, fmt,
                                   g_idx=L.g_idx, cols=cols, bias_bits=b)
        err = oracle.rel_err(oracle.half_bits_to_f64(got[:, cols], dtype), y_ref)
        assert err <= TOL, (M, err)
        assert ulp_error(got[:, cols], y_ref, dtype) <= 1.0, M
        if act_order:
            # without a workspace the kernel gathers x[:, perm] itself: same bits
            y2 = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
            w4.w4a16_gemm(x, layer.qw, layer.scales, layer.zeros, layer.perm, y2, M, N, K,
                          group, tdt, None)
            torch.cuda.synchronize()
            assert np.array_equal(half_from_dev(y2), got), M
        # deterministic: the same call gives the same bits
        y3 = torch.empty_like(y)
        w4.linear(x, layer, y=y3, bias=bias_t)
        torch.cuda.synchronize()
        assert np.array_equal(half_from_dev(y3), got), M
    assert w4.w4_device_status() == 0
