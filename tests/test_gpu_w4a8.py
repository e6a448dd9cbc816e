"""w4a8_gemm (INT4 weights x per-tensor FP8 activations, tcgen05 kind::f8f6f4)
against the FP8 oracle (oracle/fp8_oracle.py).

The activation codes the device writes (the first M*K bytes of the workspace)
must equal the oracle's e4m3 codes bit for bit (negative zero read as zero):
both sides take the rounding decisions in fp32. y must match the oracle's fp64 result within 4e-3 relative
and within one output ulp (fp32 accumulation, one rounding to the output dtype).
Shapes cover several 128 x 128 tiles with ragged rows, a partial last column
group, groups 128 and -1, both activation dtypes and symmetric weights.
"""
import numpy as np
import pytest

import oracle
import synth
from libutil import ensure_built, half_from_dev, half_to_dev, to_dev
from oracle import fp8_oracle as f8

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


CASES = [
    # K, N, group, dtype, fmt, symmetric, M
    (256, 256, 128, "bf16", "awq", False, 7),
    (512, 384, 128, "fp16", "awq", False, 200),
    (1024, 288, 128, "bf16", "gptq", False, 129),
    (768, 512, -1, "bf16", "awq", False, 64),
    (512, 256, 128, "bf16", "awq", True, 33),
    (4096, 1024, 128, "bf16", "awq", False, 1024),
]


@pytest.mark.parametrize("K,N,group,dtype,fmt,symmetric,M", CASES)
def test_w4a8_vs_oracle(w4, K, N, group, dtype, fmt, symmetric, M):
    import torch
    g = K if group == -1 else group
    L = synth.make_custom_layer([150, K, N, g], K, N, group=g, dtype=dtype, fmt=fmt,
                                symmetric=symmetric)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    sc = half_to_dev(L.scales, dtype)
    qz = to_dev(L.qzeros) if L.qzeros is not None else None
    if fmt == "awq":
        layer = w4.repack_awq(to_dev(L.qweight), qz, sc, K, N, group, tdt)
    else:
        layer = w4.repack_gptq(to_dev(L.qweight), qz, sc, None, K, N, group, tdt)
    xb = synth.make_custom_x([151, K, M], M, K, dtype)
    x = half_to_dev(xb, dtype)
    ws_bytes = w4.w4a8_gemm_workspace_size(M, K)
    assert ws_bytes >= M * K
    for call in range(2):
        ws = torch.full((ws_bytes,), 0xA5 if call else 0x5A, dtype=torch.uint8, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        w4.w4a8_gemm(x, layer.qw, layer.scales, layer.zeros, y, M, N, K, group, tdt, ws)
        torch.cuda.synchronize()
        codes_ref, _ = f8.quantize_act_per_tensor(oracle.half_bits_to_f64(xb, dtype))
        got_codes = ws[:M * K].cpu().numpy().reshape(M, K)
        # a negative value that rounds to zero is -0 (0x80) on the device and +0
        # in the oracle: the same number; every other code must match exactly
        got_codes = np.where(got_codes == 0x80, 0, got_codes)
        assert np.array_equal(got_codes, codes_ref), int(np.sum(got_codes != codes_ref))
        got = half_from_dev(y)
        y_ref = f8.reference_y_w4a8(xb, L.qweight, L.qzeros, L.scales, group, dtype, fmt)
        err = oracle.rel_err(oracle.half_bits_to_f64(got, dtype), y_ref)
        assert err <= TOL, err
        assert ulp_error(got, y_ref, dtype) <= 1.0
    assert w4.w4_device_status() == 0


def test_w4a8_zero_activations(w4):
    """x = 0: s_x = 1, every code 0, y = 0 exactly."""
    import torch
    K, N, M = 256, 128, 5
    L = synth.make_custom_layer([152], K, N, group=128, dtype="bf16")
    layer = w4.repack_awq(to_dev(L.qweight), to_dev(L.qzeros), half_to_dev(L.scales, "bf16"),
                          K, N, 128, torch.bfloat16)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(w4.w4a8_gemm_workspace_size(M, K), dtype=torch.uint8, device="cuda")
    w4.w4a8_gemm(x, layer.qw, layer.scales, layer.zeros, y, M, N, K, 128, torch.bfloat16, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0


def test_w4a8_extreme_group_sums(w4):
    """Activations that drive each 128-value block's code sum to its extremes: the
    zero point enters the tensor cores as the seven base-16 digits of 512 * (the
    block's code sum), so a block of 448s (the largest sum, every digit used), a
    block of -448s (negative), blocks that cancel exactly (sum 0) and blocks of
    small codes must all match the oracle. K = 640: five blocks, the last of a
    second digit row."""
    import torch
    K, N, M = 640, 256, 6
    L = synth.make_custom_layer([153, K, N], K, N, group=128, dtype="bf16")
    layer = w4.repack_awq(to_dev(L.qweight), to_dev(L.qzeros), half_to_dev(L.scales, "bf16"),
                          K, N, 128, torch.bfloat16)
    c = 3.5
    xf = np.zeros((M, K), dtype=np.float64)
    xf[0, :] = c                                   # every code 448: the largest block sums
    xf[1, :] = -c                                  # the most negative
    xf[2, :] = np.where(np.arange(K) % 2 == 0, c, -c)  # every block sums to zero
    xf[3, :] = c * 2.0 ** -12                      # codes far below 448
    xf[3, 0] = c                                   # ... with one at 448 setting s_x
    xf[4, :] = np.where((np.arange(K) // 128) % 2 == 0, c, -c)  # alternate sign per block
    xf[5, :] = np.linspace(-c, c, K)
    xb = synth.f32_to_bits(xf.astype(np.float32), "bf16")
    x = half_to_dev(xb, "bf16")
    ws = torch.empty(w4.w4a8_gemm_workspace_size(M, K), dtype=torch.uint8, device="cuda")
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    w4.w4a8_gemm(x, layer.qw, layer.scales, layer.zeros, y, M, N, K, 128, torch.bfloat16, ws)
    torch.cuda.synchronize()
    codes_ref, _ = f8.quantize_act_per_tensor(oracle.half_bits_to_f64(xb, "bf16"))
    got_codes = np.where(ws[:M * K].cpu().numpy().reshape(M, K) == 0x80, 0,
                         ws[:M * K].cpu().numpy().reshape(M, K))
    assert np.array_equal(got_codes, codes_ref)
    got = half_from_dev(y)
    y_ref = f8.reference_y_w4a8(xb, L.qweight, L.qzeros, L.scales, 128, "bf16", "awq")
    assert oracle.rel_err(oracle.half_bits_to_f64(got, "bf16"), y_ref) <= TOL
    assert ulp_error(got, y_ref, "bf16") <= 1.0
    assert w4.w4_device_status() == 0
