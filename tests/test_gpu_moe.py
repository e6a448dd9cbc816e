"""Grouped W4A16 GEMM over the experts of an MoE layer (w4a16_moe_gemm) against
the oracle: every expert's rows of y against that expert's oracle reference."""
import numpy as np
import pytest

import synth
from libutil import ensure_built, half_from_dev, half_to_dev, to_dev
from oracle import w4a16_oracle as oracle

pytestmark = pytest.mark.gpu

W4_ERR_EXPERT_ROWS = 13


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    import int4_weight_only_repack_gb300 as mod
    return mod


def hdt(dtype):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float16


def make_experts(w4, E, K, N, dtype, seed):
    layers = [synth.make_custom_layer([seed, e, K, N], K, N, group=128, dtype=dtype)
              for e in range(E)]
    experts = w4.repack_awq_experts([to_dev(L.qweight) for L in layers],
                                    [to_dev(L.qzeros) for L in layers],
                                    [half_to_dev(L.scales, dtype) for L in layers],
                                    K, N, 128, dtype)
    return layers, experts


def ulp_error(y_bits, y_ref, dtype):
    y = oracle.half_bits_to_f64(y_bits, dtype)
    mant = 11 if dtype == "fp16" else 8
    e = np.floor(np.log2(np.maximum(np.abs(y_ref), 1e-30)))
    if dtype == "fp16":
        e = np.maximum(e, -14)
    ulp = np.exp2(e - (mant - 1))
    return float(np.max(np.abs(y - y_ref) / (ulp + 1e-5 * np.max(np.abs(y_ref)))))


@pytest.mark.parametrize("E,K,N,dtype,rows", [
    (8, 1024, 512, "bf16", [3, 0, 16, 1, 0, 7, 2, 5]),   # mixed counts, empty experts
    (4, 512, 272, "fp16", [64, 1, 33, 0]),                # up to 64 rows, N % 32 != 0
    (3, 4096, 256, "bf16", [1, 1, 1]),                    # K split across a cluster
])
def test_moe_gemm_vs_oracle(w4, E, K, N, dtype, rows):
    import torch
    layers, experts = make_experts(w4, E, K, N, dtype, 135)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    T = int(off[-1])
    x = synth.make_custom_x([136, E, K], T, K, dtype)
    y = torch.full((T, N), float("nan"), dtype=hdt(dtype), device="cuda")
    w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), max(rows), y=y)
    torch.cuda.synchronize()
    yb = half_from_dev(y).reshape(T, N)
    for e, L in enumerate(layers):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        y_ref = oracle.reference_y(x[r0:r1], L.qweight, L.qzeros, L.scales, 128, dtype, "awq")
        assert oracle.rel_err(oracle.half_bits_to_f64(yb[r0:r1], dtype), y_ref) <= 4e-3, e
        assert ulp_error(yb[r0:r1], y_ref, dtype) <= 1.0, (e, ulp_error(yb[r0:r1], y_ref, dtype))
    assert w4.w4_device_status() == 0


def test_moe_gemm_rejects_oversized_expert(w4):
    """An expert with more rows than max_rows_per_expert records
    W4_ERR_EXPERT_ROWS and leaves its rows of y unwritten; the others are exact."""
    import torch
    E, K, N, dtype = 3, 512, 256, "bf16"
    layers, experts = make_experts(w4, E, K, N, dtype, 137)
    rows = [2, 6, 3]  # expert 1 has more than max_rows_per_expert = 4
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    T = int(off[-1])
    x = synth.make_custom_x([138], T, K, dtype)
    y = torch.zeros((T, N), dtype=hdt(dtype), device="cuda")
    assert w4.w4_device_status(clear=True) == 0
    w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), 4, y=y)
    torch.cuda.synchronize()
    assert w4.w4_device_status(clear=True) == W4_ERR_EXPERT_ROWS
    yb = half_from_dev(y).reshape(T, N)
    assert not yb[2:8].any()  # expert 1's rows untouched
    for e in (0, 2):
        r0, r1 = int(off[e]), int(off[e + 1])
        y_ref = oracle.reference_y(x[r0:r1], layers[e].qweight, layers[e].qzeros,
                                   layers[e].scales, 128, dtype, "awq")
        assert ulp_error(yb[r0:r1], y_ref, dtype) <= 1.0, e
    with pytest.raises(w4.W4Error):
        w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), 65, y=y)  # above 64
