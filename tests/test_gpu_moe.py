"""Grouped W4A16 GEMM over the experts of an MoE layer (w4a16_moe_gemm) against
the oracle: every expert's rows of y against that expert's oracle reference."""
import numpy as np
import pytest

import synth
from libutil import ensure_built, half_from_dev, half_to_dev, rounded_w_reference, to_dev
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


def make_experts(w4, E, K, N, dtype, seed, group=128, symmetric=False):
    layers = [synth.make_custom_layer([seed, e, K, N], K, N, group=group, dtype=dtype,
                                      symmetric=symmetric) for e in range(E)]
    experts = w4.repack_awq_experts([to_dev(L.qweight) for L in layers],
                                    [None if L.qzeros is None else to_dev(L.qzeros)
                                     for L in layers],
                                    [half_to_dev(L.scales, dtype) for L in layers],
                                    K, N, group, dtype)
    return layers, experts


def ulp_error(y_bits, y_ref, dtype):
    y = oracle.half_bits_to_f64(y_bits, dtype)
    mant = 11 if dtype == "fp16" else 8
    e = np.floor(np.log2(np.maximum(np.abs(y_ref), 1e-30)))
    if dtype == "fp16":
        e = np.maximum(e, -14)
    ulp = np.exp2(e - (mant - 1))
    return float(np.max(np.abs(y - y_ref) / (ulp + 1e-5 * np.max(np.abs(y_ref)))))


@pytest.mark.parametrize("E,K,N,dtype,rows,group", [
    # small-M kernel (at most 16 rows an expert, or N % 32 != 0)
    (8, 1024, 512, "bf16", [3, 0, 16, 1, 0, 7, 2, 5], 128),   # mixed counts, empty experts
    (4, 512, 272, "fp16", [64, 1, 33, 0], 128),                # up to 64 rows, N % 32 != 0
    (3, 4096, 256, "bf16", [1, 1, 1], 128),                    # K split across a cluster
    # tcgen05 kernel (more than 16 rows an expert)
    (4, 1024, 512, "bf16", [300, 0, 129, 17], 128),            # ragged 128-row tiles, empty expert
    (3, 512, 384, "fp16", [17, 200, 65], 128),                 # odd column groups per expert
    (2, 256, 256, "bf16", [100, 40], 32),                      # two group rows per k-block
    (5, 640, 96, "bf16", [0, 33, 0, 0, 260], 64),              # N < one N block, leading empties
    (3, 512, 512, "bf16", [520, 0, 300], 128),                 # 256-row tiles (mean rows > 256)
    (2, 768, 320, "fp16", [390, 257], 64),                     # 256-row tiles, odd column groups
])
def test_moe_gemm_vs_oracle(w4, E, K, N, dtype, rows, group):
    import torch
    layers, experts = make_experts(w4, E, K, N, dtype, 135, group)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    T = int(off[-1])
    x = synth.make_custom_x([136, E, K], T, K, dtype)
    y = torch.full((T, N), float("nan"), dtype=hdt(dtype), device="cuda")
    w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), max(rows), y=y)
    torch.cuda.synchronize()
    yb = half_from_dev(y).reshape(T, N)
    large = max(rows) > 16 and N % 32 == 0
    y_all = oracle.moe_reference_y(x, [(L.qweight, L.qzeros, L.scales) for L in layers], off,
                                   group, dtype, "awq")
    for e, L in enumerate(layers):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        y_ref = y_all[r0:r1]
        assert oracle.rel_err(oracle.half_bits_to_f64(yb[r0:r1], dtype), y_ref) <= 4e-3, e
        if large:
            # the tcgen05 kernel's B operand is W rounded once to the activation
            # dtype: within one output ulp of that product
            y_ref = rounded_w_reference(x[r0:r1], L, group)
        assert ulp_error(yb[r0:r1], y_ref, dtype) <= 1.0, (e, ulp_error(yb[r0:r1], y_ref, dtype))
    assert w4.w4_device_status() == 0


@pytest.mark.parametrize("rows", [[5, 0, 12], [40, 0, 150]])
def test_moe_gemm_symmetric_experts(w4, rows):
    """Symmetric experts (no qzeros: zero point 8) on both kernels."""
    import torch
    E, K, N, dtype = 3, 512, 256, "fp16"
    layers, experts = make_experts(w4, E, K, N, dtype, 146, symmetric=True)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    T = int(off[-1])
    x = synth.make_custom_x([147, T], T, K, dtype)
    y = torch.full((T, N), float("nan"), dtype=hdt(dtype), device="cuda")
    w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), max(rows), y=y)
    torch.cuda.synchronize()
    yb = half_from_dev(y).reshape(T, N)
    y_all = oracle.moe_reference_y(x, [(L.qweight, None, L.scales) for L in layers], off, 128,
                                   dtype, "awq")
    large = max(rows) > 16
    for e, L in enumerate(layers):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        assert oracle.rel_err(oracle.half_bits_to_f64(yb[r0:r1], dtype), y_all[r0:r1]) <= 4e-3
        y_ref = rounded_w_reference(x[r0:r1], L, 128) if large else y_all[r0:r1]
        assert ulp_error(yb[r0:r1], y_ref, dtype) <= 1.0, e
    assert w4.w4_device_status() == 0


def test_moe_gemm_many_experts(w4):
    """More experts than fit the 256-row pipeline's table (128-row tiles): 300
    small experts, most of them without rows."""
    import torch
    E, K, N, dtype = 300, 128, 64, "bf16"
    layers, experts = make_experts(w4, E, K, N, dtype, 143)
    rng = np.random.default_rng(144)
    rows = np.zeros(E, dtype=np.int64)
    busy = rng.choice(E, 24, replace=False)
    rows[busy] = rng.integers(1, 140, size=24)
    rows[busy[0]] = 139
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    T = int(off[-1])
    x = synth.make_custom_x([145], T, K, dtype)
    y = torch.full((T, N), float("nan"), dtype=hdt(dtype), device="cuda")
    w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), int(rows.max()), y=y)
    torch.cuda.synchronize()
    yb = half_from_dev(y).reshape(T, N)
    for e in busy:
        r0, r1 = int(off[e]), int(off[e + 1])
        y_ref = rounded_w_reference(x[r0:r1], layers[e], 128)
        assert ulp_error(yb[r0:r1], y_ref, dtype) <= 1.0, e
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
        w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), 0, y=y)


def test_moe_gemm_large_rejects_oversized_expert(w4):
    """The same rule on the tcgen05 kernel (more than 16 rows an expert): the
    expert past max_rows_per_expert is left out, the others are exact."""
    import torch
    E, K, N, dtype = 3, 512, 256, "bf16"
    layers, experts = make_experts(w4, E, K, N, dtype, 139)
    rows = [40, 300, 20]  # expert 1 has more than max_rows_per_expert = 100
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    T = int(off[-1])
    x = synth.make_custom_x([140], T, K, dtype)
    y = torch.zeros((T, N), dtype=hdt(dtype), device="cuda")
    assert w4.w4_device_status(clear=True) == 0
    w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), 100, y=y)
    torch.cuda.synchronize()
    assert w4.w4_device_status(clear=True) == W4_ERR_EXPERT_ROWS
    yb = half_from_dev(y).reshape(T, N)
    assert not yb[40:340].any()  # expert 1's rows untouched
    for e in (0, 2):
        r0, r1 = int(off[e]), int(off[e + 1])
        y_ref = rounded_w_reference(x[r0:r1], layers[e], 128)
        assert ulp_error(yb[r0:r1], y_ref, dtype) <= 1.0, e


def test_moe_gemm_small_kernel_row_limit(w4):
    """With N % 32 != 0 only the small-M kernel serves the call: more than 64
    rows an expert is refused on the host."""
    import torch
    E, K, N, dtype = 2, 256, 272, "bf16"
    _, experts = make_experts(w4, E, K, N, dtype, 141)
    off = np.array([0, 10, 20], dtype=np.int32)
    x = synth.make_custom_x([142], 20, K, dtype)
    y = torch.zeros((20, N), dtype=hdt(dtype), device="cuda")
    with pytest.raises(w4.W4Error):
        w4.moe_linear(half_to_dev(x, dtype), experts, to_dev(off), 65, y=y)
