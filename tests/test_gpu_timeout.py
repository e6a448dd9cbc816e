"""Failure detection without a GPU fault: the timeout path of the pipeline waits.

Every wait inside the kernels is bounded (one second). w4_test_stalled_gemm runs
the small-M kernel with its weight copies withheld, so its ring waits run out:
the kernel must record W4_ERR_TIMEOUT in the device status word (read through
w4_device_status), let its other copies land, exit, and leave the context
usable for the next call.
"""
import time

import numpy as np
import pytest

import synth
from libutil import ensure_built, half_from_dev, half_to_dev
from oracle import w4a16_oracle as oracle

pytestmark = pytest.mark.gpu

W4_ERR_TIMEOUT = 12


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    import int4_weight_only_repack_gb300 as mod
    return mod


def test_stalled_kernel_reports_timeout_and_recovers(w4):
    import torch
    K, N, M = 512, 256, 4
    L = synth.make_custom_layer([130], K, N, group=128, dtype="bf16")
    qweight = torch.from_numpy(L.qweight).cuda()
    qzeros = torch.from_numpy(L.qzeros).cuda()
    scales = half_to_dev(L.scales, "bf16")
    layer = w4.repack_awq(qweight, qzeros, scales, K, N, 128, torch.bfloat16)
    xb = synth.make_custom_x([131], M, K, "bf16")
    x = half_to_dev(xb, "bf16")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    assert w4.w4_device_status(clear=True) == 0

    t0 = time.monotonic()
    w4.w4_test_stalled_gemm(x, layer.qw, layer.scales, layer.zeros, y, M, N, K, 128, "bf16")
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert w4.w4_device_status() == W4_ERR_TIMEOUT
    assert 0.5 < elapsed < 60, elapsed  # the one-second wait limit, not a hang
    assert w4.w4_device_status(clear=True) == W4_ERR_TIMEOUT
    assert w4.w4_device_status() == 0

    # the context is intact: the same call without the stall is exact again
    y2 = w4.linear(x, layer)
    torch.cuda.synchronize()
    y_ref = oracle.reference_y(xb, L.qweight, L.qzeros, L.scales, 128, "bf16", "awq")
    got = oracle.half_bits_to_f64(half_from_dev(y2).reshape(M, N), "bf16")
    assert oracle.rel_err(got, y_ref) <= 4e-3
    assert w4.w4_device_status() == 0


def test_stall_hook_rejects_large_m(w4):
    import torch
    x = torch.empty((32, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((32, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4_test_stalled_gemm(x, x, x, x, y, 32, 32, 64, 64, "bf16")
    assert e.value.status == 2  # W4_ERR_SHAPE
