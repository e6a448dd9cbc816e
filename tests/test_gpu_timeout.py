"""Failure detection without a GPU fault: the timeout path of the pipeline waits.

Every wait inside the kernels is bounded (one second). w4_test_stalled_gemm runs
the kernel a call would run with the loads its pipeline waits on withheld (the
small-M kernel's weight copies; all of the tcgen05 kernel's TMA loads), so its
waits run out: the kernel must record W4_ERR_TIMEOUT in the device status word
(read through w4_device_status), wind down, exit, and leave the context usable
for the next call.
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


# M = 4: the small-M kernel; 64: the tcgen05 kernel with 64-row x tiles; 200:
# its 128-row tiles over two row blocks
@pytest.mark.parametrize("M", [4, 64, 200])
def test_stalled_kernel_reports_timeout_and_recovers(w4, M):
    import torch
    K, N = 512, 256
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
    # (the tcgen05 path multiplies weights rounded to bf16: 5e-3, as in its parity tests)
    assert oracle.rel_err(got, y_ref) <= (4e-3 if M <= 16 else 5e-3)
    assert w4.w4_device_status() == 0


def test_stall_hook_rejects_unsupported_large_m(w4):
    """Above M = 16 the hook needs the tcgen05 kernel (N % 32 == 0)."""
    import torch
    x = torch.empty((32, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((32, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4_test_stalled_gemm(x, x, x, x, y, 32, 48, 64, 64, "bf16")
    assert e.value.status == 2  # W4_ERR_SHAPE
