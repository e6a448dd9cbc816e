"""w4a16_gemm_noalloc against w4a16_gemm, through the C ABI.

Some callers of this library cannot allocate device memory when they call the
GEMM, for instance code running under CUDA-graph capture (where cudaMalloc is
not allowed) or a host that embeds the library behind an interface without an
allocator. w4a16_gemm_noalloc serves them: it stages act-order activations in a
static device array the library owns instead of a caller workspace. This file
checks that it gives the same result as the workspace entry point, twice in a
row (the array keeps the previous call's contents), and that it refuses sizes
beyond the array. It is collected last so that a failure here does not stop
the rest of the suite from running first.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from libutil import ensure_built, half_from_dev, half_to_dev, to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-3
W4_ERR_WORKSPACE = 10


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    import int4_weight_only_repack_gb300 as mod
    return mod


def _act_order_layer(w4, K, N, group, seed):
    import torch
    L = synth.make_custom_layer([seed, K, N], K, N, group=group, dtype="fp16", fmt="gptq",
                                act_order=True)
    layer = w4.repack_gptq(to_dev(L.qweight), to_dev(L.qzeros), half_to_dev(L.scales, "fp16"),
                           to_dev(L.g_idx), K, N, group, torch.float16)
    torch.cuda.synchronize()
    assert int(layer.status[0].item()) == 0
    return L, layer


def _noalloc(w4, x, layer, y, M):
    lib = w4.lib()
    import torch
    return lib.w4a16_gemm_noalloc(x.data_ptr(), layer.qw.data_ptr(), layer.scales.data_ptr(),
                                  layer.zeros.data_ptr(), layer.perm.data_ptr(), y.data_ptr(),
                                  M, layer.N, layer.K, layer.group, w4.W4_F16,
                                  torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("K,N,group,M", [(512, 256, 128, 100), (1024, 320, 64, 200),
                                         (256, 256, 128, 16)])
def test_noalloc_matches_workspace_entry(w4, K, N, group, M):
    import torch
    L, layer = _act_order_layer(w4, K, N, group, 130)
    ref = w4.linear(half_to_dev(synth.make_custom_x([131, K, M], M, K, "fp16"), "fp16"), layer)
    torch.cuda.synchronize()
    ref_bits = half_from_dev(ref)
    for call in range(2):
        # a different input on the first call leaves other data in the static array
        xb = synth.make_custom_x([131 if call else 132, K, M], M, K, "fp16")
        x = half_to_dev(xb, "fp16")
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(w4, x, layer, y, M) == 0
        torch.cuda.synchronize()
        got = half_from_dev(y)
        if call == 1:
            err = oracle.rel_err(oracle.half_bits_to_f64(got, "fp16"),
                                 oracle.half_bits_to_f64(ref_bits, "fp16"))
            assert err <= TOL, err
            assert np.array_equal(got, ref_bits)
        else:
            y_ref = oracle.reference_y(xb, L.qweight, L.qzeros, L.scales, group, "fp16", "gptq",
                                       g_idx=L.g_idx)
            assert oracle.rel_err(oracle.half_bits_to_f64(got, "fp16"), y_ref) <= TOL


def test_noalloc_refuses_oversized_staging(w4):
    import torch
    K, N, group = 1024, 256, 128
    _, layer = _act_order_layer(w4, K, N, group, 133)
    M = (32 << 20) // (K * 2) + 64   # M * K * 2 bytes beyond the static array
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert _noalloc(w4, x, layer, y, M) == W4_ERR_WORKSPACE
