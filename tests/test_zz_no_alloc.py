"""w4a16_gemm_noalloc against w4a16_gemm, through the C ABI.

Some callers of this library cannot allocate device memory when they call the
GEMM: a host that embeds the library behind a plain-function interface with no
device allocator, or a serving runtime that reserves all of its device memory
up front. w4a16_gemm_noalloc serves them: where w4a16_gemm uses a workspace
(act-order staging of x[:, perm], split-K partial tiles of the large-M kernel)
it uses a static device array the library owns. This file checks that it gives
the same result as the workspace entry point, twice in a row (the array keeps
the previous call's contents), on act-order layers and on layers whose large-M
calls split K, and that it refuses sizes beyond the array. It is collected last
so that a failure here does not stop the rest of the suite from running first.
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


def _awq_layer(w4, K, N, group, seed):
    import torch
    L = synth.make_custom_layer([seed, K, N], K, N, group=group, dtype="bf16")
    layer = w4.repack_awq(to_dev(L.qweight), to_dev(L.qzeros), half_to_dev(L.scales, "bf16"),
                          K, N, group, torch.bfloat16)
    torch.cuda.synchronize()
    return L, layer


# Large-M calls without act-order whose output tiles cannot fill the GPU: the
# tcgen05 kernel splits K and keeps fp32 partial tiles in the static array.
@pytest.mark.parametrize("K,N,M", [(4096, 256, 128), (8192, 256, 64)])
def test_noalloc_split_k_partials(w4, K, N, M):
    import torch
    lib = w4.lib()
    assert lib.w4a16_gemm_workspace_size(M, N, K, 128, w4.W4_BF16, 0) > 0, "shape must split K"
    L, layer = _awq_layer(w4, K, N, 128, 134)
    stream = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(lib.w4a16_gemm_workspace_size(M, N, K, 128, w4.W4_BF16, 0),
                     dtype=torch.uint8, device="cuda")
    xb = synth.make_custom_x([135, K, M], M, K, "bf16")
    x = half_to_dev(xb, "bf16")
    y_ref = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert lib.w4a16_gemm(x.data_ptr(), layer.qw.data_ptr(), layer.scales.data_ptr(),
                          layer.zeros.data_ptr(), None, y_ref.data_ptr(), M, N, K, 128,
                          w4.W4_BF16, ws.data_ptr(), ws.numel(), stream) == 0
    torch.cuda.synchronize()
    ref_bits = half_from_dev(y_ref)
    exact = oracle.reference_y(xb, L.qweight, L.qzeros, L.scales, 128, "bf16", "awq")
    for call in range(2):
        # the first call runs on another input, so the array holds other partials
        xc = x if call else half_to_dev(synth.make_custom_x([136, K, M], M, K, "bf16"), "bf16")
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert lib.w4a16_gemm_noalloc(xc.data_ptr(), layer.qw.data_ptr(), layer.scales.data_ptr(),
                                      layer.zeros.data_ptr(), None, y.data_ptr(), M, N, K, 128,
                                      w4.W4_BF16, stream) == 0
        torch.cuda.synchronize()
        if call == 1:
            got = half_from_dev(y)
            assert np.array_equal(got, ref_bits)
            assert oracle.rel_err(oracle.half_bits_to_f64(got, "bf16"), exact) <= TOL


def test_noalloc_refuses_oversized_staging(w4):
    import torch
    K, N, group = 1024, 256, 128
    _, layer = _act_order_layer(w4, K, N, group, 133)
    M = (32 << 20) // (K * 2) + 64   # M * K * 2 bytes beyond the static array
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert _noalloc(w4, x, layer, y, M) == W4_ERR_WORKSPACE
