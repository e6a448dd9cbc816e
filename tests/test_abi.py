"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments with the documented status before touching
the GPU (these run on a machine without one)."""
import ctypes

import pytest

from libutil import declared_symbols, ensure_built

W4_OK, W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_GROUP, W4_ERR_ALIGN = 0, 1, 2, 3, 4
W4_ERR_DTYPE, W4_ERR_LAYOUT, W4_ERR_ALIAS, W4_ERR_WORKSPACE = 5, 6, 7, 10


@pytest.fixture(scope="module")
def lib():
    return ensure_built()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert set(names) >= {"w4_repack_awq", "w4_repack_gptq", "w4a16_gemm", "w4_dequant",
                          "w4_repack_sizes", "w4a16_gemm_workspace_size", "w4_status_string",
                          "w4_abi_version"}
    for name in names:
        assert hasattr(lib, name), name


def test_no_internal_symbols_leak(lib):
    # the library hides everything but the C ABI
    for name in ("launch_decode", "_ZN2w413launch_decodeERKNS_8GemmArgsEP11CUstream_st"):
        with pytest.raises(AttributeError):
            getattr(lib, name)


def test_status_strings_and_version():
    import int4_weight_only_repack_gb300 as w4
    ensure_built()
    assert w4.w4_abi_version() == 2
    for st in range(12):
        assert w4.w4_status_string(st)
    assert w4.w4_last_cuda_error() == "no CUDA error"
    assert "unknown" in w4.w4_status_string(99)


def test_repack_sizes():
    import int4_weight_only_repack_gb300 as w4
    ensure_built()
    # tiny layer: K=256, N=256, group 128 -> 32 KB codes, 2 groups
    assert w4.w4_repack_sizes(256, 256, 128, w4.W4_LAYOUT_STD) == (256 * 256 // 2, 2 * 256 // 2,
                                                                    2 * 256 * 2)
    assert w4.w4_repack_sizes(4096, 22016, 128, w4.W4_LAYOUT_TILE) == (4096 * 22016 // 2,
                                                                        32 * 22016 // 2,
                                                                        32 * 22016 * 2)
    assert w4.w4_repack_sizes(256, 64, -1, w4.W4_LAYOUT_TILE)[1] == 64 // 2
    # TILE pads N to whole 128-column groups; STD does not
    assert w4.w4_repack_sizes(256, 272, 128, w4.W4_LAYOUT_TILE)[0] == 256 * 384 // 2
    assert w4.w4_repack_sizes(256, 272, 128, w4.W4_LAYOUT_STD)[0] == 256 * 272 // 2


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced


@pytest.mark.parametrize("args,status", [
    ((0, 256, 128, 0), W4_ERR_SHAPE),
    ((256, 0, 128, 0), W4_ERR_SHAPE),
    ((256, 256, 96, 0), W4_ERR_GROUP),
    ((200, 256, 128, 0), W4_ERR_GROUP),
    ((256, 260, 128, 0), W4_ERR_SHAPE),
    ((256, 264, 128, 1), W4_ERR_SHAPE),     # TILE needs N % 16
    ((288, 256, 32, 1), W4_ERR_SHAPE),      # TILE needs K % 64
    ((256, 256, 128, 7), W4_ERR_LAYOUT),
    ((1 << 21, 256, 128, 0), W4_ERR_SHAPE),
])
def test_repack_sizes_rejects(lib, args, status):
    a = ctypes.c_size_t()
    assert lib.w4_repack_sizes(*args, ctypes.byref(a), None, None) == status


def _gemm(lib, x=FAKE, qw=FAKE * 2, sc=FAKE * 3, z=FAKE * 4, perm=None, y=FAKE * 5, M=4, N=256,
          K=256, group=128, dtype=1, ws=None, ws_b=0):
    return lib.w4a16_gemm(x, qw, sc, z, perm, y, M, N, K, group, dtype, ws, ws_b, None)


def test_gemm_rejects_bad_arguments(lib):
    assert _gemm(lib, x=None) == W4_ERR_NULL
    assert _gemm(lib, y=None) == W4_ERR_NULL
    assert _gemm(lib, qw=None) == W4_ERR_NULL
    assert _gemm(lib, x=FAKE + 2) == W4_ERR_ALIGN
    assert _gemm(lib, y=FAKE * 5 + 8) == W4_ERR_ALIGN
    assert _gemm(lib, N=264) == W4_ERR_SHAPE
    assert _gemm(lib, K=288, group=32) == W4_ERR_SHAPE
    assert _gemm(lib, M=-1) == W4_ERR_SHAPE
    assert _gemm(lib, group=16) == W4_ERR_GROUP
    assert _gemm(lib, dtype=2) == W4_ERR_DTYPE
    # y overlapping x
    assert _gemm(lib, y=FAKE + 256) == W4_ERR_ALIAS
    # M == 0 is a no-op that succeeds without touching the device
    assert _gemm(lib, M=0) == W4_OK


def test_repack_rejects_bad_arguments(lib):
    f = lib.w4_repack_awq
    ok = dict(qweight=FAKE, qzeros=FAKE * 3, scales=FAKE * 5, K=256, N=256, group=128, dtype=0,
              layout=1, qw_out=FAKE * 7, zeros_out=FAKE * 9, scales_out=FAKE * 11, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*a.values())

    assert call(qweight=None) == W4_ERR_NULL
    assert call(scales_out=None) == W4_ERR_NULL
    assert call(qw_out=FAKE * 7 + 4) == W4_ERR_ALIGN
    assert call(qw_out=FAKE) == W4_ERR_ALIAS          # output over the input
    assert call(zeros_out=FAKE * 7) == W4_ERR_ALIAS   # two outputs overlap
    assert call(layout=2) == W4_ERR_LAYOUT
    assert call(dtype=-1) == W4_ERR_DTYPE
    g = lib.w4_repack_gptq
    # act-order needs perm_out and status_out
    assert g(FAKE, FAKE * 3, FAKE * 5, FAKE * 13, 256, 256, 128, 0, 1, FAKE * 7, FAKE * 9,
             FAKE * 11, None, None, None) == W4_ERR_NULL
    # too many groups for the act-order sort
    assert g(FAKE, FAKE * 3, FAKE * 5, FAKE * 13, 1 << 19, 256, 32, 0, 1, FAKE * 7 * 1024,
             FAKE * 9 * 1024, FAKE * 11 * 1024, FAKE * 15 * 1024, FAKE * 17 * 1024,
             None) == W4_ERR_SHAPE


def test_dequant_rejects_bad_arguments(lib):
    d = lib.w4_dequant
    assert d(None, FAKE, FAKE * 2, 256, 256, 128, 0, 1, 1, FAKE * 3, None) == W4_ERR_NULL
    assert d(FAKE, FAKE * 2, FAKE * 3, 256, 256, 128, 0, 1, 1, FAKE, None) == W4_ERR_ALIAS
    assert d(FAKE, FAKE * 2, FAKE * 3, 256, 256, 128, 0, 3, 1, FAKE * 9, None) == W4_ERR_LAYOUT


def test_binding_raises_on_error():
    import int4_weight_only_repack_gb300 as w4
    ensure_built()
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemm(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, FAKE * 5, 4, 264, 256, 128,
                      "bf16", stream=0)
    assert e.value.status == W4_ERR_SHAPE


def _moe(lib, x=FAKE, qw=FAKE * 2, sc=FAKE * 3, z=FAKE * 4, off=FAKE * 6, y=FAKE * 5, E=4,
         max_rows=16, total_rows=64, N=256, K=256, group=128, dtype=1):
    return lib.w4a16_moe_gemm(x, qw, sc, z, off, y, E, max_rows, total_rows, N, K, group, dtype,
                              None)


def test_moe_gemm_rejects_bad_arguments(lib):
    """Host-side checks of w4a16_moe_gemm, and which kernel's row limit applies:
    a call that passes the shape checks is stopped by an aliased y (x == y), so
    no case reaches a launch."""
    assert _moe(lib, E=0) == W4_ERR_SHAPE
    assert _moe(lib, E=65536) == W4_ERR_SHAPE
    assert _moe(lib, max_rows=0) == W4_ERR_SHAPE
    assert _moe(lib, total_rows=-1) == W4_ERR_SHAPE
    assert _moe(lib, total_rows=(1 << 20) + 1) == W4_ERR_SHAPE
    assert _moe(lib, off=None) == W4_ERR_NULL
    assert _moe(lib, x=None) == W4_ERR_NULL
    assert _moe(lib, y=FAKE * 5 + 8) == W4_ERR_ALIGN
    assert _moe(lib, off=FAKE * 6 + 4) == W4_ERR_ALIGN
    assert _moe(lib, N=264) == W4_ERR_SHAPE                      # TILE needs N % 16
    assert _moe(lib, group=16) == W4_ERR_GROUP
    assert _moe(lib, y=FAKE) == W4_ERR_ALIAS
    # N % 32 == 0, more than 16 rows an expert: the tcgen05 kernel (no 64-row limit)
    assert _moe(lib, max_rows=65, y=FAKE) == W4_ERR_ALIAS
    assert _moe(lib, max_rows=1 << 20, total_rows=1 << 20, y=FAKE) == W4_ERR_ALIAS
    assert _moe(lib, max_rows=(1 << 20) + 1, y=FAKE) == W4_ERR_SHAPE
    # N % 32 != 0: the small-M kernel only, up to 64 rows an expert
    assert _moe(lib, N=272, max_rows=64, y=FAKE) == W4_ERR_ALIAS
    assert _moe(lib, N=272, max_rows=65, y=FAKE) == W4_ERR_SHAPE
    # more than 4096 experts: beyond the tcgen05 kernel's table, so 64 rows at most
    assert _moe(lib, E=4097, max_rows=64, y=FAKE) == W4_ERR_ALIAS
    assert _moe(lib, E=4097, max_rows=65, y=FAKE) == W4_ERR_SHAPE


def test_linear_caches_workspace_size(monkeypatch):
    """linear() asks the library for a call's workspace size once per (device,
    M, layer shape): a fake library counts the calls (no GPU needed)."""
    import torch
    import int4_weight_only_repack_gb300 as w4

    class FakeLib:
        def __init__(self):
            self.size_calls = []
            self.gemm_calls = 0

        def w4a16_gemm_workspace_size(self, M, N, K, group, dtype, has_perm):
            self.size_calls.append((M, N, K, group, dtype, has_perm))
            return 0 if M <= 16 else 4096

        def w4a16_gemm_bias(self, *args):
            self.gemm_calls += 1
            return W4_OK

    fake = FakeLib()
    monkeypatch.setattr(w4, "_LIB", fake)
    monkeypatch.setattr(w4, "_WS_SIZES", {})
    monkeypatch.setattr(w4, "gemm_workspace", lambda nbytes, device, stream=None:
                        torch.empty(nbytes, dtype=torch.uint8))
    K, N = 256, 128
    layer = w4.RepackedLayer(K, N, 128, torch.bfloat16, w4.W4_LAYOUT_TILE,
                             torch.zeros(8), torch.zeros(8), torch.zeros(8))
    act = w4.RepackedLayer(K, N, 128, torch.bfloat16, w4.W4_LAYOUT_TILE,
                           torch.zeros(8), torch.zeros(8), torch.zeros(8),
                           perm=torch.zeros(K, dtype=torch.int32))
    for M in (1, 1, 4, 1, 64, 64):
        w4.linear(torch.zeros(M, K, dtype=torch.bfloat16), layer)
    w4.linear(torch.zeros(4, K, dtype=torch.bfloat16), act)
    w4.linear(torch.zeros(4, K, dtype=torch.bfloat16), act)
    assert fake.gemm_calls == 8
    assert [c[0] for c in fake.size_calls] == [1, 4, 64, 4]
    assert [c[5] for c in fake.size_calls] == [0, 0, 0, 1]


def _declared_signatures():
    """{name: [parameter type strings]} for every W4_API function of the header."""
    import re
    from libutil import HEADER
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    out = {}
    for m in re.finditer(r"W4_API\s+([\w\s\*]+?)\b(\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(3).split(",")]
        if params == ["void"] or params == [""]:
            params = []
        out[m.group(2)] = (m.group(1).strip(), params)
    return out


def test_binding_matches_header():
    """The ctypes binding declares every header function with the same number
    of parameters, pointers where the header has pointers, and integers of the
    header's widths elsewhere."""
    import ctypes
    import int4_weight_only_repack_gb300 as w4
    decl = _declared_signatures()
    assert set(decl) == set(w4._SIGNATURES), set(decl) ^ set(w4._SIGNATURES)
    for name, (ret, params) in decl.items():
        res, args = w4._SIGNATURES[name]
        assert len(args) == len(params), name
        for p, a in zip(params, args):
            if "*" in p:
                assert a is ctypes.c_void_p or a is ctypes.c_char_p or \
                    issubclass(a, ctypes._Pointer), (name, p, a)
            elif p.split()[0] == "size_t":
                assert a is ctypes.c_size_t, (name, p)
            else:
                assert a in (ctypes.c_int, ctypes.c_int32), (name, p, a)
        if "char" in ret:
            assert res is ctypes.c_char_p, name
        elif ret.split()[-1] in ("w4_status", "int"):
            assert res in (ctypes.c_int, ctypes.c_int32), name
        else:
            assert ret == "size_t" and res is ctypes.c_size_t, (name, ret)


def _w4a8(lib, x=FAKE, qw=FAKE * 2, sc=FAKE * 3, z=FAKE * 4, y=FAKE * 5, M=4, N=256, K=256,
          group=128, dtype=1, ws=FAKE * 6, ws_b=1 << 20):
    import int4_weight_only_repack_gb300 as w4
    w4.lib()
    return lib.w4a8_gemm(x, qw, sc, z, y, M, N, K, group, dtype, ws, ws_b, None)


def test_w4a8_gemm_rejects(lib):
    """w4a8_gemm's host checks: group 128 or -1 only, K % 128, the workspace
    size and presence, alignment, aliasing; M == 0 is a no-op."""
    import int4_weight_only_repack_gb300 as w4
    w4.lib()
    assert _w4a8(lib, group=64) == W4_ERR_GROUP
    assert _w4a8(lib, group=32) == W4_ERR_GROUP
    assert _w4a8(lib, K=320, group=64) == W4_ERR_GROUP
    assert _w4a8(lib, K=384 + 64, group=-1) == W4_ERR_SHAPE      # K % 128
    assert _w4a8(lib, N=272) == W4_ERR_SHAPE                      # N % 32
    assert _w4a8(lib, ws=None) == W4_ERR_NULL
    assert _w4a8(lib, ws_b=16) == W4_ERR_WORKSPACE
    assert _w4a8(lib, x=FAKE + 8) == W4_ERR_ALIGN
    assert _w4a8(lib, y=FAKE * 6) == W4_ERR_ALIAS                 # y on the workspace
    assert _w4a8(lib, M=0, x=None, y=None, ws=None) == W4_OK
    assert _w4a8(lib, dtype=3) == W4_ERR_DTYPE
    assert w4.w4a8_gemm_workspace_size(4, 256) >= 4 * 256
    assert w4.w4a8_gemm_workspace_size(4, 320) == 0
