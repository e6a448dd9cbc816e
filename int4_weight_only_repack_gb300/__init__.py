"""Python binding of libw4a16.so, the GB300 W4A16 linear-layer library.

Argument marshalling only: every entry point below forwards device pointers,
sizes and the current CUDA stream to the C ABI declared in include/w4a16.h and
raises W4Error on a non-zero status. All computation runs in the library's CUDA
kernels; there is no fallback path. If the shared library has not been built
the first call raises, naming the build step.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "W4_F16", "W4_BF16", "W4_LAYOUT_STD", "W4_LAYOUT_TILE", "W4Error", "lib", "library_path",
    "dtype_code", "w4_status_string", "w4_last_cuda_error", "w4_abi_version", "w4_repack_sizes", "w4_repack_awq",
    "w4_repack_gptq", "w4a16_gemm_workspace_size", "w4a16_gemm", "w4a16_gemm_bias",
    "w4a16_gemm_noalloc", "w4a8_gemm_workspace_size", "w4a8_gemm", "linear_fp8",
    "w4_dequant", "gemm_workspace",
    "w4_device_status", "w4_test_stalled_gemm", "w4_test_prefill_plan",
    "RepackedLayer", "repack_awq", "repack_gptq", "linear", "w4a16_moe_gemm", "RepackedExperts",
    "repack_awq_experts", "moe_linear",
]

W4_F16, W4_BF16 = 0, 1
W4_LAYOUT_STD, W4_LAYOUT_TILE = 0, 1
W4_OK = 0
W4_ERR_CUDA = 9
W4_ERR_GIDX = 11

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG_DIR, "libw4a16.so")
_LIB: Optional[ctypes.CDLL] = None

_c_int, _c_size, _c_void_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
_SIGNATURES = {
    "w4_status_string": (ctypes.c_char_p, [_c_int]),
    "w4_last_cuda_error": (ctypes.c_char_p, []),
    "w4_abi_version": (_c_int, []),
    "w4_repack_sizes": (_c_int, [_c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_c_size),
                                 ctypes.POINTER(_c_size), ctypes.POINTER(_c_size)]),
    "w4_repack_awq": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int,
                               _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "w4_repack_gptq": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                _c_int, _c_int, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                _c_void_p, _c_void_p, _c_void_p]),
    "w4a16_gemm_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "w4a16_gemm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                            _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_size,
                            _c_void_p]),
    "w4a16_moe_gemm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                _c_void_p]),
    "w4_test_stalled_gemm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                      _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "w4_test_prefill_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_c_int)]),
    "w4a16_gemm_bias": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                 _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                 _c_void_p, _c_size, _c_void_p]),
    "w4_dequant": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int,
                            _c_int, _c_int, _c_void_p, _c_void_p]),
    "w4_device_status": (_c_int, [ctypes.POINTER(ctypes.c_int32), _c_int]),
    "w4a16_gemm_noalloc": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                    _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_void_p]),
    "w4a8_gemm_workspace_size": (_c_size, [_c_int, _c_int]),
    "w4a8_gemm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int,
                           _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_size, _c_void_p]),
}


class W4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libw4a16.so (built in-tree); raise if it is missing."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def w4_status_string(status: int) -> str:
    return lib().w4_status_string(status).decode()


def w4_last_cuda_error() -> str:
    return lib().w4_last_cuda_error().decode()


def w4_abi_version() -> int:
    return lib().w4_abi_version()


def _check(status: int):
    if status != W4_OK:
        msg = w4_status_string(status)
        if status == W4_ERR_CUDA:
            msg += f" ({w4_last_cuda_error()})"
        raise W4Error(status, msg)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device_index: Optional[int] = None) -> Optional[int]:
    """The cudaStream_t handle to pass: `stream` itself (a torch stream or a raw
    handle), else torch's current stream on `device_index` (the current device
    when None)."""
    if stream is None:
        if not torch.cuda.is_available():
            return None
        if _RAW_STREAM is not None:
            if device_index is None:
                device_index = torch.cuda.current_device()
            return _RAW_STREAM(device_index)
        return torch.cuda.current_stream(device_index).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(dtype) -> int:
    if dtype in (W4_F16, W4_BF16):
        return dtype
    if dtype in (torch.float16, "fp16", "float16"):
        return W4_F16
    if dtype in (torch.bfloat16, "bf16", "bfloat16"):
        return W4_BF16
    raise ValueError(f"unsupported activation dtype {dtype}")


# --------------------------------------------------------------------------- #
# Raw entry points (same names and argument order as the C ABI)                 #
# --------------------------------------------------------------------------- #
def w4_repack_sizes(K: int, N: int, group: int, layout: int):
    a, b, c = _c_size(), _c_size(), _c_size()
    _check(lib().w4_repack_sizes(K, N, group, layout, ctypes.byref(a), ctypes.byref(b),
                                 ctypes.byref(c)))
    return a.value, b.value, c.value


def w4_repack_awq(qweight, qzeros, scales, K, N, group, dtype, layout, qw_out, zeros_out,
                  scales_out, stream=None):
    _check(lib().w4_repack_awq(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group,
                               dtype_code(dtype), layout, _ptr(qw_out), _ptr(zeros_out),
                               _ptr(scales_out), _stream(stream)))


def w4_repack_gptq(qweight, qzeros, scales, g_idx, K, N, group, dtype, layout, qw_out, zeros_out,
                   scales_out, perm_out=None, status_out=None, stream=None):
    _check(lib().w4_repack_gptq(_ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), K, N,
                                group, dtype_code(dtype), layout, _ptr(qw_out), _ptr(zeros_out),
                                _ptr(scales_out), _ptr(perm_out), _ptr(status_out),
                                _stream(stream)))


def w4a16_gemm_workspace_size(M, N, K, group, dtype, has_perm) -> int:
    return lib().w4a16_gemm_workspace_size(M, N, K, group, dtype_code(dtype), int(bool(has_perm)))


def w4a16_gemm(x, qw, scales, zeros, perm, y, M, N, K, group, dtype, workspace=None,
               workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().w4a16_gemm(_ptr(x), _ptr(qw), _ptr(scales), _ptr(zeros), _ptr(perm), _ptr(y),
                            M, N, K, group, dtype_code(dtype), _ptr(workspace), workspace_bytes,
                            _stream(stream)))


def w4a16_gemm_bias(x, qw, scales, zeros, perm, bias, y, M, N, K, group, dtype, workspace=None,
                    workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().w4a16_gemm_bias(_ptr(x), _ptr(qw), _ptr(scales), _ptr(zeros), _ptr(perm),
                                 _ptr(bias), _ptr(y), M, N, K, group, dtype_code(dtype),
                                 _ptr(workspace), workspace_bytes, _stream(stream)))


def w4a16_moe_gemm(x, qw, scales, zeros, expert_offsets, y, num_experts, max_rows_per_expert,
                   total_rows, N, K, group, dtype, stream=None):
    _check(lib().w4a16_moe_gemm(_ptr(x), _ptr(qw), _ptr(scales), _ptr(zeros), _ptr(expert_offsets),
                                _ptr(y), num_experts, max_rows_per_expert, total_rows, N, K, group,
                                dtype_code(dtype), _stream(stream)))


class RepackedExperts:
    """Device buffers of an MoE layer's experts, one expert after another."""

    def __init__(self, E, K, N, group, dtype, qw, zeros, scales):
        self.E, self.K, self.N, self.group, self.dtype = E, K, N, group, dtype
        self.qw, self.zeros, self.scales = qw, zeros, scales


def repack_awq_experts(qweights, qzeros, scales, K, N, group, dtype, stream=None):
    """Per-expert w4_repack_awq (TILE layout) into stacked buffers: qweights /
    qzeros / scales are sequences of the experts' checkpoint tensors (qzeros
    entries may be None for symmetric experts)."""
    E = len(qweights)
    qw_b, z_b, s_b = w4_repack_sizes(K, N, group, W4_LAYOUT_TILE)
    dev = qweights[0].device
    qw = torch.empty(E * qw_b // 4, dtype=torch.int32, device=dev)
    zeros = torch.empty(E * z_b // 4, dtype=torch.int32, device=dev)
    sc = torch.empty(E * s_b // 2, dtype=_half_dtype(dtype), device=dev)
    nq, nz, ns = qw_b // 4, z_b // 4, s_b // 2
    for e in range(E):
        w4_repack_awq(qweights[e], qzeros[e], scales[e], K, N, group, dtype, W4_LAYOUT_TILE,
                      qw[e * nq:(e + 1) * nq], zeros[e * nz:(e + 1) * nz],
                      sc[e * ns:(e + 1) * ns], stream)
    return RepackedExperts(E, K, N, group, dtype, qw, zeros, sc)


def moe_linear(x, experts: RepackedExperts, expert_offsets, max_rows_per_expert, y=None,
               stream=None):
    """y[m] = x[m] · W_e for the rows m of expert e ([off[e], off[e+1]), x sorted
    by expert); expert_offsets: int32 [E + 1] on the device."""
    T = x.shape[0]
    if y is None:
        y = torch.empty((T, experts.N), dtype=x.dtype, device=x.device)
    w4a16_moe_gemm(x, experts.qw, experts.scales, experts.zeros, expert_offsets, y, experts.E,
                   max_rows_per_expert, T, experts.N, experts.K, experts.group, experts.dtype,
                   stream)
    return y


def w4_test_stalled_gemm(x, qw, scales, zeros, y, M, N, K, group, dtype, stream=None):
    """The small-M GEMM with its weight copies withheld (the timeout test hook)."""
    _check(lib().w4_test_stalled_gemm(_ptr(x), _ptr(qw), _ptr(scales), _ptr(zeros), _ptr(y), M, N,
                                      K, group, dtype_code(dtype), _stream(stream)))


def w4_test_prefill_plan(M, N, K, sm_count):
    """The large-M kernel's plan for an M x N x K call on sm_count SMs (host
    only): (rows per tile, output tiles, split tiles, K slices of each)."""
    out = (_c_int * 4)()
    _check(lib().w4_test_prefill_plan(M, N, K, sm_count, out))
    return tuple(out)


def w4a16_gemm_noalloc(x, qw, scales, zeros, perm, y, M, N, K, group, dtype, stream=None):
    """w4a16_gemm for callers that cannot allocate device memory: act-order
    staging goes to the library's static device array instead of a workspace."""
    _check(lib().w4a16_gemm_noalloc(_ptr(x), _ptr(qw), _ptr(scales), _ptr(zeros), _ptr(perm),
                                    _ptr(y), M, N, K, group, dtype_code(dtype), _stream(stream)))


def w4a8_gemm_workspace_size(M, K) -> int:
    return lib().w4a8_gemm_workspace_size(M, K)


def w4a8_gemm(x, qw, scales, zeros, y, M, N, K, group, dtype, workspace, workspace_bytes=None,
              stream=None):
    """INT4 weights x per-tensor FP8 activations (quantised on the device)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().w4a8_gemm(_ptr(x), _ptr(qw), _ptr(scales), _ptr(zeros), _ptr(y), M, N, K, group,
                           dtype_code(dtype), _ptr(workspace), workspace_bytes, _stream(stream)))


def w4_device_status(clear: bool = False) -> int:
    v = ctypes.c_int32(0)
    _check(lib().w4_device_status(ctypes.byref(v), int(bool(clear))))
    return v.value


def w4_dequant(qw, scales, zeros, K, N, group, dtype, layout, out_f32, w_out, stream=None):
    _check(lib().w4_dequant(_ptr(qw), _ptr(scales), _ptr(zeros), K, N, group, dtype_code(dtype),
                            layout, int(bool(out_f32)), _ptr(w_out), _stream(stream)))


# --------------------------------------------------------------------------- #
# Convenience: allocate outputs with torch, then call the entry points          #
# --------------------------------------------------------------------------- #
class RepackedLayer:
    """Device buffers of one repacked layer (what the GEMM reads)."""

    def __init__(self, K, N, group, dtype, layout, qw, zeros, scales, perm=None, status=None):
        self.K, self.N, self.group, self.dtype, self.layout = K, N, group, dtype, layout
        self.qw, self.zeros, self.scales, self.perm, self.status = qw, zeros, scales, perm, status


def _half_dtype(dtype) -> torch.dtype:
    return torch.bfloat16 if dtype_code(dtype) == W4_BF16 else torch.float16


def _alloc_repacked(K, N, group, dtype, layout, device):
    qw_b, z_b, s_b = w4_repack_sizes(K, N, group, layout)
    qw = torch.empty(qw_b // 4, dtype=torch.int32, device=device)
    zeros = torch.empty(z_b // 4, dtype=torch.int32, device=device)
    scales = torch.empty(s_b // 2, dtype=_half_dtype(dtype), device=device)
    return qw, zeros, scales


def repack_awq(qweight, qzeros, scales, K, N, group, dtype, layout=W4_LAYOUT_TILE, stream=None):
    qw, zeros, sc = _alloc_repacked(K, N, group, dtype, layout, qweight.device)
    w4_repack_awq(qweight, qzeros, scales, K, N, group, dtype, layout, qw, zeros, sc, stream)
    return RepackedLayer(K, N, group, dtype, layout, qw, zeros, sc)


def repack_gptq(qweight, qzeros, scales, g_idx, K, N, group, dtype, layout=W4_LAYOUT_TILE,
                stream=None):
    qw, zeros, sc = _alloc_repacked(K, N, group, dtype, layout, qweight.device)
    perm = status = None
    if g_idx is not None:
        perm = torch.empty(K, dtype=torch.int32, device=qweight.device)
        status = torch.full((4,), -1, dtype=torch.int32, device=qweight.device)
    w4_repack_gptq(qweight, qzeros, scales, g_idx, K, N, group, dtype, layout, qw, zeros, sc,
                   perm, status, stream)
    return RepackedLayer(K, N, group, dtype, layout, qw, zeros, sc, perm, status)


_WORKSPACES: dict = {}


def gemm_workspace(nbytes: int, device, stream=None):
    """A workspace of at least nbytes on `device` for calls on `stream`, kept
    and reused across calls (calls on one stream run in order, so they can
    share it, and no call allocates device memory once it is big enough). It is
    allocated on that stream, so when a larger one replaces it the caching
    allocator hands the old block out again only in that stream's order (after
    the calls that may still be reading it)."""
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    handle = _stream(stream, idx)
    key = (idx, handle)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        if stream is None:
            ctx = contextlib.nullcontext()      # the current stream is the one used
        elif isinstance(stream, int):
            ext = (torch.cuda.ExternalStream(stream, device=torch.device("cuda", idx)) if stream
                   else torch.cuda.default_stream(idx))
            ctx = torch.cuda.stream(ext)
        else:
            ctx = torch.cuda.stream(stream)
        with ctx:
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _WORKSPACES[key] = ws
    return ws


_WS_SIZES: dict = {}
_WS_SIZES_MAX = 4096


def _workspace_size_cached(M, layer: RepackedLayer, device) -> int:
    """w4a16_gemm_workspace_size for (device, M, layer shape), remembered: the
    size depends only on those (and on the device's SM count), and linear()
    would otherwise pay a second library call on every call."""
    dev = device.index if device.index is not None else -1
    key = (dev, M, layer.N, layer.K, layer.group, layer.dtype, layer.perm is not None)
    need = _WS_SIZES.get(key)
    if need is None:
        need = w4a16_gemm_workspace_size(M, layer.N, layer.K, layer.group, layer.dtype,
                                         layer.perm is not None)
        if len(_WS_SIZES) >= _WS_SIZES_MAX:
            _WS_SIZES.clear()
        _WS_SIZES[key] = need
    return need


def linear_fp8(x, layer: RepackedLayer, y=None, workspace=None, stream=None):
    """y = x · W with the activations quantised per tensor to e4m3 on the device
    and the product on the fp8 tensor cores (w4a8_gemm); layer without act-order,
    group 128 or -1."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, layer.N), dtype=x.dtype, device=x.device)
    if M == 0:
        return y
    if workspace is None:
        workspace = gemm_workspace(w4a8_gemm_workspace_size(M, layer.K), x.device, stream)
    w4a8_gemm(x, layer.qw, layer.scales, layer.zeros, y, M, layer.N, layer.K, layer.group,
              layer.dtype, workspace, None, stream)
    return y


def linear(x, layer: RepackedLayer, y=None, workspace=None, stream=None, bias=None):
    """y = x · W (+ bias) for a TILE-layout layer; x is [M, K] fp16/bf16 on the
    device, bias [N] in the same dtype or None. Without `workspace`, the one kept
    for (device, stream) is used (grown as needed)."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, layer.N), dtype=x.dtype, device=x.device)
    need = _workspace_size_cached(M, layer, x.device)
    if need and workspace is None:
        workspace = gemm_workspace(need, x.device, stream)
    handle = _stream(stream, x.device.index)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().w4a16_gemm_bias(x.data_ptr(), layer.qw.data_ptr(), layer.scales.data_ptr(),
                                 layer.zeros.data_ptr(), _ptr(layer.perm), _ptr(bias),
                                 y.data_ptr(), M, layer.N, layer.K, layer.group,
                                 dtype_code(layer.dtype), _ptr(workspace), ws_bytes, handle))
    return y
