"""Test helpers: make sure the library is built, move numpy arrays to the device."""
import os
import re
import threading

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")
_lock = threading.Lock()


def ensure_built():
    """Build libw4a16.so if it is missing (nvcc cross-compiles without a GPU)."""
    import int4_weight_only_repack_gb300 as w4
    from int4_weight_only_repack_gb300 import _build

    with _lock:
        if not os.path.exists(w4.library_path):
            _build.build()
    return w4.lib()


def declared_symbols():
    """Names of every function include/w4a16.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"W4_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def half_to_dev(bits, dtype, device="cuda"):
    """uint16 bit patterns -> torch fp16 / bf16 tensor on the device."""
    import torch
    t = to_dev(np.ascontiguousarray(bits).view(np.int16), device)
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def half_from_dev(t):
    """torch fp16 / bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rounded_w_reference(x_bits, L, group, fmt="awq"):
    """fp64 y with the weight rounded once to the activation dtype (the large-M
    kernel's B operand): a composition of oracle steps, used for a tight check."""
    from oracle import w4a16_oracle as oracle
    q, z, s = oracle.layer_codes(L.qweight, L.qzeros, L.scales, L.dtype, fmt)
    K = q.shape[0]
    W = oracle.dequant(q, z, s, oracle.group_of_rows(K, group, L.g_idx))
    Wr = oracle.half_bits_to_f64(oracle.round_f64_to_half_bits(W, L.dtype), L.dtype)
    return oracle.gemm(oracle.half_bits_to_f64(x_bits, L.dtype), Wr)
