"""Seeded synthetic inputs for the W4A16 layer: the one module both sides share.

This module plays the part of the checkpoint writer (the AWQ / GPTQ quantiser and
packer), which sits outside the repack + GEMM path. It draws float weights and
activations from seeded generators, quantises the weights with a per-(group,
column) asymmetric min/max rule (or, for symmetric layers, a max-abs rule with
the zero point fixed at 8 and no zeros stored) and stores the codes in the two
checkpoint formats the path reads. It holds none of the path's own arithmetic: no unpack,
no repack, no dequantisation and no matrix product. Both the CPU oracle (which
derives every code it uses by unpacking these words itself) and the CUDA path
consume exactly the arrays produced here.

Cited pages (title, site):
  [QL]  "量化层加载:AWQ / GPTQ / Marlin / fp8" (vllm-arch-zh.pages.dev, model-loading/quant)
  [AWQ] "vLLM AWQ 4-bit 量化实践：AutoAWQ 模型加载、推理配置与内核调度原理" (discosf.com)
  [QB]  "vLLM 学习手册 · 01. 量化（Quantization）" (jwzheng96.github.io)

Formats produced:
  * AWQ checkpoint: qweight int32 [K, N/8] packed along the output dim, qzeros
    int32 [K/g, N/8] packed the same way, scales [K/g, N] in the activation
    dtype ([QL] 数据流: the three parameter shapes; [AWQ] §5.1: pack factor
    32 // 4 = 8). Inside a word, nibble position p (bits 4p..4p+3) holds column
    8c + AWQ_PACK_ORDER[p]; AWQ_PACK_ORDER is the inverse of the reverse order
    [0, 4, 1, 5, 2, 6, 3, 7] that [AWQ] §5.1 prints.
  * GPTQ checkpoint (standard packing, [QL] 设计动机, [AWQ] §5.1): qweight int32
    [K/8, N] packed along the input dim with row 8r+i at bits 4i..4i+3, qzeros
    int32 [K/g, N/8] with column 8c+i at bits 4i..4i+3, scales [K/g, N], and the
    act-order g_idx int32 [K] ([QL] 设计动机: desc_act / g_idx).

Half-precision values travel as uint16 bit patterns (fp16 or bf16), so numpy
can hold bf16 without a bf16 dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

FP16 = "fp16"
BF16 = "bf16"

# Nibble position p of an AWQ word holds column AWQ_PACK_ORDER[p] of its 8-column
# block. This is the inverse permutation of the [0,4,1,5,2,6,3,7] order that
# [AWQ] §5.1 names _REVERSE_AWQ_PACK_ORDER.
AWQ_PACK_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


# --------------------------------------------------------------------------- #
# Workloads: Llama-2-shaped projection layers and one tiny layer.
# --------------------------------------------------------------------------- #
@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    shapes: tuple          # ((K, N, layer name), ...)
    ms: tuple              # activation row counts M
    dtype: str             # activation (= scale) dtype
    fmt: str               # "awq" or "gptq"
    act_order: bool
    group: int = 128


WORKLOADS = (
    Workload(0, "tiny_awq_k256_n256", ((256, 256, "tiny"),), (4,), FP16, "awq", False),
    Workload(1, "llama2_7b_decode",
             ((4096, 12288, "qkv"), (4096, 4096, "o_proj"),
              (4096, 22016, "gate_up"), (11008, 4096, "down")),
             (1, 4, 16), BF16, "awq", False),
    Workload(2, "llama2_7b_prefill",
             ((4096, 12288, "qkv"), (4096, 4096, "o_proj"),
              (4096, 22016, "gate_up"), (11008, 4096, "down")),
             (512, 2048, 4096), BF16, "awq", False),
    Workload(3, "llama2_13b_gptq_act_order",
             ((5120, 15360, "qkv"), (5120, 27648, "gate_up"), (13824, 5120, "down")),
             (1, 16, 1024), FP16, "gptq", True),
    Workload(4, "llama2_70b_sweep",
             ((8192, 10240, "qkv"), (8192, 57344, "gate_up"), (28672, 8192, "down")),
             (1, 2, 4, 8, 16, 32, 64, 128, 256, 1024, 4096), BF16, "awq", False),
)


# --------------------------------------------------------------------------- #
# Half-precision encodings (the generator's own; round to nearest even).
# --------------------------------------------------------------------------- #
def f32_to_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == FP16:
        return a.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = a.view(np.uint32).astype(np.uint64)
        nan = np.isnan(a)
        rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
        rounded[nan] = 0x7FC0
        return rounded
    raise ValueError(dtype)


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    if dtype == FP16:
        return b.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (b.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


# --------------------------------------------------------------------------- #
# Layer generation.
# --------------------------------------------------------------------------- #
@dataclass
class Layer:
    K: int
    N: int
    group: int
    dtype: str
    fmt: str                          # "awq" or "gptq"
    qweight: np.ndarray               # int32, AWQ [K, N/8] or GPTQ [K/8, N]
    qzeros: Optional[np.ndarray]      # int32 [G, N/8] (AWQ or standard order); None: symmetric
    scales: np.ndarray                # uint16 bits [G, N]
    g_idx: Optional[np.ndarray] = None  # int32 [K] (GPTQ act-order only)
    # Writer-side codes, kept for generator self-checks only.
    q: Optional[np.ndarray] = field(default=None, repr=False)
    z: Optional[np.ndarray] = field(default=None, repr=False)
    w: Optional[np.ndarray] = field(default=None, repr=False)


def _quantise_minmax(w: np.ndarray, group: int, g_idx: Optional[np.ndarray], dtype: str):
    """Asymmetric 4-bit min/max quantiser per (group, column).

    scale = (max - min) / 15 in fp32, stored in the activation dtype (1 when the
    group is constant); zero = clamp(rint(-min / scale), 0, 15); code =
    clamp(rint(w / scale) + zero, 0, 15). rint is round-half-even.
    """
    K, N = w.shape
    G = K // group
    if g_idx is None:
        order = np.arange(K)
        gk = order // group
    else:
        order = np.argsort(g_idx, kind="stable")
        gk = g_idx
    wg = w[order].reshape(G, group, N)
    mn = wg.min(axis=1)
    mx = wg.max(axis=1)
    del wg
    s32 = ((mx - mn) / np.float32(15.0)).astype(np.float32)
    s32[mx == mn] = 1.0
    s_bits = f32_to_bits(s32, dtype)
    s_eff = bits_to_f32(s_bits, dtype)
    z = np.clip(np.rint(-mn / s_eff), 0, 15).astype(np.uint8)
    q = np.empty((K, N), dtype=np.uint8)
    step = max(1, (1 << 24) // max(N, 1))
    for k0 in range(0, K, step):
        k1 = min(K, k0 + step)
        gg = gk[k0:k1]
        v = np.rint(w[k0:k1] / s_eff[gg]) + z[gg].astype(np.float32)
        q[k0:k1] = np.clip(v, 0, 15).astype(np.uint8)
    return q, z, s_bits


def _quantise_symmetric(w: np.ndarray, group: int, g_idx: Optional[np.ndarray], dtype: str):
    """Symmetric 4-bit quantiser per (group, column), zero point fixed at 8.

    scale = max|w| / 7 in fp32, stored in the activation dtype (1 when the
    group is all zeros); code = clamp(rint(w / scale) + 8, 0, 15).
    """
    K, N = w.shape
    G = K // group
    if g_idx is None:
        order = np.arange(K)
        gk = order // group
    else:
        order = np.argsort(g_idx, kind="stable")
        gk = g_idx
    amax = np.abs(w[order].reshape(G, group, N)).max(axis=1)
    s32 = (amax / np.float32(7.0)).astype(np.float32)
    s32[amax == 0] = 1.0
    s_bits = f32_to_bits(s32, dtype)
    s_eff = bits_to_f32(s_bits, dtype)
    q = np.empty((K, N), dtype=np.uint8)
    step = max(1, (1 << 24) // max(N, 1))
    for k0 in range(0, K, step):
        k1 = min(K, k0 + step)
        v = np.rint(w[k0:k1] / s_eff[gk[k0:k1]]) + np.float32(8.0)
        q[k0:k1] = np.clip(v, 0, 15).astype(np.uint8)
    return q, np.full((G, N), 8, dtype=np.uint8), s_bits


def _pack_awq(codes: np.ndarray) -> np.ndarray:
    """[R, C*8] codes -> [R, C] int32 words; column 8c+AWQ_PACK_ORDER[p] at nibble p."""
    R, C8 = codes.shape
    blk = codes.reshape(R, C8 // 8, 8).astype(np.uint32)
    out = np.zeros((R, C8 // 8), dtype=np.uint32)
    for p, col in enumerate(AWQ_PACK_ORDER):
        out |= blk[:, :, col] << np.uint32(4 * p)
    return out.view(np.int32)


def _pack_rows_std(codes: np.ndarray) -> np.ndarray:
    """[K, N] codes -> [K/8, N] int32 words; row 8r+i at nibble i."""
    K, N = codes.shape
    blk = codes.reshape(K // 8, 8, N).astype(np.uint32)
    out = np.zeros((K // 8, N), dtype=np.uint32)
    for i in range(8):
        out |= blk[:, i, :] << np.uint32(4 * i)
    return out.view(np.int32)


def _pack_cols_std(codes: np.ndarray) -> np.ndarray:
    """[R, N] codes -> [R, N/8] int32 words; column 8c+i at nibble i."""
    R, N = codes.shape
    blk = codes.reshape(R, N // 8, 8).astype(np.uint32)
    out = np.zeros((R, N // 8), dtype=np.uint32)
    for i in range(8):
        out |= blk[:, :, i] << np.uint32(4 * i)
    return out.view(np.int32)


def act_order_gidx(rng: np.random.Generator, K: int, group: int) -> np.ndarray:
    """g_idx[k] = P[k] // group for a seeded random permutation P of 0..K-1.

    Every group then holds exactly `group` input rows, scattered over K, which is
    what a desc_act GPTQ checkpoint carries ([QL] 设计动机, desc_act / g_idx).
    """
    P = rng.permutation(K)
    return (P // group).astype(np.int32)


def make_layer_from_rng(rng: np.random.Generator, K: int, N: int, group: int, dtype: str,
                        fmt: str = "awq", act_order: bool = False,
                        keep_codes: bool = False, keep_float: bool = False,
                        sigma: float = 0.02, symmetric: bool = False) -> Layer:
    """symmetric: no zero points (qzeros None), every code's zero point is 8."""
    w = rng.standard_normal((K, N), dtype=np.float32)
    w *= np.float32(sigma)
    g_idx = act_order_gidx(rng, K, group) if act_order else None
    quantise = _quantise_symmetric if symmetric else _quantise_minmax
    q, z, s_bits = quantise(w, group, g_idx, dtype)
    if fmt == "awq":
        if act_order:
            raise ValueError("AWQ checkpoints carry no g_idx")
        qweight = _pack_awq(q)
        qzeros = None if symmetric else _pack_awq(z)
    elif fmt == "gptq":
        qweight = _pack_rows_std(q)
        qzeros = None if symmetric else _pack_cols_std(z)
    else:
        raise ValueError(fmt)
    return Layer(K, N, group, dtype, fmt, qweight, qzeros, s_bits, g_idx,
                 q=q if keep_codes else None, z=z if keep_codes else None,
                 w=w if keep_float else None)


def make_x_from_rng(rng: np.random.Generator, M: int, K: int, dtype: str) -> np.ndarray:
    return f32_to_bits(rng.standard_normal((M, K), dtype=np.float32), dtype)


def layer_seed(cfg: int, layer: int):
    return [0, cfg, layer]


def x_seed(cfg: int, layer: int, M: int):
    return [0, cfg, layer, M]


def make_workload_layer(cfg: int, layer: int, **kw) -> Layer:
    """Layer `layer` of workload `cfg`, from its fixed seed."""
    wl = WORKLOADS[cfg]
    K, N, _ = wl.shapes[layer]
    if cfg == 0:
        rng = np.random.default_rng(0)
    else:
        rng = np.random.default_rng(layer_seed(cfg, layer))
    return make_layer_from_rng(rng, K, N, wl.group, wl.dtype, wl.fmt, wl.act_order, **kw)


def make_workload_x(cfg: int, layer: int, M: int) -> np.ndarray:
    wl = WORKLOADS[cfg]
    K = wl.shapes[layer][0]
    if cfg == 0:
        # The tiny layer uses one stream (seed 0): weights first, then x.
        rng = np.random.default_rng(0)
        rng.standard_normal((K, wl.shapes[0][1]), dtype=np.float32)
        return make_x_from_rng(rng, M, K, wl.dtype)
    return make_x_from_rng(np.random.default_rng(x_seed(cfg, layer, M)), M, K, wl.dtype)


def make_custom_layer(seed, K: int, N: int, group: int = 128, dtype: str = BF16,
                      fmt: str = "awq", act_order: bool = False, **kw) -> Layer:
    return make_layer_from_rng(np.random.default_rng(seed), K, N, group, dtype, fmt, act_order, **kw)


def make_custom_x(seed, M: int, K: int, dtype: str = BF16) -> np.ndarray:
    return make_x_from_rng(np.random.default_rng(seed), M, K, dtype)


# --------------------------------------------------------------------------- #
# The same writer on torch tensors (for the benchmark's large layers).
# --------------------------------------------------------------------------- #
def quantise_pack_torch(w, group: int, dtype: str, fmt: str = "awq", g_idx=None):
    """The min/max writer of _quantise_minmax and the packers above, written with
    torch ops so that it can run on the device: w is a float32 [K, N] tensor (on
    any device), g_idx an int32 [K] tensor or None. Returns (qweight, qzeros,
    scales) as torch tensors on w's device: int32 words in the AWQ or GPTQ
    format and scales as the activation dtype. The rule and the word formats are
    the numpy writer's; the two agree code for code on the same w."""
    import torch
    K, N = w.shape
    G = K // group
    if g_idx is None:
        gk = torch.arange(K, device=w.device) // group
        wg = w.view(G, group, N)
    else:
        gk = g_idx.long()
        wg = w[torch.argsort(gk, stable=True)].view(G, group, N)
    mn = wg.amin(dim=1)
    mx = wg.amax(dim=1)
    del wg
    s32 = (mx - mn) / 15.0
    s32 = torch.where(mx == mn, torch.ones_like(s32), s32)
    sdt = torch.bfloat16 if dtype == BF16 else torch.float16
    s_half = s32.to(sdt)                      # round to nearest even
    s_eff = s_half.float()
    z = torch.clamp(torch.round(-mn / s_eff), 0, 15)   # round half to even
    q = torch.empty((K, N), dtype=torch.uint8, device=w.device)
    step = max(1, (1 << 26) // max(N, 1))
    for k0 in range(0, K, step):
        k1 = min(K, k0 + step)
        gg = gk[k0:k1]
        v = torch.round(w[k0:k1] / s_eff[gg]) + z[gg]
        q[k0:k1] = torch.clamp(v, 0, 15).to(torch.uint8)
    z8 = z.to(torch.uint8)

    def pack_rows(codes):                    # [K, N] -> [K/8, N]; row 8r+i at nibble i
        R, C = codes.shape
        blk = codes.view(R // 8, 8, C).to(torch.int64)
        out = torch.zeros((R // 8, C), dtype=torch.int64, device=codes.device)
        for i in range(8):
            out |= blk[:, i, :] << (4 * i)
        return _i64_to_i32_words(out)

    if fmt == "awq":
        if g_idx is not None:
            raise ValueError("AWQ checkpoints carry no g_idx")
        qweight = _pack_cols_chunked(q, AWQ_PACK_ORDER)
        qzeros = _pack_cols_chunked(z8, AWQ_PACK_ORDER)
    elif fmt == "gptq":
        qweight = torch.cat([pack_rows(q[k0:k0 + 8192]) for k0 in range(0, K, 8192)])
        qzeros = _pack_cols_chunked(z8, tuple(range(8)))
    else:
        raise ValueError(fmt)
    return qweight, qzeros, s_half


def _i64_to_i32_words(v):
    """int64 tensor of values in [0, 2^32) -> int32 tensor of the same 32 bits."""
    import torch
    return torch.where(v >= (1 << 31), v - (1 << 32), v).to(torch.int32)


def _pack_cols_chunked(codes, order):
    """[R, C*8] uint8 codes -> [R, C] int32 words, column 8c+order[p] at nibble p
    (in row chunks, to bound the int64 temporaries)."""
    import torch
    R, C8 = codes.shape
    outs = []
    step = max(1, (1 << 26) // max(C8, 1))
    for r0 in range(0, R, step):
        blk = codes[r0:r0 + step].reshape(-1, C8 // 8, 8).to(torch.int64)
        out = torch.zeros(blk.shape[:2], dtype=torch.int64, device=codes.device)
        for p, col in enumerate(order):
            out |= blk[:, :, col] << (4 * p)
        outs.append(_i64_to_i32_words(out))
    return torch.cat(outs)


def make_layer_torch(seed: int, K: int, N: int, group: int, dtype: str, fmt: str = "awq",
                     act_order: bool = False, device="cuda", sigma: float = 0.02):
    """A seeded synthetic layer drawn and quantised with torch on `device`:
    W ~ N(0, sigma) in fp32 from torch.Generator(seed), g_idx (act-order) from a
    seeded permutation as act_order_gidx does, then quantise_pack_torch. Returns
    (qweight, qzeros, scales, g_idx or None) on `device`. The benchmark's large
    layers come from here; the parity tests use the numpy writer."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    w = torch.randn((K, N), generator=gen, device=device, dtype=torch.float32)
    w *= sigma
    g_idx = None
    if act_order:
        P = torch.randperm(K, generator=gen, device=device)
        g_idx = (P // group).to(torch.int32)
    out = quantise_pack_torch(w, group, dtype, fmt, g_idx)
    del w
    return (*out, g_idx)
