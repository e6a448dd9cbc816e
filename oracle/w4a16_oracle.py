"""CPU oracle for the W4A16 (INT4 weight-only, group-quantised) linear layer.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference arm may import this module. The library's
product path never calls it, and it shares no code, table or helper with the
CUDA kernels: it re-derives every quantity from the checkpoint words itself.

Cited pages (title, site):
  [QL]  "量化层加载:AWQ / GPTQ / Marlin / fp8" (vllm-arch-zh.pages.dev, model-loading/quant)
  [AWQ] "vLLM AWQ 4-bit 量化实践：AutoAWQ 模型加载、推理配置与内核调度原理" (discosf.com)
  [QB]  "vLLM 学习手册 · 01. 量化（Quantization）" (jwzheng96.github.io)

What the path computes and where the pages say so:
  1. AWQ unpack ([AWQ] §5.1 and §5.3): a qweight word holds 8 output columns;
     column 8c+j sits at nibble REVERSE_AWQ_PACK_ORDER[j], read as
     (word >> shift) & 0xF on the unsigned bits.
  2. Standard (GPTQ-like) repack ([QL] 设计动机 "AWQ → GPTQ 格式转换";
     [AWQ] §5.1): qweight repacked along the input dim to [K/8, N] with row
     8r+i at bits 4i..4i+3 (the standard order: index i at bit 4i); qzeros
     reordered to the standard order along N.
  3. Kernel tile layout ([QL] 关键文件, MarlinLinearKernel "重排成 ... 期望布局"):
     the GEMM kernels read a layout of this library's own choosing, defined in
     `tile_pos` below and in include/w4a16.h.
  4. Act-order ([QL] 设计动机 "desc_act / g_idx"): input row k belongs to group
     g_idx[k]; the kernels sort rows by group (stable) and gather x by that
     permutation. The oracle never uses the permutation for arithmetic.
  5. Dequantisation ([AWQ] §5.3): W[k, n] = (q[k, n] - z[g(k), n]) * s[g(k), n]
     with g(k) = k // group, or g_idx[k]. Exact in fp32: |q - z| <= 15 needs 4
     bits and the scale has at most 11 significant bits.
  6. GEMM: y[m, n] = sum_k x[m, k] * W[k, n], accumulated in fp64.
  7. Grouped GEMM over MoE experts ([AWQ] §5.4, 4-bit expert weights): rows of x
     sorted by expert, expert e owning rows [off[e], off[e+1]); each row is
     multiplied by its own expert's W_e, i.e. item 6 per expert.

Parity pins for every function live in tests/test_oracle_pins.py. The TILE
layout is this library's own format: its pins are bijectivity, round trip and
agreement of the scalar index function with the vectorised packer.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

# [AWQ] §5.1: AWQ stores column j of an 8-column block at nibble position
# REVERSE_AWQ_PACK_ORDER[j]; [AWQ] §5.3 unpacks with shifts built from it.
REVERSE_AWQ_PACK_ORDER = (0, 4, 1, 5, 2, 6, 3, 7)
# [AWQ] §5.1: pack_factor = 32 // 4.
PACK_FACTOR = 32 // 4
# [AWQ] §5.3: group sizes the AWQ kernels accept (-1 = one group over all of K).
SUPPORTED_GROUPS = (-1, 32, 64, 128)

FP16 = "fp16"
BF16 = "bf16"


# --------------------------------------------------------------------------- #
# Half-precision bit patterns <-> float (the oracle's own conversions).
# --------------------------------------------------------------------------- #
def half_bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of fp16 / bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits).astype(np.uint16)
    if dtype == FP16:
        return b.view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_f64_to_half_bits(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest fp16 / bf16 (ties to even), as bits.

    Used only on values that are exact in fp32 (dequantised weights), so the
    float64 -> float32 step below is exact and the result is a single rounding.
    """
    f32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    if dtype == FP16:
        return f32.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = f32.view(np.uint32).astype(np.uint64)
        lsb = (u >> 16) & 1
        return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    raise ValueError(dtype)


def round_f64_to_half_value(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 -> fp16 / bf16 -> float64, with a single rounding step.

    For general float64 input the two-step route through fp32 could double-round,
    so the rounding is done directly on the float64 value here.
    """
    v = np.asarray(v, dtype=np.float64)
    mant_bits = 11 if dtype == FP16 else 8          # significant bits incl. implicit 1
    out = np.zeros_like(v)
    nz = v != 0
    e = np.floor(np.log2(np.abs(v[nz])))
    if dtype == FP16:
        e = np.maximum(e, -14.0)                    # fp16 subnormal spacing 2^-24
    ulp = np.exp2(e - (mant_bits - 1))
    out[nz] = np.rint(v[nz] / ulp) * ulp            # np.rint is round-half-even
    return out


# --------------------------------------------------------------------------- #
# 1. AWQ unpack                                                                 #
# --------------------------------------------------------------------------- #
def unpack_awq(words: np.ndarray) -> np.ndarray:
    """[R, C] AWQ int32 words -> [R, 8C] codes (uint8).

    [AWQ] §5.1 / §5.3: column 8c+j = (word >> 4*REVERSE_AWQ_PACK_ORDER[j]) & 0xF,
    with the word taken as unsigned bits.
    """
    u = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    R, C = u.shape
    out = np.empty((R, C, PACK_FACTOR), dtype=np.uint8)
    for j in range(PACK_FACTOR):
        out[:, :, j] = (u >> (4 * REVERSE_AWQ_PACK_ORDER[j])) & 0xF
    return out.reshape(R, C * PACK_FACTOR)


# --------------------------------------------------------------------------- #
# 2. Standard packing and the AWQ -> standard repack                            #
# --------------------------------------------------------------------------- #
def unpack_rows_std(words: np.ndarray) -> np.ndarray:
    """[K/8, N] standard words -> [K, N] codes; row 8r+i at bits 4i..4i+3."""
    u = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    R, N = u.shape
    out = np.empty((R, PACK_FACTOR, N), dtype=np.uint8)
    for i in range(PACK_FACTOR):
        out[:, i, :] = (u >> (4 * i)) & 0xF
    return out.reshape(R * PACK_FACTOR, N)


def pack_rows_std(codes: np.ndarray) -> np.ndarray:
    """[K, N] codes -> [K/8, N] int32; row 8r+i at bits 4i..4i+3 ([AWQ] §5.1)."""
    K, N = codes.shape
    c = np.asarray(codes).astype(np.int64).reshape(K // PACK_FACTOR, PACK_FACTOR, N)
    acc = np.zeros((K // PACK_FACTOR, N), dtype=np.int64)
    for i in range(PACK_FACTOR):
        acc += c[:, i, :] << (4 * i)
    return acc.astype(np.uint32).view(np.int32)


def unpack_cols_std(words: np.ndarray) -> np.ndarray:
    """[R, N/8] standard words -> [R, N] codes; column 8c+i at bits 4i..4i+3."""
    u = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    R, C = u.shape
    out = np.empty((R, C, PACK_FACTOR), dtype=np.uint8)
    for i in range(PACK_FACTOR):
        out[:, :, i] = (u >> (4 * i)) & 0xF
    return out.reshape(R, C * PACK_FACTOR)


def pack_cols_std(codes: np.ndarray) -> np.ndarray:
    """[R, N] codes -> [R, N/8] int32; column 8c+i at bits 4i..4i+3."""
    R, N = codes.shape
    c = np.asarray(codes).astype(np.int64).reshape(R, N // PACK_FACTOR, PACK_FACTOR)
    acc = np.zeros((R, N // PACK_FACTOR), dtype=np.int64)
    for i in range(PACK_FACTOR):
        acc += c[:, :, i] << (4 * i)
    return acc.astype(np.uint32).view(np.int32)


def repack_awq_to_std(qweight: np.ndarray, qzeros: np.ndarray):
    """AWQ (qweight [K, N/8], qzeros [G, N/8]) -> standard (qw [K/8, N], zeros [G, N/8]).

    [QL] 设计动机 / [AWQ] §5.1: unpack with the reverse order, then repack
    qweight along the input dim in the standard bit order; qzeros keep their
    [G, N/8] shape and take the standard order along N.
    """
    q = unpack_awq(qweight)
    z = unpack_awq(qzeros)
    return pack_rows_std(q), pack_cols_std(z)


# --------------------------------------------------------------------------- #
# 3. The kernel tile layout (this library's own format)                         #
# --------------------------------------------------------------------------- #
# Within a tile word, nibble position p holds row offset TILE_NIBBLE_ROW[p] of the
# word's 8 consecutive rows.
TILE_NIBBLE_ROW = (0, 2, 4, 6, 1, 3, 5, 7)
TILE_ATOM_K = 64
TILE_ATOM_N = 16
TILE_ATOM_WORDS = 128
TILE_GROUP_TILES = 8          # 16-column tiles per column group (128 columns)


def tile_words(K: int, N: int) -> int:
    """Number of TILE words of a K x N layer: N is padded to whole 128-column groups."""
    return K * (-(-N // (TILE_ATOM_N * TILE_GROUP_TILES)) * TILE_ATOM_N * TILE_GROUP_TILES) // 8


def tile_atom(kb: int, nt: int, K: int) -> int:
    """Index of atom (k-atom kb, column tile nt): column group outermost, then k, then the tile."""
    A = K // TILE_ATOM_K
    return ((nt // TILE_GROUP_TILES) * A + kb) * TILE_GROUP_TILES + nt % TILE_GROUP_TILES


def tile_pos(k: int, n: int, K: int, N: int):
    """(word index, nibble position) of code (k, n) in the TILE layout.

    The layout (also written out in include/w4a16.h):
      * atoms of 16 columns x 64 rows, 128 words each; columns are taken in
        groups of 8 tiles (128 columns, the last group padded with zero atoms)
        and atom (kb, nt) sits at index
        ((nt // 8) * (K // 64) + kb) * 8 + nt % 8, kb = k // 64, nt = n // 16,
        so one group's atoms at one k-atom are 8 consecutive atoms and a group's
        whole K range is one contiguous run;
      * inside an atom, word 4*lane + j with lane = 4*gg + t, where
        gg = n % 8, t = (k % 32) // 8, j = 2 * ((k % 64) // 32) + (n % 16) // 8;
      * the word holds rows 8t..8t+7 (plus the atom/half offsets) of column n,
        row offset TILE_NIBBLE_ROW[p] at nibble position p.
    """
    assert K % TILE_ATOM_K == 0 and N % TILE_ATOM_N == 0
    a = tile_atom(k // TILE_ATOM_K, n // TILE_ATOM_N, K)
    kk = k % TILE_ATOM_K
    nn = n % TILE_ATOM_N
    gg = nn % 8
    t = (kk % 32) // 8
    j = 2 * (kk // 32) + nn // 8
    lane = 4 * gg + t
    word = a * TILE_ATOM_WORDS + 4 * lane + j
    p = TILE_NIBBLE_ROW.index(kk % 8)
    return word, p


def tile_pack(codes: np.ndarray) -> np.ndarray:
    """[K, N] codes -> TILE words (int32, `tile_words(K, N)` of them), per `tile_pos`.

    Vectorised form of `tile_pos`: with N padded by zero codes to Np (a
    multiple of 128), code (k, n) with
      k = 64*kb + 32*jh + 8*t + e,  n = 128*cg + 16*w + 8*jl + gg
    goes to word (((cg*(K/64) + kb)*8 + w)*128 + 4*(4*gg + t) + 2*jh + jl),
    nibble position TILE_NIBBLE_ROW.index(e).
    """
    K, N = codes.shape
    Np = tile_words(K, N) * 8 // K
    c = np.zeros((K, Np), dtype=np.uint32)
    c[:, :N] = np.asarray(codes).astype(np.uint32)
    # axes: kb, jh, t, e, cg, w, jl, gg
    c = c.reshape(K // 64, 2, 4, 8, Np // 128, 8, 2, 8)
    # -> cg, kb, w, gg, t, jh, jl, e
    c = c.transpose(4, 0, 5, 7, 2, 1, 6, 3)
    words = np.zeros(c.shape[:-1], dtype=np.uint32)
    for p, e in enumerate(TILE_NIBBLE_ROW):
        words |= c[..., e] << np.uint32(4 * p)
    return words.reshape(-1).view(np.int32)


def tile_unpack(words: np.ndarray, K: int, N: int) -> np.ndarray:
    """Inverse of `tile_pack`: TILE words -> [K, N] codes (the padding dropped)."""
    Np = tile_words(K, N) * 8 // K
    u = np.asarray(words).view(np.uint32).reshape(Np // 128, K // 64, 8, 8, 4, 2, 2)
    c = np.empty(u.shape + (8,), dtype=np.uint8)
    for p, e in enumerate(TILE_NIBBLE_ROW):
        c[..., e] = (u >> np.uint32(4 * p)) & 0xF
    # cg, kb, w, gg, t, jh, jl, e -> kb, jh, t, e, cg, w, jl, gg
    c = c.transpose(1, 5, 4, 7, 0, 2, 6, 3)
    return np.ascontiguousarray(c).reshape(K, Np)[:, :N]


# --------------------------------------------------------------------------- #
# 4. Act-order                                                                  #
# --------------------------------------------------------------------------- #
def act_order_perm(g_idx: np.ndarray) -> np.ndarray:
    """Stable sort of input rows by group: perm[j] = j-th row in (g_idx, k) order.

    [QL] 设计动机 (desc_act / g_idx): each input row carries its group index.
    Sorting rows by group (ties kept in ascending k) makes every group contiguous.
    """
    return np.argsort(np.asarray(g_idx), kind="stable").astype(np.int32)


def gidx_is_regular(g_idx: np.ndarray, group: int) -> bool:
    """True when every group 0..K/group-1 owns exactly `group` rows."""
    g = np.asarray(g_idx)
    K = g.shape[0]
    if K % group:
        return False
    G = K // group
    if g.min(initial=0) < 0 or g.max(initial=0) >= G:
        return False
    return bool(np.all(np.bincount(g, minlength=G) == group))


# --------------------------------------------------------------------------- #
# 5. Dequantisation                                                             #
# --------------------------------------------------------------------------- #
def group_of_rows(K: int, group: int, g_idx: Optional[np.ndarray] = None) -> np.ndarray:
    """g(k): k // group, or g_idx[k] under act-order; group -1 means one group."""
    if g_idx is not None:
        return np.asarray(g_idx).astype(np.int64)
    if group == -1:
        group = K
    return np.arange(K, dtype=np.int64) // group


def dequant(q: np.ndarray, z: np.ndarray, s: np.ndarray, g_of_k: np.ndarray,
            cols: Optional[np.ndarray] = None) -> np.ndarray:
    """W[k, n] = (q[k, n] - z[g(k), n]) * s[g(k), n], as exact float32.

    [AWQ] §5.3: b = (b >> shifts) & 0xF; zeros = (zeros >> shifts) & 0xF;
    b = (b - zeros) * scales. q: [K, N] codes; z: [G, N] codes; s: [G, N]
    float64 scale values; `cols` restricts the result to those columns.
    """
    if cols is not None:
        q = q[:, cols]
        z = z[:, cols]
        s = s[:, cols]
    diff = q.astype(np.int64) - z[g_of_k].astype(np.int64)
    W = diff.astype(np.float64) * s[g_of_k]
    return W.astype(np.float32)


# --------------------------------------------------------------------------- #
# 6. GEMM                                                                       #
# --------------------------------------------------------------------------- #
def gemm(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x @ W with both operands widened to float64 (the product in fp64)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


# --------------------------------------------------------------------------- #
# Whole-layer references                                                        #
# --------------------------------------------------------------------------- #
# Zero point of every code of a symmetric checkpoint (AWQ zero_point=False, [AWQ]
# §二 quant_config: no qzeros are stored). Reading: the 4-bit codes are signed
# values stored with an offset of 8, the middle of the range, so W = (q - 8) * s.
SYMMETRIC_ZERO = 8


def layer_codes(qweight, qzeros, scales_bits, dtype: str, fmt: str):
    """Checkpoint words -> (q [K, N], z [G, N], s [G, N] float64). qzeros None:
    a symmetric checkpoint, z = SYMMETRIC_ZERO everywhere."""
    if fmt == "awq":
        q = unpack_awq(qweight)
        z = unpack_awq(qzeros) if qzeros is not None else None
    elif fmt == "gptq":
        q = unpack_rows_std(qweight)
        z = unpack_cols_std(qzeros) if qzeros is not None else None
    else:
        raise ValueError(fmt)
    s = half_bits_to_f64(scales_bits, dtype)
    if z is None:
        z = np.full(s.shape, SYMMETRIC_ZERO, dtype=np.uint8)
    return q, z, s


def reference_y(x_bits, qweight, qzeros, scales_bits, group: int, dtype: str, fmt: str,
                g_idx=None, rows=None, cols=None, col_chunk: int = 4096,
                bias_bits=None) -> np.ndarray:
    """fp64 y for the layer, optionally on a subset of rows and/or columns.

    Dequantises column chunks so memory stays bounded on the largest layers.
    bias_bits ([N] half bits): y[m, n] += bias[n], the bias of the layer's
    apply ([QL] 关键文件: apply_weights(layer, x, bias)).
    """
    q, z, s = layer_codes(qweight, qzeros, scales_bits, dtype, fmt)
    K, N = q.shape
    x = half_bits_to_f64(x_bits, dtype)
    if rows is not None:
        x = x[np.asarray(rows)]
    gk = group_of_rows(K, group, g_idx)
    col_list = np.arange(N) if cols is None else np.asarray(cols)
    y = np.empty((x.shape[0], col_list.shape[0]), dtype=np.float64)
    for c0 in range(0, col_list.shape[0], col_chunk):
        cc = col_list[c0:c0 + col_chunk]
        y[:, c0:c0 + len(cc)] = gemm(x, dequant(q, z, s, gk, cols=cc))
    if bias_bits is not None:
        y += half_bits_to_f64(np.asarray(bias_bits), dtype)[col_list][None, :]
    return y


def moe_reference_y(x_bits, experts, offsets, group: int, dtype: str, fmt: str) -> np.ndarray:
    """fp64 y of the grouped GEMM over an MoE layer's experts ([AWQ] §5.4): for
    every expert e, y[m] = x[m] . W_e for off[e] <= m < off[e+1]. experts: one
    (qweight, qzeros, scales_bits) checkpoint triple per expert; offsets: E + 1
    non-decreasing row offsets from 0 to the row count of x. Rows outside every
    range do not exist (off[E] = rows of x)."""
    off = [int(v) for v in offsets]
    if off[0] != 0 or off[-1] != len(x_bits) or any(b < a for a, b in zip(off, off[1:])):
        raise ValueError("offsets must run from 0 to the row count, non-decreasing")
    if len(off) != len(experts) + 1:
        raise ValueError("one offset more than experts")
    N = half_bits_to_f64(experts[0][2], dtype).shape[1]
    y = np.zeros((len(x_bits), N), dtype=np.float64)
    for e, (qweight, qzeros, scales_bits) in enumerate(experts):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            y[r0:r1] = reference_y(x_bits[r0:r1], qweight, qzeros, scales_bits, group, dtype, fmt)
    return y


def rel_err(y: np.ndarray, y_ref: np.ndarray) -> float:
    """max |y - y_ref| / max |y_ref|, in float64."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    den = np.max(np.abs(y_ref))
    if den == 0:
        return float(np.max(np.abs(y - y_ref)))
    return float(np.max(np.abs(y - y_ref)) / den)


def output_rounding_floor(y_ref: np.ndarray, dtype: str) -> float:
    """The error that rounding the exact y to the output dtype alone costs."""
    return rel_err(round_f64_to_half_value(y_ref, dtype), y_ref)
