// Small-M (decode) W4A16 GEMM, streaming form: y[M][N] = x[M][K] · W, M <= 8.
//
// Decode is bound by streaming the packed weights from HBM ("vLLM 学习手册 01.
// 量化" §1: decode has FLOPs/Bytes ~ 1 and moving the weights dominates). This
// kernel is built so that nothing but that stream sits on a call's critical path:
//
//  * Persistent, one CTA per SM at most, 8 warps. The layer's columns are cut
//    into slabs of 32 (two 16-column TILE tiles, adjacent in memory at every
//    k-atom: one 1 KB run) and every CTA owns a contiguous range of slabs over
//    the whole of K, so no output needs partial sums from another CTA: no
//    cluster barrier, no workspace, no atomics. Inside the CTA the (slab,
//    k-atom) items are split evenly over the warps, each warp a contiguous run.
//  * Each warp streams its own items through a private ring in shared memory:
//    one TMA tensor copy (one lane issues it) brings CHUNK consecutive
//    k-atoms of its slab (a 4D box over the TILE words, 1 KB per k-atom) and
//    completes on the slot's mbarrier; the warp refills the slot as soon as
//    it has read it. Warps never wait for one another. A bulk L2 prefetch
//    runs L2_AHEAD items ahead of the copies. One 16-byte shared-memory load
//    per lane and tile is exactly the A-fragment set of four m16n8k16 MMAs in
//    the swapped form y^T = W^T · x^T (weight columns fill the MMA's 16 rows,
//    tokens its 8 columns).
//  * Before the kernel waits for its predecessor on the stream (programmatic
//    dependent launch) every warp has issued its first RING copies and the CTA
//    has started copying all the scales and zeros of its columns into shared
//    memory (cp.async): the weights, scales and zeros do not depend on the
//    previous kernel, so their DRAM latency overlaps its tail. x is read after
//    the wait, with 16-byte loads through L1 (every warp of the SM reads it).
//  * Dequantisation ("vLLM AWQ 4-bit 量化实践" §5.3: (b - zeros) * scales): one
//    LOP3 turns a nibble pair into MAGIC + q halves and one packed subtraction
//    of MAGIC + z forms q - z, exact in both types. The scale multiplies the
//    group's fp32 partial sum.
//  * At the end each warp stores the slabs it covered whole directly and puts
//    its partial slabs in shared memory; after one CTA barrier the partial
//    slabs are summed over the warps in a fixed order (deterministic) and
//    rounded once, bias included.
//  * Every mbarrier wait is bounded (one second): a timed-out wait records
//    W4_ERR_TIMEOUT in the library's device status word, raises the CTA's
//    abort flag, and the warp lets its copies in flight land (bounded again)
//    before the CTA exits.
#include <algorithm>
#include <mutex>

#include "decode_common.cuh"
#include "sm100_ptx.cuh"
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace w4 {

namespace {

using namespace sm100;
using dec::bounded_wait;
using dec::cp_async16;
using dec::cp_async8;
using dec::cp_async_wait_all;
using dec::drain_wait;
using dec::ldg_x;
using dec::prefetch_l2;

constexpr int SW = 8;                  // warps per CTA
constexpr int ST = SW * 32;            // threads per CTA
constexpr int ATOM_K = 64;             // rows of a TILE atom
constexpr int KROW_BYTES = 4096;       // a column group's eight atoms at one k-atom
constexpr int META_BUDGET = 72 * 1024; // shared memory for the CTA's scales and zeros
#ifndef W4_STREAM_L2_AHEAD
#define W4_STREAM_L2_AHEAD 24
#endif
constexpr double STREAM_MAX_BYTES_PER_SM = 96 * 1024;
#ifndef W4_STREAM_CTAS_PER_SM
#define W4_STREAM_CTAS_PER_SM 1
#endif
#ifndef W4_STREAM_CHUNK
#define W4_STREAM_CHUNK 4
#endif
#ifndef W4_STREAM_RING
#define W4_STREAM_RING 2
#endif
constexpr int L2_AHEAD = W4_STREAM_L2_AHEAD;  // items a warp prefetches into L2 ahead of its copies
constexpr int CHUNK = W4_STREAM_CHUNK;        // k-atoms (1 KB each) per copy
constexpr int RING = W4_STREAM_RING;          // copies in flight per warp
constexpr int SLOT_BYTES = CHUNK * 1024;

struct StreamParams {
  CUtensorMap tm_w;        // TILE words, box 128 words x 2 tiles x CHUNK k-atoms x 1 group
  const uint16_t* x;       // [M][K] (act-order layers: the gathered x[:, perm] when staged)
  const int32_t* perm;     // act-order without staged x: [K], gathered here; else nullptr
  const uint8_t* qw;       // TILE words (bytes)
  const uint16_t* scales;  // [G][N]
  const uint32_t* zeros;   // [G][N/8] standard order
  uint16_t* y;             // [M][N]
  const uint16_t* bias;    // [N] or nullptr
  int M, N, K;
  int A;                   // K / 64
  int T;                   // N / 16 tiles
  int G;                   // groups
  int gshift;              // group = 1 << gshift (5, 6, 7); 31: one group over all of K
  int nslab;               // ceil(T / 2)
  int* status;             // the library's device status word
};

struct StreamLayout {
  int ring_off, bar_off, s_off, z_off, p_off, total;
};

// Shared memory of a CTA owning `ns` slabs (offsets from a 1024-byte aligned
// base): the warps' rings, their mbarriers and the abort flag, scales [G][32 ns]
// (16-bit), zeros [G][4 ns] words, then two partial-slab slots per warp of 32
// columns x MR tokens (fp32). `total` includes the alignment slack.
__host__ __device__ inline StreamLayout stream_layout(int G, int ns, int MR) {
  StreamLayout L;
  L.ring_off = 0;
  L.bar_off = SW * RING * SLOT_BYTES;
  L.s_off = L.bar_off + ((SW * RING * 8 + 16 + 15) & ~15);
  L.z_off = L.s_off + ((G * 32 * ns * 2 + 15) & ~15);
  L.p_off = (L.z_off + G * 4 * ns * 4 + 15) & ~15;
  L.total = L.p_off + SW * 2 * 32 * MR * 4 + 1024;
  return L;
}

template <bool BF16>
__device__ __forceinline__ void mma_k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Byte offset of slab s (tiles 2s, 2s + 1) at k-atom 0: both tiles sit in
// column group s / 4 at tile positions (2s) % 8 and (2s) % 8 + 1.
__device__ __forceinline__ size_t slab_base(int s, int A) {
  return ((size_t)(s >> 2) * A * 8 + ((2 * s) & 7)) * 512;
}

// MT: token tiles of 8 (M <= 8 MT). GATHER: an act-order call whose x was not
// staged (the kernel reads x through perm).
#ifndef W4_STREAM_MINB
#define W4_STREAM_MINB 2
#endif
template <int MT, bool BF16, bool GATHER>
__global__ void __launch_bounds__(ST, W4_STREAM_MINB) w4a16_stream_kernel(const __grid_constant__ StreamParams p) {
  constexpr uint32_t MAGIC = Magic<BF16>::pair;  // 128 (bf16) / 1024 (fp16) in both halves
  constexpr int MR = 8 * MT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gg = lane >> 2, t = lane & 3;
  const int s0 = (int)((long long)blockIdx.x * p.nslab / gridDim.x);
  const int s1 = (int)((long long)(blockIdx.x + 1) * p.nslab / gridDim.x);
  const int ns = s1 - s0;
  const int A = p.A;
  const StreamLayout L = stream_layout(p.G, ns, MR);
  uint16_t* sS = reinterpret_cast<uint16_t*>(smem + L.s_off);
  uint32_t* sZ = reinterpret_cast<uint32_t*>(smem + L.z_off);
  float* sP = reinterpret_cast<float*>(smem + L.p_off);
  const uint32_t ring0 = smem_addr(smem + L.ring_off) + warp * RING * SLOT_BYTES;
  const uint32_t bar0 = smem_addr(smem + L.bar_off) + warp * RING * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.bar_off + SW * RING * 8);
  const int ncols = 32 * ns;
  const int col0 = 32 * s0;

  // this warp's items: [i0, i1) of the CTA's (slab, k-atom) sequence, slab-major
  const long long I = (long long)ns * A;
  const int i0 = (int)(warp * I / SW), i1 = (int)((warp + 1) * I / SW);

  // ---- before the dependency wait: barriers, the first copies, scales and zeros --
  if (tid == 0) *abort_flag = 0;
  if (lane == 0) {
    for (int r = 0; r < RING; ++r) mbar_init(bar0 + 8 * r, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Copy cursor: the warp's items cut into chunks of at most CHUNK k-atoms that
  // stay inside one slab; chunk c goes to slot c % RING. Both the copy side and
  // the consume side walk the same sequence.
  int cs_i = i0, cs_s = i0 / A, cs_a = i0 - (i0 / A) * A;  // next chunk to copy
  int issued = 0;                                          // chunks copied so far
  auto issue_chunk = [&]() {
    if (cs_i >= i1) return;
    const int n = min(CHUNK, min(A - cs_a, i1 - cs_i));
    if (lane == 0) {
      const int slot = issued % RING;
      const int s = s0 + cs_s;
      mbar_arrive_expect_tx(bar0 + 8 * slot, SLOT_BYTES);
      tma_load_4d(ring0 + slot * SLOT_BYTES, &p.tm_w, bar0 + 8 * slot, 0, (2 * s) & 7, cs_a, s >> 2);
    }
    ++issued;
    cs_i += n;
    cs_a += n;
    if (cs_a == A) {
      cs_a = 0;
      ++cs_s;
    }
  };
  for (int r = 0; r < RING; ++r) issue_chunk();
  // L2 prefetch cursor, up to L2_AHEAD items past the copies
  int fi = cs_i, fs = cs_s, fa = cs_a;
  auto prefetch_upto = [&](int limit) {
    // one bulk prefetch per item, up to item `limit` (lanes take consecutive items)
    while (fi < limit && fi < i1) {
      const int n = min(32, min(A - fa, min(limit, i1) - fi));
      if (lane < n) {
        const int s = s0 + fs;
        prefetch_l2(p.qw + slab_base(s, A) + (size_t)(fa + lane) * KROW_BYTES, 1024);
      }
      fi += n;
      fa += n;
      if (fa == A) {
        fa = 0;
        ++fs;
      }
    }
  };
  prefetch_upto(cs_i + L2_AHEAD);
  {
    // scales: per group row, 4 ns chunks of 8 columns; zeros: 2 ns chunks of 2 words
    const int sch = 4 * ns, zch = 2 * ns;
    for (int i = tid; i < p.G * sch; i += ST) {
      const int g = i / sch, c = i - g * sch;
      const int col = col0 + 8 * c;
      const uint32_t dst = smem_addr(sS + (size_t)g * ncols + 8 * c);
      if (col < p.N) cp_async16(dst, p.scales + (size_t)g * p.N + col);
      else *reinterpret_cast<uint4*>(sS + (size_t)g * ncols + 8 * c) = make_uint4(0, 0, 0, 0);
    }
    for (int i = tid; i < p.G * zch; i += ST) {
      const int g = i / zch, c = i - g * zch;
      const int col = col0 + 16 * c;
      const uint32_t dst = smem_addr(sZ + (size_t)g * (ncols / 8) + 2 * c);
      if (col < p.N) cp_async8(dst, p.zeros + (size_t)g * (p.N / 8) + col / 8);
      else *reinterpret_cast<uint2*>(sZ + (size_t)g * (ncols / 8) + 2 * c) = make_uint2(0, 0);
    }
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every CTA of this grid is resident: the next kernel may start its prologue
  asm volatile("griddepcontrol.launch_dependents;");
  cp_async_wait_all();
  __syncthreads();  // the scales and zeros are in shared memory
  // ---- the weight loop ------------------------------------------------------------
  float acc[2][MT][4], tc[2][MT][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[h][mt][j] = tc[h][mt][j] = 0.f;

  // x of this lane's token rows (gg, gg + 8) at k-atom a: two 16-byte pieces
  // (columns 8t..8t+7 of each 32-row half); rows at or beyond M read as zero.
  // An act-order call whose x was not staged gathers x[:, perm] here.
  auto load_x = [&](int a, uint4 (&xf)[MT][2]) {
    if constexpr (GATHER) {
      const int4* pp = reinterpret_cast<const int4*>(p.perm + a * ATOM_K + 8 * t);
      const int4 q[4] = {__ldg(pp), __ldg(pp + 1), __ldg(pp + 8), __ldg(pp + 9)};
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int row = gg + 8 * mt;
        if (row < p.M) {
          const uint16_t* xr = p.x + (size_t)row * p.K;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int4 u = q[2 * hh], v = q[2 * hh + 1];
            xf[mt][hh] = make_uint4(__ldg(xr + u.x) | ((uint32_t)__ldg(xr + u.y) << 16),
                                    __ldg(xr + u.z) | ((uint32_t)__ldg(xr + u.w) << 16),
                                    __ldg(xr + v.x) | ((uint32_t)__ldg(xr + v.y) << 16),
                                    __ldg(xr + v.z) | ((uint32_t)__ldg(xr + v.w) << 16));
          }
        } else {
          xf[mt][0] = xf[mt][1] = make_uint4(0, 0, 0, 0);
        }
      }
      return;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int row = gg + 8 * mt;
      if (row < p.M) {
        const uint16_t* xr = p.x + (size_t)row * p.K + a * ATOM_K + 8 * t;
        xf[mt][0] = ldg_x(xr);
        xf[mt][1] = ldg_x(xr + 32);
      } else {
        xf[mt][0] = xf[mt][1] = make_uint4(0, 0, 0, 0);
      }
    }
  };

  int cs = i0 / A, ca = i0 - (i0 / A) * A;  // consume cursor (slab, k-atom)
  int piece_start = ca;                      // first k-atom of the current slab piece
  bool first_piece = true;
  // the open group: its index (-1: none), scales and zero terms of this lane's
  // four columns (tile h, column gg + 8 j)
  int gopen = -1;
  uint32_t zp[2][2];  // MAGIC + z pairs of the open group (tile h, column gg + 8 j)

  auto meta_col = [&](int h, int j) { return 32 * cs + 16 * h + gg + 8 * j; };
  auto zero_of = [&](int gi, int col) {
    return (sZ[(size_t)gi * (ncols / 8) + (col >> 3)] >> (4 * (col & 7))) & 0xFu;
  };
  auto open_group = [&](int gi) {
    gopen = gi;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 2; ++j) zp[h][j] = MAGIC + zero_of(gi, meta_col(h, j)) * 0x00010001u;
  };
  // tc += s * acc; acc = 0. The group's scales are read from shared memory here.
  auto flush = [&]() {
    if (gopen < 0) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int col = meta_col(h, jj);
        const float sc = half_bits_to_float<BF16>(sS[(size_t)gopen * ncols + col]);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = 2 * jj + e;
            tc[h][mt][j] = fmaf(sc, acc[h][mt][j], tc[h][mt][j]);
            acc[h][mt][j] = 0.f;
          }
        }
      }
    }
    gopen = -1;
  };
  // one 32-row half of both tiles: words (lo, hi) of tile h come from w[h]
  auto half_atom = [&](const uint32_t w0lo, const uint32_t w0hi, const uint32_t w1lo,
                       const uint32_t w1hi, const uint4 (&xh)[MT]) {
    const uint32_t wv[2][2] = {{w0lo, w0hi}, {w1lo, w1hi}};
#pragma unroll
    for (int step = 0; step < 2; ++step) {
      uint32_t a[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t lo = wv[h][0], hi = wv[h][1];
        const int sh = 8 * step;
        const uint32_t lo_a = lo >> sh, hi_a = hi >> sh;
        const uint32_t lo_b = lo >> (sh + 4), hi_b = hi >> (sh + 4);
        a[h][0] = lop3_and_or(lo_a, 0x000F000Fu, MAGIC);
        a[h][2] = lop3_and_or(lo_b, 0x000F000Fu, MAGIC);
        a[h][1] = lop3_and_or(hi_a, 0x000F000Fu, MAGIC);
        a[h][3] = lop3_and_or(hi_b, 0x000F000Fu, MAGIC);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        a[h][0] = sub_x2<BF16>(a[h][0], zp[h][0]);
        a[h][2] = sub_x2<BF16>(a[h][2], zp[h][0]);
        a[h][1] = sub_x2<BF16>(a[h][1], zp[h][1]);
        a[h][3] = sub_x2<BF16>(a[h][3], zp[h][1]);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t b0 = step ? xh[mt].z : xh[mt].x;
        const uint32_t b1 = step ? xh[mt].w : xh[mt].y;
        mma_k16<BF16>(acc[0][mt], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
        mma_k16<BF16>(acc[1][mt], a[1][0], a[1][1], a[1][2], a[1][3], b0, b1);
      }
    }
  };
  // the slab piece ends: close the group; a piece that covers the slab's whole
  // K range is final and goes straight to y, a partial one to this warp's slot
  auto end_piece = [&](int a_end) {
    flush();
    const int sr = cs;
    const bool whole = piece_start == 0 && a_end == A;
    if (whole) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int m = 8 * mt + 2 * t + (j & 1);
            const int n = col0 + 32 * sr + 16 * h + gg + 8 * (j >> 1);
            if (m < p.M && n < p.N) {
              float v = tc[h][mt][j];
              if (p.bias != nullptr) v += half_bits_to_float<BF16>(p.bias[n]);
              p.y[(size_t)m * p.N + n] = float_to_half_bits<BF16>(v);
            }
          }
        }
      }
    } else {
      float* slot = sP + (size_t)(warp * 2 + (first_piece ? 0 : 1)) * 32 * MR;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            slot[(16 * h + gg + 8 * (j >> 1)) * MR + 8 * mt + 2 * t + (j & 1)] = tc[h][mt][j];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) tc[h][mt][j] = 0.f;
    first_piece = false;
  };

  // consume the chunks in order; each chunk's slot is refilled with the chunk
  // RING ahead as soon as every lane has read it
  int consumed = 0;
  bool live = true;
  while (live && consumed < issued) {
    const int slot = consumed % RING;
    if (!bounded_wait(bar0 + 8 * slot, (uint32_t)((consumed / RING) & 1), abort_flag, p.status)) {
      live = false;
      break;
    }
    const int n = min(CHUNK, min(A - ca, i1 - (cs * A + ca)));
    const uint32_t sbase = ring0 + slot * SLOT_BYTES + lane * 16;
    // Fast path: a whole chunk of groups of 64 or 128 rows that starts on a
    // group boundary: group starts at compile-time positions, x loaded per pair
    // of k-atoms, no per-atom bookkeeping. The chunk may end its slab piece.
    const int apg = p.gshift == 7 ? 2 : 1;  // k-atoms per group
    if (n == CHUNK && (p.gshift == 6 || p.gshift == 7) && (ca & (apg - 1)) == 0) {
#pragma unroll
      for (int q = 0; q < CHUNK / 2; ++q) {
        uint4 xc[2][MT][2];
        load_x(ca + 2 * q, xc[0]);
        load_x(ca + 2 * q + 1, xc[1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int u = 2 * q + e;
          if (e == 0 || apg == 1) open_group(((ca + u) * ATOM_K) >> p.gshift);
          const uint4 w0 = dec::lds128(sbase + u * 1024);
          const uint4 w1 = dec::lds128(sbase + u * 1024 + 512);
          uint4 xh[MT];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) xh[mt] = xc[e][mt][0];
          half_atom(w0.x, w0.y, w1.x, w1.y, xh);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) xh[mt] = xc[e][mt][1];
          half_atom(w0.z, w0.w, w1.z, w1.w, xh);
          if (e == 1 || apg == 1) flush();
        }
      }
      ca += CHUNK;
      if (ca == A || cs * A + ca == i1) {
        end_piece(ca);
        if (ca == A) {
          ca = 0;
          ++cs;
        }
        piece_start = ca;
      }
    } else
    for (int u = 0; u < n; ++u) {
      const uint4 w0 = dec::lds128(sbase + u * 1024);
      const uint4 w1 = dec::lds128(sbase + u * 1024 + 512);
      uint4 xc[MT][2];
      load_x(ca, xc);
      const int kr = ca * ATOM_K;
      if (p.gshift >= 31) {
        if (gopen < 0) open_group(0);
      } else if (p.gshift >= 6) {
        const int gi = kr >> p.gshift;
        if (gi != gopen) {
          flush();
          open_group(gi);
        }
      } else {
        // groups of 32 rows: each half of the atom is a group
        flush();
        open_group(kr >> 5);
      }
      {
        uint4 xh[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) xh[mt] = xc[mt][0];
        half_atom(w0.x, w0.y, w1.x, w1.y, xh);
      }
      if (p.gshift < 6) {
        flush();
        open_group((kr >> 5) + 1);
      }
      {
        uint4 xh[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) xh[mt] = xc[mt][1];
        half_atom(w0.z, w0.w, w1.z, w1.w, xh);
      }
      // a slab piece ends at the slab's last k-atom or at the end of the items
      ++ca;
      if (ca == A || cs * A + ca == i1) {
        end_piece(ca);
        if (ca == A) {
          ca = 0;
          ++cs;
        }
        piece_start = ca;
      }
    }
    ++consumed;
    __syncwarp();
    if (lane == 0) fence_proxy_async_smem();  // the reads of the slot precede its refill
    issue_chunk();
    prefetch_upto(cs_i + L2_AHEAD);
  }
  if (!live || *abort_flag) {
    // let this warp's copies in flight land before the CTA exits
    if (lane == 0)
      for (int c = consumed; c < issued; ++c) drain_wait(bar0 + 8 * (c % RING), (uint32_t)((c / RING) & 1));
    __syncwarp();
  }

  // ---- partial slabs: sum the warps' pieces in warp order ----------------------------
  __syncthreads();
  const int outs = ns * 32 * p.M;
  for (int o = tid; o < outs; o += ST) {
    const int sr = o / (32 * p.M);
    const int rem = o - sr * 32 * p.M;
    const int m = rem / 32, c = rem - m * 32;
    const int lo = sr * A, hi = lo + A;  // the slab's items
    float v = 0.f;
    bool partial = false;
    for (int w = 0; w < SW; ++w) {
      const int wa = (int)(w * I / SW), wb_ = (int)((w + 1) * I / SW);
      if (wa >= wb_ || wa >= hi || wb_ <= lo) continue;
      if (wa <= lo && wb_ >= hi) break;  // one warp covered the slab: stored already
      partial = true;
      const int slot = (wa >= lo) ? 0 : 1;  // this slab holds the warp's first piece?
      v += sP[((size_t)(w * 2 + slot) * 32 + c) * MR + m];
    }
    const int n = col0 + 32 * sr + c;
    if (partial && n < p.N) {
      if (p.bias != nullptr) v += half_bits_to_float<BF16>(p.bias[n]);
      p.y[(size_t)m * p.N + n] = float_to_half_bits<BF16>(v);
    }
  }
}

template <int MT, bool BF16, bool GATHER>
void* stream_kernel_ptr() {
  return reinterpret_cast<void*>(&w4a16_stream_kernel<MT, BF16, GATHER>);
}

void* pick_stream_kernel(bool bf16, bool gather) {
  if (bf16) return gather ? stream_kernel_ptr<1, true, true>() : stream_kernel_ptr<1, true, false>();
  return gather ? stream_kernel_ptr<1, false, true>() : stream_kernel_ptr<1, false, false>();
}

// The kernels' dynamic shared-memory limit, raised once per (kernel, device) to
// the most any launch asks for (kept out of the launch path).
constexpr int STREAM_SMEM_MAX =
    SW * RING * SLOT_BYTES + 1024 + META_BUDGET + 32 + SW * 2 * 32 * 16 * 4 + 1024;
cudaError_t ensure_stream_smem(int which, void* fn, int bytes, int limit) {
  static std::mutex mu;
  static int done[64][8] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || which < 0 || which >= 8) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][which] >= bytes) return cudaSuccess;
  const int want = std::min(STREAM_SMEM_MAX, limit);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
  if (e == cudaSuccess) done[dev][which] = want;
  return e;
}

int log2_of(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return (1 << s) == v ? s : -1;
}

}  // namespace

cudaError_t launch_decode_stream(const GemmArgs& a, cudaStream_t stream, bool* launched) {
  *launched = false;
  // At most 8 rows: at 9-16 rows the clustered kernel is faster on these layers
  // too (measured on GB300, Llama-2-7B o_proj at M = 16: 6.7 against 7.5 us;
  // at M = 1 / 4 this kernel: 5.2 / 5.5 against 5.9 / 6.3 us)
  if (a.eoff != nullptr || a.test_stall || a.M < 1 || a.M > 8) return cudaSuccess;
  DeviceInfo info;
  cudaError_t err = device_info(&info);
  if (err != cudaSuccess) return err;
  // Layers whose packed weights come to at most STREAM_MAX_BYTES_PER_SM per SM:
  // there the clustered kernel's fixed per-CTA costs (staging x and its group
  // sums, the cluster reduction) dominate its time, and this kernel, which has
  // none of them, is faster (measured on GB300: Llama-2-7B o_proj, 57 KB per
  // SM, 5.4 against 7.7 us at M = 1). On larger layers the
  // clustered kernel's loop, with three times the warps per SM, is faster
  // (7B down, 154 KB per SM: 13.9 against 11.0 us at M = 1).
  if ((double)a.K * a.N / 2 / info.sm_count > STREAM_MAX_BYTES_PER_SM) return cudaSuccess;
  const int T = a.N / 16;
  const int nslab = (T + 1) / 2;
  const int ctas = std::min(info.sm_count * W4_STREAM_CTAS_PER_SM, nslab);
  const int ns_max = (nslab + ctas - 1) / ctas;
  int gshift = log2_of(a.group);
  if (a.group == a.K || gshift < 0) gshift = 31;
  const int G = gshift >= 31 ? 1 : a.K >> gshift;
  const int MT = 1;
  const StreamLayout L = stream_layout(G, ns_max, 8 * MT);
  // scales and zeros beyond the budget: the clustered kernel takes the call
  if (L.p_off - L.s_off > META_BUDGET || L.total > info.max_smem_optin) return cudaSuccess;
  // act-order: x[:, perm] is gathered once per call into the workspace when it
  // has room (every CTA reads all of x), else by the kernel as it reads x
  const void* xsrc = a.x;
  const int32_t* perm = a.perm;
  if (perm && a.workspace && a.workspace_bytes >= decode_workspace_bytes(a.M, a.K, true)) {
    if ((err = launch_gather_columns(a.x, perm, a.workspace, a.M, a.K, stream)) != cudaSuccess)
      return err;
    xsrc = a.workspace;
    perm = nullptr;
  }
  void* fn = pick_stream_kernel(a.bf16 != 0, perm != nullptr);
  const int which = (MT - 1) + 2 * (a.bf16 ? 1 : 0) + 4 * (perm != nullptr ? 1 : 0);
  if ((err = ensure_stream_smem(which, fn, L.total, info.max_smem_optin)) != cudaSuccess) return err;
  int* status = nullptr;
  if ((err = device_status_ptr(&status)) != cudaSuccess) return err;
  StreamParams p;
  const uint64_t NG = ((uint64_t)a.N + 127) / 128;
  if (!encode_tile_box(&p.tm_w, a.qw, a.K, NG, 2, CHUNK, 1)) return cudaErrorInvalidValue;
  p.status = status;
  p.x = static_cast<const uint16_t*>(xsrc);
  p.perm = perm;
  p.qw = reinterpret_cast<const uint8_t*>(a.qw);
  p.scales = static_cast<const uint16_t*>(a.scales);
  p.zeros = a.zeros;
  p.y = static_cast<uint16_t*>(a.y);
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.A = a.K / ATOM_K;
  p.T = T;
  p.G = G;
  p.gshift = gshift;
  p.nslab = nslab;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(ST, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  if ((err = cudaLaunchKernelExC(&cfg, fn, args)) != cudaSuccess) return err;
  *launched = true;
  return cudaSuccess;
}

}  // namespace w4
