// One-time weight repack kernels and the dense dequantisation kernel.
//
// Pages: "量化层加载:AWQ / GPTQ / Marlin / fp8" (设计动机: AWQ → GPTQ format
// conversion and desc_act / g_idx; 关键文件: the kernel's own repack after
// loading) and "vLLM AWQ 4-bit 量化实践" (§5.1: reverse-order unpack and
// repack along the input dim; §5.3: (b - zeros) * scales).
//
// Block-transform kernels here work on a block of 64 rows x 128 columns: the
// block's codes are first expanded into shared memory (one byte per code) from
// whichever packed source it comes in, then written out in the target layout.
// All of this runs once per layer at load time.
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

#include <algorithm>

namespace w4 {
namespace {

constexpr int BK = 64;    // rows per block (one TILE atom row)
constexpr int BN = 128;   // columns per block (eight TILE atoms)
constexpr int BLOCK_THREADS = 256;

enum SourceKind { SRC_AWQ = 0, SRC_STD = 1, SRC_TILE = 2 };

// Expand codes of rows [k0, k0+64) x columns [n0, n0+ncols) into codes[64][128].
// SRC_STD may gather rows through perm (stored row k <- source row perm[k]).
__device__ void load_block_codes(int kind, const uint32_t* __restrict__ src,
                                 const int32_t* __restrict__ perm, int K, int N, int k0, int n0,
                                 int nrows, int ncols, uint8_t (*codes)[BN]) {
  const int tid = threadIdx.x;
  if (kind == SRC_AWQ) {
    // qweight [K][N/8]: 16 words per block row
    const int C = N / 8;
    for (int i = tid; i < BK * (BN / 8); i += BLOCK_THREADS) {
      const int kk = i / (BN / 8), cw = i % (BN / 8);
      if (cw * 8 >= ncols || kk >= nrows) continue;
      const uint32_t w = src[(size_t)(k0 + kk) * C + n0 / 8 + cw];
#pragma unroll
      for (int j = 0; j < 8; ++j) codes[kk][cw * 8 + j] = (w >> (4 * awq_nibble_pos(j))) & 0xF;
    }
  } else if (kind == SRC_STD) {
    // qweight [K/8][N]: row k at bits 4*(k%8) of word row k/8
    for (int i = tid; i < BK * BN; i += BLOCK_THREADS) {
      const int kk = i / BN, col = i % BN;
      if (col >= ncols || kk >= nrows) continue;
      const int ks = perm ? perm[k0 + kk] : (k0 + kk);
      const uint32_t w = src[(size_t)(ks >> 3) * N + n0 + col];
      codes[kk][col] = (w >> (4 * (ks & 7))) & 0xF;
    }
  } else {
    // TILE: the eight atoms of column group n0/128 at k-atom k0/64 are adjacent
    const int A = K / BK;
    const int kb = k0 / BK;
    const uint32_t* grp = src + ((size_t)(n0 / BN) * A + kb) * 8 * 128;
    for (int i = tid; i < 8 * 128; i += BLOCK_THREADS) {
      const int at = i >> 7, wl = i & 127;
      if (at * 16 >= ncols) continue;
      const int lane = wl >> 2, j = wl & 3;
      const int gg = lane >> 2, t = lane & 3;
      const int col = at * 16 + gg + 8 * (j & 1);
      const int kk0 = 32 * (j >> 1) + 8 * t;
      const uint32_t w = grp[at * 128 + wl];
#pragma unroll
      for (int e = 0; e < 8; ++e) codes[kk0 + e][col] = (w >> (4 * tile_nibble_pos(e))) & 0xF;
    }
  }
}

// Repack any source into the TILE layout. grid = (ceil(N/128), K/64): one block
// writes the eight adjacent atoms of its column group at its k-atom (the atoms
// of a partial last group beyond N are written as zeros).
__global__ void __launch_bounds__(BLOCK_THREADS) to_tile_kernel(
    const uint32_t* __restrict__ src, int kind, const int32_t* __restrict__ perm,
    uint32_t* __restrict__ out, int K, int N) {
  __shared__ uint8_t codes[BK][BN];
  const int n0 = blockIdx.x * BN, k0 = blockIdx.y * BK;
  const int ncols = min(BN, N - n0);
  load_block_codes(kind, src, perm, K, N, k0, n0, BK, ncols, codes);
  __syncthreads();
  const int A = K / BK;
  const int kb = blockIdx.y;
  uint32_t* grp = out + ((size_t)blockIdx.x * A + kb) * 8 * 128;
  for (int i = threadIdx.x; i < 8 * 128; i += BLOCK_THREADS) {
    const int at = i >> 7, wl = i & 127;
    if (at * 16 >= ncols) {
      grp[i] = 0u;
      continue;
    }
    const int lane = wl >> 2, j = wl & 3;
    const int gg = lane >> 2, t = lane & 3;
    const int col = at * 16 + gg + 8 * (j & 1);
    const int kk0 = 32 * (j >> 1) + 8 * t;
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) w |= (uint32_t)codes[kk0 + e][col] << (4 * tile_nibble_pos(e));
    grp[i] = w;
  }
}


// ---- vectorised repacks into the TILE layout (no act-order) ---------------------
// One block per (128-column group, KA 64-row k-atoms): the group's 1024 TILE words
// per k-atom are formed in registers and leave as 4 KB of 16-byte stores staged
// in shared memory. Requires N % 32 == 0 (whole 16-byte source pieces); a partial
// last group gets zero words.
// The permutation {0, 2, 4, 6, 1, 3, 5, 7}: nibble p of an AWQ word holds column
// sigma(p) of its block, and nibble p of a TILE word holds row sigma(p).
__host__ __device__ constexpr int sigma(int p) { return p < 4 ? 2 * p : 2 * (p - 4) + 1; }

// Word index, inside a column group's eight atoms at one k-atom, of the TILE
// word holding column cl (0..127 in the group) and rows 8 r .. 8 r + 7 (r 0..7).
__device__ __forceinline__ int tile_word_index(int cl, int r) {
  const int tt = cl >> 4, c16 = cl & 15;
  return tt * 128 + 4 * (4 * (c16 & 7) + (r & 3)) + 2 * (r >> 2) + (c16 >> 3);
}

// Staged TILE words: word i of an atom sits at i with its 16-byte chunk index
// (bits 2-4) XORed with its tile (bits 7-9), so that the scatter below, whose
// warp spans the eight tiles, meets two-way bank conflicts instead of eight-way;
// a 16-byte chunk stays whole.
__device__ __forceinline__ int staged_word(int i) { return i ^ (((i >> 7) & 7) << 2); }

// In-register transpose of an 8 x 8 nibble matrix (w[i] nibble p <-> w[p] nibble i).
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // 4 x 4 blocks
    const uint32_t t = ((w[i] >> 16) ^ w[i + 4]) & 0x0000FFFFu;
    w[i] ^= t << 16;
    w[i + 4] ^= t;
  }
#pragma unroll
  for (int i = 0; i < 8; i += (i & 1) ? 3 : 1) {  // 2 x 2 blocks: pairs (0,2) (1,3) (4,6) (5,7)
    const uint32_t t = ((w[i] >> 8) ^ w[i + 2]) & 0x00FF00FFu;
    w[i] ^= t << 8;
    w[i + 2] ^= t;
  }
#pragma unroll
  for (int i = 0; i < 8; i += 2) {  // single nibbles
    const uint32_t t = ((w[i] >> 4) ^ w[i + 1]) & 0x0F0F0F0Fu;
    w[i] ^= t << 4;
    w[i + 1] ^= t;
  }
}

// AWQ qweight [K][N/8] -> TILE. Word (k, c) of AWQ holds column 8c + sigma(p) at
// nibble p (the order {0,4,1,5,2,6,3,7} read backwards), and a TILE word holds
// row 8r + sigma(p) at nibble p: taking the eight rows in sigma order makes the
// repack a plain nibble transpose whose word q is column 8c + sigma(q).
// Thread t takes column word c = t % 16 of the group and the 8-row run r8 = t / 16
// (k-atom r8 / 8): eight 4-byte loads, coalesced across the warp (two rows of
// sixteen words), straight into registers.
template <int KA>
__global__ void __launch_bounds__(256) awq_to_tile_vec_kernel(const uint32_t* __restrict__ qweight,
                                                              uint32_t* __restrict__ out, int K,
                                                              int N) {
  __shared__ __align__(16) uint32_t out_s[KA][1024];
  const int cg = blockIdx.x, a0 = blockIdx.y * KA;
  const int C = N / 8, A = K / 64;
  const int ncw = min(16, C - cg * 16);  // column words of this group present (a multiple of 4)
  const int c = threadIdx.x & 15, r8 = threadIdx.x >> 4, u = r8 >> 3, r = r8 & 7;
  if (u < KA) {
    uint32_t w[8];
#pragma unroll
    for (int p = 0; p < 8; ++p)
      w[p] = c < ncw ? __ldg(qweight + (size_t)(64 * (a0 + u) + 8 * r + sigma(p)) * C + 16 * cg + c)
                     : 0u;
    transpose8x8_nibbles(w);
#pragma unroll
    for (int q = 0; q < 8; ++q) out_s[u][staged_word(tile_word_index(8 * c + sigma(q), r))] = w[q];
  }
  __syncthreads();
#pragma unroll
  for (int v = 0; v < KA; ++v) {
    uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)cg * A + a0 + v) * 8 * 128);
    dst[threadIdx.x] = *reinterpret_cast<const uint4*>(&out_s[v][staged_word(4 * threadIdx.x)]);
  }
}

// Standard qweight [K/8][N] (row 8r + e at nibble e) -> TILE (row 8r + e at
// nibble {0,4,1,5,2,6,3,7}[e]): a nibble shuffle per word, even rows to the low
// half and odd rows to the high half.
__global__ void __launch_bounds__(256) std_to_tile_vec_kernel(const uint32_t* __restrict__ src,
                                                              uint32_t* __restrict__ out, int K,
                                                              int N) {
  __shared__ __align__(16) uint32_t out_s[1024];
  const int cg = blockIdx.x, a = blockIdx.y;
  const int A = K / 64;
  const int ncols = min(128, N - cg * 128);
  // thread: row word r = t / 32 (0..7), columns 4 (t % 32) .. + 3
  const int r = threadIdx.x >> 5, c4 = (threadIdx.x & 31) * 4;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (c4 < ncols)
    v = *reinterpret_cast<const uint4*>(src + (size_t)(8 * a + r) * N + 128 * cg + c4);
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t ev = in[j] & 0x0F0F0F0Fu, od = (in[j] >> 4) & 0x0F0F0F0Fu;
    const uint32_t ev2 = ev | (ev >> 4), od2 = od | (od >> 4);
    uint32_t o;
    asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(o) : "r"(ev2), "r"(od2));
    out_s[staged_word(tile_word_index(c4 + j, r))] = o;
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)cg * A + a) * 8 * 128);
  dst[threadIdx.x] = *reinterpret_cast<const uint4*>(&out_s[staged_word(4 * threadIdx.x)]);
}

// AWQ qweight [K][N/8] -> standard [K/8][N]: an 8 x 8 nibble transpose per thread.
__global__ void __launch_bounds__(BLOCK_THREADS) awq_to_std_kernel(
    const uint32_t* __restrict__ qweight, uint32_t* __restrict__ out, int K, int N) {
  const int C = N / 8;
  const size_t total = (size_t)(K / 8) * C;
  const size_t idx = (size_t)blockIdx.x * BLOCK_THREADS + threadIdx.x;
  if (idx >= total) return;
  const int r = (int)(idx / C), c = (int)(idx % C);
  uint32_t in[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) in[i] = qweight[(size_t)(8 * r + i) * C + c];
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int sh = 4 * awq_nibble_pos(j);
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) v |= ((in[i] >> sh) & 0xFu) << (4 * i);
    o[j] = v;
  }
  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)r * N + 8 * c);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Standard [K/8][N] -> standard [K/8][N] with rows gathered through perm.
__global__ void __launch_bounds__(BLOCK_THREADS) std_rows_permuted_kernel(
    const uint32_t* __restrict__ src, const int32_t* __restrict__ perm,
    uint32_t* __restrict__ out, int K, int N) {
  const size_t total = (size_t)(K / 8) * N;
  const size_t idx = (size_t)blockIdx.x * BLOCK_THREADS + threadIdx.x;
  if (idx >= total) return;
  const int r = (int)(idx / N), n = (int)(idx % N);
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ks = perm ? perm[8 * r + i] : 8 * r + i;
    const uint32_t w = src[(size_t)(ks >> 3) * N + n];
    v |= ((w >> (4 * (ks & 7))) & 0xFu) << (4 * i);
  }
  out[idx] = v;
}

// Zeros to standard order (from AWQ order, or copied) and scales copied.
// Both arrays have G*N/8 units: one zeros word and one 16-byte scales chunk.
__global__ void __launch_bounds__(BLOCK_THREADS) meta_kernel(
    const uint32_t* __restrict__ qzeros, int zeros_are_awq, const uint4* __restrict__ scales,
    uint32_t* __restrict__ zeros_out, uint4* __restrict__ scales_out, size_t units) {
  for (size_t i = (size_t)blockIdx.x * BLOCK_THREADS + threadIdx.x; i < units;
       i += (size_t)gridDim.x * BLOCK_THREADS) {
    // symmetric weights (no zeros stored): the zero point is 8 everywhere
    const uint32_t w = qzeros != nullptr ? qzeros[i] : 0x88888888u;
    uint32_t v = w;
    if (zeros_are_awq && qzeros != nullptr) {
      v = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) v |= ((w >> (4 * awq_nibble_pos(j))) & 0xFu) << (4 * j);
    }
    zeros_out[i] = v;
    scales_out[i] = scales[i];
  }
}

// Stable sort of rows by group for act-order. One block of 1024 threads.
// Counting pass + validation, then one warp places rows in ascending k order
// (ranks among equal groups come from a warp-wide match), so ties keep
// ascending k. Irregular g_idx -> identity perm and W4_ERR_GIDX.
constexpr int PERM_THREADS = 1024;
constexpr int PERM_MAX_GROUPS = 8192;

__global__ void __launch_bounds__(PERM_THREADS) act_order_perm_kernel(
    const int32_t* __restrict__ g_idx, int K, int group, int32_t* __restrict__ perm,
    int32_t* __restrict__ status) {
  __shared__ int cnt[PERM_MAX_GROUPS];
  __shared__ int bad;
  const int G = K / group;
  const int tid = threadIdx.x;
  for (int g = tid; g < G; g += PERM_THREADS) cnt[g] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int k = tid; k < K; k += PERM_THREADS) {
    const int g = g_idx[k];
    if (g < 0 || g >= G) {
      bad = 1;
    } else {
      atomicAdd(&cnt[g], 1);
    }
  }
  __syncthreads();
  for (int g = tid; g < G; g += PERM_THREADS)
    if (cnt[g] != group) bad = 1;
  __syncthreads();
  if (bad) {
    for (int k = tid; k < K; k += PERM_THREADS) perm[k] = k;
    if (tid == 0) *status = W4_ERR_GIDX;
    return;
  }
  // Every group owns exactly `group` rows, so group g starts at g * group.
  for (int g = tid; g < G; g += PERM_THREADS) cnt[g] = g * group;
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < K; base += 32) {
      const int k = base + lane;
      const bool valid = k < K;
      const int g = valid ? g_idx[k] : -1;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, g);
      const int rank = __popc(peers & lt_mask);
      int pos = 0;
      if (valid) pos = cnt[g] + rank;
      __syncwarp();
      if (valid) {
        perm[pos] = k;
        if (rank == 0) cnt[g] += __popc(peers);
      }
      __syncwarp();
    }
    if (lane == 0) *status = W4_OK;
  }
}

// Dense W [K][N] from a repacked layer (TILE or STD rows), fp32 or half output.
// grid = (ceil(N/128), K/64).
template <bool BF16, bool OUT_F32>
__global__ void __launch_bounds__(BLOCK_THREADS) dequant_kernel(
    const uint32_t* __restrict__ qw, int kind, const uint16_t* __restrict__ scales,
    const uint32_t* __restrict__ zeros, void* __restrict__ w_out, int K, int N, int group) {
  __shared__ uint8_t codes[BK][BN];
  const int n0 = blockIdx.x * BN, k0 = blockIdx.y * BK;
  const int ncols = min(BN, N - n0);
  const int nrows = min(BK, K - k0);
  load_block_codes(kind, qw, nullptr, K, N, k0, n0, nrows, ncols, codes);
  __syncthreads();
  for (int i = threadIdx.x; i < BK * BN; i += BLOCK_THREADS) {
    const int kk = i / BN, col = i % BN;
    if (col >= ncols || kk >= nrows) continue;
    const int k = k0 + kk, n = n0 + col;
    const int g = k / group;
    const int q = codes[kk][col];
    const int z = (zeros[(size_t)g * (N / 8) + (n >> 3)] >> (4 * (n & 7))) & 0xF;
    const float s = half_bits_to_float<BF16>(scales[(size_t)g * N + n]);
    const float v = (float)(q - z) * s;  // exact: 4-bit integer times an 11-bit scale
    if constexpr (OUT_F32) {
      static_cast<float*>(w_out)[(size_t)k * N + n] = v;
    } else {
      static_cast<uint16_t*>(w_out)[(size_t)k * N + n] = float_to_half_bits<BF16>(v);
    }
  }
}

__global__ void stream_fence_kernel() {}

inline unsigned blocks_for(size_t n, int per = BLOCK_THREADS) {
  return (unsigned)((n + per - 1) / per);
}

}  // namespace

cudaError_t launch_stream_fence(cudaStream_t s) {
  stream_fence_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_awq_to_std(const int32_t* qweight, int32_t* qw_out, int K, int N,
                              cudaStream_t s) {
  const size_t total = (size_t)(K / 8) * (N / 8);
  awq_to_std_kernel<<<blocks_for(total), BLOCK_THREADS, 0, s>>>(
      reinterpret_cast<const uint32_t*>(qweight), reinterpret_cast<uint32_t*>(qw_out), K, N);
  return cudaGetLastError();
}

cudaError_t launch_to_tile(const int32_t* src, int src_is_awq, const int32_t* perm,
                           int32_t* qw_out, int K, int N, cudaStream_t s) {
  dim3 grid((N + BN - 1) / BN, K / BK);
  if (perm == nullptr && N % 32 == 0) {
    // whole 16-byte source pieces: the vectorised repacks
    if (src_is_awq && (K / BK) % 2 == 0)
      awq_to_tile_vec_kernel<2><<<dim3(grid.x, grid.y / 2), 256, 0, s>>>(
          reinterpret_cast<const uint32_t*>(src), reinterpret_cast<uint32_t*>(qw_out), K, N);
    else if (src_is_awq)
      awq_to_tile_vec_kernel<1><<<grid, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(src),
                                                     reinterpret_cast<uint32_t*>(qw_out), K, N);
    else
      std_to_tile_vec_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(src),
                                                  reinterpret_cast<uint32_t*>(qw_out), K, N);
    return cudaGetLastError();
  }
  to_tile_kernel<<<grid, BLOCK_THREADS, 0, s>>>(reinterpret_cast<const uint32_t*>(src),
                                                 src_is_awq ? SRC_AWQ : SRC_STD, perm,
                                                 reinterpret_cast<uint32_t*>(qw_out), K, N);
  return cudaGetLastError();
}

cudaError_t launch_std_rows_permuted(const int32_t* src, const int32_t* perm, int32_t* qw_out,
                                     int K, int N, cudaStream_t s) {
  const size_t total = (size_t)(K / 8) * N;
  std_rows_permuted_kernel<<<blocks_for(total), BLOCK_THREADS, 0, s>>>(
      reinterpret_cast<const uint32_t*>(src), perm, reinterpret_cast<uint32_t*>(qw_out), K, N);
  return cudaGetLastError();
}

cudaError_t launch_meta(const int32_t* qzeros, int zeros_are_awq, const void* scales,
                        int32_t* zeros_out, void* scales_out, int G, int N, cudaStream_t s) {
  const size_t units = (size_t)G * (N / 8);
  const unsigned grid = (unsigned)std::min<size_t>(blocks_for(units), 4096);
  meta_kernel<<<grid, BLOCK_THREADS, 0, s>>>(
      reinterpret_cast<const uint32_t*>(qzeros), zeros_are_awq,
      reinterpret_cast<const uint4*>(scales), reinterpret_cast<uint32_t*>(zeros_out),
      reinterpret_cast<uint4*>(scales_out), units);
  return cudaGetLastError();
}

cudaError_t launch_act_order_perm(const int32_t* g_idx, int K, int group, int32_t* perm_out,
                                  int32_t* status_out, cudaStream_t s) {
  if (K / group > PERM_MAX_GROUPS) return cudaErrorInvalidValue;
  act_order_perm_kernel<<<1, PERM_THREADS, 0, s>>>(g_idx, K, group, perm_out, status_out);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const int32_t* qw, const void* scales, const int32_t* zeros, int K,
                           int N, int group, int bf16, int layout, int out_f32, void* w_out,
                           cudaStream_t s) {
  const int kind = layout == W4_LAYOUT_TILE ? SRC_TILE : SRC_STD;
  dim3 grid((N + BN - 1) / BN, (K + BK - 1) / BK);
  const uint32_t* q = reinterpret_cast<const uint32_t*>(qw);
  const uint16_t* sc = static_cast<const uint16_t*>(scales);
  const uint32_t* z = reinterpret_cast<const uint32_t*>(zeros);
  if (bf16) {
    if (out_f32)
      dequant_kernel<true, true><<<grid, BLOCK_THREADS, 0, s>>>(q, kind, sc, z, w_out, K, N, group);
    else
      dequant_kernel<true, false><<<grid, BLOCK_THREADS, 0, s>>>(q, kind, sc, z, w_out, K, N, group);
  } else {
    if (out_f32)
      dequant_kernel<false, true><<<grid, BLOCK_THREADS, 0, s>>>(q, kind, sc, z, w_out, K, N, group);
    else
      dequant_kernel<false, false><<<grid, BLOCK_THREADS, 0, s>>>(q, kind, sc, z, w_out, K, N, group);
  }
  return cudaGetLastError();
}

}  // namespace w4
