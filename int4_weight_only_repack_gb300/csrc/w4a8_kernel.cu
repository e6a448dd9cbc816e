// INT4 weights x FP8 activations on the 5th-generation tensor cores
// (tcgen05.mma kind::f8f6f4): y[M][N] = s_x * x8[M][K] · W, W = (q - z) * s.
//
// Pages: "量化层加载:AWQ / GPTQ / Marlin / fp8" (边界与失败: with float8_e4m3fn
// activations the 4-bit weights are preprocessed and the scales multiplied by
// 512; 职责: Fp8Config's per-tensor dynamic activation scheme) and the SGLang
// W4AFp8 article (§五: INT4 weights against FP8 activations in one GEMM).
//
//  * Activations, two small kernels: the per-tensor max|x| (one partial per
//    CTA, no initialised memory needed), then every CTA reduces the partials,
//    takes s_x = RN(max|x| / 448) and writes x8 = e4m3(RN(x / s_x)) (round to
//    nearest even, saturating) and, for every row and group of 128 columns,
//    the group's sum of the codes as seven e4m3 digits (below).
//  * Weights: a 4-bit code q becomes the e4m3 byte q itself, the number
//    q * 2^-9 (0..7 subnormal, 8..15 the first binade: exact), so the B
//    operand costs one mask, one shift, one mask and two byte permutes per
//    eight codes. The "scales x 512" of the page: 512 s restores the factor,
//    and the zero point is applied to the group's sum:
//        sum_k x8 (q - z) s = (512 s) * (sum_k x8 (q 2^-9) - z 2^-9 xs),
//    xs = sum_k x8. The second term is one more K = 32 MMA per group on the
//    tensor cores, exact: xs is a multiple of 2^-9 below 2^16, so
//    I = 512 xs is an integer below 2^25 with seven base-16 digits u_j, and
//    z 2^-9 xs = sum_j (sign(I) u_j 2^a_j) (z 2^b_j) with a_j + b_j = 4j - 18;
//    both factors are e4m3 numbers for the exponents chosen (F8_DIGIT_A / _B),
//    and the MMA adds its 32 exact products with one rounding. The digits of
//    four groups share one 128-byte swizzled row (32 bytes a group), loaded by
//    TMA once per four K blocks; the weights' side is written per block.
//  * Persistent kernel, one CTA per SM, 128 x 128 output tiles, K blocks of
//    128 = one group (group 128; group -1 applies the same per-column scale at
//    every block). Warp 0 issues TMA copies (x8 rows with the 128-byte
//    swizzle, the packed TILE atoms, one group row of scales and zeros) into a
//    STAGES-deep ring, and every fourth block the digit rows into a ring of
//    two; warps 12-15 expand the atoms into the K-major swizzled e4m3 B tile,
//    write the block's -z 2^b_j digits and stage its 512 s per column; warp 1
//    issues five UMMAs per block (M 128, N 128, K 32: four for the weights,
//    one for the zero point) into one of two TMEM accumulators; warps 4-11
//    take each block's accumulator out of TMEM and fold it into fp32 running
//    sums held in registers (one FFMA per output and block), then scale by
//    s_x, round once and store y.
//  * Every mbarrier wait is bounded (one second); a timed-out wait records
//    W4_ERR_TIMEOUT in the device status word and the CTA drains its copies
//    and MMAs before it frees its tensor memory and exits.
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
using dec::drain_wait;

constexpr int BM = 128, BN = 128, BK = 128;  // BK bytes of e4m3 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int DIGITS = 7;       // base-16 digits of 512 * (a group's sum of the codes)
constexpr int DG = 4;           // groups whose digits share one 128-byte row (32 bytes each)
constexpr int THREADS = 512;
constexpr int EPI_WARPS = 8, DEQ_WARPS = 4;
constexpr int A_BYTES = BM * BK;           // x8 tile
constexpr int B_BYTES = BN * BK;           // expanded weights
constexpr int P_BYTES = BN * BK / 2;       // packed atoms: 8 tiles x 2 k-atoms
constexpr int S_BYTES = BN * 2;            // one group row of scales
constexpr int Z_BYTES = BN / 2;            // one group row of zeros (16 words)
constexpr int AB_BYTES = BN * 4;           // 512 s per column (fp32)
constexpr int X_BYTES = BM * 128;          // digit rows of DG groups (activations)
constexpr int W_BYTES = BN * 128;          // -z 2^b_j rows (weights): a ring of 4 K slices
// Block `it` (counted over the CTA's whole run) writes the weights' digits into
// slice it % 4; block it + 4 reuses it, and its weights are only expanded once
// the TMA stage it + 4 - STAGES = it is free again, i.e. once block it's MMAs
// have completed.
static_assert(STAGES == 4, "the weights' digit slices are recycled through the stage ring");
constexpr uint32_t STAGE_TX = A_BYTES + P_BYTES + S_BYTES + Z_BYTES;
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_P = OFF_B + STAGES * B_BYTES;
constexpr int OFF_S = OFF_P + STAGES * P_BYTES;
constexpr int OFF_Z = OFF_S + STAGES * S_BYTES;
constexpr int OFF_AB = OFF_Z + STAGES * 128;  // zero rows at 128-byte slots
constexpr int OFF_XD = (OFF_AB + STAGES * AB_BYTES + 1023) & ~1023;  // swizzled tiles: 1024-aligned
constexpr int OFF_WD = OFF_XD + 2 * X_BYTES;
constexpr int OFF_BAR = OFF_WD + W_BYTES;
constexpr int NUM_BARS = 3 * STAGES + 4 + 4;
constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
constexpr int TMEM_COLS = 256;                    // two 128-column fp32 accumulators
constexpr int AMAX_PARTS = 1024;                  // partial maxima of the first pass

// Digit j of the zero-point term: the activations' factor sign(I) u_j 2^a_j and
// the weights' factor -z 2^b_j, a_j + b_j = 4j - 18, both exact in e4m3 for
// u_j, z in 0..15 (exponents within -9..4).
__host__ __device__ constexpr int f8_digit_a(int j) { return j < 4 ? 4 * j - 9 : 4; }
__host__ __device__ constexpr int f8_digit_b(int j) { return 4 * j - 18 - f8_digit_a(j); }

struct W4a8Params {
  CUtensorMap tm_a;  // x8 [M][K] bytes, box 128 x 128, 128-byte swizzle
  CUtensorMap tm_d;  // digit rows [M][ceil(K/128/DG) * 128] bytes, box 128 x 128, 128-byte swizzle
  CUtensorMap tm_p;  // TILE words [N/128][K/64][8][128], box 128 x 8 x 2 x 1
  CUtensorMap tm_s;  // scales [G][N] 16-bit, box 128 x 1
  CUtensorMap tm_z;  // zeros [G][N/8] words, box 16 x 1
  uint16_t* y;
  const float* sx;     // the per-tensor activation scale
  int* status;
  int M, N, K, group;
  int m_blocks, n_blocks, num_tiles, k_blocks;
};

// Workspace: x8 [M][K] bytes, the digit rows [M][dpitch] bytes (32 per group),
// the partial maxima, s_x.
struct W4a8Ws {
  size_t x8, xd, parts, sx, total, dpitch;
};
W4a8Ws w4a8_ws(int M, int K) {
  W4a8Ws w;
  w.dpitch = (size_t)((K / BK + DG - 1) / DG) * 128;
  w.x8 = 0;
  w.xd = ((size_t)M * K + 255) & ~(size_t)255;
  w.parts = (w.xd + (size_t)M * w.dpitch + 255) & ~(size_t)255;
  w.sx = w.parts + AMAX_PARTS * 4;
  w.total = w.sx + 256;
  return w;
}

// ---- activations --------------------------------------------------------------
// Partial max|x| of this CTA's slice (eight values per 16-byte load).
// Two fp32 lanes in one 64-bit register, and a * b + c on both lanes with one
// rounding each (fma.rn.f32x2: one instruction for two of the epilogue's FMAs).
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

template <bool BF16>
__global__ void __launch_bounds__(256) w4a8_amax_kernel(const uint4* __restrict__ x, size_t n8,
                                                        float* __restrict__ parts) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  float m = 0.f;
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n8; i += (size_t)gridDim.x * 256) {
    const uint4 v = __ldg(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = fmaxf(m, fabsf(half_bits_to_float<BF16>((uint16_t)(w[j] & 0xFFFF))));
      m = fmaxf(m, fabsf(half_bits_to_float<BF16>((uint16_t)(w[j] >> 16))));
    }
  }
  __shared__ float red[8];
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
    parts[blockIdx.x] = r;
  }
}

// 2^e for e in [-126, 127] (exact)
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return make_float2(__half2float(__ushort_as_half((uint16_t)(h & 0xFFFF))),
                     __half2float(__ushort_as_half((uint16_t)(h >> 16))));
}

// s_x from the partial maxima, then x8 and, per (row, 128-column block), the
// digits of I = 512 * (the block's sum of the codes): one warp per block, four
// values per lane. I is summed exactly in integers (every code times 512 is an
// integer of at most 229376 in magnitude; 128 of them stay below 2^25).
template <bool BF16>
__global__ void __launch_bounds__(256) w4a8_quant_kernel(const uint16_t* __restrict__ x,
                                                         const float* __restrict__ parts,
                                                         int nparts, int M, int K,
                                                         uint8_t* __restrict__ x8,
                                                         uint8_t* __restrict__ xd,
                                                         size_t dpitch,
                                                         float* __restrict__ sx_out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float red[8];
  __shared__ float s_sh;
  float m = 0.f;
  for (int i = threadIdx.x; i < nparts; i += 256) m = fmaxf(m, parts[i]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
    const float s = r > 0.f ? __fdiv_rn(r, 448.f) : 1.f;
    s_sh = s;
    if (blockIdx.x == 0) *sx_out = s;
  }
  __syncthreads();
  const float s = s_sh;
  const int lane = threadIdx.x & 31;
  const int KB = K / BK;
  const long long units = (long long)M * KB;
  for (long long u = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); u < units;
       u += (long long)gridDim.x * 8) {
    const int row = (int)(u / KB), kb = (int)(u - (long long)row * KB);
    const size_t off = (size_t)row * K + (size_t)kb * BK + 4 * lane;
    const uint2 v = *reinterpret_cast<const uint2*>(x + off);
    float f[4] = {half_bits_to_float<BF16>((uint16_t)(v.x & 0xFFFF)),
                  half_bits_to_float<BF16>((uint16_t)(v.x >> 16)),
                  half_bits_to_float<BF16>((uint16_t)(v.y & 0xFFFF)),
                  half_bits_to_float<BF16>((uint16_t)(v.y >> 16))};
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __fdiv_rn(f[j], s);
    const uint16_t c01 = e4m3x2(f[0], f[1]), c23 = e4m3x2(f[2], f[3]);
    *reinterpret_cast<uint32_t*>(x8 + off) = (uint32_t)c01 | ((uint32_t)c23 << 16);
    const float2 d01 = e4m3x2_to_float2(c01), d23 = e4m3x2_to_float2(c23);
    int isum = __float2int_rn(d01.x * 512.f) + __float2int_rn(d01.y * 512.f) +
               __float2int_rn(d23.x * 512.f) + __float2int_rn(d23.y * 512.f);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) isum += __shfl_xor_sync(0xffffffffu, isum, d);
    // lanes 0..1 write the block's 32 digit bytes: sign(I) u_j 2^a_j for j < 7, then zeros
    if (lane < 2) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (lane == 0) {
        const uint32_t u = (uint32_t)(isum < 0 ? -isum : isum);
        const float sg = isum < 0 ? -1.f : 1.f;
        float dv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dv[j] = j < DIGITS ? sg * (float)((u >> (4 * j)) & 0xFu) * pow2f(f8_digit_a(j)) : 0.f;
        w[0] = (uint32_t)e4m3x2(dv[0], dv[1]) | ((uint32_t)e4m3x2(dv[2], dv[3]) << 16);
        w[1] = (uint32_t)e4m3x2(dv[4], dv[5]) | ((uint32_t)e4m3x2(dv[6], dv[7]) << 16);
      }
      *reinterpret_cast<uint4*>(xd + (size_t)row * dpitch + 32 * (size_t)kb + 16 * lane) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ---- the GEMM -----------------------------------------------------------------------
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t bfull(int s) const { return base + 8 * (STAGES + s); }
  __device__ uint32_t empty(int s) const { return base + 8 * (2 * STAGES + s); }
  __device__ uint32_t accfull(int b) const { return base + 8 * (3 * STAGES + b); }
  __device__ uint32_t accempty(int b) const { return base + 8 * (3 * STAGES + 2 + b); }
  // the activations' digit rows: TMA landed / the MMAs reading them completed
  __device__ uint32_t dfull(int d) const { return base + 8 * (3 * STAGES + 4 + d); }
  __device__ uint32_t dempty(int d) const { return base + 8 * (3 * STAGES + 6 + d); }
};

__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

template <bool BF16>
__global__ void __launch_bounds__(THREADS, 1) w4a8_gemm_kernel(const __grid_constant__ W4a8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Bars bars{sbase + OFF_BAR};
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.bfull(s), DEQ_WARPS * 32);
      mbar_init(bars.empty(s), 1 + EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.accfull(b), 1);
      mbar_init(bars.accempty(b), EPI_WARPS);
      mbar_init(bars.dfull(b), 1);
      mbar_init(bars.dempty(b), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_a);
    prefetch_tmap(&p.tm_d);
    prefetch_tmap(&p.tm_p);
    prefetch_tmap(&p.tm_s);
    prefetch_tmap(&p.tm_z);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int KB = p.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0, dg = 0;  // blocks, and groups of DG blocks (digit rows), so far
      int last_armed[STAGES], last_dg[2] = {-1, -1};
      for (int s = 0; s < STAGES; ++s) last_armed[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int m_blk = tile % p.m_blocks, n_blk = tile / p.m_blocks;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (kb % DG == 0) {  // the digit rows of blocks kb .. kb + DG - 1
            const int d = dg & 1;
            if (!bounded_wait(bars.dempty(d), ((dg >> 1) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bars.dfull(d), X_BYTES);
            last_dg[d] = dg;
            tma_load_2d(sbase + OFF_XD + d * X_BYTES, &p.tm_d, bars.dfull(d), (kb / DG) * 128,
                        m_blk * BM);
            ++dg;
          }
          if (!bounded_wait(bars.empty(s), ((it / STAGES) & 1) ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.full(s), STAGE_TX);
          last_armed[s] = it;
          const int grow = (kb * BK) / p.group;
          tma_load_2d(sbase + OFF_A + s * A_BYTES, &p.tm_a, bars.full(s), kb * BK, m_blk * BM);
          tma_load_4d(sbase + OFF_P + s * P_BYTES, &p.tm_p, bars.full(s), 0, 0, 2 * kb, n_blk);
          tma_load_2d(sbase + OFF_S + s * S_BYTES, &p.tm_s, bars.full(s), n_blk * BN, grow);
          tma_load_2d(sbase + OFF_Z + s * 128, &p.tm_z, bars.full(s), n_blk * (BN / 8), grow);
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (last_armed[s] >= 0) drain_wait(bars.full(s), (last_armed[s] / STAGES) & 1);
        for (int d = 0; d < 2; ++d)
          if (last_dg[d] >= 0) drain_wait(bars.dfull(d), (last_dg[d] >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_f16(0, BM, BN);  // kind::f8f6f4: A, B e4m3 (0), D f32
      int it = 0, dg = -1;
      bool ok = true, issued = false;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES, buf = it & 1;
          const uint32_t ph = (it / STAGES) & 1;
          if (kb % DG == 0) ++dg;
          const int d = dg & 1;
          if (!bounded_wait(bars.accempty(buf), ((it >> 1) & 1) ^ 1, abort_flag, p.status) ||
              !bounded_wait(bars.full(s), ph, abort_flag, p.status) ||
              !bounded_wait(bars.bfull(s), ph, abort_flag, p.status) ||
              (kb % DG == 0 && !bounded_wait(bars.dfull(d), (dg >> 1) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_k128(sbase + OFF_A + s * A_BYTES);
          const uint64_t bdesc = smem_desc_k128(sbase + OFF_B + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            umma_f8(tmem + buf * BN, adesc + 2 * k, bdesc + 2 * k, IDESC, k != 0);
          // the zero point: the block's 32-byte slice of the activations' digit rows
          // against the weights' (-z 2^b_j rows), into the same accumulator
          const uint64_t xdesc = smem_desc_k128(sbase + OFF_XD + d * X_BYTES);
          const uint64_t wdesc = smem_desc_k128(sbase + OFF_WD);
          umma_f8(tmem + buf * BN, xdesc + 2 * (kb % DG), wdesc + 2 * (it % 4), IDESC, 1);
          issued = true;
          umma_commit(bars.empty(s));
          umma_commit(bars.accfull(buf));
          if (kb % DG == DG - 1 || kb == KB - 1) umma_commit(bars.dempty(d));
        }
      }
      if (!ok && issued) {
        umma_commit(bars.accfull(0));
        drain_wait(bars.accfull(0), 0);
      }
    }
  } else if (warp >= 4 && warp < 4 + EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;      // TMEM lanes 32 quarter .. + 31 (rows)
    const int half = (warp - 4) >> 2;  // columns 64 half .. + 63
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const int m_blk = tile % p.m_blocks, n_blk = tile / p.m_blocks;
      const int row = m_blk * BM + quarter * 32 + lane;
      uint64_t y2[32];  // the 64 columns' running sums, two per register
#pragma unroll
      for (int c = 0; c < 32; ++c) y2[c] = 0;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES, buf = it & 1;
        if (!bounded_wait(bars.accfull(buf), (it >> 1) & 1, abort_flag, p.status) ||
            !bounded_wait(bars.bfull(s), (it / STAGES) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* ab = reinterpret_cast<const float*>(smem + OFF_AB + s * AB_BYTES);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + buf * BN + 64 * half + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a4 = *reinterpret_cast<const float4*>(ab + 64 * half + c0 + 4 * q);
            // y = fma(512 s, acc, y), two columns per instruction (the same
            // rounding per column as a scalar FMA); acc already holds the zero point
            const int c = (c0 + 4 * q) / 2;
            y2[c] = f32x2_fma(f32x2_pack(a4.x, a4.y),
                              f32x2_pack(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1])),
                              y2[c]);
            y2[c + 1] = f32x2_fma(
                f32x2_pack(a4.z, a4.w),
                f32x2_pack(__uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])), y2[c + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bars.accempty(buf));
          mbar_arrive(bars.empty(s));
        }
      }
      if (!ok) break;
      // y = RN(s_x * sum), stored as 16-byte pieces of eight columns
      const float sx = __ldg(p.sx);
      if (row < p.M) {
        uint16_t* yrow = p.y + (size_t)row * p.N;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int n = n_blk * BN + 64 * half + 8 * q;
          if (n < p.N) {
            uint4 v;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = (uint32_t)float_to_half_bits<BF16>(sx * f32x2_lo(y2[4 * q + e])) |
                     ((uint32_t)float_to_half_bits<BF16>(sx * f32x2_hi(y2[4 * q + e])) << 16);
            v.x = w[0];
            v.y = w[1];
            v.z = w[2];
            v.w = w[3];
            *reinterpret_cast<uint4*>(yrow + n) = v;
          }
        }
      }
    }
  } else if (warp >= 16 - DEQ_WARPS) {
    // ------------------------------------------------------------ expand the weights
    const int wd = warp - (16 - DEQ_WARPS);  // 0..3
    const int dt = wd * 32 + lane;           // this thread's column for the scale terms
    const int gg = lane >> 2, t = lane & 3;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % STAGES;
        if (!bounded_wait(bars.full(s), (it / STAGES) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* sP = smem + OFF_P + s * P_BYTES;
        uint8_t* sB = smem + OFF_B + s * B_BYTES;
        // atoms (k-atom ka, tile tt) of this warp: ka = wd / 2, tt = 4 (wd & 1) .. + 3
        const int ka = wd >> 1;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int tt = 4 * (wd & 1) + r;
          const uint4 w = *reinterpret_cast<const uint4*>(sP + (ka * 8 + tt) * 512 + lane * 16);
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t lo4 = wv[j] & 0x0F0F0F0Fu, hi4 = (wv[j] >> 4) & 0x0F0F0F0Fu;
            // K order: rows 0..3 and 4..7 of the word's eight (row e at nibble {0,4,1,5,2,6,3,7}[e])
            const uint32_t b0 = prmt(lo4, hi4, 0x6420u), b1 = prmt(lo4, hi4, 0x7531u);
            const int n_loc = 16 * tt + gg + 8 * (j & 1);
            const int koff = 64 * ka + 32 * (j >> 1) + 8 * t;
            const int chunk = (koff >> 4) ^ (n_loc & 7);
            const int off = (n_loc >> 3) * 1024 + (n_loc & 7) * 128 + chunk * 16 + (koff & 8);
            *reinterpret_cast<uint2*>(sB + off) = make_uint2(b0, b1);
          }
        }
        {
          // this column's 512 s for the epilogue, and its digit row for this block:
          // -z 2^b_j for j < 7, then zeros (32 bytes at K slice it % 4 of the
          // swizzled rows: two 16-byte chunks)
          const uint16_t* sS = reinterpret_cast<const uint16_t*>(smem + OFF_S + s * S_BYTES);
          const uint32_t* sZ = reinterpret_cast<const uint32_t*>(smem + OFF_Z + s * 128);
          const float sc = half_bits_to_float<BF16>(sS[dt]);
          const float nz = -(float)((sZ[dt >> 3] >> (4 * (dt & 7))) & 0xFu);
          float* ab = reinterpret_cast<float*>(smem + OFF_AB + s * AB_BYTES);
          ab[dt] = 512.f * sc;
          float dv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) dv[j] = j < DIGITS ? nz * pow2f(f8_digit_b(j)) : 0.f;
          const uint4 lo = make_uint4(
              (uint32_t)e4m3x2(dv[0], dv[1]) | ((uint32_t)e4m3x2(dv[2], dv[3]) << 16),
              (uint32_t)e4m3x2(dv[4], dv[5]) | ((uint32_t)e4m3x2(dv[6], dv[7]) << 16), 0u, 0u);
          uint8_t* sW = smem + OFF_WD + (dt >> 3) * 1024 + (dt & 7) * 128;
          const int c0 = (2 * (it % 4)) ^ (dt & 7), c1 = (2 * (it % 4) + 1) ^ (dt & 7);
          *reinterpret_cast<uint4*>(sW + c0 * 16) = lo;
          *reinterpret_cast<uint4*>(sW + c1 * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(bars.bfull(s));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

bool encode_2d_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t ensure_w4a8_smem(void* fn, int which) {
  static std::mutex mu;
  static bool done[64][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][which]) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e == cudaSuccess) done[dev][which] = true;
  return e;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

size_t w4a8_workspace_bytes(int M, int K) { return M > 0 ? w4a8_ws(M, K).total : 0; }

cudaError_t launch_w4a8(const void* x, const uint32_t* qw, const void* scales,
                        const uint32_t* zeros, void* y, int M, int N, int K, int group, int bf16,
                        void* workspace, cudaStream_t stream) {
  DeviceInfo info;
  cudaError_t err = device_info(&info);
  if (err != cudaSuccess) return err;
  int* status = nullptr;
  if ((err = device_status_ptr(&status)) != cudaSuccess) return err;
  const W4a8Ws w = w4a8_ws(M, K);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* x8 = ws + w.x8;
  uint8_t* xd = ws + w.xd;
  size_t dpitch = w.dpitch;
  float* parts = reinterpret_cast<float*>(ws + w.parts);
  float* sx = reinterpret_cast<float*>(ws + w.sx);

  // 1) partial maxima, 2) s_x, x8 and the block sums
  const size_t n8 = (size_t)M * K / 8;
  const int g1 = (int)std::min<size_t>(AMAX_PARTS, std::max<size_t>(1, (n8 + 255) / 256));
  {
    const uint4* xv = static_cast<const uint4*>(x);
    void* args[] = {&xv, const_cast<size_t*>(&n8), &parts};
    const void* fn = bf16 ? reinterpret_cast<const void*>(&w4a8_amax_kernel<true>)
                          : reinterpret_cast<const void*>(&w4a8_amax_kernel<false>);
    if ((err = launch_pdl(fn, dim3(g1), dim3(256), 0, stream, args)) != cudaSuccess) return err;
  }
  {
    const uint16_t* xh = static_cast<const uint16_t*>(x);
    int np = g1, Mi = M, Ki = K;
    const long long units = (long long)M * (K / BK);
    const int g2 = (int)std::min<long long>((long long)info.sm_count * 8, (units + 7) / 8);
    void* args[] = {&xh, &parts, &np, &Mi, &Ki, &x8, &xd, &dpitch, &sx};
    const void* fn = bf16 ? reinterpret_cast<const void*>(&w4a8_quant_kernel<true>)
                          : reinterpret_cast<const void*>(&w4a8_quant_kernel<false>);
    if ((err = launch_pdl(fn, dim3(std::max(1, g2)), dim3(256), 0, stream, args)) != cudaSuccess)
      return err;
  }
  // 3) the GEMM
  W4a8Params p;
  const int G = K / group;
  const uint64_t NG = ((uint64_t)N + 127) / 128;
  bool ok = encode_2d_map(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, x8, K, M, (uint64_t)K, BK, BM,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_2d_map(&p.tm_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, xd, dpitch, M, dpitch, 128, BM,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tile_box(&p.tm_p, qw, K, NG, 8, 2, 1);
  ok = ok && encode_2d_map(&p.tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, N, G, (uint64_t)N * 2,
                           BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && encode_2d_map(&p.tm_z, CU_TENSOR_MAP_DATA_TYPE_UINT32, zeros, N / 8, G,
                           (uint64_t)N / 2, BN / 8, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  p.y = static_cast<uint16_t*>(y);
  p.sx = sx;
  p.status = status;
  p.M = M;
  p.N = N;
  p.K = K;
  p.group = group;
  p.m_blocks = (M + BM - 1) / BM;
  p.n_blocks = (N + BN - 1) / BN;
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.k_blocks = K / BK;
  void* fn = bf16 ? reinterpret_cast<void*>(&w4a8_gemm_kernel<true>)
                  : reinterpret_cast<void*>(&w4a8_gemm_kernel<false>);
  if ((err = ensure_w4a8_smem(fn, bf16 ? 1 : 0)) != cudaSuccess) return err;
  void* args[] = {&p};
  return launch_pdl(fn, dim3((unsigned)std::min(p.num_tiles, info.sm_count)), dim3(THREADS),
                    SMEM_BYTES, stream, args);
}

}  // namespace w4
