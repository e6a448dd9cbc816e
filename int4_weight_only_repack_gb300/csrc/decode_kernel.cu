// Small-M (decode) W4A16 GEMM: y[M][N] = x[M][K] · W, M <= 64 per launch.
//
// Decode is bound by streaming the packed weights from HBM ("vLLM 学习手册 01.
// 量化" §1: decode has FLOPs/Bytes ~ 1 and moving the weights dominates), so
// the kernel is organised around the weight stream:
//
//  * Each warp owns one 16-column tile and a contiguous run of 64-row TILE
//    atoms (512 bytes each, contiguous in memory). Lane 0 streams the run into
//    a private shared-memory ring with bulk asynchronous copies
//    (cp.async.bulk, completion counted on one mbarrier per stage), so many
//    kilobytes per warp are in flight without holding registers. Each lane
//    then reads its 16 bytes of an atom: exactly the A fragments of four
//    m16n8k16 MMAs in the swapped form y^T = W^T · x^T (the weight columns
//    fill the MMA's 16 rows, the tokens its 8 columns).
//  * Dequantisation ("vLLM AWQ 4-bit 量化实践" §5.3: (b - zeros) * scales) is
//    split: the MMA consumes (q - z), which is exact in fp16/bf16, and the
//    per-(group, column) scale multiplies the fp32 partial sum of each group.
//    One LOP3 turns a nibble pair into MAGIC + q halves and one packed
//    subtraction of MAGIC + z leaves q - z. A warp's scales and zeros are
//    staged once in shared memory.
//  * The CTA stages its slice of x in shared memory (gathering x[:, perm] for
//    act-order layers), padded so fragment loads are free of bank conflicts.
//  * Split-K across the CTAs of a thread-block cluster (up to 8 along K): each
//    CTA pushes its fp32 partial sums into the shared memory of the CTA that
//    owns those output columns (distributed shared memory stores), one
//    cluster barrier later every owner sums its slice over the peers in a
//    fixed order (deterministic, no global workspace, no atomics:
//    "vLLM AWQ 4-bit 量化实践" §5.3 names split-K for the fused kernel).
//  * Launch order inside a CTA: the small loads that gate the first MMA (x,
//    scales, zeros) are issued before the weight stream, so they are not
//    queued behind it; the weight stream is marked evict-first in L2. Launches
//    use programmatic stream serialization: a CTA may become resident while
//    the previous kernel drains, and waits for it before touching memory.
//  * Waits on the ring's mbarriers are bounded (one second); on a timeout the
//    warp records W4_ERR_TIMEOUT in the device status word, lets its copies in
//    flight land (bounded again) and stops computing.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "sm100_ptx.cuh"
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace cg = cooperative_groups;

namespace w4 {

extern __device__ int g_device_status;

namespace {

using namespace sm100;

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int ATOM_K = 64;
constexpr int ATOM_WORDS = 128;
constexpr int ATOM_BYTES = 512;
constexpr int MAX_SPLIT = 8;
constexpr int STAGE_ATOMS = 4;       // atoms per ring stage (2 KB)
constexpr int MAX_RING = 8;          // stages per warp, upper bound
constexpr int X_BUDGET = 48 * 1024;  // bytes of staged x per CTA
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

struct DecodeParams {
  const uint16_t* x;       // [M][K]
  const uint32_t* qw;      // TILE words
  const uint16_t* scales;  // [G][N]
  const uint32_t* zeros;   // [G][N/8] standard order
  const int32_t* perm;     // [K] or nullptr
  uint16_t* y;             // [M][N]
  int M, N, K;
  int gshift;              // group = 1 << gshift; 31 = one group over all of K
  int A;                   // K / 64
  int WN;                  // warps along N per CTA (WK = 8 / WN along K)
  int ring;                // stages per warp
  int chunk_atoms;         // atoms of x staged in shared memory at a time
  int x_stride;            // shared x row stride in halves
  int maxg;                // group slots of the per-warp scale / zero stage
  int xp_stride;           // row length of the x prefix sums (2 * chunk_atoms + 1)
  int slice;               // output columns owned by each CTA of a cluster
};

struct SmemLayout {
  int xs, ring, bars, meta_s, meta_z, meta_f, xpre, red, recv, total;
};

// x keeps M token rows plus one row of zeros (read by the MMA lanes whose
// token row is beyond M).
__host__ __device__ inline SmemLayout smem_layout(int MT, int m_rows, int x_stride, int ring,
                                                  int maxg, int xp_stride, int WN, int S,
                                                  int slice) {
  SmemLayout L;
  L.xs = 0;
  L.ring = (((m_rows + 1) * x_stride * 2) + 1023) & ~1023;
  L.bars = L.ring + DEC_WARPS * ring * STAGE_ATOMS * ATOM_BYTES;
  L.meta_s = (L.bars + (DEC_WARPS * ring + 1) * 8 + 15) & ~15;
  L.meta_z = L.meta_s + DEC_WARPS * maxg * 32;
  L.meta_f = (L.meta_z + DEC_WARPS * maxg * 8 + 15) & ~15;
  L.xpre = (L.meta_f + DEC_WARPS * maxg * 16 * 8 + 15) & ~15;
  L.red = (L.xpre + 8 * MT * xp_stride * 4 + 15) & ~15;
  const int red_bytes = WN < DEC_WARPS ? DEC_WARPS * 16 * 8 * MT * 4 : 0;
  L.recv = (L.red + red_bytes + 15) & ~15;
  L.total = L.recv + S * slice * 8 * MT * 4;
  return L;
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Weight-stream copy: the weights are read once per call, so they are marked
// evict-first in L2, which keeps x, scales and zeros resident.
__device__ __forceinline__ void bulk_copy_stream(uint32_t dst, const void* src, uint32_t bytes,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte shared-memory load from a 32-bit shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Bounded wait; false when the limit ran out (the caller records the timeout).
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
  return true;
}

// D += A * B for one m16n8k16 tile, fp32 accumulate (non-volatile: the
// compiler may schedule it freely; its outputs keep it alive).
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
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

// MT: token tiles of 8 (M <= 8 * MT). G64: every 64-row atom lies in one group.
// With bf16 the MMA consumes the codes as 128 + q (exact in bf16) and each
// group's partial sum is corrected by (128 + z) * sum(x) before scaling; with
// fp16 the operand is q - z (exact) and needs no correction.
#ifndef W4_DECODE_MIN_CTAS
#define W4_DECODE_MIN_CTAS 3  // resident CTAs per SM the register budget is sized for (M <= 16)
#endif

template <int MT, bool BF16, bool G64>
__global__ void __launch_bounds__(DEC_THREADS, MT <= 2 ? W4_DECODE_MIN_CTAS : 2) w4a16_decode_kernel(const DecodeParams p) {
  constexpr uint32_t MAGIC = Magic<BF16>::pair;
  constexpr bool BIAS = BF16;
  constexpr int SLOT = STAGE_ATOMS * ATOM_BYTES;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gg = lane >> 2, t = lane & 3;
  const int S = gridDim.y;          // split-K factor == cluster size along y
  const int srank = blockIdx.y;     // rank inside the cluster
  const int WN = p.WN, WK = DEC_WARPS / WN;
  const int MR = 8 * MT;
  const int RINGN = p.ring;
  const SmemLayout L = smem_layout(MT, p.M, p.x_stride, RINGN, p.maxg, p.xp_stride, WN, S, p.slice);

  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
  uint8_t* ring = smem + L.ring + warp * (RINGN * SLOT);
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar0 = smem_addr(smem + L.bars + warp * RINGN * 8);
  const uint32_t xbar = smem_addr(smem + L.bars + DEC_WARPS * RINGN * 8);
  uint16_t* meta_s = reinterpret_cast<uint16_t*>(smem + L.meta_s) + warp * p.maxg * 16;
  uint2* meta_z = reinterpret_cast<uint2*>(smem + L.meta_z) + warp * p.maxg;
  // per (group, column): {scale, (128 + zero) * scale} in fp32, the two factors
  // of the bf16 group correction
  float2* meta_f = reinterpret_cast<float2*>(smem + L.meta_f) + warp * p.maxg * 16;
  float* xpre = reinterpret_cast<float*>(smem + L.xpre);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  const int NCOL = 16 * WN;
  const uint32_t gmask = p.gshift >= 31 ? 0x7FFFFFFFu : ((1u << p.gshift) - 1u);

  // CTA K range in atoms
  const int ka0 = (int)((long long)srank * p.A / S);
  const int ka1 = (int)((long long)(srank + 1) * p.A / S);

  const int wn = warp % WN, wk = warp / WN;
  const int nt = blockIdx.x * WN + wn;
  const bool has_cols = nt < p.N / 16;
  const uint32_t* wsrc = p.qw + (size_t)nt * p.A * ATOM_WORDS;  // this tile's atom run
  uint16_t* xzero = xs + (size_t)p.M * p.x_stride;              // the zero row

  // Launched with programmatic stream serialization: the CTA may become
  // resident while the previous kernel in the stream drains. It waits for that
  // kernel (griddepcontrol.wait) before touching global memory, then lets the
  // next kernel in the stream start its own launch.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const uint64_t stream_policy = evict_first_policy();

  if (lane == 0) {
    for (int s = 0; s < RINGN; ++s) mbar_init(bar0 + 8 * s, 1);
    if (warp == 0) mbar_init(xbar, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < p.x_stride / 8; i += DEC_THREADS)
    reinterpret_cast<uint4*>(xzero)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  float acc[MT][4], tot[MT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = tot[i][j] = 0.f;
  int hs = 0;           // chunk-relative half-atom index where the open group started
  int g_first = 0;      // first group of this warp's run in the chunk
  float s_lo = 0.f, s_hi = 0.f, zs_lo = 0.f, zs_hi = 0.f;
  uint32_t zl = 0, zh = 0;
  uint32_t it = 0;      // stages consumed by this warp
  uint32_t rslot = 0;   // ring slot of the next stage to consume (== it % RINGN)
  uint32_t rphase = 0;  // its mbarrier phase parity (== (it / RINGN) & 1)
  uint32_t xphase = 0;  // phase of the x barrier
  bool alive = true;    // false once a wait gave up

  // tot += s * acc - (MAGIC + z) * s * (sum of x over halves [h0, h1)); acc = 0
  // ((MAGIC + z) * s is exact in fp32: two 8-bit significands)
  auto flush = [&](int h0, int h1) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if constexpr (BIAS) {
        const float* xp = xpre + (8 * mt + 2 * t) * p.xp_stride;
        const float c0 = xp[h1] - xp[h0];
        const float c1 = xp[p.xp_stride + h1] - xp[p.xp_stride + h0];
        tot[mt][0] = fmaf(s_lo, acc[mt][0], fmaf(-zs_lo, c0, tot[mt][0]));
        tot[mt][1] = fmaf(s_lo, acc[mt][1], fmaf(-zs_lo, c1, tot[mt][1]));
        tot[mt][2] = fmaf(s_hi, acc[mt][2], fmaf(-zs_hi, c0, tot[mt][2]));
        tot[mt][3] = fmaf(s_hi, acc[mt][3], fmaf(-zs_hi, c1, tot[mt][3]));
      } else {
        tot[mt][0] = fmaf(s_lo, acc[mt][0], tot[mt][0]);
        tot[mt][1] = fmaf(s_lo, acc[mt][1], tot[mt][1]);
        tot[mt][2] = fmaf(s_hi, acc[mt][2], tot[mt][2]);
        tot[mt][3] = fmaf(s_hi, acc[mt][3], tot[mt][3]);
      }
      acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    }
  };
  // scale / zero registers for group gi (staged in shared memory)
  auto open_group = [&](int gi) {
    const int gl = gi - g_first;
    const float2 f_lo = meta_f[gl * 16 + gg], f_hi = meta_f[gl * 16 + gg + 8];
    s_lo = f_lo.x;
    zs_lo = f_lo.y;
    s_hi = f_hi.x;
    zs_hi = f_hi.y;
    if constexpr (!BIAS) {
      const uint2 zw = meta_z[gl];
      const uint32_t z0 = (zw.x >> (4 * gg)) & 0xF;
      const uint32_t z1 = (zw.y >> (4 * gg)) & 0xF;
      zl = MAGIC | z0 | (z0 << 16);
      zh = MAGIC | z1 | (z1 << 16);
    }
  };
  // expand one group's 16 scales and 16 zeros into meta_f
  auto stage_group_f = [&](int gl, const uint4 a, const uint4 b, const uint2 z) {
    const uint32_t sv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint16_t sb = (uint16_t)(sv[c >> 1] >> (16 * (c & 1)));
      const float sf = half_bits_to_float<BF16>(sb);
      const uint32_t zc = ((c < 8 ? z.x : z.y) >> (4 * (c & 7))) & 0xF;
      meta_f[gl * 16 + c] = make_float2(sf, (float)(128 + zc) * sf);
    }
  };

  for (int c0 = ka0; c0 < ka1; c0 += p.chunk_atoms) {
    const int c1 = min(ka1, c0 + p.chunk_atoms);
    const int kx0 = c0 * ATOM_K;
    const int KC = (c1 - c0) * ATOM_K;
    const int wa0 = c0 + (int)((long long)wk * (c1 - c0) / WK);
    const int wa1 = c0 + (int)((long long)(wk + 1) * (c1 - c0) / WK);
    const int n_atoms = (has_cols && alive) ? wa1 - wa0 : 0;
    const int n_stages = (n_atoms + STAGE_ATOMS - 1) / STAGE_ATOMS;
    const bool x_async = p.perm == nullptr;

    // Stage j of this chunk goes to ring slot (it + j) % RINGN, where `it` is
    // the warp's consumed-stage count when the chunk starts.
    auto issue = [&](int j, uint32_t slot) {
      const int a = wa0 + j * STAGE_ATOMS;
      const uint32_t bytes = (uint32_t)min(STAGE_ATOMS, wa1 - a) * ATOM_BYTES;
      mbar_arrive_expect_tx(bar0 + 8 * slot, bytes);
      bulk_copy_stream(ring_s + slot * SLOT, wsrc + (size_t)a * ATOM_WORDS, bytes, bar0 + 8 * slot,
                       stream_policy);
    };

    // 1) the loads that gate the first MMA go first: x, then scales / zeros
    if (x_async && tid == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(xbar, (uint32_t)(p.M * KC * 2));
      for (int m = 0; m < p.M; ++m)
        bulk_copy(smem_addr(xs + (size_t)m * p.x_stride), p.x + (size_t)m * p.K + kx0,
                  (uint32_t)(KC * 2), xbar);
    }
    g_first = (wa0 * ATOM_K) >> p.gshift;
    const int ng = n_atoms > 0 ? ((wa1 * ATOM_K - 1) >> p.gshift) - g_first + 1 : 0;
    uint4 ms0 = make_uint4(0, 0, 0, 0), ms1 = ms0;
    uint2 mz = make_uint2(0, 0);
    if (lane < ng) {
      const int gi = g_first + lane;
      const uint4* sp = reinterpret_cast<const uint4*>(p.scales + (size_t)gi * p.N + nt * 16);
      ms0 = __ldg(sp);
      ms1 = __ldg(sp + 1);
      mz = __ldg(reinterpret_cast<const uint2*>(p.zeros + (size_t)gi * (p.N / 8) + nt * 2));
    }
    // 2) then the weight stream
    if (lane == 0 && n_stages > 0) {
      fence_proxy_async_smem();  // earlier reads of the ring precede these copies
      uint32_t sl = rslot;
      for (int j = 0; j < min(RINGN, n_stages); ++j) {
        issue(j, sl);
        sl = (sl + 1 == (uint32_t)RINGN) ? 0u : sl + 1;
      }
    }
    // 3) scales / zeros to shared memory (groups beyond 32 per warp: direct)
    if (lane < ng) {
      uint4* sd = reinterpret_cast<uint4*>(meta_s + lane * 16);
      sd[0] = ms0;
      sd[1] = ms1;
      meta_z[lane] = mz;
      stage_group_f(lane, ms0, ms1, mz);
    }
    for (int gl = lane + 32; gl < ng; gl += 32) {
      const int gi = g_first + gl;
      const uint4* sp = reinterpret_cast<const uint4*>(p.scales + (size_t)gi * p.N + nt * 16);
      uint4* sd = reinterpret_cast<uint4*>(meta_s + gl * 16);
      const uint4 a = __ldg(sp), b = __ldg(sp + 1);
      const uint2 z = __ldg(reinterpret_cast<const uint2*>(p.zeros + (size_t)gi * (p.N / 8) + nt * 2));
      sd[0] = a;
      sd[1] = b;
      meta_z[gl] = z;
      stage_group_f(gl, a, b, z);
    }
    if (!x_async) {
      // act-order: gather x[:, perm] with plain loads
      const int chunks = KC / 8;
      for (int i = tid; i < p.M * chunks; i += DEC_THREADS) {
        const int m = i / chunks, c = i - m * chunks;
        const uint16_t* xr = p.x + (size_t)m * p.K;
        uint16_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __ldg(xr + __ldg(p.perm + kx0 + 8 * c + e));
        uint4 v;
        v.x = h[0] | ((uint32_t)h[1] << 16);
        v.y = h[2] | ((uint32_t)h[3] << 16);
        v.z = h[4] | ((uint32_t)h[5] << 16);
        v.w = h[6] | ((uint32_t)h[7] << 16);
        *reinterpret_cast<uint4*>(xs + (size_t)m * p.x_stride + 8 * c) = v;
      }
      __syncthreads();
    } else {
      if (!bounded_wait(xbar, xphase & 1)) {
        if (tid == 0) atomicExch(&g_device_status, W4_ERR_TIMEOUT);
        alive = false;
      }
      ++xphase;
    }

    // 4) prefix sums of x over 32-row halves (bf16 zero correction), one token
    //    row per warp at a time, lanes over halves
    const int n32 = KC / 32;
    if constexpr (BIAS) {
      for (int m = warp; m < MR; m += DEC_WARPS) {
        float* xp = xpre + m * p.xp_stride;
        float carry = 0.f;
        if (lane == 0) xp[0] = 0.f;
        for (int h0 = 0; h0 < n32; h0 += 32) {
          const int hh = h0 + lane;
          float sum = 0.f;
          if (m < p.M && hh < n32) {
            const uint4* xr = reinterpret_cast<const uint4*>(xs + (size_t)m * p.x_stride + 32 * hh);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = xr[q];
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                sum += __uint_as_float(wv[e] << 16) + __uint_as_float(wv[e] & 0xFFFF0000u);
            }
          }
#pragma unroll
          for (int d = 1; d < 32; d <<= 1) {
            const float v = __shfl_up_sync(0xFFFFFFFFu, sum, d);
            if (lane >= d) sum += v;
          }
          if (hh < n32) xp[hh + 1] = carry + sum;
          carry += __shfl_sync(0xFFFFFFFFu, sum, 31);
        }
      }
    }
    __syncthreads();  // x prefix sums and every warp's scale / zero stage are ready

    // 5) consume the ring. Shared-memory operands are addressed with 32-bit
    //    shared-window addresses: per stage one base for the weights and one per
    //    token tile for x, with constant offsets inside the stage.
    uint32_t xa[MT];  // this lane's x row (or the zero row) at the warp's first atom, column 8t
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int row = 8 * mt + gg;
      xa[mt] = smem_addr(row < p.M ? xs + (size_t)row * p.x_stride : xzero) +
               2u * (uint32_t)(8 * t + (wa0 - c0) * ATOM_K);
    }
    hs = 2 * (wa0 - c0);
    // atoms left before the next group boundary (groups of 64 rows or more)
    const int apg = G64 ? (p.gshift >= 31 ? (1 << 30) : (1 << (p.gshift - 6))) : 1;
    int gleft = G64 ? apg - (wa0 & (apg - 1)) : 0;
    if (n_atoms > 0) open_group((wa0 * ATOM_K) >> p.gshift);

    // one atom: 64 rows x 16 columns, four m16n8k16 MMAs per token tile;
    // xo = byte offset of the atom's x columns from xa
    auto atom = [&](int a, const uint4 w, const uint32_t xo) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (G64) {
          if (h == 0 && gleft == 0) {  // a group starts at this atom
            const int hcur = 2 * (a - c0);
            flush(hs, hcur);
            hs = hcur;
            open_group((a * ATOM_K) >> p.gshift);
            gleft = apg;
          }
        } else {
          const uint32_t kabs = (uint32_t)(a * ATOM_K + 32 * h);
          if ((kabs & gmask) == 0) {
            const int hcur = 2 * (a - c0) + h;
            flush(hs, hcur);
            hs = hcur;
            open_group((int)(kabs >> p.gshift));
          }
        }
        const uint32_t wlo = h ? w.z : w.x;  // column gg
        const uint32_t whi = h ? w.w : w.y;  // column gg + 8
        uint4 xf[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) xf[mt] = lds128(xa[mt] + xo + 64u * h);
#pragma unroll
        for (int step = 0; step < 2; ++step) {
          const int sh = 8 * step;
          uint32_t a0 = lop3_and_or(wlo >> sh, 0x000F000Fu, MAGIC);
          uint32_t a2 = lop3_and_or(wlo >> (sh + 4), 0x000F000Fu, MAGIC);
          uint32_t a1 = lop3_and_or(whi >> sh, 0x000F000Fu, MAGIC);
          uint32_t a3 = lop3_and_or(whi >> (sh + 4), 0x000F000Fu, MAGIC);
          if constexpr (!BIAS) {
            a0 = sub_x2<BF16>(a0, zl);
            a2 = sub_x2<BF16>(a2, zl);
            a1 = sub_x2<BF16>(a1, zh);
            a3 = sub_x2<BF16>(a3, zh);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t b0 = step ? xf[mt].z : xf[mt].x;
            const uint32_t b1 = step ? xf[mt].w : xf[mt].y;
            mma16816<BF16>(acc[mt], a0, a1, a2, a3, b0, b1);
          }
        }
      }
      if constexpr (G64) --gleft;
    };

    const uint32_t wlane = ring_s + (uint32_t)lane * 16u;
    for (int j = 0; j < n_stages; ++j) {
      const uint32_t slot = rslot;
      if (!bounded_wait(bar0 + 8 * slot, rphase)) {
        // give up: record it, let the copies in flight land, stop streaming
        if (lane == 0) atomicExch(&g_device_status, W4_ERR_TIMEOUT);
        const int in_flight = min(RINGN, n_stages - j);
        for (int q = 0; q < in_flight; ++q)
          bounded_wait(bar0 + 8 * ((it + q) % RINGN), ((it + q) / RINGN) & 1);
        alive = false;
        break;
      }
      const uint32_t st = wlane + slot * SLOT;
      const int a_base = wa0 + j * STAGE_ATOMS;
      const uint32_t xo = (uint32_t)j * (STAGE_ATOMS * ATOM_K * 2);
      if (a_base + STAGE_ATOMS <= wa1) {
        uint4 w[STAGE_ATOMS];
#pragma unroll
        for (int u = 0; u < STAGE_ATOMS; ++u) w[u] = lds128(st + u * ATOM_BYTES);
#pragma unroll
        for (int u = 0; u < STAGE_ATOMS; ++u) atom(a_base + u, w[u], xo + u * (ATOM_K * 2));
      } else {
        for (int u = 0; u < wa1 - a_base; ++u)
          atom(a_base + u, lds128(st + u * ATOM_BYTES), xo + u * (ATOM_K * 2));
      }
      __syncwarp();
      if (lane == 0 && j + RINGN < n_stages) {
        fence_proxy_async_smem();  // the reads of this slot precede the next copy into it
        issue(j + RINGN, slot);    // slot == (it_at_chunk_start + j + RINGN) % RINGN
      }
      ++it;
      if (++rslot == (uint32_t)RINGN) {
        rslot = 0;
        rphase ^= 1u;
      }
    }
    // the prefix sums and the scale / zero stage belong to this chunk: close the group
    if (n_atoms > 0) flush(hs, 2 * (wa1 - c0));
    __syncthreads();  // the next chunk overwrites xs, xpre and the scale / zero stage
  }

  // ---- split-K: push partial sums to the CTA that owns each output column -------
  cg::cluster_group cluster = cg::this_cluster();
  const int SL = p.slice;
  auto push = [&](int col, int m, float v) {
    const int owner = col / SL;
    float* dst = cluster.map_shared_rank(recv, owner);
    dst[((size_t)srank * SL + (col - owner * SL)) * MR + m] = v;
  };
  if (WK == 1) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int m0 = 8 * mt + 2 * t;
      const int ca = wn * 16 + gg, cb = ca + 8;
      if (m0 < p.M) {
        push(ca, m0, tot[mt][0]);
        push(cb, m0, tot[mt][2]);
      }
      if (m0 + 1 < p.M) {
        push(ca, m0 + 1, tot[mt][1]);
        push(cb, m0 + 1, tot[mt][3]);
      }
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int m0 = 8 * mt + 2 * t;
      float* r0 = red + ((size_t)wk * NCOL + wn * 16 + gg) * MR;
      float* r1 = red + ((size_t)wk * NCOL + wn * 16 + gg + 8) * MR;
      r0[m0] = tot[mt][0];
      r0[m0 + 1] = tot[mt][1];
      r1[m0] = tot[mt][2];
      r1[m0 + 1] = tot[mt][3];
    }
    __syncthreads();
    for (int o = tid; o < NCOL * p.M; o += DEC_THREADS) {
      const int col = o / p.M, m = o - col * p.M;
      float v = 0.f;
      for (int q = 0; q < WK; ++q) v += red[((size_t)q * NCOL + col) * MR + m];
      push(col, m, v);
    }
  }
  cluster.sync();
  {
    const int c_lo = srank * SL;
    const int c_hi = min(NCOL, c_lo + SL);
    const int width = c_hi - c_lo;
    for (int o = tid; o < width * p.M; o += DEC_THREADS) {
      const int m = o / width, cl = o - m * width;
      const int n = blockIdx.x * NCOL + c_lo + cl;
      if (n >= p.N) continue;
      float sum = 0.f;
      for (int r = 0; r < S; ++r) sum += recv[((size_t)r * SL + cl) * MR + m];
      p.y[(size_t)m * p.N + n] = float_to_half_bits<BF16>(sum);
    }
  }
}

template <int MT, bool BF16, bool G64>
void* kernel_ptr() {
  return reinterpret_cast<void*>(&w4a16_decode_kernel<MT, BF16, G64>);
}

template <int MT>
void* pick_mt(bool bf16, bool g64) {
  if (bf16) return g64 ? kernel_ptr<MT, true, true>() : kernel_ptr<MT, true, false>();
  return g64 ? kernel_ptr<MT, false, true>() : kernel_ptr<MT, false, false>();
}

void* pick_kernel(int MT, bool bf16, bool g64) {
  switch (MT) {
    case 1: return pick_mt<1>(bf16, g64);
    case 2: return pick_mt<2>(bf16, g64);
    case 4: return pick_mt<4>(bf16, g64);
    case 8: return pick_mt<8>(bf16, g64);
    default: return nullptr;
  }
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device); the
// attribute call is then kept out of the launch path (and out of graph capture).
cudaError_t ensure_smem(void* fn, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t key = reinterpret_cast<uint64_t>(fn) ^ (static_cast<uint64_t>(dev) << 56);
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

// Rows of x (per token) a CTA stages at a time.
int max_rows_per_chunk(int M) {
  const int rows = X_BUDGET / (M * 2);
  return std::max(ATOM_K, (rows / ATOM_K) * ATOM_K);
}

struct DecodePlan {
  int WN, S;
  int ring, chunk_atoms, x_stride, maxg, xp_stride, slice;
  SmemLayout L;
};

// Shared-memory plan of one launch shape.
DecodePlan shape_plan(int WN, int S, int A, int Mc, int MT, int gshift, int ring) {
  DecodePlan d;
  d.WN = WN;
  d.S = S;
  d.ring = ring;
  const int cta_atoms = (A + S - 1) / S;
  d.chunk_atoms = std::min(cta_atoms, max_rows_per_chunk(Mc) / ATOM_K);
  d.x_stride = d.chunk_atoms * ATOM_K + 32;  // halves; row stride = 64 mod 128 bytes
  const int WK = DEC_WARPS / WN;
  const int warp_atoms = (d.chunk_atoms + WK - 1) / WK;
  d.maxg = (gshift == 31) ? 1 : (warp_atoms * ATOM_K >> gshift) + 2;
  d.xp_stride = 2 * d.chunk_atoms + 1;
  d.slice = (16 * WN + S - 1) / S;
  d.L = smem_layout(MT, Mc, d.x_stride, ring, d.maxg, d.xp_stride, WN, S, d.slice);
  return d;
}

// Deepest ring (2..MAX_RING stages, no deeper than the warp's run) that keeps
// `per_sm` CTAs resident.
DecodePlan fit_ring(int WN, int S, int A, int Mc, int MT, int gshift, int per_sm, int smem_per_sm) {
  const int WK = DEC_WARPS / WN;
  const int warp_atoms = ((A + S - 1) / S + WK - 1) / WK;
  const int need = std::max(2, std::min(MAX_RING, (warp_atoms + STAGE_ATOMS - 1) / STAGE_ATOMS));
  DecodePlan d = shape_plan(WN, S, A, Mc, MT, gshift, 2);
  for (int r = need; r >= 2; --r) {
    d = shape_plan(WN, S, A, Mc, MT, gshift, r);
    if ((d.L.total + 1024) * per_sm <= smem_per_sm) break;
  }
  return d;
}

// Choose warps-along-N and the split-K factor with a small time model. A
// wave of CTAs shares the HBM bandwidth among its members and pays a fixed
// start-up / drain cost; a CTA streams at most ~1/16 of an SM's share alone
// per warp, so fewer than two resident CTAs per SM leave bandwidth unused.
DecodePlan plan_decode(int N, int K, int Mc, int MT, int gshift, const DeviceInfo& info) {
  const int NT = N / 16, A = K / ATOM_K;
  const int reg_ctas = MT <= 2 ? W4_DECODE_MIN_CTAS : 2;
  const double overhead = 2.5e-6, bw = 6.5e12;
  const double sm_bw = bw / info.sm_count;
  DecodePlan best = shape_plan(8, 1, A, Mc, MT, gshift, 2);
  double best_t = 1e30;
  for (int WN = 8; WN >= 1; WN >>= 1) {
    const int WK = DEC_WARPS / WN;
    const int cols = (NT + WN - 1) / WN;
    for (int S = 1; S <= MAX_SPLIT && S <= A; ++S) {
      if ((double)A / (S * WK) < 1.0) continue;
      // three resident CTAs per SM (more warps to hide latency) when registers
      // allow it and a ring of at least three stages still fits; else two
      DecodePlan d = fit_ring(WN, S, A, Mc, MT, gshift, 2, info.smem_per_sm);
      if (reg_ctas >= 3) {
        const DecodePlan d3 = fit_ring(WN, S, A, Mc, MT, gshift, 3, info.smem_per_sm);
        if (d3.ring >= 3 && (d3.L.total + 1024) * 3 <= info.smem_per_sm) d = d3;
      }
      const int smem_ctas = info.smem_per_sm / (d.L.total + 1024);
      const int per_sm = std::max(1, std::min(reg_ctas, smem_ctas));
      const long long slots = (long long)per_sm * info.sm_count;
      long long left = (long long)cols * S;
      const double cta_bytes = (double)(16 * WN) * ((double)A / S) * 32.0;  // 64 rows x 16 cols / 2
      double t = 0.0;
      while (left > 0) {
        const long long now = std::min(left, slots);
        const double per_sm_ctas = (double)now / info.sm_count;
        // an SM streams at its share of HBM once it holds two CTAs
        const double rate = sm_bw * std::min(1.0, per_sm_ctas / 2.0) / std::max(1.0, per_sm_ctas);
        t += overhead + cta_bytes / rate;
        left -= now;
      }
      t += 0.05e-6 * S;
      if (t < best_t) {
        best_t = t;
        best = d;
      }
    }
  }
  return best;
}

int log2_exact(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return (1 << s) == v ? s : -1;
}

}  // namespace

cudaError_t launch_decode(const GemmArgs& a, cudaStream_t stream) {
  DeviceInfo info;
  cudaError_t err = device_info(&info);
  if (err != cudaSuccess) return err;
  int gshift = log2_exact(a.group);
  if (a.group == a.K || gshift < 0) gshift = 31;  // one group over all of K
  const int A = a.K / ATOM_K;
  const bool g64 = gshift >= 6;  // groups of 64 or more: one group per atom
  for (int r0 = 0; r0 < a.M; r0 += DECODE_MAX_M) {
    const int Mc = std::min(DECODE_MAX_M, a.M - r0);
    const int MT = Mc <= 8 ? 1 : Mc <= 16 ? 2 : Mc <= 32 ? 4 : 8;
    const DecodePlan plan = plan_decode(a.N, a.K, Mc, MT, gshift, info);
    void* fn = pick_kernel(MT, a.bf16 != 0, g64);
    if ((err = ensure_smem(fn, plan.L.total)) != cudaSuccess) return err;

    DecodeParams p;
    p.x = static_cast<const uint16_t*>(a.x) + (size_t)r0 * a.K;
    p.qw = a.qw;
    p.scales = static_cast<const uint16_t*>(a.scales);
    p.zeros = a.zeros;
    p.perm = a.perm;
    p.y = static_cast<uint16_t*>(a.y) + (size_t)r0 * a.N;
    p.M = Mc;
    p.N = a.N;
    p.K = a.K;
    p.gshift = gshift;
    p.A = A;
    p.WN = plan.WN;
    p.ring = plan.ring;
    p.chunk_atoms = plan.chunk_atoms;
    p.x_stride = plan.x_stride;
    p.maxg = plan.maxg;
    p.xp_stride = plan.xp_stride;
    p.slice = plan.slice;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.N / 16 + plan.WN - 1) / plan.WN, plan.S, 1);
    cfg.blockDim = dim3(DEC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = plan.L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = plan.S;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void* args[] = {&p};
    if ((err = cudaLaunchKernelExC(&cfg, fn, args)) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace w4
