// Small-M (decode) W4A16 GEMM: y[M][N] = x[M][K] · W, M <= 64 per launch.
//
// Decode is bound by streaming the packed weights from HBM ("vLLM 学习手册 01.
// 量化" §1: decode has FLOPs/Bytes ~ 1 and moving the weights dominates), so
// the kernel is organised around the weight stream:
//
//  * Each warp owns one 16-column tile and a contiguous run of 64-row TILE
//    atoms. One 16-byte load per lane fetches a whole atom (512 B per warp,
//    fully coalesced); the four words a lane receives are exactly the A
//    fragments of four m16n8k16 MMAs in the swapped form y^T = W^T · x^T (the
//    weight columns fill the MMA's 16 rows, the tokens its 8 columns). Loads
//    are issued PIPE atoms ahead of use to keep enough bytes in flight.
//  * Dequantisation ("vLLM AWQ 4-bit 量化实践" §5.3: (b - zeros) * scales) is
//    split: the MMA consumes (q - z), which is exact in fp16/bf16, and the
//    per-(group, column) scale is applied to the fp32 partial sum of each
//    group. One LOP3 turns a nibble pair into MAGIC + q halves and one packed
//    subtraction of MAGIC + z leaves q - z.
//  * The CTA stages its slice of x in shared memory once (gathering x[:, perm]
//    for act-order layers), padded so fragment loads are free of bank conflicts.
//  * Split-K across the CTAs of a thread-block cluster (up to 8 along K): each
//    CTA leaves its fp32 partial tile in its own shared memory, and after a
//    cluster barrier every CTA sums a slice of the outputs over all peers
//    through distributed shared memory, in a fixed order (deterministic, no
//    global workspace, no atomics, no spin waits: "vLLM AWQ 4-bit 量化实践"
//    §5.3 names split-K for the fused kernel).
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace cg = cooperative_groups;

namespace w4 {
namespace {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int ATOM_K = 64;
constexpr int ATOM_WORDS = 128;
constexpr int MAX_SPLIT = 8;

struct DecodeParams {
  const uint16_t* x;      // [M][K]
  const uint32_t* qw;     // TILE words
  const uint16_t* scales; // [G][N]
  const uint32_t* zeros;  // [G][N/8] standard order
  const int32_t* perm;    // [K] or nullptr
  uint16_t* y;            // [M][N]
  int M, N, K, group;
  int A;                  // K / 64
  int WN;                 // warps along N per CTA (WK = 8 / WN along K)
  int chunk_atoms;        // atoms of x staged in shared memory at a time
  int x_stride;           // shared x row stride in halves
};

template <int MT>
struct Pipe {
  static constexpr int depth = MT <= 2 ? 8 : (MT == 4 ? 4 : 2);
};

// Scale pair (rows gg and gg+8 of the tile) and the tile's 16 zeros for one group.
struct Meta {
  uint32_t s;    // lo 16 bits: scale of column gg, hi: column gg+8
  uint2 z;       // zeros words for columns [16nt, 16nt+8) and [16nt+8, 16nt+16)
};

__device__ __forceinline__ Meta load_meta(const DecodeParams& p, int gi, int nt, int gg) {
  Meta m;
  const uint16_t* sp = p.scales + (size_t)gi * p.N + nt * 16 + gg;
  const uint32_t lo = __ldg(sp), hi = __ldg(sp + 8);
  m.s = lo | (hi << 16);
  m.z = __ldg(reinterpret_cast<const uint2*>(p.zeros + (size_t)gi * (p.N / 8) + nt * 2));
  return m;
}

template <int MT, bool BF16, bool G32>
__global__ void __launch_bounds__(DEC_THREADS, 2) w4a16_decode_kernel(const DecodeParams p) {
  constexpr int PIPE = Pipe<MT>::depth;
  constexpr uint32_t MAGIC = Magic<BF16>::pair;
  extern __shared__ __align__(16) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gg = lane >> 2, t = lane & 3;
  const int S = gridDim.y;          // split-K factor == cluster size along y
  const int srank = blockIdx.y;     // rank inside the cluster
  const int WN = p.WN, WK = DEC_WARPS / WN;

  // CTA K range in atoms.
  const int ka0 = (int)((long long)srank * p.A / S);
  const int ka1 = (int)((long long)(srank + 1) * p.A / S);

  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)8 * MT * p.x_stride * 2);
  const int NCOL = 16 * WN;     // columns per CTA
  const int MR = 8 * MT;        // padded rows

  const int wn = warp % WN, wk = warp / WN;
  const int nt = blockIdx.x * WN + wn;
  const int NT = p.N / 16;
  const bool warp_has_cols = nt < NT;
  const uint32_t* wbase = p.qw + (size_t)nt * p.A * ATOM_WORDS + lane * 4;
  const int group = p.group;

  float acc[MT][4], tot[MT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = tot[i][j] = 0.f;
  int cur_g = -1;
  float s_lo = 0.f, s_hi = 0.f;
  uint32_t zl = 0, zh = 0;

  // The CTA range is walked in chunks whose x slice fits the shared buffer.
  for (int c0 = ka0; c0 < ka1; c0 += p.chunk_atoms) {
    const int c1 = min(ka1, c0 + p.chunk_atoms);
    const int kx0 = c0 * ATOM_K;
    const int KC = (c1 - c0) * ATOM_K;

    // ---- stage x[:, kx0:kx0+KC] (gathered through perm) ------------------------
    {
      const int chunks = KC / 8;
      for (int i = tid; i < MR * chunks; i += DEC_THREADS) {
        const int m = i / chunks, c = i % chunks;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (m < p.M) {
          const uint16_t* xr = p.x + (size_t)m * p.K;
          if (p.perm == nullptr) {
            v = __ldg(reinterpret_cast<const uint4*>(xr + kx0 + 8 * c));
          } else {
            uint16_t h[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = __ldg(xr + __ldg(p.perm + kx0 + 8 * c + e));
            v.x = h[0] | ((uint32_t)h[1] << 16);
            v.y = h[2] | ((uint32_t)h[3] << 16);
            v.z = h[4] | ((uint32_t)h[5] << 16);
            v.w = h[6] | ((uint32_t)h[7] << 16);
          }
        }
        *reinterpret_cast<uint4*>(xs + (size_t)m * p.x_stride + 8 * c) = v;
      }
    }
    __syncthreads();

    // ---- per-warp weight stream ------------------------------------------------
    const int wa0 = c0 + (int)((long long)wk * (c1 - c0) / WK);
    const int wa1 = c0 + (int)((long long)(wk + 1) * (c1 - c0) / WK);
    if (warp_has_cols && wa1 > wa0) {
      const int n_atoms = wa1 - wa0;
      uint4 wb[PIPE];
      Meta mb[PIPE][G32 ? 2 : 1];

      auto fetch = [&](int slot, int a) {
        wb[slot] = ldg_stream_v4(wbase + (size_t)a * ATOM_WORDS);
        mb[slot][0] = load_meta(p, (a * ATOM_K) / group, nt, gg);
        if constexpr (G32) mb[slot][1] = load_meta(p, (a * ATOM_K + 32) / group, nt, gg);
      };

#pragma unroll
      for (int i = 0; i < PIPE; ++i)
        if (i < n_atoms) fetch(i, wa0 + i);

      for (int base = 0; base < n_atoms; base += PIPE) {
#pragma unroll
        for (int i = 0; i < PIPE; ++i) {
          const int ai = base + i;
          if (ai < n_atoms) {
            const int a = wa0 + ai;
            const uint4 w = wb[i];
            Meta mh[G32 ? 2 : 1];
            mh[0] = mb[i][0];
            if constexpr (G32) mh[1] = mb[i][1];
            if (ai + PIPE < n_atoms) fetch(i, a + PIPE);

#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int gi = (a * ATOM_K + 32 * h) / group;
              if (gi != cur_g) {
                if (cur_g >= 0) {
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt) {
                    tot[mt][0] = fmaf(s_lo, acc[mt][0], tot[mt][0]);
                    tot[mt][1] = fmaf(s_lo, acc[mt][1], tot[mt][1]);
                    tot[mt][2] = fmaf(s_hi, acc[mt][2], tot[mt][2]);
                    tot[mt][3] = fmaf(s_hi, acc[mt][3], tot[mt][3]);
                    acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
                  }
                }
                cur_g = gi;
                const Meta& m = mh[G32 ? h : 0];
                s_lo = half_bits_to_float<BF16>((uint16_t)(m.s & 0xFFFF));
                s_hi = half_bits_to_float<BF16>((uint16_t)(m.s >> 16));
                const uint32_t z0 = (m.z.x >> (4 * gg)) & 0xF;
                const uint32_t z1 = (m.z.y >> (4 * gg)) & 0xF;
                zl = MAGIC | z0 | (z0 << 16);
                zh = MAGIC | z1 | (z1 << 16);
              }
              const uint32_t wlo = h ? w.z : w.x;  // column gg
              const uint32_t whi = h ? w.w : w.y;  // column gg + 8

              // x fragments for this 32-row block: rows 8t..8t+7 of token row 8mt+gg
              uint4 xf[MT];
              const int kl = a * ATOM_K + 32 * h - kx0 + 8 * t;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
                xf[mt] = *reinterpret_cast<const uint4*>(xs + (size_t)(8 * mt + gg) * p.x_stride + kl);

#pragma unroll
              for (int step = 0; step < 2; ++step) {
                const int sh = 8 * step;
                const uint32_t a0 = sub_x2<BF16>(lop3_and_or(wlo >> sh, 0x000F000Fu, MAGIC), zl);
                const uint32_t a2 = sub_x2<BF16>(lop3_and_or(wlo >> (sh + 4), 0x000F000Fu, MAGIC), zl);
                const uint32_t a1 = sub_x2<BF16>(lop3_and_or(whi >> sh, 0x000F000Fu, MAGIC), zh);
                const uint32_t a3 = sub_x2<BF16>(lop3_and_or(whi >> (sh + 4), 0x000F000Fu, MAGIC), zh);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  const uint32_t b0 = step ? xf[mt].z : xf[mt].x;
                  const uint32_t b1 = step ? xf[mt].w : xf[mt].y;
                  mma_16816<BF16>(acc[mt], a0, a1, a2, a3, b0, b1);
                }
              }
            }
          }
        }
      }
    }
    __syncthreads();  // the next chunk overwrites xs
  }
  if (cur_g >= 0) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      tot[mt][0] = fmaf(s_lo, acc[mt][0], tot[mt][0]);
      tot[mt][1] = fmaf(s_lo, acc[mt][1], tot[mt][1]);
      tot[mt][2] = fmaf(s_hi, acc[mt][2], tot[mt][2]);
      tot[mt][3] = fmaf(s_hi, acc[mt][3], tot[mt][3]);
    }
  }

  // ---- partial tile to shared memory: red[wk][col][m] --------------------------
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

  // ---- cluster reduction over the S CTAs that share this column block ----------
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  {
    const int total = p.M * NCOL;
    const int o0 = (int)((long long)srank * total / S);
    const int o1 = (int)((long long)(srank + 1) * total / S);
    for (int o = o0 + tid; o < o1; o += DEC_THREADS) {
      const int m = o / NCOL, col = o % NCOL;
      const int n = blockIdx.x * NCOL + col;
      if (n >= p.N) continue;
      float sum = 0.f;
      for (int r = 0; r < S; ++r) {
        const float* peer = cluster.map_shared_rank(red, r);
        for (int q = 0; q < WK; ++q) sum += peer[((size_t)q * NCOL + col) * MR + m];
      }
      p.y[(size_t)m * p.N + n] = float_to_half_bits<BF16>(sum);
    }
  }
  cluster.sync();
}

template <int MT, bool BF16, bool G32>
void* kernel_ptr() {
  return reinterpret_cast<void*>(&w4a16_decode_kernel<MT, BF16, G32>);
}

void* pick_kernel(int MT, bool bf16, bool g32) {
#define W4_PICK(mt)                                                                     \
  if (MT == mt) {                                                                       \
    if (bf16) return g32 ? kernel_ptr<mt, true, true>() : kernel_ptr<mt, true, false>(); \
    return g32 ? kernel_ptr<mt, false, true>() : kernel_ptr<mt, false, false>();        \
  }
  W4_PICK(1)
  W4_PICK(2)
  W4_PICK(4)
  W4_PICK(8)
#undef W4_PICK
  return nullptr;
}

// Largest per-CTA K range (rows) whose x slice fits the shared-memory budget.
int max_rows_per_cta(int MT) {
  const int budget = 96 * 1024;  // x slice bytes; leaves room for 2 CTAs per SM
  int rows = budget / (8 * MT * 2);
  return std::max(ATOM_K, (rows / ATOM_K) * ATOM_K);
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

struct DecodePlan {
  int WN, S;
};

// Choose warps-along-N and the split-K factor: fill the GPU's CTA slots as
// evenly as possible while keeping each warp's run long enough to pipeline.
DecodePlan plan_decode(int N, int K, int MT, int sm_count) {
  const int NT = N / 16, A = K / ATOM_K;
  const int slots = 2 * sm_count;
  DecodePlan best{8, 1};
  double best_score = -1.0;
  for (int WN = 8; WN >= 1; WN >>= 1) {
    const int WK = DEC_WARPS / WN;
    const int cols = (NT + WN - 1) / WN;
    for (int S = 1; S <= MAX_SPLIT; ++S) {
      if (S > A) break;
      const long long ctas = (long long)cols * S;
      const int per_warp = A / (S * WK);
      if (per_warp < 1) continue;
      const long long waves = (ctas + slots - 1) / slots;
      double eff = (double)ctas / (double)(waves * slots);
      // idle warps when the column count does not fill WN
      eff *= (double)NT / (double)(cols * WN);
      // short runs cannot keep enough loads in flight
      const double pipe = std::min(1.0, per_warp / 6.0);
      const double score = eff * (0.5 + 0.5 * pipe) - 0.002 * S - 0.001 * (8 / WN);
      if (score > best_score) {
        best_score = score;
        best = {WN, S};
      }
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_decode(const GemmArgs& a, cudaStream_t stream) {
  DeviceInfo info;
  cudaError_t err = device_info(&info);
  if (err != cudaSuccess) return err;
  const bool g32 = (a.group % 64) != 0;
  for (int r0 = 0; r0 < a.M; r0 += 64) {
    const int Mc = std::min(64, a.M - r0);
    const int MT = Mc <= 8 ? 1 : Mc <= 16 ? 2 : Mc <= 32 ? 4 : 8;
    const DecodePlan plan = plan_decode(a.N, a.K, MT, info.sm_count);
    const int A = a.K / ATOM_K;
    const int cta_atoms = (A + plan.S - 1) / plan.S;
    const int chunk_atoms = std::min(cta_atoms, max_rows_per_cta(MT) / ATOM_K);
    const int x_stride = chunk_atoms * ATOM_K + 32;  // halves; row stride = 64 mod 128 bytes
    const size_t smem = (size_t)8 * MT * x_stride * 2 + (size_t)DEC_WARPS * 16 * 8 * MT * 4;
    void* fn = pick_kernel(MT, a.bf16 != 0, g32);
    err = ensure_smem(fn, smem);
    if (err != cudaSuccess) return err;

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
    p.group = a.group;
    p.A = A;
    p.WN = plan.WN;
    p.chunk_atoms = chunk_atoms;
    p.x_stride = x_stride;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.N / 16 + plan.WN - 1) / plan.WN, plan.S, 1);
    cfg.blockDim = dim3(DEC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = plan.S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    err = cudaLaunchKernelExC(&cfg, fn, args);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace w4
