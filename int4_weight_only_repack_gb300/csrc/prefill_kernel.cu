// Large-M (prefill) W4A16 GEMM on the 5th-generation tensor cores (tcgen05).
//
// Prefill is bound by tensor-core throughput ("vLLM 学习手册 01. 量化" §1:
// the prefill phase is compute-bound), so the weight stream is turned into
// UMMA operands as fast as the tensor cores consume them ("vLLM 学习手册 01.
// 量化" §5.3: dequantisation fused with the multiply; "vLLM AWQ 4-bit 量化实践"
// §5.3: W = (b - zeros) * scales):
//
//  * Persistent kernel, one CTA per SM, CTA tile 128 or 256 (M) x 256 (N), K
//    blocks of 64. Tiles are walked with M fastest so neighbouring CTAs share a
//    weight column block in L2. When the output tiles cannot fill the SMs, K is
//    split into slices whose fp32 partials a second kernel sums.
//  * Grouped (MoE) calls: one launch over all experts. Each CTA builds a table
//    of the experts' tiles from the row offsets on the device; a tile maps to
//    (expert, row block, column block), reads that expert's weights and masks
//    rows at the expert's end.
//  * Warp roles (16 warps): warp 0 issues TMA copies (x tile with the 128-byte
//    swizzle, the packed weight atoms, scales and zeros) into a 3-stage ring;
//    warps 8-15 dequantise the packed atoms into the bf16/fp16 B operand,
//    written directly in the K-major 128-byte-swizzled layout UMMA reads (one
//    16-byte store per packed word); warp 1 issues the UMMAs from one thread
//    into a TMEM accumulator; warps 4-7 drain the accumulator (tcgen05.ld),
//    round to the activation dtype and store y. Warp 2 owns the TMEM
//    allocation. The accumulator is double-buffered (2 x 256 TMEM columns) so
//    the epilogue of one tile overlaps the main loop of the next.
//  * Every wait on an mbarrier is bounded: after one second the CTA raises an
//    abort flag, records W4_ERR_TIMEOUT in the library's device status word,
//    lets its copies and UMMAs drain (again bounded), frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "sm100_ptx.cuh"
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace w4 {

// Non-zero once a kernel of this library gave up on a wait (see w4_device_status).
__device__ int g_device_status = 0;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_tile_box(CUtensorMap* map, const void* qw, int K, uint64_t NG, uint32_t box_tiles,
                     uint32_t box_atoms, uint32_t box_groups) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t A = (cuuint64_t)K / 64;
  const cuuint64_t dims[4] = {128, 8, A, NG};
  const cuuint64_t strides[3] = {512, 8 * 512, A * 8 * 512};
  const cuuint32_t box[4] = {128, box_tiles, box_atoms, box_groups};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(qw), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

using namespace sm100;

// NACC accumulators of 128 rows share each dequantised B tile: the CTA tile is
// (128 * NACC) x 256. NACC = 1 double-buffers the accumulator in TMEM (epilogue
// overlaps the next tile); NACC = 2 fills TMEM with the two accumulators and
// halves the dequantisation work per MMA.
constexpr int BN = 256, BK = 64;
// warps 0-3: TMA, MMA issue, TMEM allocation, second TMA issuer; 4-7: epilogue;
// 8 onward: dequantisation (Cfg::DEQ_WARPS of them)
constexpr int EPI_THREADS = 128;  // warps 4-7
constexpr int B_BYTES = BN * BK * 2;
constexpr int P_BYTES = BN * BK / 2;
constexpr int S_BYTES = 2 * BN * 2;   // two group rows of scales
constexpr int Z_BYTES = 2 * BN / 2;   // two group rows of zeros
constexpr int Z_SLOT = 1024;
constexpr int TMEM_COLS = 512;

// Two rings: ST_T stages that TMA fills (the x tile, the packed block, two
// group rows of scales and of zeros) and ST_B dequantised B tiles. A TMA stage
// is free again once the MMAs that read its x tile have completed, a B tile
// once the MMAs that read it have; the dequantising warps need a full TMA stage
// and a free B tile. Keeping B out of the TMA ring lets that ring run deeper
// where shared memory allows (a slot's round trip - load, dequantise, MMA - is
// about 2 us on GB300, so with 3 slots the pipeline, not the MMA, set the pace
// below M = 128). HALF_A: calls of at most 64 rows load 64 rows of x per stage;
// the MMA still reads 128 rows, the last 64 from whatever follows in shared
// memory, and those accumulator rows are never stored.
template <int NACC, bool GROUPED, bool HALF_A>
struct Cfg {
  static constexpr int BM = 128 * NACC;
  static constexpr int NBUF = NACC == 1 ? 2 : 1;  // accumulator buffers in TMEM
  static constexpr int A_ROWS = HALF_A ? 64 : BM;  // rows of x the TMA loads per stage
  static constexpr int A_BYTES = A_ROWS * BK * 2;
  static constexpr int ST_T = NACC == 2 ? 3 : GROUPED ? 3 : HALF_A ? 6 : 4;
  static constexpr int ST_B = 3;
  // Dequantising warps (8 onward), one or two of a B tile's 16 atoms each.
  // Ungrouped 128-row tiles get sixteen, one atom each: the MMA does half a
  // 256-row tile's work per dequantised B tile, so the dequantisation sets
  // their pace (measured on GB300: Llama-2-70B layers at M = 32 / 64 2-4 %
  // faster, at M = 128 gate_up 183 -> 175 us and down 90 -> 86 us, Llama-2-7B
  // o_proj / down at M = 512 2 %; 72-76 registers at 768 threads, no spills).
  // Grouped (MoE) 128-row tiles keep eight: with sixteen, a Mixtral-8x7B-shaped
  // layer at 41-109 rows an expert ran about 6 % slower (w13 298 -> 316 us,
  // w2 176 -> 187 us).
  static constexpr int DEQ_WARPS = (HALF_A || (NACC == 1 && !GROUPED)) ? 16 : 8;
  static constexpr int NTHREADS = 256 + 32 * DEQ_WARPS;
  // Threads that issue the TMA ring's loads. One issuing thread starts the
  // loads of a 256-row stage (x tile of 256 rows, packed block, scale and zero
  // rows) more slowly than the MMAs consume them (measured on GB300: 0.9 us a
  // stage against 0.55 us of MMA; two threads: Llama-2-70B gate_up at
  // M = 1024 659 -> 625 us; a third, splitting the x tile, gained nothing);
  // the 128-row pipeline is not bound by it.
  static constexpr int ISSUERS = NACC == 2 ? 2 : 1;
  static constexpr uint32_t STAGE_TX = A_BYTES + P_BYTES + S_BYTES + Z_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_P = OFF_A + ST_T * A_BYTES;
  static constexpr int OFF_S = OFF_P + ST_T * P_BYTES;
  static constexpr int OFF_Z = OFF_S + ST_T * S_BYTES;
  static constexpr int OFF_B = OFF_Z + ST_T * Z_SLOT;  // 1024-byte aligned
  static constexpr int OFF_BAR = OFF_B + ST_B * B_BYTES;
  static constexpr int NUM_BARS = 2 * ST_T + 2 * ST_B + 2 * NBUF + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base to 1024
  static_assert(OFF_B % 1024 == 0, "swizzled B tiles start on 1024 bytes");
  static_assert(!HALF_A || (NACC == 1 && !GROUPED), "64-row x tiles: ungrouped 128-row tiles only");
};

constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s per wait

struct PrefillParams {
  CUtensorMap tm_a;  // x [M][K], box 64 x 128, 128-byte swizzle
  CUtensorMap tm_p;  // TILE words as [N/128][K/64][8][128], box 128 x 8 x 1 x 2
  CUtensorMap tm_s;  // scales [G][N], box 256 x 2
  CUtensorMap tm_z;  // zeros [G][N/8], box 32 x 2
  uint16_t* y;
  const uint16_t* bias;  // [N] in the activation dtype, or nullptr
  int M, N, K, group;
  int m_blocks, n_blocks, num_tiles, k_blocks;
  // Split K (ungrouped): the tiles from tail_start on run as tail_split K
  // slices each, whose fp32 partial tiles go to tail_part
  // [tail_split][tail_tiles][tail_rows][BN] (slice-major; tail_rows = min(M, BM),
  // rows at or beyond M are not stored) for tail_reduce_kernel. Either every
  // tile (tail_start = 0: the tiles cannot fill the SMs) or the few beyond
  // whole waves that would leave most SMs idle in a last wave of their own.
  float* tail_part;
  int tail_start, tail_tiles, tail_split, tail_rows;
  // Grouped (MoE) calls: eoff != nullptr. x and y hold the rows of all experts,
  // sorted by expert ([eoff[e], eoff[e+1]) for expert e); tm_p spans the
  // experts' TILE buffers one after another (ng128 column groups each), tm_s
  // and tm_z their [E * groups] group rows. M is then the most rows an expert
  // may have, and the tile count comes from the offsets on the device.
  const int32_t* eoff;
  int num_experts, groups, ng128, total_rows;
  int stall;  // test hook: the producers issue nothing (every wait on the ring runs out)
};

// Per-CTA table of a grouped call, after the pipeline's shared memory:
// tile0[E + 1] (first work unit of each expert; tile0[E] = all units), then
// the first row r0[E] and the end row r1[E] of each expert.
__host__ __device__ constexpr int grouped_table_bytes(int E) { return (12 * (E + 1) + 15) & ~15; }
// Experts one launch takes: with 128-row tiles, and with 256-row tiles (less
// shared memory left beside that pipeline).
constexpr int GROUPED_MAX_EXPERTS = 4096;
constexpr int GROUPED_MAX_EXPERTS_256 = 256;
static_assert(Cfg<1, true, false>::SMEM_BYTES + grouped_table_bytes(GROUPED_MAX_EXPERTS) <=
                  227 * 1024,
              "the grouped tile table must fit beside the 128-row pipeline");
static_assert(Cfg<2, true, false>::SMEM_BYTES + grouped_table_bytes(GROUPED_MAX_EXPERTS_256) <=
                  227 * 1024,
              "the grouped tile table must fit beside the 256-row pipeline");
static_assert(Cfg<1, false, false>::SMEM_BYTES <= 227 * 1024 &&
                  Cfg<1, false, true>::SMEM_BYTES <= 227 * 1024 &&
                  Cfg<2, false, false>::SMEM_BYTES <= 227 * 1024,
              "the pipelines fit in shared memory");

// Work unit `tile` -> (expert, M block, N block, K slice [kb0, kb1) of
// k-blocks, first row and end row of the unit's rows). Ungrouped units run M
// fastest, then N; the split tiles' units after the whole tiles, slice by
// slice. Grouped ones run expert by expert, M fastest within the expert, then
// N (no K split).
struct Unit {
  int e, m_blk, n_blk, ks, kb0, kb1, row0, row_end;
  int slot;  // partial-tile slot of a split unit in tail_part, else -1
};
template <bool GROUPED>
__device__ __forceinline__ Unit unit_of(const PrefillParams& p, const int* tab, int BM, int tile) {
  Unit u;
  if (!GROUPED) {
    u.e = 0;
    u.slot = -1;
    if (p.tail_split > 1 && tile >= p.tail_start) {
      // a split unit: slice v / tail_tiles of tile tail_start + v % tail_tiles
      const int v = tile - p.tail_start;
      const int tt = p.tail_start + v % p.tail_tiles;
      u.m_blk = tt % p.m_blocks;
      u.n_blk = tt / p.m_blocks;
      u.ks = v / p.tail_tiles;
      u.kb0 = (int)((long long)u.ks * p.k_blocks / p.tail_split);
      u.kb1 = (int)((long long)(u.ks + 1) * p.k_blocks / p.tail_split);
      u.slot = v;
    } else {
      u.m_blk = tile % p.m_blocks;
      u.n_blk = tile / p.m_blocks;
      u.ks = 0;
      u.kb0 = 0;
      u.kb1 = p.k_blocks;
    }
    u.row0 = u.m_blk * BM;
    u.row_end = p.M;
    return u;
  }
  // the last expert whose first unit is at or before `tile` (experts with no
  // units share their tile0 with the next one and are passed over)
  const int E = p.num_experts;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid] <= tile) lo = mid;
    else hi = mid;
  }
  const int* r0 = tab + (E + 1);
  const int* r1 = r0 + E;
  const int local = tile - tab[lo];
  const int mb = (r1[lo] - r0[lo] + BM - 1) / BM;
  u.e = lo;
  u.slot = -1;
  u.m_blk = local % mb;
  u.n_blk = local / mb;
  u.ks = 0;
  u.kb0 = 0;
  u.kb1 = p.k_blocks;
  u.row0 = r0[lo] + u.m_blk * BM;
  u.row_end = r1[lo];
  return u;
}

// full / empty: the TMA ring; bready / bfree: the B ring; accfull / accempty:
// the TMEM accumulators; mmadone: the abort path's last commit.
template <int ST_T, int ST_B, int NBUF>
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8 * s; }
  __device__ uint32_t empty(int s) const { return base + 8 * (ST_T + s); }
  __device__ uint32_t bready(int b) const { return base + 8 * (2 * ST_T + b); }
  __device__ uint32_t bfree(int b) const { return base + 8 * (2 * ST_T + ST_B + b); }
  __device__ uint32_t accfull(int b) const { return base + 8 * (2 * ST_T + 2 * ST_B + b); }
  __device__ uint32_t accempty(int b) const {
    return base + 8 * (2 * ST_T + 2 * ST_B + NBUF + b);
  }
  __device__ uint32_t mmadone() const { return base + 8 * (2 * ST_T + 2 * ST_B + 2 * NBUF); }
};

// Wait for an mbarrier phase. Returns false when this CTA is aborting: either
// another role raised the flag, or this wait ran past the limit (then it
// raises the flag and records the timeout).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      atomicExch(&g_device_status, W4_ERR_TIMEOUT);
      return false;
    }
  }
}

// Bounded drain wait used on the abort path only.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi, bool bf16) {
  uint32_t d;
  if (bf16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  }
  return d;
}

// GROUPED: a grouped (MoE) call, p.eoff != nullptr (its own instantiation, so
// that ungrouped calls carry none of its per-tile work).
template <bool BF16, int NACC, bool GROUPED, bool HALF_A>
__global__ void __launch_bounds__(Cfg<NACC, GROUPED, HALF_A>::NTHREADS, 1)
    w4a16_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = Cfg<NACC, GROUPED, HALF_A>;
  constexpr int DEQ_WARPS = C::DEQ_WARPS, NTHREADS = C::NTHREADS;
  constexpr int ATOMS_PER_WARP = 16 / DEQ_WARPS;
  constexpr int BM = C::BM, NBUF = C::NBUF, A_BYTES = C::A_BYTES;
  constexpr int ST_T = C::ST_T, ST_B = C::ST_B, ISSUERS = C::ISSUERS;
  constexpr int OFF_A = C::OFF_A, OFF_B = C::OFF_B, OFF_P = C::OFF_P, OFF_S = C::OFF_S;
  constexpr int OFF_Z = C::OFF_Z, OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC;
  constexpr uint32_t STAGE_TX = C::STAGE_TX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Bars<ST_T, ST_B, NBUF> bars{sbase + OFF_BAR};
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  // Launched with programmatic stream serialization: wait for the previous
  // kernel in the stream before touching global memory, then let the next one
  // start its launch.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (tid == 0) {
    for (int s = 0; s < ST_T; ++s) {
      mbar_init(bars.full(s), ISSUERS);
      mbar_init(bars.empty(s), 1);
    }
    for (int b = 0; b < ST_B; ++b) {
      mbar_init(bars.bready(b), 32 * DEQ_WARPS);
      mbar_init(bars.bfree(b), 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(bars.accfull(b), 1);
      mbar_init(bars.accempty(b), EPI_THREADS);
    }
    mbar_init(bars.mmadone(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  int* tab = reinterpret_cast<int*>(smem + C::SMEM_USED);
  if (GROUPED) {
    // grouped call: the experts' row offsets (they may come from the kernel
    // before this one), staged in tile0[] by all threads in one pass
    for (int e = tid; e <= p.num_experts; e += NTHREADS)
      tab[e] = *reinterpret_cast<const volatile int32_t*>(p.eoff + e);
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_a);
    prefetch_tmap(&p.tm_p);
    prefetch_tmap(&p.tm_s);
    prefetch_tmap(&p.tm_z);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (GROUPED) {
    if (warp == 3) {
      // Each expert's rows and its first work unit. First every lane checks
      // its experts' ranges from the staged offsets: an invalid range or one
      // longer than M records W4_ERR_EXPERT_ROWS and gets no rows (its rows of
      // y stay unwritten). Then a prefix sum over the experts, 32 at a time,
      // overwrites the staged offsets with the first unit of each expert.
      const int E = p.num_experts;
      int* r0 = tab + (E + 1);
      int* r1 = r0 + E;
      bool bad = false;
      for (int e = lane; e < E; e += 32) {
        const int a = tab[e], b = tab[e + 1];
        int rows = b - a;
        if (a < 0 || rows < 0 || b > p.total_rows || rows > p.M) {
          bad = true;
          rows = 0;
        }
        r0[e] = a;
        r1[e] = a + rows;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicExch(&g_device_status, W4_ERR_EXPERT_ROWS);
      __syncwarp();
      int carry = 0;
      for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int incl = e < E ? (r1[e] - r0[e] + C::BM - 1) / C::BM * p.n_blocks : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += v;
        }
        if (e < E) tab[e + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) tab[0] = 0;
    }
    __syncthreads();
  }
  const uint32_t tmem = *tmem_holder;
  const int num_tiles = GROUPED ? tab[p.num_experts] : p.num_tiles;

  // ------------------------------------------------------------------ producers
  // ISSUERS threads fill the TMA ring, each arming its own bytes of a stage:
  // one thread loads everything; with two, warp 0 loads the x tile and the
  // scale / zero rows and warp 3 the packed block.
  auto produce = [&](const int role) {
    if (p.stall) return;
    const uint32_t tx = ISSUERS == 1 ? STAGE_TX
                        : role == 0  ? STAGE_TX - P_BYTES
                                     : (uint32_t)P_BYTES;
    int it = 0;
    int last_armed[ST_T];
    for (int s = 0; s < ST_T; ++s) last_armed[s] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const Unit u = unit_of<GROUPED>(p, tab, BM, tile);
      const int n_blk = u.n_blk;
      for (int j = 0; j < u.kb1 - u.kb0; ++j, ++it) {
        const int kb = u.kb0 + j;
        const int s = it % ST_T;
        const uint32_t ph = (it / ST_T) & 1;
        if (!wait_phase(bars.empty(s), ph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bars.full(s), tx);
        last_armed[s] = it;
        // (a grouped call's unit reads its expert's rows of x, column groups
        // and group rows; rows past the expert's end are computed but not stored)
        const int grow = u.e * p.groups + (kb * BK) / p.group;
        if (role == 0) {
          tma_load_2d(sbase + OFF_A + s * A_BYTES, &p.tm_a, bars.full(s), kb * BK, u.row0);
          tma_load_2d(sbase + OFF_S + s * S_BYTES, &p.tm_s, bars.full(s), n_blk * BN, grow);
          tma_load_2d(sbase + OFF_Z + s * Z_SLOT, &p.tm_z, bars.full(s), n_blk * (BN / 8), grow);
        }
        if (ISSUERS == 1 || role == 1) {
          // the 16 atoms (two column groups) of this N block at k-atom kb
          tma_load_4d(sbase + OFF_P + s * P_BYTES, &p.tm_p, bars.full(s), 0, 0, kb,
                      u.e * p.ng128 + n_blk * (BN / 128));
        }
      }
    }
    if (!ok) {
      // let the copies already issued land before the CTA can exit
      for (int s = 0; s < ST_T; ++s)
        if (last_armed[s] >= 0) drain_phase(bars.full(s), (last_armed[s] / ST_T) & 1);
    }
  };
  if (warp == 0) {
    if (lane == 0) produce(0);
  } else if (warp == 3) {
    if (ISSUERS == 2 && lane == 0) produce(1);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_f16(BF16 ? 1 : 0, 128, BN);
      int it = 0, lt = 0;
      bool ok = true;
      bool issued = false;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++lt) {
        const int buf = lt % NBUF;
        const uint32_t aph = (lt / NBUF) & 1;
        if (!wait_phase(bars.accempty(buf), aph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * (BN * NACC);
        const Unit u = unit_of<GROUPED>(p, tab, BM, tile);
        // a grouped call's 256-row tile whose second half holds no rows (the
        // last rows of an expert) skips that accumulator's MMAs (the epilogue
        // still drains it, but every row it would store is masked)
        const bool second = NACC == 2 && (!GROUPED || u.row0 + 128 < u.row_end);
        for (int j = 0; j < u.kb1 - u.kb0; ++j, ++it) {
          const int s = it % ST_T, b = it % ST_B;
          const uint32_t ph = (it / ST_T) & 1, phb = (it / ST_B) & 1;
          if (!wait_phase(bars.full(s), ph, abort_flag) ||
              !wait_phase(bars.bready(b), phb, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc = smem_desc_k128(sbase + OFF_B + b * B_BYTES);
          // accumulator i: rows 128 i .. 128 i + 127 of the A tile; each MMA
          // advances 16 elements (32 bytes) along K inside the swizzled rows
          if (NACC == 1 || second) {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
#pragma unroll
              for (int i = 0; i < NACC; ++i) {
                const uint64_t adesc = smem_desc_k128(sbase + OFF_A + s * A_BYTES + i * (128 * BK * 2));
                umma_f16(d_tmem + i * BN, adesc + 2 * k, bdesc + 2 * k, IDESC, j != 0 || k != 0);
              }
            }
          } else {
            const uint64_t adesc = smem_desc_k128(sbase + OFF_A + s * A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, j != 0 || k != 0);
          }
          issued = true;
          umma_commit(bars.empty(s));  // the x tile (and the stage) is free again
          umma_commit(bars.bfree(b));  // and so is the B tile
        }
        if (ok) umma_commit(bars.accfull(buf));
      }
      if (!ok && issued) {
        umma_commit(bars.mmadone());
        drain_phase(bars.mmadone(), 0);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    int lt = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++lt) {
      const Unit u = unit_of<GROUPED>(p, tab, BM, tile);
      const int n_blk = u.n_blk;
      const int buf = lt % NBUF;
      const uint32_t aph = (lt / NBUF) & 1;
      if (!wait_phase(bars.accfull(buf), aph, abort_flag)) break;
      tc_fence_after();
#pragma unroll 1
      for (int i = 0; i < NACC; ++i) {
        const int m = u.row0 + i * 128 + quarter * 32 + lane;
        uint16_t* yrow = p.y + (size_t)m * p.N;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + buf * (BN * NACC) + i * BN + c0, r);
          tmem_ld_wait();
          const int n = n_blk * BN + c0;
          if (u.slot >= 0) {
            // split K: this slice's fp32 partial of the tile (N % 32 == 0: whole
            // 32-column chunks; m - row0 < tail_rows for every stored row)
            if (m < u.row_end && n < p.N) {
              float4* dst = reinterpret_cast<float4*>(
                  p.tail_part + ((size_t)u.slot * p.tail_rows + (m - u.row0)) * BN + c0);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                     __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            }
          } else if (m < u.row_end) {
            if (p.bias != nullptr) {
              // y = RN(acc + bias): the bias joins the fp32 sum before the one rounding
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (n + 8 * q < p.N) {
                  const uint4 b = __ldg(reinterpret_cast<const uint4*>(p.bias + n + 8 * q));
                  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                  for (int e = 0; e < 8; ++e)
                    r[8 * q + e] = __float_as_uint(
                        __uint_as_float(r[8 * q + e]) +
                        half_bits_to_float<BF16>((uint16_t)(bw[e >> 1] >> (16 * (e & 1)))));
                }
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (n + 8 * q < p.N) {
                uint4 v;
                v.x = pack_half2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]), BF16);
                v.y = pack_half2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]), BF16);
                v.z = pack_half2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]), BF16);
                v.w = pack_half2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]), BF16);
                *reinterpret_cast<uint4*>(yrow + n + 8 * q) = v;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bars.accempty(buf));
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------------- dequantise
    constexpr uint32_t MAGIC = Magic<BF16>::pair;
    const int wd = warp - 8;
    const int gg = lane >> 2, t = lane & 3;
    const bool odd = (gg & 1) != 0;
    const bool two_groups = p.group < BK;  // group 32: each K half has its own group row
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const Unit u = unit_of<GROUPED>(p, tab, BM, tile);
      for (int j = 0; j < u.kb1 - u.kb0; ++j, ++it) {
        const int s = it % ST_T, b = it % ST_B;
        const uint32_t ph = (it / ST_T) & 1, phb = (it / ST_B) & 1;
        if (!wait_phase(bars.full(s), ph, abort_flag) ||
            !wait_phase(bars.bfree(b), phb ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint16_t* sS = reinterpret_cast<const uint16_t*>(smem + OFF_S + s * S_BYTES);
        const uint32_t* sZ = reinterpret_cast<const uint32_t*>(smem + OFF_Z + s * Z_SLOT);
        const uint8_t* sP = smem + OFF_P + s * P_BYTES;
        uint8_t* sB = smem + OFF_B + b * B_BYTES;
        // the scale pairs (s | s << 16) and MAGIC + z pairs of this lane's four
        // columns (atoms wd + DEQ_WARPS r, rows gg and gg + 8), per K half when the
        // block holds two groups: read once per block, not per word
        uint32_t ss[ATOMS_PER_WARP][2][2], zz[ATOMS_PER_WARP][2][2];
#pragma unroll
        for (int r = 0; r < ATOMS_PER_WARP; ++r)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int n_loc = (wd + DEQ_WARPS * r) * 16 + gg + 8 * c;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (h == 1 && !two_groups) {
                ss[r][c][1] = ss[r][c][0];
                zz[r][c][1] = zz[r][c][0];
                continue;
              }
              const uint32_t sb = sS[h * BN + n_loc];
              const uint32_t z = (sZ[h * (BN / 8) + (n_loc >> 3)] >> (4 * (n_loc & 7))) & 0xF;
              ss[r][c][h] = sb | (sb << 16);
              zz[r][c][h] = MAGIC | z | (z << 16);
            }
          }
#pragma unroll
        for (int r = 0; r < ATOMS_PER_WARP; ++r) {
          const int at = wd + DEQ_WARPS * r;  // atom (16-column tile) inside the block
          const uint4 w = *reinterpret_cast<const uint4*>(sP + (at * 128 + 4 * lane) * 4);
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            // odd gg store the other K half first: the 8 lanes of each store
            // phase then hit 8 distinct 16-byte bank groups (word j = jj ^ 2 for
            // odd gg, picked with selects so every array index stays static)
            const uint32_t word = odd ? wv[jj ^ 2] : wv[jj];
            const int n_loc = at * 16 + gg + 8 * (jj & 1);
            const int h = (jj >> 1) ^ (odd ? 1 : 0);
            const uint32_t zzw = !two_groups ? zz[r][jj & 1][0]
                                 : odd       ? zz[r][jj & 1][(jj >> 1) ^ 1]
                                             : zz[r][jj & 1][jj >> 1];
            const uint32_t ssw = !two_groups ? ss[r][jj & 1][0]
                                 : odd       ? ss[r][jj & 1][(jj >> 1) ^ 1]
                                             : ss[r][jj & 1][jj >> 1];
            uint4 o;
            o.x = mul_x2<BF16>(sub_x2<BF16>(lop3_and_or(word, 0x000F000Fu, MAGIC), zzw), ssw);
            o.y = mul_x2<BF16>(sub_x2<BF16>(lop3_and_or(word >> 4, 0x000F000Fu, MAGIC), zzw), ssw);
            o.z = mul_x2<BF16>(sub_x2<BF16>(lop3_and_or(word >> 8, 0x000F000Fu, MAGIC), zzw), ssw);
            o.w = mul_x2<BF16>(sub_x2<BF16>(lop3_and_or(word >> 12, 0x000F000Fu, MAGIC), zzw), ssw);
            const int c = 4 * h + t;  // 16-byte chunk along K inside the 128-byte row
            const int off = (n_loc >> 3) * 1024 + (n_loc & 7) * 128 + ((c ^ (n_loc & 7)) << 4);
            *reinterpret_cast<uint4*>(sB + off) = o;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bars.bready(b));
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

// ---- act-order: x'[m][j] = x[m][perm[j]] --------------------------------------
// One thread: eight consecutive columns, for the rows blockIdx.y, blockIdx.y +
// gridDim.y, ... (grid: column blocks x up to 65535 rows). perm comes in as two
// 16-byte loads, the eight x values of a row as independent 2-byte loads, and
// they leave as one 16-byte store (K % 64 == 0, 16-byte aligned buffers).
__global__ void __launch_bounds__(256) gather_columns_kernel(const uint16_t* __restrict__ x,
                                                             const int32_t* __restrict__ perm,
                                                             uint16_t* __restrict__ xg, int M,
                                                             int K) {
  // launched with programmatic stream serialization: x may come from the kernel
  // before this one; the GEMM after it may start its weight prologue at once
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int c = blockIdx.x * 256 + threadIdx.x;  // eight-column chunk
  if (c >= K / 8) return;
  const int4* pp = reinterpret_cast<const int4*>(perm) + 2 * c;
  const int4 pa = __ldg(pp), pb = __ldg(pp + 1);
  for (size_t m = blockIdx.y; m < (size_t)M; m += gridDim.y) {
    const uint16_t* xr = x + m * K;
    uint4 v;
    v.x = __ldg(xr + pa.x) | ((uint32_t)__ldg(xr + pa.y) << 16);
    v.y = __ldg(xr + pa.z) | ((uint32_t)__ldg(xr + pa.w) << 16);
    v.z = __ldg(xr + pb.x) | ((uint32_t)__ldg(xr + pb.y) << 16);
    v.w = __ldg(xr + pb.z) | ((uint32_t)__ldg(xr + pb.w) << 16);
    reinterpret_cast<uint4*>(xg + m * K)[c] = v;
  }
}

// ---- split K: y = RN(sum over the slices + bias) for the split tiles --------------
// One thread per four consecutive outputs of a split tile (R = tail_rows rows of
// partials a tile); the slices are summed in order (deterministic).
template <bool BF16>
__global__ void __launch_bounds__(256) tail_reduce_kernel(const float4* __restrict__ part,
                                                          uint16_t* __restrict__ y,
                                                          const uint16_t* __restrict__ bias,
                                                          int M, int N, int BM, int R,
                                                          int m_blocks, int tail_start,
                                                          int tail_tiles, int tail_split) {
  const size_t per_tile = (size_t)R * (BN / 4);
  const size_t total = (size_t)tail_tiles * per_tile;
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (size_t)gridDim.x * 256) {
    const int ti = (int)(i / per_tile);
    const int rr = (int)((i - (size_t)ti * per_tile) / (BN / 4));
    const int c4 = (int)(i % (BN / 4));
    const int tt = tail_start + ti;
    const int m = (tt % m_blocks) * BM + rr;
    const int n = (tt / m_blocks) * BN + 4 * c4;
    if (m >= M || n >= N) continue;
    float4 a = part[i];
    for (int sl = 1; sl < tail_split; ++sl) {
      const float4 b = part[(size_t)sl * total + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if (bias != nullptr) {
      a.x += half_bits_to_float<BF16>(bias[n]);
      a.y += half_bits_to_float<BF16>(bias[n + 1]);
      a.z += half_bits_to_float<BF16>(bias[n + 2]);
      a.w += half_bits_to_float<BF16>(bias[n + 3]);
    }
    *reinterpret_cast<uint2*>(y + (size_t)m * N + n) =
        make_uint2(pack_half2(a.x, a.y, BF16), pack_half2(a.z, a.w, BF16));
  }
}

// ---- host side ------------------------------------------------------------------
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
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

// TILE words viewed as [column group][k-atom][tile in group][word] (NG column
// groups): one box is the 8 atoms of `box_groups` consecutive column groups at
// one k-atom.
bool encode_tile_4d(CUtensorMap* map, const void* qw, int K, uint64_t NG, uint32_t box_groups) {
  return encode_tile_box(map, qw, K, NG, 8, 1, box_groups);
}

cudaError_t ensure_prefill_smem(void* fn, int which, int bytes) {
  static std::mutex mu;
  static bool done[64][10] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && done[dev][which]) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done[dev][which] = true;
  return e;
}

// Tiling and K split of a call, chosen by an estimate of its time. A CTA
// computes one 128 x 256 tile (NACC = 1) or one 256 x 256 tile (NACC = 2: it
// dequantises each B tile once for both accumulators). One SM's measured rate
// on GB300 is about 5.8 TFLOP/s with 128-row tiles and 8.7 with 256-row ones,
// over a long K. Tiles beyond whole waves (all of them when they cannot fill
// the SMs) may be split into K slices of at least 8 k-blocks, each slice's
// fp32 partial tile written out and summed by tail_reduce_kernel. The estimate
// of a split: ceil(split tiles * slices / SMs) waves of 1/slices of a tile's
// time, every wave plus about 4 k-blocks of pipeline fill and drain, plus
// writing and reading the partials (8 bytes an output a slice at about
// 6.6 TB/s) and the reduce launch (about 3 us). Among the splits, one wave's
// worth (as many slices as the SMs hold, when the tiles cannot fill them) or
// none (for the tiles of a last wave) is kept unless another is estimated at
// least 10 % faster. Measured on GB300 against the former fixed choices:
// Llama-2-70B gate_up at M = 128 175 -> 142 us (its last wave split), 7B down
// at M = 512 70 -> 62 us (256-row tiles split 3-4 ways), 70B qkv at M = 1024
// 211 -> 133 us and 7B gate_up at M = 512 116 -> 85 us (the last wave split).
struct PrefillPlan {
  int nacc, m_blocks, n_blocks;
  int tail_tiles, tail_split;  // split K (tail_split > 1): the last tail_tiles tiles and their slices
  double seconds;              // the estimate
};

PrefillPlan plan_tiles(int M, int N, int K, int sm_count, int nacc) {
  PrefillPlan pl;
  pl.nacc = nacc;
  pl.n_blocks = (N + BN - 1) / BN;
  pl.m_blocks = (M + 128 * nacc - 1) / (128 * nacc);
  pl.tail_tiles = 0;
  pl.tail_split = 1;
  const long long tiles = (long long)pl.m_blocks * pl.n_blocks;
  const int kb_total = K / BK;
  const int kmax = std::max(1, kb_total / 8);
  const double tile_s = 2.0 * 128 * nacc * BN * (double)K / (nacc == 2 ? 8.7e12 : 5.8e12);
  const double fill = 4.0 / kb_total;
  const long long full = tiles / sm_count;
  const long long rem = tiles - full * sm_count;
  const double whole = (double)full * tile_s * (1.0 + fill);
  pl.seconds = whole;
  if (rem == 0) return pl;
  // partial bytes of one slice of the rem tiles: their stored rows x BN x 8
  const double rows = (double)std::min<long long>(M, 128LL * nacc * pl.m_blocks) / pl.m_blocks;
  const double slice_s = 8.0 * (double)rem * rows * BN / 6.6e12;
  auto cost = [&](int ks) {
    const double waves = (double)((rem * ks + sm_count - 1) / sm_count);
    return waves * tile_s * (1.0 / ks + fill) + (ks > 1 ? slice_s * ks + 3e-6 : 0.0);
  };
  const int base = full == 0 ? (int)std::max(1LL, std::min<long long>(kmax, sm_count / rem)) : 1;
  int best = base;
  for (int ks = 1; ks <= kmax; ++ks)
    if (cost(ks) < cost(best)) best = ks;
  const int ks = cost(best) < 0.9 * cost(base) ? best : base;
  if (ks > 1) {
    pl.tail_tiles = (int)rem;
    pl.tail_split = ks;
  }
  pl.seconds = whole + cost(ks);
  return pl;
}

PrefillPlan prefill_plan(int M, int N, int K, int sm_count) {
  PrefillPlan pl = plan_tiles(M, N, K, sm_count, 1);
  if (M > 128) {
    const PrefillPlan p2 = plan_tiles(M, N, K, sm_count, 2);
    if (p2.seconds < pl.seconds) pl = p2;
  }
  return pl;
}

// fp32 partials of a plan's split tiles (rows at or beyond M are not stored)
size_t tail_bytes(const PrefillPlan& pl, int M) {
  const size_t rows = (size_t)std::min(M, 128 * pl.nacc);
  return pl.tail_split > 1 ? (size_t)pl.tail_split * pl.tail_tiles * rows * BN * 4 : 0;
}

}  // namespace

cudaError_t launch_gather_columns(const void* x, const int32_t* perm, void* xg, int M, int K,
                                  cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((K / 8 + 255) / 256), (unsigned)std::min(M, 65535), 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint16_t* xd = static_cast<uint16_t*>(xg);
  return cudaLaunchKernelEx(&cfg, gather_columns_kernel, xs, perm, xd, M, K);
}

size_t prefill_workspace_bytes(int M, int K, bool has_perm) {
  if (!has_perm) return 0;
  return ((size_t)M * K * 2 + 255) & ~(size_t)255;
}

void prefill_plan_query(int M, int N, int K, int sm_count, int* out) {
  const PrefillPlan pl = prefill_plan(M, N, K, sm_count);
  out[0] = 128 * pl.nacc;
  out[1] = pl.m_blocks * pl.n_blocks;
  out[2] = pl.tail_split > 1 ? pl.tail_tiles : 0;
  out[3] = pl.tail_split;
}

size_t prefill_split_workspace_bytes(int M, int N, int K) {
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return 0;
  return tail_bytes(prefill_plan(M, N, K, info.sm_count), M);
}

bool prefill_supported(int M, int N, int K) {
  return M > 0 && N % 32 == 0 && K % BK == 0;
}

bool grouped_prefill_supported(int N, int K, int num_experts) {
  return N % 32 == 0 && K % BK == 0 && num_experts >= 1 && num_experts <= GROUPED_MAX_EXPERTS;
}

bool use_prefill(int M, int N, int K, int sm_count) {
  (void)sm_count;
  return M > 16 && prefill_supported(M, N, K);
}

cudaError_t launch_prefill(const GemmArgs& a, cudaStream_t stream) {
  DeviceInfo info;
  cudaError_t err = device_info(&info);
  if (err != cudaSuccess) return err;
  const void* x = a.x;
  if (a.perm) {
    if ((err = launch_gather_columns(a.x, a.perm, a.workspace, a.M, a.K, stream)) != cudaSuccess)
      return err;
    x = a.workspace;
  }
  const bool grouped = a.eoff != nullptr;
  PrefillPlan pl;
  if (grouped) {
    // experts: no K split (the units come from the offsets, which only the
    // device reads). 256-row tiles when an expert may have more than 128 rows
    // and the experts' table fits beside that pipeline: an expert's last tile
    // skips its second accumulator when it holds no more than 128 rows, so
    // they never do more MMA work than 128-row tiles, and they dequantise each
    // B tile once for 256 rows. When every expert fits one 128-row tile, the
    // 128-row pipeline is faster: it double-buffers the accumulator and loads
    // half the x tile (measured on GB300 over a Mixtral-8x7B-shaped layer,
    // 23-75 rows per expert: 10-12 % faster; 115-143 rows: the 256-row tiles
    // 18-38 % faster).
    pl.nacc = (a.M > 128 && a.num_experts <= GROUPED_MAX_EXPERTS_256) ? 2 : 1;
    pl.n_blocks = (a.N + BN - 1) / BN;
    pl.m_blocks = 0;
    pl.tail_tiles = 0;
    pl.tail_split = 1;
    pl.seconds = 0.0;
  } else {
    pl = prefill_plan(a.M, a.N, a.K, info.sm_count);
  }
  // the split-K partials go after the act-order staging, when the workspace
  // has room for them; with less room the split shrinks (down to none)
  const size_t staged = prefill_workspace_bytes(a.M, a.K, a.perm != nullptr);
  const size_t room = a.workspace_bytes > staged ? a.workspace_bytes - staged : 0;
  while (pl.tail_split > 1 && (a.workspace == nullptr || tail_bytes(pl, a.M) > room))
    --pl.tail_split;
  const int nacc = pl.nacc;
  const int BM = 128 * nacc;
  // 64-row x tiles (and a deeper TMA ring) for ungrouped calls of at most 64 rows
  const bool half_a = !grouped && nacc == 1 && a.M <= 64;
  const int n_blocks = pl.n_blocks;
  PrefillParams p;
  const int G = a.K / a.group;
  const int E = grouped ? a.num_experts : 1;
  const int x_rows = grouped ? a.total_rows : a.M;
  const int ng128 = (a.N + 127) / 128;
  const CUtensorMapDataType act = a.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  bool ok = encode_2d(&p.tm_a, act, x, a.K, x_rows, (uint64_t)a.K * 2, BK, half_a ? 64 : BM,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  // stacked experts are further column groups of one TILE tensor, and further
  // group rows of the scales and zeros
  ok = ok && encode_tile_4d(&p.tm_p, a.qw, a.K, (uint64_t)E * ng128, BN / 128);
  ok = ok && encode_2d(&p.tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, a.N, (uint64_t)E * G,
                       (uint64_t)a.N * 2, BN, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && encode_2d(&p.tm_z, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.zeros, a.N / 8, (uint64_t)E * G,
                       (uint64_t)a.N / 2, BN / 8, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  p.y = static_cast<uint16_t*>(a.y);
  p.bias = static_cast<const uint16_t*>(a.bias);
  p.tail_part = pl.tail_split > 1
                    ? reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + staged)
                    : nullptr;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.group = a.group;
  p.m_blocks = (a.M + BM - 1) / BM;
  p.n_blocks = n_blocks;
  p.num_tiles = p.m_blocks * n_blocks;
  p.tail_split = pl.tail_split;
  p.tail_tiles = pl.tail_split > 1 ? pl.tail_tiles : 0;
  p.tail_start = p.num_tiles - p.tail_tiles;
  p.tail_rows = std::min(a.M, BM);
  if (pl.tail_split > 1) p.num_tiles = p.tail_start + pl.tail_tiles * pl.tail_split;
  p.k_blocks = a.K / BK;
  p.eoff = a.eoff;
  p.num_experts = E;
  p.groups = G;
  p.ng128 = ng128;
  p.total_rows = x_rows;
  p.stall = a.test_stall;
  // CTAs: one per SM at most; a grouped call has at most
  // (total_rows / 128 + E) row tiles over the N blocks
  const long long max_units =
      grouped ? (long long)n_blocks * ((x_rows + BM - 1) / BM + E) : (long long)p.num_tiles;

  // [variant][bf16]: 0 ungrouped 128-row, 1 ungrouped 128-row with 64-row x
  // tiles, 2 ungrouped 256-row, 3 grouped 128-row, 4 grouped 256-row
  static void* const kernels[5][2] = {
      {reinterpret_cast<void*>(&w4a16_prefill_kernel<false, 1, false, false>),
       reinterpret_cast<void*>(&w4a16_prefill_kernel<true, 1, false, false>)},
      {reinterpret_cast<void*>(&w4a16_prefill_kernel<false, 1, false, true>),
       reinterpret_cast<void*>(&w4a16_prefill_kernel<true, 1, false, true>)},
      {reinterpret_cast<void*>(&w4a16_prefill_kernel<false, 2, false, false>),
       reinterpret_cast<void*>(&w4a16_prefill_kernel<true, 2, false, false>)},
      {reinterpret_cast<void*>(&w4a16_prefill_kernel<false, 1, true, false>),
       reinterpret_cast<void*>(&w4a16_prefill_kernel<true, 1, true, false>)},
      {reinterpret_cast<void*>(&w4a16_prefill_kernel<false, 2, true, false>),
       reinterpret_cast<void*>(&w4a16_prefill_kernel<true, 2, true, false>)}};
  const int variant = grouped ? (nacc == 2 ? 4 : 3) : (nacc == 2 ? 2 : half_a ? 1 : 0);
  void* fn = kernels[variant][a.bf16 ? 1 : 0];
  static const int cfg_bytes[5] = {Cfg<1, false, false>::SMEM_BYTES, Cfg<1, false, true>::SMEM_BYTES,
                                   Cfg<2, false, false>::SMEM_BYTES, Cfg<1, true, false>::SMEM_BYTES,
                                   Cfg<2, true, false>::SMEM_BYTES};
  const int table_max = variant == 3 ? grouped_table_bytes(GROUPED_MAX_EXPERTS)
                        : variant == 4 ? grouped_table_bytes(GROUPED_MAX_EXPERTS_256)
                                       : 0;
  const int smem_bytes = cfg_bytes[variant] + (grouped ? grouped_table_bytes(E) : 0);
  const int smem_max = cfg_bytes[variant] + table_max;
  const int which = (a.bf16 ? 1 : 0) + 2 * variant;
  if ((err = ensure_prefill_smem(fn, which, smem_max)) != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<long long>(max_units, info.sm_count), 1, 1);
  static const int cfg_threads[5] = {Cfg<1, false, false>::NTHREADS, Cfg<1, false, true>::NTHREADS,
                                     Cfg<2, false, false>::NTHREADS, Cfg<1, true, false>::NTHREADS,
                                     Cfg<2, true, false>::NTHREADS};
  cfg.blockDim = dim3((unsigned)cfg_threads[variant], 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  if ((err = cudaLaunchKernelExC(&cfg, fn, args)) != cudaSuccess) return err;
  if (pl.tail_split > 1) {
    const size_t total = (size_t)pl.tail_tiles * p.tail_rows * (BN / 4);
    const unsigned g = (unsigned)std::min<size_t>((total + 255) / 256, (size_t)info.sm_count * 8);
    const float4* part = reinterpret_cast<const float4*>(p.tail_part);
    uint16_t* yy = static_cast<uint16_t*>(a.y);
    const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
    if (a.bf16)
      tail_reduce_kernel<true><<<g, 256, 0, stream>>>(part, yy, bias, a.M, a.N, BM, p.tail_rows,
                                                      p.m_blocks, p.tail_start, pl.tail_tiles,
                                                      pl.tail_split);
    else
      tail_reduce_kernel<false><<<g, 256, 0, stream>>>(part, yy, bias, a.M, a.N, BM, p.tail_rows,
                                                       p.m_blocks, p.tail_start, pl.tail_tiles,
                                                       pl.tail_split);
    err = cudaGetLastError();
  }
  return err;
}

// ---- static scratch for w4a16_gemm_noalloc ------------------------------------
// One array per GPU that loads the library, held until exit. Host code must
// not pass the symbol itself to a kernel (it names a host-side stand-in): the
// device address comes from cudaGetSymbolAddress, once per device.
__device__ __align__(256) uint8_t g_noalloc_scratch[W4_NOALLOC_SCRATCH_BYTES];

cudaError_t noalloc_scratch(void** out, size_t* bytes) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  *bytes = W4_NOALLOC_SCRATCH_BYTES;
  return cudaSuccess;
}

// Device address of the status word, for the kernels of the other translation
// units (each .cu compiles on its own, so they cannot name the symbol).
cudaError_t device_status_ptr(int** out) {
  static std::mutex mu;
  static int* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) return e;
    addr[dev] = static_cast<int*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t read_device_status(int* out, int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear && v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace w4
