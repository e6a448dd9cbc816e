// Small-M (decode) W4A16 GEMM: y[M][N] = x[M][K] · W, M <= 64 per launch.
//
// Decode is bound by streaming the packed weights from HBM ("vLLM 学习手册 01.
// 量化" §1: decode has FLOPs/Bytes ~ 1 and moving the weights dominates), so
// the kernel is organised around the weight stream:
//
//  * A CTA owns one 128-column group (eight 16-column tiles, one warp each)
//    and a K range. In the TILE layout that group's atoms are one contiguous
//    run along K (the eight tiles of a k-atom are adjacent, 4 KB), so the CTA
//    reads its weights as a single sequential stream: bulk asynchronous copies
//    (cp.async.bulk) of several k-atoms at a time into a CTA-wide ring, each
//    completion counted on one mbarrier per stage. Every warp reads its tile's
//    atom of each k-atom; the last warp to finish a stage refills its slot
//    with the stage one ring-length ahead. The CTA's first stages are also
//    prefetched into L2 before the kernel waits for its predecessor in the
//    stream (L2 is the device's point of coherence, so this never reads stale
//    data), and the stream keeps a prefetch a few stages ahead of the ring.
//  * One 16-byte shared-memory load per lane is exactly the A-fragment set of
//    four m16n8k16 MMAs in the swapped form y^T = W^T · x^T (the weight
//    columns fill the MMA's 16 rows, the tokens its 8 columns).
//  * Dequantisation ("vLLM AWQ 4-bit 量化实践" §5.3: (b - zeros) * scales) is
//    split: one LOP3 turns a nibble pair into MAGIC + q halves and the
//    per-(group, column) scale multiplies the fp32 partial sum of each group.
//    With bf16 one packed subtraction of 128 + z per register forms q - z
//    exactly (on the FMA pipe, beside the LOP3s on the ALU pipe); with fp16
//    nibbles of two slots are taken per shift and one packed fma or
//    subtraction forms q - z, exact as well.
//  * The CTA stages its slice of x in shared memory (gathering x[:, perm] for
//    act-order layers), padded so fragment loads are free of bank conflicts;
//    when it does not fit, x is staged in double-buffered chunks while the
//    weight stream runs on across chunk boundaries.
//  * Split-K across the CTAs of a thread-block cluster (up to 16 along K): each
//    CTA pushes its fp32 partial sums into the shared memory of the CTA that
//    owns those output columns (distributed shared memory stores), one
//    cluster barrier later every owner sums its slice over the peers in a
//    fixed order (deterministic, no global workspace, no atomics:
//    "vLLM AWQ 4-bit 量化实践" §5.3 names split-K for the fused kernel).
//  * Launches use programmatic stream serialization: a CTA may become resident
//    while the previous kernel drains. It requests its weights, scales and
//    zeros at once, waits for that kernel (griddepcontrol.wait) before reading
//    x or writing anything, and then lets the next kernel on the stream launch
//    so that its prologue overlaps this kernel's tail.
//  * Every wait is bounded (one second). A timed-out wait records
//    W4_ERR_TIMEOUT in the device status word and raises a CTA abort flag that
//    ends every other wait at once; the CTA lets its copies in flight land
//    (bounded again) before it exits.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <type_traits>
#include <unordered_map>

#include "decode_common.cuh"
#include "sm100_ptx.cuh"
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace cg = cooperative_groups;

namespace w4 {

namespace {

using namespace sm100;
using namespace dec;

constexpr int DEC_WARPS = 8;                  // one warp per tile of a 128-column group
constexpr int DEC_THREADS = DEC_WARPS * 32;
constexpr int ATOM_K = 64;
constexpr int ATOM_BYTES = 512;
constexpr int KROW_BYTES = DEC_WARPS * ATOM_BYTES;  // a column group's atoms at one k-atom
constexpr int MAX_SPLIT = 16;                // cluster size (above 8: non-portable)
#ifndef W4_DECODE_SA
#define W4_DECODE_SA 4  // k-atoms per ring stage
#endif
constexpr int SA = W4_DECODE_SA;
constexpr int STAGE_BYTES = SA * KROW_BYTES;  // 16 KB
constexpr int MAX_RING = 8;
constexpr int X_BUDGET = 48 * 1024;           // bytes of staged x per CTA
#ifndef W4_DECODE_PF
#define W4_DECODE_PF 2  // stages prefetched into L2 beyond the ring
#endif

struct DecodeParams {
  const uint16_t* x;       // [M][K]
  const uint32_t* qw;      // TILE words
  const uint16_t* scales;  // [G][N]
  const uint32_t* zeros;   // [G][N/8] standard order
  const int32_t* perm;     // [K] or nullptr
  uint16_t* y;             // [M][N]
  const uint16_t* bias;    // [N] or nullptr
  int M, N, K;
  int gshift;              // group = 1 << gshift; 31 = one group over all of K
  int A;                   // K / 64
  int ring;                // stages of the CTA's ring
  int pf;                  // stages prefetched into L2 beyond the ring
  int chunk_atoms;         // k-atoms of x staged at a time (a multiple of SA when chunked)
  int nbuf;                // x chunk buffers: 2 when the CTA's K range spans several chunks
  int x_stride;            // shared x row stride in halves
  int maxg;                // group slots per chunk
  int slice;               // output columns owned by each CTA of a cluster
  int* status;             // the library's device status word
  int stall;               // test hook: withhold the weight copies (every ring wait runs out)
  // grouped (expert) calls: blockIdx.z is the expert, whose weights sit qw_estride
  // words / s_estride scales / z_estride zero words after the previous expert's
  // and whose rows of x and y are [eoff[e], eoff[e+1]) (at most M of them)
  const int32_t* eoff;
  size_t qw_estride, s_estride, z_estride;
  int total_rows;
};

struct SmemLayout {
  int xs, ring, bars, cnt, meta, recv, total;
};

// xs: nbuf buffers of M token rows (the MMA lanes whose token row is beyond M
// read row 0: their output columns are never stored). bars: ring mbarriers, then one per x
// buffer. cnt: per slot the count of warps done with it (monotonic), per slot
// the last stage copied into it, per x buffer the last chunk copied into it,
// and the abort flag. meta: per warp and group slot, the scales of the tile's
// 16 columns as they are stored (one 32-bit word per lane group: columns gg
// and gg + 8), then per warp and group slot the tile's two zero words.
// recv: the cluster peers' partial sums of this CTA's output columns, [peer]
// [token][column] (the reducing threads walk consecutive columns).
__host__ __device__ inline SmemLayout smem_layout(int MT, int m_rows, int x_stride, int nbuf,
                                                  int ring, int maxg, int S, int slice) {
  SmemLayout L;
  L.xs = 0;
  L.ring = ((nbuf * m_rows * x_stride * 2) + 1023) & ~1023;
  L.bars = L.ring + ring * STAGE_BYTES;
  L.cnt = L.bars + (ring + 2) * 8;
  L.meta = (L.cnt + (2 * ring + 2 + 1) * 4 + 15) & ~15;
  L.recv = L.meta + DEC_WARPS * maxg * (8 * 4 + 8);
  L.total = L.recv + S * slice * 8 * MT * 4;
  return L;
}

// MT: token tiles of 8 (M <= 8 * MT). G64: every 64-row atom lies in one group.
#ifndef W4_DECODE_MIN_CTAS
#define W4_DECODE_MIN_CTAS 3  // resident CTAs per SM the M <= 8 register budget is sized for
#endif
constexpr int decode_min_ctas(int MT) { return MT == 1 ? W4_DECODE_MIN_CTAS : 2; }

// The MMA consumes q - z, exact in both types (the zero pairs are built per
// group from the staged zero words), and the loop adds s * acc per group.
template <int MT, bool BF16, bool G64>
__global__ void __launch_bounds__(DEC_THREADS, decode_min_ctas(MT))
    w4a16_decode_kernel(const DecodeParams p) {
  constexpr uint32_t MAGIC = Magic<BF16>::pair;  // 128 (bf16) / 1024 (fp16) in both halves
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gg = lane >> 2, t = lane & 3;
  const int S = gridDim.y;          // split-K factor == cluster size along y
  const int srank = blockIdx.y;     // rank inside the cluster
  const int MR = 8 * MT;
  const int D = p.ring;
  const int NB = p.nbuf;
  const SmemLayout L = smem_layout(MT, p.M, p.x_stride, NB, D, p.maxg, S, p.slice);
  // grouped calls: this CTA's expert and its weights; its rows come after the wait
  const bool grouped = p.eoff != nullptr;
  const int ex = blockIdx.z;
  const uint32_t* qwp = p.qw + (size_t)ex * p.qw_estride;
  const uint16_t* scp = p.scales + (size_t)ex * p.s_estride;
  const uint32_t* zp = p.zeros + (size_t)ex * p.z_estride;
  int M = p.M;  // rows of this call (the shared-memory layout is sized for p.M)
  const uint16_t* xg = p.x;
  uint16_t* yg = p.y;
  __shared__ int grp_rows[2];

  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
  const uint32_t ring_s = smem_addr(smem + L.ring);
  const uint32_t full0 = smem_addr(smem + L.bars);       // + 8 * slot
  const uint32_t xbar0 = full0 + 8 * D;                   // + 8 * buffer
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);        // [D] warps done with each slot
  int* last_stage = cnt + D;                              // [D] last stage copied into each slot
  int* last_chunk = last_stage + D;                       // [2] last x chunk copied into each buffer
  volatile int* abort_flag = last_chunk + 2;
  // per (group slot, lane group gg): the scales of columns gg and gg + 8 of the
  // warp's tile; then per group slot the tile's two zero words
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + L.meta) + warp * p.maxg * 8;
  uint2* zraw = reinterpret_cast<uint2*>(smem + L.meta + DEC_WARPS * p.maxg * 32) + warp * p.maxg;
  // a meta word as the fp32 scales of columns gg and gg + 8 (exact)
  auto scale_pair = [](const uint32_t w) {
    return make_float2(half_bits_to_float<BF16>((uint16_t)(w & 0xFFFFu)),
                       half_bits_to_float<BF16>((uint16_t)(w >> 16)));
  };
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  constexpr int NCOL = 16 * DEC_WARPS;

  // CTA K range: whole stages of SA k-atoms (the last one may be partial), so
  // stage starts are aligned to SA k-atoms and a group of 128 rows or fewer
  // never straddles a stage
  const int nst_all = (p.A + SA - 1) / SA;
  const int ka0 = min(p.A, (int)((long long)srank * nst_all / S) * SA);
  const int ka1 = min(p.A, (int)((long long)(srank + 1) * nst_all / S) * SA);
  const int NS = (ka1 - ka0 + SA - 1) / SA;
  const int nchunks = (ka1 - ka0 + p.chunk_atoms - 1) / p.chunk_atoms;

  const int cgi = blockIdx.x;  // column group
  const int nt = cgi * DEC_WARPS + warp;
  const bool has_cols = nt < p.N / 16;
  // the column group's run: k-atom a at byte offset a * KROW_BYTES
  const uint8_t* gsrc = reinterpret_cast<const uint8_t*>(qwp) + (size_t)cgi * p.A * KROW_BYTES;
  const uint64_t stream_policy = evict_first_policy();
  const bool x_async = p.perm == nullptr;

  // x of chunk ci into buffer ci % NB, completion on that buffer's barrier (tid 0)
  auto issue_x = [&](int ci) {
    const int c0 = ka0 + ci * p.chunk_atoms;
    const int KC = (min(ka1, c0 + p.chunk_atoms) - c0) * ATOM_K;
    const int b = NB == 2 ? (ci & 1) : 0;
    uint16_t* dst = xs + (size_t)b * p.M * p.x_stride;
    last_chunk[b] = ci;
    mbar_arrive_expect_tx(xbar0 + 8 * b, (uint32_t)(M * KC * 2));
    for (int m = 0; m < M; ++m)
      bulk_copy(smem_addr(dst + (size_t)m * p.x_stride), xg + (size_t)m * p.K + c0 * ATOM_K,
                (uint32_t)(KC * 2), xbar0 + 8 * b);
  };
  // stage j (k-atoms [ka0 + j*SA, ...)) into ring slot j % D (one thread)
  auto issue_stage = [&](int j) {
    const int a = ka0 + j * SA;
    const uint32_t bytes = (uint32_t)min(SA, ka1 - a) * KROW_BYTES;
    const int slot = j % D;
    last_stage[slot] = j;
    mbar_arrive_expect_tx(full0 + 8 * slot, bytes);
    bulk_copy_stream(ring_s + slot * STAGE_BYTES, gsrc + (size_t)a * KROW_BYTES, bytes,
                     full0 + 8 * slot, stream_policy);
    // stage j + pf into L2 (stages below D + pf were prefetched at the start)
    const int pa = a + p.pf * SA;
    if (p.pf > 0 && pa < ka1 && j >= D)
      prefetch_l2(gsrc + (size_t)pa * KROW_BYTES, (uint32_t)min(SA, ka1 - pa) * KROW_BYTES);
  };
  // one group's 16 scales (of this warp's tile) into its 8 meta entries (entry
  // c: column c in the low half, column c + 8 in the high half), and its zero
  // words
  auto stage_meta = [&](int gl, const uint4 a, const uint4 b, const uint2 z) {
    const uint32_t sv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int c = 0; c < 8; ++c)
      meta[gl * 8 + c] = __byte_perm(sv[c >> 1], sv[4 + (c >> 1)], (c & 1) ? 0x7632u : 0x5410u);
    zraw[gl] = z;
  };
  // the first ring stages, and the pf stages beyond the ring into L2 (one thread)
  auto fill_ring = [&]() {
    for (int j = 0; j < min(D, NS); ++j) issue_stage(j);
    const int a0 = ka0 + min(D, NS) * SA, a1 = min(ka1, ka0 + (D + p.pf) * SA);
    if (a1 > a0) prefetch_l2(gsrc + (size_t)a0 * KROW_BYTES, (uint32_t)(a1 - a0) * KROW_BYTES);
  };
  // scales / zeros of the groups of chunk ci for this warp's tile; in the first
  // chunk the ring fill waits until every warp has issued these loads, so they
  // are not queued behind the weight stream
  auto stage_chunk_meta = [&](int ci) {
    const int c0 = ka0 + ci * p.chunk_atoms;
    const int c1 = min(ka1, c0 + p.chunk_atoms);
    const int g_first = (c0 * ATOM_K) >> p.gshift;
    const int ng = ((c1 * ATOM_K - 1) >> p.gshift) - g_first + 1;
    uint4 ms0 = make_uint4(0, 0, 0, 0), ms1 = ms0;
    uint2 mz = make_uint2(0, 0);
    const bool mine = has_cols && lane < ng;
    if (mine) {
      const int gi = g_first + lane;
      const uint4* sp = reinterpret_cast<const uint4*>(scp + (size_t)gi * p.N + nt * 16);
      ms0 = __ldg(sp);
      ms1 = __ldg(sp + 1);
      mz = __ldg(reinterpret_cast<const uint2*>(zp + (size_t)gi * (p.N / 8) + nt * 2));
    }
    if (ci == 0) {
      __syncthreads();  // every warp has issued its gating loads
      if (tid == 0 && !p.stall && !grouped) fill_ring();
    }
    if (mine) stage_meta(lane, ms0, ms1, mz);
    for (int gl = lane + 32; has_cols && gl < ng; gl += 32) {
      const int gi = g_first + gl;
      const uint4* sp = reinterpret_cast<const uint4*>(scp + (size_t)gi * p.N + nt * 16);
      const uint4 a = __ldg(sp), bb = __ldg(sp + 1);
      const uint2 z =
          __ldg(reinterpret_cast<const uint2*>(zp + (size_t)gi * (p.N / 8) + nt * 2));
      stage_meta(gl, a, bb, z);
    }
  };

  // ---- before the dependency wait: everything that does not read x ------------
  // The weights, scales and zeros are read here, before the kernel waits for its
  // predecessor on the stream: the library's contract is that they are not
  // written by the kernel launched just before the GEMM (the repack entry points
  // end with an empty kernel for that reason).
  if (tid == 0) {
    for (int s = 0; s < D; ++s) {
      mbar_init(full0 + 8 * s, 1);
      cnt[s] = 0;
      last_stage[s] = -1;
    }
    for (int b = 0; b < NB; ++b) mbar_init(xbar0 + 8 * b, 1);
    last_chunk[0] = last_chunk[1] = -1;
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();  // barrier initialisation and counters
  if (nchunks > 0) stage_chunk_meta(0);

  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every CTA of this grid is resident: the next kernel may start its own
  // prologue as resources free up
  asm volatile("griddepcontrol.launch_dependents;");
  if (grouped) {
    // the expert's rows (the offsets may come from the kernel before this one);
    // an expert with no rows skips its weight stream altogether
    if (tid == 0) {
      const int r0 = *reinterpret_cast<const volatile int32_t*>(p.eoff + ex);
      const int r1 = *reinterpret_cast<const volatile int32_t*>(p.eoff + ex + 1);
      int m = r1 - r0;
      if (r0 < 0 || m < 0 || r1 > p.total_rows || m > p.M) {
        atomicExch(p.status, W4_ERR_EXPERT_ROWS);
        m = 0;
      }
      grp_rows[0] = r0;
      grp_rows[1] = m;
    }
    __syncthreads();
    M = grp_rows[1];
    xg = p.x + (size_t)grp_rows[0] * p.K;
    yg = p.y + (size_t)grp_rows[0] * p.N;
    if (tid == 0 && M > 0 && !p.stall) fill_ring();
  }
  if (tid == 0 && x_async && nchunks > 0 && M > 0) {
    issue_x(0);
    if (NB == 2 && nchunks > 1) issue_x(1);
  }

  // acc: the open group's MMA sums; tc: the CTA's total
  float acc[MT][4], tc[MT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = tc[i][j] = 0.f;
  float2 gf = make_float2(0.f, 0.f);  // scales of the open group (columns gg, gg + 8)
  uint32_t zl = 0, zh = 0;            // MAGIC + z pairs of the open group
  uint32_t nl = 0, nh = 0;            // fp16: -(64 + z) pairs (the high slot's offset)
  int gslot = -1;                     // its slot in meta (-1: none open)
  uint32_t rslot = 0, rphase = 0;     // ring slot of the next stage, its parity

  // tc += s * acc; acc = 0
  auto flush = [&]() {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      tc[mt][0] = fmaf(gf.x, acc[mt][0], tc[mt][0]);
      tc[mt][1] = fmaf(gf.x, acc[mt][1], tc[mt][1]);
      tc[mt][2] = fmaf(gf.y, acc[mt][2], tc[mt][2]);
      tc[mt][3] = fmaf(gf.y, acc[mt][3], tc[mt][3]);
      acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    }
  };
  // close the open group (if any) and open the next one
  auto next_group = [&]() {
    if (gslot >= 0) flush();
    ++gslot;
    gf = scale_pair(meta[gslot * 8 + gg]);
    {
      const uint2 zw = zraw[gslot];
      const uint32_t z0 = (zw.x >> (4 * gg)) & 0xFu, z1 = (zw.y >> (4 * gg)) & 0xFu;
      zl = MAGIC + z0 * 0x00010001u;
      zh = MAGIC + z1 * 0x00010001u;
      if constexpr (!BF16) {
        // -(64 + z) in fp16: 64 is 0x5400, whose last mantissa bit is 1/16
        nl = (0xD400u + 16u * z0) * 0x00010001u;
        nh = (0xD400u + 16u * z1) * 0x00010001u;
      }
    }
  };

  for (int ci = 0; M > 0 && ci < nchunks; ++ci) {
    const int c0 = ka0 + ci * p.chunk_atoms;
    const int c1 = min(ka1, c0 + p.chunk_atoms);
    const int KC = (c1 - c0) * ATOM_K;
    const int b = NB == 2 ? (ci & 1) : 0;
    const bool live = !*abort_flag;

    // 1) scales / zeros (the first chunk's were staged before the wait)
    if (ci > 0 && live) stage_chunk_meta(ci);
    // 2) x of this chunk
    uint16_t* xb = xs + (size_t)b * p.M * p.x_stride;
    if (!x_async) {
      // act-order: gather x[:, perm] with plain loads
      const int chunks = KC / 8;
      const int kx0 = c0 * ATOM_K;
      for (int i = tid; live && i < M * chunks; i += DEC_THREADS) {
        const int m = i / chunks, c = i - m * chunks;
        const uint16_t* xr = xg + (size_t)m * p.K;
        uint16_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __ldg(xr + __ldg(p.perm + kx0 + 8 * c + e));
        uint4 v;
        v.x = h[0] | ((uint32_t)h[1] << 16);
        v.y = h[2] | ((uint32_t)h[3] << 16);
        v.z = h[4] | ((uint32_t)h[5] << 16);
        v.w = h[6] | ((uint32_t)h[7] << 16);
        *reinterpret_cast<uint4*>(xb + (size_t)m * p.x_stride + 8 * c) = v;
      }
    } else if (live) {
      bounded_wait(xbar0 + 8 * b, (uint32_t)((NB == 2 ? ci >> 1 : ci) & 1), abort_flag, p.status);
    }
    __syncthreads();  // x and every warp's scale / zero stage are ready
    // 3) consume this chunk's stages. Shared-memory operands are addressed with
    //    32-bit shared-window addresses with constant offsets inside a stage.
    // this lane's x row at the chunk's first atom, column 8t; lanes whose token
    // row is beyond M read row 0 (their output columns are discarded)
    uint32_t xa[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int row = 8 * mt + gg;
      xa[mt] = smem_addr(xb + (size_t)(row < M ? row : 0) * p.x_stride) + 16u * (uint32_t)t;
    }
    // k-atoms per group (groups of 64 rows or more); a chunk that starts inside
    // a group (only possible for groups longer than a stage) opens it at once
    const int apg = G64 ? (p.gshift >= 31 ? (1 << 30) : (1 << (p.gshift - 6))) : 1;
    gslot = -1;
    if (has_cols && G64 && (c0 & (apg - 1)) != 0) next_group();

    // one half atom (32 rows x 16 columns): two k-steps, one x load and two MMAs
    // per token tile; xo = byte offset of the atom's x columns from xa
    auto half_atom = [&](const uint32_t wlo, const uint32_t whi, const uint32_t xo) {
      uint32_t af[2][4];
#pragma unroll
      for (int step = 0; step < 2; ++step) {
        const int sh = 8 * step;
        if constexpr (BF16) {
          // 128 + q minus 128 + z: q - z exactly
          af[step][0] = sub_x2<true>(lop3_and_or(wlo >> sh, 0x000F000Fu, MAGIC), zl);
          af[step][2] = sub_x2<true>(lop3_and_or(wlo >> (sh + 4), 0x000F000Fu, MAGIC), zl);
          af[step][1] = sub_x2<true>(lop3_and_or(whi >> sh, 0x000F000Fu, MAGIC), zh);
          af[step][3] = sub_x2<true>(lop3_and_or(whi >> (sh + 4), 0x000F000Fu, MAGIC), zh);
        } else {
          // fp16 has two 4-bit slots below its 10 mantissa bits: the nibbles
          // at bits 4-7 / 20-23 give 1024 + 16q in place, and one fused
          // multiply-add by 1/16 takes it to q - z exactly (64 + q is exact),
          // so one shift serves four nibble pairs instead of three shifts
          const uint32_t lo = wlo >> sh, hi = whi >> sh;
          af[step][0] = sub_x2<false>(lop3_and_or(lo, 0x000F000Fu, MAGIC), zl);
          af[step][2] = fma_x2_f16(lop3_and_or(lo, 0x00F000F0u, MAGIC), 0x2C002C00u, nl);
          af[step][1] = sub_x2<false>(lop3_and_or(hi, 0x000F000Fu, MAGIC), zh);
          af[step][3] = fma_x2_f16(lop3_and_or(hi, 0x00F000F0u, MAGIC), 0x2C002C00u, nh);
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint4 xf = lds128(xa[mt] + xo);
        mma16816<BF16>(acc[mt], af[0][0], af[0][1], af[0][2], af[0][3], xf.x, xf.y);
        mma16816<BF16>(acc[mt], af[1][0], af[1][1], af[1][2], af[1][3], xf.z, xf.w);
      }
    };
    // one atom (64 rows x 16 columns); `start` says whether a group starts here
    auto atom = [&](const uint4 w, const uint32_t xo, const bool start) {
      if constexpr (G64) {
        if (start) next_group();
        half_atom(w.x, w.y, xo);
        half_atom(w.z, w.w, xo + 64u);
      } else {  // groups of 32 rows: each half atom is a group
        next_group();
        half_atom(w.x, w.y, xo);
        next_group();
        half_atom(w.z, w.w, xo + 64u);
      }
    };
    // a full stage with group starts at compile-time positions: every P-th atom
    // (P = 1, 2), or (P = 0) at most one, at the first atom
    auto full_stage = [&](const uint32_t st, const uint32_t xo, const int a_base, auto P) {
      constexpr int PP = decltype(P)::value;
      const bool first = (a_base & (apg - 1)) == 0;
#pragma unroll
      for (int u = 0; u < SA; ++u) {
        const bool start = PP == 0 ? (u == 0 && first) : (u % PP == 0);
        atom(lds128(st + u * KROW_BYTES), xo + u * (ATOM_K * 2), start);
      }
    };

    const int j0 = (c0 - ka0) / SA;
    const int j1 = min(NS, (c1 - ka0 + SA - 1) / SA);
    const uint32_t wbase = ring_s + (uint32_t)warp * ATOM_BYTES + (uint32_t)lane * 16u;
    for (int j = j0; j < j1; ++j) {
      const bool ready = live && bounded_wait(full0 + 8 * rslot, rphase, abort_flag, p.status);
      if (ready && has_cols) {
        const int a_base = ka0 + j * SA;
        const uint32_t st = wbase + rslot * STAGE_BYTES;
        const uint32_t xo = (uint32_t)(a_base - c0) * (ATOM_K * 2);
        if (a_base + SA <= c1) {
          if (!G64 || apg >= SA)
            full_stage(st, xo, a_base, std::integral_constant<int, 0>());
          else if (apg == 2)
            full_stage(st, xo, a_base, std::integral_constant<int, 2>());
          else if (apg == 1)
            full_stage(st, xo, a_base, std::integral_constant<int, 1>());
          else
            full_stage(st, xo, a_base, std::integral_constant<int, 4>());
        } else {
          for (int u = 0; u < c1 - a_base; ++u)
            atom(lds128(st + u * KROW_BYTES), xo + u * (ATOM_K * 2),
                 ((a_base + u) & (apg - 1)) == 0);
        }
        // groups longer than a stage are flushed at every stage as well (the
        // flush is linear and the zero-point part was removed up front), which
        // bounds the length of an fp32 MMA accumulation to one stage
        if (G64 && apg > SA && gslot >= 0) flush();
      }
      __syncwarp();
      // release the slot; the last of the eight warps refills it with stage j + D
      if (lane == 0 && ready) {
        __threadfence_block();  // this warp's reads of the slot precede its count
        const int old = atomicAdd(&cnt[rslot], 1);
        if ((old & (DEC_WARPS - 1)) == DEC_WARPS - 1 && j + D < NS) {
          __threadfence_block();     // every warp's reads precede the refill
          fence_proxy_async_smem();  // ... which the async proxy performs
          issue_stage(j + D);
        }
      }
      if (++rslot == (uint32_t)D) {
        rslot = 0;
        rphase ^= 1u;
      }
    }
    // the scale / zero stage and the sums belong to this chunk: close the group
    if (has_cols && gslot >= 0) flush();
    __syncthreads();  // the chunk's x buffer, sums and scale / zero stage are free again
    if (x_async && tid == 0 && NB == 2 && ci + 2 < nchunks && !*abort_flag) {
      fence_proxy_async_smem();  // the reads of the buffer precede the copy into it
      issue_x(ci + 2);
    }
  }

  // ---- after an abort: let every copy in flight land before the CTA exits ------
  if (*abort_flag) {
    __syncthreads();
    if (tid == 0) {
      for (int s = 0; s < D; ++s)
        if (last_stage[s] >= 0) drain_wait(full0 + 8 * s, (uint32_t)((last_stage[s] / D) & 1));
      for (int bb = 0; bb < NB; ++bb)
        if (last_chunk[bb] >= 0)
          drain_wait(xbar0 + 8 * bb,
                     (uint32_t)((NB == 2 ? last_chunk[bb] >> 1 : last_chunk[bb]) & 1));
    }
  }

  // ---- split-K: push partial sums to the CTA that owns each output column -------
  cg::cluster_group cluster = cg::this_cluster();
  const int SL = p.slice;
  auto push = [&](int col, int m, float v) {
    const int owner = col / SL;
    float* dst = cluster.map_shared_rank(recv, owner);
    dst[((size_t)srank * MR + m) * SL + (col - owner * SL)] = v;
  };
  if (has_cols) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int m0 = 8 * mt + 2 * t;
      const int ca = warp * 16 + gg, cb = ca + 8;
      if (m0 < M) {
        push(ca, m0, tc[mt][0]);
        push(cb, m0, tc[mt][2]);
      }
      if (m0 + 1 < M) {
        push(ca, m0 + 1, tc[mt][1]);
        push(cb, m0 + 1, tc[mt][3]);
      }
    }
  }
  cluster.sync();
  {
    const int c_lo = srank * SL;
    const int c_hi = min(NCOL, c_lo + SL);
    const int width = c_hi - c_lo;
    for (int o = tid; o < width * M; o += DEC_THREADS) {
      const int m = o / width, cl = o - m * width;
      const int n = cgi * NCOL + c_lo + cl;
      if (n >= p.N) continue;
      float sum = 0.f;
      for (int r = 0; r < S; ++r) sum += recv[((size_t)r * MR + m) * SL + cl];
      if (p.bias != nullptr) sum += half_bits_to_float<BF16>(p.bias[n]);  // one rounding below
      yg[(size_t)m * p.N + n] = float_to_half_bits<BF16>(sum);
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

// Raise a kernel's dynamic shared-memory limit (and allow clusters above the
// portable size of 8) once per (kernel, device); the attribute calls are then
// kept out of the launch path (and out of graph capture).
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
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

struct DecodePlan {
  int S;
  int ring, pf, chunk_atoms, nbuf, x_stride, maxg, slice;
  SmemLayout L;
};

// Shared-memory plan of one launch shape. x of the CTA's whole K range is
// staged at once when it fits X_BUDGET; otherwise in chunks of a multiple of
// SA k-atoms, double-buffered so the next chunk's x lands while the current
// one is consumed.
DecodePlan shape_plan(int S, int A, int Mc, int MT, int gshift, int ring) {
  DecodePlan d;
  d.S = S;
  d.ring = ring;
  d.pf = W4_DECODE_PF;
  const int cta_atoms = ((A + SA - 1) / SA + S - 1) / S * SA;  // whole stages
  if (cta_atoms * ATOM_K * Mc * 2 <= X_BUDGET) {
    d.nbuf = 1;
    d.chunk_atoms = cta_atoms;
  } else {
    d.nbuf = 2;
    d.chunk_atoms = std::max(SA, X_BUDGET / 2 / (Mc * 2) / ATOM_K / SA * SA);
  }
  d.x_stride = d.chunk_atoms * ATOM_K + 32;  // halves; row stride = 64 mod 128 bytes
  d.maxg = (gshift == 31) ? 1 : (d.chunk_atoms * ATOM_K >> gshift) + 2;
  d.slice = (16 * DEC_WARPS + S - 1) / S;
  d.L = smem_layout(MT, Mc, d.x_stride, d.nbuf, ring, d.maxg, S, d.slice);
  return d;
}

// CTAs of `fn` resident per SM with `smem` bytes of dynamic shared memory, as
// the runtime's occupancy calculator counts them (registers, shared memory with
// its allocation granularity and per-CTA reservation); 0 on an error.
int resident_ctas(void* fn, int smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, DEC_THREADS, (size_t)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();  // a failed query must not surface in a later launch's check
    return 0;
  }
  return n;
}

// Deepest ring (2..MAX_RING stages, no deeper than the CTA's stage count) that
// keeps `per_sm` CTAs resident.
DecodePlan fit_ring(int S, int A, int Mc, int MT, int gshift, int per_sm, void* fn) {
  const int stages = ((A + SA - 1) / SA + S - 1) / S;
  const int need = std::max(2, std::min(MAX_RING, stages));
  DecodePlan d = shape_plan(S, A, Mc, MT, gshift, 2);
  for (int r = need; r >= 2; --r) {
    d = shape_plan(S, A, Mc, MT, gshift, r);
    if (resident_ctas(fn, d.L.total) >= per_sm) break;
  }
  return d;
}

// Clusters of the launch (grid gx x S x gz, clusters 1 x S x 1, `smem` bytes of
// dynamic shared memory) that the device runs at once, as the runtime counts
// them (residency per SM and the packing of a cluster's CTAs into one GPC); 0
// on an error.
int resident_clusters(void* fn, int gx, int S, int gz, int smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gx, (unsigned)S, (unsigned)gz);
  cfg.blockDim = dim3(DEC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)S;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();  // a failed query must not surface in a later launch's check
    return 0;
  }
  return n;
}

// Choose the split-K factor S and the ring. For every S the ring is as deep as
// keeps 3 CTAs per SM resident (2 when the register budget allows only 2; the
// runtime's occupancy count), and the runtime says how many clusters of S CTAs
// run at once: a cluster's CTAs must fit on S SMs of one GPC, so the number of
// waves of a split depends on how clusters pack into GPCs, not only on CTAs per
// SM. Then:
//  * the largest S whose clusters run in one wave with at least two CTAs per SM
//    on average (the most warps per SM and the shortest K range per CTA);
//  * failing that, the S with the least waves x (k-atoms per CTA + 8): the
//    busiest SM's share of the stream plus a fixed cost per wave (prologue,
//    pipeline fill, cluster reduction) worth about 8 k-atoms; fewer waves on a
//    tie.
// Measured on GB300 against the S that each shape ran best with (sweeps over
// S = 1..16 of the Llama-2 7B / 70B decode calls at M = 1, 4, 16), this picks
// the best split on every call; the rule it replaced (about 2.6 CTAs per SM
// from the CTA count alone) ran Llama-2-70B down at 42.5 / 63.5 us against
// 35.3 / 52.7 us at M = 1 / 16 (its split took a second wave of clusters).
// CTA and cluster counts include every (column group, expert) pair of a grouped
// call.
DecodePlan plan_decode(int N, int K, int Mc, int MT, int gshift, int experts,
                       const DeviceInfo& info, void* fn) {
  const int NG = (N / 16 + DEC_WARPS - 1) / DEC_WARPS, A = K / ATOM_K;
  const long long units = (long long)NG * experts;  // (column group, expert) pairs of the grid
  const int nst_all = (A + SA - 1) / SA;
  auto cta_atoms = [&](int S) { return (nst_all + S - 1) / S * SA; };
  const int s_cap = std::min(MAX_SPLIT, nst_all);
  const int reg_ctas = decode_min_ctas(MT);
  DecodePlan one_wave{}, best{};
  bool have_one = false, have_best = false;
  long long best_cost = 0, best_waves = 0;
  for (int S = 1; S <= s_cap; ++S) {
    if (S > 1 && cta_atoms(S) == cta_atoms(S - 1)) continue;  // the same K ranges, more CTAs idle
    DecodePlan d = fit_ring(S, A, Mc, MT, gshift, std::min(3, reg_ctas), fn);
    if (resident_ctas(fn, d.L.total) < std::min(3, reg_ctas)) d = fit_ring(S, A, Mc, MT, gshift, 2, fn);
    const int clusters = resident_clusters(fn, NG, S, experts, d.L.total);
    if (clusters <= 0) continue;
    const long long waves = (units + clusters - 1) / clusters;
    if (waves == 1 && units * S >= 2LL * info.sm_count) {
      one_wave = d;
      have_one = true;
    }
    const long long cost = waves * (cta_atoms(S) + 8);
    if (!have_best || cost < best_cost || (cost == best_cost && waves < best_waves)) {
      best = d;
      best_cost = cost;
      best_waves = waves;
      have_best = true;
    }
  }
  if (have_one) return one_wave;
  if (have_best) return best;
  // no occupancy answer: the smallest split, two CTAs per SM
  return fit_ring(1, A, Mc, MT, gshift, 2, fn);
}

// Plans are cached per (device, shape): planning costs tens of microseconds of
// host time, more than a decode launch.
struct PlanKey {
  int dev, N, K, Mc, gshift, experts;
  void* fn;  // the kernel (its register budget decides residency)
  bool operator==(const PlanKey& o) const {
    return dev == o.dev && N == o.N && K == o.K && Mc == o.Mc && gshift == o.gshift &&
           experts == o.experts && fn == o.fn;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey& k) const {
    uint64_t h = (uint64_t)k.dev * 0x9E3779B97F4A7C15ull;
    h ^= (uint64_t)k.N + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    h ^= (uint64_t)k.K + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    h ^= (uint64_t)k.Mc + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    h ^= (uint64_t)k.gshift + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    h ^= (uint64_t)k.experts + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    h ^= reinterpret_cast<uint64_t>(k.fn) + 0x7F4A7C15ull + (h << 6) + (h >> 2);
    return (size_t)h;
  }
};

cudaError_t cached_plan(int N, int K, int Mc, int MT, int gshift, int experts,
                        const DeviceInfo& info, void* fn, DecodePlan* out) {
  static std::mutex mu;
  static std::unordered_map<PlanKey, DecodePlan, PlanKeyHash> plans;
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const PlanKey key{dev, N, K, Mc, gshift, experts, fn};
  std::lock_guard<std::mutex> lock(mu);
  auto it = plans.find(key);
  if (it == plans.end())
    it = plans.emplace(key, plan_decode(N, K, Mc, MT, gshift, experts, info, fn)).first;
  *out = it->second;
  return cudaSuccess;
}

int log2_exact(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return (1 << s) == v ? s : -1;
}

}  // namespace

size_t decode_workspace_bytes(int M, int K, bool has_perm) {
  return has_perm && M > 0 ? ((size_t)M * K * 2 + 255) & ~(size_t)255 : 0;
}

cudaError_t launch_decode(const GemmArgs& a, cudaStream_t stream) {
  // M <= 8 on a small layer (at most 96 KB of packed weights per SM), no
  // experts: the streaming kernel (decode_stream_kernel.cu); otherwise this one
  bool launched = false;
  cudaError_t err = launch_decode_stream(a, stream, &launched);
  if (err != cudaSuccess || launched) return err;
  DeviceInfo info;
  err = device_info(&info);
  if (err != cudaSuccess) return err;
  int gshift = log2_exact(a.group);
  if (a.group == a.K || gshift < 0) gshift = 31;  // one group over all of K
  const int A = a.K / ATOM_K;
  const bool g64 = gshift >= 6;  // groups of 64 or more: one group per atom
  int* status = nullptr;
  if ((err = device_status_ptr(&status)) != cudaSuccess) return err;
  // act-order with room in the workspace: gather x[:, perm] once for all CTAs
  // instead of once per CTA (every column group's CTAs read the same columns)
  const void* xsrc = a.x;
  const int32_t* perm = a.perm;
  if (perm && a.workspace && a.workspace_bytes >= decode_workspace_bytes(a.M, a.K, true)) {
    if ((err = launch_gather_columns(a.x, perm, a.workspace, a.M, a.K, stream)) != cudaSuccess)
      return err;
    xsrc = a.workspace;
    perm = nullptr;
  }
  for (int r0 = 0; r0 < a.M; r0 += DECODE_MAX_M) {
    const int Mc = std::min(DECODE_MAX_M, a.M - r0);
    const int MT = Mc <= 8 ? 1 : Mc <= 16 ? 2 : Mc <= 32 ? 4 : 8;
    DecodePlan plan;
    const int experts = a.eoff != nullptr ? a.num_experts : 1;
    void* fn = pick_kernel(MT, a.bf16 != 0, g64);
    // the occupancy queries of the plan need the kernel's dynamic limit at the
    // device's maximum (the opt-in limit less the kernel's static shared memory)
    cudaFuncAttributes fa;
    if ((err = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return err;
    if ((err = ensure_smem(fn, (size_t)info.max_smem_optin - fa.sharedSizeBytes)) != cudaSuccess)
      return err;
    if ((err = cached_plan(a.N, a.K, Mc, MT, gshift, experts, info, fn, &plan)) != cudaSuccess)
      return err;

    DecodeParams p;
    p.x = static_cast<const uint16_t*>(xsrc) + (size_t)r0 * a.K;
    p.qw = a.qw;
    p.scales = static_cast<const uint16_t*>(a.scales);
    p.zeros = a.zeros;
    p.perm = perm;
    p.y = static_cast<uint16_t*>(a.y) + (size_t)r0 * a.N;
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.M = Mc;
    p.N = a.N;
    p.K = a.K;
    p.gshift = gshift;
    p.A = A;
    p.ring = plan.ring;
    p.pf = plan.pf;
    p.chunk_atoms = plan.chunk_atoms;
    p.nbuf = plan.nbuf;
    p.x_stride = plan.x_stride;
    p.maxg = plan.maxg;
    p.slice = plan.slice;
    p.status = status;
    p.stall = a.test_stall;
    p.eoff = a.eoff;
    p.qw_estride = a.qw_estride;
    p.s_estride = a.s_estride;
    p.z_estride = a.z_estride;
    p.total_rows = a.total_rows;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.N / 16 + DEC_WARPS - 1) / DEC_WARPS, plan.S,
                       a.eoff != nullptr ? (unsigned)a.num_experts : 1u);
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
