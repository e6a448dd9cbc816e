// Device-side helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w4 {

// Nibble position of row offset e inside a TILE word (rows 2i and 2i+1 share
// bit ranges 4i and 16+4i, so one mask extracts an (even, odd) row pair).
__host__ __device__ constexpr int tile_nibble_pos(int e) {
  return (e & 1) ? 4 + (e >> 1) : (e >> 1);
}
// AWQ stores column j of its 8-column block at nibble awq_nibble_pos(j):
// the order {0,4,1,5,2,6,3,7}.
__host__ __device__ constexpr int awq_nibble_pos(int j) {
  return (j & 1) ? 4 + (j >> 1) : (j >> 1);
}

// (a & b) | c in one instruction.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Exponent pattern that turns a 4-bit code q in the low mantissa bits into the
// half value MAGIC + q (bf16: 128 + q, fp16: 1024 + q), in both halves.
template <bool BF16> struct Magic;
template <> struct Magic<true> {
  static constexpr uint32_t pair = 0x43004300u;
};
template <> struct Magic<false> {
  static constexpr uint32_t pair = 0x64006400u;
};

template <bool BF16>
__device__ __forceinline__ uint32_t sub_x2(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF16) {
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  } else {
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  }
  return d;
}

// a * b + c on fp16 pairs, one rounding.
__device__ __forceinline__ uint32_t fma_x2_f16(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t mul_x2(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF16) {
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  } else {
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  }
  return d;
}

template <bool BF16>
__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    return __half2float(__ushort_as_half(h));
  }
}

template <bool BF16>
__device__ __forceinline__ uint16_t float_to_half_bits(float f) {
  if constexpr (BF16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  } else {
    return __half_as_ushort(__float2half_rn(f));
  }
}

// Streaming 16-byte load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// D += A * B for one m16n8k16 tile, fp32 accumulate.
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

}  // namespace w4
