// wq_tmem_dequant.cuh -- dequantisation of packed cells into tensor memory,
// shared by the tcgen05 kernels whose A operand is the dequantised weights
// (wq_gemm_wt.cu, wq_gemm_skinny.cu).
#pragma once

#include <cstdint>

#include "wq_device.cuh"
#include "wq_tcgen05.cuh"

namespace wq {

// Byte offset, within one cell of a chunk, of the 16-byte packed lane
// 4c + t4 of column n (INT8: of k half h) after the 128-byte swizzle: chunk
// `ch` of 128-byte row `row` sits at chunk position ch ^ (row % 8).
template <int BITS>
__device__ __forceinline__ uint32_t wt_lane_offset(int n, int h, int t4) {
  const int j8 = (n >> 3) & 7, c = n & 7;
  const int row = BITS == 4 ? j8 * 4 + (c >> 1) : (j8 * 2 + h) * 4 + (c >> 1);
  const int ch = (4 * (c & 1) + t4) ^ (row & 7);
  return row * 128 + ch * 16;
}

// Dequantise one group (128 k) of this thread's column into bf16(s * q)
// and store it into TMEM columns [taddr, taddr + 64) of its lane: column j
// holds k = 2j, 2j + 1 (low half k = 2j).
template <int BITS>
__device__ __forceinline__ void dequant_group_to_tmem(uint32_t cell, int n, uint32_t s2,
                                                      uint32_t taddr) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kLo = 0x43004300u;  // bf16 128
  constexpr uint32_t kHi = 0x45004500u;  // bf16 2048
  if constexpr (BITS == 4) {
    constexpr uint32_t kB4 = 0x43084308u;  // 136
    // lane 4c + t4 holds words kb = 0..3 of k = 32 kb + 8 t4 + 0..7
    uint4 w[4];
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) w[t4] = ld_shared_v4(cell + wt_lane_offset<4>(n, 0, t4));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t r[32];
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int kb = 2 * h + b;
          const uint32_t word = kb == 0 ? w[t4].x : kb == 1 ? w[t4].y : kb == 2 ? w[t4].z : w[t4].w;
          const int col = 4 * (4 * b + t4);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            r[col + j] = bf16x2_mul(bf16x2_sub(lop3_and_or(word >> (4 * j), kMask, kLo), kB4), s2);
        }
      }
      tmem_st_32x32b_x32(taddr + 32 * h, r);
    }
  } else {
    constexpr uint32_t kB8Lo = 0x43004300u;  // 128
    constexpr uint32_t kB8Hi = 0x45084508u;  // 2176 = 2048 + 128
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // half h: lane 4c + t4 holds words wi = 0..3,
      // k = 32 (2h + wi/2) + 8 t4 + 4 (wi & 1) + 0..3
      uint32_t r[32];
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) {
        const uint4 w = ld_shared_v4(cell + wt_lane_offset<8>(n, h, t4));
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          const uint32_t word = wi == 0 ? w.x : wi == 1 ? w.y : wi == 2 ? w.z : w.w;
          const int col = 4 * (4 * (wi >> 1) + t4) + 2 * (wi & 1);
          const uint32_t lo01 = bf16x2_sub(lop3_and_or(word, kMask, kLo), kB8Lo);
          const uint32_t hi01 = bf16x2_sub(lop3_and_or(word >> 4, kMask, kHi), kB8Hi);
          const uint32_t lo23 = bf16x2_sub(lop3_and_or(word >> 8, kMask, kLo), kB8Lo);
          const uint32_t hi23 = bf16x2_sub(lop3_and_or(word >> 12, kMask, kHi), kB8Hi);
          r[col] = bf16x2_mul(bf16x2_add(hi01, lo01), s2);
          r[col + 1] = bf16x2_mul(bf16x2_add(hi23, lo23), s2);
        }
      }
      tmem_st_32x32b_x32(taddr + 32 * h, r);
    }
  }
}

}  // namespace wq

namespace wq {

__device__ __forceinline__ uint2 ld_shared_v2_u32(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Byte offsets of this thread's four 16-byte packed chunks within a cell
// (after the 128-byte swizzle), for half h of the INT8 layout (h = 0 for
// INT4, whose chunks hold both halves): loop-invariant per thread, so a
// kernel computes them once instead of per group.
template <int BITS>
struct LaneOffsets {
  uint32_t o[2][4];
  __device__ __forceinline__ explicit LaneOffsets(int n) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) o[h][t4] = wt_lane_offset<BITS>(n, BITS == 4 ? 0 : h, t4);
  }
};

// Half h (k in [64h, 64h + 64)) of one group of this thread's column:
// bf16(s * q) into the 32 TMEM columns [taddr, taddr + 32) of its lane
// (column j holds k = 64h + 2j, 64h + 2j + 1, the low half k even).  The
// work of one group is split this way between warps, so that a group's
// dequantisation is spread over more warps.  `lo` holds the thread's
// chunk offsets (LaneOffsets).
template <int BITS>
__device__ __forceinline__ void dequant_half_to_tmem(uint32_t cell, const LaneOffsets<BITS>& lo,
                                                     int h, uint32_t s2, uint32_t taddr) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kLo = 0x43004300u;  // bf16 128
  constexpr uint32_t kHi = 0x45004500u;  // bf16 2048
  uint32_t r[32];
  if constexpr (BITS == 4) {
    constexpr uint32_t kB4 = 0x43084308u;  // 136
    // lane 4c + t4 holds words kb = 0..3 (k = 32 kb + 8 t4 + 0..7) in one
    // 16-byte chunk; half h needs kb = 2h, 2h + 1, its bytes 8h .. 8h + 7
    const uint32_t base = cell + 8 * h;
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) {
      const uint2 w = ld_shared_v2_u32(base + lo.o[0][t4]);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t word = b == 0 ? w.x : w.y;
        const int col = 4 * (4 * b + t4);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          r[col + j] = bf16x2_mul(bf16x2_sub(lop3_and_or(word >> (4 * j), kMask, kLo), kB4), s2);
      }
    }
  } else {
    constexpr uint32_t kB8Lo = 0x43004300u;  // 128
    constexpr uint32_t kB8Hi = 0x45084508u;  // 2176 = 2048 + 128
    // half h: lane 4c + t4 holds words wi = 0..3,
    // k = 32 (2h + wi/2) + 8 t4 + 4 (wi & 1) + 0..3
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) {
      const uint4 w = ld_shared_v4(cell + (h ? lo.o[1][t4] : lo.o[0][t4]));
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const uint32_t word = wi == 0 ? w.x : wi == 1 ? w.y : wi == 2 ? w.z : w.w;
        const int col = 4 * (4 * (wi >> 1) + t4) + 2 * (wi & 1);
        const uint32_t lo01 = bf16x2_sub(lop3_and_or(word, kMask, kLo), kB8Lo);
        const uint32_t hi01 = bf16x2_sub(lop3_and_or(word >> 4, kMask, kHi), kB8Hi);
        const uint32_t lo23 = bf16x2_sub(lop3_and_or(word >> 8, kMask, kLo), kB8Lo);
        const uint32_t hi23 = bf16x2_sub(lop3_and_or(word >> 12, kMask, kHi), kB8Hi);
        r[col] = bf16x2_mul(bf16x2_add(hi01, lo01), s2);
        r[col + 1] = bf16x2_mul(bf16x2_add(hi23, lo23), s2);
      }
    }
  }
  tmem_st_32x32b_x32(taddr, r);
}

}  // namespace wq
