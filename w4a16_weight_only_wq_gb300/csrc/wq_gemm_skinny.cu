// wq_gemm_skinny.cu -- tensor-memory W4A16 / W8A16 GEMM for M <= 16.
//
// Y[M,N] = X[M,K] . (s (.) q)[K,N] for the verifier's 16-token block
// ("Quantize the Target, Quantize the Drafter": the INT4 target verifies an
// anchor plus 15 drafted tokens in one forward).  The product is computed
// transposed, Y^T = W^T . X^T, so that the weights are the 128-row operand
// of tcgen05.mma and live in tensor memory, and the 16 tokens are its
// N = 16 operand in shared memory:
//
//  * A CTA owns 128 output columns (two packed cells) and a contiguous
//    range of 128-deep groups; a cluster of `cs` CTAs splits one column
//    tile's K range and reduces through distributed shared memory.
//  * Producer warp: per group, the two packed cells by TMA (the packed
//    buffer seen as rows of 128 bytes, with the 128-byte swizzle so that the
//    dequant threads' reads spread over the banks) and 128 scales by bulk
//    copy, both issued before the programmatic-launch dependency resolves,
//    then the group's X tile [16 tokens x 128 k] by TMA with the 128-byte
//    swizzle (after it), into a ring of shared-memory slots.
//  * Dequant warps: one LOP3 per pair of codes makes the exact bf16 values
//    136 + q (INT4) or the planes 128 + lo and 2048 + 16 hi (INT8); each
//    thread owns one weight column (a TMEM lane) and stores 64 k of it with
//    one tcgen05.st.  No bf16 arithmetic and no rounding happen here.
//  * MMA thread: per group, 8 (INT4) or 16 (INT8) MMAs of the codes plus 8
//    MMAs of a constant -136 (-2304) matrix against the same X tile, which
//    removes the bias exactly; each group accumulates into its own small
//    TMEM accumulator [128 columns x 16 tokens].
//  * Accumulate warps: read a finished group's accumulator (tcgen05.ld) and
//    add s[group, n] * value into fp32 registers, then release it.
//  Every wait is bounded; an abort drains copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tcgen05.cuh"

namespace wq {
namespace {

constexpr int kTok = 16;             // tokens per CTA (the MMA's N)
constexpr int kCols = 128;           // output columns per CTA (the MMA's M)
constexpr int kXStage = kTok * 128;  // one k64 X tile: 16 rows x 128 B (swizzled)
constexpr int kDequantWarps = 8;     // two per TMEM lane quadrant (k halves)
constexpr int kAccWarps = 4;         // one per TMEM lane quadrant
constexpr int kFirstDequantWarp = 2;
constexpr int kFirstAccWarp = kFirstDequantWarp + kDequantWarps;  // 10
constexpr int kThreads = (kFirstAccWarp + kAccWarps) * 32;         // 448
constexpr int kTD = 4;               // TMEM accumulators in flight
constexpr uint32_t kTmemCols = 512;

template <int BITS>
struct SkCfg {
  static constexpr int kCellWords = BITS == 4 ? 1024 : 2048;
  static constexpr int kCellBytes = kCellWords * 4;
  static constexpr int kPlanes = BITS == 4 ? 1 : 2;  // TMEM A planes per stage
  static constexpr int kTA = BITS == 4 ? 4 : 2;      // groups of A in TMEM
  static constexpr int kAColsPerGroup = 2 * 32 * kPlanes;
  static constexpr int kBiasCol = kTA * kAColsPerGroup;  // 256
  static constexpr int kDCol = kBiasCol + 16;            // 272
  // slot: [X: 2 stages x 2 KiB][cells: 2 x cell][scales: 128 x bf16], 1 KiB aligned
  static constexpr int kSlotX = 0;
  static constexpr int kSlotW = 2 * kXStage;
  static constexpr int kSlotS = kSlotW + 2 * kCellBytes;
  static constexpr int kSlot = ((kSlotS + kCols * 2) + 1023) / 1024 * 1024;
  static constexpr uint32_t kBias2 = BITS == 4 ? 0xC308C308u    // -136
                                               : 0xC510C510u;   // -2304
};

struct SkParams {
  const uint32_t* Wp;
  const uint16_t* S;
  __nv_bfloat16* Y;
  int M, N, K, G, cs, slots;
  KernelDiag diag;
};

__host__ __device__ constexpr int sk_fixed_bytes() {
  // part [16][128] fp32 + barriers + flags + alignment slack
  return kTok * kCols * 4 + 64 * 8 + 64 + 1024;
}

// Byte offset, within a slot's cells, of the 16-byte packed lane 4c + t4
// that holds k half `h` of column `n` (the bytes of half h only, for INT4),
// as the 128-byte swizzled TMA load placed it: 16-byte chunk `ch` of 128-byte
// row `row` sits at chunk position ch ^ (row % 8).
template <int BITS>
__device__ __forceinline__ uint32_t sk_lane_offset(int n, int h, int t4) {
  using C = SkCfg<BITS>;
  const int ci = n >> 6, j8 = (n >> 3) & 7, c = n & 7;
  const int row = BITS == 4 ? j8 * 4 + (c >> 1) : (j8 * 2 + h) * 4 + (c >> 1);
  const int ch = (4 * (c & 1) + t4) ^ (row & 7);
  return ci * C::kCellBytes + row * 128 + ch * 16 + (BITS == 4 ? 8 * h : 0);
}

// Write the k64 half `h` of column `n` (this thread's TMEM lane) of the
// packed group at `cells` into TMEM columns [col, col + 32) (INT4) or
// [col, col + 64) (INT8: low plane, then high plane).  Column j of a stage
// holds the bf16 pair for k = 2j, 2j + 1 of the half.  off[t4] =
// sk_lane_offset(n, h, t4).
template <int BITS>
__device__ __forceinline__ void dequant_to_tmem(uint32_t cells, const uint32_t (&off)[4],
                                                uint32_t taddr) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kLo = 0x43004300u;  // bf16 128
  constexpr uint32_t kHi = 0x45004500u;  // bf16 2048
  if constexpr (BITS == 4) {
    // lane 4c + t4 holds words kb = 0..3 (k = 32 kb + 8 t4 + 0..7); this
    // half needs kb = 2h, 2h + 1.
    uint32_t r[32];
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) {
      const uint2 w = ld_shared_v2(cells + off[t4]);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t word = b ? w.y : w.x;
        const int col = 4 * (4 * b + t4);  // k8 chunk (b, t4) -> 4 columns
        r[col + 0] = lop3_and_or(word, kMask, kLo);
        r[col + 1] = lop3_and_or(word >> 4, kMask, kLo);
        r[col + 2] = lop3_and_or(word >> 8, kMask, kLo);
        r[col + 3] = lop3_and_or(word >> 12, kMask, kLo);
      }
    }
    tmem_st_32x32b_x32(taddr, r);
  } else {
    // half h: lane 4c + t4 holds words wi = 0..3,
    // k = 32 (2h + wi/2) + 8 t4 + 4 (wi & 1) + 0..3
    uint32_t lo[32], hi[32];
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) {
      const uint4 w = ld_shared_v4(cells + off[t4]);
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const uint32_t word = wi == 0 ? w.x : wi == 1 ? w.y : wi == 2 ? w.z : w.w;
        const int col = 4 * (4 * (wi >> 1) + t4) + 2 * (wi & 1);
        lo[col + 0] = lop3_and_or(word, kMask, kLo);
        hi[col + 0] = lop3_and_or(word >> 4, kMask, kHi);
        lo[col + 1] = lop3_and_or(word >> 8, kMask, kLo);
        hi[col + 1] = lop3_and_or(word >> 12, kMask, kHi);
      }
    }
    tmem_st_32x32b_x32(taddr, lo);
    tmem_st_32x32b_x32(taddr + 32, hi);
  }
}


__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, uint32_t v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(taddr),
      "r"(v)
      : "memory");
}

// Bounded wait that gives up as soon as another role has aborted.
__device__ __forceinline__ bool sk_wait(uint64_t* bar, uint32_t parity, const KernelDiag& d,
                                        volatile int* abort_flag, uint32_t hint_ns = 0) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (hint_ns ? mbar_try_wait_sleep(a, parity, hint_ns) : mbar_try_wait(a, parity))
        return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > d.wait_limit_ns) {
      atomicMax(d.err, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                   const SkParams p) {
  using C = SkCfg<BITS>;
  constexpr int kTA = C::kTA;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

  const int cs = p.cs, D = p.slots;
  const int tile = blockIdx.x / cs;
  const int rank = blockIdx.x % cs;  // == %cluster_ctarank for cluster (cs,1,1)
  const int g0 = (p.G * rank) / cs;
  const int ng = (p.G * (rank + 1)) / cs - g0;
  const int n0 = tile * kCols;
  const int cells = min(2, (p.N - n0) / 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Same offsets in every CTA of the cluster (`part` is read remotely).
  uint8_t* slots = smem;
  float* part = reinterpret_cast<float*>(smem + D * C::kSlot);  // [16 tokens][128 cols]
  uint64_t* bars = reinterpret_cast<uint64_t*>(part + kTok * kCols);
  uint64_t* s_full = bars;                // [D] slot landed
  uint64_t* s_empty = s_full + D;         // [D] MMA done + scales read
  uint64_t* a_full = s_empty + D;         // [kTA] group's codes in TMEM
  uint64_t* a_empty = a_full + kTA;       // [kTA] MMA done with them
  uint64_t* d_full = a_empty + kTA;       // [kTD] group accumulator ready
  uint64_t* d_empty = d_full + kTD;       // [kTD] accumulator read
  uint64_t* never_bar = d_empty + kTD;    // test hook
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < D; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 1 + kAccWarps);
    }
    for (int i = 0; i < kTA; ++i) {
      mbar_init(&a_full[i], kDequantWarps);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kTD; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], kAccWarps);
    }
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  int issued = 0, mma_last = -1;
  float acc[kTok];
#pragma unroll
  for (int m = 0; m < kTok; ++m) acc[m] = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------- producer ---
    if (lane != 0) pdl_wait_primary();
    if (lane == 0) {
      prefetch_tensor_map(&tmx);
      prefetch_tensor_map(&tmw);
      const int first = min(ng, D);
      auto issue_w = [&](int i, int slot) {
        uint8_t* dst = slots + slot * C::kSlot;
        const int g = g0 + i;
        mbar_arrive_expect_tx(&s_full[slot], 2 * kXStage + cells * C::kCellBytes + cells * 128);
        for (int ci = 0; ci < cells; ++ci)
          tma_load_2d(dst + C::kSlotW + ci * C::kCellBytes, &tmw, 0,
                      ((n0 / 64 + ci) * p.G + g) * (C::kCellBytes / 128), &s_full[slot]);
        bulk_g2s(dst + C::kSlotS, p.S + static_cast<size_t>(g) * p.N + n0, cells * 128,
                 &s_full[slot]);
      };
      auto issue_x = [&](int i, int slot) {
        uint8_t* dst = slots + slot * C::kSlot;
        const int k = (g0 + i) * 128;
        tma_load_2d(dst + C::kSlotX, &tmx, k, 0, &s_full[slot]);
        tma_load_2d(dst + C::kSlotX + kXStage, &tmx, k + 64, 0, &s_full[slot]);
      };
      // weights first: they do not depend on the preceding kernel
      for (int i = 0; i < first; ++i) issue_w(i, i);
      pdl_wait_primary();
      for (int i = 0; i < first; ++i) issue_x(i, i);
      issued = first;
      for (int i = D; i < ng; ++i) {
        const int slot = i % D;
        if (!sk_wait(&s_empty[slot], ((i / D) - 1) & 1, p.diag, abort_flag)) break;
        issue_w(i, slot);
        issue_x(i, slot);
        issued = i + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer ---
    pdl_wait_primary();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kCols, kTok);
      for (int i = 0; i < ng; ++i) {
        const int slot = i % D, ga = i % kTA, d = i % kTD;
        // Test hook 2: halfway through, wait on a barrier nothing completes,
        // so that the give-up-and-drain path runs with copies in flight.
        const bool hook = p.diag.force_timeout == 2 && i == ng / 2;
        if (!sk_wait(hook ? never_bar : &s_full[slot], hook ? 0u : (i / D) & 1, p.diag,
                     abort_flag) ||
            !sk_wait(&a_full[ga], (i / kTA) & 1, p.diag, abort_flag) ||
            (i >= kTD && !sk_wait(&d_empty[d], ((i / kTD) - 1) & 1, p.diag, abort_flag)))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + C::kDCol + d * kTok;
        const uint32_t a_tmem = tmem_base + ga * C::kAColsPerGroup;
        const uint32_t x0 = smem_addr(slots + slot * C::kSlot + C::kSlotX);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t b_desc = smem_desc_sw128(x0 + h * kXStage);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int pl = 0; pl < C::kPlanes; ++pl)
              umma_bf16_ts(d_tmem, a_tmem + h * 32 * C::kPlanes + pl * 32 + 8 * j,
                           b_desc + 2 * j, idesc, (h | j | pl) != 0);
            // remove the code bias exactly: D += (-bias) * X
            umma_bf16_ts(d_tmem, tmem_base + C::kBiasCol, b_desc + 2 * j, idesc, 1);
          }
        }
        umma_commit(&a_empty[ga]);
        umma_commit(&s_empty[slot]);
        umma_commit(&d_full[d]);
        mma_last = i;
      }
    }
  } else if (warp < kFirstAccWarp) {
    // ------------------------------------------------- dequant warps ---
    // TMEM lane quadrant = warp % 4; warps 2-5 take the first k64 half of
    // every group, warps 6-9 the second.
    pdl_wait_primary();
    const int q = warp & 3, h = (warp - kFirstDequantWarp) >> 2;
    const int n = 32 * q + lane;  // this thread's weight column (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    uint32_t off[4];
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) off[t4] = sk_lane_offset<BITS>(n, h, t4);
    if (h == 0) {
      tmem_st_32x32b_x8(tmem_base + lane_addr + C::kBiasCol, C::kBias2);
    }
    for (int i = 0; i < ng; ++i) {
      const int slot = i % D, ga = i % kTA;
      if (!sk_wait(&s_full[slot], (i / D) & 1, p.diag, abort_flag) ||
          (i >= kTA && !sk_wait(&a_empty[ga], ((i / kTA) - 1) & 1, p.diag, abort_flag)))
        break;
      dequant_to_tmem<BITS>(smem_addr(slots + slot * C::kSlot + C::kSlotW), off,
                            tmem_base + lane_addr + ga * C::kAColsPerGroup + h * 32 * C::kPlanes);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[ga]);
    }
  } else {
    // ------------------------------------------------ accumulate warps ---
    pdl_wait_primary();  // these warps store Y
    const int q = warp & 3;
    const int n = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    for (int i = 0; i < ng; ++i) {
      const int slot = i % D, d = i % kTD;
      if (!sk_wait(&s_full[slot], (i / D) & 1, p.diag, abort_flag, 2000)) break;
      const float sc = __uint_as_float(
          static_cast<uint32_t>(ld_shared_u16(smem_addr(slots + slot * C::kSlot + C::kSlotS) +
                                              2 * n))
          << 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[slot]);
      if (!sk_wait(&d_full[d], (i / kTD) & 1, p.diag, abort_flag, 2000)) break;
      tc_fence_after();
      uint32_t v[kTok];
      tmem_ld_32x32b_x16(tmem_base + lane_addr + C::kDCol + d * kTok, v);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[d]);
#pragma unroll
      for (int m = 0; m < kTok; ++m) acc[m] = fmaf(sc, __uint_as_float(v[m]), acc[m]);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    KernelDiag drain = p.diag;
    if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
    if (warp == 0 && lane == 0) {
      for (int slot = 0; slot < D && slot < issued; ++slot) {
        const int last = slot + ((issued - 1 - slot) / D) * D;
        mbar_wait_bounded(&s_full[slot], (last / D) & 1, drain);
      }
    }
    if (warp == 1 && lane == 0 && mma_last >= 0)
      mbar_wait_bounded(&a_empty[mma_last % kTA], (mma_last / kTA) & 1, drain);
    __syncthreads();
  }

  // CTA partial [16 tokens][128 columns] -> Y (cs == 1) or the cluster.
  const int rows = min(kTok, p.M);
  if (warp >= kFirstAccWarp) {
    const int n = 32 * (warp & 3) + lane;
    if (cs == 1) {
      if (n0 + n < p.N) {
#pragma unroll
        for (int m = 0; m < kTok; ++m)
          if (m < rows)
            p.Y[static_cast<size_t>(m) * p.N + n0 + n] = __float2bfloat16_rn(acc[m]);
      }
    } else {
#pragma unroll
      for (int m = 0; m < kTok; ++m) part[m * kCols + n] = acc[m];
    }
  }
  if (cs > 1) {
    cluster_sync();
    const int ncol = cells * 64;
    const int total = rows * kCols;
    const int e_end = (total * (rank + 1)) / cs;
    for (int e = (total * rank) / cs + threadIdx.x; e < e_end; e += kThreads) {
      const int m = e / kCols, n = e % kCols;
      if (n >= ncol) continue;
      float v = 0.f;
      for (int r = 0; r < cs; ++r) v += dsmem_ld_f32(dsmem_map(part + e, r));
      p.Y[static_cast<size_t>(m) * p.N + n0 + n] = __float2bfloat16_rn(v);
    }
    cluster_sync();  // keep `part` alive until every peer has read it
  }
  pdl_launch_dependents();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side ---
typedef CUresult (*SkEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                               const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                               const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

SkEncodeFn sk_encode_fn() {
  static SkEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<SkEncodeFn>(f);
  });
  return fn;
}

template <int BITS>
struct SkInit {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
  int max_dyn[64] = {};
  cudaError_t ensure(int device, int* out) {
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> lk(mu);
      if (!(done.load() & bit)) {
        int optin = 0;
        cudaError_t e =
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_skinny_kernel<BITS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
        max_dyn[device & 63] = optin;
        done.fetch_or(bit, std::memory_order_release);
      }
    }
    *out = max_dyn[device & 63];
    return cudaSuccess;
  }
};
SkInit<4> g_sk4;
SkInit<8> g_sk8;

int sk_split(int64_t K, int64_t N, int num_sms, int hint) {
  const int64_t tiles = (N + kCols - 1) / kCols, G = K / 128;
  if (hint > 0) return (hint <= 8 && hint <= G) ? hint : -1;
  int best = 1;
  for (int cs = 1; cs <= 8 && cs <= G; ++cs)
    if (tiles * cs <= num_sms) best = cs;
  return best;
}

}  // namespace

cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t stream) {
  if (a.M > kTok) return cudaErrorNotSupported;
  // TMA coordinates are signed 32-bit: the packed buffer's 128-byte rows
  // must be indexable.
  if ((a.bits == 4 ? a.K * a.N / 256 : a.K * a.N / 128) > INT32_MAX) return cudaErrorNotSupported;
  SkEncodeFn enc = sk_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int cs = sk_split(a.K, a.N, a.num_sms, a.split_hint);
  if (cs < 0) return cudaErrorNotSupported;
  int max_dyn = 0;
  cudaError_t e = a.bits == 4 ? g_sk4.ensure(a.device, &max_dyn) : g_sk8.ensure(a.device, &max_dyn);
  if (e != cudaSuccess) return e;

  const int G = static_cast<int>(a.K / 128);
  const int ng_max = (G + cs - 1) / cs;
  const int slot = a.bits == 4 ? SkCfg<4>::kSlot : SkCfg<8>::kSlot;
  int D = (max_dyn - sk_fixed_bytes()) / slot;
  if (D > ng_max) D = ng_max;
  if (D > 20) D = 20;
  if (D < 1) return cudaErrorNotSupported;
  // At least ~60% of an SM's shared memory, so that one CTA (and its 512
  // TMEM columns) occupies an SM and no two CTAs of a cluster share one.
  int smem = D * slot + sk_fixed_bytes();
  const int floor_bytes = (max_dyn * 6) / 10;
  if (smem < floor_bytes) smem = floor_bytes;

  // X as a 2-D bf16 tensor [M rows, K cols]; box 64 x 16 with the 128-byte
  // swizzle; rows past M read as zeros.
  CUtensorMap tmx;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.M)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(a.K) * 2};
  const cuuint32_t box[2] = {64, kTok};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.X), gdim,
                   gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  // The packed weights as a 2-D u32 tensor [K N / 256 (INT4) or K N / 128
  // (INT8) rows, 32 words]; one box is one packed cell.
  CUtensorMap tmw;
  const int64_t words = a.bits == 4 ? a.K * a.N / 8 : a.K * a.N / 4;
  const cuuint64_t wdim[2] = {32, static_cast<cuuint64_t>(words / 32)};
  const cuuint64_t wstride[1] = {128};
  const cuuint32_t wbox[2] = {32, static_cast<cuuint32_t>(
                                      (a.bits == 4 ? SkCfg<4>::kCellBytes : SkCfg<8>::kCellBytes) / 128)};
  r = enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(a.Wp), wdim, wstride, wbox,
          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  SkParams p;
  p.Wp = a.Wp;
  p.S = static_cast<const uint16_t*>(a.S);
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.G = G;
  p.cs = cs;
  p.slots = D;
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;

  const int tiles = static_cast<int>((a.N + kCols - 1) / kCols);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = cs;
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  if (a.pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  if (a.bits == 4) return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<4>, tmx, tmw, p);
  return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<8>, tmx, tmw, p);
}

}  // namespace wq
