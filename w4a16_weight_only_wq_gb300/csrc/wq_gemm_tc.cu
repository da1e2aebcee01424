// wq_gemm_tc.cu -- tensor-core (tcgen05) W4A16 / W8A16 GEMM for large M.
//
// Y[M,N] = X[M,K] . (s (.) q)[K,N] for prefill-sized M ("Quantize the
// Target, Quantize the Drafter": the INT4 target served as W4A16; the Long
// setting's 8,192-token prompt).  Here the product is a dense contraction,
// so it runs on the 5th-generation tensor cores:
//
//  * Persistent CTAs walk 128 x 256 output tiles (M fastest, so CTAs that
//    run together share a weight tile in L2).  K is consumed 64 at a time.
//  * Producer warp: TMA (tensor map, 128-byte swizzle) loads the X tile
//    [128 rows x 64 k] of every k-step, and bulk-copies the packed cells of
//    the 256 columns and their scales once per 128-deep group.
//  * Eight dequant warps turn the packed codes into bf16 s*q (one rounding)
//    and store them in the canonical 128-byte-swizzled K-major layout the
//    MMA reads, then hand the stage to the MMA with an mbarrier.
//  * One thread issues tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> f32)
//    into a TMEM accumulator; two accumulators alternate so the epilogue of
//    one tile overlaps the main loop of the next.
//  * Four epilogue warps read TMEM (tcgen05.ld), round to bf16 and store Y.
//  Every mbarrier wait is bounded; a wait that runs out flags the error
//  word, stops the pipeline, lets in-flight copies and MMAs finish and frees
//  TMEM before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tcgen05.cuh"
#include "wq_tensor_map.h"

namespace wq {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kAStages = 4;      // k64 stages of X (TMA)
constexpr int kBStages = 4;      // k64 stages of dequantized W (even: a group per pass)
constexpr int kEpiWarps = 4;
constexpr int kFirstDequantWarp = 2;
constexpr int kABytes = kBM * kBK * 2;   // 16 KiB
constexpr int kBdBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kTmemCols = 2 * kBN;  // two accumulators

template <int BITS>
struct TcCfg {
  // INT4: two dequant threads per column (each takes two of its four
  // 16-byte lanes); INT8 (more registers per thread): one.
  static constexpr int kDequantWarps = BITS == 4 ? 16 : 8;
  static constexpr int kFirstEpiWarp = kFirstDequantWarp + kDequantWarps;
  static constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;
  static constexpr int kQStages = BITS == 4 ? 2 : 1;          // packed groups in flight
  static constexpr int kCellWords = BITS == 4 ? 1024 : 2048;  // 64 cols x 128 k
  static constexpr int kCellBytes = kCellWords * 4;
  static constexpr int kQBytes = 4 * kCellBytes + kBN * 2;    // 4 cells + scales
  static constexpr int kOffA = 0;
  static constexpr int kOffBd = kOffA + kAStages * kABytes;
  static constexpr int kOffQ = kOffBd + kBStages * kBdBytes;
  static constexpr int kOffBar = kOffQ + kQStages * kQBytes;
  static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kQStages + 4 + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + align slack
};

struct TcParams {
  const uint32_t* Wp;
  const uint16_t* S;
  __nv_bfloat16* Y;
  int M, N, K, G;
  int mt, nt;  // tile counts
  KernelDiag diag;
};

// Dequantize one packed 128-deep group (4 cells of 64 columns + 256 scales
// at `q_base`) into the two bf16 k64 stages at `bd0` (k 0..63) and `bd1`
// (k 64..127): 256 rows of 128 bytes, 16-byte chunk j of row r stored at
// chunk j ^ (r % 8) (the 128-byte-swizzled K-major layout).  One thread per
// column n = row.  The row's packed words are 64 (INT4) or 2 x 64 (INT8)
// contiguous bytes of the cell, four 16-byte lanes t4 = 0..3; lane
// t4 = i ^ (c/2) is handled in step i so that both the loads and the
// chunk stores (at chunk ^ c) of a quarter-warp fall on distinct banks.
template <int BITS>
__device__ __forceinline__ void dequant_group(uint32_t q_base, uint32_t bd0, uint32_t bd1,
                                              int n, int part, bool valid) {
  using C = TcCfg<BITS>;
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kLo = 0x43004300u;  // bf16 128
  constexpr uint32_t kHi = 0x45004500u;  // bf16 2048
  if (!valid) return;
  const int ci = n >> 6, j8 = (n >> 3) & 7, c = n & 7;
  const uint32_t s1 = ld_shared_u16(q_base + 4 * C::kCellBytes + n * 2);
  const uint32_t s2 = s1 | (s1 << 16);
  const uint32_t row0 = bd0 + (n >> 3) * 1024 + c * 128;
  const uint32_t row1 = bd1 + (n >> 3) * 1024 + c * 128;
  const int rot = c >> 1;
  if constexpr (BITS == 4) {
    constexpr uint32_t kB4 = 0x43084308u;  // 136
    // lane 4c + t4 holds words kb = 0..3: k = 32 kb + 8 t4 + 0..7
    // this thread takes steps i = 2 part, 2 part + 1
    const uint32_t base = q_base + ci * C::kCellBytes + (j8 * 32 + 4 * c) * 16;
    uint4 w[2];
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) w[ii] = ld_shared_v4(base + ((2 * part + ii) ^ rot) * 16);
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const int i = ii;
      const int t4 = (2 * part + ii) ^ rot;
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const uint32_t word = kb == 0 ? w[i].x : kb == 1 ? w[i].y : kb == 2 ? w[i].z : w[i].w;
        const uint32_t q0 = bf16x2_sub(lop3_and_or(word, kMask, kLo), kB4);
        const uint32_t q1 = bf16x2_sub(lop3_and_or(word >> 4, kMask, kLo), kB4);
        const uint32_t q2 = bf16x2_sub(lop3_and_or(word >> 8, kMask, kLo), kB4);
        const uint32_t q3 = bf16x2_sub(lop3_and_or(word >> 12, kMask, kLo), kB4);
        const int chunk = 4 * (kb & 1) + t4;
        st_shared_v4((kb < 2 ? row0 : row1) + ((chunk ^ c) << 4), bf16x2_mul(q0, s2),
                     bf16x2_mul(q1, s2), bf16x2_mul(q2, s2), bf16x2_mul(q3, s2));
      }
    }
  } else {
    constexpr uint32_t kB8Lo = 0x43004300u;  // 128
    constexpr uint32_t kB8Hi = 0x45084508u;  // 2176
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // half h: lane 4c + t4 holds words wi = 0..3,
      // k = 32 (2h + wi/2) + 8 t4 + 4 (wi & 1) + 0..3
      const uint32_t base = q_base + ci * C::kCellBytes + ((j8 * 2 + h) * 32 + 4 * c) * 16;
      uint4 w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = ld_shared_v4(base + (i ^ rot) * 16);
      const uint32_t row = h == 0 ? row0 : row1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t4 = i ^ rot;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          uint32_t v[4];
#pragma unroll
          for (int hw = 0; hw < 2; ++hw) {
            const int wi = 2 * b + hw;
            const uint32_t word = wi == 0 ? w[i].x : wi == 1 ? w[i].y : wi == 2 ? w[i].z : w[i].w;
            const uint32_t lo01 = bf16x2_sub(lop3_and_or(word, kMask, kLo), kB8Lo);
            const uint32_t hi01 = bf16x2_sub(lop3_and_or(word >> 4, kMask, kHi), kB8Hi);
            const uint32_t lo23 = bf16x2_sub(lop3_and_or(word >> 8, kMask, kLo), kB8Lo);
            const uint32_t hi23 = bf16x2_sub(lop3_and_or(word >> 12, kMask, kHi), kB8Hi);
            v[2 * hw] = bf16x2_mul(bf16x2_add(hi01, lo01), s2);
            v[2 * hw + 1] = bf16x2_mul(bf16x2_add(hi23, lo23), s2);
          }
          const int chunk = 4 * b + t4;
          st_shared_v4(row + ((chunk ^ c) << 4), v[0], v[1], v[2], v[3]);
        }
      }
    }
  }
}

// Bounded wait that also gives up as soon as another role has aborted.
// `hint_ns` lets a long waiter sleep inside try_wait rather than spin.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              const KernelDiag& d, volatile int* abort_flag,
                                              uint32_t hint_ns = 0) {
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
__global__ void __launch_bounds__(TcCfg<BITS>::kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmx, const TcParams p) {
  using C = TcCfg<BITS>;
  constexpr int kQStages = C::kQStages;
  constexpr int kDequantWarps = C::kDequantWarps;
  constexpr int kFirstEpiWarp = C::kFirstEpiWarp;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment (of the shared-window offset) for the swizzled stages.
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* a_full = bars;                       // [kAStages] X tile landed
  uint64_t* a_empty = a_full + kAStages;         // [kAStages] MMA done with X tile
  uint64_t* bd_full = a_empty + kAStages;        // [kBStages] W tile dequantized
  uint64_t* bd_empty = bd_full + kBStages;       // [kBStages] MMA done with W tile
  uint64_t* q_full = bd_empty + kBStages;        // [kQStages] packed group landed
  uint64_t* q_empty = q_full + kQStages;         // [kQStages] packed group consumed
  uint64_t* acc_full = q_empty + kQStages;       // [2] accumulator ready
  uint64_t* acc_empty = acc_full + 2;            // [2] accumulator drained
  uint64_t* never_bar = acc_empty + 2;           // test hook
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.K / kBK;
  const int tiles = p.mt * p.nt;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&bd_full[i], kDequantWarps);
      mbar_init(&bd_empty[i], 1);
    }
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kDequantWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
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
  // The next kernel may launch now: it reads nothing this grid writes
  // before this grid completes.
  pdl_launch_dependents();

  // X and Y may belong to the preceding kernel on the stream.
  pdl_wait_primary();
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  // Progress counters used to drain after an abort.
  int a_issued = 0, q_issued = 0, mma_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------- producer ---
    if (lane == 0) {
      prefetch_tensor_map(&tmx);
      int it = 0, iq = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        const int m0 = (t % p.mt) * kBM, n0 = (t / p.mt) * kBN;
        const int cells = min(4, (p.N - n0) / 64);
        for (int kk = 0; kk < nk; ++kk, ++it) {
          if ((kk & 1) == 0) {  // first half of a group: fetch the packed group
            const int q = iq % kQStages, g = kk >> 1;
            if (iq >= kQStages &&
                !wait_or_abort(&q_empty[q], ((iq / kQStages) - 1) & 1, p.diag, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* qd = smem + C::kOffQ + q * C::kQBytes;
            mbar_arrive_expect_tx(&q_full[q], cells * C::kCellBytes + cells * 128);
            for (int ci = 0; ci < cells; ++ci)
              bulk_g2s(qd + ci * C::kCellBytes,
                       p.Wp + (static_cast<size_t>(n0 / 64 + ci) * p.G + g) * C::kCellWords,
                       C::kCellBytes, &q_full[q]);
            bulk_g2s(qd + 4 * C::kCellBytes, p.S + static_cast<size_t>(g) * p.N + n0,
                     cells * 128, &q_full[q]);
            ++iq;
            q_issued = iq;
          }
          const int sa = it % kAStages;
          if (it >= kAStages &&
              !wait_or_abort(&a_empty[sa], ((it / kAStages) - 1) & 1, p.diag, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&a_full[sa], kABytes);
          tma_load_2d(smem + C::kOffA + sa * kABytes, &tmx, kk * kBK, m0, &a_full[sa]);
          a_issued = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      int it = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++tl) {
        const int b = tl & 1;
        if (tl >= 2 && !wait_or_abort(&acc_empty[b], ((tl >> 1) - 1) & 1, p.diag, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kBN;
        for (int kk = 0; kk < nk; ++kk, ++it) {
          const int sa = it % kAStages, sb = it % kBStages;
          if (!wait_or_abort(&a_full[sa], (it / kAStages) & 1, p.diag, abort_flag) ||
              !wait_or_abort(&bd_full[sb], (it / kBStages) & 1, p.diag, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = smem_desc_sw128(smem_addr(smem + C::kOffA + sa * kABytes));
          const uint64_t b_desc = smem_desc_sw128(smem_addr(smem + C::kOffBd + sb * kBdBytes));
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)  // +32 bytes per K=16 step
            umma_bf16(d_tmem, a_desc + 2 * j, b_desc + 2 * j, idesc, (kk | j) != 0);
          umma_commit(&a_empty[sa]);
          umma_commit(&bd_empty[sb]);
          mma_issued = it + 1;
        }
        if (ok) umma_commit(&acc_full[b]);
      }
    }
  } else if (warp < kFirstEpiWarp) {
    // ------------------------------------------------- dequant warps ---
    // One (INT8) or two (INT4) threads per column of the 256-column tile; a
    // whole group (two k64 stages) per pass.
    const int dwi = warp - kFirstDequantWarp;
    const int n = (dwi & 7) * 32 + lane;
    const int part = dwi >> 3;
    int it = 0, iq = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
      const int n0 = (t / p.mt) * kBN;
      const bool valid = n0 + n < p.N;
      for (int kk = 0; kk < nk; kk += 2, it += 2, ++iq) {
        const int s0 = it % kBStages, s1 = (it + 1) % kBStages, q = iq % kQStages;
        if (!wait_or_abort(&q_full[q], (iq / kQStages) & 1, p.diag, abort_flag) ||
            (it >= kBStages &&
             (!wait_or_abort(&bd_empty[s0], ((it / kBStages) - 1) & 1, p.diag, abort_flag) ||
              !wait_or_abort(&bd_empty[s1], (((it + 1) / kBStages) - 1) & 1, p.diag,
                             abort_flag)))) {
          ok = false;
          break;
        }
        dequant_group<BITS>(smem_addr(smem + C::kOffQ + q * C::kQBytes),
                            smem_addr(smem + C::kOffBd + s0 * kBdBytes),
                            smem_addr(smem + C::kOffBd + s1 * kBdBytes), n, part, valid);
        fence_proxy_async_smem();  // generic stores -> tensor-core reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bd_full[s0]);
          mbar_arrive(&bd_full[s1]);
          mbar_arrive(&q_empty[q]);
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps ---
    const int lane_base = 32 * (warp & 3);  // TMEM lanes this warp may read
    int tl = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
      const int b = tl & 1;
      if (!wait_or_abort(&acc_full[b], (tl >> 1) & 1, p.diag, abort_flag, 20000)) break;
      tc_fence_after();
      const int m0 = (t % p.mt) * kBM, n0 = (t / p.mt) * kBN;
      const int m = m0 + lane_base + lane;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        if (n0 + 32 * c >= p.N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(lane_base) << 16) + b * kBN + 32 * c, r);
        tmem_ld_wait();
        if (m < p.M) {
          __nv_bfloat16* dst = p.Y + static_cast<size_t>(m) * p.N + n0 + 32 * c;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_global_v4(dst + 8 * v,
                         pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                         pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                         pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                         pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }

  // Roles that ran on one lane (MMA issue, copy issue) rejoin their warp
  // before the block-wide barrier, which a diverged warp must not reach.
  __syncwarp();
  __syncthreads();
  if (*abort_flag) {
    // Let every issued copy land and every issued MMA finish (bounded, at
    // least 1 s) before the shared memory and TMEM are released.  The
    // latest phase of a barrier covers the earlier ones.
    KernelDiag drain = p.diag;
    if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < kAStages && s < a_issued; ++s) {
        const int last = s + ((a_issued - 1 - s) / kAStages) * kAStages;
        mbar_wait_bounded(&a_full[s], (last / kAStages) & 1, drain);
      }
      for (int q = 0; q < kQStages && q < q_issued; ++q) {
        const int last = q + ((q_issued - 1 - q) / kQStages) * kQStages;
        mbar_wait_bounded(&q_full[q], (last / kQStages) & 1, drain);
      }
    }
    if (warp == 1 && lane == 0 && mma_issued > 0) {
      const int last = mma_issued - 1;
      mbar_wait_bounded(&a_empty[last % kAStages], (last / kAStages) & 1, drain);
    }
    __syncwarp();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side ---

template <int BITS>
struct TcInit {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
  cudaError_t ensure(int device) {
    const uint64_t bit = 1ull << (device & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu);
    if (done.load() & bit) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BITS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcCfg<BITS>::kSmem);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
  }
};
TcInit<4> g_tc4;
TcInit<8> g_tc8;

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t stream) {
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  cudaError_t e = a.bits == 4 ? g_tc4.ensure(a.device) : g_tc8.ensure(a.device);
  if (e != cudaSuccess) return e;

  // X as a 2-D bf16 tensor [M rows, K cols]; box 64 x 128 with the 128-byte
  // swizzle the MMA descriptors expect; rows past M read as zeros.
  CUtensorMap tmx;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.M)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(a.K) * 2};
  const cuuint32_t box[2] = {kBK, kBM};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.X), gdim,
                   gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  TcParams p;
  p.Wp = a.Wp;
  p.S = static_cast<const uint16_t*>(a.S);
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.G = static_cast<int>(a.K / 128);
  p.mt = static_cast<int>((a.M + kBM - 1) / kBM);
  p.nt = static_cast<int>((a.N + kBN - 1) / kBN);
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;

  const int tiles = p.mt * p.nt;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles < a.num_sms ? tiles : a.num_sms));
  cfg.blockDim = dim3(a.bits == 4 ? TcCfg<4>::kThreads : TcCfg<8>::kThreads);
  cfg.dynamicSmemBytes = a.bits == 4 ? TcCfg<4>::kSmem : TcCfg<8>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  int na = 0;
  if (a.pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  if (a.bits == 4) return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<4>, tmx, p);
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<8>, tmx, p);
}

}  // namespace wq
