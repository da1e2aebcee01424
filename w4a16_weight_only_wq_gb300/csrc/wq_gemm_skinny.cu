// wq_gemm_skinny.cu -- tcgen05 W4A16 / W8A16 GEMM for M <= 16 with the
// dequantised weights in tensor memory.
//
// Y[M,N] = X[M,K] . (s (.) q)[K,N] for the verifier's 16-token block
// ("Quantize the Target, Quantize the Drafter": the INT4 target verifies an
// anchor plus 15 drafted tokens in one forward), computed as
// Y^T = W^T . X^T: the dequantised weights bf16(s*q) are the tcgen05.mma A
// operand (M = 128 weight columns, one per TMEM lane, written from
// registers with tcgen05.st) and the 16 tokens of X are the N = 16 operand
// in shared memory.  At M = 16 the packed weights dominate the bytes, so
// the kernel is organised around streaming them:
//
//  * Work unit: 128 weight columns x a contiguous range of packed chunks
//    (two groups each); a cluster of `cs` CTAs splits one
//    column tile's K range and every CTA accumulates its range in one TMEM
//    accumulator [128 x 16].  Partial sums are pushed into the owning CTA's
//    shared memory (distributed shared memory) and added there in rank
//    order.  `cs` is the largest split whose clusters are all resident.
//  * Producer (warp 0): the packed cells of a chunk for both cell columns
//    per TMA (128-byte swizzle) and their scales, issued before the
//    programmatic-launch wait (they do not depend on the preceding
//    kernel); then X: when the CTA's K range fits, all of it in one TMA
//    over a 3-D view of X (64-deep blocks as the outer dimension), else 64
//    deep per TMA.  (Each TMA costs the SM's copy engine ~0.1 us to issue.)
//  * Dequant (warps 2-17, four per TMEM lane quadrant): LOP3 extraction,
//    an exact bf16x2 subtraction of the offset and a bf16x2 multiply by the
//    scale give bf16(s*q) (one rounding), stored into the thread's lane.
//  * MMA (warp 1, one thread): eight 128x16x16 MMAs per group, spread
//    over four accumulators so that consecutive MMAs do not serialise.
//  * Epilogue (warps 18-21): tcgen05.ld of the accumulator, then Y (one
//    CTA) or the cluster reduction.
//  Every wait is bounded; an abort drains copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tcgen05.cuh"
#include "wq_tensor_map.h"
#include "wq_tmem_dequant.cuh"

namespace wq {
namespace {

constexpr int kTok = 16;            // tokens (MMA N)
constexpr int kCols = 128;          // weight columns per CTA (MMA M, TMEM lanes)
constexpr int kNX = 32;             // X stages (64 deep) in shared memory
constexpr int kGA = 4;              // groups of A in tensor memory
constexpr int kNQ = 3;              // packed chunks in flight
constexpr int kDequantWarps = 16;
constexpr int kFirstDequantWarp = 2;
constexpr int kFirstEpiWarp = kFirstDequantWarp + kDequantWarps;  // 18
constexpr int kEpiWarps = 4;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;        // 704
constexpr uint32_t kTmemCols = 512;
constexpr int kACol = 256;          // A slots: TMEM columns 256..511
// Independent accumulators (TMEM columns 16 i .. 16 i + 15): consecutive
// MMAs of 128 x 16 x 16 into one accumulator serialise on it, so k-step j
// goes to accumulator (4h + j) % kAcc and the epilogue adds them in order.
constexpr int kAcc = 4;
constexpr int kXStage = kTok * 128; // 2 KiB: 16 tokens x 64 bf16
constexpr int kPartFloats = (kCols + 8) * kTok;  // cs slices of ceil(128 / cs) columns x 16

template <int BITS>
struct SkCfg {
  static constexpr int kChunk = 2;                             // groups per packed chunk
  static constexpr int kCellBytes = BITS == 4 ? 4096 : 8192;
  static constexpr int kCellRows = kCellBytes / 128;
  static constexpr int kColBytes = kChunk * kCellBytes;        // one cell column of a chunk
  static constexpr int kScaleOff = 2 * kColBytes;
  static constexpr int kQBytes = (kScaleOff + kChunk * kCols * 2 + 1023) / 1024 * 1024;
  static constexpr int kOffX = 0;
  static constexpr int kOffQ = kOffX + kNX * kXStage;
  static constexpr int kOffPart = kOffQ + kNQ * kQBytes;
  static constexpr int kOffBar = kOffPart + kPartFloats * 4;
  static constexpr int kNumBars = 2 * kNX + 2 * kNQ + 2 * kGA + 3;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
};

struct SkParams {
  const uint16_t* S;
  __nv_bfloat16* Y;
  int M, N, K, G, cs;
  int xblocks;  // > 0: X in one 3-D TMA of this many 64-deep blocks
  KernelDiag diag;
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                   const SkParams p) {
  using C = SkCfg<BITS>;
  constexpr int kChunk = C::kChunk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

  float* part = reinterpret_cast<float*>(smem + C::kOffPart);  // same offset in every CTA
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* x_full = bars;                 // [kNX] X stage landed
  uint64_t* x_empty = x_full + kNX;        // [kNX] MMAs done with it
  uint64_t* q_full = x_empty + kNX;        // [kNQ] packed chunk + scales landed
  uint64_t* q_empty = q_full + kNQ;        // [kNQ] chunk dequantised
  uint64_t* a_full = q_empty + kNQ;        // [kGA] group of A written
  uint64_t* a_empty = a_full + kGA;        // [kGA] MMAs done with it
  uint64_t* d_full = a_empty + kGA;        // every MMA of this CTA has completed
  uint64_t* never_bar = d_full + 1;        // test hook
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = p.cs;
  const int tile = blockIdx.x / cs;
  const int rank = blockIdx.x % cs;       // == %cluster_ctarank for cluster (cs,1,1)
  // K split in whole chunks, so that every chunk is complete
  const int nchunks = p.G / kChunk;
  const int c0 = (nchunks * rank) / cs;
  const int nch = (nchunks * (rank + 1)) / cs - c0;
  const int g0 = c0 * kChunk, ng = nch * kChunk;
  const int n0 = tile * kCols;
  const int rows = min(kTok, p.M);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
    }
    for (int i = 0; i < kNQ; ++i) {
      mbar_init(&q_full[i], 1 + 32);       // TMA arrival + one per producer lane (cp.async)
      mbar_init(&q_empty[i], 4 * kChunk);  // every dequant warp that reads the chunk
    }
    for (int i = 0; i < kGA; ++i) {
      mbar_init(&a_full[i], 4);            // one warp per TMEM lane quadrant
      mbar_init(&a_empty[i], 1);
    }
    mbar_init(d_full, 1);
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
  // every CTA of the cluster has started before any remote store (epilogue)
  if (cs > 1) cluster_arrive_relaxed();
  const uint32_t tmem_base = *tmem_slot;
  // The next kernel may launch now: it reads nothing this grid writes
  // before this grid completes.
  pdl_launch_dependents();
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  int issued_q = 0, issued_x = 0;
  if (warp == 0) {
    // ------------------------------------------------------- producer ---
    if (lane == 0) {
      prefetch_tensor_map(&tmx);
      prefetch_tensor_map(&tmw);
    }
    const int ncells = min(2, (p.N - n0) / 64);
    bool ok = true;
    auto issue_q = [&](int qc) -> bool {
      const int slot = qc % kNQ;
      const int g = g0 + qc * kChunk;
      int okw = 1;
      if (lane == 0) {
        if (qc >= kNQ) okw = role_wait(&q_empty[slot], ((qc / kNQ) - 1) & 1, p.diag, abort_flag);
        if (okw) {
          uint8_t* dst = smem + C::kOffQ + slot * C::kQBytes;
          mbar_arrive_expect_tx(&q_full[slot], ncells * C::kColBytes);
          for (int ci = 0; ci < ncells; ++ci)
            tma_load_2d(dst + ci * C::kColBytes, &tmw, 0,
                        ((n0 / 64 + ci) * p.G + g) * C::kCellRows, &q_full[slot]);
        }
      }
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (!okw) return false;
      const uint32_t sdst = smem_addr(smem + C::kOffQ + slot * C::kQBytes + C::kScaleOff);
      for (int piece = lane; piece < kChunk * 16; piece += 32) {
        const int gi = piece >> 4, col = (piece & 15) * 8;
        const bool live = n0 + col < p.N;
        const uint16_t* src = live ? p.S + static_cast<size_t>(g + gi) * p.N + n0 + col : p.S;
        cp_async_16(sdst + (gi * kCols + col) * 2, src, live ? 16u : 0u);
      }
      cp_async_mbar_arrive_noinc(&q_full[slot]);
      return true;
    };
    auto issue_x = [&](int si) -> bool {
      if (p.xblocks > 0) {  // every stage in one copy, on x_full[0]
        if (lane == 0) {
          mbar_arrive_expect_tx(&x_full[0], p.xblocks * kXStage);
          tma_load_3d(smem + C::kOffX, &tmx, 0, 0, g0 * 2, &x_full[0]);
        }
        __syncwarp();
        return true;
      }
      const int slot = si % kNX;
      int okx = 1;
      if (lane == 0) {
        if (si >= kNX) okx = role_wait(&x_empty[slot], ((si / kNX) - 1) & 1, p.diag, abort_flag);
        if (okx) {
          mbar_arrive_expect_tx(&x_full[slot], kXStage);
          tma_load_2d(smem + C::kOffX + slot * kXStage, &tmx, (g0 * 2 + si) * 64, 0, &x_full[slot]);
        }
      }
      return __shfl_sync(0xffffffffu, okx, 0) != 0;
    };
    // weights first: they do not depend on the preceding kernel
    for (int qc = 0; qc < min(kNQ, nch) && ok; ++qc) {
      ok = issue_q(qc);
      if (ok) issued_q = qc + 1;
    }
    pdl_wait_primary();
    const int nstages = p.xblocks > 0 ? 0 : 2 * ng;
    if (p.xblocks > 0) {
      ok = issue_x(0);
      issued_x = 1;
    }
    for (int si = 0; si < min(kNX, nstages) && ok; ++si) {
      ok = issue_x(si);
      if (ok) issued_x = si + 1;
    }
    // refills, in the order the MMAs need them
    int qc = min(kNQ, nch), si = min(kNX, nstages);
    while (ok && (qc < nch || si < nstages)) {
      if (qc < nch && (si >= nstages || qc * kChunk * 2 <= si)) {
        ok = issue_q(qc);
        if (ok) issued_q = ++qc;
      } else {
        ok = issue_x(si);
        if (ok) issued_x = ++si;
      }
    }
    cp_async_wait_all();
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kCols, kTok);
      for (int u = 0; u < ng; ++u) {
        const int as = u % kGA;
        const bool hook = p.diag.force_timeout == 2 && u == ng / 2;
        if (!role_wait(hook ? never_bar : &a_full[as], hook ? 0u : (u / kGA) & 1, p.diag,
                       abort_flag))
          break;
        bool ok = true;
        for (int h = 0; h < 2; ++h) {
          const int si = 2 * u + h, xs = si % kNX;
          const bool xwait = p.xblocks > 0 ? si == 0 : true;
          if (xwait && !role_wait(&x_full[p.xblocks > 0 ? 0 : xs], p.xblocks > 0 ? 0u : (si / kNX) & 1,
                                  p.diag, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t b_desc = smem_desc_sw128(smem_addr(smem + C::kOffX + xs * kXStage));
          const uint32_t a_tmem = tmem_base + kACol + as * 64 + h * 32;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma_bf16_ts(tmem_base + ((4 * h + j) % kAcc) * kTok, a_tmem + 8 * j, b_desc + 2 * j,
                         idesc, (u | ((4 * h + j) / kAcc)) != 0);
          if (p.xblocks == 0) umma_commit(&x_empty[xs]);
        }
        if (!ok) break;
        umma_commit(&a_empty[as]);
      }
      // arrives when every MMA issued above has completed
      umma_commit(d_full);
    }
  } else if (warp < kFirstEpiWarp) {
    // ------------------------------------------------- dequant warps ---
    // Quadrant q = warp % 4 (the TMEM lanes this warp may write); warp r =
    // (warp - 2) / 4 takes the groups whose A slot is r.
    const int q = warp & 3, r = (warp - kFirstDequantWarp) >> 2;
    const int n = 32 * q + lane;  // weight column within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    for (int qc = 0; qc < nch; ++qc) {
      const int pos = r - (qc * kChunk) % kGA;
      if (pos < 0 || pos >= kChunk) continue;  // not this warp's chunk
      const int slot = qc % kNQ;
      const int u = qc * kChunk + pos;
      if (!role_wait(&q_full[slot], (qc / kNQ) & 1, p.diag, abort_flag) ||
          (u >= kGA && !role_wait(&a_empty[r], ((u / kGA) - 1) & 1, p.diag, abort_flag)))
        break;
      const uint32_t qbase = smem_addr(smem + C::kOffQ + slot * C::kQBytes);
      const uint32_t s1 = ld_shared_u16(qbase + C::kScaleOff + (pos * kCols + n) * 2);
      dequant_group_to_tmem<BITS>(qbase + (n >> 6) * C::kColBytes + pos * C::kCellBytes, n,
                                  s1 | (s1 << 16), tmem_base + lane_addr + kACol + r * 64);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[r]);
        mbar_arrive(&q_empty[slot]);
      }
    }
  }

  // ------------------------------------------------------- epilogue ---
  // Accumulator D[column n][token m] (128 lanes x 16 columns).  Element
  // e = m * 128 + n of the tile; with a cluster, rank r owns elements
  // [r E / cs, (r + 1) E / cs) and receives every rank's partial of them in
  // its `part` (slice q at q * slice) by remote stores.
  float v[kTok];
#pragma unroll
  for (int m = 0; m < kTok; ++m) v[m] = 0.f;
  if (warp >= kFirstEpiWarp) {
    pdl_wait_primary();  // these warps store Y
    const int lane_base = 32 * (warp & 3);
    if (role_wait(d_full, 0, p.diag, abort_flag, 2000)) {
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < kAcc; ++i) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(lane_base) << 16) + i * kTok, r);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < kTok; ++m) v[m] += __uint_as_float(r[m]);
      }
    }
  }
  // Roles that ran on one lane (MMA issue, copy issue) rejoin their warp
  // before the block-wide barrier, which a diverged warp must not reach.
  __syncwarp();
  __syncthreads();
  if (*abort_flag) {
    // Let every issued copy land and every issued MMA finish (bounded, at
    // least 1 s) before shared and tensor memory are released.
    KernelDiag drain = p.diag;
    if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < kNQ && s < issued_q; ++s) {
        const int last = s + ((issued_q - 1 - s) / kNQ) * kNQ;
        mbar_wait_bounded(&q_full[s], (last / kNQ) & 1, drain);
      }
      for (int s = 0; s < kNX && s < issued_x; ++s) {
        const int last = s + ((issued_x - 1 - s) / kNX) * kNX;
        mbar_wait_bounded(&x_full[s], (last / kNX) & 1, drain);
      }
    }
    if (warp == 1 && lane == 0) mbar_wait_bounded(d_full, 0, drain);
    __syncwarp();
    __syncthreads();
  }
  if (cs == 1) {
    if (warp >= kFirstEpiWarp) {
      const int n = 32 * (warp & 3) + lane;
      if (n0 + n < p.N) {
#pragma unroll
        for (int m = 0; m < kTok; ++m)
          if (m < rows) p.Y[static_cast<size_t>(m) * p.N + n0 + n] = __float2bfloat16_rn(v[m]);
      }
    }
  } else {
    // Rank r owns the tile's columns [128 r / cs, 128 (r + 1) / cs) and
    // receives, per source rank q, the 16 token partials of each of its
    // columns at part[(q * cslice + local column) * 16 ..] (64 bytes, four
    // 16-byte remote stores per column).
    const int cslice = (kCols + cs - 1) / cs;
    cluster_wait();
    if (warp >= kFirstEpiWarp) {
      const int n = 32 * (warp & 3) + lane;
      int owner = (n * cs) / kCols;
      while (owner + 1 < cs && n >= ((owner + 1) * kCols) / cs) ++owner;
      while (n < (owner * kCols) / cs) --owner;
      const uint32_t dst = dsmem_map(part + (rank * cslice + n - (owner * kCols) / cs) * kTok, owner);
#pragma unroll
      for (int i = 0; i < kTok / 4; ++i)
        dsmem_st_v4_f32(dst + 16 * i, v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    cluster_sync();  // every partial has arrived in its owner's `part`
    const int cb0 = (rank * kCols) / cs, ncol = ((rank + 1) * kCols) / cs - cb0;
    for (int e = threadIdx.x; e < rows * ncol; e += kThreads) {
      const int m = e / ncol, c = e % ncol;
      if (n0 + cb0 + c >= p.N) continue;
      float acc = 0.f;
      for (int qq = 0; qq < cs; ++qq) acc += part[(qq * cslice + c) * kTok + m];
      p.Y[static_cast<size_t>(m) * p.N + n0 + cb0 + c] = __float2bfloat16_rn(acc);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side ---

// Per device: the kernel's shared-memory attribute, and for every cluster
// size 1..8 how many clusters can be resident at once.
template <int BITS>
struct SkInit {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
  int max_clusters[64][9] = {};
  cudaError_t ensure(int device, int (&out)[9]) {
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> lk(mu);
      if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SkCfg<BITS>::kSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_skinny_kernel<BITS>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        (void)e;  // sizes up to 8 are portable
        for (int c = 1; c <= 8; ++c) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(c);
          cfg.blockDim = dim3(kThreads);
          cfg.dynamicSmemBytes = SkCfg<BITS>::kSmem;
          cudaLaunchAttribute at;
          at.id = cudaLaunchAttributeClusterDimension;
          at.val.clusterDim.x = c;
          at.val.clusterDim.y = 1;
          at.val.clusterDim.z = 1;
          cfg.attrs = &at;
          cfg.numAttrs = 1;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, gemm_skinny_kernel<BITS>, &cfg) != cudaSuccess)
            n = 0;
          max_clusters[device & 63][c] = n;
        }
        cudaGetLastError();  // a refused size above is not an error of this call
        done.fetch_or(bit, std::memory_order_release);
      }
    }
    for (int c = 0; c <= 8; ++c) out[c] = max_clusters[device & 63][c];
    return cudaSuccess;
  }
};
SkInit<4> g_sk4;
SkInit<8> g_sk8;

// The largest split (in whole chunks) whose clusters all fit at once and
// whose CTAs fit one per SM.
int sk_split(int64_t tiles, int nchunks, int num_sms, int hint, const int (&max_cl)[9]) {
  if (hint > 0) return (hint <= 8 && hint <= nchunks) ? hint : -1;
  int best = 1;
  for (int cs = 1; cs <= 8 && cs <= nchunks; ++cs)
    if (tiles * cs <= num_sms && tiles <= max_cl[cs]) best = cs;
  return best;
}

}  // namespace

bool gemm_skinny_fits(int bits, int64_t K, int64_t N) {
  if ((K / 128) % 2 != 0) return false;  // whole packed chunks
  return (bits == 4 ? K * N / 256 : K * N / 128) <= INT32_MAX;
}

cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t stream) {
  if (a.M > kTok || !gemm_skinny_fits(a.bits, a.K, a.N)) return cudaErrorNotSupported;
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  int max_cl[9];
  cudaError_t e = a.bits == 4 ? g_sk4.ensure(a.device, max_cl) : g_sk8.ensure(a.device, max_cl);
  if (e != cudaSuccess) return e;
  const int chunk = a.bits == 4 ? SkCfg<4>::kChunk : SkCfg<8>::kChunk;
  const int G = static_cast<int>(a.K / 128);
  const int64_t tiles = (a.N + kCols - 1) / kCols;
  const int cs = sk_split(tiles, G / chunk, a.num_sms, a.split_hint, max_cl);
  if (cs < 0) return cudaErrorNotSupported;

  // X as a 2-D bf16 tensor [M rows, K cols]; box 64 x 16, 128-byte
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
  // The packed weights as a 2-D u32 tensor of 128-byte rows; one box is the
  // cells of one chunk of one cell column.
  CUtensorMap tmw;
  const int64_t words = a.bits == 4 ? a.K * a.N / 8 : a.K * a.N / 4;
  const int box_rows = a.bits == 4 ? SkCfg<4>::kChunk * SkCfg<4>::kCellRows
                                   : SkCfg<8>::kChunk * SkCfg<8>::kCellRows;
  const cuuint64_t wdim[2] = {32, static_cast<cuuint64_t>(words / 32)};
  const cuuint64_t wstride[1] = {128};
  const cuuint32_t wbox[2] = {32, static_cast<cuuint32_t>(box_rows)};
  r = enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(a.Wp), wdim, wstride,
          wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  // When a CTA's K range fits the X stages, X comes in one TMA over the
  // 3-D view [K/64 blocks][M rows][64] (box 64 x 16 x blocks); the same
  // shared-memory layout as the 2-D boxes, block after block.
  const int nchunks = G / chunk;
  const int xblocks = ((nchunks + cs - 1) / cs) * chunk * 2;
  int use3d = 0;
  if (xblocks <= kNX) {
    CUtensorMap t3;
    const cuuint64_t d3[3] = {64, static_cast<cuuint64_t>(a.M), static_cast<cuuint64_t>(a.K / 64)};
    const cuuint64_t s3[2] = {static_cast<cuuint64_t>(a.K) * 2, 128};
    const cuuint32_t b3[3] = {64, kTok, static_cast<cuuint32_t>(xblocks)};
    const cuuint32_t e3[3] = {1, 1, 1};
    if (enc(&t3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.X), d3, s3, b3, e3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      tmx = t3;
      use3d = 1;
    }
  }

  SkParams p;
  p.xblocks = use3d ? xblocks : 0;
  p.S = static_cast<const uint16_t*>(a.S);
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.G = G;
  p.cs = cs;
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.bits == 4 ? SkCfg<4>::kSmem : SkCfg<8>::kSmem;
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
