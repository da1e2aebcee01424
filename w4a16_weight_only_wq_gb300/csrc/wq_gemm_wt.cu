// wq_gemm_wt.cu -- tcgen05 W4A16 / W8A16 GEMM for large M with the
// dequantised weights in tensor memory.
//
// Y[M,N] = X[M,K] . (s (.) q)[K,N] ("Quantize the Target, Quantize the
// Drafter": the INT4 target's prefill of a long prompt and batched
// verification of several draft blocks), computed as
// Y^T = W^T . X^T so that the dequantised weights are the tcgen05.mma A
// operand (M = 128 weight columns, one per TMEM lane) written straight
// from registers into tensor memory, and X is the B operand (N = 128
// tokens) read from shared memory.  The weights never pass through shared
// memory as bf16, which is what bounds a kernel that stages dequantised
// weights there: only X tiles (TMA) and packed codes (TMA) are stored in
// shared memory, and only the MMA and the dequant warps read it.
//
//  * Persistent: one CTA per SM walks tiles of 128 tokens x 128 weight
//    columns (M < 512: double-buffered accumulator, so the epilogue of a
//    tile overlaps the next tile's MMAs) or x 256 weight columns as two
//    128-lane halves that share every X stage (M >= 512: half the L2
//    traffic of X per FLOP, one accumulator of 2 x 128 columns).
//  * Producer (warp 0): packed cells of four (INT4) or two (INT8) groups of
//    both 64-column cell columns per TMA (the packed buffer seen as rows of
//    128 bytes, 128-byte swizzle) plus their scales (cp.async), one chunk
//    ahead; X in 64-deep stages (TMA, 128-byte swizzle).
//  * MMA (warp 1, one thread): per 64-deep stage, four 128x128x16 MMAs
//    with A from tensor memory and B from the X stage.
//  * Dequant (warps 2-17, four per TMEM lane quadrant): a thread owns one
//    weight column of one group: LOP3 extraction of the codes, an exact
//    bf16x2 subtraction of the offset and one bf16x2 multiply by the scale
//    give bf16(s*q), stored with two tcgen05.st into its lane.
//  * Epilogue (warps 18-21): tcgen05.ld of the accumulator; a thread holds
//    one weight column of 32 tokens, so each warp transposes its 32 x 32
//    block through shared memory and stores Y rows with 16-byte stores.
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

constexpr int kTM = 128;          // tokens per tile (MMA N)
constexpr int kNB = 8;            // X stages (64 deep) in shared memory
constexpr int kXG = kNB / 2;      // ... filled a group (two stages) per copy
constexpr int kNQ = 2;            // packed chunks in flight
constexpr int kDequantWarps = 16;
constexpr int kFirstDequantWarp = 2;
constexpr int kFirstEpiWarp = kFirstDequantWarp + kDequantWarps;  // 18
constexpr int kEpiWarps = 4;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;        // 704
constexpr uint32_t kTmemCols = 512;
constexpr int kACol = 256;        // A slots: TMEM columns 256..511
constexpr int kXStage = kTM * 128;  // 16 KiB: 128 tokens x 64 bf16

// HALVES = 1: tiles of 128 weight columns, the accumulator (128 columns)
// double-buffered, four groups of A in flight.  HALVES = 2: tiles of 256
// weight columns as two 128-lane halves that share every X stage (half the
// L2 traffic of X per FLOP), one accumulator of 2 x 128 columns, two groups
// of A in flight; the epilogue of a tile briefly holds up the next one.
template <int BITS, int HALVES>
struct WtCfg {
  static constexpr int kTN = 128 * HALVES;                     // weight columns per tile
  static constexpr int kGA = HALVES == 1 ? 4 : 2;              // groups of A in TMEM
  static constexpr int kAGroupCols = 64 * HALVES;              // TMEM columns per group of A
  static constexpr int kDBufs = HALVES == 1 ? 2 : 1;           // accumulators
  static constexpr int kChunk = (BITS == 4 ? 4 : 2) / HALVES;  // groups per packed chunk
  static constexpr int kCellCols = 2 * HALVES;                 // 64-column cell columns per tile
  static constexpr int kCellBytes = BITS == 4 ? 4096 : 8192;   // 64 columns x 128 k
  static constexpr int kCellRows = kCellBytes / 128;
  static constexpr int kColBytes = kChunk * kCellBytes;        // one cell column of a chunk
  static constexpr int kScaleOff = kCellCols * kColBytes;
  // + scales [group][128]; a multiple of 1024 so every slot's cells keep the
  // 1024-byte alignment the 128-byte swizzle pattern is anchored to
  static constexpr int kQBytes = (kScaleOff + kChunk * kTN * 2 + 1023) / 1024 * 1024;
  static constexpr int kOffX = 0;
  static constexpr int kOffQ = kOffX + kNB * kXStage;
  static constexpr int kOffT = kOffQ + kNQ * kQBytes;              // epilogue transposes
  static constexpr int kOffBar = kOffT + kEpiWarps * 32 * 64;
  static constexpr int kNumBars = 2 * kNB + 2 * kNQ + 2 * 4 + 4 + 2;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 32 + 1024;  // + alignment slack
};

struct WtParams {
  const uint16_t* S;
  __nv_bfloat16* Y;
  int M, N, K, G;
  int mt, nt;  // tile counts along M and N
  int ks;      // CTAs of a cluster that split one tile's K range (1: none)
  int tn;      // tokens per MMA (N): 64 when M <= 64, else kTM
  KernelDiag diag;
};

template <int BITS, int HALVES, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_wt_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
               const WtParams p) {
  using C = WtCfg<BITS, HALVES>;
  constexpr int kChunk = C::kChunk;
  constexpr int kGA = C::kGA;
  constexpr int kTN = C::kTN;
  static_assert(HALVES == 2 || kGA == kXG, "one-accumulator tiles share the A and X slot ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* b_full = bars;                 // [kXG] X stages of a group landed
  uint64_t* b_empty = b_full + kNB;        // [kXG] MMAs done with them
  uint64_t* q_full = b_empty + kNB;        // [kNQ] packed chunk + scales landed
  uint64_t* q_empty = q_full + kNQ;        // [kNQ] chunk dequantised
  uint64_t* a_full = q_empty + kNQ;        // [kGA] group of A written
  uint64_t* a_empty = a_full + 4;          // [kGA] MMAs done with it
  uint64_t* d_full = a_empty + 4;          // [kDBufs] accumulator finished
  uint64_t* d_empty = d_full + 2;          // [2] accumulator read out
  uint64_t* mma_done = d_empty + 2;       // every MMA of this CTA has completed
  uint64_t* never_bar = mma_done + 1;      // test hook
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);


  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = p.G / kChunk;            // chunks per tile
  // Tiles: cluster cl (of ncl; one CTA unless the K range is split) takes
  // tiles t = cl + k ncl: token tile t % mt, column tile t / mt.  With a
  // split, CTA `rank` of the cluster takes chunks [kc0, kc0 + kch) of each
  // of its tiles' K range.
  const int ks = HALVES == 1 ? p.ks : 1;
  const int rank = ks > 1 ? static_cast<int>(blockIdx.x) % ks : 0;
  const int cl = blockIdx.x / ks, ncl = gridDim.x / ks;
  const int kc0 = (nch * rank) / ks, kch = (nch * (rank + 1)) / ks - kc0;
  const int ptiles = p.mt * p.nt;
  const int my_tiles = ptiles > cl ? (ptiles - 1 - cl) / ncl + 1 : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kXG; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < kNQ; ++i) {
      mbar_init(&q_full[i], 1 + 32);       // TMA arrival + one per producer lane (cp.async)
      mbar_init(&q_empty[i], 4 * HALVES * kChunk);  // every dequant warp that reads the chunk
    }
    for (int i = 0; i < kGA; ++i) {
      mbar_init(&a_full[i], 4 * HALVES);   // one warp per TMEM lane quadrant and half
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], kEpiWarps);
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
  // The next kernel may launch now: its CTAs take SMs this grid leaves
  // free, and it reads nothing this grid writes before it completes.
  pdl_launch_dependents();
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  int issued_q = 0, issued_b = 0;
  if (warp == 0) {
    // ------------------------------------------------------- producer ---
    if (lane == 0) {
      prefetch_tensor_map(&tmx);
      prefetch_tensor_map(&tmw);
    }
    const int total_q = my_tiles * kch;
    bool ok = true;
    // chunk qc (global over this CTA's tiles) -> tile and first group
    auto issue_q = [&](int qc) -> bool {
      const int slot = qc % kNQ;
      const int t2 = cl + (qc / kch) * ncl;
      const int g0 = (kc0 + qc % kch) * kChunk;
      const int nt = t2 / p.mt;
      int okw = 1;
      if (lane == 0) {
        if (qc >= kNQ) okw = role_wait(&q_empty[slot], ((qc / kNQ) - 1) & 1, p.diag, abort_flag);
        if (okw) {
          // every cell column of the tile in one copy; a column past N reads
          // as zeros and still counts in the transaction
          mbar_arrive_expect_tx(&q_full[slot], C::kCellCols * C::kColBytes);
          tma_load_3d(smem + C::kOffQ + slot * C::kQBytes, &tmw, 0, g0 * C::kCellRows,
                      nt * C::kCellCols, &q_full[slot]);
        }
      }
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (!okw) return false;
      // scales: kChunk groups x kTN columns, 16-byte pieces (8 columns)
      const uint32_t sdst = smem_addr(smem + C::kOffQ + slot * C::kQBytes + C::kScaleOff);
      for (int piece = lane; piece < kChunk * (kTN / 8); piece += 32) {
        const int gi = piece / (kTN / 8), col = (piece % (kTN / 8)) * 8;
        const bool live = nt * kTN + col < p.N;
        const uint16_t* src = live ? p.S + static_cast<size_t>(g0 + gi) * p.N + nt * kTN + col : p.S;
        cp_async_16(sdst + (gi * kTN + col) * 2, src, live ? 16u : 0u);
      }
      cp_async_mbar_arrive_noinc(&q_full[slot]);
      return true;
    };
    // X of chunk qc: one copy per group (two 64-deep stages)
    auto issue_x = [&](int qc) -> bool {
      const int t2 = cl + (qc / kch) * ncl;
      const int g0 = (kc0 + qc % kch) * kChunk;
      const int m0 = (t2 % p.mt) * kTM;
      for (int s = 0; s < kChunk; ++s) {
        const int gi = qc * kChunk + s;
        const int slot = gi % kXG;
        int okx = 1;
        if (lane == 0) {
          // with one accumulator half the A and X rings coincide (slot u % 4)
          // and the MMAs release both with one commit on a_empty
          if (gi >= kXG)
            okx = role_wait(HALVES == 1 ? &a_empty[slot] : &b_empty[slot], ((gi / kXG) - 1) & 1,
                            p.diag, abort_flag);
          if (okx) {
            mbar_arrive_expect_tx(&b_full[slot], 2 * p.tn * 128);
            tma_load_3d(smem + C::kOffX + slot * 2 * kXStage, &tmx, 0, m0, (g0 + s) * 2,
                        &b_full[slot]);
          }
        }
        okx = __shfl_sync(0xffffffffu, okx, 0);
        if (!okx) return false;
        issued_b = gi + 1;
      }
      return true;
    };
    // The packed weights and scales do not depend on the preceding kernel:
    // the first chunks are requested before waiting for it (programmatic
    // launch); X, which it may write, after.
    for (int qc = 0; qc < min(kNQ, total_q) && ok; ++qc) {
      ok = issue_q(qc);
      if (ok) issued_q = qc + 1;
    }
    pdl_wait_primary();
    for (int qc = 0; qc < total_q && ok; ++qc) {
      ok = issue_x(qc);
      if (ok && qc + kNQ < total_q) {
        ok = issue_q(qc + kNQ);
        if (ok) issued_q = qc + kNQ + 1;
      }
    }
    cp_async_wait_all();
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      // N = p.tn tokens: a 64-token MMA when M <= 64 (the rows past it would
      // be zeros), which costs about half a 128-token one
      const uint32_t idesc = p.tn == 64 ? idesc_bf16_f32(128, 64) : idesc_bf16_f32(128, kTM);
      // a group's X copy lands as [stage][p.tn rows][128 bytes]
      const uint32_t x_stage = HALVES == 2 ? kXStage : p.tn * 128;
      int u = 0;  // global group index of this CTA
      bool ok = true;
      for (int tl = 0; ok && tl < my_tiles; ++tl) {
        const int buf = tl % C::kDBufs, use = tl / C::kDBufs;
        if (tl >= C::kDBufs && !role_wait(&d_empty[buf], (use - 1) & 1, p.diag, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int g = 0; g < kch * kChunk; ++g, ++u) {
          const int as = u % kGA;
          const bool hook = p.diag.force_timeout == 2 && tl == 0 && g == kch * kChunk / 2;
          if (!role_wait(hook ? never_bar : &a_full[as], hook ? 0u : (u / kGA) & 1, p.diag,
                         abort_flag)) {
            ok = false;
            break;
          }
          const int xs = u % kXG;
          // HALVES == 1: the dequant warps saw the group's X land before
          // marking its A slot full, so one wait covers both
          if (HALVES == 2 && !role_wait(&b_full[xs], (u / kXG) & 1, p.diag, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t b_desc =
                smem_desc_sw128(smem_addr(smem + C::kOffX + 2 * xs * kXStage + h * x_stage));
#pragma unroll
            for (int hf = 0; hf < HALVES; ++hf) {
              // half hf of the weight columns: its own accumulator and A
              const uint32_t d_tmem = tmem_base + (HALVES == 1 ? buf : hf) * 128;
              const uint32_t a_tmem = tmem_base + kACol + as * C::kAGroupCols + hf * 64 + h * 32;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                umma_bf16_ts(d_tmem, a_tmem + 8 * j, b_desc + 2 * j, idesc, (g | h | j) != 0);
            }
          }
          if (HALVES == 2) umma_commit(&b_empty[xs]);
          umma_commit(&a_empty[as]);
        }
        if (ok) umma_commit(&d_full[buf]);
      }
      // every MMA has completed before shared and tensor memory are released
      umma_commit(mma_done);
      KernelDiag drain = p.diag;
      if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
      mbar_wait_bounded(mma_done, 0, drain);
    }
  } else if (warp < kFirstEpiWarp) {
    // ------------------------------------------------- dequant warps ---
    // Quadrant q = warp % 4 (the TMEM lanes this warp may write); with
    // r = (warp - 2) / 4, the warp takes half hf of the columns of the
    // groups whose A slot is r (HALVES = 1) or r / 2 (HALVES = 2).
    const int q = warp & 3, r = (warp - kFirstDequantWarp) >> 2;
    const int hf = HALVES == 1 ? 0 : (r & 1);
    const int aslot = HALVES == 1 ? r : (r >> 1);
    const int n = hf * 128 + 32 * q + lane;  // weight column within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const int total_q = my_tiles * kch;
    bool ok = true;
    for (int qc = 0; qc < total_q && ok; ++qc) {
      // groups u = qc * kChunk + pos, A slot u % kGA; this warp takes aslot
      const int pos = aslot - (qc * kChunk) % kGA;
      if (pos < 0 || pos >= kChunk) continue;  // not this warp's chunk
      const int slot = qc % kNQ;
      const int u = qc * kChunk + pos;
      if (!role_wait(&q_full[slot], (qc / kNQ) & 1, p.diag, abort_flag) ||
          (u >= kGA && !role_wait(&a_empty[aslot], ((u / kGA) - 1) & 1, p.diag, abort_flag))) {
        ok = false;
        break;
      }
      const uint32_t qbase = smem_addr(smem + C::kOffQ + slot * C::kQBytes);
      const uint32_t s1 = ld_shared_u16(qbase + C::kScaleOff + (pos * kTN + n) * 2);
      dequant_group_to_tmem<BITS>(qbase + (n >> 6) * C::kColBytes + pos * C::kCellBytes, n,
                                  s1 | (s1 << 16),
                                  tmem_base + lane_addr + kACol + aslot * C::kAGroupCols + hf * 64);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // HALVES == 1: the group's X (same slot) has landed too
        if (HALVES == 1 && !role_wait(&b_full[aslot], (u / kXG) & 1, p.diag, abort_flag)) ok = false;
        mbar_arrive(&a_full[aslot]);
        mbar_arrive(&q_empty[slot]);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
  } else {
    // ------------------------------------------------ epilogue warps ---
    pdl_wait_primary();  // these warps store Y
    const int lane_base = 32 * (warp & 3);
    for (int tl = 0; tl < my_tiles; ++tl) {
      const int buf = tl % C::kDBufs, use = tl / C::kDBufs;
      if (!role_wait(&d_full[buf], use & 1, p.diag, abort_flag, 20000)) break;
      tc_fence_after();
      if (ks > 1) break;  // one tile per CTA: partials are reduced after the roles
      const int t2 = cl + tl * ncl;
      const int m0 = (t2 % p.mt) * kTM;
#pragma unroll 1
      for (int cc = 0; cc < HALVES * (kTM / 32); ++cc) {
        const int hf = cc / (kTM / 32), c = cc % (kTM / 32);
        if (m0 + 32 * c >= p.M) continue;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(lane_base) << 16) +
                               (HALVES == 1 ? buf : hf) * 128 + 32 * c,
                           v);
        tmem_ld_wait();
        // transpose: T[token i][column lane] (bf16, rows of 64 bytes), then
        // lane l stores 16 bytes (8 columns) of rows l/4 + 8k
        const uint32_t tb = smem_addr(smem + C::kOffT + (warp - kFirstEpiWarp) * 32 * 64);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          st_shared_u16(tb + i * 64 + lane * 2,
                        __bfloat16_as_ushort(
                            __float2bfloat16_rn(apply_act(__uint_as_float(v[i]), ACT))));
        __syncwarp();
        const int ncol0 = (t2 / p.mt) * kTN + hf * 128 + lane_base;  // first column of the block
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int row = (lane >> 2) + 8 * k, seg = lane & 3;
          const uint4 w = ld_shared_v4(tb + row * 64 + seg * 16);
          const int m = m0 + 32 * c + row, nc = ncol0 + seg * 8;
          if (m < p.M && nc < p.N)  // N is a multiple of 64: a segment is all in or all out
            st_global_v4(p.Y + static_cast<size_t>(m) * p.N + nc, w.x, w.y, w.z, w.w);
        }
        __syncwarp();  // the block is read before the next chunk overwrites it
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[buf]);
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
      for (int s = 0; s < kXG && s < issued_b; ++s) {
        const int last = s + ((issued_b - 1 - s) / kXG) * kXG;
        mbar_wait_bounded(&b_full[s], (last / kXG) & 1, drain);
      }
    }
    // the MMA thread waited for mma_done
    __syncwarp();
    __syncthreads();
  }
  if (HALVES == 1 && ks > 1) {
    // ------------------------------------------- K-split reduction ---
    // The tile's 128 weight columns are dealt to the cluster's CTAs in
    // groups of 8: rank r owns groups [16 r / ks, 16 (r + 1) / ks).  Every
    // CTA pushes its fp32 partial of each column to the column's owner, into
    // the owner's X stages (idle once every CTA of the cluster has passed its
    // roles), as part[source rank][owned column][token], the 16-byte token
    // quads of a column rotated by the column's low three bits so that a
    // warp's stores (32 columns) spread over the banks.  The owner adds the
    // partials in rank order and writes Y.
    const int slice = 8 * ((16 + ks - 1) / ks);  // columns of the widest share
    auto part_off = [&](int src, int local, int tok) -> uint32_t {
      return static_cast<uint32_t>((((src * slice + local) * 32 + ((tok >> 2) ^ (local & 7))) << 4) +
                                   ((tok & 3) << 2));
    };
    const int m0 = (cl % p.mt) * kTM;
    // every owner's X stages are free: their last readers, the owner's MMAs,
    // completed before its roles ended, so this rendezvous needs no release
    // (a relaxed arrive; a release/acquire barrier here measured slower)
    __syncwarp();
    cluster_arrive_relaxed();
    cluster_wait();
    if (warp >= kFirstEpiWarp) {
      tc_fence_after();
      const int lane_base = 32 * (warp & 3);
      const int col = lane_base + lane, owner = (((col >> 3) + 1) * ks - 1) / 16;
      const int local = col - 8 * ((16 * owner) / ks);
      const uint32_t dst = dsmem_map(smem + C::kOffX, static_cast<uint32_t>(owner));
#pragma unroll 1
      for (int c = 0; c < kTM / 32 && m0 + 32 * c < p.M; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(lane_base) << 16) + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dsmem_st_v4_f32(dst + part_off(rank, local, 32 * c + 4 * k), __uint_as_float(v[4 * k]),
                          __uint_as_float(v[4 * k + 1]), __uint_as_float(v[4 * k + 2]),
                          __uint_as_float(v[4 * k + 3]));
      }
    }
    cluster_sync();  // every partial has arrived at its owner
    pdl_wait_primary();  // every thread below may store Y
    const int gs = (16 * rank) / ks, ng = (16 * (rank + 1)) / ks - gs;
    const int rows = min(kTM, p.M - m0);
    const int ncol0 = (cl / p.mt) * kTN + 8 * gs;
    const uint32_t base = smem_addr(smem + C::kOffX);
    // consecutive threads take consecutive tokens of one 8-column group: a
    // warp's loads of one column are 32 consecutive words
    for (int it = threadIdx.x; it < rows * ng; it += kThreads) {
      const int tok = it % rows, cg = it / rows;
      const int nc = ncol0 + 8 * cg;
      if (nc >= p.N) continue;  // N is a multiple of 64: a group is all in or all out
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
      for (int src = 0; src < ks; ++src) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          acc[j] += __uint_as_float(ld_shared_u32(base + part_off(src, 8 * cg + j, tok)));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = apply_act(acc[j], ACT);
      st_global_v4(p.Y + static_cast<size_t>(m0 + tok) * p.N + nc, pack_bf16x2(acc[0], acc[1]),
                   pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side ---

// Per device: the kernel's shared-memory attribute and, for every cluster
// size 1..8, how many clusters can be resident at once (tiles of 128 columns
// only: the K split is used there alone).
template <int BITS, int HALVES, int ACT>
struct WtInit {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
  int max_clusters[64][9] = {};
  cudaError_t ensure(int device, int (&out)[9]) {
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> lk(mu);
      if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_wt_kernel<BITS, HALVES, ACT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             WtCfg<BITS, HALVES>::kSmem);
        if (e != cudaSuccess) return e;
        for (int c = 1; HALVES == 1 && c <= 8; ++c) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(c);
          cfg.blockDim = dim3(kThreads);
          cfg.dynamicSmemBytes = WtCfg<BITS, HALVES>::kSmem;
          cudaLaunchAttribute at;
          at.id = cudaLaunchAttributeClusterDimension;
          at.val.clusterDim.x = c;
          at.val.clusterDim.y = 1;
          at.val.clusterDim.z = 1;
          cfg.attrs = &at;
          cfg.numAttrs = 1;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, gemm_wt_kernel<BITS, HALVES, ACT>, &cfg) != cudaSuccess)
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
// One per kernel variant: bits, tile halves, activation (the fused MLP's
// up-projection).
template <int BITS, int HALVES, int ACT>
WtInit<BITS, HALVES, ACT> g_wt_init;

// K split of a tile over a cluster when the tiles alone leave at least half
// the SMs idle: the largest split (in whole chunks, at most 8) whose CTAs fit
// one per SM and whose clusters are all resident at once.  A positive hint
// forces the split (any split up to 8 and the chunk count is correct).
int wt_split(int64_t tiles, int nchunks, int num_sms, int hint, const int (&max_cl)[9]) {
  if (hint > 0) return (hint <= 8 && hint <= nchunks && max_cl[hint] > 0) ? hint : -1;
  int best = 1;
  if (tiles * 2 > num_sms) return best;
  for (int cs = 2; cs <= 8 && cs <= nchunks; ++cs)
    if (tiles * cs <= num_sms && tiles <= max_cl[cs]) best = cs;
  return best;
}

template <int BITS, int HALVES, int ACT>
cudaError_t launch_wt(const GemmArgs& a, cudaStream_t stream, TensorMapEncodeFn enc) {
  using C = WtCfg<BITS, HALVES>;
  constexpr int kTN = C::kTN;
  int max_cl[9];
  cudaError_t e = g_wt_init<BITS, HALVES, ACT>.ensure(a.device, max_cl);
  if (e != cudaSuccess) return e;

  // X as a 3-D bf16 tensor [K/64 blocks][M rows][64]: one box is the two
  // 64-deep stages of a group for 128 rows (128-byte swizzle); rows past M
  // read as zeros.  A copy costs the copy engine about the same whatever its
  // size, so each group's X is one copy.
  CUtensorMap tmx;
  const cuuint64_t gdim[3] = {64, static_cast<cuuint64_t>(a.M), static_cast<cuuint64_t>(a.K / 64)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(a.K) * 2, 128};
  const int tn = a.M <= 64 ? 64 : kTM;  // tokens per MMA and per X box
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(tn), 2};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.X), gdim,
                   gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // The packed weights as a 3-D u32 tensor [N/64 cell columns][G cells x
  // 128-byte rows][32 words]; one box is kChunk consecutive cells of every
  // cell column of a tile.
  CUtensorMap tmw;
  const cuuint64_t groups = static_cast<cuuint64_t>(a.K / 128);
  const cuuint64_t wdim[3] = {32, groups * C::kCellRows,
                              static_cast<cuuint64_t>(a.N / 64)};
  const cuuint64_t wstride[2] = {128, groups * C::kCellBytes};
  const cuuint32_t wbox[3] = {32, static_cast<cuuint32_t>(C::kChunk * C::kCellRows),
                              static_cast<cuuint32_t>(C::kCellCols)};
  r = enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(a.Wp), wdim, wstride,
          wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  WtParams p;
  p.S = static_cast<const uint16_t*>(a.S);
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.G = static_cast<int>(a.K / 128);
  p.mt = static_cast<int>((a.M + kTM - 1) / kTM);
  p.nt = static_cast<int>((a.N + kTN - 1) / kTN);
  p.tn = tn;
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;
  const int64_t tiles = static_cast<int64_t>(p.mt) * p.nt;
  const int ks = HALVES == 1 ? wt_split(tiles, p.G / C::kChunk, a.num_sms, a.split_hint, max_cl) : 1;
  if (ks < 1) return cudaErrorNotSupported;
  p.ks = ks;

  cudaLaunchConfig_t cfg = {};
  // K split: one cluster of ks CTAs per tile; else persistent, one CTA per SM
  cfg.gridDim = dim3(static_cast<unsigned>(ks > 1 ? tiles * ks : (tiles < a.num_sms ? tiles : a.num_sms)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (ks > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = ks;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  if (a.pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_wt_kernel<BITS, HALVES, ACT>, tmx, tmw, p);
}

}  // namespace

// Tiles of 256 weight columns from this M on (measured at K = 2560,
// N = 9728: below it the 128-column tiles fill the GPU better).
constexpr int64_t kWideMinM = 512;

bool gemm_wt_fits(int bits, int64_t M, int64_t K, int64_t N) {
  const int64_t chunk = bits == 4 ? 4 : 2;
  if ((K / 128) % chunk != 0) return false;
  // tile counts and TMA row coordinates stay within 32-bit signed range
  if ((M + kTM - 1) / kTM * ((N + 127) / 128) > INT32_MAX) return false;
  return (bits == 4 ? K * N / 256 : K * N / 128) <= INT32_MAX;
}

cudaError_t launch_gemm_wt(const GemmArgs& a, cudaStream_t stream) {
  if (!gemm_wt_fits(a.bits, a.M, a.K, a.N)) return cudaErrorNotSupported;
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const bool wide = a.M >= kWideMinM;
  if (a.act != 0) {
    if (a.bits == 4)
      return wide ? launch_wt<4, 2, 1>(a, stream, enc) : launch_wt<4, 1, 1>(a, stream, enc);
    return wide ? launch_wt<8, 2, 1>(a, stream, enc) : launch_wt<8, 1, 1>(a, stream, enc);
  }
  if (a.bits == 4)
    return wide ? launch_wt<4, 2, 0>(a, stream, enc) : launch_wt<4, 1, 0>(a, stream, enc);
  return wide ? launch_wt<8, 2, 0>(a, stream, enc) : launch_wt<8, 1, 0>(a, stream, enc);
}

}  // namespace wq
