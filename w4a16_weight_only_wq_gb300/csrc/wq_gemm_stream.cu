// wq_gemm_stream.cu -- tcgen05 W4A16 / W8A16 GEMM for M <= 64 (one launch
// per 16, 32 or 64 tokens) that keeps the weight stream going across
// consecutive launches.
//
// Y[M,N] = X[M,K] . (s (.) q)[K,N] for the verifier's 16-token block
// ("Quantize the Target, Quantize the Drafter": the INT4 target checks an
// anchor plus 15 drafted tokens in one forward), computed as
// Y^T = W^T . X^T on the tensor cores: the dequantised weights bf16(s*q) are
// the tcgen05.mma A operand in tensor memory (M = 128 weight columns, one per
// TMEM lane) and the 16 tokens are the N = 16 operand in shared memory.
//
// At M = 16 a call is bound by streaming the packed weights, and a lone
// launch cannot keep HBM busy: it starts, waits for its first bytes, and
// ends with a reduction while no weight bytes move.  So a CTA here takes
// under half an SM (512 threads, ~108 KiB of shared memory, 256 TMEM
// columns) and the next launch on the stream, started early by programmatic
// dependent launch, shares the SM with it: while this launch multiplies and
// reduces, the next one streams its weights into shared memory and
// dequantises its first groups into tensor memory.  Only the parts that read
// X (the MMAs) or write Y wait for the preceding kernel.
//
//  * Work unit: 128 weight columns x a contiguous range of 128-deep groups;
//    a cluster of `cs` CTAs splits one column tile's K range and each CTA
//    accumulates its range in one TMEM accumulator [128 x 16].  Partial sums
//    go to the owning CTA's shared memory as staged bulk copies counted on
//    the owner's mbarrier, and are added there in rank order.  At a split of
//    2 rank 0 owns the whole tile and takes one group more than half: rank
//    1 finishes earlier and its partial travels while rank 0 still works
//    (the lead split).
//  * Producer (warp 0): the scales of the CTA's range (one TMA), the packed
//    cells of each group (one TMA per group, both 64-column cells, 128-byte
//    swizzle) into a ring, and an L2 prefetch of the groups beyond the ring,
//    all before the programmatic-launch wait.
//  * Three pipelines, one per group residue: pipeline w takes the groups
//    u = w, w + 3, ... with its own dequant set, MMA warp, two half-group
//    A slots in tensor memory (64 k x 128 columns, 32 TMEM columns each:
//    half h of a group goes to slot 2w + h), three X stages and
//    accumulator.  Every barrier thus has one waiting warp, which waits
//    its phases in order (a parity wait two phases ahead would pass at
//    once).  The producer's weight ring is shared, but it holds a
//    multiple of three groups, so each of its slots serves one set.
//  * Dequant (warps 4-15: set w = warps 4 + 4w .. 7 + 4w, one per TMEM lane
//    quadrant): LOP3 extraction, an exact bf16x2 subtraction of the offset
//    and one bf16x2 multiply by the scale give bf16(s*q), stored with
//    tcgen05.st, a group as two halves so that the MMAs of one half run
//    while the other is dequantised.
//  * MMA (warps 1-3, warp-uniform, one elected thread issues): four
//    128x16x16 MMAs per half group.  (Per-CTA traces: a warp needs ~650
//    cycles around each batch of MMAs, so a single MMA warp paced the whole
//    pipeline.)  Each warp waits for the preceding kernel before its first
//    X request (one TMA per group); warp 1 lets the next launch start.
//  * 32 and 64 tokens (M = 17..64 in one launch): the accumulator is TOK
//    columns wide, so only one MMA pipeline fits beside the six A
//    half-slots; warp 1 waits once per group and issues both halves' MMAs,
//    warp 2 requests X, and the epilogue reads the accumulator in 16-token
//    chunks, one per group of four warps.  The cluster's partials go column
//    by column (padded rows, 16-byte accesses), one bulk copy per owner after
//    a relaxed rendezvous, into the owners' idle weight rings, where all 512
//    threads add them.
//  * Epilogue (warps 0-3 once their roles are done, one per lane
//    quadrant): tcgen05.ld of the three accumulators, added in a fixed
//    order, then Y or the cluster reduction.
//  Every wait is bounded; an abort drains copies and MMAs, completes the
//  cluster exchange and frees TMEM.
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

constexpr int kCols = 128;           // weight columns per CTA (MMA M, TMEM lanes)
constexpr int kDqSets = 3;           // sets of four dequant warps (one per quadrant)
constexpr int kHS = 2 * kDqSets;     // half-group A slots in tensor memory, two per set
constexpr uint32_t kTmemCols = 256;  // half of an SM's tensor memory
constexpr int kACol = 64;            // accumulators below column 64, A slots 64..255
constexpr int kMaxGroups = 32;       // groups per CTA (the scales buffer)
constexpr int kMaxSplit = 8;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kEpiWarps = 4;
constexpr int kFirstDqWarp = 4;      // warps 1-3 issue MMAs (as many as there are pipelines)
constexpr int kDqWarps = 4 * kDqSets;
constexpr uint32_t kMmaWaitHintNs = 1000;  // suspend hint of the MMA warps' waits
constexpr int kThreads = (kFirstDqWarp + kDqWarps) * 32;  // 512
constexpr int kChunk = 16;           // tokens per epilogue chunk (16 fp32 registers)
constexpr int kXRegion = 48 * 1024;  // X stages (and, after the MMAs, staged partials)
constexpr int kLeadGroups = 1;       // split 2: rank 0's groups beyond half (see the epilogue)

// TOK tokens per launch (the MMA's N: 16, 32 or 64).  At 16 there are three
// MMA pipelines (one per dequant set, each with its own accumulator); at 32
// and 64 one MMA warp takes every group in order, so that one accumulator of
// TOK columns plus the six A half-slots fit 256 TMEM columns.  Either way
// every mbarrier keeps a single waiting warp that takes its phases in order.
template <int TOK>
struct TokCfg {
  static_assert(TOK == 16 || TOK == 32 || TOK == 64, "16, 32 or 64 tokens");
  static constexpr int kPipes = TOK == 16 ? 3 : 1;
  static_assert(kPipes * TOK <= kACol, "accumulators below the A slots");
  static constexpr int kXGroupBytes = TOK * 256;  // a group's two 64-deep blocks
  static constexpr int kXBlockBytes = TOK * 128;  // one block: TOK rows x 128 bytes
  // X stages: per pipeline kXPer, in all kXG (36 / 48 / 48 KiB)
  static constexpr int kXG = TOK == 16 ? 9 : kXRegion / kXGroupBytes;
  static constexpr int kXPer = kXG / kPipes;
  static_assert(kXG % kPipes == 0 && kXPer >= 2, "X stages per pipeline");
  // 16 tokens: a dedicated buffer receives the cluster's partials at any
  // time; 32 and 64: they are received in the idle weight ring, after a
  // rendezvous that says every CTA of the cluster is done with its ring
  static constexpr int kPartBytes = TOK == 16 ? 10752 : 0;  // >= cs * ceil(128/cs) * (16 + 4) * 4
};

template <int BITS, int TOK>
struct StCfg {
  using T = TokCfg<TOK>;
  static constexpr int kCellBytes = BITS == 4 ? 4096 : 8192;
  static constexpr int kCellRows = kCellBytes / 128;
  static constexpr int kWBytes = 2 * kCellBytes;    // one group of both cells
  // weight groups in the ring: a multiple of the dequant sets, so that slot
  // s only ever holds groups of set s % 3 and its w_full barrier has one
  // waiter taking its phases in order.  (With 7 slots, a set could reach
  // its next group in a slot while another set's earlier group there had
  // not landed yet: its parity wait passed a phase early, and the ring's
  // phases fell out of step.)
  static constexpr int kRing = BITS == 4 ? 6 : 3;
  static_assert(kRing % kDqSets == 0, "one dequant set per ring slot");
  static constexpr int kOffW = 0;
  static constexpr int kOffX = kOffW + kRing * kWBytes;
  static constexpr int kOffS = kOffX + T::kXG * T::kXGroupBytes;
  static constexpr int kOffP = kOffS + kMaxGroups * kCols * 2;
  static constexpr int kOffBar = kOffP + T::kPartBytes;
  static constexpr int kNumBars = 2 * kRing + 2 * T::kXG + 2 * kHS + 4;
  // after the barriers: the TMEM address word and the abort flag (16 bytes),
  // then [kXG] the last group requested per X stage
  static constexpr int kOffXLast = kOffBar + kNumBars * 8 + 16;
  static constexpr int kSmem = kOffXLast + T::kXG * 4 + 1024;  // + alignment slack
  static_assert(kSmem <= 113 * 1024, "two CTAs must fit one SM");
  // partials: staged in the X region (128 columns x at most TOK + 4 floats);
  // received (TOK >= 32) in the weight ring, cs slices of ceil(128 / cs)
  // columns x (TOK + 4) floats (<= 36 KiB)
  static_assert(kCols * (TOK + 4) * 4 <= T::kXG * T::kXGroupBytes, "staged partials fit the X stages");
  static_assert(TOK == 16 || 7 * 19 * (TOK + 4) * 4 <= kRing * kWBytes,
                "received partials fit the ring");
};

struct StParams {
  __nv_bfloat16* Y;
  int M, N, G, cs;
  int lead;           // > 0 (16 tokens, cs = 2): rank 0 takes G / 2 + lead groups and all
                      // 128 columns, rank 1 sends it the partials of the rest
  int ngmax;          // groups of the longest CTA range (scales box rows)
  int act;            // 0 none, 1 SiLU applied to the stored bf16 result
  int prefetch_x;     // pull the CTA's X rows into L2 before the wait
  const uint8_t* Wp;  // packed words (for the L2 prefetch)
  const uint8_t* X;   // X rows (for the L2 prefetch)
  KernelDiag diag;
};

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Y[m][col] = bf16(act(v[m])) for the first `rows` tokens of a 16-token chunk
// of one column (row stride N).  The activation is chosen once, outside the
// stores: inside them the compiler evaluated SiLU for every value even when
// none was asked for (~2,600 cycles per column of 16).
__device__ __forceinline__ void store_column(__nv_bfloat16* y, int N, const float (&v)[kChunk],
                                             int rows, int act) {
  if (act == 0) {
#pragma unroll
    for (int m = 0; m < kChunk; ++m)
      if (m < rows) y[static_cast<size_t>(m) * N] = __float2bfloat16_rn(v[m]);
  } else {
#pragma unroll
    for (int m = 0; m < kChunk; ++m)
      if (m < rows) y[static_cast<size_t>(m) * N] = __float2bfloat16_rn(apply_act(v[m], 1));
  }
}

// Y[m][col] = bf16(act(a.m)) for tokens m = 0..3 (those below `left`) of
// one column (row stride N), the activation chosen outside the stores.
__device__ __forceinline__ void store_quad(__nv_bfloat16* y, int N, float4 a, int left, int act) {
  const size_t n = static_cast<size_t>(N);
  if (act == 0) {
    y[0] = __float2bfloat16_rn(a.x);
    if (left > 1) y[n] = __float2bfloat16_rn(a.y);
    if (left > 2) y[2 * n] = __float2bfloat16_rn(a.z);
    if (left > 3) y[3 * n] = __float2bfloat16_rn(a.w);
  } else {
    y[0] = __float2bfloat16_rn(apply_act(a.x, 1));
    if (left > 1) y[n] = __float2bfloat16_rn(apply_act(a.y, 1));
    if (left > 2) y[2 * n] = __float2bfloat16_rn(apply_act(a.z, 1));
    if (left > 3) y[3 * n] = __float2bfloat16_rn(apply_act(a.w, 1));
  }
}

template <int BITS, int TOK>
__global__ void __launch_bounds__(kThreads, 2)
gemm_stream_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                   const __grid_constant__ CUtensorMap tms, const StParams p) {
  using C = StCfg<BITS, TOK>;
  using T = TokCfg<TOK>;
  constexpr int kRing = C::kRing;
  constexpr int kPipes = T::kPipes, kXG = T::kXG, kXPer = T::kXPer;
  // with one MMA pipeline, warp 2 requests X so that the MMA warp only waits
  // and issues (with three, each MMA warp requests its own pipeline's X)
  constexpr bool kXWarp = kPipes == 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

  float* part = reinterpret_cast<float*>(smem + C::kOffP);  // same offset in every CTA
  const uint16_t* sc = reinterpret_cast<const uint16_t*>(smem + C::kOffS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* w_full = bars;              // [kRing] a group's packed cells landed
  uint64_t* w_empty = w_full + kRing;   // [kRing] dequantised
  uint64_t* x_full = w_empty + kRing;   // [kXG] a group of X landed
  uint64_t* x_empty = x_full + kXG;     // [kXG] MMAs done with it
  uint64_t* a_full = x_empty + kXG;     // [kHS] half group of A written
  uint64_t* a_empty = a_full + kHS;     // [kHS] MMAs done with it
  uint64_t* s_full = a_empty + kHS;     // scales landed
  uint64_t* d_full = s_full + 1;        // every MMA of this CTA has completed
  uint64_t* part_full = d_full + 1;     // every rank's partials of my columns landed
  uint64_t* never_bar = part_full + 1;  // test hook
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* x_last = reinterpret_cast<int*>(smem + C::kOffXLast);  // [kXG] for the drain

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = p.cs;
  const int tile = blockIdx.x / cs;
  const int rank = blockIdx.x % cs;  // == %cluster_ctarank for cluster (cs,1,1)
  // the CTA's groups [g0, g0 + ng): an even split, or with a lead, rank 0
  // ahead by 2 lead groups so that rank 1's partials travel while it works
  const bool lead = TOK == 16 && cs == 2 && p.lead > 0;
  const int g_lead = p.G / 2 + p.lead;
  const int g0 = lead ? (rank == 0 ? 0 : g_lead) : (p.G * rank) / cs;
  const int ng = lead ? (rank == 0 ? g_lead : p.G - g_lead) : (p.G * (rank + 1)) / cs - g0;
  const int n0 = tile * kCols;
  const int rows = min(TOK, p.M);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 4);  // the four quadrant warps of the group's set
    }
    for (int i = 0; i < kXG; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);  // the group's MMA warp
      x_last[i] = -1;
    }
    for (int i = 0; i < kHS; ++i) {
      mbar_init(&a_full[i], 4);  // one dequant warp per lane quadrant
      mbar_init(&a_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(d_full, kPipes);  // one commit per MMA warp
    mbar_init(part_full, 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA of the cluster has initialised its barriers before any remote
  // copy; waited for here, before the weights stream, where it costs
  // nothing (~800 cycles when waited for just before the exchange)
  if (cs > 1) {
    cluster_arrive_relaxed();
    cluster_wait();
  }
  const uint32_t tmem_base = *tmem_slot;
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  int issued_w = 0;
  if (warp == kProducerWarp) {
    // ------------------------------------------------------- producer ---
    // Weights and scales do not depend on the preceding kernel: everything
    // here may run before it completes.
    if (lane == 0) {
      prefetch_tensor_map(&tmw);
      prefetch_tensor_map(&tms);
      mbar_arrive_expect_tx(s_full, p.ngmax * kCols * 2);
      tma_load_2d(smem + C::kOffS, &tms, n0, g0, s_full);
      for (int c = 0; c < min(kRing, ng); ++c) {
        mbar_arrive_expect_tx(&w_full[c], C::kWBytes);
        tma_load_3d(smem + C::kOffW + c * C::kWBytes, &tmw, 0, (g0 + c) * C::kCellRows, 2 * tile,
                    &w_full[c]);
        issued_w = c + 1;
      }
      // the groups beyond the ring: into L2 now, into the ring when a slot
      // frees up (after this launch's MMAs start)
      if (ng > kRing) {
        const int ncells = min(2, (p.N - n0) / 64);
        for (int ci = 0; ci < ncells; ++ci) {
          const size_t cell0 = (static_cast<size_t>(2 * tile + ci) * p.G + g0 + kRing);
          prefetch_l2_bulk(p.Wp + cell0 * C::kCellBytes,
                           static_cast<uint32_t>((ng - kRing) * C::kCellBytes));
        }
      }
      int slot = 0;
      uint32_t ph = 0;  // phase of the slot's previous use
      for (int c = kRing; c < ng; ++c) {
        if (!role_wait(&w_empty[slot], ph, p.diag, abort_flag, 2000)) break;
        mbar_arrive_expect_tx(&w_full[slot], C::kWBytes);
        tma_load_3d(smem + C::kOffW + slot * C::kWBytes, &tmw, 0, (g0 + c) * C::kCellRows,
                    2 * tile, &w_full[slot]);
        issued_w = c + 1;
        if (++slot == kRing) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp < kMmaWarp + kPipes + (kXWarp ? 1 : 0)) {
    // --------------------------------------------------- MMA issuers ---
    // Warp kMmaWarp + w (w < kPipes) takes the groups u = w, w + kPipes, ...
    // (group u's A slots are its dequant set's, 2 (u % 3) and 2 (u % 3) + 1;
    // its X stages w, w + kPipes, ... in turn) into its own accumulator (TMEM
    // columns TOK w .. TOK w + TOK - 1).  With one pipeline, warp
    // kMmaWarp + 1 requests the X stages instead of the MMA warp.
    const int w = warp - kMmaWarp;
    auto issue_x = [&](int u, int xs) {
      if (elect_one()) {
        mbar_arrive_expect_tx(&x_full[xs], T::kXGroupBytes);
        tma_load_3d(smem + C::kOffX + xs * T::kXGroupBytes, &tmx, 0, 0, 2 * (g0 + u), &x_full[xs]);
        x_last[xs] = u;
      }
      __syncwarp();
    };
    const bool x_issuer = kXWarp ? w == kPipes : true;  // requests X for pipeline (kXWarp ? 0 : w)
    if (x_issuer) {
      if ((kXWarp || w == 0) && p.prefetch_x) {
        // X rows of this CTA's K range into L2: harmless before the wait (a
        // prefetch changes no data) and it hides HBM latency when X is cold
        for (int r = lane; r < rows; r += 32)
          prefetch_l2_bulk(p.X + (static_cast<size_t>(r) * p.G + g0) * 256,
                           static_cast<uint32_t>(ng) * 256);
      }
      if (lane == 0) prefetch_tensor_map(&tmx);
      pdl_wait_primary();  // X may be the preceding kernel's output
      if (kXWarp || w == 0) pdl_launch_dependents();  // the next launch may stream its weights
      const int pw = kXWarp ? 0 : w;
      for (int k = 0; k < kXPer && pw + kPipes * k < ng; ++k)
        issue_x(pw + kPipes * k, pw + kPipes * k);
    }
    if (kXWarp && w == kPipes) {
      // the X warp: refill stage u % kXPer with group u once group
      // u - kXPer's MMAs are done with it
      for (int u = kXPer; u < ng; ++u) {
        if (!role_wait(&x_empty[u % kXPer], static_cast<uint32_t>((u / kXPer - 1) & 1), p.diag,
                       abort_flag, kMmaWaitHintNs))
          break;
        issue_x(u, u % kXPer);
      }
    } else {
    constexpr uint32_t idesc = idesc_bf16_f32(kCols, TOK);
    const uint64_t xdesc0 = smem_desc_sw128(smem_addr(smem + C::kOffX));
    const uint32_t d_tmem = tmem_base + TOK * w;
    int xk = 0;  // this group's X stage among the pipeline's kXPer
    for (int u = w, k = 0; u < ng; u += kPipes, ++k) {
      const int xs = w + kPipes * xk;
      const uint32_t xph = static_cast<uint32_t>((k / kXPer) & 1);
      const bool hook = p.diag.force_timeout == 2 && 2 * u >= ng;
      bool ok = true;
      // group u's dequant set and the phase of its A slots (with one
      // pipeline per set these are the warp's own and k)
      const int set = kPipes == kDqSets ? w : u % kDqSets;
      const uint32_t aph = static_cast<uint32_t>((kPipes == kDqSets ? k : u / kDqSets) & 1);
      if constexpr (kPipes == 1) {
        // One warp issues every group, so its per-group steps are the MMA
        // phase's pace: one wait for A, one for X, then both halves' MMAs
        // from one elected thread.  Each warp of the set arrives on half 1's
        // barrier after its half-0 stores and arrival, so half 1 complete
        // means the whole group's A is in tensor memory.  (Waiting and
        // issuing per half, with the SM shared by the dequant warps, took
        // ~1,000 cycles per group.)
        if (!role_wait(hook ? never_bar : &a_full[2 * set + 1], hook ? 0u : aph, p.diag, abort_flag,
                       kMmaWaitHintNs) ||
            !role_wait(&x_full[xs], xph, p.diag, abort_flag, kMmaWaitHintNs)) {
          ok = false;
        } else {
          tc_fence_after();
          const uint64_t bd = xdesc0 + static_cast<uint64_t>((xs * T::kXGroupBytes) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a_tmem = tmem_base + kACol + (2 * set + h) * 32;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                umma_bf16_ts(d_tmem, a_tmem + 8 * j,
                             bd + static_cast<uint64_t>((h * T::kXBlockBytes) >> 4) +
                                 static_cast<uint64_t>(2 * j),
                             idesc, (k | h | j) != 0);
              umma_commit(&a_empty[2 * set + h]);
            }
            umma_commit(&x_empty[xs]);
          }
          __syncwarp();
        }
      } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int hs = 2 * set + h;
        // (the waits suspend the warp instead of spinning: the next
        // launch's MMA warps wait here for microseconds while this SM's
        // other CTA dequantises)
        if (!role_wait(hook ? never_bar : &a_full[hs], hook ? 0u : aph, p.diag, abort_flag,
                       kMmaWaitHintNs) ||
            (h == 0 && !role_wait(&x_full[xs], xph, p.diag, abort_flag, kMmaWaitHintNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_tmem = tmem_base + kACol + hs * 32;
        // block h of the group's X stage
        const uint64_t bd =
            xdesc0 + static_cast<uint64_t>((xs * T::kXGroupBytes + h * T::kXBlockBytes) >> 4);
        // one elected thread issues the half's four MMAs and the commits (a
        // probe: ~22 cycles per MMA this way, 40 with an election per MMA)
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma_bf16_ts(d_tmem, a_tmem + 8 * j, bd + static_cast<uint64_t>(2 * j), idesc,
                         (k | h | j) != 0);
          umma_commit(&a_empty[hs]);
          if (h == 1) umma_commit(&x_empty[xs]);
        }
        __syncwarp();
      }
      }
      if (!ok) break;
      // refill the X stage of this pipeline's previous group (whose MMAs
      // have most likely completed) with the group kXPer after it
      if (!kXWarp && k >= 1) {
        const int pk = (xk + kXPer - 1) % kXPer, pu = u - kPipes;
        if (pu + kPipes * kXPer < ng) {
          if (!role_wait(&x_empty[w + kPipes * pk], static_cast<uint32_t>(((k - 1) / kXPer) & 1),
                         p.diag, abort_flag, kMmaWaitHintNs))
            break;
          issue_x(pu + kPipes * kXPer, w + kPipes * pk);
        }
      }
      if (++xk == kXPer) xk = 0;
    }
    // arrives when every MMA this warp issued has completed
    if (elect_one()) umma_commit(d_full);
    __syncwarp();
    }
  } else if (warp >= kFirstDqWarp) {
    // ------------------------------------------------- dequant warps ---
    // Quadrant q = warp % 4 (the TMEM lanes this warp may write); set ds
    // takes the groups u = ds, ds + 3, ..., half h into A slot 2 ds + h.
    const int q = warp & 3, ds = (warp - kFirstDqWarp) >> 2;
    const int n = 32 * q + lane;  // weight column within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t cell_off = (n >> 6) * C::kCellBytes;
    const LaneOffsets<BITS> lo(n & 63);  // the thread's chunk offsets, once
    if (role_wait(s_full, 0, p.diag, abort_flag, 2000)) {
      bool ok = true;
      for (int u = ds, k = 0; u < ng && ok; u += 3, ++k) {
        const int slot = u % kRing;
        if (!role_wait(&w_full[slot], (u / kRing) & 1, p.diag, abort_flag, 2000)) break;
        const uint32_t s1 = sc[u * kCols + n];
        const uint32_t cell = smem_addr(smem + C::kOffW + slot * C::kWBytes) + cell_off;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int hs = 2 * ds + h;
          if (k > 0 && !role_wait(&a_empty[hs], static_cast<uint32_t>((k - 1) & 1), p.diag,
                                  abort_flag, 2000)) {
            ok = false;
            break;
          }
          tc_fence_after();
          dequant_half_to_tmem<BITS>(cell, lo, h, s1 | (s1 << 16),
                                     tmem_base + lane_addr + kACol + hs * 32);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[hs]);
        }
        // (the slot was only read here; the barrier hand-off orders those
        // reads before the producer's refill)
        if (ok && lane == 0) mbar_arrive(&w_empty[slot]);
      }
    }
  }

  // ------------------------------------------------------- epilogue ---
  // Two forms of the same steps: at 16 tokens the thread's 16 partials are
  // read once into registers (this form needs no register spill); at 32 and
  // 64 tokens the epilogue works in 16-token chunks, which also changes
  // where the cluster's partials are received.
  if constexpr (TOK == 16) {
    // Accumulators D_w[column n][token m] (w = 0..2): thread n of warps 0-3
    // (lane quadrant = warp) adds its column's three 16-token partials in
    // order.  (A warp without a task, when the CTA has a single group, left
    // its accumulator unwritten.)
    float v[TOK];
#pragma unroll
    for (int m = 0; m < TOK; ++m) v[m] = 0.f;
    const bool epi = warp < kEpiWarps;
    const int en = 32 * warp + lane;  // the epilogue thread's column
    if (epi) {
      pdl_wait_primary();  // Y may be read or written by the preceding kernel
      if (role_wait(d_full, 0, p.diag, abort_flag, 200)) {
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * warp) << 16);
        uint32_t r0[16], r1[16];
        tmem_ld_32x32b_x16(taddr, r0);
        if (ng > 1) tmem_ld_32x32b_x16(taddr + 16, r1);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < TOK; ++m)
          v[m] = __uint_as_float(r0[m]) + (ng > 1 ? __uint_as_float(r1[m]) : 0.f);
        if (ng > 2) {  // pipeline 2 starts at the third group
          tmem_ld_32x32b_x16(taddr + 32, r0);
          tmem_ld_wait();
#pragma unroll
          for (int m = 0; m < TOK; ++m) v[m] += __uint_as_float(r0[m]);
        }
      }
    }
    // Roles that ran on one lane rejoin their warp before the block-wide
    // barrier, which a diverged warp must not reach.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
      // Let every issued copy land and every issued MMA finish (bounded, at
      // least 1 s) before shared and tensor memory are released.
      KernelDiag drain = p.diag;
      if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
      if (warp == kProducerWarp && lane == 0) {
        mbar_wait_bounded(s_full, 0, drain);
        for (int s = 0; s < kRing && s < issued_w; ++s) {
          const int last = s + ((issued_w - 1 - s) / kRing) * kRing;
          mbar_wait_bounded(&w_full[s], (last / kRing) & 1, drain);
        }
      }
      if (warp == kMmaWarp && lane == 0) {
        // group u sits in stage u % kPipes + kPipes ((u / kPipes) % kXPer), phase (u / kPipes / kXPer) & 1
        for (int s = 0; s < kXG; ++s)
          if (x_last[s] >= 0)
            mbar_wait_bounded(&x_full[s], static_cast<uint32_t>((x_last[s] / kPipes / kXPer) & 1), drain);
        mbar_wait_bounded(d_full, 0, drain);
      }
      __syncwarp();
      __syncthreads();
    }
    if (cs == 1) {
      if (epi && n0 + en < p.N) store_column(p.Y + n0 + en, p.N, v, rows, p.act);
    } else {
      // Rank r owns the tile's columns [128 r / cs, 128 (r + 1) / cs).  Each
      // CTA stages its 16 token partials per column in its (now idle) X ring,
      // column-major in rows of 16 + 4 floats (with the pad a warp's 16-byte
      // accesses of consecutive columns fall on distinct banks), so that
      // every owner's columns are one contiguous block, and sends each owner
      // its block with one bulk copy counted on the owner's part_full; slice
      // q of the owner's `part` holds rank q's block.  Every thread of the
      // owner then adds the slices, in rank order, for one (column, 4
      // tokens).  Measured against the alternatives: byte-counted 16-byte
      // remote stores serialise on the owner's barrier (1.2 us more), and
      // plain remote stores need a release/acquire cluster barrier (0.3 us
      // more).  Every rank sends its blocks even after an abort, so every
      // owner's count completes.
      constexpr int kRow = TOK + 4;  // floats per staged column
      const int slice = (kCols + cs - 1) / cs;
      const int cb0 = (rank * kCols) / cs, ncol = ((rank + 1) * kCols) / cs - cb0;
      float* stage = reinterpret_cast<float*>(smem + C::kOffX);
      if (lead) {
        // Rank 0 owns all 128 columns and ran G / 2 + lead groups; rank 1,
        // with fewer, finished earlier and sends all of its partials (8 KiB)
        // while rank 0 still works, so their transfer is off the critical
        // path.  Rank 0 adds its own partial and rank 1's, in rank order.
        if (rank == 0 && threadIdx.x == 0)
          mbar_arrive_expect_tx(part_full, static_cast<uint32_t>(kCols * kRow * 4));
        if (epi && rank == 1) {
          const uint32_t dst = smem_addr(stage + en * kRow);
#pragma unroll
          for (int i = 0; i < TOK / 4; ++i)
            st_shared_v4(dst + 16 * i, __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                         __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
          fence_proxy_async_smem();  // the bulk copy reads what these threads wrote
          named_barrier_sync(1, kEpiWarps * 32);
          if (en == 0)
            dsmem_bulk_copy(dsmem_map(part, 0), smem_addr(stage),
                            static_cast<uint32_t>(kCols * kRow * 4), dsmem_map(part_full, 0));
        }
        if (epi && rank == 0) {
          if (!mbar_wait_bounded(part_full, 0, p.diag)) {
            // a peer can be late by its own timed-out wait plus its drain
            KernelDiag late = p.diag;
            late.wait_limit_ns = p.diag.wait_limit_ns + 2000000000ull;
            mbar_wait_bounded(part_full, 0, late);
          }
          const uint32_t src = smem_addr(part + en * kRow);
#pragma unroll
          for (int i = 0; i < TOK / 4; ++i) {
            const float4 f = ld_shared_v4_f32(src + 16 * i);
            v[4 * i] += f.x;
            v[4 * i + 1] += f.y;
            v[4 * i + 2] += f.z;
            v[4 * i + 3] += f.w;
          }
          if (n0 + en < p.N) store_column(p.Y + n0 + en, p.N, v, rows, p.act);
        }
      } else if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(part_full, static_cast<uint32_t>(cs * ncol * kRow * 4));
      }
      if (!lead && epi) {
        const uint32_t dst = smem_addr(stage + en * kRow);
#pragma unroll
        for (int i = 0; i < TOK / 4; ++i)
          st_shared_v4(dst + 16 * i, __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                       __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
        fence_proxy_async_smem();  // the bulk copies read what these threads wrote
        named_barrier_sync(1, kEpiWarps * 32);
        if (en < cs) {
          const int r = en;  // one thread per destination rank
          const int rb0 = (r * kCols) / cs, rn = ((r + 1) * kCols) / cs - rb0;
          dsmem_bulk_copy(dsmem_map(part + rank * slice * kRow, r), smem_addr(stage + rb0 * kRow),
                          static_cast<uint32_t>(rn * kRow * 4), dsmem_map(part_full, r));
        }
      }
      // one (column c, 4 tokens t4) per thread, c the faster index: at most
      // 128 columns x 4 quads = kThreads items
      const int nq = (rows + 3) / 4;
      if (!lead && static_cast<int>(threadIdx.x) < ncol * nq) {
        const int t4 = threadIdx.x / ncol, c = threadIdx.x - t4 * ncol;
        if (!mbar_wait_bounded(part_full, 0, p.diag)) {
          // a peer can be late by its own timed-out wait plus its drain
          KernelDiag late = p.diag;
          late.wait_limit_ns = p.diag.wait_limit_ns + 2000000000ull;
          mbar_wait_bounded(part_full, 0, late);
        }
        float4 a = ld_shared_v4_f32(smem_addr(part + c * kRow) + 16 * t4);
        for (int qq = 1; qq < cs; ++qq) {
          const float4 f = ld_shared_v4_f32(smem_addr(part + (qq * slice + c) * kRow) + 16 * t4);
          a.x += f.x;
          a.y += f.y;
          a.z += f.z;
          a.w += f.w;
        }
        if (n0 + cb0 + c < p.N)
          store_quad(p.Y + static_cast<size_t>(4 * t4) * p.N + n0 + cb0 + c, p.N, a, rows - 4 * t4,
                     p.act);
      }
      // No CTA leaves while a peer's copy may still read or write its shared
      // memory.  The owners have waited for all of their bytes before
      // arriving, so every copy has completed once all have arrived; the
      // barrier orders nothing else (relaxed: it does not wait for this CTA's
      // Y stores to become visible).
      __syncwarp();
      cluster_arrive_relaxed();
      cluster_wait();
    }
  } else {
    // Accumulators D_w[column n][token m] (w < kPipes, TMEM columns TOK w ..)
    // are read in chunks of 16 tokens, the pipelines' partials added in
    // order: warp w reads chunk w / 4 of the columns of its lane quadrant
    // w % 4 (thread n = 32 (w % 4) + lane, column n), so the TOK / 16 chunks
    // are read by as many groups of four warps at once.  Warps 0-3 read
    // chunk 0 as soon as the MMAs complete, the others after the block-wide
    // barrier that passes that on.  (A pipeline without a group, when the
    // CTA has fewer groups than pipelines, left its accumulator unwritten.)
    const bool epi = warp < kEpiWarps;
    const int en = 32 * (warp & 3) + lane;  // the thread's column
    const int cw = warp >> 2;               // the warp's chunk of tokens
    const bool has_chunk = cw < TOK / kChunk && kChunk * cw < rows;
    bool have = false;
    if (epi) {
      pdl_wait_primary();  // Y may be read or written by the preceding kernel
      have = role_wait(d_full, 0, p.diag, abort_flag, 200);
    }
    auto load_chunk = [&](int c, float (&v)[kChunk]) {
#pragma unroll
      for (int m = 0; m < kChunk; ++m) v[m] = 0.f;
      if (!have) return;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kChunk * c;
      if constexpr (kPipes == 3) {
        uint32_t r0[kChunk], r1[kChunk];
        tmem_ld_32x32b_x16(taddr, r0);
        if (ng > 1) tmem_ld_32x32b_x16(taddr + TOK, r1);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < kChunk; ++m)
          v[m] = __uint_as_float(r0[m]) + (ng > 1 ? __uint_as_float(r1[m]) : 0.f);
        if (ng > 2) {  // pipeline 2 starts at the third group
          tmem_ld_32x32b_x16(taddr + 2 * TOK, r0);
          tmem_ld_wait();
#pragma unroll
          for (int m = 0; m < kChunk; ++m) v[m] += __uint_as_float(r0[m]);
        }
      } else {
        uint32_t r0[kChunk];
        tmem_ld_32x32b_x16(taddr, r0);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < kChunk; ++m) v[m] = __uint_as_float(r0[m]);
      }
    };
    float v0[kChunk];  // tokens 0..15, read before the block-wide barrier
    if (epi) {
      tc_fence_after();
      load_chunk(0, v0);
    }
    // Roles that ran on one lane rejoin their warp before the block-wide
    // barrier, which a diverged warp must not reach.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
      // Let every issued copy land and every issued MMA finish (bounded, at
      // least 1 s) before shared and tensor memory are released.
      KernelDiag drain = p.diag;
      if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
      if (warp == kProducerWarp && lane == 0) {
        mbar_wait_bounded(s_full, 0, drain);
        for (int s = 0; s < kRing && s < issued_w; ++s) {
          const int last = s + ((issued_w - 1 - s) / kRing) * kRing;
          mbar_wait_bounded(&w_full[s], (last / kRing) & 1, drain);
        }
      }
      if (warp == kMmaWarp && lane == 0) {
        // group u sits in stage u % kPipes + kPipes ((u / kPipes) % kXPer),
        // phase (u / kPipes / kXPer) & 1; each X stage's MMA warp issued its
        // copies, and x_last holds the last group requested per stage
        for (int s = 0; s < kXG; ++s)
          if (x_last[s] >= 0)
            mbar_wait_bounded(&x_full[s], static_cast<uint32_t>((x_last[s] / kPipes / kXPer) & 1),
                              drain);
        mbar_wait_bounded(d_full, 0, drain);
      }
      __syncwarp();
      __syncthreads();
    }
    if (!epi && has_chunk) {
      // the MMAs completed before the barrier (warps 0-3 saw d_full); after
      // an abort the chunk stays zero (the result is reported as failed)
      have = *abort_flag == 0;
      tc_fence_after();
      load_chunk(cw, v0);
    }
    if (cs == 1) {
      if (has_chunk && n0 + en < p.N)
        store_column(p.Y + static_cast<size_t>(kChunk * cw) * p.N + n0 + en, p.N, v0,
                     rows - kChunk * cw, p.act);
    } else {
      // Rank r owns the tile's columns [128 r / cs, 128 (r + 1) / cs).  Each
      // CTA stages its partials in its (now idle) X stages column by column,
      // TOK + 4 floats per column (a thread's 16 tokens are four 16-byte
      // stores; with the 16-byte pad a warp's consecutive columns fall on
      // distinct banks), so that every owner's columns are one contiguous
      // block, and sends every other owner its block with one bulk copy
      // counted on the owner's part_full, into the owner's weight ring, after
      // a relaxed cluster rendezvous (every CTA is done with its ring).  Slice
      // q of the receive buffer is rank q's block, and the owner's own block
      // is read in place from its stage (copying it to itself through the
      // cluster cost 0.9 us at M = 64, 2560 x 9728): all 512 threads then add
      // the slices in rank order, four tokens of one column at a time,
      // consecutive threads on consecutive columns, so the Y stores of a row
      // coalesce.
      // (Token-major blocks added one float at a time took ~500 cycles per
      // item at a split of 2: a chain of dependent accesses per thread, with
      // only 16 warps to hide it.)  Every rank sends its blocks even after an
      // abort, so every owner's count completes.
      constexpr int kRow = TOK + 4;  // floats per staged column
      const int cb0 = (rank * kCols) / cs, ncol = ((rank + 1) * kCols) / cs - cb0;
      float* stage = reinterpret_cast<float*>(smem + C::kOffX);
      const float4* recv = reinterpret_cast<const float4*>(smem + C::kOffW);
      if (threadIdx.x == 0)
        mbar_arrive_expect_tx(part_full, static_cast<uint32_t>((cs - 1) * ncol * kRow * 4));
      // (chunks of tokens past M are not staged: the owners never read them)
      if (has_chunk) {
        float4* dst = reinterpret_cast<float4*>(stage + en * kRow + kChunk * cw);
#pragma unroll
        for (int i = 0; i < kChunk / 4; ++i)
          dst[i] = make_float4(v0[4 * i], v0[4 * i + 1], v0[4 * i + 2], v0[4 * i + 3]);
        fence_proxy_async_smem();  // the bulk copies read what these threads wrote
      }
      __syncthreads();
      cluster_arrive_relaxed();
      cluster_wait();  // every CTA of the cluster is done with its weight ring
      if (threadIdx.x < cs && threadIdx.x != rank) {
        const int r = threadIdx.x;  // one thread per other rank (its own block is read in place)
        const int rb0 = (r * kCols) / cs, rn = ((r + 1) * kCols) / cs - rb0;
        dsmem_bulk_copy(
            dsmem_map_addr(smem_addr(smem + C::kOffW) + static_cast<uint32_t>(rank * rn * kRow * 4), r),
            smem_addr(stage) + static_cast<uint32_t>(rb0 * kRow * 4),
            static_cast<uint32_t>(rn * kRow * 4), dsmem_map(part_full, r));
      }
      if (!mbar_wait_bounded(part_full, 0, p.diag)) {
        // a peer can be late by its own timed-out wait plus its drain
        KernelDiag late = p.diag;
        late.wait_limit_ns = p.diag.wait_limit_ns + 2000000000ull;
        mbar_wait_bounded(part_full, 0, late);
      }
      // item (column c, token quad t4), c the faster index; a thread's next
      // item is kThreads further, so (t4, c) advance by a fixed step
      constexpr int kRow4 = kRow / 4;
      const int nq = (rows + 3) / 4;  // quads holding a token below M
      const int dq = kThreads / ncol, dc = kThreads - dq * ncol;
      const float4* own = reinterpret_cast<const float4*>(stage + cb0 * kRow);
      auto owner_sum = [&](int t4, int c) {
        float4 acc = rank == 0 ? own[c * kRow4 + t4] : recv[c * kRow4 + t4];
        for (int q = 1; q < cs; ++q) {
          const float4 v = q == rank ? own[c * kRow4 + t4] : recv[(q * ncol + c) * kRow4 + t4];
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        return acc;
      };
      const int q0 = threadIdx.x / ncol, c0 = threadIdx.x - q0 * ncol;
      if (p.act == 0) {
        for (int t4 = q0, c = c0; t4 < nq;) {
          if (n0 + cb0 + c < p.N) {
            const float4 a = owner_sum(t4, c);
            __nv_bfloat16* y = p.Y + static_cast<size_t>(4 * t4) * p.N + n0 + cb0 + c;
            const int left = rows - 4 * t4;
            y[0] = __float2bfloat16_rn(a.x);
            if (left > 1) y[p.N] = __float2bfloat16_rn(a.y);
            if (left > 2) y[2 * static_cast<size_t>(p.N)] = __float2bfloat16_rn(a.z);
            if (left > 3) y[3 * static_cast<size_t>(p.N)] = __float2bfloat16_rn(a.w);
          }
          t4 += dq;
          c += dc;
          if (c >= ncol) {
            c -= ncol;
            ++t4;
          }
        }
      } else {
        for (int t4 = q0, c = c0; t4 < nq;) {
          if (n0 + cb0 + c < p.N) {
            const float4 a = owner_sum(t4, c);
            __nv_bfloat16* y = p.Y + static_cast<size_t>(4 * t4) * p.N + n0 + cb0 + c;
            const int left = rows - 4 * t4;
            y[0] = __float2bfloat16_rn(apply_act(a.x, 1));
            if (left > 1) y[p.N] = __float2bfloat16_rn(apply_act(a.y, 1));
            if (left > 2) y[2 * static_cast<size_t>(p.N)] = __float2bfloat16_rn(apply_act(a.z, 1));
            if (left > 3) y[3 * static_cast<size_t>(p.N)] = __float2bfloat16_rn(apply_act(a.w, 1));
          }
          t4 += dq;
          c += dc;
          if (c >= ncol) {
            c -= ncol;
            ++t4;
          }
        }
      }
      // No CTA leaves while a peer's copy may still read or write its shared
      // memory.  The owners have waited for all of their bytes before
      // arriving, so every copy has completed once all have arrived; the
      // barrier orders nothing else (relaxed: it does not wait for this CTA's
      // Y stores to become visible).
      __syncwarp();
      cluster_arrive_relaxed();
      cluster_wait();
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kProducerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side ---

// Never launched: its occupancy answers how many clusters of each size find
// room when only one CTA fits an SM.
__global__ void __launch_bounds__(128, 1) st_room_probe_kernel() {}
constexpr int kProbeSmem = 160 * 1024;  // more than half of an SM

// Per device: the kernel's shared-memory attributes, and for every cluster
// size 1..8 how many clusters fit at once in one CTA slot per SM -- the room
// a launch finds while its neighbour holds the other slot.  (The occupancy
// calculator counts one CTA of this kernel per SM, while two run side by
// side, so the count is taken on the probe kernel above.)
template <int BITS, int TOK>
struct StInit {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
  int room[64][kMaxSplit + 1] = {};
  cudaError_t ensure(int device, int (&out)[kMaxSplit + 1]) {
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> lk(mu);
      if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_stream_kernel<BITS, TOK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             StCfg<BITS, TOK>::kSmem);
        if (e != cudaSuccess) return e;
        // all of the unified L1/shared memory as shared, so that two CTAs
        // (this launch's and the next one's) fit one SM
        e = cudaFuncSetAttribute(gemm_stream_kernel<BITS, TOK>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(st_room_probe_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
        if (e != cudaSuccess) return e;
        for (int c = 1; c <= kMaxSplit; ++c) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(c);
          cfg.blockDim = dim3(128);
          cfg.dynamicSmemBytes = kProbeSmem;
          cudaLaunchAttribute at;
          at.id = cudaLaunchAttributeClusterDimension;
          at.val.clusterDim.x = c;
          at.val.clusterDim.y = 1;
          at.val.clusterDim.z = 1;
          cfg.attrs = &at;
          cfg.numAttrs = 1;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, st_room_probe_kernel, &cfg) != cudaSuccess) n = 0;
          room[device & 63][c] = n;
        }
        cudaGetLastError();  // a refused size above is not an error of this call
        done.fetch_or(bit, std::memory_order_release);
      }
    }
    for (int c = 0; c <= kMaxSplit; ++c) out[c] = room[device & 63][c];
    return cudaSuccess;
  }
};
StInit<4, 16> g_st4_16;
StInit<4, 32> g_st4_32;
StInit<4, 64> g_st4_64;
StInit<8, 16> g_st8_16;
StInit<8, 32> g_st8_32;
StInit<8, 64> g_st8_64;

// The kernel attributes of (bits, TOK) on `device`, and the cluster room
// (the same for every TOK: the footprints differ by a few KiB at most).
cudaError_t st_ensure(int bits, int tok, int device, int (&room)[kMaxSplit + 1]) {
  if (bits == 4)
    return tok == 16 ? g_st4_16.ensure(device, room)
                     : tok == 32 ? g_st4_32.ensure(device, room) : g_st4_64.ensure(device, room);
  return tok == 16 ? g_st8_16.ensure(device, room)
                   : tok == 32 ? g_st8_32.ensure(device, room) : g_st8_64.ensure(device, room);
}

// The K split: the largest cs <= 8 (and <= the groups) whose CTAs fill at
// most one slot per SM (the other slot is for the neighbouring launch) and
// whose clusters find room in one slot per SM (room[cs], with 10% slack:
// the neighbour's CTAs do not always sit one per SM).  Clusters that find no
// room start only when the neighbouring launch ends (a 9728 x 2560 call with
// 20 clusters of 7 had some CTAs start 6 us late).  room == nullptr (no
// device to ask): the SM count alone.
int st_split(int64_t tiles, int64_t G, int num_sms, int hint, const int* room) {
  if (hint > 0) return (hint <= kMaxSplit && hint <= G) ? hint : -1;
  int best = 1;
  for (int cs = 1; cs <= kMaxSplit && cs <= G; ++cs) {
    if (tiles * cs > num_sms) continue;
    if (room != nullptr && cs > 1 && tiles * 10 > room[cs] * 11) continue;
    best = cs;
  }
  return best;
}

const int* st_caps(int bits, int device) {
  static thread_local int caps[kMaxSplit + 1];
  if (device < 0) return nullptr;
  const cudaError_t e = st_ensure(bits, 16, device, caps);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return caps;
}

}  // namespace

int gemm_stream_split(int bits, int64_t K, int64_t N, int split_hint, int num_sms, int device) {
  const int64_t G = K / 128, tiles = (N + kCols - 1) / kCols;
  const int cs = st_split(tiles, G, num_sms, split_hint, st_caps(bits, device));
  if (cs < 1) return -1;
  if ((G + cs - 1) / cs > kMaxGroups) return -1;  // the scales of a CTA's range
  const int64_t cell_rows = bits == 4 ? 32 : 64;
  if (G * cell_rows >= (int64_t(1) << 31) || N / 64 >= (int64_t(1) << 31)) return -1;
  return cs;
}

bool gemm_stream_fits(int bits, int64_t K, int64_t N, int split_hint, int num_sms, int device) {
  return gemm_stream_split(bits, K, N, split_hint, num_sms, device) > 0;
}

cudaError_t launch_gemm_stream(const GemmArgs& a, cudaStream_t stream) {
  if (a.M > kMaxStreamRows || a.M < 1) return cudaErrorNotSupported;
  // the MMA's N: the smallest of 16, 32, 64 tokens that holds M
  const int tok = a.M <= 16 ? 16 : a.M <= 32 ? 32 : 64;
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  int room[kMaxSplit + 1];
  cudaError_t e = st_ensure(a.bits, tok, a.device, room);
  if (e != cudaSuccess) return e;
  const int cs = gemm_stream_split(a.bits, a.K, a.N, a.split_hint, a.num_sms, a.device);
  if (cs < 1 || room[cs] < 1) return cudaErrorNotSupported;
  const int64_t G = a.K / 128, tiles = (a.N + kCols - 1) / kCols;
  // split 2 at 16 tokens: rank 0 takes kLeadGroups more than half (both
  // ranks keep at least one group, and rank 0 at most the scales buffer)
  int lead = 0;
  if (tok == 16 && cs == 2) {
    lead = kLeadGroups;
    while (lead > 0 && (G / 2 + lead > G - 1 || G / 2 + lead > kMaxGroups)) --lead;
  }
  const int ngmax = lead > 0 ? static_cast<int>(G / 2 + lead) : static_cast<int>((G + cs - 1) / cs);

  // X as a 3-D bf16 tensor [K/64 blocks][M rows][64]; one box is a group's
  // two 64-deep blocks for `tok` rows (128-byte swizzle); rows past M read as
  // zeros.
  CUtensorMap tmx;
  const cuuint64_t xdim[3] = {64, static_cast<cuuint64_t>(a.M), static_cast<cuuint64_t>(a.K / 64)};
  const cuuint64_t xstride[2] = {static_cast<cuuint64_t>(a.K) * 2, 128};
  const cuuint32_t xbox[3] = {64, static_cast<cuuint32_t>(tok), 2};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.X), xdim,
                   xstride, xbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // The packed weights as a 3-D u32 tensor [N/64 cell columns][G cells x
  // 128-byte rows][32 words]; one box is one group's cell of both cell
  // columns of a tile (a column past N reads as zeros).
  CUtensorMap tmw;
  const int cell_rows = a.bits == 4 ? StCfg<4, 16>::kCellRows : StCfg<8, 16>::kCellRows;
  const int cell_bytes = a.bits == 4 ? StCfg<4, 16>::kCellBytes : StCfg<8, 16>::kCellBytes;
  const cuuint64_t wdim[3] = {32, static_cast<cuuint64_t>(G) * cell_rows,
                              static_cast<cuuint64_t>(a.N / 64)};
  const cuuint64_t wstride[2] = {128, static_cast<cuuint64_t>(G) * cell_bytes};
  const cuuint32_t wbox[3] = {32, static_cast<cuuint32_t>(cell_rows), 2};
  r = enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(a.Wp), wdim, wstride,
          wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // The scales as a 2-D bf16 tensor [G rows][N]; one box is 128 columns of
  // the longest CTA range (rows and columns past the tensor read as zeros).
  CUtensorMap tms;
  const cuuint64_t sdim[2] = {static_cast<cuuint64_t>(a.N), static_cast<cuuint64_t>(G)};
  const cuuint64_t sstride[1] = {static_cast<cuuint64_t>(a.N) * 2};
  const cuuint32_t sbox[2] = {kCols, static_cast<cuuint32_t>(ngmax)};
  r = enc(&tms, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.S), sdim, sstride, sbox,
          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  StParams p;
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.G = static_cast<int>(G);
  p.cs = cs;
  p.ngmax = ngmax;
  p.lead = lead;
  p.act = a.act;
  p.prefetch_x = 1;
  p.Wp = reinterpret_cast<const uint8_t*>(a.Wp);
  p.X = static_cast<const uint8_t*>(a.X);
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(
      a.bits == 4 ? (tok == 16 ? StCfg<4, 16>::kSmem : tok == 32 ? StCfg<4, 32>::kSmem : StCfg<4, 64>::kSmem)
                  : (tok == 16 ? StCfg<8, 16>::kSmem : tok == 32 ? StCfg<8, 32>::kSmem : StCfg<8, 64>::kSmem));
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
  if (a.bits == 4) {
    if (tok == 16) return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<4, 16>, tmx, tmw, tms, p);
    if (tok == 32) return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<4, 32>, tmx, tmw, tms, p);
    return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<4, 64>, tmx, tmw, tms, p);
  }
  if (tok == 16) return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<8, 16>, tmx, tmw, tms, p);
  if (tok == 32) return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<8, 32>, tmx, tmw, tms, p);
  return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<8, 64>, tmx, tmw, tms, p);
}

}  // namespace wq
