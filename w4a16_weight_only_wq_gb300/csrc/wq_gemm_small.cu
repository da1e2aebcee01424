// wq_gemm_small.cu -- memory-bound W4A16 / W8A16 GEMM for M <= 16.
//
// Y[M,N] = X[M,K] . (s (.) q)[K,N]: the quantized Linear of the verifier
// ("Quantize the Target, Quantize the Drafter": the INT4 target verifies a
// 16-token draft block in one forward; "Qwen3.5-4B-DFlash-W8A16": the int8
// drafter's projections).  At M = 16 the packed weights are read once and
// dominate the traffic, so the kernel is organised around streaming them.
//
//  * Work unit: a 64-column tile x a contiguous range of 128-deep groups.
//    A thread-block cluster of `cs` CTAs shares one tile and splits its K
//    range; each CTA pushes its partial sums into the owning CTA's shared
//    memory (distributed shared memory), where they are added in rank order
//    (deterministic, no global workspace).  The split is chosen so that
//    every CTA of the grid is resident at once (one per SM).
//  * Copies are few and large, because the copy engine of an SM issues one
//    copy every ~30 ns whatever its size: the tile's packed cells over the
//    CTA's K range are contiguous, so a chunk of four groups (16 KiB INT4 /
//    32 KiB INT8; two groups for a K split with long CTA ranges) is one
//    bulk copy, and X is one bulk copy per row for the whole K range.  The
//    producer warp issues weight chunk 0, waits for the preceding kernel
//    (programmatic launch), issues X, then the rest of the weight ring;
//    scales travel with their chunk (16-byte cp.async).
//  * Sixteen consumer warps each take half a group (32 columns) at a time.
//    Dequant happens in registers: one LOP3 turns two 4-bit fields into the
//    bf16 values 128 + u (INT8: 128 + lo and 2048 + 16 hi), one exact
//    bf16x2 subtract removes the bias, and the codes feed mma.sync m16n8k16
//    (bf16 in, fp32 accumulate) as the B operand; A is X read from shared
//    memory.  The group's partial is scaled by s[group, n] in fp32.
//  * X rows sit (256 x groups + 64) bytes apart, 64 modulo 128, so that the
//    16-byte fragment loads of a quarter-warp hit distinct banks.
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRedStride = 36;             // floats per row of a half-tile partial (16-byte rows)
constexpr int kRedBytes = kConsumerWarps * 16 * kRedStride * 4;
constexpr int kPartFloats = 1024 + 64;     // cs slices of ceil(256 / cs) quads of floats

// CH groups per weight chunk (one bulk copy): 4, or 2 (see launch_gemm_small).
template <int BITS, int CH>
struct Cell {
  static constexpr int kWords = BITS == 4 ? 1024 : 2048;
  static constexpr int kBytes = kWords * 4;
  // weight chunk slot: CH cells, then CH x 64 scales
  static constexpr int kSlot = CH * kBytes + CH * 128;
  static constexpr int kScaleOff = CH * kBytes;
};

struct SmallParams {
  const __nv_bfloat16* X;
  const uint32_t* Wp;
  const uint16_t* S;
  __nv_bfloat16* Y;
  int M, N, K, G, cs, wslots, xstride;
  int act;                  // apply_act on the stored result
  const uint8_t* pf;        // L2 prefetch range (the next GEMM's weights), or null
  int64_t pf_bytes;
  KernelDiag diag;
};

// Four adjacent outputs as bf16.  The activation is chosen once here rather
// than per value inside the store: as a per-value select the compiler
// evaluated SiLU for every output even when none was asked for.
__device__ __forceinline__ void store4(__nv_bfloat16* y, float4 v, int act) {
  if (act != 0) {
    v.x = apply_act(v.x, 1);
    v.y = apply_act(v.y, 1);
    v.z = apply_act(v.z, 1);
    v.w = apply_act(v.w, 1);
  }
  st_global_v2(y, pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
}

// Shared memory: [weight ring | CTA reduction][X rows][part][barriers]
__host__ __device__ constexpr int wregion_bytes(int wslots, int slot) {
  return wslots * slot > kRedBytes ? wslots * slot : kRedBytes;
}
__host__ __device__ constexpr int smem_bytes_for(int wslots, int slot, int xstride) {
  return wregion_bytes(wslots, slot) + 16 * xstride + kPartFloats * 4 + (2 * wslots + 3) * 8 + 16;
}
// X row stride for ng groups: 256 bytes per group, plus 64 so that rows g
// and g + 1 sit 64 bytes apart modulo 128 (conflict-free fragment loads).
__host__ __device__ constexpr int x_stride(int ng) { return ng * 256 + 64; }

// Half a group (slabs 4h .. 4h+3, 32 columns) of one 64-column tile:
// tmp = X_group . codes, then acc += s[group, n] * tmp per output column.
template <int BITS>
__device__ __forceinline__ void process_half(float (&acc)[4][4], uint32_t slot_addr,
                                             uint32_t s_addr, uint32_t x_addr, int xstride,
                                             int half, int lane) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kLo = 0x43004300u;    // bf16 128.0 in both halves
  constexpr uint32_t kHi = 0x45004500u;    // bf16 2048.0 in both halves
  constexpr uint32_t kB4 = 0x43084308u;    // 136 = 128 + 8
  constexpr uint32_t kB8Lo = 0x43004300u;  // 128
  constexpr uint32_t kB8Hi = 0x45084508u;  // 2176 = 2048 + 128
  const int g = lane >> 2, t4 = lane & 3;
  const uint32_t xa_addr = x_addr + g * xstride + 16 * t4;
  const uint32_t xb_addr = xa_addr + 8 * xstride;
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  float tmp[4][4];

  if constexpr (BITS == 4) {
    uint4 w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      w[t] = ld_shared_v4(slot_addr + (half * 4 + t) * 512 + lane * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 xa = ld_shared_v4(xa_addr + 64 * j);
      const uint4 xb = ld_shared_v4(xb_addr + 64 * j);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t word = j == 0 ? w[t].x : j == 1 ? w[t].y : j == 2 ? w[t].z : w[t].w;
        const uint32_t e0 = bf16x2_sub(lop3_and_or(word, kMask, kLo), kB4);
        const uint32_t e1 = bf16x2_sub(lop3_and_or(word >> 4, kMask, kLo), kB4);
        const uint32_t e2 = bf16x2_sub(lop3_and_or(word >> 8, kMask, kLo), kB4);
        const uint32_t e3 = bf16x2_sub(lop3_and_or(word >> 12, kMask, kLo), kB4);
        if (j == 0)
          mma_bf16_16816(tmp[t], xa.x, xb.x, xa.y, xb.y, e0, e1, zero);
        else
          mma_bf16_16816(tmp[t], xa.x, xb.x, xa.y, xb.y, e0, e1, tmp[t]);
        mma_bf16_16816(tmp[t], xa.z, xb.z, xa.w, xb.w, e2, e3, tmp[t]);
      }
    }
  } else {
    // INT8: 8 words per lane per slab in two 16-byte halves (k32 blocks
    // 0-1 and 2-3); each word is one k16 step in two 4-bit planes.
    uint4 w[4][2];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t base = slot_addr + (half * 4 + t) * 1024 + lane * 16;
      w[t][0] = ld_shared_v4(base);
      w[t][1] = ld_shared_v4(base + 512);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 xa = ld_shared_v4(xa_addr + 64 * j);
      const uint4 xb = ld_shared_v4(xb_addr + 64 * j);
#pragma unroll
      for (int step = 0; step < 2; ++step) {
        const uint32_t a0 = step ? xa.z : xa.x, a1 = step ? xb.z : xb.x;
        const uint32_t a2 = step ? xa.w : xa.y, a3 = step ? xb.w : xb.y;
        const int wi = 2 * j + step;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4& h = w[t][wi >> 2];
          const int q = wi & 3;
          const uint32_t word = q == 0 ? h.x : q == 1 ? h.y : q == 2 ? h.z : h.w;
          const uint32_t lo01 = bf16x2_sub(lop3_and_or(word, kMask, kLo), kB8Lo);
          const uint32_t hi01 = bf16x2_sub(lop3_and_or(word >> 4, kMask, kHi), kB8Hi);
          const uint32_t lo23 = bf16x2_sub(lop3_and_or(word >> 8, kMask, kLo), kB8Lo);
          const uint32_t hi23 = bf16x2_sub(lop3_and_or(word >> 12, kMask, kHi), kB8Hi);
          if (wi == 0)
            mma_bf16_16816(tmp[t], a0, a1, a2, a3, lo01, lo23, zero);
          else
            mma_bf16_16816(tmp[t], a0, a1, a2, a3, lo01, lo23, tmp[t]);
          mma_bf16_16816(tmp[t], a0, a1, a2, a3, hi01, hi23, tmp[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int tt = half * 4 + t;
    const uint32_t s2 = ld_shared_u32(s_addr + (tt * 8 + 2 * t4) * 2);
    const float s0 = bf16_lo_to_f32(s2), s1 = bf16_hi_to_f32(s2);
    acc[t][0] = fmaf(s0, tmp[t][0], acc[t][0]);
    acc[t][1] = fmaf(s1, tmp[t][1], acc[t][1]);
    acc[t][2] = fmaf(s0, tmp[t][2], acc[t][2]);
    acc[t][3] = fmaf(s1, tmp[t][3], acc[t][3]);
  }
}

template <int BITS, int CH>
__global__ void __launch_bounds__(kThreads, 1)
gemm_small_kernel(const SmallParams p) {
  using C = Cell<BITS, CH>;
  constexpr int kChunk = CH;
  extern __shared__ __align__(16) uint8_t smem[];

  const int cs = p.cs, DW = p.wslots, xs = p.xstride;
  const int tile = blockIdx.x / cs;
  const int rank = blockIdx.x % cs;  // == %cluster_ctarank for cluster (cs,1,1)
  const int g0 = (p.G * rank) / cs;
  const int ng = (p.G * (rank + 1)) / cs - g0;
  const int nch = (ng + kChunk - 1) / kChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = warp & 1;
  const int rows = min(16, p.M);

  uint8_t* wring = smem;
  float* red = reinterpret_cast<float*>(smem);  // aliases the drained weight ring
  const int wregion = wregion_bytes(DW, C::kSlot);
  uint8_t* xbuf = smem + wregion;
  float* part = reinterpret_cast<float*>(xbuf + 16 * xs);
  uint64_t* wfull = reinterpret_cast<uint64_t*>(part + kPartFloats);
  uint64_t* wempty = wfull + DW;
  uint64_t* xfull = wempty + DW;
  uint64_t* never_bar = xfull + 1;
  uint64_t* part_full = never_bar + 1;  // every rank's partials of my quads landed
  int& s_err = *reinterpret_cast<int*>(part_full + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < DW; ++i) {
      mbar_init(&wfull[i], 1 + 32);       // bulk-copy arrival + one per producer lane
      mbar_init(&wempty[i], 2 * kChunk);  // both halves of every group of the chunk
    }
    mbar_init(xfull, 1);
    mbar_init(never_bar, 1);
    mbar_init(part_full, 1);
    fence_mbar_init();
    s_err = 0;
  }
  __syncthreads();
  // Every CTA of the cluster has started before any remote store (below).
  if (cs > 1) cluster_arrive_relaxed();
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  float acc[4][4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[t][c] = 0.f;

  int issued = 0;  // producer: chunks whose copies were issued
  if (warp == kProducerWarp) {
    // ------------------------------------------------------- producer ---
    // Weights and scales do not depend on the preceding kernel: the first
    // ring of chunks is requested before the programmatic-launch wait.
    auto issue_chunk = [&](int c) {
      const int slot = c % DW;
      const int gc = min(kChunk, ng - c * kChunk);  // groups in this chunk
      uint8_t* dst = wring + slot * C::kSlot;
      if (lane == 0) {
        mbar_arrive_expect_tx(&wfull[slot], gc * C::kBytes);
        bulk_g2s(dst, p.Wp + (static_cast<size_t>(tile) * p.G + g0 + c * kChunk) * C::kWords,
                 gc * C::kBytes, &wfull[slot]);
      }
      // scales: gc x 128 bytes, 16 bytes per lane (up to kChunk x 8 pieces)
      for (int piece = lane; piece < gc * 8; piece += 32) {
        const int gi = piece >> 3, part16 = piece & 7;
        cp_async_16(smem_addr(dst + C::kScaleOff + gi * 128 + part16 * 16),
                    p.S + static_cast<size_t>(g0 + c * kChunk + gi) * p.N + tile * 64 + part16 * 8,
                    16u);
      }
      cp_async_mbar_arrive_noinc(&wfull[slot]);
    };
    // Chunk 0 first, then (once the preceding kernel is done) X, so that the
    // first group can start as early as possible; then the rest of the ring.
    const int first = min(nch, DW);
    issue_chunk(0);
    pdl_launch_dependents();
    pdl_wait_primary();
    // X: the rows' whole K range of this CTA, one bulk copy per row.
    if (lane == 0) mbar_arrive_expect_tx(xfull, rows * ng * 256);
    __syncwarp();
    if (lane < rows)
      bulk_g2s(xbuf + lane * xs, p.X + static_cast<size_t>(lane) * p.K + static_cast<size_t>(g0) * 128,
               ng * 256, xfull);
    for (int c = 1; c < first; ++c) issue_chunk(c);
    issued = first;
    for (int c = first; c < nch; ++c) {
      const int slot = c % DW;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&wempty[slot], ((c / DW) - 1) & 1, p.diag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        s_err = 1;
        break;
      }
      issue_chunk(c);
      issued = c + 1;
    }
    cp_async_wait_all();
    if (p.pf != nullptr && issued == nch && lane == 0) {
      // Once this CTA's last chunk has landed (HBM is then left to the other
      // CTAs' tails), pull this CTA's share of the next GEMM's weights into L2.
      const int last = nch - 1;
      if (mbar_wait_bounded(&wfull[last % DW], (last / DW) & 1, p.diag)) {
        const int64_t share = ((p.pf_bytes / gridDim.x + 15) / 16) * 16;
        const int64_t b0 = share * blockIdx.x;
        const int64_t nb = min(share, p.pf_bytes - b0);
        if (nb > 0) prefetch_l2_bulk(p.pf + b0, static_cast<uint32_t>(nb));
      } else {
        s_err = 1;
      }
    }
  } else {
    pdl_launch_dependents();
    pdl_wait_primary();  // consumers store Y, which the preceding kernel may use
    // ------------------------------------------------------ consumers ---
    // Warp w handles half (w & 1) of groups (w >> 1), (w >> 1) + 8, ...
    bool have_x = false;
    for (int i = warp >> 1; i < ng; i += kConsumerWarps / 2) {
      const int c = i / kChunk, slot = c % DW, gi = i % kChunk;
      // Test hook 2: halfway through, wait on a barrier nothing completes,
      // so that the give-up-and-drain path runs with copies in flight.
      const bool hook = p.diag.force_timeout == 2 && i == ng / 2;
      if (!mbar_wait_bounded(hook ? never_bar : &wfull[slot], hook ? 0u : (c / DW) & 1, p.diag) ||
          (!have_x && !mbar_wait_bounded(xfull, 0, p.diag))) {
        s_err = 1;  // stop here; the slot is not handed back
        break;
      }
      have_x = true;
      const uint32_t wbase = smem_addr(wring + slot * C::kSlot);
      process_half<BITS>(acc, wbase + gi * C::kBytes, wbase + C::kScaleOff + gi * 128,
                         smem_addr(xbuf) + i * 256, xs, half, lane);
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();  // our reads of the slot precede its refill
        mbar_arrive(&wempty[slot]);
      }
    }
  }
  // Roles that ran on one lane (MMA issue, copy issue) rejoin their warp
  // before the block-wide barrier, which a diverged warp must not reach.
  __syncwarp();
  __syncthreads();
  if (s_err) {
    // Some wait gave up: let every issued copy land (bounded, at least 1 s)
    // before the shared memory is reused or released.
    if (warp == kProducerWarp && lane == 0) {
      KernelDiag drain = p.diag;
      if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
      for (int slot = 0; slot < DW && slot < issued; ++slot) {
        const int last = slot + ((issued - 1 - slot) / DW) * DW;
        mbar_wait_bounded(&wfull[slot], (last / DW) & 1, drain);
      }
      mbar_wait_bounded(xfull, 0, drain);
    }
    __syncwarp();
    __syncthreads();
  }

  // CTA reduction in a fixed order: every consumer warp stores its partial
  // half tile ([16 rows][32 cols], rows padded to 36 floats), then each
  // thread sums a quad of 4 consecutive columns over the eight warps of that
  // half, in order, with 16-byte loads.
  const int gl = lane >> 2, t4 = lane & 3;
  if (warp < kConsumerWarps) {
    const uint32_t dst = smem_addr(red + warp * 16 * kRedStride);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int col = t * 8 + 2 * t4;
      st_shared_v2_f32(dst + (gl * kRedStride + col) * 4, acc[t][0], acc[t][1]);
      st_shared_v2_f32(dst + ((gl + 8) * kRedStride + col) * 4, acc[t][2], acc[t][3]);
    }
  }
  __syncthreads();
  // Quad e = row * 16 + col / 4 of the tile.  With a cluster, rank r owns
  // quads [r E / cs, (r + 1) E / cs) and receives every rank's partial of
  // them in its `part` (slice q at q * slice quads) by 16-byte asynchronous
  // remote stores that count their bytes on its `part_full` barrier, so the
  // owner waits for exactly its bytes instead of a second cluster barrier.
  const int E = rows * 16;
  const int slice = (E + cs - 1) / cs;
  const int e0 = (rank * E) / cs, e1 = ((rank + 1) * E) / cs;
  if (cs > 1) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(part_full, cs * (e1 - e0) * 16);
    cluster_wait();  // every CTA of the cluster has initialised its barriers
  }
  for (int e = threadIdx.x; e < E; e += kThreads) {
    const int r = e >> 4, c = (e & 15) * 4, h = c >> 5, cc = c & 31;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kConsumerWarps / 2; ++k) {
      const float4 w =
          ld_shared_v4_f32(smem_addr(red + (2 * k + h) * 16 * kRedStride + r * kRedStride + cc));
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    if (cs == 1) {
      store4(p.Y + static_cast<size_t>(r) * p.N + tile * 64 + c, v, p.act);
    } else {
      int owner = (e * cs) / E;  // first rank whose range holds e
      while (owner + 1 < cs && e >= ((owner + 1) * E) / cs) ++owner;
      while (e < (owner * E) / cs) --owner;
      const int off = e - (owner * E) / cs;
      dsmem_st_async_v4_f32(dsmem_map(part + (rank * slice + off) * 4, owner),
                            dsmem_map(part_full, owner), v.x, v.y, v.z, v.w);
    }
  }
  if (cs == 1 || e0 + static_cast<int>(threadIdx.x) >= e1) return;
  if (!mbar_wait_bounded(part_full, 0, p.diag)) {
    // A peer can be late by its own timed-out wait plus its drain (at least
    // 1 s) before it sends; this CTA's shared memory must outlive those
    // remote stores, so keep waiting (bounded) for them before exiting.
    KernelDiag late = p.diag;
    late.wait_limit_ns = p.diag.wait_limit_ns + 2000000000ull;
    mbar_wait_bounded(part_full, 0, late);
    return;
  }
  for (int e = e0 + threadIdx.x; e < e1; e += kThreads) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < cs; ++q) {
      const float4 w = ld_shared_v4_f32(smem_addr(part + (q * slice + (e - e0)) * 4));
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    store4(p.Y + static_cast<size_t>(e >> 4) * p.N + tile * 64 + (e & 15) * 4, v, p.act);
  }
}

// ------------------------------------------------------------ host side ---
template <int BITS, int CH>
struct KernelInit {
  std::atomic<uint64_t> done{0};  // one bit per device
  std::mutex mu;
  int max_dyn[64] = {};           // dynamic shared bytes a CTA may use
  cudaError_t ensure(int device, int* max_dyn_out) {
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> lk(mu);
      if (!(done.load() & bit)) {
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(
            &optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, gemm_small_kernel<BITS, CH>);
        if (e != cudaSuccess) return e;
        const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
        e = cudaFuncSetAttribute(gemm_small_kernel<BITS, CH>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (e != cudaSuccess) return e;
        max_dyn[device & 63] = dyn;
        done.fetch_or(bit, std::memory_order_release);
      }
    }
    *max_dyn_out = max_dyn[device & 63];
    return cudaSuccess;
  }
};
KernelInit<4, 4> g_init44;
KernelInit<4, 2> g_init42;
KernelInit<8, 4> g_init84;
KernelInit<8, 2> g_init82;

int slot_bytes(int bits, int ch) {
  if (bits == 4) return ch == 4 ? Cell<4, 4>::kSlot : Cell<4, 2>::kSlot;
  return ch == 4 ? Cell<8, 4>::kSlot : Cell<8, 2>::kSlot;
}

// Cluster split along K: the largest cs in 1..8 (and <= groups) for which
// tiles * cs CTAs still fit one per SM, so the whole grid is resident and
// the per-SM share of cells is as even as the shape allows.
int choose_split(int64_t K, int64_t N, int num_sms, int hint) {
  const int64_t tiles = N / 64, G = K / 128;
  if (hint > 0) return (hint <= 8 && hint <= G) ? hint : -1;
  int best = 1;
  for (int cs = 1; cs <= 8 && cs <= G; ++cs)
    if (tiles * cs <= num_sms) best = cs;
  return best;
}

}  // namespace

bool gemm_small_fits(int bits, int64_t K, int64_t N, int split_hint, int num_sms) {
  const int cs = choose_split(K, N, num_sms, split_hint);
  if (cs <= 0) return false;
  // X for the CTA's K range and at least one weight chunk must fit the
  // 227 KiB a CTA may use on sm_103.
  const int64_t ng_max = (K / 128 + cs - 1) / cs;
  if (ng_max > 4096) return false;
  return smem_bytes_for(1, slot_bytes(bits, 2), x_stride(static_cast<int>(ng_max))) <= 232448;
}

cudaError_t launch_gemm_small(const GemmArgs& a, cudaStream_t stream) {
  if (a.M > 16) return cudaErrorNotSupported;
  const int cs = choose_split(a.K, a.N, a.num_sms, a.split_hint);
  if (cs < 0) return cudaErrorNotSupported;
  int max_dyn = 0;  // the same for every variant (none uses static shared memory)
  cudaError_t e = a.bits == 4 ? g_init44.ensure(a.device, &max_dyn)
                              : g_init84.ensure(a.device, &max_dyn);
  if (e != cudaSuccess) return e;

  SmallParams p;
  p.X = static_cast<const __nv_bfloat16*>(a.X);
  p.Wp = a.Wp;
  p.S = static_cast<const uint16_t*>(a.S);
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.G = static_cast<int>(a.K / 128);
  p.cs = cs;
  const int ng_max = (p.G + cs - 1) / cs;
  p.xstride = x_stride(ng_max);
  // Chunks of four groups; of two for a K split with long CTA ranges
  // streamed from HBM (measured at M = 16: 9728 x 2560, 26 groups per CTA,
  // 8.23 -> 8.09 us; short ranges such as 2560 x 2560, 7 groups, unsplit
  // tiles and weights already in L2 are slower with them).
  const int ch = cs > 1 && ng_max >= 16 && !a.weights_in_l2 ? 2 : 4;
  const int nch_max = (ng_max + ch - 1) / ch;
  const int sb = slot_bytes(a.bits, ch);
  int dw = nch_max;
  while (dw > 0 && smem_bytes_for(dw, sb, p.xstride) > max_dyn) --dw;
  if (dw < 1) return cudaErrorNotSupported;
  if (a.bits == 4)
    e = ch == 4 ? g_init44.ensure(a.device, &max_dyn) : g_init42.ensure(a.device, &max_dyn);
  else
    e = ch == 4 ? g_init84.ensure(a.device, &max_dyn) : g_init82.ensure(a.device, &max_dyn);
  if (e != cudaSuccess) return e;
  p.wslots = dw;
  p.act = a.act;
  p.pf = static_cast<const uint8_t*>(a.l2_prefetch);
  p.pf_bytes = a.l2_prefetch != nullptr ? a.l2_prefetch_bytes : 0;
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.N / 64) * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for(p.wslots, sb, p.xstride);
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
  if (a.bits == 4)
    return ch == 4 ? cudaLaunchKernelEx(&cfg, gemm_small_kernel<4, 4>, p)
                   : cudaLaunchKernelEx(&cfg, gemm_small_kernel<4, 2>, p);
  return ch == 4 ? cudaLaunchKernelEx(&cfg, gemm_small_kernel<8, 4>, p)
                 : cudaLaunchKernelEx(&cfg, gemm_small_kernel<8, 2>, p);
}

}  // namespace wq
