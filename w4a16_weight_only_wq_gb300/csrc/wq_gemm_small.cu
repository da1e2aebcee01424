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
//    range; the partial sums meet in distributed shared memory and are
//    added in rank order (deterministic, no global workspace).  The split is
//    chosen so that every CTA of the grid is resident at once (one per SM).
//  * A producer warp fills a ring of shared-memory slots, one group per
//    slot: the tile's packed cell (4 KiB INT4 / 8 KiB INT8, contiguous) by
//    one bulk copy (TMA, no tensor map), and the group's 16 rows of X and 64
//    scales by 16-byte LDGSTS (cp.async).  The slot's "full" mbarrier
//    completes when the bulk bytes have landed and every producer lane's
//    cp.async have landed; an "empty" mbarrier hands the slot back.
//  * Sixteen consumer warps each take half a group (32 columns) at a time.
//    Dequant happens in registers: one LOP3 turns two 4-bit fields into the
//    bf16 values 128 + u (INT8: 128 + lo and 2048 + 16 hi), one exact
//    bf16x2 subtract removes the bias, and the codes feed mma.sync m16n8k16
//    (bf16 in, fp32 accumulate) as the B operand; A is X read from the slot.
//    The group's partial is scaled by s[group, n] in fp32 and accumulated.
//  * X rows sit 320 bytes apart in a slot so that the 16-byte fragment loads
//    of a warp hit distinct banks.
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
constexpr int kXRowStride = 320;  // bytes
constexpr int kXBytes = 16 * kXRowStride;
constexpr int kPartBytes = 16 * 64 * 4;
constexpr int kRedStride = 33;  // floats per row of a half-tile partial
constexpr int kRedBytes = kConsumerWarps * 16 * kRedStride * 4;

template <int BITS>
struct Cell {
  static constexpr int kWords = BITS == 4 ? 1024 : 2048;
  static constexpr int kBytes = kWords * 4;
  static constexpr int kScaleOff = kBytes;
  static constexpr int kXOff = kBytes + 128;
  static constexpr int kSlot = kXOff + kXBytes;
};

struct SmallParams {
  const __nv_bfloat16* X;
  const uint32_t* Wp;
  const uint16_t* S;
  __nv_bfloat16* Y;
  int M, N, K, G, cs, slots;
  KernelDiag diag;
};

__host__ __device__ constexpr int slot_region(int slots, int slot_bytes) {
  return slots * slot_bytes > kRedBytes ? slots * slot_bytes : kRedBytes;
}
__host__ __device__ constexpr int smem_bytes_for(int slots, int slot_bytes) {
  return slot_region(slots, slot_bytes) + kPartBytes + (2 * slots + 1) * 8 + 16;
}

// Half a group (slabs 4h .. 4h+3, 32 columns) of one 64-column tile:
// tmp = X_group . codes, then acc += s[group, n] * tmp per output column.
template <int BITS>
__device__ __forceinline__ void process_half(float (&acc)[4][4], uint32_t slot_addr,
                                             int half, int lane) {
  using C = Cell<BITS>;
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kLo = 0x43004300u;    // bf16 128.0 in both halves
  constexpr uint32_t kHi = 0x45004500u;    // bf16 2048.0 in both halves
  constexpr uint32_t kB4 = 0x43084308u;    // 136 = 128 + 8
  constexpr uint32_t kB8Lo = 0x43004300u;  // 128
  constexpr uint32_t kB8Hi = 0x45084508u;  // 2176 = 2048 + 128
  const int g = lane >> 2, t4 = lane & 3;
  const uint32_t xa_addr = slot_addr + C::kXOff + g * kXRowStride + 16 * t4;
  const uint32_t xb_addr = xa_addr + 8 * kXRowStride;
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
    const uint32_t s2 = ld_shared_u32(slot_addr + C::kScaleOff + (tt * 8 + 2 * t4) * 2);
    const float s0 = bf16_lo_to_f32(s2), s1 = bf16_hi_to_f32(s2);
    acc[t][0] = fmaf(s0, tmp[t][0], acc[t][0]);
    acc[t][1] = fmaf(s1, tmp[t][1], acc[t][1]);
    acc[t][2] = fmaf(s0, tmp[t][2], acc[t][2]);
    acc[t][3] = fmaf(s1, tmp[t][3], acc[t][3]);
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
gemm_small_kernel(const SmallParams p) {
  using C = Cell<BITS>;
  extern __shared__ __align__(16) uint8_t smem[];

  const int cs = p.cs, D = p.slots;
  const int tile = blockIdx.x / cs;
  const int rank = blockIdx.x % cs;  // == %cluster_ctarank for cluster (cs,1,1)
  const int g0 = (p.G * rank) / cs;
  const int ng = (p.G * (rank + 1)) / cs - g0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Each consumer warp owns one half (32 columns) of the tile.
  const int half = warp & 1;

  // Same offsets in every CTA of the cluster (`part` is read remotely).
  uint8_t* slots = smem;
  float* red = reinterpret_cast<float*>(smem);  // aliases the drained slots
  const int region = slot_region(D, C::kSlot);
  float* part = reinterpret_cast<float*>(smem + region);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + region + kPartBytes);
  uint64_t* empty = full + D;
  uint64_t* never_bar = empty + D;  // test hook: nothing ever arrives here
  int& s_err = *reinterpret_cast<int*>(never_bar + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < D; ++i) {
      mbar_init(&full[i], 1 + 32);  // bulk-copy arrival + one per producer lane
      mbar_init(&empty[i], 2);      // both halves consumed
    }
    mbar_init(never_bar, 1);
    fence_mbar_init();
    s_err = 0;
  }
  __syncthreads();
  // Test hook 1: a wait that nothing completes runs out, reports, and the
  // kernel then carries on normally.
  if (p.diag.force_timeout == 1) mbar_wait_bounded(never_bar, 0, p.diag);

  float acc[4][4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[t][c] = 0.f;

  int issued = 0;  // producer: groups whose copies were issued
  if (warp == kProducerWarp) {
    // ------------------------------------------------------- producer ---
    // Weights are not written by the preceding kernel, so the first round
    // of cells is fetched before the programmatic-launch dependency
    // resolves; X (which may be) is fetched after it.
    const int first = min(ng, D);
    const int mrows = min(p.M, 16);
    auto issue_w = [&](int i, int slot) {
      mbar_arrive_expect_tx(&full[slot], C::kBytes);
      bulk_g2s(slots + slot * C::kSlot,
               p.Wp + (static_cast<size_t>(tile) * p.G + g0 + i) * C::kWords, C::kBytes,
               &full[slot]);
    };
    auto issue_xs = [&](int i, int slot) {
      const int g = g0 + i;
      const uint32_t base = smem_addr(slots + slot * C::kSlot);
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int c = lane + 32 * it, row = c >> 4, col = c & 15;
        const bool live = row < mrows;
        const __nv_bfloat16* src =
            live ? p.X + static_cast<size_t>(row) * p.K + static_cast<size_t>(g) * 128 + col * 8
                 : p.X;
        cp_async_16(base + C::kXOff + row * kXRowStride + col * 16, src, live ? 16u : 0u);
      }
      if (lane < 8)
        cp_async_16(base + C::kScaleOff + lane * 16,
                    p.S + static_cast<size_t>(g) * p.N + tile * 64 + lane * 8, 16u);
      cp_async_mbar_arrive_noinc(&full[slot]);
    };
    if (lane == 0)
      for (int i = 0; i < first; ++i) issue_w(i, i);
    pdl_launch_dependents();
    pdl_wait_primary();
    for (int i = 0; i < first; ++i) issue_xs(i, i);
    issued = first;
    for (int i = D; i < ng; ++i) {
      const int slot = i % D;
      int e_ok = 1;
      if (lane == 0) e_ok = mbar_wait_bounded(&empty[slot], ((i / D) - 1) & 1, p.diag);
      e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
      if (!e_ok) {
        s_err = 1;
        break;
      }
      if (lane == 0) issue_w(i, slot);
      issue_xs(i, slot);
      issued = i + 1;
    }
    cp_async_wait_all();
  } else {
    pdl_launch_dependents();
    pdl_wait_primary();  // consumers store Y, which the preceding kernel may use
    // ------------------------------------------------------ consumers ---
    // Warp w handles half (w & 1) of groups (w >> 1), (w >> 1) + 8, ...
    for (int i = warp >> 1; i < ng; i += kConsumerWarps / 2) {
      const int slot = i % D;
      // Test hook 2: look for the phase after the real one, which never
      // completes, so the give-up-and-drain path runs.
      const uint32_t parity = ((i / D) + (p.diag.force_timeout == 2 ? 1 : 0)) & 1;
      if (!mbar_wait_bounded(&full[slot], parity, p.diag)) {
        s_err = 1;  // stop here; the slot is not handed back
        break;
      }
      process_half<BITS>(acc, smem_addr(slots + slot * C::kSlot), half, lane);
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();  // our reads of the slot precede its refill
        mbar_arrive(&empty[slot]);
      }
    }
  }
  __syncthreads();
  if (s_err) {
    // Some wait gave up: let the latest fill of every slot land (bounded,
    // at least 1 s) before the shared memory is reused or released.  Phases
    // of a slot complete in order, so the latest one covers the earlier.
    if (warp == kProducerWarp && lane == 0) {
      KernelDiag drain = p.diag;
      if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
      for (int slot = 0; slot < D && slot < issued; ++slot) {
        const int last = slot + ((issued - 1 - slot) / D) * D;
        mbar_wait_bounded(&full[slot], (last / D) & 1, drain);
      }
    }
    __syncthreads();
  }

  // CTA reduction in a fixed order: every consumer warp stores its partial
  // half tile ([16 rows][32 cols], rows padded to 33 floats), then each
  // thread sums one element over the eight warps of that half, in order.
  const int gl = lane >> 2, t4 = lane & 3;
  if (warp < kConsumerWarps) {
    float* dst = red + warp * 16 * kRedStride;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int col = t * 8 + 2 * t4;
      dst[gl * kRedStride + col] = acc[t][0];
      dst[gl * kRedStride + col + 1] = acc[t][1];
      dst[(gl + 8) * kRedStride + col] = acc[t][2];
      dst[(gl + 8) * kRedStride + col + 1] = acc[t][3];
    }
  }
  __syncthreads();
  const int rows = min(16, p.M);
  for (int e = threadIdx.x; e < 1024; e += kThreads) {
    const int r = e >> 6, c = e & 63, h = c >> 5, cc = c & 31;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < kConsumerWarps / 2; ++k)
      v += red[(2 * k + h) * 16 * kRedStride + r * kRedStride + cc];
    if (cs == 1) {
      if (r < rows)
        p.Y[static_cast<size_t>(r) * p.N + tile * 64 + c] = __float2bfloat16_rn(v);
    } else {
      part[e] = v;
    }
  }
  if (cs == 1) return;

  // Cluster reduction: CTA `rank` finalises elements [rank*E/cs, ...) of
  // the tile's E = rows x 64 outputs, adding the cs partials in rank order.
  cluster_sync();
  const int e_end = (rows * 64 * (rank + 1)) / cs;
  for (int e = (rows * 64 * rank) / cs + threadIdx.x; e < e_end; e += kThreads) {
    float v = 0.f;
    for (int q = 0; q < cs; ++q) v += dsmem_ld_f32(dsmem_map(part + e, q));
    p.Y[static_cast<size_t>(e >> 6) * p.N + tile * 64 + (e & 63)] = __float2bfloat16_rn(v);
  }
  cluster_sync();  // keep this CTA's `part` alive until every peer has read it
}

// ------------------------------------------------------------ host side ---
template <int BITS>
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
        e = cudaFuncGetAttributes(&fa, gemm_small_kernel<BITS>);
        if (e != cudaSuccess) return e;
        const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
        e = cudaFuncSetAttribute(gemm_small_kernel<BITS>,
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
KernelInit<4> g_init4;
KernelInit<8> g_init8;

int slot_bytes(int bits) { return bits == 4 ? Cell<4>::kSlot : Cell<8>::kSlot; }

// Ring depth: every group of the CTA when it fits, else as many slots as
// the shared memory holds.
int ring_slots(int bits, int ng_max, int max_dyn) {
  const int sb = slot_bytes(bits);
  int d = (max_dyn - kPartBytes - 64) / (sb + 16);
  if (ng_max < d) d = ng_max;
  while (d > 0 && smem_bytes_for(d, sb) > max_dyn) --d;
  return d;
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

bool gemm_small_fits(int bits, int64_t K, int64_t N, int split_hint) {
  (void)bits;
  return choose_split(K, N, 152, split_hint) > 0;
}

cudaError_t launch_gemm_small(const GemmArgs& a, cudaStream_t stream) {
  if (a.M > 16) return cudaErrorNotSupported;
  const int cs = choose_split(a.K, a.N, a.num_sms, a.split_hint);
  if (cs < 0) return cudaErrorNotSupported;
  int max_dyn = 0;
  cudaError_t e = a.bits == 4 ? g_init4.ensure(a.device, &max_dyn)
                              : g_init8.ensure(a.device, &max_dyn);
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
  p.slots = ring_slots(a.bits, (p.G + cs - 1) / cs, max_dyn);
  if (p.slots < 1) return cudaErrorNotSupported;
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.N / 64) * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for(p.slots, slot_bytes(a.bits));
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
  if (a.bits == 4) return cudaLaunchKernelEx(&cfg, gemm_small_kernel<4>, p);
  return cudaLaunchKernelEx(&cfg, gemm_small_kernel<8>, p);
}

}  // namespace wq
