// wq_swa.cu -- the drafter's attention with a symmetric sliding window.
//
// A block of B <= 16 query tokens (anchor + drafted tokens) sits at the end
// of a sequence of T tokens whose keys and values are all cached; each query
// attends bidirectionally to the keys within half a window on either side of
// its position, or to all keys when the sequence fits the window ("Quantize
// the Target, Quantize the Drafter", drafter-SWA paragraph: the window is
// applied in the attention kernel only, the cache is kept whole).
//
//  * Work unit: one query head x one contiguous slice of the keys its block
//    can see.  A thread-block cluster of S CTAs covers the slices of one
//    head; each CTA keeps a running (max, sum, weighted values) per query row
//    and sends it to rank 0 of the cluster with 16-byte asynchronous remote
//    stores counted on rank 0's mbarrier; rank 0 merges the S partial
//    softmaxes in rank order and writes the output (deterministic).
//  * Keys in chunks of 128 rows (16 per warp, eight warps), K and V staged
//    by 16-byte cp.async into rows padded to 272 bytes (conflict-free
//    fragment loads), double-buffered.  Scores and the weighted sum use mma.sync m16n8k16
//    (bf16 in, fp32 accumulate); the probabilities are re-packed from the
//    score accumulators into the A operand of the second MMA, and V is read
//    transposed with ldmatrix.
//  * The pass is bound by reading each head's visible K and V once.
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kD = 128;                 // head dimension
constexpr int kRows = 16;               // query rows per CTA (the block, padded)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 128;             // keys per chunk, 16 per warp
constexpr int kNB = 2;                  // chunk buffers in flight
constexpr int kRow = kD * 2 + 16;       // 272-byte shared-memory rows
constexpr int kMaxCluster = 8;
constexpr int kPartFloats = 2 * kRows + kRows * kD;  // max[16], sum[16], values[16][128]
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kRows * kRow;          // kNB K chunk buffers
constexpr int kOffV = kOffK + kNB * kChunk * kRow;   // kNB V chunk buffers
constexpr int kOffW = kOffV + kNB * kChunk * kRow;   // per-warp max / sum [warps][2][16]
constexpr int kORow = kD + 4;                        // fp32 rows of 132: conflict-free
constexpr int kOffO = kOffW + kWarps * 2 * kRows * 4;  // the CTA's values [16][132] fp32
constexpr int kOffRecv = kOffO + kRows * kORow * 4;  // rank 0: [S][kPartFloats]
constexpr int kOffBar = kOffRecv + kMaxCluster * kPartFloats * 4;
constexpr int kSmem = kOffBar + 24;  // two barriers, then rank 0's "bytes arrived" flag
// scores are kept in base 2: q.k / sqrt(128) * log2(e), so the softmax
// weights are exp2f of differences (the same weights, a cheaper function)
constexpr float kScale2 = 0.0883883476483184405f * 1.44269504088896341f;

struct SwaParams {
  const __nv_bfloat16* Q;  // [B][Hq][128]
  const __nv_bfloat16* K;  // [Hkv][T][128]
  const __nv_bfloat16* V;  // [Hkv][T][128]
  __nv_bfloat16* O;        // [B][Hq][128]
  int B, Hq, group, S;
  int64_t T, window;
  KernelDiag diag;
};

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__global__ void __launch_bounds__(kThreads, 1) swa_attention_kernel(const SwaParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int S = p.S;
  const int h = blockIdx.x / S, rank = blockIdx.x % S;  // rank == %cluster_ctarank
  const int kv = h / p.group;
  const int64_t T = p.T;
  const int64_t p0 = T - p.B;  // position of query 0
  const bool full = p.window == 0 || T <= p.window;
  const int64_t half = p.window / 2;
  const int ihalf = static_cast<int>(half < (int64_t(1) << 30) ? half : (int64_t(1) << 30));
  const int64_t klo = full ? 0 : (p0 - half > 0 ? p0 - half : 0);
  const int64_t nk = T - klo;
  const int64_t c0 = klo + nk * rank / S, c1 = klo + nk * (rank + 1) / S;
  const int nchunks = static_cast<int>((c1 - c0 + kChunk - 1) / kChunk);
  uint64_t* recv_bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* never_bar = recv_bar + 1;  // test hook: a barrier nothing completes
  const uint32_t sbase = smem_addr(smem);

  if (threadIdx.x == 0) {
    mbar_init(recv_bar, 1);
    mbar_init(never_bar, 1);
    fence_mbar_init();
    if (rank == 0) mbar_arrive_expect_tx(recv_bar, S * kPartFloats * 4);
  }
  __syncthreads();
  cluster_arrive_relaxed();  // every CTA's barrier is initialised before any remote store

  // ---- staging: Q once, then K / V chunks (rows past the slice read as 0)
  for (int i = threadIdx.x; i < kRows * 16; i += kThreads) {
    const int r = i >> 4, piece = i & 15;
    const bool live = r < p.B;
    const __nv_bfloat16* src = live ? p.Q + (static_cast<int64_t>(r) * p.Hq + h) * kD + piece * 8 : p.Q;
    cp_async_16(sbase + kOffQ + r * kRow + piece * 16, src, live ? 16u : 0u);
  }
  auto load_chunk = [&](int c) {
    const int buf = c % kNB;
    const int64_t j0 = c0 + static_cast<int64_t>(c) * kChunk;
    for (int i = threadIdx.x; i < kChunk * 16; i += kThreads) {
      const int r = i >> 4, piece = i & 15;
      const int64_t j = j0 + r;
      const bool live = j < c1;
      const int64_t off = live ? (static_cast<int64_t>(kv) * T + j) * kD + piece * 8 : 0;
      cp_async_16(sbase + kOffK + (buf * kChunk + r) * kRow + piece * 16, p.K + off, live ? 16u : 0u);
      cp_async_16(sbase + kOffV + (buf * kChunk + r) * kRow + piece * 16, p.V + off, live ? 16u : 0u);
    }
  };
  // chunk c is cp.async group c (Q travels with chunk 0); up to kNB ahead
  const int first = nchunks < kNB ? nchunks : kNB;
  for (int c = 0; c < first; ++c) {
    load_chunk(c);
    cp_async_commit();
  }
  if (first == 0) cp_async_commit();

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int db = 0; db < 16; ++db)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[db][e] = 0.f;
  uint32_t qa[8][4];

  for (int c = 0; c < nchunks; ++c) {
    // groups committed after chunk c's: min(kNB - 1, nchunks - 1 - c)
    const int later = nchunks - 1 - c < kNB - 1 ? nchunks - 1 - c : kNB - 1;
    if (later >= 3) cp_async_wait_group<3>();
    else if (later == 2) cp_async_wait_group<2>();
    else if (later == 1) cp_async_wait_group<1>();
    else cp_async_wait_group<0>();
    __syncthreads();
    if (c == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t a = sbase + kOffQ + g * kRow + (16 * ks + 2 * t4) * 2;
        qa[ks][0] = ld_shared_u32(a);
        qa[ks][1] = ld_shared_u32(a + 8 * kRow);
        qa[ks][2] = ld_shared_u32(a + 16);
        qa[ks][3] = ld_shared_u32(a + 8 * kRow + 16);
      }
    }
    const int buf = c % kNB;
    const int rb = buf * kChunk + 16 * warp;  // this warp's first row in the buffers
    const int64_t kb = c0 + static_cast<int64_t>(c) * kChunk + 16 * warp;  // its first key
    // scores s[nb]: rows g / g + 8, keys kb + 8 nb + 2 t4 + {0, 1}
    float s[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
      const uint32_t kaddr = sbase + kOffK + (rb + 8 * nb + g) * kRow + 4 * t4;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t b0 = ld_shared_u32(kaddr + 32 * ks);
        const uint32_t b1 = ld_shared_u32(kaddr + 32 * ks + 16);
        mma_bf16_16816(s[nb], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1, s[nb]);
      }
    }
    // mask (slice end, window) and scale; running max / sum per row.  A step
    // whose 16 keys lie in every query's window and before the slice end
    // needs no mask.
    float mx[2] = {-INFINITY, -INFINITY};
    const bool interior =
        kb + 16 <= c1 && (full || (kb >= p0 + p.B - 1 - half && kb + 15 <= p0 + half));
    if (interior) {
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s[nb][e] *= kScale2;
          mx[e >> 1] = fmaxf(mx[e >> 1], s[nb][e]);
        }
    } else {
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = g + 8 * (e >> 1);
          const int jr = static_cast<int>(kb - p0) + 8 * nb + 2 * t4 + (e & 1) - r;  // j - p_r
          const bool vis = jr + r < static_cast<int>(c1 - p0) &&
                           (full || r >= p.B || (jr >= -ihalf && jr <= ihalf));
          s[nb][e] = vis ? s[nb][e] * kScale2 : -INFINITY;
          mx[e >> 1] = fmaxf(mx[e >> 1], s[nb][e]);
        }
      }
    }
    float alpha[2], psum[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float mnew = fmaxf(m_run[i], mx[i]);
      alpha[i] = mnew == -INFINITY ? 1.f : exp2f(m_run[i] - mnew);
      m_run[i] = mnew;
    }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = e >> 1;
        s[nb][e] = m_run[i] == -INFINITY ? 0.f : exp2f(s[nb][e] - m_run[i]);
        psum[i] += s[nb][e];
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      psum[i] += __shfl_xor_sync(0xffffffffu, psum[i], 1);
      psum[i] += __shfl_xor_sync(0xffffffffu, psum[i], 2);
      l_run[i] = l_run[i] * alpha[i] + psum[i];
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {  // a row's max moved
#pragma unroll
      for (int db = 0; db < 16; ++db) {
        o[db][0] *= alpha[0];
        o[db][1] *= alpha[0];
        o[db][2] *= alpha[1];
        o[db][3] *= alpha[1];
      }
    }
    // probabilities as the A operand (16 rows x 16 keys)
    const uint32_t pa0 = pack_bf16x2_rn(s[0][0], s[0][1]);
    const uint32_t pa1 = pack_bf16x2_rn(s[0][2], s[0][3]);
    const uint32_t pa2 = pack_bf16x2_rn(s[1][0], s[1][1]);
    const uint32_t pa3 = pack_bf16x2_rn(s[1][2], s[1][3]);
    // values: V rows rb .. rb + 15 read transposed, 16 dims per ldmatrix
    const int mi = lane >> 3;
    const uint32_t vaddr =
        sbase + kOffV + (rb + 8 * (mi & 1) + (lane & 7)) * kRow + 8 * (mi >> 1) * 2;
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(vaddr + 32 * dp, r0, r1, r2, r3);
      mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, r0, r1, o[2 * dp]);
      mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, r2, r3, o[2 * dp + 1]);
    }
    __syncthreads();  // every warp is done with the buffer: refill it
    if (c + kNB < nchunks) {
      load_chunk(c + kNB);
      cp_async_commit();
    }
  }
  cp_async_wait_group<0>();  // a CTA with no chunk still waits for its Q copies

  // ---- the CTA's partial: merge the warps in order
  float* wml = reinterpret_cast<float*>(smem + kOffW);  // [warp][0: max, 1: sum][row]
  float* co = reinterpret_cast<float*>(smem + kOffO);   // [row][132]
  float* wo = reinterpret_cast<float*>(smem + kOffK);   // [warp][row][132], K/V are done
  if (t4 == 0) {
    wml[(warp * 2 + 0) * kRows + g] = m_run[0];
    wml[(warp * 2 + 0) * kRows + g + 8] = m_run[1];
    wml[(warp * 2 + 1) * kRows + g] = l_run[0];
    wml[(warp * 2 + 1) * kRows + g + 8] = l_run[1];
  }
  __syncthreads();
  float f[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = g + 8 * i;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wml[(w * 2) * kRows + r]);
    f[i] = (M == -INFINITY || m_run[i] == -INFINITY) ? 0.f : exp2f(m_run[i] - M);
  }
  float* mine = wo + warp * kRows * kORow;
#pragma unroll
  for (int db = 0; db < 16; ++db) {
    const int col = 8 * db + 2 * t4;
    mine[g * kORow + col] = o[db][0] * f[0];
    mine[g * kORow + col + 1] = o[db][1] * f[0];
    mine[(g + 8) * kORow + col] = o[db][2] * f[1];
    mine[(g + 8) * kORow + col + 1] = o[db][3] * f[1];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRows * kD; i += kThreads) {
    const int r = i / kD, col = i % kD;
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v += wo[(w * kRows + r) * kORow + col];
    co[r * kORow + col] = v;
  }
  // max and sum of the CTA's rows go in front of the values: part = wml[0 .. 31]
  float rowmax = -INFINITY, rowsum = 0.f;
  if (threadIdx.x < kRows) {
    const int r = threadIdx.x;
    for (int w = 0; w < kWarps; ++w) rowmax = fmaxf(rowmax, wml[(w * 2) * kRows + r]);
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wml[(w * 2) * kRows + r];
      if (mw != -INFINITY) rowsum += wml[(w * 2 + 1) * kRows + r] * exp2f(mw - rowmax);
    }
  }
  __syncthreads();  // everyone has read wml and written co
  float* part = wml;
  if (threadIdx.x < kRows) {
    part[threadIdx.x] = rowmax;
    part[kRows + threadIdx.x] = rowsum;
  }
  __syncthreads();
  cluster_wait();
  const uint32_t recv = dsmem_map(smem + kOffRecv, 0) + rank * kPartFloats * 4;
  const uint32_t rbar = dsmem_map(recv_bar, 0);
  for (int q = threadIdx.x; q < kPartFloats / 4; q += kThreads) {
    const float* src = q < 8 ? part + 4 * q : co + ((q - 8) / 32) * kORow + 4 * ((q - 8) % 32);
    dsmem_st_async_v4_f32(recv + 16 * q, rbar, src[0], src[1], src[2], src[3]);
  }
  if (rank != 0) return;

  // ---- rank 0: merge the S partials in rank order and write O
  int* okflag = reinterpret_cast<int*>(smem + kOffBar + 16);
  if (threadIdx.x == 0) {
    // Test hook 2: wait on a barrier nothing completes; the wait gives up,
    // reports the timeout, and the partials are still drained below before
    // the CTA (whose shared memory they land in) exits, without an output.
    const bool hooked = p.diag.force_timeout == 2 && !mbar_wait_bounded(never_bar, 0, p.diag);
    KernelDiag drain = p.diag;
    if (hooked && drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
    *okflag = mbar_wait_bounded(recv_bar, 0, drain) && !hooked ? 1 : 0;
  }
  __syncthreads();
  if (*okflag == 0) return;
  const float* rp = reinterpret_cast<const float*>(smem + kOffRecv);
  float* wts = reinterpret_cast<float*>(smem + kOffW + 2 * kRows * 4);  // [S][16] after part
  if (threadIdx.x < kRows) {
    const int r = threadIdx.x;
    float M = -INFINITY;
    for (int q = 0; q < S; ++q) M = fmaxf(M, rp[q * kPartFloats + r]);
    float L = 0.f;
    for (int q = 0; q < S; ++q) {
      const float mq = rp[q * kPartFloats + r];
      const float w = mq == -INFINITY ? 0.f : exp2f(mq - M);
      wts[q * kRows + r] = w;
      L += rp[q * kPartFloats + kRows + r] * w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int q = 0; q < S; ++q) wts[q * kRows + r] *= inv;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.B * (kD / 2); i += kThreads) {
    const int r = i / (kD / 2), d = 2 * (i % (kD / 2));
    float v0 = 0.f, v1 = 0.f;
    for (int q = 0; q < S; ++q) {
      const float w = wts[q * kRows + r];
      v0 += rp[q * kPartFloats + 2 * kRows + r * kD + d] * w;
      v1 += rp[q * kPartFloats + 2 * kRows + r * kD + d + 1] * w;
    }
    *reinterpret_cast<uint32_t*>(p.O + (static_cast<int64_t>(r) * p.Hq + h) * kD + d) =
        pack_bf16x2_rn(v0, v1);
  }
}

struct SwaInit {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
  int max_clusters[64][kMaxCluster + 1] = {};
  cudaError_t ensure(int device, int (&out)[kMaxCluster + 1]) {
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> lk(mu);
      if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(swa_attention_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        for (int c = 1; c <= kMaxCluster; ++c) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(c);
          cfg.blockDim = dim3(kThreads);
          cfg.dynamicSmemBytes = kSmem;
          cudaLaunchAttribute at;
          at.id = cudaLaunchAttributeClusterDimension;
          at.val.clusterDim.x = c;
          at.val.clusterDim.y = 1;
          at.val.clusterDim.z = 1;
          cfg.attrs = &at;
          cfg.numAttrs = 1;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, swa_attention_kernel, &cfg) != cudaSuccess) n = 0;
          max_clusters[device & 63][c] = n;
        }
        cudaGetLastError();  // a refused size above is not an error of this call
        done.fetch_or(bit, std::memory_order_release);
      }
    }
    for (int c = 0; c <= kMaxCluster; ++c) out[c] = max_clusters[device & 63][c];
    return cudaSuccess;
  }
};
SwaInit g_swa;

}  // namespace

cudaError_t launch_swa_attention(const SwaArgs& a, cudaStream_t stream) {
  int max_cl[kMaxCluster + 1];
  cudaError_t e = g_swa.ensure(a.device, max_cl);
  if (e != cudaSuccess) return e;
  const int64_t p0 = a.T - a.B;
  const bool full = a.window == 0 || a.T <= a.window;
  const int64_t klo = full ? 0 : (p0 - a.window / 2 > 0 ? p0 - a.window / 2 : 0);
  const int64_t nk = a.T - klo;
  // slices per head: fill the SMs, at least one chunk each, clusters resident
  int S = 1;
  for (int c = 2; c <= kMaxCluster; ++c)
    if (a.Hq * c <= a.num_sms && (nk + c - 1) / c >= kChunk && max_cl[c] > 0) S = c;
  if (a.split_hint > 0 && a.split_hint <= kMaxCluster && max_cl[a.split_hint] > 0) S = a.split_hint;
  SwaParams p;
  p.Q = static_cast<const __nv_bfloat16*>(a.Q);
  p.K = static_cast<const __nv_bfloat16*>(a.K);
  p.V = static_cast<const __nv_bfloat16*>(a.V);
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.B = a.B;
  p.Hq = a.Hq;
  p.group = a.Hq / a.Hkv;
  p.S = S;
  p.T = a.T;
  p.window = a.window;
  p.diag.err = a.diag.err;
  p.diag.wait_limit_ns = a.diag.wait_limit_ns;
  p.diag.force_timeout = a.diag.force_timeout;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.Hq * S));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = S;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, swa_attention_kernel, p);
}

}  // namespace wq
