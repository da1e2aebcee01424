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
//    and sends each row's partial to the row's owner (rank row % S) with
//    16-byte asynchronous remote stores counted on the owner's mbarrier;
//    every owner merges the S partials of its rows in rank order and writes
//    them (deterministic).
//  * Keys in chunks of 128 rows (16 per warp, eight warps).  K and V come
//    by TMA, four copies per chunk (each 64-dimension half of K and of V)
//    with the 128-byte swizzle, so the fragment loads are conflict-free;
//    three chunks in flight; a slice's last, partial chunk in 16-row boxes.
//    Keys past the slice are masked.  The warps walk the chunks at their own
//    pace (no block-wide barrier per chunk); the last warp to release a
//    buffer issues its refill.
//  * Scores and the weighted sum use mma.sync m16n8k16 (bf16 in, fp32
//    accumulate) with an online softmax in base 2; the probabilities are
//    re-packed from the score accumulators into the A operand of the second
//    MMA, and V is read transposed with ldmatrix.
//  * With programmatic launch the kernel sets up while the preceding kernel
//    drains and reads nothing global before it completes.
//  * Its bytes are each head's visible K and V read once; at the drafter's
//    sizes the pass is bound by latency (copy landing, the per-chunk
//    dependent MMA and softmax steps, the merges), not by those bytes.
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tcgen05.cuh"
#include "wq_tensor_map.h"

namespace wq {
namespace {

constexpr int kD = 128;                 // head dimension
constexpr int kRows = 16;               // query rows per CTA (the block, padded)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 128;             // keys per chunk, 16 per warp
constexpr int kNB = 3;                  // chunk buffers in flight
constexpr int kRow = kD * 2;            // 256-byte Q rows (pieces permuted)
constexpr int kMaxCluster = 8;
// One row's partial: (max, sum, 0, 0) then the 128 weighted values.
constexpr int kRowPart = 4 + kD;
// A K or V chunk buffer: two 64-dimension halves of 128 rows x 128 bytes,
// each as TMA writes it with the 128-byte swizzle (1024-byte aligned).
constexpr int kHalfBytes = kChunk * 128;
constexpr int kChunkBytes = 2 * kHalfBytes;
constexpr int kOffK = 0;                             // kNB K chunk buffers
constexpr int kOffV = kOffK + kNB * kChunkBytes;     // kNB V chunk buffers
constexpr int kOffQ = kOffV + kNB * kChunkBytes;     // Q [16][256 bytes]
constexpr int kOffW = kOffQ + kRows * kRow;          // per-warp max / sum [warps][2][16]
constexpr int kORow = kD + 8;                        // fp32 rows of 136: conflict-free 8-byte stores
// Owner's receive buffer: [source rank][owned row][kRowPart] for up to
// ceil(16 / S) owned rows; the largest over S = 1..8 is 7 x 3 rows.
constexpr int kRecvRows = 21;
constexpr int kOffRecv = kOffW + kWarps * 2 * kRows * 4;
constexpr int kOffBar = kOffRecv + kRecvRows * kRowPart * 4;
// barriers: receive, test hook, kNB chunks landed; then the int flags
// (partials arrived, abort, chunks issued, kNB release counters)
constexpr int kNumBars = 2 + kNB;
constexpr int kNumFlags = 3 + kNB;
constexpr int kSmem = kOffBar + kNumBars * 8 + kNumFlags * 4 + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory of one CTA");
static_assert(kWarps * kRows * kORow * 4 <= kNB * kChunkBytes, "warp merge fits the K buffers");

// Byte offset of byte `b` (0..255) of row `r` in a K or V chunk buffer: the
// half b / 128, then the 128-byte row with its 16-byte pieces permuted by
// r % 8 (the TMA 128-byte swizzle).
__host__ __device__ constexpr uint32_t kv_off(int r, int b) {
  return static_cast<uint32_t>((b >> 7) * kHalfBytes + r * 128 +
                               (((((b & 127) >> 4) ^ (r & 7))) << 4) + (b & 15));
}

// Byte offset of byte `b` of row `r` in a 256-byte-row buffer whose 16-byte
// pieces are permuted by r % 8, so that the eight rows a quarter-warp reads
// at one column fall on distinct banks.
__host__ __device__ constexpr uint32_t swz(int r, int b) {
  return static_cast<uint32_t>(r * kRow + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15)));
}
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

__global__ void __launch_bounds__(kThreads, 1)
swa_attention_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmk16,
                     const __grid_constant__ CUtensorMap tmv16, const SwaParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the swizzled TMA buffers want 1024-byte alignment; every CTA of the
  // cluster gets the same offset, so remote addresses match
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
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
  uint64_t* chunk_full = never_bar + 1;  // [kNB] a chunk's K and V landed
  int* okflag = reinterpret_cast<int*>(chunk_full + kNB);  // rank's partials arrived
  volatile int* abort_flag = okflag + 1;                     // some wait gave up
  int* issued = okflag + 2;    // chunks whose copies were issued
  int* released = okflag + 3;  // [kNB] warps done with each buffer, over all its uses
  const uint32_t sbase = smem_addr(smem);

  if (threadIdx.x == 0) {
    prefetch_tensor_map(&tmk);
    prefetch_tensor_map(&tmv);
    prefetch_tensor_map(&tmk16);
    prefetch_tensor_map(&tmv16);
    mbar_init(recv_bar, 1);
    mbar_init(never_bar, 1);
    for (int i = 0; i < kNB; ++i) {
      mbar_init(&chunk_full[i], 1);
      released[i] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
    // this CTA owns rows rank, rank + S, ...: S partials of each arrive here
    const int owned = (kRows - rank + S - 1) / S;
    mbar_arrive_expect_tx(recv_bar, S * owned * kRowPart * 4);
  }
  __syncthreads();
  // every CTA's barrier is initialised before any remote store; waited for
  // here, where it overlaps the launch wait and the first chunks, rather
  // than just before the merges
  cluster_arrive_relaxed();
  cluster_wait();
  // Q, K and V may come from the preceding kernel (programmatic launch):
  // nothing global is read before it completes; the next kernel may start
  // launching now.
  pdl_wait_primary();
  pdl_launch_dependents();

  // ---- staging: K / V chunks by TMA, Q by cp.async.  A chunk covers key
  // rows kv * T + j0 .. + 127 of the [Hkv * T][128] view; rows past the
  // slice are real keys of the cache (or zeros past its end) and are masked
  // below.  The last warp to release a buffer refills it, so the warps walk
  // the chunks at their own pace, with no block-wide barrier per chunk.
  // A chunk with fewer than 128 keys left in the slice (its last) comes in
  // boxes of 16 rows, as many as cover its keys.
  auto load_chunk = [&](int c) {
    const int buf = c % kNB;
    const int64_t j0 = c0 + static_cast<int64_t>(c) * kChunk;
    const int y = static_cast<int>(static_cast<int64_t>(kv) * T + j0);
    uint8_t* kb = smem + kOffK + buf * kChunkBytes;
    uint8_t* vb = smem + kOffV + buf * kChunkBytes;
    const int64_t left = c1 - j0;
    if (left >= kChunk) {
      mbar_arrive_expect_tx(&chunk_full[buf], 2 * kChunkBytes);
      tma_load_2d(kb, &tmk, 0, y, &chunk_full[buf]);
      tma_load_2d(kb + kHalfBytes, &tmk, 64, y, &chunk_full[buf]);
      tma_load_2d(vb, &tmv, 0, y, &chunk_full[buf]);
      tma_load_2d(vb + kHalfBytes, &tmv, 64, y, &chunk_full[buf]);
    } else {
      const int nblk = static_cast<int>((left + 15) / 16);
      mbar_arrive_expect_tx(&chunk_full[buf], static_cast<uint32_t>(4 * nblk * 16 * 128));
      for (int b = 0; b < nblk; ++b) {
        const int off = b * 16 * 128;
        tma_load_2d(kb + off, &tmk16, 0, y + 16 * b, &chunk_full[buf]);
        tma_load_2d(kb + kHalfBytes + off, &tmk16, 64, y + 16 * b, &chunk_full[buf]);
        tma_load_2d(vb + off, &tmv16, 0, y + 16 * b, &chunk_full[buf]);
        tma_load_2d(vb + kHalfBytes + off, &tmv16, 64, y + 16 * b, &chunk_full[buf]);
      }
    }
  };
  const int first = nchunks < kNB ? nchunks : kNB;
  if (threadIdx.x == 0) {
    for (int c = 0; c < first; ++c) load_chunk(c);
    *issued = first;
  }
  for (int i = threadIdx.x; i < kRows * 16; i += kThreads) {
    const int r = i >> 4, piece = i & 15;
    const bool live = r < p.B;
    const __nv_bfloat16* src = live ? p.Q + (static_cast<int64_t>(r) * p.Hq + h) * kD + piece * 8 : p.Q;
    cp_async_16(sbase + kOffQ + swz(r, piece * 16), src, live ? 16u : 0u);
  }
  cp_async_commit();

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int db = 0; db < 16; ++db)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[db][e] = 0.f;
  uint32_t qa[8][4];

  cp_async_wait_group<0>();  // Q
  __syncthreads();           // every thread's Q pieces have landed
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % kNB;
    // Lane 0 waits (bounded) and tells its warp, so that the warp leaves
    // the loop as a whole if the wait gives up.
    int ok = 1;
    if (lane == 0) {
      // test hook 2: the last chunk's wait looks for a phase that never completes
      const bool hook = p.diag.force_timeout == 2 && c == nchunks - 1;
      ok = role_wait(hook ? never_bar : &chunk_full[buf], hook ? 0u : (c / kNB) & 1, p.diag,
                     abort_flag);
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    // completes at once: makes the landed bytes visible to this thread
    mbar_wait_bounded(&chunk_full[buf], (c / kNB) & 1, p.diag);
    if (c == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int b = 32 * ks + 4 * t4;
        qa[ks][0] = ld_shared_u32(sbase + kOffQ + swz(g, b));
        qa[ks][1] = ld_shared_u32(sbase + kOffQ + swz(g + 8, b));
        qa[ks][2] = ld_shared_u32(sbase + kOffQ + swz(g, b + 16));
        qa[ks][3] = ld_shared_u32(sbase + kOffQ + swz(g + 8, b + 16));
      }
    }
    const uint32_t kbase = sbase + kOffK + buf * kChunkBytes;
    const uint32_t vbase = sbase + kOffV + buf * kChunkBytes;
    const int rb = 16 * warp;  // this warp's first row in the chunk
    const int64_t kb = c0 + static_cast<int64_t>(c) * kChunk + 16 * warp;  // its first key
    // a warp whose 16 keys all lie past the slice end has nothing to add
    if (kb < c1) {
      // scores s[nb]: rows g / g + 8, keys kb + 8 nb + 2 t4 + {0, 1}
      float s[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nb][e] = 0.f;
        const int kr = rb + 8 * nb + g;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t b0 = ld_shared_u32(kbase + kv_off(kr, 32 * ks + 4 * t4));
          const uint32_t b1 = ld_shared_u32(kbase + kv_off(kr, 32 * ks + 16 + 4 * t4));
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
      // l_run is this thread's share of the row sum (its four keys of each
      // step); alpha is the same across the quad, so the shares are added
      // once, after the loop
#pragma unroll
      for (int i = 0; i < 2; ++i) l_run[i] = l_run[i] * alpha[i] + psum[i];
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
      const int vr = rb + 8 * (mi & 1) + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4_trans(vbase + kv_off(vr, 32 * dp + 16 * (mi >> 1)), r0, r1, r2, r3);
        mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, r0, r1, o[2 * dp]);
        mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, r2, r3, o[2 * dp + 1]);
      }
    }
    // This warp is done with the buffer: when a later chunk goes into it,
    // its reads are ordered before the async-proxy writes of the refill, and
    // the warp whose release completes the buffer's use (the count reaches
    // kWarps times its uses) refills it.
    if (c + kNB >= nchunks) continue;
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      const int prev = atomicAdd(&released[buf], 1);
      if (prev == (c / kNB + 1) * kWarps - 1) {
        __threadfence_block();
        fence_proxy_async_smem();
        load_chunk(c + kNB);
        atomicMax(issued, c + kNB + 1);
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // A wait gave up: let every issued copy land (bounded, at least 1 s)
    // before the buffers are reused below or the CTA exits.
    KernelDiag drain = p.diag;
    if (drain.wait_limit_ns < 1000000000ull) drain.wait_limit_ns = 1000000000ull;
    const int n = *issued;
    for (int b = 0; b < kNB && b < n; ++b) {
      const int last = b + ((n - 1 - b) / kNB) * kNB;
      mbar_wait_bounded(&chunk_full[b], (last / kNB) & 1, drain);
    }
  }
  __syncthreads();

  // ---- the CTA's partial: merge the warps in order and send every row's
  // share to its owner (rank row % S), slot (this rank, row / S) of the
  // owner's receive buffer: piece 0 is (max, sum, 0, 0), pieces 1..32 the
  // values, as 16-byte asynchronous remote stores counted on the owner's
  // barrier.
  float* wml = reinterpret_cast<float*>(smem + kOffW);  // [warp][0: max, 1: sum][row]
  float* wo = reinterpret_cast<float*>(smem + kOffK);   // [warp][row][136], K/V are done
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
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
  // the warp's row sums rescaled to the CTA's row maxima replace its sums
  // (only the maxima are read above)
  if (t4 == 0) {
    wml[(warp * 2 + 1) * kRows + g] = l_run[0] * f[0];
    wml[(warp * 2 + 1) * kRows + g + 8] = l_run[1] * f[1];
  }
  const uint32_t mine = smem_addr(wo + warp * kRows * kORow);
#pragma unroll
  for (int db = 0; db < 16; ++db) {
    const int col = 8 * db + 2 * t4;
    st_shared_v2_f32(mine + (g * kORow + col) * 4, o[db][0] * f[0], o[db][1] * f[0]);
    st_shared_v2_f32(mine + ((g + 8) * kORow + col) * 4, o[db][2] * f[1], o[db][3] * f[1]);
  }
  __syncthreads();
  const int max_owned = (kRows + S - 1) / S;
  const uint32_t recv_local = smem_addr(smem + kOffRecv);
  for (int q = threadIdx.x; q < kRows * kD / 4; q += kThreads) {
    const int r = q / (kD / 4), col = 4 * (q % (kD / 4));
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < kWarps; ++w) {
      const float4 x = ld_shared_v4_f32(smem_addr(wo + (w * kRows + r) * kORow + col));
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    const int owner = r % S;
    const uint32_t dst = recv_local + ((rank * max_owned + r / S) * kRowPart + 4 + col) * 4;
    dsmem_st_async_v4_f32(dsmem_map_addr(dst, owner), dsmem_map(recv_bar, owner), v.x, v.y, v.z,
                          v.w);
  }
  if (threadIdx.x < kRows) {
    const int r = threadIdx.x;
    float rowmax = -INFINITY, rowsum = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      rowmax = fmaxf(rowmax, wml[(w * 2) * kRows + r]);
      rowsum += wml[(w * 2 + 1) * kRows + r];  // already rescaled to the row maximum
    }
    const int owner = r % S;
    const uint32_t dst = recv_local + ((rank * max_owned + r / S) * kRowPart) * 4;
    dsmem_st_async_v4_f32(dsmem_map_addr(dst, owner), dsmem_map(recv_bar, owner), rowmax, rowsum,
                          0.f, 0.f);
  }

  // ---- every rank: merge the S partials of its rows in rank order, write O
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
  // Thread (row i, dimension pair d) weighs the S partials of its row
  // itself: w_q = exp2(m_q - M) / sum_q' l_q' exp2(m_q' - M).
  const float* rp = reinterpret_cast<const float*>(smem + kOffRecv);
  const int owned = (kRows - rank + S - 1) / S;
  for (int e = threadIdx.x; e < owned * (kD / 2); e += kThreads) {
    const int i = e / (kD / 2), d = 2 * (e % (kD / 2));
    const int r = rank + i * S;
    if (r >= p.B) continue;
    float M = -INFINITY;
    for (int q = 0; q < S; ++q) M = fmaxf(M, rp[(q * max_owned + i) * kRowPart]);
    float L = 0.f, v0 = 0.f, v1 = 0.f;
    for (int q = 0; q < S; ++q) {
      const float* src = rp + (q * max_owned + i) * kRowPart;
      const float w = src[0] == -INFINITY ? 0.f : exp2f(src[0] - M);
      L += src[1] * w;
      v0 += src[4 + d] * w;
      v1 += src[5 + d] * w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<uint32_t*>(p.O + (static_cast<int64_t>(r) * p.Hq + h) * kD + d) =
        pack_bf16x2_rn(v0 * inv, v1 * inv);
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
  // K and V as 2-D bf16 tensors [Hkv * T rows][128]; a box is 64
  // dimensions x one chunk of rows, written with the 128-byte swizzle;
  // rows past the end read as zeros.
  TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // A second pair of maps with 16-row boxes serves a slice's last chunk.
  CUtensorMap maps[4];  // K, V (128-row boxes), K, V (16-row boxes)
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(kD),
                              static_cast<cuuint64_t>(a.Hkv) * static_cast<cuuint64_t>(a.T)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t estride[2] = {1, 1};
  for (int i = 0; i < 4; ++i) {
    const cuuint32_t box[2] = {64, i < 2 ? static_cast<cuuint32_t>(kChunk) : 16u};
    const CUresult r = enc(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                           const_cast<void*>(i % 2 == 0 ? a.K : a.V), gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.Hq * S));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = S;
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
  return cudaLaunchKernelEx(&cfg, swa_attention_kernel, maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace wq
