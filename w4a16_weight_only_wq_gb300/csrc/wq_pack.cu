// wq_pack.cu -- the pack step and its inverse, on the GPU.
//
// Pack ("Quantize the Target, Quantize the Drafter", packing paragraph: the
// updated weights are rounded back onto the same grid under the original
// scales; "Qwen3.5-4B-DFlash-W8A16" card: RTN, symmetric, group 128):
//   s = given scale, or bf16_rne(absmax / qpos) (qpos 7 / 127; 1 if absmax 0)
//   q = clamp(rint(w / s), qmin, qmax)      (IEEE fp32 divide, ties to even)
// followed by the tile-interleaved word layout documented in include/wq.h.
//
// One CTA handles one (64-column tile, 128-deep group) cell: it stages the
// 128 x 64 weight block in shared memory with coalesced row loads, and
// writes the cell's 4 KiB (INT4) / 8 KiB (INT8) of words contiguously.
#include <cuda_bf16.h>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kPackThreads = 256;

__device__ __forceinline__ float widen_bf16(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

template <int BITS>
struct Fmt {
  static constexpr int kWords = BITS == 4 ? 1024 : 2048;  // words per cell
  static constexpr int kQmin = BITS == 4 ? -8 : -128;
  static constexpr int kQmax = BITS == 4 ? 7 : 127;
  static constexpr int kOff = BITS == 4 ? 8 : 128;
  static constexpr float kQpos = BITS == 4 ? 7.0f : 127.0f;
  static constexpr int kPerWord = BITS == 4 ? 8 : 4;
};

// Position of code `p` (0 .. kPerWord-1) of word `i` of a cell: the local
// row (k within the group), column (n within the tile) and bit shift.
template <int BITS>
__device__ __forceinline__ void cell_slot(int i, int p, int& kl, int& nl,
                                          int& shift) {
  int j8, lane, kb, r;
  if (BITS == 4) {
    j8 = i >> 7;
    lane = (i >> 2) & 31;
    kb = i & 3;
    r = p;  // the word holds 8 consecutive k
    shift = 4 * ((r >> 1) + 4 * (r & 1));
  } else {
    j8 = i >> 8;
    const int half = (i >> 7) & 1;
    lane = (i >> 2) & 31;
    const int w = 4 * half + (i & 3);  // 0..7
    kb = w >> 1;
    r = 4 * (w & 1) + p;  // the word holds 4 consecutive k
    const int rr = p;
    shift = 8 * ((rr >> 1) + 2 * (rr & 1));
  }
  const int c = lane >> 2, t4 = lane & 3;
  kl = 32 * kb + 8 * t4 + r;
  nl = 8 * j8 + c;
}

template <int BITS, typename TIn>
__global__ void __launch_bounds__(kPackThreads)
pack_symmetric_kernel(const TIn* __restrict__ W, int64_t K, int64_t N,
                      const uint16_t* scales_in, uint16_t* scales_out,
                      uint32_t* __restrict__ packed) {
  using F = Fmt<BITS>;
  __shared__ float tile[128][65];
  __shared__ float sc[64];
  __shared__ float red[4][64];
  const int64_t nt = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  for (int e = tid; e < 128 * 64; e += kPackThreads) {
    const int r = e >> 6, c = e & 63;
    const int64_t idx = (g * 128 + r) * N + nt * 64 + c;
    float v;
    if constexpr (sizeof(TIn) == 4)
      v = W[idx];
    else
      v = widen_bf16(W[idx]);
    tile[r][c] = v;
  }
  __syncthreads();
  const int64_t srow = g * N + nt * 64;
  if (scales_in == nullptr) {
    // absmax over the 128 rows: 4 threads per column, 32 rows each.
    const int c = tid & 63, part = tid >> 6;
    float m = 0.0f;
    for (int r = part * 32; r < part * 32 + 32; ++r) m = fmaxf(m, fabsf(tile[r][c]));
    red[part][c] = m;
    __syncthreads();
    if (tid < 64) {
      const float amax = fmaxf(fmaxf(red[0][tid], red[1][tid]),
                               fmaxf(red[2][tid], red[3][tid]));
      const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, F::kQpos);
      const uint16_t sb = __bfloat16_as_ushort(__float2bfloat16_rn(s));
      scales_out[srow + tid] = sb;
      sc[tid] = widen_bf16(sb);
    }
  } else if (tid < 64) {
    const uint16_t sb = scales_in[srow + tid];
    scales_out[srow + tid] = sb;
    sc[tid] = widen_bf16(sb);
  }
  __syncthreads();
  uint32_t* out = packed + (nt * (K / 128) + g) * F::kWords;
  for (int i = tid; i < F::kWords; i += kPackThreads) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < F::kPerWord; ++p) {
      int kl, nl, sh;
      cell_slot<BITS>(i, p, kl, nl, sh);
      int q = __float2int_rn(__fdiv_rn(tile[kl][nl], sc[nl]));
      q = min(max(q, F::kQmin), F::kQmax);
      word |= static_cast<uint32_t>(q + F::kOff) << sh;
    }
    out[i] = word;
  }
}

template <int BITS>
__global__ void __launch_bounds__(kPackThreads)
pack_codes_kernel(const int8_t* __restrict__ codes, int64_t K, int64_t N,
                  uint32_t* __restrict__ packed) {
  using F = Fmt<BITS>;
  __shared__ int8_t tile[128][64 + 4];
  const int64_t nt = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  for (int e = tid; e < 128 * 64; e += kPackThreads) {
    const int r = e >> 6, c = e & 63;
    tile[r][c] = codes[(g * 128 + r) * N + nt * 64 + c];
  }
  __syncthreads();
  constexpr uint32_t kMask = BITS == 4 ? 0xFu : 0xFFu;
  uint32_t* out = packed + (nt * (K / 128) + g) * F::kWords;
  for (int i = tid; i < F::kWords; i += kPackThreads) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < F::kPerWord; ++p) {
      int kl, nl, sh;
      cell_slot<BITS>(i, p, kl, nl, sh);
      word |= (static_cast<uint32_t>(tile[kl][nl] + F::kOff) & kMask) << sh;
    }
    out[i] = word;
  }
}

// Import of a layer stored output-channel-major with its codes packed along
// the input dimension: qweight[n][j] holds the 32 / BITS consecutive codes
// k = (32 / BITS) j + p at bits BITS p, offset-binary (q + 8 / q + 128);
// scales_nk[n][g] is the bf16 scale of group g of column n.  One CTA per
// (64-column tile, group) cell: decode the tile's 64 rows x 128 k into the
// shared tile, pack it as pack_codes_kernel does, and write the tile's 64
// scales of the group into the [K/128, N] scale matrix.
template <int BITS>
__global__ void __launch_bounds__(kPackThreads)
import_nk_kernel(const uint32_t* __restrict__ qweight, const uint16_t* __restrict__ scales_nk,
                 int64_t K, int64_t N, uint32_t* __restrict__ packed,
                 uint16_t* __restrict__ scales_out) {
  using F = Fmt<BITS>;
  constexpr int kPer = 32 / BITS;            // codes per external word
  constexpr int kRowWords = 128 / kPer;      // external words of one row per group
  constexpr uint32_t kMask = BITS == 4 ? 0xFu : 0xFFu;
  __shared__ int8_t tile[128][64 + 4];
  const int64_t nt = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t row_words = K / kPer;
  for (int e = tid; e < 64 * kRowWords; e += kPackThreads) {
    const int nl = e / kRowWords, w = e % kRowWords;
    const uint32_t word = qweight[(nt * 64 + nl) * row_words + g * kRowWords + w];
#pragma unroll
    for (int p = 0; p < kPer; ++p)
      tile[w * kPer + p][nl] =
          static_cast<int8_t>(static_cast<int>((word >> (BITS * p)) & kMask) - F::kOff);
  }
  if (tid < 64) scales_out[g * N + nt * 64 + tid] = scales_nk[(nt * 64 + tid) * (K / 128) + g];
  __syncthreads();
  uint32_t* out = packed + (nt * (K / 128) + g) * F::kWords;
  for (int i = tid; i < F::kWords; i += kPackThreads) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < F::kPerWord; ++p) {
      int kl, nl, sh;
      cell_slot<BITS>(i, p, kl, nl, sh);
      word |= (static_cast<uint32_t>(tile[kl][nl] + F::kOff) & kMask) << sh;
    }
    out[i] = word;
  }
}

template <int BITS>
__global__ void __launch_bounds__(kPackThreads)
unpack_kernel(const uint32_t* __restrict__ packed, int64_t K, int64_t N,
              int8_t* __restrict__ codes) {
  using F = Fmt<BITS>;
  __shared__ int8_t tile[128][64 + 4];
  const int64_t nt = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  constexpr uint32_t kMask = BITS == 4 ? 0xFu : 0xFFu;
  const uint32_t* in = packed + (nt * (K / 128) + g) * F::kWords;
  for (int i = tid; i < F::kWords; i += kPackThreads) {
    const uint32_t word = in[i];
#pragma unroll
    for (int p = 0; p < F::kPerWord; ++p) {
      int kl, nl, sh;
      cell_slot<BITS>(i, p, kl, nl, sh);
      tile[kl][nl] = static_cast<int8_t>(static_cast<int>((word >> sh) & kMask) - F::kOff);
    }
  }
  __syncthreads();
  for (int e = tid; e < 128 * 64; e += kPackThreads) {
    const int r = e >> 6, c = e & 63;
    codes[(g * 128 + r) * N + nt * 64 + c] = tile[r][c];
  }
}

// Dequantise one packed cell: W[k][n] = bf16(fp32(s[k/128][n]) * q[k][n]),
// the product exact in fp32 and rounded once (ties to even).  Codes are
// scattered into a shared tile by the packed layout, then rows of 64
// columns are written as bf16 pairs.
template <int BITS>
__global__ void __launch_bounds__(kPackThreads)
dequantize_kernel(const uint32_t* __restrict__ packed, const uint16_t* __restrict__ scales,
                  int64_t K, int64_t N, uint32_t* __restrict__ W) {
  using F = Fmt<BITS>;
  __shared__ int8_t tile[128][64 + 4];
  __shared__ float s[64];
  const int64_t nt = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  constexpr uint32_t kMask = BITS == 4 ? 0xFu : 0xFFu;
  const uint32_t* in = packed + (nt * (K / 128) + g) * F::kWords;
  if (tid < 64) s[tid] = widen_bf16(scales[g * N + nt * 64 + tid]);
  for (int i = tid; i < F::kWords; i += kPackThreads) {
    const uint32_t word = in[i];
#pragma unroll
    for (int p = 0; p < F::kPerWord; ++p) {
      int kl, nl, sh;
      cell_slot<BITS>(i, p, kl, nl, sh);
      tile[kl][nl] = static_cast<int8_t>(static_cast<int>((word >> sh) & kMask) - F::kOff);
    }
  }
  __syncthreads();
  for (int e = tid; e < 128 * 32; e += kPackThreads) {
    const int r = e >> 5, c = (e & 31) * 2;
    const float lo = s[c] * static_cast<float>(tile[r][c]);
    const float hi = s[c + 1] * static_cast<float>(tile[r][c + 1]);
    const uint32_t v = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
                       (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
    W[((g * 128 + r) * N + nt * 64 + c) / 2] = v;
  }
}

dim3 cell_grid(int64_t K, int64_t N) {
  return dim3(static_cast<unsigned>(N / 64), static_cast<unsigned>(K / 128));
}

}  // namespace

cudaError_t launch_pack_symmetric(const void* W, int wdt, int64_t K, int64_t N,
                                  int bits, const uint16_t* scales_in,
                                  uint16_t* scales_out, uint32_t* packed,
                                  cudaStream_t stream) {
  const dim3 grid = cell_grid(K, N);
  if (bits == 4 && wdt == 0)
    pack_symmetric_kernel<4, float><<<grid, kPackThreads, 0, stream>>>(
        static_cast<const float*>(W), K, N, scales_in, scales_out, packed);
  else if (bits == 4)
    pack_symmetric_kernel<4, uint16_t><<<grid, kPackThreads, 0, stream>>>(
        static_cast<const uint16_t*>(W), K, N, scales_in, scales_out, packed);
  else if (wdt == 0)
    pack_symmetric_kernel<8, float><<<grid, kPackThreads, 0, stream>>>(
        static_cast<const float*>(W), K, N, scales_in, scales_out, packed);
  else
    pack_symmetric_kernel<8, uint16_t><<<grid, kPackThreads, 0, stream>>>(
        static_cast<const uint16_t*>(W), K, N, scales_in, scales_out, packed);
  return cudaGetLastError();
}

cudaError_t launch_pack_codes(const int8_t* codes, int64_t K, int64_t N,
                              int bits, uint32_t* packed, cudaStream_t stream) {
  const dim3 grid = cell_grid(K, N);
  if (bits == 4)
    pack_codes_kernel<4><<<grid, kPackThreads, 0, stream>>>(codes, K, N, packed);
  else
    pack_codes_kernel<8><<<grid, kPackThreads, 0, stream>>>(codes, K, N, packed);
  return cudaGetLastError();
}

cudaError_t launch_import_nk(const uint32_t* qweight, const uint16_t* scales_nk, int bits,
                             int64_t K, int64_t N, uint32_t* packed, uint16_t* scales_out,
                             cudaStream_t stream) {
  const dim3 grid = cell_grid(K, N);
  if (bits == 4)
    import_nk_kernel<4><<<grid, kPackThreads, 0, stream>>>(qweight, scales_nk, K, N, packed,
                                                           scales_out);
  else
    import_nk_kernel<8><<<grid, kPackThreads, 0, stream>>>(qweight, scales_nk, K, N, packed,
                                                           scales_out);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint32_t* packed, const uint16_t* scales, int bits,
                              int64_t K, int64_t N, uint16_t* W, cudaStream_t stream) {
  const dim3 grid = cell_grid(K, N);
  uint32_t* out = reinterpret_cast<uint32_t*>(W);
  if (bits == 4)
    dequantize_kernel<4><<<grid, kPackThreads, 0, stream>>>(packed, scales, K, N, out);
  else
    dequantize_kernel<8><<<grid, kPackThreads, 0, stream>>>(packed, scales, K, N, out);
  return cudaGetLastError();
}

namespace {
// One bf16 pair per thread iteration (n is even for every caller: N % 64 == 0).
__global__ void silu_inplace_kernel(uint32_t* h2, int64_t npairs) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < npairs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t w = h2[i];
    const float lo = apply_act(__uint_as_float(w << 16), 1);
    const float hi = apply_act(__uint_as_float(w & 0xFFFF0000u), 1);
    h2[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
  }
}
}  // namespace

cudaError_t launch_silu_inplace(uint16_t* H, int64_t n, cudaStream_t stream) {
  const int64_t npairs = n / 2;
  if (npairs == 0) return cudaSuccess;
  const int64_t blocks = (npairs + 255) / 256;
  silu_inplace_kernel<<<static_cast<unsigned>(blocks < 1184 ? blocks : 1184), 256, 0, stream>>>(
      reinterpret_cast<uint32_t*>(H), npairs);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* packed, int bits, int64_t K,
                          int64_t N, int8_t* codes, cudaStream_t stream) {
  const dim3 grid = cell_grid(K, N);
  if (bits == 4)
    unpack_kernel<4><<<grid, kPackThreads, 0, stream>>>(packed, K, N, codes);
  else
    unpack_kernel<8><<<grid, kPackThreads, 0, stream>>>(packed, K, N, codes);
  return cudaGetLastError();
}

}  // namespace wq
