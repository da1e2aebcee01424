// wq_internal.h -- launch functions shared between the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace wq {

struct DiagHost {
  uint32_t* err;
  uint64_t wait_limit_ns;
  int force_timeout;
};

// Pack / unpack (wq_pack.cu).  Shapes and pointers are validated by the
// caller.  wdt: 0 = fp32, 1 = bf16.
cudaError_t launch_pack_symmetric(const void* W, int wdt, int64_t K, int64_t N,
                                  int bits, const uint16_t* scales_in,
                                  uint16_t* scales_out, uint32_t* packed,
                                  cudaStream_t stream);
cudaError_t launch_pack_codes(const int8_t* codes, int64_t K, int64_t N,
                              int bits, uint32_t* packed, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* packed, int bits, int64_t K,
                          int64_t N, int8_t* codes, cudaStream_t stream);
cudaError_t launch_import_nk(const uint32_t* qweight, const uint16_t* scales_nk, int bits,
                             int64_t K, int64_t N, uint32_t* packed, uint16_t* scales_out,
                             cudaStream_t stream);
cudaError_t launch_dequantize(const uint32_t* packed, const uint16_t* scales, int bits,
                              int64_t K, int64_t N, uint16_t* W, cudaStream_t stream);
// H[i] = bf16(silu(H[i])) for n bf16 values (wq_pack.cu).
cudaError_t launch_silu_inplace(uint16_t* H, int64_t n, cudaStream_t stream);

// Small-M split-K GEMM (wq_gemm_small.cu).
struct GemmArgs {
  const void* X;
  const uint32_t* Wp;
  const void* S;
  void* Y;
  int64_t M, N, K;
  int bits;
  int num_sms;
  int device;
  int pdl;          // launch with programmatic stream serialization
  int split_hint;   // 0 = automatic cluster split
  int act;          // 0: none; 1: Y = bf16(silu(bf16(X . W))) (small and wt kernels only)
  const void* l2_prefetch;    // small kernel: bytes to pull into L2 once its weights have
  int64_t l2_prefetch_bytes;  // landed (the next GEMM's weights); 16-byte aligned and sized
  int weights_in_l2;          // the preceding GEMM pulled these weights into L2
  DiagHost diag;
};
// Returns cudaErrorNotSupported when the shape does not fit this kernel.
cudaError_t launch_gemm_small(const GemmArgs& a, cudaStream_t stream);
// num_sms: the device's SM count (the cluster split fills the SMs).
bool gemm_small_fits(int bits, int64_t K, int64_t N, int split_hint, int num_sms);

// Tensor-memory GEMM for M <= 16 (wq_gemm_skinny.cu).  Needs K / 128 to
// be even.
cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t stream);
bool gemm_skinny_fits(int bits, int64_t K, int64_t N);

// Tensor-memory GEMM for M <= 64 (16, 32 or 64 tokens per launch) whose
// CTAs take half an SM, so that consecutive launches overlap
// (wq_gemm_stream.cu).
// device < 0: no device to query, the split follows the SM count alone.
// Rows one launch of it takes (the MMA's N is 16, 32 or 64 tokens).
constexpr int kMaxStreamRows = 64;
cudaError_t launch_gemm_stream(const GemmArgs& a, cudaStream_t stream);
bool gemm_stream_fits(int bits, int64_t K, int64_t N, int split_hint, int num_sms, int device);
int gemm_stream_split(int bits, int64_t K, int64_t N, int split_hint, int num_sms, int device);

// Tensor-core GEMM for large M, dequantised weights staged in shared
// memory (wq_gemm_tc.cu).
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t stream);

// Tensor-core GEMM for large M, dequantised weights in tensor memory
// (wq_gemm_wt.cu).  Needs K / 128 to be a multiple of 4 (INT4) or 2 (INT8).
cudaError_t launch_gemm_wt(const GemmArgs& a, cudaStream_t stream);
bool gemm_wt_fits(int bits, int64_t M, int64_t K, int64_t N);

// The drafter's sliding-window attention (wq_swa.cu).  Q, O [B][Hq][128],
// K, V [Hkv][T][128], bf16; arguments checked by the caller.
struct SwaArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  int B, Hq, Hkv;
  int64_t T, window;
  int num_sms;
  int device;
  int pdl;          // launch with programmatic stream serialization
  int split_hint;   // 0 = automatic number of key slices per head
  DiagHost diag;
};
cudaError_t launch_swa_attention(const SwaArgs& a, cudaStream_t stream);

}  // namespace wq
