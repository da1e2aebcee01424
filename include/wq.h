/*
 * wq.h -- C ABI of the GB300 (sm_103a) weight-only quantized GEMM library.
 *
 * The operation is the quantized Linear of a weight-only INT4 / INT8 model:
 *
 *     Y[M,N] = X[M,K] . dequant(Wq)[K,N],   dequant(Wq)[k,n] = s[k/128,n] * q[k,n]
 *
 * with symmetric integer codes q, one bf16 scale per 128-element group along
 * K, bf16 activations X and output Y, fp32 accumulation.  Sources:
 *   - "Quantize the Target, Quantize the Drafter: Efficient Inference with
 *     Qwen3.5-4B" (arXiv 2607.04244 HTML): QAD paragraph (student weights are
 *     the dequantized s (.) Wq with frozen symmetric per-group scales),
 *     packing paragraph (round the updated weights back onto the same grid,
 *     served as W4A16), drafter-PTQ paragraph (group-wise symmetric INT4,
 *     group size 128).
 *   - "Qwen3.5-4B-DFlash-W8A16" model card, "What changed vs upstream" table
 *     (int8 weight-only, RTN, symmetric, group 128) and "Required vLLM
 *     patches" item 3 (the drafter's qkv projection runs the int8 GEMM).
 *
 * Conventions for every entry point
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference to them after the call returns.
 *   - Work is enqueued on `stream` and never synchronised; results are
 *     ready when the stream reaches that point.  Calls on different streams
 *     may run concurrently.
 *   - Arguments are checked before anything is launched: a non-OK status
 *     means nothing was enqueued.  A launch failure returns WQ_ERR_CUDA.
 *   - Every wait inside a kernel is bounded; a wait that runs out records
 *     WQ_ERR_DEVICE_TIMEOUT in a per-device error word that
 *     wq_last_device_error() reads after the caller synchronises.
 *   - Layouts are row-major and contiguous: X [M,K], Y [M,N], W [K,N],
 *     scales [K/128, N] (bf16 bit patterns).  A torch Linear weight
 *     [N,K] is passed transposed.  Pointers must be 16-byte aligned.
 *   - Shapes: group == 128, K % 128 == 0, N % 64 == 0, M >= 0 (M == 0 is a
 *     no-op), K*N < 2^40.
 *
 * Packed weight layout (tile-interleaved, uint32 words; the pages fix no
 * layout, this one is the library's own).  Element (k, n):
 *   nt = n/64, j8 = (n%64)/8, c = n%8, g = k/128, kk = k%128,
 *   kb = kk/32, t4 = (kk%32)/8, r = kk%8, lane = 4c + t4,
 *   slab = (nt*(K/128) + g)*8 + j8
 *   INT4: word index (slab*32 + lane)*4 + kb, nibble r/2 + 4*(r%2),
 *         field value q + 8
 *   INT8: w = 2kb + r/4, word index ((slab*2 + w/4)*32 + lane)*4 + w%4,
 *         byte (r%4)/2 + 2*((r%4)%2), field value q + 128
 * A 64-column x 128-deep (tile, group) cell is one contiguous 4 KiB (INT4)
 * or 8 KiB (INT8) block.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define WQ_API __attribute__((visibility("default")))
#else
#define WQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WQ_OK = 0,
  WQ_ERR_NULL = 1,           /* a required pointer is NULL */
  WQ_ERR_SHAPE = 2,          /* K, N, M or group outside the supported set */
  WQ_ERR_UNSUPPORTED = 3,    /* bits not 4/8, dtype unknown, no sm_103 GPU */
  WQ_ERR_ALIGN = 4,          /* a pointer is not 16-byte aligned */
  WQ_ERR_CUDA = 5,           /* a CUDA runtime call failed */
  WQ_ERR_DEVICE_TIMEOUT = 6  /* a bounded in-kernel wait ran out */
} wq_status;

typedef enum { WQ_F32 = 0, WQ_BF16 = 1 } wq_dtype;

/* Activation between the two projections of wq_mlp_w4a16 / wq_mlp_w8a16. */
typedef enum { WQ_ACT_NONE = 0, WQ_ACT_SILU = 1 } wq_act;

/* Number of uint32 words in a packed [K,N] weight with `bits` (4 or 8)
   bits per code: K*N/8 or K*N/4 -- the "8 per int32" packing of the INT4
   target ("Quantize the Target, Quantize the Drafter", packing paragraph:
   the weights are served as W4A16, group-wise INT4) and one byte per code
   for the int8 drafter ("Qwen3.5-4B-DFlash-W8A16" card, "What changed vs
   upstream" table, int8 weight-only).  Returns 0 for unsupported arguments
   (bits not 4/8, K % 128, N % 64, sizes out of range).  Pure host
   arithmetic: no device is needed. */
WQ_API size_t wq_packed_words(int bits, int64_t K, int64_t N);

/* Device bytes a packed [K,N] layer occupies: the codes (bits*K*N/8) plus
   its bf16 scales, one per 128-deep group and column (2*(K/128)*N).  This is
   the storage accounting of the "Qwen3.5-4B-DFlash-W8A16" card's "What
   changed vs upstream" table (1.00 GB of bf16 weights -> 521 MB as W8A16):
   one byte per INT8 weight (half a byte per INT4 weight) plus 2/128 of a
   byte per weight for the scales.  Returns 0 for unsupported arguments, as
   wq_packed_words.  Pure host arithmetic. */
WQ_API size_t wq_packed_bytes(int bits, int64_t K, int64_t N);

/*
 * Pack step (one-off per weight, "at packing time" in the packing paragraph
 * of the paper above; RTN per the W8A16 card's recipe).
 *   W          [K,N] fp32 or bf16 (wdt), finite values.
 *   scales_in  bf16 [K/128,N] or NULL.  Given: the grid is fixed and the
 *              codes are q = clamp(rint(w/s), qmin, qmax) (round half to
 *              even, IEEE fp32 divide) -- re-rounding onto a frozen grid.
 *              Values must be positive and finite.  NULL: RTN scales
 *              s = bf16_rne(absmax_group / qpos), qpos = 7 (INT4) or 127
 *              (INT8), s = 1 for an all-zero group.
 *   scales_out bf16 [K/128,N]: the scales used (a copy of scales_in when
 *              given; may equal scales_in).
 *   packed     wq_packed_words(bits,K,N) words, layout above.
 *   [qmin,qmax] = [-8,7] for bits 4, [-128,127] for bits 8.
 */
WQ_API wq_status wq_pack_symmetric(const void* W, wq_dtype wdt, int64_t K, int64_t N,
                            int bits, int group, const uint16_t* scales_in,
                            uint16_t* scales_out, uint32_t* packed,
                            cudaStream_t stream);

/* Interleave ready-made int8 codes [K,N] into the packed layout, without
   rounding: the codes are already on the grid, as when a GPTQ-quantized
   layer is packed ("Quantize the Target, Quantize the Drafter" project
   README, pipeline table: the GPTQ drafter export and pack_ct.sh; the
   packing paragraph of the paper: codes on a fixed symmetric grid).  Each
   code must lie in [qmin,qmax] ([-8,7] for bits 4, [-128,127] for bits 8);
   other values are wrapped to the field width.  `codes` and `packed` are
   caller-owned device memory, 16-byte aligned; `packed` holds
   wq_packed_words(bits,K,N) words.  Errors: WQ_ERR_NULL, WQ_ERR_UNSUPPORTED
   (bits), WQ_ERR_SHAPE (K % 128, N % 64), WQ_ERR_ALIGN, WQ_ERR_CUDA.
   Stream-ordered; allocates nothing. */
WQ_API wq_status wq_pack_codes(const int8_t* codes, int64_t K, int64_t N, int bits,
                        uint32_t* packed, cudaStream_t stream);

/* Import a layer stored the way its serving checkpoint stores it: output-
   channel-major, codes packed along the input dimension.  The target model
   is served as a compressed-tensors checkpoint ("Quantize the Target,
   Quantize the Drafter" project README, pipeline table: pack_ct.sh; the
   GPTQ-W4A16 drafter card: --quantization compressed-tensors); the pages do
   not print its layout, and this call reads the format's definition:
     qweight    [N][K * bits / 32] uint32, row-major: word j of row n holds
                the 32/bits consecutive codes k = (32/bits) j + p of column n
                at bits [bits p, bits p + bits), offset-binary (q + 8 for
                INT4, q + 128 for INT8);
     scales_nk  [N][K / 128] bf16, row-major.
   Writes this library's packed layout (`packed`, wq_packed_words(bits, K,
   N) words) and the scales as [K/128, N] bf16 (`scales_out`), bit-exact.
   Errors: WQ_ERR_NULL, WQ_ERR_UNSUPPORTED (bits), WQ_ERR_SHAPE (group !=
   128, K % 128, N % 64), WQ_ERR_ALIGN (qweight, packed, scales_out 16 bytes;
   scales_nk 2 bytes), WQ_ERR_CUDA.  Stream-ordered; allocates nothing. */
WQ_API wq_status wq_import_packed_nk(const uint32_t* qweight, const uint16_t* scales_nk, int bits,
                                     int64_t K, int64_t N, int group, uint32_t* packed,
                                     uint16_t* scales_out, cudaStream_t stream);

/* The effective weight of a packed layer, W[k][n] = bf16(s[k/128][n] *
   q[k][n]) as a row-major bf16 [K,N] matrix (s times q is exact in fp32 and
   rounded once, ties to even).  This is what the fused-KV patch of the
   "naveenrajk/Qwen3.5-4B-DFlash-W8A16" card ("Required vLLM patches",
   item 2) recovers by running an identity matrix through the quantized
   projection; this call returns it without a GEMM.  `packed` and `scales`
   are as for the GEMMs (bits 4 or 8, group 128); `W` is caller-owned device
   memory of K*N bf16.  Errors: WQ_ERR_NULL, WQ_ERR_UNSUPPORTED (bits),
   WQ_ERR_SHAPE (group != 128, K % 128, N % 64), WQ_ERR_ALIGN (16 bytes),
   WQ_ERR_CUDA.  Stream-ordered; allocates nothing. */
WQ_API wq_status wq_dequantize(const uint32_t* packed, const uint16_t* scales, int bits,
                               int64_t K, int64_t N, int group, uint16_t* W,
                               cudaStream_t stream);

/* Inverse of the interleave: the int8 codes q [K,N] (row-major, values in
   [qmin,qmax]) of a packed weight -- the codes the QAD paragraph of
   "Quantize the Target, Quantize the Drafter" multiplies by the frozen
   scales (student weights s (.) Wq).  `packed` (wq_packed_words words) and
   `codes` (K*N bytes) are caller-owned device memory, 16-byte aligned.
   Errors as wq_pack_codes.  Stream-ordered; allocates nothing. */
WQ_API wq_status wq_unpack(const uint32_t* packed, int bits, int64_t K, int64_t N,
                    int8_t* codes, cudaStream_t stream);

/*
 * W4A16 GEMM (the verifier's quantized Linear): Y = X . dequant(Wp, scales).
 *   X bf16 [M,K], Wp packed INT4 (bits 4), scales bf16 [K/128,N],
 *   Y bf16 [M,N] (fp32 accumulation, round to nearest even on store).
 *   group must be 128.  Y must not overlap X, Wp or scales.
 * Small M (one speculative block of 16 tokens, a few blocks) runs the
 * memory-bound kernel; large M (prefill) runs the tensor-core kernel.
 */
WQ_API wq_status wq_gemm_w4a16(const void* X, const uint32_t* Wp, const void* scales,
                        void* Y, int64_t M, int64_t N, int64_t K, int group,
                        cudaStream_t stream);

/* W8A16 GEMM (the int8 drafter's quantized Linear): as wq_gemm_w4a16 with a
   packed INT8 weight (bits 8). */
WQ_API wq_status wq_gemm_w8a16(const void* X, const uint32_t* Wp, const void* scales,
                        void* Y, int64_t M, int64_t N, int64_t K, int group,
                        cudaStream_t stream);

/*
 * The two quantized projections of one MLP block in one call (the INT4
 * target's verifier forward, "Quantize the Target, Quantize the Drafter"):
 *   H = act(bf16(X . dequant(Wu, Su)))   X bf16 [M,K], Wu [K,N1], H bf16 [M,N1]
 *   Y = bf16(H . dequant(Wd, Sd))        Wd [N1,N2], Y bf16 [M,N2]
 * act: WQ_ACT_NONE, or WQ_ACT_SILU = the up-projection's bf16 result h
 * mapped to h / (1 + e^-h) in fp32 and rounded to bf16 (the pages name no
 * activation; SiLU is the one the target family uses).  H is caller-owned
 * device memory and holds the activated intermediate on return.  Each
 * projection runs the kernel wq_gemm_w4a16 would pick (the activation is
 * applied in the store of the warp-MMA and tensor-memory tiled kernels, in a
 * separate pass otherwise); with the warp-MMA kernel the up-projection also
 * pulls Wd into L2 once its own weights have landed.  Shapes and errors as
 * for the GEMMs (K, N1 multiples of 128; N1, N2 multiples of 64; 16-byte
 * aligned pointers), plus WQ_ERR_UNSUPPORTED for an unknown act.  H and Y
 * must not overlap each other or the inputs.  Stream-ordered; allocates
 * nothing.  wq_mlp_w8a16: the same with packed INT8 weights.
 */
WQ_API wq_status wq_mlp_w4a16(const void* X, const uint32_t* Wu, const void* Su,
                              const uint32_t* Wd, const void* Sd, void* H, void* Y,
                              int64_t M, int64_t K, int64_t N1, int64_t N2, int group,
                              int act, cudaStream_t stream);
/*
 * The drafter's attention with a symmetric sliding window ("Quantize the
 * Target, Quantize the Drafter", drafter-SWA paragraph): a block of B
 * query tokens (1..16: the anchor and the drafted tokens) at positions
 * p_b = T - B + b, the last B of a sequence of T tokens whose keys and values
 * are all cached, attends bidirectionally; query b sees key j iff
 * |j - p_b| <= window / 2.  window == 0, or T <= window (a sequence the
 * window covers), is full attention.  Scores q.k / sqrt(128), softmax over
 * the visible keys, weighted sum of the values (fp32 accumulation, output
 * rounded to bf16).
 *   Q [B][Hq][128], K and V [Hkv][T][128], O [B][Hq][128], all bf16,
 *   row-major and contiguous, 16-byte aligned, caller-owned device memory;
 *   query head h reads key/value head h / (Hq / Hkv).
 * Errors: WQ_ERR_NULL, WQ_ERR_UNSUPPORTED (head dim other than 128),
 * WQ_ERR_SHAPE (B outside 1..16, Hq not a multiple of Hkv, Hq > 4096, T < B,
 * T > 2^30, Hkv * T > 2^31 - 256, window < 0), WQ_ERR_ALIGN, WQ_ERR_CUDA,
 * and WQ_ERR_DEVICE_TIMEOUT through wq_last_device_error().  Stream-ordered;
 * allocates nothing.
 */
WQ_API wq_status wq_swa_attention(const void* Q, const void* K, const void* V, void* O,
                                  int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t T,
                                  int64_t window, cudaStream_t stream);

WQ_API wq_status wq_mlp_w8a16(const void* X, const uint32_t* Wu, const void* Su,
                              const uint32_t* Wd, const void* Sd, void* H, void* Y,
                              int64_t M, int64_t K, int64_t N1, int64_t N2, int group,
                              int act, cudaStream_t stream);

/* The per-device error word of the current device: WQ_OK or
   WQ_ERR_DEVICE_TIMEOUT.  Synchronous (reads device memory); call after
   synchronising the streams of interest.  wq_clear_device_error() resets it. */
WQ_API wq_status wq_last_device_error(void);
WQ_API wq_status wq_clear_device_error(void);

/* Human-readable name of a status. */
WQ_API const char* wq_status_string(wq_status status);

/* The CUDA error behind the calling thread's last WQ_ERR_CUDA, as text. */
WQ_API const char* wq_last_cuda_error(void);

/* Diagnostics for tests.  wq_debug_set_wait_limit_ns: the time limit of
   every in-kernel wait in nanoseconds (0 restores the default of 2 s).
   wq_debug_force_timeout(mode): 0 off; 1 every CTA of the next GEMMs first
   waits on a barrier nothing completes -- the wait runs out, is reported,
   and the GEMM then runs normally; 2 the data waits look for a phase that
   never completes, so the GEMM gives up, lets its copies land and reports
   (its output is then undefined).  Both report WQ_ERR_DEVICE_TIMEOUT
   through wq_last_device_error() without any fault. */
WQ_API void wq_debug_set_wait_limit_ns(uint64_t ns);
WQ_API void wq_debug_force_timeout(int mode);

/* Tuning and test hooks: force the number of CTAs of a cluster that split
   one tile's K range in the small-M kernels and in the tensor-memory kernel
   at M < 512 (1..8, at most the tile's packed chunks; 0 restores the
   automatic choice; a split the tensor-memory kernel cannot take makes the
   call report WQ_ERR_UNSUPPORTED; for wq_swa_attention, the number of key
   slices per head), and enable programmatic dependent launch, which lets a
   GEMM start streaming its weights while the preceding kernel on the stream
   finishes, and lets the attention kernel launch and set up meanwhile (it
   reads nothing before that kernel completes).  With it on, the weights and
   scales of a GEMM must not be written by the kernel immediately before it
   on the same stream (X and Y may be).  Both settings are process-wide:
   they apply to every later call from every thread of the process (not
   thread-safe with respect to calls in flight on other threads), and
   programmatic launch is off until a caller turns it on. */
WQ_API void wq_debug_set_split(int cs);
WQ_API void wq_set_programmatic_launch(int on);

/* Test hook: run every GEMM on one kernel family regardless of M (0 the
   warp-MMA small-M kernel, 1 the tiled tensor-core kernel with dequantised
   weights in shared memory, 2 the tensor-memory small-M kernel, which needs
   K/128 to be even and otherwise falls back to 0, 3 the
   tiled tensor-core kernel with dequantised weights in tensor memory, which
   needs K/128 to be a multiple of 4 (INT4) or 2 (INT8) and otherwise falls
   back to 1, 4 the tensor-memory small-M kernel whose launches overlap
   (weights streamed by TMA, a K split reduced across a thread-block
   cluster; up to 64 rows per launch, taller inputs in 64-row slices),
   which needs at most 32 groups per CTA and otherwise falls back to 0;
   any other value restores the automatic choice: M <= 64 kernel 4 (one
   launch), or where kernel 4 does not apply kernel 0 in 16-row slices
   (M <= 32) or kernel 3 (M from 33 to 64); larger M kernel 3, or kernel 1
   where kernel 3 does not apply). */
WQ_API void wq_debug_force_regime(int regime);

/* Which kernel family a GEMM of this shape runs (numbering as in
   wq_debug_force_regime).  -1 for unsupported shapes. */
WQ_API int wq_gemm_regime(int bits, int64_t M, int64_t N, int64_t K);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
