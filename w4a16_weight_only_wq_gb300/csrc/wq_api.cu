// wq_api.cu -- the C ABI declared in include/wq.h: argument checks, regime
// selection, launches on the caller's stream, and the per-device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "wq.h"
#include "wq_internal.h"

namespace {

// Per-device error word written by bounded waits that ran out.
__device__ uint32_t g_wq_device_error;

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_pdl{0};
std::atomic<int> g_split_hint{0};
std::atomic<int> g_force_regime{-1};

// Rows up to which the stream kernel (one launch takes up to 64 rows) is
// used; larger M runs on the tiled tensor-memory kernel.  Of the shapes the
// stream kernel cannot take, those up to kSmallMaxM rows go to the warp-MMA
// kernel (16 rows per launch), taller ones to the tiled kernel.
constexpr int64_t kStreamMaxM = wq::kMaxStreamRows;
constexpr int64_t kSmallMaxM = 32;

// 0: warp-MMA small-M kernel (16 rows per launch), 1: tensor-core tiled
// kernel with dequantised weights in shared memory, 2: tensor-memory
// small-M kernel (16 rows per launch), 3: tensor-core tiled kernel with
// dequantised weights in tensor memory, 4: tensor-memory small-M kernel
// whose launches overlap (16 rows per launch).
constexpr int kNumRegimes = 5;
int pick_regime(int64_t M) {
  const int f = g_force_regime.load();
  if (f >= 0 && f < kNumRegimes) return f;
  // measured at K = 2560, N = 9728: kernel 3 is faster than kernel 1 at
  // every M from 64 to 8192; kernel 1 takes the shapes kernel 3 cannot.
  // At M <= 32, kernel 4 (whose launches overlap) beats kernel 0 on the
  // INT4 decode shapes.  From 33 to 64 rows kernel 4's single launch beats
  // kernel 3 on K x N = 2560 x 9728, 2560 x 2560 and 9728 x 2560, INT4 and
  // INT8 (M = 64, INT4: 8.1 against 12.1 us, 5.8 against 7.9, 9.6 against
  // 14.6); above 64 rows it needs a second launch and kernel 3 wins.
  return M <= kStreamMaxM ? 4 : 3;
}

// The family that takes a shape kernel 4 cannot index.
int stream_fallback(int64_t M) { return M <= kSmallMaxM ? 0 : 3; }
thread_local cudaError_t t_last_cuda = cudaSuccess;

wq_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return WQ_OK;
  t_last_cuda = e;
  return WQ_ERR_CUDA;
}

struct DeviceInfo {
  int num_sms = 0;
  int cc = 0;
  uint32_t* err = nullptr;
};
DeviceInfo g_dev[64];
std::atomic<uint64_t> g_dev_ready{0};
std::mutex g_dev_mu;

wq_status device_info(int* dev_out, DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WQ_ERR_CUDA;
  *dev_out = dev;
  const uint64_t bit = 1ull << dev;
  if (!(g_dev_ready.load(std::memory_order_acquire) & bit)) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!(g_dev_ready.load() & bit)) {
      DeviceInfo d;
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return WQ_ERR_CUDA;
      d.cc = major * 10 + minor;
      if (d.cc != 103) return WQ_ERR_UNSUPPORTED;  // built for sm_103a only
      if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_wq_device_error) != cudaSuccess)
        return WQ_ERR_CUDA;
      g_dev[dev] = d;
      g_dev_ready.fetch_or(bit, std::memory_order_release);
    }
  }
  *info = g_dev[dev];
  return WQ_OK;
}

// SM count of the current device for host-side queries; 152 (a GB300) when
// no device is visible, so that the answer is defined on a build machine.
int sm_count_or_default() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  cudaGetLastError();  // no device: not an error of a later call
  return 152;
}

// The current device if it is an sm_103 GPU, else -1 (host-side queries).
int current_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return major * 10 + minor == 103 ? dev : -1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

wq_status check_kn(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 64 != 0) return WQ_ERR_SHAPE;
  if (K > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K * N >= (int64_t(1) << 40))
    return WQ_ERR_SHAPE;
  if (K / 128 > 65535) return WQ_ERR_SHAPE;
  return WQ_OK;
}

wq::DiagHost diag_for(const DeviceInfo& d) {
  wq::DiagHost h;
  h.err = d.err;
  h.wait_limit_ns = g_wait_limit_ns.load();
  h.force_timeout = g_force_timeout.load();
  return h;
}

wq_status check_gemm(const void* X, const uint32_t* Wp, const void* scales, const void* Y,
                     int64_t M, int64_t N, int64_t K, int group) {
  if (!X || !Wp || !scales || !Y) return M == 0 ? WQ_OK : WQ_ERR_NULL;
  if (group != 128) return WQ_ERR_SHAPE;
  if (M < 0 || M > (int64_t(1) << 30)) return WQ_ERR_SHAPE;
  wq_status st = check_kn(K, N);
  if (st != WQ_OK) return st;
  if (M * K >= (int64_t(1) << 40) || M * N >= (int64_t(1) << 40)) return WQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(Wp) || !aligned16(scales) || !aligned16(Y))
    return WQ_ERR_ALIGN;
  return WQ_OK;
}

// One GEMM on the chosen kernel family, arguments already checked.  act: the
// activation of the fused MLP's up-projection; *act_done tells whether the
// kernel applied it (the warp-MMA and tensor-memory tiled kernels do).
// pf / pf_bytes: the next GEMM's weights, for the warp-MMA small-M kernel
// to pull into L2 once its own weights have landed; *prefetched tells
// whether a launch was given them.  weights_in_l2: this GEMM's weights were
// pulled so by the one before it.
wq_status gemm_run(int bits, const void* X, const uint32_t* Wp, const void* scales, void* Y,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream, int act,
                   const void* pf, int64_t pf_bytes, bool weights_in_l2, bool* act_done,
                   bool* prefetched) {
  *act_done = act == 0;
  *prefetched = false;
  if (M == 0) return WQ_OK;
  int dev;
  DeviceInfo d;
  wq_status st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  wq::GemmArgs a;
  a.X = X;
  a.Wp = Wp;
  a.S = scales;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = bits;
  a.num_sms = d.num_sms;
  a.device = dev;
  a.pdl = g_pdl.load();
  a.split_hint = g_split_hint.load();
  a.act = 0;
  a.l2_prefetch = nullptr;
  a.l2_prefetch_bytes = 0;
  a.weights_in_l2 = weights_in_l2 ? 1 : 0;
  a.diag = diag_for(d);
  int regime = pick_regime(M);
  if (regime == 4 && !wq::gemm_stream_fits(bits, K, N, a.split_hint, d.num_sms, dev))
    regime = stream_fallback(M);
  if (regime == 0 && !wq::gemm_small_fits(bits, K, N, a.split_hint, d.num_sms)) regime = 1;
  if (regime == 3 && !wq::gemm_wt_fits(bits, M, K, N)) regime = 1;
  if (regime == 3) {
    a.act = act;
    cudaError_t e = wq::launch_gemm_wt(a, stream);
    if (e == cudaErrorNotSupported) return WQ_ERR_UNSUPPORTED;
    *act_done = true;
    return cuda_status(e);
  }
  if (regime == 1) {
    cudaError_t e = wq::launch_gemm_tc(a, stream);
    if (e == cudaErrorNotSupported) return WQ_ERR_UNSUPPORTED;
    return cuda_status(e);
  }
  // The small-M kernels take a bounded number of rows per launch (the
  // stream kernel 64, the others 16); taller inputs are processed in slices.
  const size_t xrow = static_cast<size_t>(K) * 2, yrow = static_cast<size_t>(N) * 2;
  // the activation is applied in the store of kernels 0 and 4; kernel 2 has none
  if (regime == 0 || regime == 4) a.act = act;
  // rows [r0, r0 + h) on the warp-MMA kernel in 16-row slices, each slice
  // that does not fit it on the tiled kernel
  auto run_small = [&](int64_t r0, int64_t h, bool last_rows) -> wq_status {
    for (int64_t m0 = r0; m0 < r0 + h; m0 += 16) {
      wq::GemmArgs b = a;
      b.X = static_cast<const char*>(X) + m0 * xrow;
      b.Y = static_cast<char*>(Y) + m0 * yrow;
      b.M = (r0 + h - m0) < 16 ? (r0 + h - m0) : 16;
      const bool last = last_rows && m0 + 16 >= r0 + h;
      b.l2_prefetch = last && pf != nullptr ? pf : nullptr;
      b.l2_prefetch_bytes = b.l2_prefetch != nullptr ? pf_bytes : 0;
      cudaError_t e = wq::launch_gemm_small(b, stream);
      if (e == cudaErrorNotSupported) {
        // the slice does not fit the small-M kernel: the tiled kernel takes it
        b.act = 0;
        e = wq::launch_gemm_tc(b, stream);
        if (e == cudaErrorNotSupported) return WQ_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return cuda_status(e);
        if (a.act != 0) {  // the caller counts on this slice being activated
          const wq_status st2 = cuda_status(wq::launch_silu_inplace(
              static_cast<uint16_t*>(b.Y), b.M * N, stream));
          if (st2 != WQ_OK) return st2;
        }
        continue;
      }
      if (e != cudaSuccess) return cuda_status(e);
      if (b.l2_prefetch != nullptr) *prefetched = true;
    }
    return WQ_OK;
  };
  const int64_t step = regime == 4 ? wq::kMaxStreamRows : 16;
  for (int64_t m0 = 0; m0 < M; m0 += step) {
    const int64_t h = (M - m0) < step ? (M - m0) : step;
    const bool last = m0 + step >= M;
    cudaError_t e = cudaErrorNotSupported;
    if (regime == 4 || regime == 2) {
      a.X = static_cast<const char*>(X) + m0 * xrow;
      a.Y = static_cast<char*>(Y) + m0 * yrow;
      a.M = h;
      a.l2_prefetch = nullptr;
      a.l2_prefetch_bytes = 0;
      e = regime == 4 ? wq::launch_gemm_stream(a, stream) : wq::launch_gemm_skinny(a, stream);
      if (e != cudaSuccess && e != cudaErrorNotSupported) return cuda_status(e);
    }
    // shapes the tensor-memory kernels cannot index go to the warp-MMA kernel
    if (regime == 0 || e == cudaErrorNotSupported) {
      const wq_status st = run_small(m0, h, last);
      if (st != WQ_OK) return st;
    }
  }
  *act_done = act == 0 || regime == 0 || regime == 4;
  return WQ_OK;
}

wq_status gemm_common(int bits, const void* X, const uint32_t* Wp, const void* scales, void* Y,
                      int64_t M, int64_t N, int64_t K, int group, cudaStream_t stream) {
  wq_status st = check_gemm(X, Wp, scales, Y, M, N, K, group);
  if (st != WQ_OK || M == 0) return st;
  bool act_done, prefetched;
  return gemm_run(bits, X, Wp, scales, Y, M, N, K, stream, 0, nullptr, 0, false, &act_done,
                  &prefetched);
}

// The fused MLP pair: H = act(bf16(X . Wu)), Y = bf16(H . Wd).
wq_status mlp_common(int bits, const void* X, const uint32_t* Wu, const void* Su,
                     const uint32_t* Wd, const void* Sd, void* H, void* Y, int64_t M, int64_t K,
                     int64_t N1, int64_t N2, int group, int act, cudaStream_t stream) {
  if (act != WQ_ACT_NONE && act != WQ_ACT_SILU) return WQ_ERR_UNSUPPORTED;
  wq_status st = check_gemm(X, Wu, Su, H, M, N1, K, group);
  if (st != WQ_OK) return st;
  st = check_gemm(H, Wd, Sd, Y, M, N2, N1, group);
  if (st != WQ_OK || M == 0) return st;
  const int64_t wd_bytes = bits == 4 ? N1 * N2 / 2 : N1 * N2;
  bool act_done = false, prefetched = false, unused = false;
  st = gemm_run(bits, X, Wu, Su, H, M, N1, K, stream, act, Wd, wd_bytes, false, &act_done,
                &prefetched);
  if (st != WQ_OK) return st;
  if (!act_done) {
    st = cuda_status(wq::launch_silu_inplace(static_cast<uint16_t*>(H), M * N1, stream));
    if (st != WQ_OK) return st;
  }
  // the down-projection's copy sizes assume its weights are in L2 only when
  // the up-projection actually pulled them there
  return gemm_run(bits, H, Wd, Sd, Y, M, N2, N1, stream, 0, nullptr, 0, prefetched, &act_done,
                  &unused);
}

}  // namespace

extern "C" {

size_t wq_packed_words(int bits, int64_t K, int64_t N) {
  if ((bits != 4 && bits != 8) || check_kn(K, N) != WQ_OK) return 0;
  return static_cast<size_t>(bits == 4 ? K * N / 8 : K * N / 4);
}

size_t wq_packed_bytes(int bits, int64_t K, int64_t N) {
  const size_t words = wq_packed_words(bits, K, N);
  if (words == 0) return 0;
  return words * 4 + static_cast<size_t>(K / 128) * static_cast<size_t>(N) * 2;
}

wq_status wq_pack_symmetric(const void* W, wq_dtype wdt, int64_t K, int64_t N,
                            int bits, int group, const uint16_t* scales_in,
                            uint16_t* scales_out, uint32_t* packed,
                            cudaStream_t stream) {
  if (!W || !scales_out || !packed) return WQ_ERR_NULL;
  if (bits != 4 && bits != 8) return WQ_ERR_UNSUPPORTED;
  if (wdt != WQ_F32 && wdt != WQ_BF16) return WQ_ERR_UNSUPPORTED;
  if (group != 128) return WQ_ERR_SHAPE;
  wq_status st = check_kn(K, N);
  if (st != WQ_OK) return st;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(scales_out) ||
      (scales_in && !aligned16(scales_in)))
    return WQ_ERR_ALIGN;
  int dev;
  DeviceInfo d;
  st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  cudaError_t e = wq::launch_pack_symmetric(W, wdt == WQ_F32 ? 0 : 1, K, N, bits,
                                            scales_in, scales_out, packed, stream);
  return cuda_status(e);
}

wq_status wq_pack_codes(const int8_t* codes, int64_t K, int64_t N, int bits,
                        uint32_t* packed, cudaStream_t stream) {
  if (!codes || !packed) return WQ_ERR_NULL;
  if (bits != 4 && bits != 8) return WQ_ERR_UNSUPPORTED;
  wq_status st = check_kn(K, N);
  if (st != WQ_OK) return st;
  if (!aligned16(codes) || !aligned16(packed)) return WQ_ERR_ALIGN;
  int dev;
  DeviceInfo d;
  st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  cudaError_t e = wq::launch_pack_codes(codes, K, N, bits, packed, stream);
  return cuda_status(e);
}

wq_status wq_import_packed_nk(const uint32_t* qweight, const uint16_t* scales_nk, int bits,
                              int64_t K, int64_t N, int group, uint32_t* packed,
                              uint16_t* scales_out, cudaStream_t stream) {
  if (!qweight || !scales_nk || !packed || !scales_out) return WQ_ERR_NULL;
  if (bits != 4 && bits != 8) return WQ_ERR_UNSUPPORTED;
  if (group != 128) return WQ_ERR_SHAPE;
  wq_status st = check_kn(K, N);
  if (st != WQ_OK) return st;
  if (!aligned16(qweight) || !aligned16(packed) || !aligned16(scales_out) ||
      reinterpret_cast<uintptr_t>(scales_nk) % 2 != 0)
    return WQ_ERR_ALIGN;
  int dev;
  DeviceInfo d;
  st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  return cuda_status(
      wq::launch_import_nk(qweight, scales_nk, bits, K, N, packed, scales_out, stream));
}

wq_status wq_dequantize(const uint32_t* packed, const uint16_t* scales, int bits, int64_t K,
                        int64_t N, int group, uint16_t* W, cudaStream_t stream) {
  if (!packed || !scales || !W) return WQ_ERR_NULL;
  if (bits != 4 && bits != 8) return WQ_ERR_UNSUPPORTED;
  if (group != 128) return WQ_ERR_SHAPE;
  wq_status st = check_kn(K, N);
  if (st != WQ_OK) return st;
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(W)) return WQ_ERR_ALIGN;
  int dev;
  DeviceInfo d;
  st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  return cuda_status(wq::launch_dequantize(packed, scales, bits, K, N, W, stream));
}

wq_status wq_unpack(const uint32_t* packed, int bits, int64_t K, int64_t N,
                    int8_t* codes, cudaStream_t stream) {
  if (!codes || !packed) return WQ_ERR_NULL;
  if (bits != 4 && bits != 8) return WQ_ERR_UNSUPPORTED;
  wq_status st = check_kn(K, N);
  if (st != WQ_OK) return st;
  if (!aligned16(codes) || !aligned16(packed)) return WQ_ERR_ALIGN;
  int dev;
  DeviceInfo d;
  st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  cudaError_t e = wq::launch_unpack(packed, bits, K, N, codes, stream);
  return cuda_status(e);
}

wq_status wq_gemm_w4a16(const void* X, const uint32_t* Wp, const void* scales,
                        void* Y, int64_t M, int64_t N, int64_t K, int group,
                        cudaStream_t stream) {
  return gemm_common(4, X, Wp, scales, Y, M, N, K, group, stream);
}

wq_status wq_gemm_w8a16(const void* X, const uint32_t* Wp, const void* scales,
                        void* Y, int64_t M, int64_t N, int64_t K, int group,
                        cudaStream_t stream) {
  return gemm_common(8, X, Wp, scales, Y, M, N, K, group, stream);
}

wq_status wq_swa_attention(const void* Q, const void* K, const void* V, void* O, int64_t B,
                           int64_t Hq, int64_t Hkv, int64_t D, int64_t T, int64_t window,
                           cudaStream_t stream) {
  if (B == 0) return WQ_OK;
  if (!Q || !K || !V || !O) return WQ_ERR_NULL;
  if (D != 128) return WQ_ERR_UNSUPPORTED;
  if (B < 1 || B > 16 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 4096 || T < B ||
      T > (int64_t(1) << 30) || window < 0 || Hkv * T > (int64_t(1) << 31) - 256)
    return WQ_ERR_SHAPE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return WQ_ERR_ALIGN;
  int dev;
  DeviceInfo d;
  wq_status st = device_info(&dev, &d);
  if (st != WQ_OK) return st;
  wq::SwaArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.B = static_cast<int>(B);
  a.Hq = static_cast<int>(Hq);
  a.Hkv = static_cast<int>(Hkv);
  a.T = T;
  a.window = window;
  a.num_sms = d.num_sms;
  a.device = dev;
  a.pdl = g_pdl.load();
  a.split_hint = g_split_hint.load();
  a.diag = diag_for(d);
  return cuda_status(wq::launch_swa_attention(a, stream));
}

wq_status wq_mlp_w4a16(const void* X, const uint32_t* Wu, const void* Su, const uint32_t* Wd,
                       const void* Sd, void* H, void* Y, int64_t M, int64_t K, int64_t N1,
                       int64_t N2, int group, int act, cudaStream_t stream) {
  return mlp_common(4, X, Wu, Su, Wd, Sd, H, Y, M, K, N1, N2, group, act, stream);
}

wq_status wq_mlp_w8a16(const void* X, const uint32_t* Wu, const void* Su, const uint32_t* Wd,
                       const void* Sd, void* H, void* Y, int64_t M, int64_t K, int64_t N1,
                       int64_t N2, int group, int act, cudaStream_t stream) {
  return mlp_common(8, X, Wu, Su, Wd, Sd, H, Y, M, K, N1, N2, group, act, stream);
}

wq_status wq_last_device_error(void) {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_wq_device_error, sizeof(v)) != cudaSuccess)
    return WQ_ERR_CUDA;
  return static_cast<wq_status>(v);
}

wq_status wq_clear_device_error(void) {
  const uint32_t z = 0;
  if (cudaMemcpyToSymbol(g_wq_device_error, &z, sizeof(z)) != cudaSuccess)
    return WQ_ERR_CUDA;
  return WQ_OK;
}

const char* wq_status_string(wq_status s) {
  switch (s) {
    case WQ_OK: return "WQ_OK";
    case WQ_ERR_NULL: return "WQ_ERR_NULL: a required pointer is NULL";
    case WQ_ERR_SHAPE: return "WQ_ERR_SHAPE: unsupported M/N/K/group";
    case WQ_ERR_UNSUPPORTED: return "WQ_ERR_UNSUPPORTED: bits, dtype or device not supported";
    case WQ_ERR_ALIGN: return "WQ_ERR_ALIGN: pointer not 16-byte aligned";
    case WQ_ERR_CUDA: return "WQ_ERR_CUDA: a CUDA runtime call failed";
    case WQ_ERR_DEVICE_TIMEOUT: return "WQ_ERR_DEVICE_TIMEOUT: an in-kernel wait ran out";
  }
  return "unknown wq_status";
}

void wq_debug_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns);
}

void wq_debug_force_timeout(int mode) {
  g_force_timeout.store(mode == 1 || mode == 2 ? mode : 0);
}

const char* wq_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda); }

void wq_debug_set_split(int cs) { g_split_hint.store(cs < 0 || cs > 8 ? 0 : cs); }

void wq_set_programmatic_launch(int on) { g_pdl.store(on ? 1 : 0); }

void wq_debug_force_regime(int regime) {
  g_force_regime.store(regime >= 0 && regime < kNumRegimes ? regime : -1);
}

int wq_gemm_regime(int bits, int64_t M, int64_t N, int64_t K) {
  if ((bits != 4 && bits != 8) || M < 0 || check_kn(K, N) != WQ_OK) return -1;
  int r = pick_regime(M);
  const int sms = sm_count_or_default();
  if (r == 4 && !wq::gemm_stream_fits(bits, K, N, g_split_hint.load(), sms, current_sm103()))
    r = stream_fallback(M);
  if (r == 2 && !wq::gemm_skinny_fits(bits, K, N)) r = 0;
  // shapes whose X slice does not fit the small-M kernel run on the tiled one
  if (r == 0 && !wq::gemm_small_fits(bits, K, N, g_split_hint.load(), sms)) r = 1;
  if (r == 3 && !wq::gemm_wt_fits(bits, M, K, N)) r = 1;
  return r;
}

}  // extern "C"
