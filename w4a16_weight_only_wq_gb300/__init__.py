"""Thin Python binding of libwq (include/wq.h): argument marshalling only.

Every step of the path (packing, dequant, GEMM) runs in the library's CUDA
kernels; this module converts torch tensors to device pointers and the
current torch stream to a ``cudaStream_t``.  There is no fallback: if the
library is missing, importing the binding raises.

Two layers:
  * ``wq_*`` functions with the C names and C arguments (integer device
    pointers, sizes, stream handle) -- the ABI as-is;
  * tensor helpers (``pack_symmetric``, ``pack_codes``, ``unpack``,
    ``gemm_w4a16``, ``gemm_w8a16``) that allocate outputs with torch and
    call the ABI on the current stream.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libwq.so")

WQ_OK = 0
WQ_ERR_NULL = 1
WQ_ERR_SHAPE = 2
WQ_ERR_UNSUPPORTED = 3
WQ_ERR_ALIGN = 4
WQ_ERR_CUDA = 5
WQ_ERR_DEVICE_TIMEOUT = 6
WQ_F32 = 0
WQ_BF16 = 1
WQ_ACT_NONE = 0
WQ_ACT_SILU = 1
GROUP = 128

EXPORTED = (
    "wq_packed_words", "wq_packed_bytes", "wq_pack_symmetric", "wq_pack_codes", "wq_unpack", "wq_dequantize",
    "wq_import_packed_nk",
    "wq_gemm_w4a16", "wq_gemm_w8a16", "wq_mlp_w4a16", "wq_mlp_w8a16", "wq_swa_attention",
    "wq_last_device_error",
    "wq_clear_device_error", "wq_status_string", "wq_debug_set_wait_limit_ns",
    "wq_debug_force_timeout", "wq_gemm_regime", "wq_debug_set_split",
    "wq_set_programmatic_launch", "wq_last_cuda_error", "wq_debug_force_regime",
)


class WQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)}"
        if status == WQ_ERR_CUDA:
            msg += f" ({wq_last_cuda_error()})"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libwq.so not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    sig = {
        "wq_packed_words": ([I, I64, I64], ctypes.c_size_t),
        "wq_packed_bytes": ([I, I64, I64], ctypes.c_size_t),
        "wq_pack_symmetric": ([P, I, I64, I64, I, I, P, P, P, P], I),
        "wq_pack_codes": ([P, I64, I64, I, P, P], I),
        "wq_unpack": ([P, I, I64, I64, P, P], I),
        "wq_dequantize": ([P, P, I, I64, I64, I, P, P], I),
        "wq_import_packed_nk": ([P, P, I, I64, I64, I, P, P, P], I),
        "wq_gemm_w4a16": ([P, P, P, P, I64, I64, I64, I, P], I),
        "wq_gemm_w8a16": ([P, P, P, P, I64, I64, I64, I, P], I),
        "wq_mlp_w4a16": ([P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, P], I),
        "wq_mlp_w8a16": ([P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, P], I),
        "wq_swa_attention": ([P, P, P, P, I64, I64, I64, I64, I64, I64, P], I),
        "wq_last_device_error": ([], I),
        "wq_clear_device_error": ([], I),
        "wq_status_string": ([I], ctypes.c_char_p),
        "wq_debug_set_wait_limit_ns": ([ctypes.c_uint64], None),
        "wq_debug_force_timeout": ([I], None),
        "wq_gemm_regime": ([I, I64, I64, I64], I),
        "wq_debug_set_split": ([I], None),
        "wq_set_programmatic_launch": ([I], None),
        "wq_last_cuda_error": ([], ctypes.c_char_p),
        "wq_debug_force_regime": ([I], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


# ------------------------------------------------------------ raw C ABI ---
def wq_packed_words(bits: int, K: int, N: int) -> int:
    return int(_lib.wq_packed_words(bits, K, N))


def wq_packed_bytes(bits: int, K: int, N: int) -> int:
    return int(_lib.wq_packed_bytes(bits, K, N))


def wq_pack_symmetric(W, wdt, K, N, bits, group, scales_in, scales_out, packed,
                      stream) -> int:
    return _lib.wq_pack_symmetric(W, wdt, K, N, bits, group, scales_in,
                                  scales_out, packed, stream)


def wq_pack_codes(codes, K, N, bits, packed, stream) -> int:
    return _lib.wq_pack_codes(codes, K, N, bits, packed, stream)


def wq_unpack(packed, bits, K, N, codes, stream) -> int:
    return _lib.wq_unpack(packed, bits, K, N, codes, stream)


def wq_import_packed_nk(qweight, scales_nk, bits, K, N, group, packed, scales_out,
                        stream) -> int:
    return _lib.wq_import_packed_nk(qweight, scales_nk, bits, K, N, group, packed,
                                    scales_out, stream)


def wq_dequantize(packed, scales, bits, K, N, group, W, stream) -> int:
    return _lib.wq_dequantize(packed, scales, bits, K, N, group, W, stream)


def wq_gemm_w4a16(X, Wp, scales, Y, M, N, K, group, stream) -> int:
    return _lib.wq_gemm_w4a16(X, Wp, scales, Y, M, N, K, group, stream)


def wq_gemm_w8a16(X, Wp, scales, Y, M, N, K, group, stream) -> int:
    return _lib.wq_gemm_w8a16(X, Wp, scales, Y, M, N, K, group, stream)


def wq_last_device_error() -> int:
    return int(_lib.wq_last_device_error())


def wq_clear_device_error() -> int:
    return int(_lib.wq_clear_device_error())


def wq_last_cuda_error() -> str:
    return _lib.wq_last_cuda_error().decode()


def status_string(status: int) -> str:
    return _lib.wq_status_string(int(status)).decode()


def wq_debug_set_wait_limit_ns(ns: int) -> None:
    _lib.wq_debug_set_wait_limit_ns(int(ns))


def wq_debug_force_timeout(mode) -> None:
    """0 off, 1 a wait on a barrier nothing completes, 2 data waits that
    give up (see include/wq.h)."""
    _lib.wq_debug_force_timeout(int(mode))


def wq_gemm_regime(bits: int, M: int, N: int, K: int) -> int:
    return int(_lib.wq_gemm_regime(bits, M, N, K))


def wq_debug_set_split(cs: int) -> None:
    _lib.wq_debug_set_split(int(cs))


def wq_debug_force_regime(regime: int) -> None:
    """0 small-M kernel, 1 tensor-core kernel, -1 automatic."""
    _lib.wq_debug_force_regime(int(regime))


def wq_set_programmatic_launch(on: bool) -> None:
    _lib.wq_set_programmatic_launch(1 if on else 0)


# ---------------------------------------------------------- tensor layer ---
def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _check(status: int, what: str) -> None:
    if status != WQ_OK:
        raise WQError(status, what)


def pack_symmetric(W: torch.Tensor, bits: int, scales: torch.Tensor | None = None,
                   stream=None):
    """Round W [K,N] (fp32/bf16) onto the group-128 grid and pack it.
    Returns (packed int32 words, bf16 scales [K/128, N])."""
    K, N = W.shape
    wdt = {torch.float32: WQ_F32, torch.bfloat16: WQ_BF16}.get(W.dtype)
    if wdt is None:
        raise ValueError("W must be float32 or bfloat16")
    words = wq_packed_words(bits, K, N)
    if words == 0:
        raise WQError(WQ_ERR_SHAPE, "pack_symmetric")
    packed = torch.empty(words, dtype=torch.int32, device=W.device)
    s_out = torch.empty((K // GROUP, N), dtype=torch.bfloat16, device=W.device)
    _check(wq_pack_symmetric(_ptr(W), wdt, K, N, bits, GROUP, _ptr(scales),
                             _ptr(s_out), _ptr(packed), _stream(stream)),
           "wq_pack_symmetric")
    return packed, s_out


def pack_codes(codes: torch.Tensor, bits: int, stream=None) -> torch.Tensor:
    """Interleave int8 codes [K,N] into packed words."""
    K, N = codes.shape
    words = wq_packed_words(bits, K, N)
    if words == 0:
        raise WQError(WQ_ERR_SHAPE, "pack_codes")
    packed = torch.empty(words, dtype=torch.int32, device=codes.device)
    _check(wq_pack_codes(_ptr(codes), K, N, bits, _ptr(packed), _stream(stream)),
           "wq_pack_codes")
    return packed


def unpack(packed: torch.Tensor, K: int, N: int, bits: int,
           stream=None) -> torch.Tensor:
    codes = torch.empty((K, N), dtype=torch.int8, device=packed.device)
    _check(wq_unpack(_ptr(packed), bits, K, N, _ptr(codes), _stream(stream)),
           "wq_unpack")
    return codes


def import_packed_nk(qweight: torch.Tensor, scales_nk: torch.Tensor, bits: int,
                     stream=None):
    """Repack an output-channel-major checkpoint layer (qweight int32
    [N, K*bits/32], scales [N, K/128] bf16) into this library's layout:
    returns (packed words, scales [K/128, N])."""
    if scales_nk.dtype != torch.bfloat16:
        raise ValueError("scales must be bfloat16")
    N, G = scales_nk.shape
    K = G * GROUP
    packed = torch.empty((wq_packed_words(bits, K, N),), dtype=torch.int32,
                         device=qweight.device)
    scales = torch.empty((G, N), dtype=torch.bfloat16, device=qweight.device)
    _check(wq_import_packed_nk(_ptr(qweight), _ptr(scales_nk), bits, K, N, GROUP,
                               _ptr(packed), _ptr(scales), _stream(stream)),
           "wq_import_packed_nk")
    return packed, scales


def dequantize(packed: torch.Tensor, scales: torch.Tensor, bits: int,
               stream=None) -> torch.Tensor:
    """The effective bf16 weight [K, N] = bf16(s * q) of a packed layer."""
    if scales.dtype != torch.bfloat16:
        raise ValueError("scales must be bfloat16")
    K, N = scales.shape[0] * GROUP, scales.shape[1]
    W = torch.empty((K, N), dtype=torch.bfloat16, device=packed.device)
    _check(wq_dequantize(_ptr(packed), _ptr(scales), bits, K, N, GROUP, _ptr(W),
                         _stream(stream)), "wq_dequantize")
    return W


def _gemm(fn, name, X, Wp, scales, N, Y=None, stream=None):
    M, K = X.shape
    if X.dtype != torch.bfloat16 or scales.dtype != torch.bfloat16:
        raise ValueError("X and scales must be bfloat16")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _check(fn(_ptr(X), _ptr(Wp), _ptr(scales), _ptr(Y), M, N, K, GROUP,
              _stream(stream)), name)
    return Y


def gemm_w4a16(X: torch.Tensor, Wp: torch.Tensor, scales: torch.Tensor,
               N: int | None = None, Y: torch.Tensor | None = None, stream=None):
    """Y[M,N] = X[M,K] . dequant(Wp INT4, scales)."""
    N = scales.shape[1] if N is None else N
    return _gemm(wq_gemm_w4a16, "wq_gemm_w4a16", X, Wp, scales, N, Y, stream)


def gemm_w8a16(X: torch.Tensor, Wp: torch.Tensor, scales: torch.Tensor,
               N: int | None = None, Y: torch.Tensor | None = None, stream=None):
    """Y[M,N] = X[M,K] . dequant(Wp INT8, scales)."""
    N = scales.shape[1] if N is None else N
    return _gemm(wq_gemm_w8a16, "wq_gemm_w8a16", X, Wp, scales, N, Y, stream)


def wq_mlp_w4a16(X, Wu, Su, Wd, Sd, H, Y, M, K, N1, N2, group, act, stream) -> int:
    return _lib.wq_mlp_w4a16(X, Wu, Su, Wd, Sd, H, Y, M, K, N1, N2, group, act, stream)


def wq_mlp_w8a16(X, Wu, Su, Wd, Sd, H, Y, M, K, N1, N2, group, act, stream) -> int:
    return _lib.wq_mlp_w8a16(X, Wu, Su, Wd, Sd, H, Y, M, K, N1, N2, group, act, stream)


_ACTS = {"none": WQ_ACT_NONE, "silu": WQ_ACT_SILU}


def mlp(X: torch.Tensor, Wu: torch.Tensor, Su: torch.Tensor, Wd: torch.Tensor,
        Sd: torch.Tensor, bits: int, act: str = "none", H: torch.Tensor | None = None,
        Y: torch.Tensor | None = None, stream=None):
    """The two projections of an MLP block: H = act(bf16(X . Wu)),
    Y = bf16(H . Wd).  Returns (H, Y)."""
    M, K = X.shape
    N1, N2 = Su.shape[1], Sd.shape[1]
    if X.dtype != torch.bfloat16 or Su.dtype != torch.bfloat16 or Sd.dtype != torch.bfloat16:
        raise ValueError("X and scales must be bfloat16")
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(_ACTS)}")
    if H is None:
        H = torch.empty((M, N1), dtype=torch.bfloat16, device=X.device)
    if Y is None:
        Y = torch.empty((M, N2), dtype=torch.bfloat16, device=X.device)
    fn, name = (wq_mlp_w4a16, "wq_mlp_w4a16") if bits == 4 else (wq_mlp_w8a16, "wq_mlp_w8a16")
    _check(fn(_ptr(X), _ptr(Wu), _ptr(Su), _ptr(Wd), _ptr(Sd), _ptr(H), _ptr(Y), M, K, N1, N2,
              GROUP, _ACTS[act], _stream(stream)), name)
    return H, Y


def wq_swa_attention(Q, K, V, O, B, Hq, Hkv, D, T, window, stream) -> int:
    return _lib.wq_swa_attention(Q, K, V, O, B, Hq, Hkv, D, T, window, stream)


def swa_attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, window: int,
                  O: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The drafter's symmetric sliding-window attention.  Q [B, Hq, 128],
    K and V [Hkv, T, 128] (bf16); query b sits at position T - B + b and
    sees keys within window // 2 of it (window 0: all keys).  Returns
    O [B, Hq, 128]."""
    if Q.dtype != torch.bfloat16 or K.dtype != torch.bfloat16 or V.dtype != torch.bfloat16:
        raise ValueError("Q, K and V must be bfloat16")
    B, Hq, D = Q.shape
    Hkv, T, _ = K.shape
    if O is None:
        O = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=Q.device)
    _check(wq_swa_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), B, Hq, Hkv, D, T, window,
                            _stream(stream)), "wq_swa_attention")
    return O
