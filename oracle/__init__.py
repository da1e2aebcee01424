"""CPU oracle for the group-wise symmetric weight-only quantized GEMM.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The product path (the CUDA library and its binding) never imports
this package, and this package never imports the product.

The arithmetic lives in ``wq_oracle.c`` (plain C, fp32 quantization with IEEE
divide and round-half-even, exact fp32 dequant, fp64 GEMM); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Sources of each step:
  * "Quantize the Target, Quantize the Drafter" (arXiv 2607.04244): QAD
    paragraph (dequantized weights s (.) Wq, frozen symmetric per-group
    scales), packing paragraph (round back onto the same grid), drafter-PTQ
    paragraph (group-wise symmetric INT4, group size 128).
  * "Qwen3.5-4B-DFlash-W8A16" card, "What changed vs upstream" table (int8
    RTN symmetric, group 128).

Every function here is pinned by tests/test_oracle.py against closed forms,
brute force and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libwq_oracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 128


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, IEEE-strict flags) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.wqo_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.wqo_f32_to_bf16.restype = ctypes.c_uint16
    lib.wqo_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.wqo_bf16_to_f32.restype = ctypes.c_float
    lib.wqo_rtn_scales.argtypes = [P, I64, I64, I, I, P]
    lib.wqo_quantize.argtypes = [P, P, I64, I64, I, I, P]
    lib.wqo_widen_bf16.argtypes = [P, I64, P]
    lib.wqo_round_bf16.argtypes = [P, I64, P]
    lib.wqo_round_bf16_f64.argtypes = [P, I64, P]
    lib.wqo_silu_bf16.argtypes = [P, I64, P]
    lib.wqo_swa_attention.argtypes = [P, P, P, I, I, I, I, I64, I64, P]
    lib.wqo_packed_words.argtypes = [I, I64, I64]
    lib.wqo_packed_words.restype = I64
    lib.wqo_pack.argtypes = [P, I64, I64, I, P]
    lib.wqo_unpack.argtypes = [P, I64, I64, I, P]
    lib.wqo_dequant.argtypes = [P, P, I64, I64, I, P]
    lib.wqo_import_nk.argtypes = [P, P, I64, I64, I, I, P, P]
    lib.wqo_gemm_rows.argtypes = [P, P, P, P, I64, I64, I64, I, I, I, P]
    lib.wqo_gemm_rows.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used only by the
    mutation tests, which plant mistakes to show the pins catch them)."""
    c_path = out_path[:-3] + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off",
                    "-fno-fast-math", "-fPIC", "-shared", "-pthread", c_path,
                    "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _check_shape(K: int, N: int, group: int):
    if group != GROUP:
        raise ValueError("group size must be 128")
    if K % 128 or N % 64 or K <= 0 or N <= 0:
        raise ValueError("need K % 128 == 0 and N % 64 == 0")


# ------------------------------------------------------------------ bf16 ---
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (in C)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().wqo_round_bf16(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().wqo_widen_bf16(_ptr(h), h.size, _ptr(out))
    return out


# --------------------------------------------------------- quantization ---
def rtn_scales(W: np.ndarray, bits: int, group: int = GROUP) -> np.ndarray:
    """Per-(group, column) RTN scales, bf16 bits [K/group, N]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    K, N = W.shape
    _check_shape(K, N, group)
    s = np.empty((K // group, N), dtype=np.uint16)
    _load().wqo_rtn_scales(_ptr(W), K, N, group, bits, _ptr(s))
    return s


def quantize(W: np.ndarray, s: np.ndarray, bits: int,
             group: int = GROUP) -> np.ndarray:
    """Codes q = clamp(rint(W / s), qmin, qmax) as int8 [K, N]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    K, N = W.shape
    _check_shape(K, N, group)
    q = np.empty((K, N), dtype=np.int8)
    _load().wqo_quantize(_ptr(W), _ptr(s), K, N, group, bits, _ptr(q))
    return q


def packed_words(bits: int, K: int, N: int) -> int:
    return int(_load().wqo_packed_words(bits, K, N))


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    """Interleave int8 codes [K, N] into the packed uint32 word layout."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    K, N = q.shape
    _check_shape(K, N, GROUP)
    out = np.empty(packed_words(bits, K, N), dtype=np.uint32)
    _load().wqo_pack(_ptr(q), K, N, bits, _ptr(out))
    return out


def unpack(packed: np.ndarray, K: int, N: int, bits: int) -> np.ndarray:
    """Inverse of :func:`pack`: canonical int8 codes [K, N]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    _check_shape(K, N, GROUP)
    if packed.size != packed_words(bits, K, N):
        raise ValueError("packed buffer has the wrong size")
    q = np.empty((K, N), dtype=np.int8)
    _load().wqo_unpack(_ptr(packed), K, N, bits, _ptr(q))
    return q


def pack_symmetric(W: np.ndarray, bits: int, scales_in: np.ndarray | None = None,
                   group: int = GROUP):
    """The pack step: (scales or RTN scales) -> codes -> packed words.

    W is fp32 [K, N] (bf16 weights: pass ``bf16_bits_to_f32(Wh)``).
    Returns (packed uint32, scales bf16 bits [K/group, N], codes int8).
    """
    W = np.ascontiguousarray(W, dtype=np.float32)
    s = rtn_scales(W, bits, group) if scales_in is None else \
        np.ascontiguousarray(scales_in, dtype=np.uint16)
    q = quantize(W, s, bits, group)
    return pack(q, bits), s, q


def import_packed_nk(qweight: np.ndarray, s_nk: np.ndarray, K: int, N: int, bits: int,
                     group: int = GROUP):
    """Codes q [K, N] and scales s [K/group, N] of a layer stored output-
    channel-major with codes packed along K (qweight uint32 [N, K*bits/32],
    offset-binary, first code in the low bits; s_nk bf16 [N, K/group])."""
    _check_shape(K, N, group)
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    s_nk = np.ascontiguousarray(s_nk, dtype=np.uint16)
    assert qweight.size == N * K * bits // 32 and s_nk.size == N * (K // group)
    q = np.empty((K, N), dtype=np.int8)
    s = np.empty((K // group, N), dtype=np.uint16)
    _load().wqo_import_nk(_ptr(qweight), _ptr(s_nk), K, N, group, bits, _ptr(q), _ptr(s))
    return q, s


def dequant(q: np.ndarray, s: np.ndarray, group: int = GROUP) -> np.ndarray:
    """w^ = s * q in fp32 (exact), [K, N]."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    K, N = q.shape
    out = np.empty((K, N), dtype=np.float32)
    _load().wqo_dequant(_ptr(q), _ptr(s), K, N, group, _ptr(out))
    return out


# ------------------------------------------------------------------ GEMM ---
def gemm(X_bf16: np.ndarray, packed: np.ndarray, s: np.ndarray, K: int, N: int,
         bits: int, rows=None, group: int = GROUP,
         nthreads: int | None = None) -> np.ndarray:
    """Y_ref = X . dequant(unpack(packed)) with fp64 accumulation.

    X_bf16: uint16 bf16 bits [M, K].  ``rows`` selects output rows (default
    all).  Returns fp64 [len(rows), N].
    """
    X_bf16 = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    M = X_bf16.shape[0]
    assert X_bf16.shape[1] == K
    _check_shape(K, N, group)
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise ValueError("row index out of range")
    Y = np.zeros((rows.size, N), dtype=np.float64)
    if rows.size == 0:
        return Y
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().wqo_gemm_rows(_ptr(X_bf16), _ptr(packed), _ptr(s), _ptr(rows),
                               rows.size, N, K, group, bits, int(nthreads),
                               _ptr(Y))
    if rc != 0:
        raise MemoryError("oracle GEMM could not allocate its dequant buffer")
    return Y


def round_bf16_f64(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16), round to nearest even, directly."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().wqo_round_bf16_f64(_ptr(x), x.size, _ptr(out))
    return out


def silu_bf16(h_bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> bf16 bits of silu(h) = h / (1 + e^-h) (fp64, then RNE)."""
    h = np.ascontiguousarray(h_bits, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.uint16)
    _load().wqo_silu_bf16(_ptr(h), h.size, _ptr(out))
    return out


def mlp(X_bf16: np.ndarray, packed_up: np.ndarray, s_up: np.ndarray, packed_down: np.ndarray,
        s_down: np.ndarray, K: int, N1: int, N2: int, bits: int, act: str = "none",
        rows=None, nthreads=None):
    """The MLP pair: H = act(bf16(X . Wu)) as bf16 bits [M, N1] and
    Y_ref = H . Wd in fp64 ([len(rows), N2]).  act is "none" or "silu"."""
    if act not in ("none", "silu"):
        raise ValueError("act must be 'none' or 'silu'")
    H = round_bf16_f64(gemm(X_bf16, packed_up, s_up, K, N1, bits, nthreads=nthreads))
    if act == "silu":
        H = silu_bf16(H)
    return H, gemm(H, packed_down, s_down, N1, N2, bits, rows=rows, nthreads=nthreads)


def swa_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, T: int, window: int) -> np.ndarray:
    """The drafter's symmetric sliding-window attention, fp64 [B, Hq, D].

    Q bf16 bits [B, Hq, D]; K, V bf16 bits [Hkv, T, D].  Query b sits at
    position T - B + b and sees keys j with |j - (T - B + b)| <= window / 2;
    window 0 or T <= window is full attention."""
    Q = np.ascontiguousarray(Q, dtype=np.uint16)
    K = np.ascontiguousarray(K, dtype=np.uint16)
    V = np.ascontiguousarray(V, dtype=np.uint16)
    B, Hq, D = Q.shape
    Hkv = K.shape[0]
    if K.shape != (Hkv, T, D) or V.shape != (Hkv, T, D) or Hq % Hkv != 0 or B > T:
        raise ValueError("shape mismatch")
    O = np.zeros((B, Hq, D), dtype=np.float64)
    _load().wqo_swa_attention(_ptr(Q), _ptr(K), _ptr(V), B, Hq, Hkv, D, T, window, _ptr(O))
    return O


def tolerance(Y_ref: np.ndarray) -> float:
    """Allowed max |Y_gpu - Y_ref|: 1e-2 * max|Y_ref| + 1e-3 (bf16 output,
    fp32 accumulation)."""
    peak = float(np.max(np.abs(Y_ref))) if Y_ref.size else 0.0
    return 1e-2 * peak + 1e-3
