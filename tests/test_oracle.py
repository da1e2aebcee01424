"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: hand-derived
golden values, closed forms, brute force in plain Python, invariants of the
fixed grid, or an fp64 library matmul.  A plausible slip anywhere in the
oracle (a wrong nibble or byte position, a dropped scale, a transposed
operand, a wrong offset, round-half-up instead of half-even, a wrong clamp)
fails at least one of them; tests/test_oracle_mutants.py checks that claim
by compiling planted mistakes into the oracle.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


# ------------------------------------------------------------ P-h storage ---
def test_storage_accounting_matches_printed_sizes():
    """Packed bytes per weight (bits/8) plus one bf16 scale per 128-group
    reproduce the W8A16 card's 1.00 GB -> 521 MB within the fixture's bound."""
    kv = {k: float(v) for k, v in _rows("storage_accounting.txt")}
    K, N = 2560, 9728
    for bits in (4, 8):
        words = oracle.packed_words(bits, K, N)
        assert words * 4 == K * N * bits // 8
    per_weight_w8 = 1 + 2 / 128
    predicted = kv["params"] * per_weight_w8 / (kv["params"] * 2)
    printed = kv["w8a16_bytes_printed"] / kv["bf16_bytes_printed"]
    assert abs(predicted - printed) / printed < kv["ratio_tolerance"]
    # bf16 size of the parameters is the printed "1.00 GB" (GiB-ish units)
    assert abs(kv["params"] * 2 / 2**30 - 1.0) < 0.01


# -------------------------------------------------------- RTN scale pins ---
def test_rtn_scales_golden():
    for bits, amax, want in _rows("rtn_scales.txt"):
        bits, amax, want = int(bits), float(amax), int(want, 16)
        W = np.zeros((128, 64), dtype=np.float32)
        W[5, 3] = amax
        W[77, 3] = -amax / 2
        s = oracle.rtn_scales(W, bits)
        assert s[0, 3] == want, (bits, amax, hex(s[0, 3]))
        # columns with absmax 0 get scale 1.0
        assert s[0, 0] == 0x3F80


def test_rtn_negative_absmax_and_code_extremes():
    """absmax is taken over |w|: a group whose largest magnitude is negative
    gets the same scale, and RTN codes reach exactly -qpos .. qpos."""
    for bits, qpos in ((4, 7), (8, 127)):
        W = np.zeros((256, 64), dtype=np.float32)
        W[3, 0], W[9, 0] = -1.0, 0.25
        W[130, 1], W[200, 1] = 1.0, -0.5
        s = oracle.rtn_scales(W, bits)
        assert s[0, 0] == s[1, 1]
        q = oracle.quantize(W, s, bits)
        assert q[3, 0] == -qpos and q[130, 1] == qpos


# ---------------------------------------------------------- P-c rounding ---
def test_rounding_ties_and_clamp_golden():
    for bits, sb, w, want in _rows("rounding.txt"):
        bits, sb, w, want = int(bits), int(sb, 16), float(w), int(want)
        W = np.zeros((128, 64), dtype=np.float32)
        W[17, 9] = w
        s = np.full((1, 64), sb, dtype=np.uint16)
        q = oracle.quantize(W, s, bits)
        assert q[17, 9] == want, (bits, hex(sb), w, q[17, 9])


@pytest.mark.parametrize("bits", [4, 8])
def test_codes_stay_in_range(bits):
    rng = np.random.default_rng(7)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    for scale in (1e-30, 1e-3, 1.0, 1e3, 1e30):
        W = (rng.standard_normal((256, 128)) * scale).astype(np.float32)
        W[0, :] = np.float32(scale * 50)  # outliers
        packed, s, q = oracle.pack_symmetric(W, bits)
        assert q.min() >= lo and q.max() <= hi
        # RTN codes never use the extra negative code
        assert q.min() >= -hi
        # supplied (too small) scales clamp
        s_small = np.full_like(s, 0x0080)  # smallest normal bf16
        q2 = oracle.quantize(W, s_small, bits)
        assert q2.min() >= lo and q2.max() <= hi


# ------------------------------------------------------- P-a round trip ---
@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_round_trip(bits):
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    rng = np.random.default_rng(bits)
    for K, N in ((128, 64), (256, 192), (384, 128)):
        q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
        p = oracle.pack(q, bits)
        assert p.size * 32 == K * N * bits
        assert np.array_equal(oracle.unpack(p, K, N, bits), q)


@pytest.mark.parametrize("bits", [4, 8])
def test_every_value_at_every_position(bits):
    """Brute force: every code value at every slot position survives."""
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    K, N = 128, 64
    idx = np.arange(K * N).reshape(K, N)
    for v in range(hi - lo + 1):
        q = (((idx + v) % (hi - lo + 1)) + lo).astype(np.int8)
        assert np.array_equal(oracle.unpack(oracle.pack(q, bits), K, N, bits), q)


@pytest.mark.parametrize("bits", [4, 8])
def test_layout_is_a_bijection(bits):
    """Read every field of every packed word directly (no layout formula):
    the element indices stored there, written in base-16 (or base-256)
    digit planes, must be a permutation of all elements."""
    K, N = 256, 128
    width = bits
    mask = (1 << width) - 1
    off = 8 if bits == 4 else 128
    idx = np.arange(K * N, dtype=np.int64).reshape(K, N)
    nplanes = int(np.ceil(np.log2(K * N) / width))
    recovered = None
    fields = 32 // width
    for p in range(nplanes):
        digit = (idx >> (width * p)) & mask
        packed = oracle.pack((digit - off).astype(np.int8), bits)
        vals = np.stack([(packed >> (width * f)) & mask for f in range(fields)],
                        axis=1).astype(np.int64).ravel()
        recovered = vals << (width * p) if recovered is None else \
            recovered | (vals << (width * p))
    assert np.array_equal(np.sort(recovered), np.arange(K * N))


def test_layout_positions_golden():
    for bits, K, N, k, n, w, sh in _rows("layout_positions.txt"):
        bits, K, N, k, n, w, sh = map(int, (bits, K, N, k, n, w, sh))
        lo = -8 if bits == 4 else -128
        q = np.full((K, N), lo, dtype=np.int8)  # stored field value 0
        q[k, n] = lo + 1                          # stored field value 1
        p = oracle.pack(q, bits)
        nz = np.flatnonzero(p)
        assert list(nz) == [w], (bits, k, n, nz[:4])
        assert int(p[w]) == 1 << sh, (bits, k, n, hex(int(p[w])))


# --------------------------------------------------- P-b grid idempotence ---
@pytest.mark.parametrize("bits", [4, 8])
def test_fixed_grid_idempotence(bits):
    """s*q is exact in fp32, so re-rounding it with the same s returns q."""
    rng = np.random.default_rng(11)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    K, N = 512, 128
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    # random bf16 scales over many binades, including subnormal-free tiny ones
    sf = np.exp(rng.uniform(np.log(1e-6), np.log(1e3), size=(K // 128, N)))
    s = oracle.f32_to_bf16_bits(sf.astype(np.float32))
    sv = oracle.bf16_bits_to_f32(s).astype(np.float64)
    W64 = np.repeat(sv, 128, axis=0) * q.astype(np.float64)
    W = W64.astype(np.float32)
    assert np.array_equal(W.astype(np.float64), W64)  # exactness of s*q
    packed, s_out, q_out = oracle.pack_symmetric(W, bits, scales_in=s)
    assert np.array_equal(q_out, q)
    assert np.array_equal(s_out, s)
    assert np.array_equal(oracle.unpack(packed, K, N, bits), q)
    # and re-packing the dequantized weights is a fixed point
    W2 = oracle.dequant(q_out, s_out)
    assert np.array_equal(W2, W)


# ----------------------------------------------------------- P-g s = 1 ---
def test_unit_scale_dequant_is_the_codes():
    K, N = 256, 64
    q = np.empty((K, N), dtype=np.int8)
    for k in range(K):          # hand enumeration of all codes
        for n in range(N):
            q[k, n] = ((k * 7 + n * 3) % 16) - 8
    s = np.full((K // 128, N), 0x3F80, dtype=np.uint16)
    W = oracle.dequant(q, s)
    assert np.array_equal(W, q.astype(np.float32))


# ------------------------------------------------------ P-d identity probe ---
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K", [128, 256])
def test_identity_probe_recovers_weights(bits, K):
    """Running the identity through the quantized product gives back the
    effective dense weight (the identity-probe of the W8A16 card's fused-KV
    patch, site 2)."""
    X, q, s = synth.small_case(K, K, 64, bits, seed=K + bits)
    eye = np.zeros((K, K), dtype=np.float32)
    np.fill_diagonal(eye, 1.0)
    X = oracle.f32_to_bf16_bits(eye)
    packed = oracle.pack(q, bits)
    Y = oracle.gemm(X, packed, s, K, 64, bits)
    sv = oracle.bf16_bits_to_f32(s).astype(np.float64)
    expect = np.repeat(sv, 128, axis=0) * q.astype(np.float64)
    assert np.array_equal(Y, expect)


# --------------------------------------------- P-e exact integer brute force ---
@pytest.mark.parametrize("bits", [4, 8])
def test_exact_bruteforce_power_of_two_scales(bits):
    """Tiny shape, powers-of-two scales, small integer activations: compare
    the oracle with a pure-Python exact-rational triple loop."""
    rng = np.random.default_rng(3 + bits)
    M, K, N = 3, 256, 64
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    e = rng.integers(-6, 3, size=(K // 128, N))
    s = oracle.f32_to_bf16_bits((2.0 ** e).astype(np.float32))
    Xi = rng.integers(-4, 5, size=(M, K))
    X = oracle.f32_to_bf16_bits(Xi.astype(np.float32))
    Y = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(int(Xi[m, k])) * Fraction(2) ** int(e[k // 128, n]) \
                    * int(q[k, n])
            assert Fraction(Y[m, n]) == acc, (m, n)


def test_scale_row_selection_bruteforce():
    """Distinct scale per group and per column: a wrong group index or a
    transposed scale tensor is caught."""
    M, K, N = 2, 384, 64
    q = np.ones((K, N), dtype=np.int8)
    e = np.arange(K // 128)[:, None] * 2 + (np.arange(N)[None, :] % 5)
    s = oracle.f32_to_bf16_bits((2.0 ** e).astype(np.float32))
    X = oracle.f32_to_bf16_bits(np.ones((M, K), dtype=np.float32))
    Y = oracle.gemm(X, oracle.pack(q, 4), s, K, N, 4)
    for n in range(N):
        want = sum(128 * 2.0 ** int(e[g, n]) for g in range(K // 128))
        assert Y[0, n] == want and Y[1, n] == want


# -------------------------------------------------- P-f on-grid agreement ---
@pytest.mark.parametrize("bits", [4, 8])
def test_on_grid_weights_match_fp64_matmul(bits):
    """Weights already on the grid: quantization is lossless, so the oracle
    equals an fp64 library matmul of X and W (up to fp64 summation order)."""
    X, q, s = synth.small_case(5, 384, 192, bits, seed=21)
    sv = oracle.bf16_bits_to_f32(s).astype(np.float64)
    W = (np.repeat(sv, 128, axis=0) * q).astype(np.float32)
    packed, s2, q2 = oracle.pack_symmetric(W, bits, scales_in=s)
    Y = oracle.gemm(X, packed, s2, 384, 192, bits)
    Xf = oracle.bf16_bits_to_f32(X).astype(np.float64)
    ref = Xf @ W.astype(np.float64)
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_row_subset_and_threads_agree():
    X, q, s = synth.small_case(9, 256, 128, 4, seed=5)
    p = oracle.pack(q, 4)
    full = oracle.gemm(X, p, s, 256, 128, 4, nthreads=1)
    sub = oracle.gemm(X, p, s, 256, 128, 4, rows=[8, 0, 3], nthreads=3)
    assert np.array_equal(sub, full[[8, 0, 3]])
    assert oracle.gemm(X, p, s, 256, 128, 4, rows=[]).shape == (0, 128)


def test_bf16_rounding_helpers():
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3e38, 1e-40],
                    dtype=np.float32)
    # 1.00390625 = 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0);
    # 1.01171875 = 1 + 3*2^-8 is a tie between 1+2^-7 and 1+2^-6 -> 1+2^-6
    want = np.array([0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F62, 0x0001],
                    dtype=np.uint16)
    got = oracle.f32_to_bf16_bits(vals)
    assert np.array_equal(got, want), [hex(int(x)) for x in got]
    assert np.array_equal(oracle.bf16_bits_to_f32(want[:4]),
                          np.array([1.0, 1.0, 1.015625, -2.5], np.float32))


def test_shape_checks():
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((100, 64), np.int8), 4)
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((128, 48), np.int8), 4)
    with pytest.raises(ValueError):
        oracle.rtn_scales(np.zeros((128, 64), np.float32), 4, group=64)


# ----------------------------------------------------- checkpoint import ---
def _encode_nk(q, bits):
    """Test-side writer of the output-channel-major format: word j of row n
    holds codes k = per*j .. per*j + per - 1, offset-binary, first in the
    low bits."""
    K, N = q.shape
    per, off = 32 // bits, (8 if bits == 4 else 128)
    u = (q.astype(np.int64) + off).T.reshape(N, K // per, per)
    shifts = (bits * np.arange(per, dtype=np.int64))[None, None, :]
    return np.ascontiguousarray((u << shifts).sum(axis=2).astype(np.uint32))


def test_import_nk_reads_hand_made_words():
    """Values fixed by the format definition: consecutive codes in rising
    nibble (byte) positions, offset 8 (128)."""
    qw = np.full((64, 16), 0x88888888, dtype=np.uint32)
    qw[0, 0], qw[0, 1], qw[5, 15] = 0x76543210, 0xFEDCBA98, 0x0000000F
    s_nk = np.arange(64, dtype=np.uint16).reshape(64, 1) + 0x3F00
    q, s = oracle.import_packed_nk(qw, s_nk, 128, 64, 4)
    assert q[:16, 0].tolist() == list(range(-8, 8))
    assert q[120:128, 5].tolist() == [7] + [-8] * 7
    assert np.all(q[:, 1:5] == 0) and np.all(q[16:, 0] == 0)
    assert np.array_equal(s, s_nk.T)
    qw8 = np.full((64, 32), 0x80808080, dtype=np.uint32)
    qw8[3, 0], qw8[3, 31] = 0x83828180, 0x00FF7F01
    q8, _ = oracle.import_packed_nk(qw8, s_nk, 128, 64, 8)
    assert q8[0:4, 3].tolist() == [0, 1, 2, 3]
    assert q8[124:128, 3].tolist() == [-127, -1, 127, -128]


@pytest.mark.parametrize("bits", [4, 8])
def test_import_nk_round_trip(bits):
    rng = np.random.default_rng(51 + bits)
    K, N = 384, 128
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    s = rng.integers(0x3C00, 0x3F80, size=(K // 128, N)).astype(np.uint16)
    got_q, got_s = oracle.import_packed_nk(_encode_nk(q, bits), np.ascontiguousarray(s.T), K, N,
                                           bits)
    assert np.array_equal(got_q, q)
    assert np.array_equal(got_s, s)


# ------------------------------------------------------------- MLP pair ---
def _bits(x: float) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0] >> 16)


def test_round_bf16_f64_ties_and_ranges():
    """Direct fp64 -> bf16 rounding: ties go to the even neighbour, a value
    just past a tie rounds away (an fp32 step would make it a tie), the
    subnormal grid is 2^-133, and past the largest bf16 lies infinity."""
    cases = [
        (1.0 + 2.0 ** -8, 0x3F80),                  # tie -> even (1.0)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),              # tie -> even (1 + 2^-6)
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),     # just past the tie
        (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -140, 0x0000),                      # below half the subnormal step
        (1.5 * 2.0 ** -133, 0x0002),                # subnormal tie -> even
        (2.0 ** 130, 0x7F80),                       # overflow
        (3.0, 0x4040),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float64)
    got = oracle.round_bf16_f64(x)
    assert [int(v) for v in got] == [c[1] for c in cases]


def test_silu_closed_form_values():
    """silu(h) = h * sigma(h): silu(0) = 0, silu(1) = e / (1 + e),
    silu(-1) = -1 / (1 + e), silu(h) -> h for large h and -> -0 for very
    negative h."""
    e = 2.718281828459045
    h = np.array([_bits(v) for v in (0.0, 1.0, -1.0, 30.0, -200.0, 2.0)], dtype=np.uint16)
    got = oracle.silu_bf16(h)
    want = oracle.round_bf16_f64(np.array([0.0, e / (1 + e), -1 / (1 + e), 30.0, -0.0,
                                           2 * e * e / (1 + e * e)]))
    assert [int(v) for v in got] == [int(v) for v in want]
    assert int(got[1]) == 0x3F3B and int(got[2]) == 0xBE8A  # 0.73046875, -0.26953125


def test_silu_minimum_and_odd_part():
    """Over every bf16 value in [-16, 16]: silu never goes below its global
    minimum (-0.2784645...), and silu(h) - silu(-h) = h up to the two
    roundings."""
    grid = np.arange(0x0000, 0x4180, dtype=np.uint32)        # 0 .. 16
    pos = grid.astype(np.uint16)
    neg = (grid | 0x8000).astype(np.uint16)
    sp = oracle.bf16_bits_to_f32(oracle.silu_bf16(pos)).astype(np.float64)
    sn = oracle.bf16_bits_to_f32(oracle.silu_bf16(neg)).astype(np.float64)
    h = oracle.bf16_bits_to_f32(pos).astype(np.float64)
    assert sn.min() >= -0.2784645428 * (1 + 2.0 ** -7)
    ulp = np.maximum(np.abs(sp), np.abs(h)) * 2.0 ** -7 + 2.0 ** -133
    assert np.all(np.abs((sp - sn) - h) <= ulp)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_mlp_one_hot_rows_bruteforce(bits, act):
    """One-hot rows of X pick rows of the up-projection's weight: H row k =
    act(bf16(s q)[k, :]), and Y = H . dequant(Wd) by a plain fp64 matmul."""
    K, N1, N2 = 256, 128, 64
    rng = np.random.default_rng(70 + bits)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    qu = rng.integers(lo, hi + 1, size=(K, N1)).astype(np.int8)
    qd = rng.integers(lo, hi + 1, size=(N1, N2)).astype(np.int8)
    su = oracle.f32_to_bf16_bits(rng.uniform(0.01, 0.05, size=(K // 128, N1)).astype(np.float32))
    sd = oracle.f32_to_bf16_bits(rng.uniform(0.01, 0.05, size=(N1 // 128, N2)).astype(np.float32))
    ks = np.array([0, 5, 127, 128, 255])
    X = np.zeros((ks.size, K), dtype=np.float32)
    X[np.arange(ks.size), ks] = 1.0
    H, Y = oracle.mlp(oracle.f32_to_bf16_bits(X), oracle.pack(qu, bits), su,
                      oracle.pack(qd, bits), sd, K, N1, N2, bits, act=act)
    wu = oracle.dequant(qu, su)            # exact fp32 s * q
    Hk = oracle.f32_to_bf16_bits(wu[ks])   # one rounding of the exact s * q
    if act == "silu":
        Hk = oracle.silu_bf16(Hk)
    assert np.array_equal(H, Hk)
    Yk = oracle.bf16_bits_to_f32(Hk).astype(np.float64) @ oracle.dequant(qd, sd).astype(np.float64)
    assert np.allclose(Y, Yk, rtol=1e-12, atol=1e-12)


# ------------------------------------------------ drafter attention (SWA) ---
def _bf16(a) -> np.ndarray:
    return oracle.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


@pytest.mark.parametrize("T,W,B", [(200, 64, 16), (200, 2, 4), (100, 128, 16), (200, 0, 16),
                                   (40, 38, 16), (17, 16, 16)])
def test_swa_window_bounds_by_uniform_scores(T, W, B):
    """Equal keys make every visible score equal, so the output is the mean
    of the visible values; with value j at key j that mean is
    (lo + hi) / 2, lo = max(0, p - W/2), hi = min(T - 1, p + W/2), p = T - B
    + b, and the whole sequence when W = 0 or T <= W."""
    Hq, Hkv, D = 2, 1, 128
    rng = np.random.default_rng(T + W)
    Q = _bf16(rng.normal(size=(B, Hq, D)))
    K = _bf16(np.broadcast_to(rng.normal(size=(1, 1, D)), (Hkv, T, D)))
    V = _bf16(np.broadcast_to(np.arange(T, dtype=np.float32)[None, :, None], (Hkv, T, D)))
    O = oracle.swa_attention(Q, K, V, T, W)
    for b in range(B):
        p = T - B + b
        if W == 0 or T <= W:
            lo, hi = 0, T - 1
        else:
            lo, hi = max(0, p - W // 2), min(T - 1, p + W // 2)
        assert np.allclose(O[b], (lo + hi) / 2, rtol=0, atol=1e-9), (b, lo, hi)


def test_swa_grouped_heads_read_their_kv_head():
    """Query head h reads key/value head h / (Hq / Hkv): with a constant
    value per key/value head the output names the head."""
    B, Hq, Hkv, D, T = 16, 8, 2, 128, 64
    rng = np.random.default_rng(3)
    Q = _bf16(rng.normal(size=(B, Hq, D)))
    K = _bf16(rng.normal(size=(Hkv, T, D)))
    V = _bf16(np.broadcast_to((np.arange(Hkv, dtype=np.float32) + 1)[:, None, None], (Hkv, T, D)))
    O = oracle.swa_attention(Q, K, V, T, 32)
    for h in range(Hq):
        assert np.allclose(O[:, h, :], h // (Hq // Hkv) + 1, rtol=0, atol=1e-12)


def test_swa_single_peak_closed_form():
    """One key aligned with the query: its weight is e^s / (e^s + n - 1)
    with s = |q|^2 / sqrt(D) and every other visible key scoring 0 (keys
    orthogonal to q); a key outside the window gets no weight at all."""
    B, Hq, Hkv, D, T, W = 16, 1, 1, 128, 300, 100
    Q = np.zeros((B, Hq, D), dtype=np.float32)
    Q[:, :, 0] = 2.0
    K = np.zeros((Hkv, T, D), dtype=np.float32)
    K[:, :, 1] = 1.0                                   # orthogonal to q: score 0
    jstar = T - B - 10                                 # visible to queries b with p - 50 <= jstar
    K[0, jstar, 0] = 3.0
    K[0, 0, 0] = 3.0                                   # outside every window
    V = np.zeros((Hkv, T, D), dtype=np.float32)
    V[0, jstar, :] = 1.0
    V[0, 0, :] = -7.0
    O = oracle.swa_attention(_bf16(Q), _bf16(K), _bf16(V), T, W)
    s = 6.0 / np.sqrt(D)
    for b in range(B):
        p = T - B + b
        lo, hi = max(0, p - W // 2), min(T - 1, p + W // 2)
        n = hi - lo + 1
        want = np.exp(s) / (np.exp(s) + n - 1) if lo <= jstar <= hi else 0.0
        assert np.allclose(O[b, 0, :], want, rtol=1e-12, atol=1e-15), b


def test_swa_output_is_a_convex_combination_and_permutation_invariant():
    """The output lies between the smallest and largest visible value, and
    does not change when the visible keys and values are permuted together."""
    B, Hq, Hkv, D, T, W = 16, 4, 2, 128, 96, 0
    rng = np.random.default_rng(9)
    Q = _bf16(rng.normal(size=(B, Hq, D)))
    K = _bf16(rng.normal(size=(Hkv, T, D)))
    V = _bf16(rng.normal(size=(Hkv, T, D)))
    O = oracle.swa_attention(Q, K, V, T, W)
    Vf = oracle.bf16_bits_to_f32(V).astype(np.float64)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        assert np.all(O[:, h, :] <= Vf[kv].max(axis=0) + 1e-12)
        assert np.all(O[:, h, :] >= Vf[kv].min(axis=0) - 1e-12)
    perm = rng.permutation(T)
    O2 = oracle.swa_attention(Q, K[:, perm], V[:, perm], T, W)
    assert np.allclose(O, O2, rtol=1e-12, atol=1e-12)
