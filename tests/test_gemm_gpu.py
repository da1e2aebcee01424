"""GPU GEMM against the oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from tests import synth
from tests.gpu_util import (assert_close_to_oracle, bf16_to_dev,
                            bf16_to_host_bits, f32_to_dev, i8_to_dev,
                            words_to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wq():
    import __graft_entry__
    __graft_entry__.build()
    import w4a16_weight_only_wq_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    return m


def _gemm(wq, bits, Xt, Wp, st, N=None, Y=None):
    fn = wq.gemm_w4a16 if bits == 4 else wq.gemm_w8a16
    return fn(Xt, Wp, st, N=N, Y=Y)


def _run_codes_case(wq, X, q, s, bits, rows=None):
    K, N = q.shape
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(X), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    p_ref = oracle.pack(q, bits)
    assert np.array_equal(words_to_host(Wp), p_ref)
    Yref = oracle.gemm(X, p_ref, s, K, N, bits, rows=rows)
    Ysel = Y if rows is None else Y[torch.as_tensor(rows, device=Y.device)]
    return assert_close_to_oracle(Ysel, Yref, f"W{bits} M={X.shape[0]} K={K} N={N}")


@pytest.fixture(params=[0, 2, 4], ids=["warpmma", "tmem", "stream"])
def small_kernel(wq, request):
    """Run the test on each small-M kernel: 0 the warp-MMA kernel, 2 the
    tensor-memory kernel, 4 the tensor-memory kernel whose launches overlap
    (the default for M <= 32)."""
    wq.wq_debug_force_regime(request.param)
    yield request.param
    wq.wq_debug_force_regime(-1)


# ------------------------------------------------ small shapes, many tiles ---
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 5, 16, 17, 40])
@pytest.mark.parametrize("K,N", [(128, 64), (640, 192), (1280, 576), (3840, 128)])
def test_small_shapes(wq, small_kernel, bits, M, K, N):
    # the tensor-memory kernel takes whole two-group chunks only
    want = small_kernel if small_kernel != 2 or (K // 128) % 2 == 0 else 0
    assert wq.wq_gemm_regime(bits, M, N, K) == want
    X, q, s = synth.small_case(M, K, N, bits, seed=M * 7 + K + N + bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_small_m_long_k_falls_back_to_tiled(wq, bits):
    """K = 128000 with one column tile: X of a CTA's K range does not fit
    the small-M kernel's shared memory, so the tiled kernel runs it."""
    M, K, N = 16, 128 * 1000, 64
    assert wq.wq_gemm_regime(bits, M, N, K) == 1
    X, q, s = synth.small_case(M, K, N, bits, seed=91 + bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.fixture
def skinny_regime(wq):
    wq.wq_debug_force_regime(2)
    yield
    wq.wq_debug_force_regime(-1)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 7, 16, 24])
@pytest.mark.parametrize("K,N", [(256, 64), (512, 192), (1280, 576), (3840, 128),
                                 (9728, 2560)])
def test_tmem_small_m_shapes(wq, skinny_regime, bits, M, K, N):
    """The tensor-memory small-M kernel on ragged tiles, every split the
    occupancy rule picks, and M > 16 in 16-row slices."""
    assert wq.wq_gemm_regime(bits, M, N, K) == 2
    X, q, s = synth.small_case(M, K, N, bits, seed=M * 3 + K + N + bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_tmem_small_m_every_split(wq, skinny_regime, bits):
    M, K, N = 11, 2048, 320   # 8 chunks, 3 column tiles (the last one half)
    X, q, s = synth.small_case(M, K, N, bits, seed=66)
    try:
        for cs in range(1, 9):
            wq.wq_debug_set_split(cs)
            _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)


def test_default_kernel_choice(wq):
    for M, want in [(1, 4), (16, 4), (32, 4), (33, 4), (64, 4), (65, 3), (384, 3), (8192, 3)]:
        assert wq.wq_gemm_regime(4, M, 2560, 2560) == want


# --------------------------------------------------------- exact cases ---
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K", [128, 256])
def test_identity_probe_bit_exact(wq, small_kernel, bits, K):
    """X = I recovers bf16(s * q) exactly (identity probe of the W8A16
    card's fused-KV patch)."""
    N = 128
    _, q, s = synth.small_case(1, K, N, bits, seed=K + bits)
    eye = oracle.f32_to_bf16_bits(np.eye(K, dtype=np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(eye), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(eye, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(bf16_to_host_bits(Y), want)


@pytest.mark.parametrize("bits", [4, 8])
def test_integer_exact_bruteforce_bit_exact(wq, small_kernel, bits):
    """Powers-of-two scales and small integer X: every partial sum is exact,
    so the GPU result must be the oracle's value rounded once to bf16."""
    M, K, N = 16, 1024, 256
    rng = np.random.default_rng(17 + bits)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    s = oracle.f32_to_bf16_bits(
        (2.0 ** rng.integers(-8, -2, size=(K // 128, N))).astype(np.float32))
    X = oracle.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(X), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(Yref.astype(np.float32).astype(np.float64), Yref)
    assert np.array_equal(bf16_to_host_bits(Y), want)


# ------------------------------------------------------ edge behaviours ---
def test_m_zero_is_a_noop(wq):
    K, N = 256, 128
    _, q, s = synth.small_case(1, K, N, 4, seed=3)
    Wp = wq.pack_codes(i8_to_dev(q), 4)
    X = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    assert wq.wq_gemm_w4a16(X.data_ptr() or None, Wp.data_ptr(), None, None, 0, N,
                            K, 128, 0) == wq.WQ_OK
    wq.gemm_w4a16(X, Wp, bf16_to_dev(s), Y=Y)


@pytest.mark.parametrize("bits", [4, 8])
def test_output_rows_beyond_m_untouched_and_deterministic(wq, small_kernel, bits):
    M, K, N = 5, 1280, 640
    X, q, s = synth.small_case(M, K, N, bits, seed=31)
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    canary = torch.full((M + 3, N), 7.0, dtype=torch.bfloat16, device="cuda")
    Yv = canary[:M]
    _gemm(wq, bits, Xt, Wp, st, Y=Yv)
    Y2 = _gemm(wq, bits, Xt, Wp, st)
    torch.cuda.synchronize()
    assert torch.all(canary[M:] == 7.0)
    assert torch.equal(Yv, Y2), "two calls differ"
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    assert_close_to_oracle(Yv, Yref, "canary case")


@pytest.mark.parametrize("bits", [4, 8])
def test_every_cluster_split(wq, small_kernel, bits):
    """Force each K split 1..8 of the cluster reduction on a ragged shape."""
    M, K, N = 9, 1152, 320   # 9 groups, 5 tiles
    X, q, s = synth.small_case(M, K, N, bits, seed=44)
    try:
        for cs in range(1, 9):
            wq.wq_debug_set_split(cs)
            _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)


# ------------------------------------------------ the benchmark workloads ---
def _case_ids(cases):
    return [c.name for c in cases]


FULL = synth.C1 + synth.C2 + synth.C3 + [c for c in synth.C4 if c.kind == "codes"]


@pytest.mark.parametrize("case", FULL, ids=_case_ids(FULL))
def test_workload_codes(wq, case):
    d = case.draw()
    _run_codes_case(wq, d["X"], d["q"], d["s"], case.bits)


@pytest.mark.parametrize("case", [c for c in synth.C4 if c.kind == "rtn"],
                         ids=_case_ids([c for c in synth.C4 if c.kind == "rtn"]))
def test_workload_drafter_rtn(wq, case):
    d = case.draw()
    K, N = case.K, case.N
    packed, st = wq.pack_symmetric(f32_to_dev(d["W"]), 8)
    Y = wq.gemm_w8a16(bf16_to_dev(d["X"]), packed, st)
    torch.cuda.synchronize()
    p_ref, s_ref, _ = oracle.pack_symmetric(d["W"], 8)
    assert np.array_equal(words_to_host(packed), p_ref)
    Yref = oracle.gemm(d["X"], p_ref, s_ref, K, N, 8)
    assert_close_to_oracle(Y, Yref, case.name)


@pytest.mark.parametrize("case", synth.C5, ids=_case_ids(synth.C5))
def test_workload_prefill_sampled_rows(wq, case):
    """M = 8192: rows sampled from the first and last 128-row tiles and at
    random are checked one by one against the oracle."""
    d = case.draw()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(120, 136),
                                     np.arange(case.M - 8, case.M),
                                     rng.integers(0, case.M, 24)]))
    _run_codes_case(wq, d["X"], d["q"], d["s"], case.bits, rows=rows)


@pytest.mark.parametrize("case", synth.C5, ids=_case_ids(synth.C5))
def test_workload_prefill_full(wq, case):
    """M = 8192 in full: every one of the 8192 x 9728 outputs against the
    oracle, on the default kernel (weights in tensor memory, 256-column
    tiles, persistent tile scheduler over 64 x 38 tiles) and on the tiled
    kernel with the weights in shared memory."""
    d = case.draw()
    K, N = case.K, case.N
    Wp = wq.pack_codes(i8_to_dev(d["q"]), case.bits)
    Xt, st = bf16_to_dev(d["X"]), bf16_to_dev(d["s"])
    assert wq.wq_gemm_regime(case.bits, case.M, N, K) == 3
    Y3 = _gemm(wq, case.bits, Xt, Wp, st)
    try:
        wq.wq_debug_force_regime(1)
        Y1 = _gemm(wq, case.bits, Xt, Wp, st)
    finally:
        wq.wq_debug_force_regime(-1)
    torch.cuda.synchronize()
    p_ref = oracle.pack(d["q"], case.bits)
    assert np.array_equal(words_to_host(Wp), p_ref)
    Yref = oracle.gemm(d["X"], p_ref, d["s"], K, N, case.bits)
    assert_close_to_oracle(Y3, Yref, case.name + " (weights in tensor memory)")
    assert_close_to_oracle(Y1, Yref, case.name + " (weights in shared memory)")


# --------------------------------------------- the tensor-core (tcgen05) path ---
@pytest.fixture
def tc_regime(wq):
    wq.wq_debug_force_regime(1)
    yield
    wq.wq_debug_force_regime(-1)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [(1, 128, 64), (100, 640, 320), (129, 1280, 576),
                                   (300, 384, 256), (256, 2560, 512)])
def test_tc_ragged_shapes(wq, tc_regime, bits, M, K, N):
    assert wq.wq_gemm_regime(bits, M, N, K) == 1
    X, q, s = synth.small_case(M, K, N, bits, seed=M + K + N + bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_tc_identity_probe_bit_exact(wq, tc_regime, bits):
    """X = I through the tensor-core path gives bf16(s*q) exactly."""
    K, N = 256, 320
    _, q, s = synth.small_case(1, K, N, bits, seed=5 + bits)
    eye = oracle.f32_to_bf16_bits(np.eye(K, dtype=np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(eye), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(eye, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(bf16_to_host_bits(Y), want)


@pytest.mark.parametrize("bits", [4, 8])
def test_tc_integer_exact_bit_exact(wq, tc_regime, bits):
    M, K, N = 200, 1024, 512
    rng = np.random.default_rng(23 + bits)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    s = oracle.f32_to_bf16_bits(
        (2.0 ** rng.integers(-8, -2, size=(K // 128, N))).astype(np.float32))
    X = oracle.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(X), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(bf16_to_host_bits(Y), want)


def test_tc_deterministic_and_rows_beyond_m_untouched(wq, tc_regime):
    M, K, N = 130, 768, 384
    X, q, s = synth.small_case(M, K, N, 4, seed=77)
    Wp = wq.pack_codes(i8_to_dev(q), 4)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    canary = torch.full((M + 5, N), 3.0, dtype=torch.bfloat16, device="cuda")
    wq.gemm_w4a16(Xt, Wp, st, Y=canary[:M])
    Y2 = wq.gemm_w4a16(Xt, Wp, st)
    torch.cuda.synchronize()
    assert torch.all(canary[M:] == 3.0)
    assert torch.equal(canary[:M], Y2)


# ------------------------------- tensor-core kernel, weights in tensor memory ---
@pytest.fixture
def wt_regime(wq):
    wq.wq_debug_force_regime(3)
    yield
    wq.wq_debug_force_regime(-1)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [(1, 512, 64), (100, 1024, 320), (129, 512, 576),
                                   (300, 1536, 256), (256, 2560, 512), (16, 1024, 192)])
def test_wt_ragged_shapes(wq, wt_regime, bits, M, K, N):
    assert wq.wq_gemm_regime(bits, M, N, K) == 3
    X, q, s = synth.small_case(M, K, N, bits, seed=M + K + N + 3 * bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [(512, 512, 320), (700, 1024, 576), (640, 2560, 1024),
                                   (513, 512, 64)])
def test_wt_wide_tiles_ragged(wq, wt_regime, bits, M, K, N):
    """M >= 512 takes tiles of 256 weight columns (two 128-lane halves
    sharing each X stage); N = 320, 576 and 64 leave partial tiles."""
    assert wq.wq_gemm_regime(bits, M, N, K) == 3
    X, q, s = synth.small_case(M, K, N, bits, seed=M + 2 * K + N + bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_wt_wide_integer_exact_bit_exact(wq, wt_regime, bits):
    M, K, N = 600, 512, 768
    rng = np.random.default_rng(43 + bits)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    s = oracle.f32_to_bf16_bits(
        (2.0 ** rng.integers(-8, -2, size=(K // 128, N))).astype(np.float32))
    X = oracle.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(X), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(bf16_to_host_bits(Y), want)


@pytest.mark.parametrize("bits", [4, 8])
def test_wt_unsupported_depth_falls_back(wq, wt_regime, bits):
    """K / 128 = 5 is not a multiple of the packed chunk: the tiled kernel
    with weights in shared memory runs instead."""
    M, K, N = 40, 640, 128
    assert wq.wq_gemm_regime(bits, M, N, K) == 1
    X, q, s = synth.small_case(M, K, N, bits, seed=5)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_wt_identity_probe_bit_exact(wq, wt_regime, bits):
    """X = I through the tensor-memory kernel gives bf16(s*q) exactly."""
    K, N = 512, 320
    _, q, s = synth.small_case(1, K, N, bits, seed=15 + bits)
    eye = oracle.f32_to_bf16_bits(np.eye(K, dtype=np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(eye), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(eye, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(bf16_to_host_bits(Y), want)


@pytest.mark.parametrize("bits", [4, 8])
def test_wt_integer_exact_bit_exact(wq, wt_regime, bits):
    M, K, N = 200, 1024, 512
    rng = np.random.default_rng(33 + bits)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    s = oracle.f32_to_bf16_bits(
        (2.0 ** rng.integers(-8, -2, size=(K // 128, N))).astype(np.float32))
    X = oracle.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Y = _gemm(wq, bits, bf16_to_dev(X), Wp, bf16_to_dev(s))
    torch.cuda.synchronize()
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    assert np.array_equal(bf16_to_host_bits(Y), want)


def test_wt_deterministic_and_rows_beyond_m_untouched(wq, wt_regime):
    M, K, N = 130, 1024, 384
    X, q, s = synth.small_case(M, K, N, 4, seed=78)
    Wp = wq.pack_codes(i8_to_dev(q), 4)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    canary = torch.full((M + 5, N), 3.0, dtype=torch.bfloat16, device="cuda")
    wq.gemm_w4a16(Xt, Wp, st, Y=canary[:M])
    Y2 = wq.gemm_w4a16(Xt, Wp, st)
    torch.cuda.synchronize()
    assert torch.all(canary[M:] == 3.0)
    assert torch.equal(canary[:M], Y2)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,N", [(64, 640), (100, 320), (128, 128)])
def test_wt_every_k_split(wq, wt_regime, bits, M, N):
    """A cluster of 1..8 CTAs splits each tile's K range (K = 2560: 5 packed
    chunks for INT4, 10 for INT8); the owners of each column add the fp32
    partials.  N = 320 leaves a half tile whose upper columns are owned but
    never stored."""
    K = 2560
    X, q, s = synth.small_case(M, K, N, bits, seed=M + N + bits)
    nchunks = (K // 128) // (4 if bits == 4 else 2)
    try:
        for ks in range(1, min(8, nchunks) + 1):
            wq.wq_debug_set_split(ks)
            _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)


@pytest.mark.parametrize("bits", [4, 8])
def test_wt_k_split_integer_exact_and_deterministic(wq, wt_regime, bits):
    """Partial sums that fp32 holds exactly: every split gives the same bits
    as the oracle, and a repeated call the same bits again."""
    M, K, N = 96, 2048, 256
    rng = np.random.default_rng(53 + bits)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    q = rng.integers(lo, hi + 1, size=(K, N)).astype(np.int8)
    s = oracle.f32_to_bf16_bits(
        (2.0 ** rng.integers(-8, -2, size=(K // 128, N))).astype(np.float32))
    X = oracle.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    want = oracle.f32_to_bf16_bits(Yref.astype(np.float32))
    nchunks = (K // 128) // (4 if bits == 4 else 2)
    try:
        for ks in range(1, min(8, nchunks) + 1):
            wq.wq_debug_set_split(ks)
            Y1 = _gemm(wq, bits, Xt, Wp, st)
            Y2 = _gemm(wq, bits, Xt, Wp, st)
            torch.cuda.synchronize()
            assert np.array_equal(bf16_to_host_bits(Y1), want), f"split {ks}"
            assert torch.equal(Y1, Y2), f"split {ks}"
    finally:
        wq.wq_debug_set_split(0)


def test_wt_k_split_beyond_chunks_is_refused(wq, wt_regime):
    """A forced split above the tile's chunk count is reported, not run."""
    M, K, N = 64, 512, 128  # one INT4 chunk
    X, q, s = synth.small_case(M, K, N, 4, seed=3)
    Wp = wq.pack_codes(i8_to_dev(q), 4)
    try:
        wq.wq_debug_set_split(2)
        with pytest.raises(wq.WQError) as ei:
            wq.gemm_w4a16(bf16_to_dev(X), Wp, bf16_to_dev(s))
        assert ei.value.status == wq.WQ_ERR_UNSUPPORTED
    finally:
        wq.wq_debug_set_split(0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", synth.C5, ids=_case_ids(synth.C5))
def test_wt_workload_prefill_sampled_rows(wq, wt_regime, case):
    d = case.draw()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(120, 136),
                                     np.arange(case.M - 8, case.M),
                                     rng.integers(0, case.M, 24)]))
    _run_codes_case(wq, d["X"], d["q"], d["s"], case.bits, rows=rows)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("cs", [2, 3])
def test_two_group_chunks_ragged(wq, bits, cs):
    """Warp-MMA kernel with two-group weight chunks (a K split over 16 or
    more groups per CTA): 33 groups split 2 or 3 ways, so a CTA's last chunk
    holds a single group; 7 rows, 3 tiles."""
    M, K, N = 7, 128 * 33, 192
    X, q, s = synth.small_case(M, K, N, bits, seed=70 + cs + bits)
    try:
        wq.wq_debug_force_regime(0)
        wq.wq_debug_set_split(cs)
        assert wq.wq_gemm_regime(bits, M, N, K) == 0
        _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)
        wq.wq_debug_force_regime(-1)


# ------------------------- tensor-memory small-M kernel with overlapping launches ---
@pytest.fixture
def stream_regime(wq):
    wq.wq_debug_force_regime(4)
    yield
    wq.wq_debug_force_regime(-1)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 7, 16, 24, 33, 64, 100])
@pytest.mark.parametrize("K,N", [(128, 64), (384, 192), (1280, 576), (3840, 128),
                                 (9728, 2560), (2560, 9728)])
def test_stream_shapes(wq, stream_regime, bits, M, K, N):
    """Ragged tiles (N = 64, 192, 576 leave a half tile), one to many groups
    per CTA, the splits the SM count picks; 16-, 32- and 64-token launches
    (M = 24 and 33 leave rows of the launch past M), and M = 100 as a
    64-row slice plus a 36-row one."""
    assert wq.wq_gemm_regime(bits, M, N, K) == 4
    X, q, s = synth.small_case(M, K, N, bits, seed=M * 5 + K + N + bits)
    _run_codes_case(wq, X, q, s, bits)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [11, 30, 50])
def test_stream_every_split(wq, stream_regime, bits, M):
    """Each K split 1..8 of the cluster reduction: 16 groups, 3 column tiles
    (the last one half), 11 rows (16-token launches, partials received in a
    dedicated buffer), 30 or 50 rows (32- and 64-token launches, partials
    received in the weight ring after a cluster rendezvous; the last 4-token
    quad and 16-token chunk part past M)."""
    K, N = 2048, 320
    X, q, s = synth.small_case(M, K, N, bits, seed=67 + bits + M)
    try:
        for cs in range(1, 9):
            wq.wq_debug_set_split(cs)
            _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("G", [9, 30, 32])
@pytest.mark.parametrize("M", [16, 64])
def test_stream_ring_refills(wq, stream_regime, bits, G, M):
    """One CTA per tile (split 1) walks G groups: more than the weight ring
    (6 groups INT4, 3 INT8), the X stages (9 at 16 tokens, 3 at 64) and the
    tensor-memory A slots (3) hold, up to the 32 groups its scales buffer
    takes."""
    K, N = 128 * G, 192
    X, q, s = synth.small_case(M, K, N, bits, seed=G + bits + M)
    try:
        wq.wq_debug_set_split(1)
        assert wq.wq_gemm_regime(bits, M, N, K) == 4
        _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("G", [5, 63, 64])
def test_stream_lead_split_limits(wq, stream_regime, bits, G):
    """A split of 2 gives rank 0 one group past half and sends rank 1's
    partials to it (the lead split): G = 5 (3 + 2 groups) and G = 63 (32 +
    31, rank 0 at the scales buffer's limit); at G = 64 the lead would take
    rank 0 past it, so the even split and the per-owner reduction run."""
    M, K, N = 16, 128 * G, 192
    X, q, s = synth.small_case(M, K, N, bits, seed=300 + G + bits)
    try:
        wq.wq_debug_set_split(2)
        assert wq.wq_gemm_regime(bits, M, N, K) == 4
        _run_codes_case(wq, X, q, s, bits)
    finally:
        wq.wq_debug_set_split(0)


def test_stream_too_many_groups_per_cta_falls_back(wq, stream_regime):
    """33 groups in one CTA exceed the scales buffer: the warp-MMA kernel
    takes the shape."""
    M, K, N = 16, 128 * 33, 128
    X, q, s = synth.small_case(M, K, N, 4, seed=33)
    try:
        wq.wq_debug_set_split(1)
        assert wq.wq_gemm_regime(4, M, N, K) == 0
        _run_codes_case(wq, X, q, s, 4)
    finally:
        wq.wq_debug_set_split(0)


def _chain_weights(wq, bits, L, K, seed):
    """L square weights whose scales keep |Y| about |X| along a chain."""
    rng = np.random.default_rng(seed)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    out = []
    for _ in range(L):
        q = rng.integers(lo, hi + 1, size=(K, K)).astype(np.int8)
        s_f = (0.25 / (np.sqrt(K) * (4.6 if bits == 4 else 73.0))) * \
            (np.abs(rng.standard_normal((K // 128, K))) + 0.5)
        s = oracle.f32_to_bf16_bits(s_f.astype(np.float32))
        out.append((q, s, wq.pack_codes(i8_to_dev(q), bits), bf16_to_dev(s)))
    return out


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [16, 64])
def test_stream_chain_reads_the_preceding_output(wq, stream_regime, bits, M):
    """Eight GEMMs on one stream with programmatic launch on, each reading
    the previous one's output as X: the launches overlap, so each must still
    see its predecessor's complete result.  Every step is checked against
    the oracle run on the step's actual input (16 rows: 16-token launches;
    64 rows: 64-token launches)."""
    K, L = 2560, 8
    ws = _chain_weights(wq, bits, L, K, seed=100 + bits)
    rng = np.random.default_rng(7)
    X0 = oracle.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    assert wq.wq_gemm_regime(bits, M, K, K) == 4
    outs = []
    try:
        wq.wq_set_programmatic_launch(True)
        x = bf16_to_dev(X0)
        for q, s, Wp, st in ws:
            x = _gemm(wq, bits, x, Wp, st)
            outs.append(x)
        torch.cuda.synchronize()
    finally:
        wq.wq_set_programmatic_launch(False)
    assert wq.wq_last_device_error() == wq.WQ_OK
    xin = X0
    for i, ((q, s, _, _), y) in enumerate(zip(ws, outs)):
        Yref = oracle.gemm(xin, oracle.pack(q, bits), s, K, K, bits)
        assert_close_to_oracle(y, Yref, f"chain step {i}")
        xin = bf16_to_host_bits(y)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [16, 64])
def test_stream_ping_pong_matches_serial_launches(wq, stream_regime, bits, M):
    """The same chain through two ping-pong buffers, so each launch also
    overwrites the buffer its predecessor read: with programmatic launch the
    bits equal those of launches that do not overlap."""
    K, L = 2560, 8
    ws = _chain_weights(wq, bits, L, K, seed=200 + bits)
    rng = np.random.default_rng(8)
    X0 = bf16_to_dev(oracle.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32)))

    def run(pdl):
        bufs = [X0.clone(), torch.empty_like(X0)]
        try:
            wq.wq_set_programmatic_launch(pdl)
            for i, (_, _, Wp, st) in enumerate(ws):
                _gemm(wq, bits, bufs[i % 2], Wp, st, Y=bufs[(i + 1) % 2])
            torch.cuda.synchronize()
        finally:
            wq.wq_set_programmatic_launch(False)
        return bufs[L % 2].clone()

    serial = run(False)
    for _ in range(3):
        assert torch.equal(run(True), serial)
    assert wq.wq_last_device_error() == wq.WQ_OK
