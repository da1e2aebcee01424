"""Bounded waits: a wait that runs out reports WQ_ERR_DEVICE_TIMEOUT and the
context stays usable.  The wait is made to run out by pointing it at a
barrier nothing completes (no fault, no trap, no hang)."""
import numpy as np
import pytest
import torch

import oracle
from tests import synth
from tests.gpu_util import assert_close_to_oracle, bf16_to_dev, i8_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wq():
    import __graft_entry__
    __graft_entry__.build()
    import w4a16_weight_only_wq_gb300 as m
    return m


@pytest.fixture(params=[0, 1, 2, 3, 4], ids=["warpmma", "tc", "tmem", "wt", "stream"])
def regime(wq, request):
    wq.wq_debug_force_regime(request.param)
    yield request.param
    wq.wq_debug_force_regime(-1)


@pytest.mark.parametrize("bits", [4, 8])
def test_forced_timeout_reports_and_recovers(wq, regime, bits):
    M, K, N = 16, 1024, 256
    X, q, s = synth.small_case(M, K, N, bits, seed=8)
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    fn = wq.gemm_w4a16 if bits == 4 else wq.gemm_w8a16
    torch.cuda.synchronize()
    assert wq.wq_clear_device_error() == wq.WQ_OK
    try:
        wq.wq_debug_set_wait_limit_ns(200_000)  # 0.2 ms
        wq.wq_debug_force_timeout(1)
        fn(Xt, Wp, st)
        torch.cuda.synchronize()
    finally:
        wq.wq_debug_force_timeout(0)
        wq.wq_debug_set_wait_limit_ns(0)
    assert wq.wq_last_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.wq_clear_device_error() == wq.WQ_OK
    Y = fn(Xt, Wp, st)
    torch.cuda.synchronize()
    assert wq.wq_last_device_error() == wq.WQ_OK
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    assert_close_to_oracle(Y, Yref, "after timeout")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("small", [0, 2, 3, 4], ids=["warpmma", "tmem", "wt", "stream"])
def test_abandoned_data_wait_drains_and_recovers(wq, small, bits):
    """The data waits look for a phase that never completes: the kernel gives
    up, lets its copies land, reports the timeout, and a normal call
    afterwards is correct."""
    M, K, N = 16, 9728, 2560  # split across a cluster, ring refills for INT8
    X, q, s = synth.small_case(M, K, N, bits, seed=12)
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    fn = wq.gemm_w4a16 if bits == 4 else wq.gemm_w8a16
    torch.cuda.synchronize()
    assert wq.wq_clear_device_error() == wq.WQ_OK
    try:
        wq.wq_debug_force_regime(small)
        wq.wq_debug_set_wait_limit_ns(1_000_000)  # 1 ms
        wq.wq_debug_force_timeout(2)
        fn(Xt, Wp, st)
        torch.cuda.synchronize()
    finally:
        wq.wq_debug_force_timeout(0)
        wq.wq_debug_set_wait_limit_ns(0)
        wq.wq_debug_force_regime(-1)
    assert wq.wq_last_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.wq_clear_device_error() == wq.WQ_OK
    Y = fn(Xt, Wp, st)
    torch.cuda.synchronize()
    assert wq.wq_last_device_error() == wq.WQ_OK
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    assert_close_to_oracle(Y, Yref, "after an abandoned wait")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [(16, 2560, 9728), (32, 2560, 9728), (64, 2560, 2560)],
                         ids=["lead_split", "tok32", "tok64_cluster6"])
def test_stream_abandoned_wait_paths(wq, bits, M, K, N):
    """The stream kernel's other reductions under an abandoned wait: the
    lead split (a split of 2: rank 1 sends its whole partial to rank 0), and
    the 32- and 64-token launches (partials received in the owners' weight
    rings after a rendezvous).  Every rank still sends and every thread
    reaches the cluster barriers; the error is reported and a normal call
    afterwards is correct."""
    X, q, s = synth.small_case(M, K, N, bits, seed=13 + M)
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    Xt, st = bf16_to_dev(X), bf16_to_dev(s)
    fn = wq.gemm_w4a16 if bits == 4 else wq.gemm_w8a16
    torch.cuda.synchronize()
    assert wq.wq_clear_device_error() == wq.WQ_OK
    try:
        wq.wq_debug_force_regime(4)
        assert wq.wq_gemm_regime(bits, M, N, K) == 4
        wq.wq_debug_set_wait_limit_ns(1_000_000)  # 1 ms
        wq.wq_debug_force_timeout(2)
        fn(Xt, Wp, st)
        torch.cuda.synchronize()
        assert wq.wq_last_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
        assert wq.wq_clear_device_error() == wq.WQ_OK
        wq.wq_debug_force_timeout(0)
        wq.wq_debug_set_wait_limit_ns(0)
        Y = fn(Xt, Wp, st)
        torch.cuda.synchronize()
    finally:
        wq.wq_debug_force_timeout(0)
        wq.wq_debug_set_wait_limit_ns(0)
        wq.wq_debug_force_regime(-1)
    assert wq.wq_last_device_error() == wq.WQ_OK
    Yref = oracle.gemm(X, oracle.pack(q, bits), s, K, N, bits)
    assert_close_to_oracle(Y, Yref, "after an abandoned wait")


def test_attention_abandoned_wait_reports_and_recovers(wq):
    """The wait for the last key/value chunk and the merge wait of the
    sliding-window attention look at a barrier that never completes: the
    kernel gives up, lets its copies and the partials land, reports the
    timeout, and a normal call afterwards is correct."""
    B, Hq, Hkv, T, W = 16, 8, 2, 700, 256
    rng = np.random.default_rng(21)
    Q = oracle.f32_to_bf16_bits(rng.normal(size=(B, Hq, 128)).astype(np.float32))
    K = oracle.f32_to_bf16_bits(rng.normal(size=(Hkv, T, 128)).astype(np.float32))
    V = oracle.f32_to_bf16_bits(rng.normal(size=(Hkv, T, 128)).astype(np.float32))
    Qt, Kt, Vt = bf16_to_dev(Q), bf16_to_dev(K), bf16_to_dev(V)
    torch.cuda.synchronize()
    assert wq.wq_clear_device_error() == wq.WQ_OK
    try:
        wq.wq_debug_set_wait_limit_ns(1_000_000)  # 1 ms
        wq.wq_debug_force_timeout(2)
        wq.swa_attention(Qt, Kt, Vt, W)
        torch.cuda.synchronize()
    finally:
        wq.wq_debug_force_timeout(0)
        wq.wq_debug_set_wait_limit_ns(0)
    assert wq.wq_last_device_error() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.wq_clear_device_error() == wq.WQ_OK
    O = wq.swa_attention(Qt, Kt, Vt, W)
    torch.cuda.synchronize()
    assert wq.wq_last_device_error() == wq.WQ_OK
    assert_close_to_oracle(O, oracle.swa_attention(Q, K, V, T, W), "after an abandoned wait")
