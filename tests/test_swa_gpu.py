"""The drafter's symmetric sliding-window attention (wq_swa_attention)
against the oracle: random heads at several window / sequence lengths,
every split of the keys over a cluster, the window bounds through equal
scores, grouped heads, and determinism."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_close_to_oracle, bf16_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wq():
    import __graft_entry__
    __graft_entry__.build()
    import w4a16_weight_only_wq_gb300 as m
    return m


def _bf16(a):
    return oracle.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _case(B, Hq, Hkv, T, seed):
    rng = np.random.default_rng(seed)
    Q = _bf16(rng.normal(size=(B, Hq, 128)))
    K = _bf16(rng.normal(size=(Hkv, T, 128)))
    V = _bf16(rng.normal(size=(Hkv, T, 128)))
    return Q, K, V


def _run(wq, Q, K, V, T, W):
    O = wq.swa_attention(bf16_to_dev(Q), bf16_to_dev(K), bf16_to_dev(V), W)
    torch.cuda.synchronize()
    assert wq.wq_last_device_error() == wq.WQ_OK
    return O


@pytest.mark.parametrize("B,Hq,Hkv,T,W", [
    (16, 4, 2, 300, 64),        # window inside the sequence
    (16, 32, 8, 4096, 2048),    # the drafter's shape: 32 query heads, 8 key/value heads
    (16, 8, 8, 1037, 0),        # full attention, ragged chunk tail
    (16, 4, 1, 500, 1024),      # sequence within the window: full attention
    (5, 4, 2, 700, 128),        # a short block
    (1, 2, 1, 90, 16),
    (16, 2, 2, 16, 8),          # the block alone
    (16, 6, 2, 900, 512),       # three query heads per key/value head: one CTA per query head
    (16, 16, 8, 2000, 600),     # two query heads per key/value head: one CTA per key/value head
])
def test_swa_matches_oracle(wq, B, Hq, Hkv, T, W):
    Q, K, V = _case(B, Hq, Hkv, T, seed=B + T + W)
    O = _run(wq, Q, K, V, T, W)
    assert_close_to_oracle(O, oracle.swa_attention(Q, K, V, T, W), f"T={T} W={W}")


def test_swa_every_split(wq):
    B, Hq, Hkv, T, W = 16, 4, 2, 1500, 1024
    Q, K, V = _case(B, Hq, Hkv, T, seed=4)
    ref = oracle.swa_attention(Q, K, V, T, W)
    try:
        for S in range(1, 9):
            wq.wq_debug_set_split(S)
            assert_close_to_oracle(_run(wq, Q, K, V, T, W), ref, f"split {S}")
    finally:
        wq.wq_debug_set_split(0)


@pytest.mark.parametrize("T,W", [(200, 64), (250, 100), (120, 0), (64, 2)])
def test_swa_window_bounds_exact_means(wq, T, W):
    """Equal keys give every visible key the same weight; with value j at key
    j the output is (lo + hi) / 2, which bf16 holds exactly (a multiple of
    1/2 below 256)."""
    B, Hq, Hkv = 16, 2, 1
    rng = np.random.default_rng(T)
    Q = _bf16(rng.normal(size=(B, Hq, 128)))
    K = _bf16(np.broadcast_to(rng.normal(size=(1, 1, 128)), (Hkv, T, 128)))
    V = _bf16(np.broadcast_to(np.arange(T, dtype=np.float32)[None, :, None], (Hkv, T, 128)))
    O = _run(wq, Q, K, V, T, W).float().cpu().numpy()
    for b in range(B):
        p = T - B + b
        lo, hi = (0, T - 1) if (W == 0 or T <= W) else (max(0, p - W // 2), min(T - 1, p + W // 2))
        # equal fp32 weights sum to n exactly; the mean is rounded once to bf16
        want = oracle.bf16_bits_to_f32(_bf16([(lo + hi) / 2]))[0]
        assert np.all(np.abs(O[b] - want) <= abs(want) * 2.0 ** -7 + 1e-6), (b, lo, hi)


def test_swa_grouped_heads_and_determinism(wq):
    B, Hq, Hkv, T, W = 16, 8, 2, 600, 256
    rng = np.random.default_rng(8)
    Q = _bf16(rng.normal(size=(B, Hq, 128)))
    K = _bf16(rng.normal(size=(Hkv, T, 128)))
    V = _bf16(np.broadcast_to((np.arange(Hkv, dtype=np.float32) + 1)[:, None, None], (Hkv, T, 128)))
    O1 = _run(wq, Q, K, V, T, W)
    O2 = _run(wq, Q, K, V, T, W)
    assert torch.equal(O1, O2)
    got = O1.float().cpu().numpy()
    for h in range(Hq):
        assert np.allclose(got[:, h, :], h // (Hq // Hkv) + 1, rtol=2.0 ** -7, atol=0)


@pytest.mark.parametrize("S", [1, 2])
def test_swa_long_slices_refill_every_buffer(wq, S):
    """Full attention over 4,096 keys in one or two slices per head: 32 or 16
    chunks of 128 keys per CTA, so each of the three chunk buffers is
    refilled many times by whichever warp releases it last; the result is
    deterministic and matches the oracle."""
    B, Hq, Hkv, T, W = 16, 2, 1, 4096, 0
    Q, K, V = _case(B, Hq, Hkv, T, seed=60 + S)
    ref = oracle.swa_attention(Q, K, V, T, W)
    try:
        wq.wq_debug_set_split(S)
        O1 = _run(wq, Q, K, V, T, W)
        O2 = _run(wq, Q, K, V, T, W)
    finally:
        wq.wq_debug_set_split(0)
    assert torch.equal(O1, O2)
    assert_close_to_oracle(O1, ref, f"split {S}")


@pytest.mark.parametrize("T,W", [(8192, 2048), (8192, 1024), (2048, 4096)])
def test_swa_bench_workloads(wq, T, W):
    """The three attention workloads bench.py times (16-token block, 32 query
    heads over 8 key/value heads of 128), in the same launch configuration,
    against the oracle over every output."""
    B, Hq, Hkv = 16, 32, 8
    Q, K, V = _case(B, Hq, Hkv, T, seed=T + W)
    assert_close_to_oracle(_run(wq, Q, K, V, T, W), oracle.swa_attention(Q, K, V, T, W),
                           f"T={T} W={W}")
