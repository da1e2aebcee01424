"""The fused MLP pair (wq_mlp_w4a16 / wq_mlp_w8a16) against the oracle's
pair: H = act(bf16(X . Wu)) and Y = H . Wd, on every kernel family the
up-projection can take (the activation in the store of the warp-MMA
small-M kernel, the overlapping-launch small-M kernel and the
tensor-memory tiled kernel, in a separate pass for the others)."""
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


def _run_pair(wq, M, K, N1, N2, bits, act, seed):
    X, qu, su = synth.small_case(M, K, N1, bits, seed=seed)
    _, qd, sd = synth.small_case(1, N1, N2, bits, seed=seed + 1)
    Hg, Yg = wq.mlp(bf16_to_dev(X), wq.pack_codes(i8_to_dev(qu), bits), bf16_to_dev(su),
                    wq.pack_codes(i8_to_dev(qd), bits), bf16_to_dev(sd), bits, act=act)
    torch.cuda.synchronize()
    assert wq.wq_last_device_error() == wq.WQ_OK
    H, Y = oracle.mlp(X, oracle.pack(qu, bits), su, oracle.pack(qd, bits), sd, K, N1, N2,
                      bits, act=act)
    assert_close_to_oracle(Hg, oracle.bf16_bits_to_f32(H).astype(np.float64), "H")
    assert_close_to_oracle(Yg, Y, "Y")
    return Hg, Yg


@pytest.mark.parametrize("act", ["none", "silu"])
def test_mlp_pair_workload_shape(wq, act):
    """The MLP-shaped pair at M = 16 (up 2560 -> 9728, down 9728 -> 2560)."""
    _run_pair(wq, 16, 2560, 9728, 2560, 4, act, seed=91)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("act", ["none", "silu"])
@pytest.mark.parametrize("M,K,N1,N2", [(1, 256, 128, 64), (16, 512, 256, 320),
                                       (40, 512, 256, 320), (130, 1024, 384, 192)])
def test_mlp_pair_shapes(wq, bits, act, M, K, N1, N2):
    """M = 1 and 16 (16-token launches of the small-M kernel with
    overlapping launches), 40 (one 64-token launch of it, K split over a
    cluster), 130 (tensor-memory tiled kernel, K split and ragged tiles)."""
    _run_pair(wq, M, K, N1, N2, bits, act, seed=M + K + bits)


@pytest.mark.parametrize("regime,M", [(1, 40), (2, 16), (0, 33), (4, 33), (3, 40)])
def test_mlp_pair_every_family(wq, regime, M):
    """Forced kernel families: the tiled shared-memory kernel and the
    tensor-memory small-M kernel take the activation as a separate pass; the
    warp-MMA kernel runs M = 33 in two 16-row slices plus one row, the
    overlapping-launch kernel in one 64-token launch; the tensor-memory tiled
    kernel applies it in its store."""
    try:
        wq.wq_debug_force_regime(regime)
        _run_pair(wq, M, 512, 256, 192, 4, "silu", seed=7 + regime)
    finally:
        wq.wq_debug_force_regime(-1)


def test_mlp_silu_matches_oracle_bits_on_exact_inputs(wq):
    """Integer X, power-of-two scales: the up-projection is exact in fp32,
    so H must carry the oracle's bits wherever fp32 SiLU rounds like fp64."""
    M, K, N1, N2, bits = 16, 256, 128, 64, 4
    rng = np.random.default_rng(5)
    qu = rng.integers(-8, 8, size=(K, N1)).astype(np.int8)
    qd = rng.integers(-8, 8, size=(N1, N2)).astype(np.int8)
    su = oracle.f32_to_bf16_bits((2.0 ** rng.integers(-6, -2, size=(K // 128, N1))).astype(np.float32))
    sd = oracle.f32_to_bf16_bits((2.0 ** rng.integers(-6, -2, size=(N1 // 128, N2))).astype(np.float32))
    X = oracle.f32_to_bf16_bits(rng.integers(-2, 3, size=(M, K)).astype(np.float32))
    Hg, _ = wq.mlp(bf16_to_dev(X), wq.pack_codes(i8_to_dev(qu), bits), bf16_to_dev(su),
                   wq.pack_codes(i8_to_dev(qd), bits), bf16_to_dev(sd), bits, act="silu")
    torch.cuda.synchronize()
    H, _ = oracle.mlp(X, oracle.pack(qu, bits), su, oracle.pack(qd, bits), sd, K, N1, N2, bits,
                      act="silu")
    got = Hg.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    # fp32 SiLU against fp64 SiLU, both rounded once more to bf16: at most a
    # handful of last-bit differences, never more than one bf16 step
    diff = np.abs(got.astype(np.int32) - H.astype(np.int32))
    assert diff.max() <= 1
    assert np.count_nonzero(diff) <= max(4, got.size // 200)


def test_mlp_empty_and_errors(wq):
    X = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    s = torch.zeros((2, 128), dtype=torch.bfloat16, device="cuda")
    sd = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256 * 128 // 8,), dtype=torch.int32, device="cuda")
    Wd = torch.zeros((128 * 64 // 8,), dtype=torch.int32, device="cuda")
    H, Y = wq.mlp(X, W, s, Wd, sd, 4, act="silu")
    assert H.shape == (0, 128) and Y.shape == (0, 64)
    with pytest.raises(ValueError):
        wq.mlp(X, W, s, Wd, sd, 4, act="gelu")


@pytest.mark.parametrize("M", [16, 40])
def test_mlp_without_activation_equals_two_gemm_calls(wq, M):
    """With no activation the pair is exactly the two GEMMs: the same kernels
    run, so H and Y match two wq_gemm_w4a16 calls bit for bit."""
    K, N1, N2, bits = 1024, 512, 256, 4
    X, qu, su = synth.small_case(M, K, N1, bits, seed=40 + M)
    _, qd, sd = synth.small_case(1, N1, N2, bits, seed=41 + M)
    Xt, sut, sdt = bf16_to_dev(X), bf16_to_dev(su), bf16_to_dev(sd)
    Wu, Wd = wq.pack_codes(i8_to_dev(qu), bits), wq.pack_codes(i8_to_dev(qd), bits)
    H, Y = wq.mlp(Xt, Wu, sut, Wd, sdt, bits, act="none")
    H2 = wq.gemm_w4a16(Xt, Wu, sut)
    Y2 = wq.gemm_w4a16(H2, Wd, sdt)
    torch.cuda.synchronize()
    assert torch.equal(H, H2)
    assert torch.equal(Y, Y2)
