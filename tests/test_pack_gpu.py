"""GPU pack / unpack against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from tests import synth
from tests.gpu_util import (bf16_to_dev, bf16_to_host_bits, f32_to_dev,
                            i8_to_dev, words_to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wq():
    import __graft_entry__
    __graft_entry__.build()
    import w4a16_weight_only_wq_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    return m


def _special_weights(K, N, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    W[:, 0] = 0.0                        # all-zero column -> s = 1, q = 0
    W[5, 1] = 3.0                        # outlier
    W[:, 2] = 0.125                      # constant column
    W[:, 3] = np.float32(-1.0)           # negative absmax
    W[: K // 2, 4] = np.float32(1e-30)   # tiny values
    return W


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [(128, 64), (384, 192), (640, 320)])
def test_pack_rtn_fp32_bit_exact(wq, bits, K, N):
    W = _special_weights(K, N, seed=K + N + bits)
    packed, s = wq.pack_symmetric(f32_to_dev(W), bits)
    torch.cuda.synchronize()
    p_ref, s_ref, _ = oracle.pack_symmetric(W, bits)
    assert np.array_equal(bf16_to_host_bits(s), s_ref)
    assert np.array_equal(words_to_host(packed), p_ref)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_rtn_bf16_input_bit_exact(wq, bits):
    K, N = 384, 128
    W = _special_weights(K, N, seed=9)
    Wb = oracle.f32_to_bf16_bits(W)
    packed, s = wq.pack_symmetric(bf16_to_dev(Wb), bits)
    torch.cuda.synchronize()
    p_ref, s_ref, _ = oracle.pack_symmetric(oracle.bf16_bits_to_f32(Wb), bits)
    assert np.array_equal(bf16_to_host_bits(s), s_ref)
    assert np.array_equal(words_to_host(packed), p_ref)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_fixed_grid_round_trip(wq, bits):
    """Weights on the grid of supplied scales come back as the same codes
    (the packing step of grid-preserving QAD)."""
    K, N = 512, 256
    X, q, s = synth.small_case(1, K, N, bits, seed=77)
    sv = oracle.bf16_bits_to_f32(s).astype(np.float64)
    W = (np.repeat(sv, 128, axis=0) * q).astype(np.float32)
    packed, s_out = wq.pack_symmetric(f32_to_dev(W), bits, scales=bf16_to_dev(s))
    codes = wq.unpack(packed, K, N, bits)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_host_bits(s_out), s)
    assert np.array_equal(codes.cpu().numpy(), q)
    assert np.array_equal(words_to_host(packed), oracle.pack(q, bits))


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_supplied_scales_clamp_and_ties(wq, bits):
    K, N = 128, 64
    rng = np.random.default_rng(5)
    W = (rng.integers(-300, 300, size=(K, N)) * 0.5).astype(np.float32)  # ties
    s = np.full((1, N), 0x3F80, dtype=np.uint16)  # s = 1
    packed, _ = wq.pack_symmetric(f32_to_dev(W), bits, scales=bf16_to_dev(s))
    torch.cuda.synchronize()
    p_ref, _, _ = oracle.pack_symmetric(W, bits, scales_in=s)
    assert np.array_equal(words_to_host(packed), p_ref)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_codes_and_unpack_bit_exact(wq, bits):
    for K, N, seed in ((128, 64, 1), (1280, 576, 2)):
        _, q, _ = synth.small_case(1, K, N, bits, seed)
        packed = wq.pack_codes(i8_to_dev(q), bits)
        codes = wq.unpack(packed, K, N, bits)
        torch.cuda.synchronize()
        assert np.array_equal(words_to_host(packed), oracle.pack(q, bits))
        assert np.array_equal(codes.cpu().numpy(), q)


@pytest.mark.parametrize("name,K,N,seed", synth.PACK_CASES)
def test_pack_mlp_pair_weights_bit_exact(wq, name, K, N, seed):
    """The MLP-pair pack check: fp32 weights ~ N(0, 0.02), both shapes, INT4."""
    W = synth.pack_weights(K, N, seed)
    packed, s = wq.pack_symmetric(f32_to_dev(W), 4)
    torch.cuda.synchronize()
    p_ref, s_ref, _ = oracle.pack_symmetric(W, 4)
    assert np.array_equal(bf16_to_host_bits(s), s_ref), name
    assert np.array_equal(words_to_host(packed), p_ref), name


@pytest.mark.parametrize("n", [2560, 9728])
def test_pack_drafter_int8_rtn_bit_exact(wq, n):
    case = [c for c in synth.C4 if c.kind == "rtn" and c.N == n][0]
    W = case.draw()["W"]
    packed, s = wq.pack_symmetric(f32_to_dev(W), 8)
    torch.cuda.synchronize()
    p_ref, s_ref, q_ref = oracle.pack_symmetric(W, 8)
    assert np.array_equal(bf16_to_host_bits(s), s_ref)
    assert np.array_equal(words_to_host(packed), p_ref)
    assert q_ref.min() >= -127 and q_ref.max() <= 127


# ------------------------------------------------------ effective weight ---
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [(128, 64), (384, 192), (1280, 576)])
def test_dequantize_bit_exact(wq, bits, K, N):
    """bf16(s * q) for every weight, against the oracle's exact fp32 dequant
    rounded once."""
    _, q, s = synth.small_case(1, K, N, bits, seed=K + N + bits)
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    W = wq.dequantize(Wp, bf16_to_dev(s), bits)
    torch.cuda.synchronize()
    want = oracle.f32_to_bf16_bits(oracle.dequant(q, s))
    assert np.array_equal(bf16_to_host_bits(W), want)


@pytest.mark.parametrize("bits", [4, 8])
def test_dequantize_equals_identity_probe(wq, bits):
    """The effective weight equals what an identity matrix run through the
    quantized GEMM returns (the W8A16 card's fused-KV extraction)."""
    K, N = 256, 320
    _, q, s = synth.small_case(1, K, N, bits, seed=40 + bits)
    Wp = wq.pack_codes(i8_to_dev(q), bits)
    st = bf16_to_dev(s)
    W = wq.dequantize(Wp, st, bits)
    eye = torch.eye(K, dtype=torch.bfloat16, device="cuda")
    fn = wq.gemm_w4a16 if bits == 4 else wq.gemm_w8a16
    Y = fn(eye, Wp, st)
    torch.cuda.synchronize()
    assert torch.equal(W, Y)


# ------------------------------------------------------ checkpoint import ---
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [(128, 64), (384, 192), (2560, 576)])
def test_import_packed_nk_bit_exact(wq, bits, K, N):
    """An output-channel-major checkpoint layer (codes packed along K) is
    repacked into exactly the words the oracle packs from its codes."""
    from tests.test_oracle import _encode_nk
    _, q, s = synth.small_case(1, K, N, bits, seed=K + N + 7 * bits)
    qw = torch.from_numpy(_encode_nk(q, bits).view(np.int32)).cuda()
    s_nk = torch.from_numpy(np.ascontiguousarray(s.T).view(np.int16)).view(torch.bfloat16).cuda()
    packed, scales = wq.import_packed_nk(qw, s_nk, bits)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.import_packed_nk(_encode_nk(q, bits), np.ascontiguousarray(s.T), K, N,
                                           bits)
    assert np.array_equal(words_to_host(packed), oracle.pack(q_ref, bits))
    assert np.array_equal(bf16_to_host_bits(scales), s_ref)
