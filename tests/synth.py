"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests
and bench.py.

This module only draws random numbers (torch.Generator on the CPU, so the
same seed gives the same tensors on every machine) and rounds them to the
storage types; it contains none of the quantization, packing or GEMM
arithmetic.  All arrays are numpy; bf16 values travel as their uint16 bit
patterns.

Workloads (shapes from the pages, distributions from the benchmark
definition):
  * M = 16 is one speculative block verify: the anchor token plus 15
    drafted tokens ("num_speculative_tokens": 15, block size 16).
  * K = 2560 is the hidden size of the 4B-class target / 5-layer drafter.
  * N = 9728 is the MLP width used for the up/down projection pair.
  * M = 8192 is the "Long" prompt length of the latency protocol.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

GROUP = 128


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Round an fp32 CPU tensor to bf16 (torch RNE) and return the bits."""
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(
        np.uint16).copy()


def activations(g: torch.Generator, M: int, K: int) -> np.ndarray:
    """X ~ N(0, 1) in bf16, [M, K]."""
    return bf16_bits(torch.randn(M, K, generator=g, dtype=torch.float32))


def codes_uniform(g: torch.Generator, K: int, N: int, lo: int,
                  hi: int) -> np.ndarray:
    """Integer codes uniform in [lo, hi], int8 [K, N]."""
    return torch.randint(lo, hi + 1, (K, N), generator=g,
                         dtype=torch.int32).to(torch.int8).numpy()


def scales_abs_normal(g: torch.Generator, K: int, N: int) -> np.ndarray:
    """s = bf16(0.02 * |N(0,1)| + 1e-3), [K/128, N]."""
    z = torch.randn(K // GROUP, N, generator=g, dtype=torch.float32)
    return bf16_bits(0.02 * z.abs() + 1e-3)


def weights_normal(g: torch.Generator, K: int, N: int,
                   std: float = 0.02) -> np.ndarray:
    """fp32 weights ~ N(0, std), [K, N]."""
    return (torch.randn(K, N, generator=g, dtype=torch.float32) * std).numpy()


@dataclass
class GemmCase:
    """One GEMM problem.  Codes are either drawn directly (kind 'codes') or
    produced by the pack step from Gaussian weights (kind 'rtn')."""
    name: str
    M: int
    K: int
    N: int
    bits: int
    seed: int
    kind: str = "codes"  # 'codes' | 'rtn' | 'codes_full'

    def draw(self):
        """Returns dict with X (bf16 bits), and either (q, s) or W."""
        g = _gen(self.seed)
        out = {"X": activations(g, self.M, self.K)}
        if self.kind == "rtn":
            out["W"] = weights_normal(g, self.K, self.N)
        else:
            lo, hi = (-8, 7) if self.bits == 4 else (-127, 127)
            out["q"] = codes_uniform(g, self.K, self.N, lo, hi)
            out["s"] = scales_abs_normal(g, self.K, self.N)
        return out


# The five benchmark workloads.
C1 = [GemmCase("c1_verify_w4_m16_2560x2560", 16, 2560, 2560, 4, 0)]
C2 = [GemmCase("c2_mlp_up_w4_m16_2560x9728", 16, 2560, 9728, 4, 1),
      GemmCase("c2_mlp_down_w4_m16_9728x2560", 16, 9728, 2560, 4, 1)]
C3 = [GemmCase(f"c3_sweep_w4_m{m}_2560x{n}", m, 2560, n, 4, 2)
      for n in (2560, 9728) for m in (1, 16, 64, 128)]
C4 = [GemmCase(f"c4_drafter_w8_rtn_m16_2560x{n}", 16, 2560, n, 8, 3, "rtn")
      for n in (2560, 9728)] + \
     [GemmCase(f"c4_drafter_w8_codes_m16_2560x{n}", 16, 2560, n, 8, 3, "codes")
      for n in (2560, 9728)]
C5 = [GemmCase("c5_prefill_w4_m8192_2560x9728", 8192, 2560, 9728, 4, 4)]
ALL_CASES = C1 + C2 + C3 + C4 + C5

# The pack check of the MLP pair: fp32 weights ~ N(0, 0.02) of both shapes.
PACK_CASES = [("c2_pack_up_2560x9728", 2560, 9728, 1),
              ("c2_pack_down_9728x2560", 9728, 2560, 1)]


def pack_weights(K: int, N: int, seed: int) -> np.ndarray:
    return weights_normal(_gen(seed + 1000), K, N)


def small_case(M: int, K: int, N: int, bits: int, seed: int):
    """Random codes/scales/activations of any small shape."""
    g = _gen(seed)
    lo, hi = (-8, 7) if bits == 4 else (-128, 127)
    return (activations(g, M, K), codes_uniform(g, K, N, lo, hi),
            scales_abs_normal(g, K, N))
