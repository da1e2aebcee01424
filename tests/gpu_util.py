"""Helpers shared by the GPU parity tests (host <-> device marshalling)."""
import numpy as np
import torch

import oracle


def dev():
    return torch.device("cuda:0")


def bf16_to_dev(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bfloat16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).to(dev())


def f32_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def i8_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int8)).to(dev())


def words_to_host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def bf16_to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close_to_oracle(Y_gpu: torch.Tensor, Y_ref: np.ndarray, what=""):
    """The parity bar for the GEMM: max|Y_gpu - Y_ref| <= 1e-2 max|Y_ref| + 1e-3."""
    Yg = bf16_to_host_f64(Y_gpu)
    assert Yg.shape == Y_ref.shape, (Yg.shape, Y_ref.shape)
    assert np.all(np.isfinite(Yg)), f"{what}: non-finite output"
    err = float(np.max(np.abs(Yg - Y_ref))) if Y_ref.size else 0.0
    tol = oracle.tolerance(Y_ref)
    assert err <= tol, f"{what}: max|err| {err:.4e} > tol {tol:.4e}"
    return err, tol
