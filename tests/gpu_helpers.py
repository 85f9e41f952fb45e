"""Shared plumbing of the GPU parity tests: numpy <-> torch transfers of bf16
bit patterns, e4m3 bytes and int32 tensors, and the error measures the
tests use.  No arithmetic of the layer lives here."""
import numpy as np
import pytest
import torch

from grouped_gemm_serving_gb300.synth import bf16_bits_to_f32


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from grouped_gemm_serving_gb300 import build as gbuild
    gbuild.build()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32_from_bf16(t: torch.Tensor) -> np.ndarray:
    return bf16_bits_to_f32(host_bf16_bits(t))


def host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy()


def row_rel_err(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per row: max |y - ref| / max |ref| (rows with ref == 0 must be 0: inf otherwise)."""
    y = y.astype(np.float64)
    ref = ref.astype(np.float64)
    num = np.abs(y - ref).max(axis=1)
    den = np.abs(ref).max(axis=1)
    out = np.where(den > 0, num / np.where(den > 0, den, 1), np.where(num == 0, 0.0, np.inf))
    return out


def assert_close_bf16(y: np.ndarray, ref: np.ndarray, rtol=2.0 ** -7, row_atol=1e-3):
    """Elementwise |y - ref| <= rtol |ref| + row_atol * max_row |ref|; bf16 output rounding is 2^-9."""
    y = y.astype(np.float64)
    ref = ref.astype(np.float64)
    scale = np.abs(ref).max(axis=1, keepdims=True)
    bad = np.abs(y - ref) > rtol * np.abs(ref) + row_atol * scale
    assert not bad.any(), (np.argwhere(bad)[:5], y[bad][:5], ref[bad][:5])
