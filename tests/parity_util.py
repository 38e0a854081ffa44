"""Helpers shared by the GPU parity tests: host <-> device marshalling and the
tolerance checks.

Tolerances (written out here, used by every parity test):

* fp32 outputs: max_i |y_i - y*_i| / max_i |y*_i| <= 1e-5, y* the oracle's
  exact (binary64) value.
* bf16 outputs: the same scale-normalised bound, 2e-3, applied to the error
  beyond the output type's own rounding:
      max_i max(0, |y_i - y*_i| - ulp_bf16(y*_i)/2) / max_i |y*_i| <= 2e-3,
  because a bf16 value cannot be closer to y* than half a bf16 spacing (2^-9
  relative, above 2e-3 for elements near the maximum).  The plain metric
  max|y - bf16(y*)| / max|bf16(y*)| and the count of elements that differ
  from bf16(y*) are reported alongside.
* integer / byte / index work (packed codes, scales, biases, out_sum,
  exact-arithmetic indexing cases): bit-exact.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

TOL_BF16 = 2e-3
TOL_F32 = 1e-5


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> bfloat16 CUDA tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor -> uint16 bit patterns on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return oracle.f64_from_bf16(host_bits(t))
    return t.detach().cpu().numpy().astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (2^(floor(log2|x|) - 7), normal range)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(int))


def bf16_error(y_bits: np.ndarray, y_exact: np.ndarray):
    """Returns (err_beyond_rounding, plain_err, n_diff) for a bf16 output."""
    y = oracle.f64_from_bf16(y_bits)
    ref = np.asarray(y_exact, dtype=np.float64)
    scale = np.max(np.abs(ref))
    if scale == 0:
        scale = 1.0
    excess = np.maximum(0.0, np.abs(y - ref) - 0.5 * ulp_bf16(ref))
    ref_b = oracle.bf16_from_f64(ref)
    plain = np.max(np.abs(y - oracle.f64_from_bf16(ref_b))) / scale
    n_diff = int(np.count_nonzero(y_bits != ref_b))
    return float(np.max(excess) / scale), float(plain), n_diff


def assert_bf16_close(y_bits, y_exact, what=""):
    err, plain, nd = bf16_error(y_bits, y_exact)
    assert np.all(np.isfinite(oracle.f64_from_bf16(y_bits))), f"{what}: non-finite output"
    assert err <= TOL_BF16, f"{what}: scale-normalised error {err:.3e} > {TOL_BF16} " \
                            f"(plain {plain:.3e}, {nd} elements differ from bf16(oracle))"
    return err, plain, nd


def assert_f32_close(y, y_exact, what=""):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(y_exact, dtype=np.float64)
    scale = np.max(np.abs(ref)) or 1.0
    err = float(np.max(np.abs(y - ref)) / scale)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    assert err <= TOL_F32, f"{what}: scale-normalised error {err:.3e} > {TOL_F32}"
    return err
