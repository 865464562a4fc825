"""Helpers for the GPU parity tests: moving stored arrays to the device and the
tolerance rules.

Tolerances (stated once, used by every GPU test):
* wnorm, g: relative error <= 1e-4 for bf16 inputs, <= 1e-6 for fp32 inputs,
  per element, against the float64 oracle.
* compose, bf16 output: within 1 bf16 ulp of the oracle rounded once to bf16
  (distance in representable steps <= 1).
* compose, fp32 output: within 2 fp32 ulp of the oracle rounded to fp32.
* training path (inner, d_base, d_lora): the compose rule above.
* dmag: |dmag - ref| <= 1e-5 * sum_t |d_out_tj * inner_tj| / max(wnorm_j, eps).
  The kernel sums at most ceil(T / parts) exact products per thread in fp32,
  then the parts (<= 256) compensated, then divides once: an error bound of
  about (T / parts + 3) * 2^-24 of the absolute sum, 1e-6 at T / parts <= 16;
  1e-5 leaves a factor of ten.
"""
from __future__ import annotations

import numpy as np
import torch

from synthetic import configs

NORM_RTOL = {configs.BF16: 1e-4, configs.F32: 1e-6}


def to_dev(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == configs.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def to_host_stored(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def rel_err(got, ref) -> np.ndarray:
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    return np.abs(got - ref) / np.maximum(np.abs(ref), np.finfo(np.float64).tiny)


def ordered_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers in the same order as the values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ordered_f32(x: np.ndarray) -> np.ndarray:
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.int64)
    return np.where(b & 0x80000000, -(b & 0x7FFFFFFF), b)


def ulp_distance(got_stored: np.ndarray, ref_stored: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == configs.BF16:
        return np.abs(ordered_bf16(got_stored) - ordered_bf16(ref_stored))
    return np.abs(ordered_f32(got_stored) - ordered_f32(ref_stored))


COMPOSE_MAX_ULP = {configs.BF16: 1, configs.F32: 2}

DM_RTOL = 1e-5
