"""Seeded synthetic inputs in their stored formats.

Every tensor is cut into fixed row chunks; chunk ``c`` of tensor ``t`` of
module ``k`` in config ``i`` is drawn from its own Philox stream keyed by
``(seed, i, t, k, c)`` (numpy's ``SeedSequence``), so any subset of rows can be
regenerated without drawing the rest, and the chunks can be drawn in parallel.

Stored formats (what the library and the oracle both receive):

* ``bf16``: ``numpy.uint16`` holding the bfloat16 bit pattern, obtained from a
  float32 draw by round-to-nearest-even on the top 16 bits;
* ``f32``: ``numpy.float32``.

The magnitude vector follows the DoRA initialisation the paper write-up
describes (magnitude initialised to the row norm of W, so g starts near 1;
"Scaling DoRA" section 2.1.1): ``m_j = ||W_j|| * (1 + 0.0015 z_j)`` with
``||W_j||`` taken from the stored W in float64, then stored in W's dtype.
That is input construction only: nothing here evaluates the factored norm,
the magnitude scale or the compose.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterable, Optional, Sequence

import numpy as np

from .configs import BF16, F32, Config

CHUNK_ELEMS = 1 << 22

# tensor ids inside the Philox key
T_W, T_A, T_B, T_M, T_BASE, T_LORA, T_G, T_DOUT = range(8)

_POOL: Optional[ThreadPoolExecutor] = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4))
    return _POOL


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit pattern, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit pattern -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(stored: np.ndarray, dtype: str) -> np.ndarray:
    """Stored array -> float64 (exact)."""
    if dtype == BF16:
        return bf16_bits_to_f32(stored).astype(np.float64)
    return np.asarray(stored, dtype=np.float32).astype(np.float64)


def _rows_per_chunk(n_cols: int) -> int:
    return max(1, CHUNK_ELEMS // max(1, n_cols))


def _draw_chunk(key: Sequence[int], n: int, std: float, mean: float, dtype: str) -> np.ndarray:
    rng = np.random.Generator(np.random.Philox(np.random.SeedSequence(list(key))))
    x = rng.standard_normal(n, dtype=np.float32)
    x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    if dtype == BF16:
        return f32_to_bf16_bits(x)
    return x


def normal(key: Sequence[int], n_rows: int, n_cols: int, std: float, dtype: str,
           rows: Optional[Iterable[int]] = None, mean: float = 0.0) -> np.ndarray:
    """Seeded N(mean, std) matrix [n_rows x n_cols] in stored format.

    With ``rows`` given, only those rows are returned (in the given order),
    drawing only the chunks that hold them; the values equal the corresponding
    rows of the full matrix.
    """
    rpc = _rows_per_chunk(n_cols)
    n_chunks = (n_rows + rpc - 1) // rpc
    out_dtype = np.uint16 if dtype == BF16 else np.float32
    if rows is None:
        out = np.empty((n_rows, n_cols), dtype=out_dtype)

        def job(c: int) -> None:
            r0, r1 = c * rpc, min(n_rows, (c + 1) * rpc)
            out[r0:r1] = _draw_chunk(tuple(key) + (c,), (r1 - r0) * n_cols, std, mean,
                                     dtype).reshape(r1 - r0, n_cols)

        list(_pool().map(job, range(n_chunks)))
        return out
    rows = np.asarray(list(rows), dtype=np.int64)
    out = np.empty((len(rows), n_cols), dtype=out_dtype)
    for c in np.unique(rows // rpc):
        r0, r1 = int(c) * rpc, min(n_rows, (int(c) + 1) * rpc)
        chunk = _draw_chunk(tuple(key) + (int(c),), (r1 - r0) * n_cols, std, mean,
                            dtype).reshape(r1 - r0, n_cols)
        sel = np.nonzero(rows // rpc == c)[0]
        out[sel] = chunk[rows[sel] - r0]
    return out


def norm_inputs(cfg: Config, module: int = 0, seed: int = 0,
                rows: Optional[Iterable[int]] = None) -> Dict[str, np.ndarray]:
    """W, A, B, m of one module in stored format.  With ``rows``, W, B and m
    hold only those rows (A is always whole)."""
    mod = cfg.modules[module]
    base_key = (seed, cfg.index)
    if rows is not None:
        rows = list(rows)
    W = normal(base_key + (T_W, module), mod.d_out, mod.d_in, cfg.std_w, cfg.dtype, rows)
    A = normal(base_key + (T_A, module), cfg.r, mod.d_in, cfg.std_a(mod.d_in), cfg.dtype)
    B = normal(base_key + (T_B, module), mod.d_out, cfg.r, cfg.std_b, cfg.dtype, rows)
    z = normal(base_key + (T_M, module), mod.d_out, 1, 1.0, F32, rows).reshape(-1)
    w64 = to_f64(W, cfg.dtype)
    row_len = np.sqrt(np.einsum("ij,ij->i", w64, w64))
    m32 = (row_len * (1.0 + cfg.std_m_rel * z.astype(np.float64))).astype(np.float32)
    m = f32_to_bf16_bits(m32) if cfg.dtype == BF16 else m32
    return {"W": W, "A": A, "B": B, "m": m}


def compose_inputs(cfg: Config, module: int = 0, seed: int = 0,
                   tokens: Optional[int] = None) -> Dict[str, np.ndarray]:
    """base, lora [T x d_out] in stored format; plus g (fp32) when the config
    draws g directly instead of taking it from the norm."""
    mod = cfg.modules[module]
    T = cfg.tokens if tokens is None else tokens
    base_key = (seed, cfg.index)
    out = {
        "base": normal(base_key + (T_BASE, module), T, mod.d_out, cfg.std_base, cfg.dtype),
        "lora": normal(base_key + (T_LORA, module), T, mod.d_out, cfg.std_lora, cfg.dtype),
    }
    if cfg.g_mode == "synthetic":
        out["g"] = normal(base_key + (T_G, module), 1, mod.d_out, cfg.g_std, F32,
                          mean=1.0).reshape(-1)
    return out


def grad_inputs(cfg: Config, module: int = 0, seed: int = 0,
                tokens: Optional[int] = None) -> np.ndarray:
    """Upstream gradient d out [T x d_out] of the compose, in stored format,
    N(0, cfg.std_grad)."""
    mod = cfg.modules[module]
    T = cfg.tokens if tokens is None else tokens
    return normal((seed, cfg.index, T_DOUT, module), T, mod.d_out, cfg.std_grad, cfg.dtype)


def stack_inputs_shared_w(cfg: Config, module: int, W: np.ndarray, w_row_len: np.ndarray,
                          seed: int = 0) -> Dict[str, np.ndarray]:
    """W, A, B, m of stack module ``module`` when its frozen weight is the
    stored W of another module of the same shape (drawn once, passed in with
    its float64 row lengths ``w_row_len``).  A, B and the magnitude noise z
    come from ``module``'s own Philox keys, and m is built as in
    :func:`norm_inputs` (``||W_j|| * (1 + 0.0015 z_j)`` in W's dtype), so
    modules that share W still differ in every adapter tensor.  This keeps a
    whole 196-module stack cheap to draw for a parity test."""
    mod = cfg.modules[module]
    assert W.shape == (mod.d_out, mod.d_in) and w_row_len.shape == (mod.d_out,)
    base_key = (seed, cfg.index)
    A = normal(base_key + (T_A, module), cfg.r, mod.d_in, cfg.std_a(mod.d_in), cfg.dtype)
    B = normal(base_key + (T_B, module), mod.d_out, cfg.r, cfg.std_b, cfg.dtype)
    z = normal(base_key + (T_M, module), mod.d_out, 1, 1.0, F32).reshape(-1)
    m32 = (w_row_len * (1.0 + cfg.std_m_rel * z.astype(np.float64))).astype(np.float32)
    m = f32_to_bf16_bits(m32) if cfg.dtype == BF16 else m32
    return {"W": W, "A": A, "B": B, "m": m}


def row_lengths(W: np.ndarray, dtype: str) -> np.ndarray:
    """float64 Euclidean length of every row of a stored matrix (input
    construction of m)."""
    w64 = to_f64(W, dtype)
    return np.sqrt(np.einsum("ij,ij->i", w64, w64))
