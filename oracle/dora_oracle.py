"""Plain, slow, obviously correct CPU oracle for the DoRA per-module hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library in ``dora_parameter_efficient_gb300`` never imports, links
or calls it, and shares no code with it.

Everything is evaluated in float64 from the stored input values, decoded
exactly.  The sources are the two write-ups of "Scaling DoRA: High-Rank
Adaptation via Factored Norms and Fused Kernels" (Zelenin, Zhuravlyova):

* the DoRA weight ``W' = m * (W + sBA) / ||W + sBA||_row`` -- English summary,
  "The Problem"; Chinese write-up section 1.1.  The row norm is taken over d_in
  for each of the d_out output rows.  The oracle evaluates that definition
  directly: it forms each row of ``W + s*B*A`` densely and takes its Euclidean
  length.  It deliberately does NOT use the factored decomposition (base +
  cross + BA-norm terms) that the GPU path uses; the tests pin the two against
  each other only through exact rational arithmetic on tiny inputs.
* the magnitude scale ``g = m / max(wnorm, eps)`` -- Chinese write-up section
  1.2.2 (the clamp before the divide).  The pages call eps "dtype dependent"
  without a value; here it is an explicit argument.
* the stable compose ``out = (g - 1) * base + g * (s * lora)`` -- Chinese
  write-up sections 2.1 and 2.1.1; English summary, "Fused Kernels".  g is one
  value per output feature and broadcasts along the token axis.  The naive
  algebraic twin ``g * (s * lora + base) - base`` (section 2.1.1, the form that
  cancels catastrophically near g = 1) is provided only as a comparator.
* rounding of a float64 result to the stored dtype: IEEE 754
  roundTiesToEven, done once, directly from float64.

The d_in-sharded form of the norm (each term of the factored norm is a sum
over d_in, so devices holding column slices add their shares; section 1.2.1)
is given by ``norm_partials`` and ``norm_from_partials``.

Each function names the passage it follows.  No function here is "parity
unpinned": ``tests/test_oracle_pins.py`` checks every one against exact
rational arithmetic, closed forms or hand-worked fixtures.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np

BF16 = "bf16"
F32 = "f32"


# ---------------------------------------------------------------- decoding
def decode(stored: np.ndarray, dtype: str) -> np.ndarray:
    """Stored tensor -> float64, exactly.

    bf16 is a bit pattern in uint16: the float32 with those 16 bits on top and
    zeros below has exactly the bf16 value."""
    if dtype == BF16:
        bits = np.asarray(stored, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == F32:
        return np.asarray(stored, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------- rounding
def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit pattern, one roundTiesToEven step.

    bf16 has 8 significant bits.  For |x| in [2^e, 2^(e+1)) the spacing is
    2^(e-7); below the smallest normal (2^-126) the spacing is fixed at the
    subnormal quantum 2^-133.  x / spacing is exact (a power-of-two scale), and
    numpy.rint rounds half to even."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    ax = np.abs(np.where(finite, x, 0.0))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    # guard log2 rounding at exact powers of two
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -126.0)
    q = np.ldexp(1.0, (e - 7).astype(np.int64))
    out[finite] = (np.rint(x[finite] / q[finite]) * q[finite])
    out[~finite] = x[~finite]
    # the rounded value has <= 8 significant bits, so float32 holds it exactly
    # (values beyond the bf16 range become inf here, as roundTiesToEven says)
    with np.errstate(over="ignore"):
        f = out.astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> stored dtype (bf16 bits or float32), one RNE rounding."""
    if dtype == BF16:
        return round_to_bf16_bits(x)
    if dtype == F32:
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    raise ValueError(dtype)


# ---------------------------------------------------------------- the norm
def row_norm(W: np.ndarray, A: np.ndarray, B: np.ndarray, s: float) -> np.ndarray:
    """wnorm_j = || W_j + s * (B A)_j ||_2 for every output row j.

    DoRA weight definition ("Scaling DoRA", English summary "The Problem";
    Chinese write-up section 1.1).  Dense: the full row W_j + s*B_j*A is formed
    (one float64 matrix product, B @ A), squared and summed along d_in."""
    W = np.asarray(W, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    V = W + float(s) * (B @ A)
    return np.sqrt(np.sum(V * V, axis=1))


def magnitude_scale(m: np.ndarray, wnorm: np.ndarray, eps: float) -> np.ndarray:
    """g_j = m_j / max(wnorm_j, eps)  (Chinese write-up section 1.2.2)."""
    m = np.asarray(m, dtype=np.float64)
    return m / np.maximum(np.asarray(wnorm, dtype=np.float64), float(eps))


def norm_and_scale(W, A, B, m, s: float, eps: float, dtype: str
                   ) -> Tuple[np.ndarray, np.ndarray]:
    """Stored W [d_out x d_in], A [r x d_in], B [d_out x r], m [d_out] ->
    (wnorm, g) in float64.  Rows of W, B and m may be any subset of the
    module's rows: every row is independent."""
    wnorm = row_norm(decode(W, dtype), decode(A, dtype), decode(B, dtype), s)
    return wnorm, magnitude_scale(decode(m, dtype), wnorm, eps)


# ---------------------------------------------------------------- d_in-sharded norm
# Every term of the factored norm is a sum over the d_in columns (Chinese
# write-up section 1.2.1; Algorithm 1 of section 5.1, steps 4a-f accumulate
# them chunk by chunk over d_in): ||W_j||^2, rowsum(B o U)_j with U = W A^T,
# and G = A A^T.  A device holding only the columns [k0, k1) of W and A can
# form its share of each; the shares add up to the whole.  These functions
# state the three sums by their definitions and apply the identity of
# section 1.2.1 to summed shares; tests/test_oracle_pins.py pins them to the
# dense norm above with exact rational arithmetic.
def norm_partials(W: np.ndarray, A: np.ndarray, B: np.ndarray):
    """(base, cross, G) of the columns of W [d_out x k] and A [r x k], float64:
    base_j = sum_k W_jk^2;  cross_j = sum_l B_jl * sum_k W_jk A_lk;
    G_lm = sum_k A_lk A_mk."""
    W = np.asarray(W, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    base = np.sum(W * W, axis=1)
    U = W @ A.T
    cross = np.sum(B * U, axis=1)
    G = A @ A.T
    return base, cross, G


def norm_from_partials(base: np.ndarray, cross: np.ndarray, G: np.ndarray, B: np.ndarray,
                       s: float) -> np.ndarray:
    """wnorm_j = sqrt(max(base_j + 2 s cross_j + s^2 B_j G B_j^T, 0)) from shares
    summed over all of d_in (section 1.2.1's three terms; the clamp of section
    1.2.2), float64."""
    B = np.asarray(B, dtype=np.float64)
    ba = np.sum((B @ np.asarray(G, dtype=np.float64)) * B, axis=1)
    w2 = np.asarray(base, np.float64) + 2.0 * float(s) * np.asarray(cross, np.float64) \
        + float(s) * float(s) * ba
    return np.sqrt(np.maximum(w2, 0.0))


# ---------------------------------------------------------------- the compose
def compose(base: np.ndarray, lora: np.ndarray, g: np.ndarray, s: float) -> np.ndarray:
    """out_ij = (g_j - 1) * base_ij + g_j * (s * lora_ij), float64.

    Stable compose of the Chinese write-up sections 2.1 / 2.1.1 (and the
    English summary, "Fused Kernels").  base and lora are [T x d_out]; g is
    [d_out], one scale per output feature, broadcast over the T rows."""
    base = np.asarray(base, dtype=np.float64)
    lora = np.asarray(lora, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)[None, :]
    return (g - 1.0) * base + g * (float(s) * lora)


def compose_stored(base, lora, g, s: float, dtype: str) -> np.ndarray:
    """Stored base/lora + float32 g -> the float64 compose, rounded once to
    the stored dtype."""
    return round_to(compose(decode(base, dtype), decode(lora, dtype),
                            np.asarray(g, dtype=np.float32), s), dtype)


def naive_compose_f32(base32: np.ndarray, lora32: np.ndarray, g32: np.ndarray,
                      s: float) -> np.ndarray:
    """Comparator only: g * (s * lora + base) - base with every operation
    rounded to float32 -- the algebraically equal form the Chinese write-up
    (section 2.1.1) warns cancels catastrophically when g is close to 1."""
    base32 = np.asarray(base32, dtype=np.float32)
    lora32 = np.asarray(lora32, dtype=np.float32)
    g32 = np.asarray(g32, dtype=np.float32)[None, :]
    t = np.float32(s) * lora32
    t = t + base32
    t = g32 * t
    return t - base32


# ---------------------------------------------------------------- training path of the compose
# The Chinese write-up (sections 2.2, 4.2 and 5.2) describes the training
# tier of the compose: the forward also keeps `inner`, one activation-sized
# tensor, for the magnitude gradient; the backward is a dual-output kernel
# (the gradients of the base and adapter branches) and dmag is a separate,
# deterministic column reduction, skipped when the magnitude is frozen.  The
# norm is a detached constant in the backward (section 1.2.2, following the
# DoRA paper), so g = m / max(wnorm, eps) depends on m alone.  The functions
# below are the plain derivatives of compose() under that reading.
def compose_inner(base: np.ndarray, lora: np.ndarray, s: float) -> np.ndarray:
    """inner_ij = base_ij + s * lora_ij, float64: d out_ij / d g_j of
    out = (g - 1) * base + g * (s * lora)."""
    return np.asarray(base, dtype=np.float64) + float(s) * np.asarray(lora, dtype=np.float64)


def compose_inner_stored(base, lora, s: float, dtype: str) -> np.ndarray:
    """Stored base/lora -> inner rounded once to the stored dtype."""
    return round_to(compose_inner(decode(base, dtype), decode(lora, dtype), s), dtype)


def compose_backward(d_out: np.ndarray, g: np.ndarray, s: float):
    """Gradients of out = (g - 1) * base + g * (s * lora) with respect to the
    two activations, float64: d_base = (g - 1) * d_out, d_lora = g * s * d_out
    (g broadcast over the T rows)."""
    d_out = np.asarray(d_out, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)[None, :]
    return (g - 1.0) * d_out, g * float(s) * d_out


def compose_backward_stored(d_out, g, s: float, dtype: str):
    """Stored d_out + float32 g -> (d_base, d_lora), each rounded once to dtype."""
    d_base, d_lora = compose_backward(decode(d_out, dtype), np.asarray(g, dtype=np.float32), s)
    return round_to(d_base, dtype), round_to(d_lora, dtype)


def magnitude_grad(d_out: np.ndarray, inner: np.ndarray, wnorm: np.ndarray,
                   eps: float) -> np.ndarray:
    """dL/dm_j = sum_t d_out_tj * inner_tj / max(wnorm_j, eps), float64 [d_out]
    (the chain rule through g_j = m_j / max(wnorm_j, eps) with wnorm constant)."""
    d_out = np.asarray(d_out, dtype=np.float64)
    inner = np.asarray(inner, dtype=np.float64)
    col = np.sum(d_out * inner, axis=0)
    return col / np.maximum(np.asarray(wnorm, dtype=np.float64), float(eps))


def magnitude_grad_stored(d_out, inner, wnorm, eps: float, dtype: str) -> np.ndarray:
    """Stored d_out / inner + float32 wnorm -> dm in float64."""
    return magnitude_grad(decode(d_out, dtype), decode(inner, dtype),
                          np.asarray(wnorm, dtype=np.float32), float(np.float32(eps)))


# ---------------------------------------------------------------- memory facts
def dense_ba_bytes(d_out: int, d_in: int, elem_bytes: int) -> int:
    """Bytes of the dense [d_out x d_in] product B*A that the factored norm
    never forms (Chinese write-up section 1.3, Table 1)."""
    return d_out * d_in * elem_bytes


def factored_intermediate_bytes(d_out: int, r: int, elem_bytes: int) -> int:
    """Bytes of the factored intermediates U [d_out x r] and G [r x r]
    (Chinese write-up section 1.3, Table 1)."""
    return (d_out * r + r * r) * elem_bytes
