"""Pins for the oracle's training-path compose (the forward's saved `inner`,
the dual-output backward and the magnitude gradient), against things other
than the oracle's own formulas:

* central finite differences of the scalar loss L = sum(d_out * out), with
  out from the oracle's forward compose and g = m / max(wnorm, eps) -- an
  independent route to every derivative (L is linear in m, base and lora, so
  the difference quotients are exact up to float64 rounding);
* closed forms: g = 1, s = 0, d_out = 0;
* small-integer inputs, where every float64 step is exact;
* the bf16 rounding of the stored outputs against the generator's
  independent round-to-nearest-even on float32 bits.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from synthetic import gen

RNG = np.random.default_rng(99)


def _loss(base, lora, m, wnorm, eps, s, d_out):
    g = m / np.maximum(wnorm, eps)
    return float(np.sum(d_out * oracle.compose(base, lora, g, s)))


@pytest.mark.parametrize("s", [1.0, -0.5, 2.0])
def test_backward_matches_finite_differences(s):
    T, d = 4, 6
    base = RNG.standard_normal((T, d))
    lora = RNG.standard_normal((T, d)) * 0.05
    d_out = RNG.standard_normal((T, d))
    wnorm = np.abs(RNG.standard_normal(d)) + 0.5
    wnorm[2] = 1e-9                       # below eps: the divisor is eps
    eps = 1e-6
    m = wnorm * (1.0 + 0.01 * RNG.standard_normal(d))
    m[2] = 3e-6
    g = m / np.maximum(wnorm, eps)
    d_base, d_lora = oracle.compose_backward(d_out, g, s)
    dm = oracle.magnitude_grad(d_out, oracle.compose_inner(base, lora, s), wnorm, eps)
    for j in range(d):
        h = 1e-6 * max(abs(m[j]), 1e-6)
        mp, mm = m.copy(), m.copy()
        mp[j] += h
        mm[j] -= h
        fd = (_loss(base, lora, mp, wnorm, eps, s, d_out) -
              _loss(base, lora, mm, wnorm, eps, s, d_out)) / (2 * h)
        assert fd == pytest.approx(dm[j], rel=1e-6, abs=1e-9 * np.sum(np.abs(d_out[:, j])) / eps)
    for t in range(T):
        for j in range(d):
            for arr, grad in ((base, d_base), (lora, d_lora)):
                h = 1e-3
                ap, am = arr.copy(), arr.copy()
                ap[t, j] += h
                am[t, j] -= h
                args_p = (ap, lora) if arr is base else (base, ap)
                args_m = (am, lora) if arr is base else (base, am)
                fd = (_loss(*args_p, m, wnorm, eps, s, d_out) -
                      _loss(*args_m, m, wnorm, eps, s, d_out)) / (2 * h)
                assert fd == pytest.approx(grad[t, j], rel=1e-7, abs=1e-12)


def test_backward_closed_forms():
    T, d = 5, 7
    d_out = RNG.standard_normal((T, d))
    base = RNG.standard_normal((T, d))
    lora = RNG.standard_normal((T, d))
    # g = 1: the base branch gets nothing, the adapter branch s * d_out
    d_base, d_lora = oracle.compose_backward(d_out, np.ones(d), 1.5)
    assert np.all(d_base == 0.0)
    assert np.array_equal(d_lora, 1.5 * d_out)
    # s = 0: no adapter gradient, inner is the base activation
    g = 1.0 + 0.01 * RNG.standard_normal(d)
    d_base, d_lora = oracle.compose_backward(d_out, g, 0.0)
    assert np.all(d_lora == 0.0)
    assert np.array_equal(oracle.compose_inner(base, lora, 0.0), base)
    # zero upstream gradient: every output is zero
    z = np.zeros((T, d))
    d_base, d_lora = oracle.compose_backward(z, g, 1.0)
    assert not d_base.any() and not d_lora.any()
    assert not oracle.magnitude_grad(z, base, np.ones(d), 1e-6).any()


def test_magnitude_grad_small_integers_exact():
    T, d = 64, 9
    d_out = RNG.integers(-3, 4, size=(T, d)).astype(np.float32)
    inner = RNG.integers(-3, 4, size=(T, d)).astype(np.float32)
    wnorm = (2.0 ** RNG.integers(-3, 4, size=d)).astype(np.float32)
    ds = gen.f32_to_bf16_bits(d_out)
    ins = gen.f32_to_bf16_bits(inner)
    dm = oracle.magnitude_grad_stored(ds, ins, wnorm, 1e-6, oracle.BF16)
    for j in range(d):
        exact = sum(int(d_out[t, j]) * int(inner[t, j]) for t in range(T))
        assert dm[j] == exact / float(wnorm[j])


def test_stored_backward_rounding():
    T, d = 33, 40
    d_out = (RNG.standard_normal((T, d)) * 0.1).astype(np.float32)
    ds = gen.f32_to_bf16_bits(d_out)
    d32 = gen.bf16_bits_to_f32(ds)
    # g = 1, s = 2: d_lora = 2 d_out exactly, d_base = 0
    db, dl = oracle.compose_backward_stored(ds, np.ones(d, np.float32), 2.0, oracle.BF16)
    assert np.array_equal(dl, gen.f32_to_bf16_bits(2.0 * d32))
    assert np.all(gen.bf16_bits_to_f32(db) == 0.0)
    # g = 0.5 exactly: both products exact in float32, one rounding to bf16
    g = np.full(d, 0.5, np.float32)
    db, dl = oracle.compose_backward_stored(ds, g, 1.0, oracle.BF16)
    assert np.array_equal(db, gen.f32_to_bf16_bits(np.float32(-0.5) * d32))
    assert np.array_equal(dl, gen.f32_to_bf16_bits(np.float32(0.5) * d32))
    # inner of bf16 values with s = 1 where base + lora is exact in float32
    base = gen.f32_to_bf16_bits(np.round(RNG.standard_normal((T, d)) * 8) / 8)
    lora = gen.f32_to_bf16_bits(np.round(RNG.standard_normal((T, d)) * 8) / 8)
    exact = gen.bf16_bits_to_f32(base) + gen.bf16_bits_to_f32(lora)
    assert np.array_equal(oracle.compose_inner_stored(base, lora, 1.0, oracle.BF16),
                          gen.f32_to_bf16_bits(exact))
