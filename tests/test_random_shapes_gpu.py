"""Seeded sweeps of shapes for the norm and the compose against the float64
oracle: odd row counts (ragged pair tiles), K tails, ranks from 8 to 512
(one or two N chunks, one or two fp32 N passes), scales including 0 and
negative values, both dtypes; every row (norm) or element (compose) checked."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import (COMPOSE_MAX_ULP, NORM_RTOL, rel_err, to_dev, to_host_stored,
                               ulp_distance)

pytestmark = pytest.mark.gpu


def _norm_shapes(n=14, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = configs.BF16 if i % 2 == 0 else configs.F32
        step = 8 if dtype == configs.BF16 else 4      # 16-byte rows
        d_out = int(rng.integers(1, 1600))
        d_in = int(rng.integers(1, 380)) * step
        r = int(rng.integers(1, 65)) * 8
        s = float(rng.choice([0.0, -0.75, 0.5, 1.0, 2.0]))
        out.append((dtype, d_out, d_in, r, s))
    return out


@pytest.mark.parametrize("dtype,d_out,d_in,r,s", _norm_shapes())
def test_norm_random_shape(dtype, d_out, d_in, r, s):
    cfg = configs.Config(f"rand-{dtype}-{d_out}x{d_in}-r{r}", 70 + d_out % 17, dtype,
                         (configs.Module("rand", d_out, d_in),), r=r, s=s, eps=1e-6, tokens=4)
    x = gen.norm_inputs(cfg, seed=d_in)
    W, A, B, m = (to_dev(x[k], dtype) for k in ("W", "A", "B", "m"))
    wn, g = api.dora_factored_norm(W, A, B, s, m, cfg.eps)
    wn_ref, g_ref = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], s,
                                          float(np.float32(cfg.eps)), dtype)
    tol = NORM_RTOL[dtype]
    assert rel_err(wn.cpu().numpy(), wn_ref).max() <= tol
    assert rel_err(g.cpu().numpy(), g_ref).max() <= tol


def _compose_shapes(n=10, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = configs.BF16 if i % 2 == 0 else configs.F32
        T = int(rng.integers(1, 300))
        d_out = int(rng.choice([int(rng.integers(1, 3000)), 2048 * int(rng.integers(1, 3))]))
        s = float(rng.choice([0.0, 0.5, 1.0, 2.0, -1.25]))
        out.append((dtype, T, d_out, s))
    return out


@pytest.mark.parametrize("dtype,T,d_out,s", _compose_shapes())
def test_compose_random_shape(dtype, T, d_out, s):
    cfg = configs.Config(f"randc-{dtype}-{T}x{d_out}", 90 + T % 13, dtype,
                         (configs.Module("randc", d_out, 8),), r=8, s=s, eps=1e-6, tokens=T,
                         g_mode="synthetic")
    c = gen.compose_inputs(cfg, seed=d_out)
    g32 = c["g"].astype(np.float32)
    import torch
    out = api.dora_compose(to_dev(c["base"], dtype), to_dev(c["lora"], dtype),
                           torch.from_numpy(g32).cuda(), s)
    ref = oracle.compose_stored(c["base"], c["lora"], g32, s, dtype)
    assert ulp_distance(to_host_stored(out), ref, dtype).max() <= COMPOSE_MAX_ULP[dtype]
