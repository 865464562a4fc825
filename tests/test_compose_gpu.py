"""GPU parity of dora_compose against the float64 oracle.

g for the compose is the oracle's g (configs 0-2, "g from the norm") or the
config's synthetic N(1, 0.0015) draw (configs 3-4), rounded to fp32; both
sides receive the same stored arrays."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import COMPOSE_MAX_ULP, to_dev, to_host_stored, ulp_distance

pytestmark = pytest.mark.gpu


def _g_for(cfg, module=0):
    c = gen.compose_inputs(cfg, module=module, tokens=1)
    if "g" in c:
        return c["g"].astype(np.float32)
    x = gen.norm_inputs(cfg, module=module)
    _, g = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s,
                                 float(np.float32(cfg.eps)), cfg.dtype)
    return g.astype(np.float32)


def _check_rows(cfg, base, lora, g32, got_stored, rows=None):
    if rows is not None:
        base, lora, got_stored = base[rows], lora[rows], got_stored[rows]
    ref = oracle.compose_stored(base, lora, g32, cfg.s, cfg.dtype)
    d = ulp_distance(got_stored, ref, cfg.dtype)
    assert d.max() <= COMPOSE_MAX_ULP[cfg.dtype], (
        f"{cfg.name}: {d.max()} ulp at {np.unravel_index(d.argmax(), d.shape)}")
    return ref


def _run(cfg, base, lora, g32, s=None):
    out = api.dora_compose(to_dev(base, cfg.dtype), to_dev(lora, cfg.dtype),
                           torch.from_numpy(g32).cuda(), cfg.s if s is None else s)
    return to_host_stored(out)


@pytest.mark.parametrize("index", [0, 1, 2])
def test_config_full(index):
    cfg = configs.get(index)
    c = gen.compose_inputs(cfg)
    g32 = _g_for(cfg)
    got = _run(cfg, c["base"], c["lora"], g32)
    _check_rows(cfg, c["base"], c["lora"], g32, got)


def _token_sample(T, n=256, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(min(16, T))) | set(range(max(0, T - 16), T))
    rows |= set(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(rows))


def test_config3_moe_sampled_tokens():
    cfg = configs.get(3)
    c = gen.compose_inputs(cfg)
    got = _run(cfg, c["base"], c["lora"], c["g"])
    _check_rows(cfg, c["base"], c["lora"], c["g"], got, rows=_token_sample(cfg.tokens))


@pytest.mark.parametrize("module", [0, 1, 4, 6])
def test_config4_stack_modules(module):
    cfg = configs.get(4)
    c = gen.compose_inputs(cfg, module=module)
    got = _run(cfg, c["base"], c["lora"], c["g"])
    _check_rows(cfg, c["base"], c["lora"], c["g"], got, rows=_token_sample(cfg.tokens, seed=module))


@pytest.mark.parametrize("index", [1, 3])
def test_no_worse_than_naive_near_one(index):
    """Against the fp64 oracle, the kernel's peak error is no larger than that
    of the naive g*(s*lora+base)-base evaluated in fp32 (Chinese write-up
    section 2.1.1), on the g ~ 1 distribution."""
    cfg = configs.get(index)
    T = 512
    c = gen.compose_inputs(cfg, tokens=T)
    g32 = c["g"] if "g" in c else _g_for(cfg)
    got = _run(cfg, c["base"], c["lora"], g32)
    base, lora = oracle.decode(c["base"], cfg.dtype), oracle.decode(c["lora"], cfg.dtype)
    exact = oracle.compose(base, lora, g32, cfg.s)
    naive = oracle.naive_compose_f32(base.astype(np.float32), lora.astype(np.float32), g32, cfg.s)
    naive_stored = oracle.round_to(naive.astype(np.float64), cfg.dtype)
    err_ours = np.abs(oracle.decode(got, cfg.dtype) - exact).max()
    err_naive = np.abs(oracle.decode(naive_stored, cfg.dtype) - exact).max()
    assert err_ours <= err_naive


# ------------------------------------------------------------------ edge cases
def _small(dtype, T, d, seed=0):
    cfg = configs.Config("edge", 0, dtype, (configs.Module("edge", d, 8),), r=8, s=1.5, eps=1e-6,
                         tokens=T, g_mode="synthetic", g_std=0.01)
    c = gen.compose_inputs(cfg, seed=seed)
    return cfg, c


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
@pytest.mark.parametrize("T,d", [(1, 8), (7, 37), (33, 1), (5, 4100), (129, 24)])
def test_ragged_shapes(dtype, T, d):
    cfg, c = _small(dtype, T, d)
    got = _run(cfg, c["base"], c["lora"], c["g"])
    _check_rows(cfg, c["base"], c["lora"], c["g"], got)


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_unaligned_pointers_take_scalar_path(dtype):
    cfg, c = _small(dtype, 9, 64)
    tdtype = torch.bfloat16 if dtype == configs.BF16 else torch.float32
    n = 9 * 64
    bufs = []
    for key in ("base", "lora"):
        big = torch.empty(n + 1, dtype=tdtype, device="cuda")
        big[1:].copy_(to_dev(c[key], dtype).reshape(-1))
        bufs.append(big[1:].view(9, 64))            # 2- or 4-byte offset: not 16-byte aligned
    out_big = torch.empty(n + 1, dtype=tdtype, device="cuda")
    out = out_big[1:].view(9, 64)
    api.dora_compose(bufs[0], bufs[1], torch.from_numpy(c["g"]).cuda(), cfg.s, out=out)
    _check_rows(cfg, c["base"], c["lora"], c["g"], to_host_stored(out))


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_in_place(dtype):
    cfg, c = _small(dtype, 64, 256)
    base = to_dev(c["base"], dtype)
    api.dora_compose(base, to_dev(c["lora"], dtype), torch.from_numpy(c["g"]).cuda(), cfg.s,
                     out=base)
    _check_rows(cfg, c["base"], c["lora"], c["g"], to_host_stored(base))


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_special_scales(dtype):
    cfg, c = _small(dtype, 16, 128)
    base, lora = c["base"], c["lora"]
    one = np.ones(128, np.float32)
    zero = np.zeros(128, np.float32)
    # g = 1: out = s * lora exactly for s = 2
    got = _run(cfg, base, lora, one, s=2.0)
    np.testing.assert_array_equal(got, oracle.round_to(2.0 * oracle.decode(lora, dtype), dtype))
    # g = 0: out = -base exactly
    got = _run(cfg, base, lora, zero, s=2.0)
    np.testing.assert_array_equal(oracle.decode(got, dtype), -oracle.decode(base, dtype))


def test_empty_tokens():
    base = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    out = api.dora_compose(base, base.clone(), torch.ones(64, device="cuda"), 1.0)
    assert out.shape == (0, 64)
