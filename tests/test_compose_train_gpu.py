"""GPU parity of the training path of the compose (dora_compose_train and
dora_compose_backward) against the float64 oracle.

Inputs: the configs' compose activations, the upstream gradient from
gen.grad_inputs, g from the oracle's norm (configs 0-2) or the config's
synthetic draw (configs 3-4), and wnorm from the oracle (or a synthetic
positive vector where only its use as a divisor matters).  The oracle's
inner (rounded to the stored dtype) feeds both sides of the dmag check, so
no oracle input comes from the GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import COMPOSE_MAX_ULP, DM_RTOL, to_dev, to_host_stored, ulp_distance

pytestmark = pytest.mark.gpu


def _norm_for(cfg, module=0):
    """(g, wnorm) as fp32: the oracle's, or synthetic g with a matching wnorm."""
    c = gen.compose_inputs(cfg, module=module, tokens=1)
    d_out = cfg.modules[module].d_out
    if "g" in c:
        wn = 1.0 + np.abs(gen.normal((7, cfg.index, module), 1, d_out, 0.5, configs.F32).reshape(-1))
        return c["g"].astype(np.float32), wn.astype(np.float32)
    x = gen.norm_inputs(cfg, module=module)
    wn, g = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s,
                                  float(np.float32(cfg.eps)), cfg.dtype)
    return g.astype(np.float32), wn.astype(np.float32)


def _check_ulp(got, ref, dtype, what):
    d = ulp_distance(got, ref, dtype)
    assert d.max() <= COMPOSE_MAX_ULP[dtype], (
        f"{what}: {d.max()} ulp at {np.unravel_index(d.argmax(), d.shape)}")


def _check_dm(got, d_out, inner, wnorm, eps, dtype):
    ref = oracle.magnitude_grad_stored(d_out, inner, wnorm, eps, dtype)
    absum = np.sum(np.abs(oracle.decode(d_out, dtype) * oracle.decode(inner, dtype)), axis=0)
    bound = DM_RTOL * absum / np.maximum(wnorm.astype(np.float64), float(np.float32(eps)))
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.all(err <= bound + 1e-30), f"dmag err {err.max()} vs bound at {err.argmax()}"


def _run_all(cfg, base, lora, d_out, g32, wn32, s, eps=1e-6, want_dm=True):
    dt = cfg.dtype
    out, inner = api.dora_compose_train(to_dev(base, dt), to_dev(lora, dt),
                                        torch.from_numpy(g32).cuda(), s)
    inner_ref = oracle.compose_inner_stored(base, lora, s, dt)
    db, dl, dm = api.dora_compose_backward(
        to_dev(d_out, dt), torch.from_numpy(g32).cuda(), s,
        inner=to_dev(inner_ref, dt) if want_dm else None,
        wnorm=torch.from_numpy(wn32).cuda() if want_dm else None, eps=eps)
    torch.cuda.synchronize()
    return (to_host_stored(out), to_host_stored(inner), to_host_stored(db), to_host_stored(dl),
            None if dm is None else dm.cpu().numpy(), inner_ref)


def _check_all(cfg, base, lora, d_out, g32, wn32, s, res, eps=1e-6):
    out, inner, db, dl, dm, inner_ref = res
    dt = cfg.dtype
    _check_ulp(out, oracle.compose_stored(base, lora, g32, s, dt), dt, "out")
    _check_ulp(inner, inner_ref, dt, "inner")
    rb, rl = oracle.compose_backward_stored(d_out, g32, s, dt)
    _check_ulp(db, rb, dt, "d_base")
    _check_ulp(dl, rl, dt, "d_lora")
    if dm is not None:
        _check_dm(dm, d_out, inner_ref, wn32, eps, dt)


@pytest.mark.parametrize("index", [0, 1, 2])
def test_config_full(index):
    cfg = configs.get(index)
    c = gen.compose_inputs(cfg)
    d_out = gen.grad_inputs(cfg)
    g32, wn32 = _norm_for(cfg)
    res = _run_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s)
    _check_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s, res)


@pytest.mark.parametrize("module", [0, 1, 4, 6])
def test_config4_stack_modules(module):
    cfg = configs.get(4)
    c = gen.compose_inputs(cfg, module=module, tokens=256)
    d_out = gen.grad_inputs(cfg, module=module, tokens=256)
    g32, wn32 = _norm_for(cfg, module)
    res = _run_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s)
    _check_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s, res)


def _edge(dtype, T, d, s=1.5):
    cfg = configs.Config("edge", 0, dtype, (configs.Module("edge", d, 8),), r=8, s=s, eps=1e-6,
                         tokens=T)
    c = gen.compose_inputs(cfg)
    d_out = gen.grad_inputs(cfg)
    rng = np.random.default_rng(T * 1000 + d)
    g32 = (1.0 + 0.01 * rng.standard_normal(d)).astype(np.float32)
    wn32 = (0.5 + rng.random(d)).astype(np.float32)
    wn32[0] = 1e-9            # below eps: divide by eps
    return cfg, c, d_out, g32, wn32


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
@pytest.mark.parametrize("T,d", [(1, 8), (7, 37), (33, 1), (5, 4100), (129, 24), (300, 2048),
                                 (1000, 64)])
def test_ragged_shapes(dtype, T, d):
    cfg, c, d_out, g32, wn32 = _edge(dtype, T, d)
    res = _run_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s)
    _check_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s, res)


def test_frozen_magnitude_skips_dmag():
    cfg, c, d_out, g32, wn32 = _edge(configs.BF16, 64, 256)
    res = _run_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s, want_dm=False)
    assert res[4] is None
    _check_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s, res)


def test_misaligned_rows_take_the_elementwise_kernels():
    cfg, c, d_out, g32, wn32 = _edge(configs.BF16, 16, 64)
    dt = cfg.dtype
    # the same values in a view that starts one element into its buffer:
    # not 16-byte aligned
    def shifted(a):
        t = to_dev(np.concatenate([a.reshape(-1)[:1], a.reshape(-1)]), dt)
        return t[1:].view(a.shape)
    dev_g = torch.from_numpy(g32).cuda()
    out, inner = api.dora_compose_train(shifted(c["base"]), shifted(c["lora"]), dev_g, cfg.s)
    inner_ref = oracle.compose_inner_stored(c["base"], c["lora"], cfg.s, dt)
    db, dl, dm = api.dora_compose_backward(shifted(d_out), dev_g, cfg.s,
                                           inner=shifted(inner_ref),
                                           wnorm=torch.from_numpy(wn32).cuda(), eps=1e-6)
    res = (to_host_stored(out), to_host_stored(inner), to_host_stored(db), to_host_stored(dl),
           dm.cpu().numpy(), inner_ref)
    _check_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s, res)


def test_g_one_and_zero_scale_closed_forms():
    cfg, c, d_out, _, wn32 = _edge(configs.BF16, 40, 512, s=2.0)
    ones = np.ones(512, np.float32)
    res = _run_all(cfg, c["base"], c["lora"], d_out, ones, wn32, 2.0)
    d32 = gen.bf16_bits_to_f32(d_out)
    assert np.all(gen.bf16_bits_to_f32(res[2]) == 0.0)                  # d_base = 0
    assert np.array_equal(res[3], gen.f32_to_bf16_bits(2.0 * d32))     # d_lora = 2 d_out
    res0 = _run_all(cfg, c["base"], c["lora"], d_out, ones, wn32, 0.0)
    assert np.all(gen.bf16_bits_to_f32(res0[3]) == 0.0)                 # s = 0: no adapter grad
    assert np.array_equal(res0[1], c["base"])                            # inner = base


def test_dmag_deterministic_across_calls():
    cfg, c, d_out, g32, wn32 = _edge(configs.BF16, 2048, 4096)
    a = _run_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s)
    b = _run_all(cfg, c["base"], c["lora"], d_out, g32, wn32, cfg.s)
    assert np.array_equal(a[4].view(np.uint32), b[4].view(np.uint32))
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
