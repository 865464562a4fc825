"""GPU parity of the grouped calls (one launch sequence for a stack of
modules) against the float64 oracle and against the per-module calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import COMPOSE_MAX_ULP, NORM_RTOL, rel_err, to_dev, to_host_stored, ulp_distance

pytestmark = pytest.mark.gpu


def _sample_rows(d_out, n=256, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(min(32, d_out))) | set(range(max(0, d_out - 32), d_out))
    rows |= set(rng.choice(d_out, size=min(n, d_out), replace=False).tolist())
    return np.array(sorted(rows))


def _dev_module(x, dtype):
    return tuple(to_dev(x[k], dtype) for k in ("W", "A", "B", "m"))


def _check_norm(cfg, x, wn, g, rows):
    wn_ref, g_ref = oracle.norm_and_scale(x["W"][rows], x["A"], x["B"][rows], x["m"][rows],
                                          cfg.s, float(np.float32(cfg.eps)), cfg.dtype)
    tol = NORM_RTOL[cfg.dtype]
    assert rel_err(wn[rows], wn_ref).max() <= tol
    assert rel_err(g[rows], g_ref).max() <= tol


def test_stack_layer_grouped_norm():
    """The seven modules of one layer of the 7B-like stack in one grouped call."""
    cfg = configs.get(4)
    xs = [gen.norm_inputs(cfg, module=k) for k in range(7)]
    mods = [_dev_module(x, cfg.dtype) for x in xs]
    wns, gs = api.dora_factored_norm_grouped(mods, cfg.s, cfg.eps)
    torch.cuda.synchronize()
    for k, x in enumerate(xs):
        rows = _sample_rows(cfg.modules[k].d_out, seed=k)
        _check_norm(cfg, x, wns[k].cpu().numpy(), gs[k].cpu().numpy(), rows)
        # and close to the per-module call (same arithmetic, K segments may differ)
        wn1, g1 = api.dora_factored_norm(*mods[k][:3], cfg.s, mods[k][3], cfg.eps)
        assert rel_err(wns[k].cpu().numpy(), wn1.cpu().numpy()).max() <= 2e-6


def test_full_stack_plan_every_module_sampled_rows():
    """All 196 modules of the 7B-like stack (r = 128) in one grouped plan run,
    four seeded rows of every module against the oracle.  The 28 layers share
    the seven layer-0 weights W (read-only, the same buffers), while A, B and
    m are drawn per module, so a work item mapped to the wrong module of its
    shape class, or a wrong per-module table entry, still changes the result
    (Chinese write-up sections 2.2 and 4.2: the stack of small projections)."""
    cfg = configs.get(4)
    n = len(cfg.modules)
    assert n == 196
    shared = {}
    for k in range(7):
        W = gen.norm_inputs(cfg, module=k)["W"]
        shared[k] = (W, gen.row_lengths(W, cfg.dtype), to_dev(W, cfg.dtype))
    xs, mods, rows = [], [], []
    rng = np.random.default_rng(196)
    for k in range(n):
        W, row_len, W_dev = shared[k % 7]
        x = gen.stack_inputs_shared_w(cfg, k, W, row_len)
        d_out = cfg.modules[k].d_out
        xs.append(x)
        mods.append((W_dev, to_dev(x["A"], cfg.dtype), to_dev(x["B"], cfg.dtype),
                     to_dev(x["m"], cfg.dtype)))
        rows.append(np.unique(np.concatenate([[0, d_out - 1], rng.choice(d_out, 2, replace=False)])))
    ws = torch.empty(api.norm_grouped_workspace_size(mods, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    plan = api.dora_norm_grouped_plan_create(mods, workspace=ws)
    try:
        for _ in range(2):          # two runs of the same plan: the second starts from the first's state
            plan.run(cfg.s, cfg.eps)
        torch.cuda.synchronize()
        assert api.dora_check_status(ws) == 0
        for k in range(n):
            wn = plan.wnorms[k].cpu().numpy()
            g = plan.gs[k].cpu().numpy()
            _check_norm(cfg, xs[k], wn, g, rows[k])
    finally:
        plan.destroy()


def _mixed(dtype, r, s, shapes, seed=0):
    out = []
    for i, (d_out, d_in) in enumerate(shapes):
        cfg = configs.Config(f"g{i}", 20 + i, dtype, (configs.Module(f"g{i}", d_out, d_in),), r=r,
                             s=s, eps=1e-6, tokens=8)
        out.append((cfg, gen.norm_inputs(cfg, seed=seed)))
    return out


@pytest.mark.parametrize("dtype,r,s", [(configs.BF16, 40, 1.5), (configs.BF16, 384, 1.0),
                                       (configs.BF16, 128, -0.5), (configs.F32, 24, 2.0),
                                       (configs.BF16, 64, 0.0)])
def test_mixed_shapes_group(dtype, r, s):
    shapes = [(200, 136), (129, 64), (1, 8), (640, 1000), (256, 512), (70, 2048)]
    if dtype == configs.F32:
        shapes = [(200, 136), (65, 36), (33, 100)]
    group = _mixed(dtype, r, s, shapes)
    mods = [_dev_module(x, dtype) for _, x in group]
    wns, gs = api.dora_factored_norm_grouped(mods, s, 1e-6)
    torch.cuda.synchronize()
    for (cfg, x), wn, g in zip(group, wns, gs):
        _check_norm(cfg, x, wn.cpu().numpy(), g.cpu().numpy(), np.arange(cfg.module.d_out))


def test_group_with_empty_module_and_repeat_calls():
    group = _mixed(configs.BF16, 32, 1.0, [(300, 256), (0, 256), (128, 64)])
    mods = [_dev_module(x, configs.BF16) for _, x in group]
    ws = torch.empty(api.norm_grouped_workspace_size(mods, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    first = None
    for _ in range(3):     # the workspace is reused: every call must start from its own state
        wns, gs = api.dora_factored_norm_grouped(mods, 1.0, 1e-6, workspace=ws)
        torch.cuda.synchronize()
        cur = [w.cpu().numpy().copy() for w in wns]
        if first is None:
            first = cur
        for a, b in zip(first, cur):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for (cfg, x), wn, g in zip(group, wns, gs):
        if cfg.module.d_out:
            _check_norm(cfg, x, wn.cpu().numpy(), g.cpu().numpy(), np.arange(cfg.module.d_out))


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_grouped_compose_matches_oracle_and_single_calls(dtype):
    cfg4 = configs.get(4)
    mods, refs = [], []
    for k in range(7):
        d_out = cfg4.modules[k].d_out
        cfg = configs.Config("gc", 4, dtype, cfg4.modules, r=8, s=cfg4.s, eps=1e-6, tokens=48,
                             g_mode="synthetic")
        c = gen.compose_inputs(cfg, module=k, tokens=48 + 3 * k)
        g32 = c["g"].astype(np.float32)
        mods.append((to_dev(c["base"], dtype), to_dev(c["lora"], dtype), torch.from_numpy(g32).cuda()))
        refs.append(oracle.compose_stored(c["base"], c["lora"], g32, cfg.s, dtype))
    outs = api.dora_compose_grouped(mods, cfg4.s)
    torch.cuda.synchronize()
    for (b, l, g), out, ref in zip(mods, outs, refs):
        got = to_host_stored(out)
        assert ulp_distance(got, ref, dtype).max() <= COMPOSE_MAX_ULP[dtype]
        single = to_host_stored(api.dora_compose(b, l, g, cfg4.s))
        assert np.array_equal(got, single)


def test_grouped_compose_misaligned_falls_back():
    cfg = configs.Config("gm", 0, configs.BF16, (configs.Module("gm", 37, 8),), r=8, s=1.5,
                         eps=1e-6, tokens=9)
    c = gen.compose_inputs(cfg)
    g32 = (1.0 + 0.01 * np.random.default_rng(0).standard_normal(37)).astype(np.float32)
    mods = [(to_dev(c["base"], cfg.dtype), to_dev(c["lora"], cfg.dtype), torch.from_numpy(g32).cuda())]
    out = api.dora_compose_grouped(mods, cfg.s)[0]
    ref = oracle.compose_stored(c["base"], c["lora"], g32, cfg.s, cfg.dtype)
    assert ulp_distance(to_host_stored(out), ref, cfg.dtype).max() <= 1


def _bits(ts):
    return [t.cpu().numpy().view(np.uint32).copy() for t in ts]


def test_plan_matches_grouped_call_across_in_place_updates():
    """A plan created once gives, run after run, the grouped call's bits, also
    after W, A, B and m are rewritten in place (the training-loop use)."""
    cfg = configs.get(4)
    xs = [gen.norm_inputs(cfg, module=k) for k in range(7)]
    mods = [_dev_module(x, cfg.dtype) for x in xs]
    plan = api.dora_norm_grouped_plan_create(mods)
    for step in range(3):
        if step:
            xs = [gen.norm_inputs(cfg, module=k, seed=step) for k in range(7)]
            for dst, x in zip(mods, xs):
                for t, src in zip(dst, _dev_module(x, cfg.dtype)):
                    t.copy_(src)
        wns, gs = plan.run(cfg.s, cfg.eps)
        got_w, got_g = _bits(wns), _bits(gs)
        ref_w, ref_g = api.dora_factored_norm_grouped(mods, cfg.s, cfg.eps)
        torch.cuda.synchronize()
        for a, b in zip(got_w + got_g, _bits(ref_w) + _bits(ref_g)):
            assert np.array_equal(a, b)
    for k, x in enumerate(xs):
        rows = _sample_rows(cfg.modules[k].d_out, n=64, seed=k)
        _check_norm(cfg, x, plan.wnorms[k].cpu().numpy(), plan.gs[k].cpu().numpy(), rows)
    plan.destroy()


def test_plan_per_module_fallback_keeps_tables():
    """s = 0 takes the per-module path through the same workspace; the next
    s != 0 run must still find the one-launch tables intact."""
    group = _mixed(configs.BF16, 48, 1.25, [(300, 256), (129, 64), (512, 1024)])
    mods = [_dev_module(x, configs.BF16) for _, x in group]
    plan = api.dora_norm_grouped_plan_create(mods)
    for s in (1.25, 0.0, 1.25, -0.75):
        wns, gs = plan.run(s, 1e-6)
        torch.cuda.synchronize()
        for (cfg, x), wn, g in zip(group, wns, gs):
            c = configs.Config(cfg.name, cfg.index, cfg.dtype, cfg.modules, r=cfg.r, s=s,
                               eps=cfg.eps, tokens=cfg.tokens)
            _check_norm(c, x, wn.cpu().numpy(), g.cpu().numpy(), np.arange(cfg.module.d_out))
    plan.destroy()


def test_plan_f32_group():
    group = _mixed(configs.F32, 24, 2.0, [(200, 136), (65, 36)])
    mods = [_dev_module(x, configs.F32) for _, x in group]
    plan = api.dora_norm_grouped_plan_create(mods)
    wns, gs = plan.run(2.0, 1e-6)
    torch.cuda.synchronize()
    for (cfg, x), wn, g in zip(group, wns, gs):
        _check_norm(cfg, x, wn.cpu().numpy(), g.cpu().numpy(), np.arange(cfg.module.d_out))
    plan.destroy()


def test_many_modules_whole_k_items():
    """Enough pair tiles to fill the persistent grid several times over: every
    module runs as whole-K items, numbered longest K first."""
    rng = np.random.default_rng(5)
    shapes = [(int(rng.choice([512, 1000, 2048, 2304])), int(rng.choice([64, 200, 512, 1024, 1536])))
              for _ in range(80)]
    # four waves of the 76 CTA pairs of a 152-SM part
    assert sum((d + 255) // 256 for d, _ in shapes) >= 4 * 76
    group = _mixed(configs.BF16, 32, 0.75, shapes, seed=3)
    mods = [_dev_module(x, configs.BF16) for _, x in group]
    plan = api.dora_norm_grouped_plan_create(mods)
    wns, gs = plan.run(0.75, 1e-6)
    torch.cuda.synchronize()
    for k, ((cfg, x), wn, g) in enumerate(zip(group, wns, gs)):
        rows = _sample_rows(cfg.module.d_out, n=32, seed=k)
        _check_norm(cfg, x, wn.cpu().numpy(), g.cpu().numpy(), rows)
    for k in (0, 17, 79):
        wn1, _ = api.dora_factored_norm(*mods[k][:3], 0.75, mods[k][3], 1e-6)
        assert rel_err(wns[k].cpu().numpy(), wn1.cpu().numpy()).max() <= 2e-6
    plan.destroy()


def test_more_modules_than_the_shared_memory_cache():
    """2100 modules: more than the main pass keeps in shared memory, so the
    item -> module search reads the module table in global memory."""
    n = 2100
    cfg = configs.Config("many", 60, configs.BF16, (configs.Module("many", 256, 64),), r=16,
                         s=1.0, eps=1e-6, tokens=8)
    x = gen.norm_inputs(cfg, seed=9)
    base = _dev_module(x, configs.BF16)
    # distinct modules: each a copy scaled by a power of two (exact in bf16),
    # so every result follows from the first module's (the norm is homogeneous
    # of degree 1 in W and B; g = m / wnorm with m scaled alike is unchanged)
    scales = [2.0 ** ((i % 5) - 2) for i in range(n)]
    mods = [(base[0] * sc, base[1], base[2] * sc, base[3] * sc) for sc in scales]
    plan = api.dora_norm_grouped_plan_create(mods)
    wns, gs = plan.run(cfg.s, cfg.eps)
    torch.cuda.synchronize()
    wn_ref, g_ref = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s,
                                          float(np.float32(cfg.eps)), cfg.dtype)
    for i in (0, 1, 777, 2047, 2048, 2099):
        assert rel_err(wns[i].cpu().numpy() / scales[i], wn_ref).max() <= NORM_RTOL[cfg.dtype]
        assert rel_err(gs[i].cpu().numpy(), g_ref).max() <= NORM_RTOL[cfg.dtype]
    plan.destroy()
