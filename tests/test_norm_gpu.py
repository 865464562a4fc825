"""GPU parity of dora_factored_norm against the float64 oracle.

Every call goes through the C ABI (the ctypes binding).  Inputs come from the
seeded generator; the oracle sees the same stored values.  Full-size configs
are checked on every row where the oracle finishes in seconds (8192 x 8192)
and on seeded row samples otherwise (rows are independent)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import NORM_RTOL, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _run(x, cfg, s=None, r=None):
    s = cfg.s if s is None else s
    dev = {k: to_dev(x[k], cfg.dtype) for k in ("W", "A", "B", "m")}
    ws = api.alloc_workspace(dev["W"].shape[0], dev["W"].shape[1], dev["A"].shape[0],
                             dev["W"].dtype)
    wn, g = api.dora_factored_norm(dev["W"], dev["A"], dev["B"], s, dev["m"], cfg.eps,
                                   workspace=ws)
    assert api.dora_check_status(ws) == 0
    return wn.cpu().numpy(), g.cpu().numpy()


def _oracle(x, cfg, s=None, rows=None):
    s = cfg.s if s is None else s
    W, B, m = x["W"], x["B"], x["m"]
    if rows is not None:
        W, B, m = W[rows], B[rows], m[rows]
    return oracle.norm_and_scale(W, x["A"], B, m, s, float(np.float32(cfg.eps)), cfg.dtype)


def _check(cfg, wn, g, wn_ref, g_ref):
    tol = NORM_RTOL[cfg.dtype]
    ew, eg = rel_err(wn, wn_ref), rel_err(g, g_ref)
    assert ew.max() <= tol, f"{cfg.name}: wnorm rel err {ew.max():.3e} at row {ew.argmax()}"
    assert eg.max() <= tol, f"{cfg.name}: g rel err {eg.max():.3e} at row {eg.argmax()}"


def _custom(name, dtype, d_out, d_in, r, s, index=0):
    return configs.Config(name, index, dtype, (configs.Module(name, d_out, d_in),), r=r, s=s,
                          eps=1e-6, tokens=16)


# ------------------------------------------------------------------ configs
@pytest.mark.parametrize("index", [0, 1, 2])
def test_config_full(index):
    cfg = configs.get(index)
    x = gen.norm_inputs(cfg)
    wn, g = _run(x, cfg)
    wn_ref, g_ref = _oracle(x, cfg)
    _check(cfg, wn, g, wn_ref, g_ref)


def _sample_rows(d_out, n=512, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(min(64, d_out))) | set(range(max(0, d_out - 64), d_out))
    rows |= set(rng.choice(d_out, size=min(n, d_out), replace=False).tolist())
    return np.array(sorted(rows))


def test_config3_moe_sampled_rows():
    cfg = configs.get(3)
    x = gen.norm_inputs(cfg)
    wn, g = _run(x, cfg)
    rows = _sample_rows(cfg.module.d_out)
    wn_ref, g_ref = _oracle(x, cfg, rows=rows)
    _check(cfg, wn[rows], g[rows], wn_ref, g_ref)


@pytest.mark.parametrize("module", range(7))
def test_config4_stack_layer0_sampled_rows(module):
    """One full layer of the 7B-like stack: q, k, v, o, gate, up, down shapes."""
    cfg = configs.get(4)
    x = gen.norm_inputs(cfg, module=module)
    wn, g = _run(x, cfg)
    rows = _sample_rows(cfg.modules[module].d_out, n=256, seed=module)
    wn_ref, g_ref = _oracle(x, cfg, rows=rows)
    _check(cfg, wn[rows], g[rows], wn_ref, g_ref)


# ------------------------------------------------------------------ ragged and edge shapes
@pytest.mark.parametrize("dtype,d_out,d_in,r,s", [
    (configs.BF16, 200, 136, 24, 1.5),       # ragged rows, K tail of 8, N padded 24 -> 32
    (configs.BF16, 129, 64, 8, 2.0),         # one row past a tile, r = 8 (N padded to 16)
    (configs.BF16, 1, 8, 8, 1.0),            # single row, single short K tile
    (configs.BF16, 300, 1000, 16, -0.5),     # negative scale
    (configs.BF16, 130, 520, 200, 1.0),      # N = 208 in one MMA
    (configs.BF16, 256, 512, 264, 1.0),      # N = 272: two MMAs (256 + 16)
    (configs.BF16, 128, 1024, 512, 0.25),    # the largest rank
    (configs.BF16, 640, 4096, 384, 1.0),     # several K splits
    # more pair tiles than CTA pairs: static ranges (each pair owns a run of
    # (tile, K tile) iterations; a tile is cut where a range ends)
    (configs.BF16, 19500, 4104, 40, 1.0),    # ragged rows, K tail, N padded 40 -> 48
    (configs.BF16, 19500, 4104, 296, -1.25), # two MMAs (160 + 144), ragged everywhere
    # fewer pair tiles than pairs: K segments
    (configs.BF16, 8100, 4104, 40, 1.0),
    (configs.BF16, 9000, 4104, 296, -1.25),
    (configs.F32, 200, 136, 24, 1.5),
    (configs.F32, 65, 36, 4, 2.0),
    (configs.F32, 70, 100, 512, 0.5),        # two N passes of 256
    (configs.F32, 300, 260, 300, 1.0),       # two N passes of 160 (80-row Y halves), K tail
    (configs.F32, 1000, 1028, 384, -0.75),   # two N passes of 192, four pair tiles, K tail
    (configs.F32, 520, 2048, 128, 2.0),      # one pass of 128, many K segments
    (configs.F32, 1, 4, 8, 1.0),             # single row, single short K tile
])
def test_edge_shapes(dtype, d_out, d_in, r, s):
    cfg = _custom(f"edge-{dtype}-{d_out}x{d_in}-r{r}", dtype, d_out, d_in, r, s)
    x = gen.norm_inputs(cfg)
    wn, g = _run(x, cfg)
    wn_ref, g_ref = _oracle(x, cfg)
    _check(cfg, wn, g, wn_ref, g_ref)


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_zero_scale_takes_base_norm_only(dtype):
    cfg = _custom("s0", dtype, 300, 264, 32, 0.0)
    x = gen.norm_inputs(cfg)
    wn, g = _run(x, cfg)
    wn_ref, g_ref = _oracle(x, cfg)
    _check(cfg, wn, g, wn_ref, g_ref)


def test_rank_zero():
    cfg = _custom("r0", configs.BF16, 96, 128, 0, 1.0)
    x = gen.norm_inputs(configs.Config("r0", 0, configs.BF16, cfg.modules, r=8, s=1.0, eps=1e-6,
                                       tokens=4))
    W, m = to_dev(x["W"], cfg.dtype), to_dev(x["m"], cfg.dtype)
    A = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((96, 0), dtype=torch.bfloat16, device="cuda")
    wn, g = api.dora_factored_norm(W, A, B, 1.0, m, 1e-6)
    wn_ref, g_ref = oracle.norm_and_scale(x["W"], np.zeros((0, 128), np.uint16),
                                          np.zeros((96, 0), np.uint16), x["m"], 1.0,
                                          float(np.float32(1e-6)), cfg.dtype)
    _check(cfg, wn.cpu().numpy(), g.cpu().numpy(), wn_ref, g_ref)


def test_empty_input_dim_gives_eps_branch():
    W = torch.empty((10, 0), dtype=torch.bfloat16, device="cuda")
    A = torch.empty((8, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((10, 8), dtype=torch.bfloat16, device="cuda")
    m = torch.full((10,), 3.0, dtype=torch.bfloat16, device="cuda")
    wn, g = api.dora_factored_norm(W, A, B, 1.0, m, 0.5)
    assert torch.all(wn == 0).item()
    assert torch.all(g == 6.0).item()


def test_empty_output_dim_is_noop():
    W = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((0, 8), dtype=torch.bfloat16, device="cuda")
    m = torch.empty((0,), dtype=torch.bfloat16, device="cuda")
    wn, g = api.dora_factored_norm(W, A, B, 1.0, m, 1e-6)
    assert wn.numel() == 0 and g.numel() == 0


# ------------------------------------------------------------------ exact cases
def _int_case(dtype, d_out, d_in, r, seed, ab_max=3):
    rng = np.random.default_rng(seed)
    W = rng.integers(-3, 4, (d_out, d_in)).astype(np.float32)
    A = rng.integers(-ab_max, ab_max + 1, (r, d_in)).astype(np.float32)
    B = rng.integers(-ab_max, ab_max + 1, (d_out, r)).astype(np.float32)
    m = rng.integers(1, 9, d_out).astype(np.float32)
    # Bound every partial sum of every term by the sum of absolute values:
    # all stay below 2^24, so fp32 accumulation in any order is exact.
    aW, aA, aB = (np.abs(v.astype(np.int64)) for v in (W, A, B))
    aU = aW @ aA.T                     # |U| partial sums
    aG = aA @ aA.T                     # |G| partial sums
    aT = aB @ aG                       # |B G| partial sums
    # the bf16 path accumulates U + (s/2) B G in one accumulator (s = 2 here)
    bounds = [(aW * aW).sum(1), aU + aT, (aB * (aU + aT)).sum(1), aG, aT, (aB * aT).sum(1)]
    assert max(int(np.max(b)) for b in bounds) < 2 ** 24
    if dtype == configs.BF16:
        conv = gen.f32_to_bf16_bits
        return {"W": conv(W), "A": conv(A), "B": conv(B), "m": conv(m)}
    return {"W": W, "A": A, "B": B, "m": m}


@pytest.mark.parametrize("dtype,d_out,d_in,r,ab_max", [
    (configs.BF16, 200, 256, 32, 3), (configs.BF16, 130, 200, 8, 3),
    (configs.BF16, 64, 64, 384, 1), (configs.F32, 200, 256, 32, 3), (configs.F32, 33, 60, 12, 3),
])
def test_small_integers_bit_exact(dtype, d_out, d_in, r, ab_max):
    """Small-integer inputs, s = 2: every product and partial sum is an integer
    below 2^24, so every fp32 step is exact and wnorm, g must equal the
    oracle's values rounded to fp32, bit for bit."""
    cfg = _custom("int", dtype, d_out, d_in, r, 2.0)
    x = _int_case(dtype, d_out, d_in, r, seed=d_out + r, ab_max=ab_max)
    wn, g = _run(x, cfg)
    wn_ref, g_ref = _oracle(x, cfg)
    np.testing.assert_array_equal(wn, wn_ref.astype(np.float32))
    np.testing.assert_array_equal(g, g_ref.astype(np.float32))


def test_fp32_low_bits_reach_the_tensor_cores():
    """fp32 operands whose bits below the TF32 precision are set, chosen so
    that the part the tensor core does not read (v minus v truncated to 10
    fraction bits) is itself a TF32 value: the three-term product is then
    exact.  U, the cross term and the BA-norm term are of the size of the
    base term, so a pass that dropped or double-counted those bits (2^-10
    relative) would miss the oracle by about 1e-4; the tolerance is 1e-6."""
    d_out, d_in, r, s = 256, 64, 16, 1.0
    j = np.arange(d_out)
    sign = np.where(j % 2 == 0, 1.0, -1.0)
    a = sign * (1.0 + (j % 7) * 2.0 ** -10 + 2.0 ** -11 + 2.0 ** -13 + 2.0 ** -19)
    b = 1.0 + 2.0 ** -11 + 2.0 ** -15
    W = np.zeros((d_out, d_in), np.float32)
    W[:, 0] = a                      # low bits in W
    W[:, 1] = 1.0
    A = np.zeros((r, d_in), np.float32)
    A[0, 0] = 1.0
    A[1, 1] = b                      # low bits in A
    B = np.zeros((d_out, r), np.float32)
    B[:, :2] = 1.0
    m = np.ones(d_out, np.float32)
    for v in (W, A):
        assert np.all(v.astype(np.float64) == v)          # exactly representable
    x = {"W": W, "A": A, "B": B, "m": m}
    cfg = _custom("tf32bits", configs.F32, d_out, d_in, r, s)
    wn, g = _run(x, cfg)
    wn_ref, g_ref = _oracle(x, cfg)
    _check(cfg, wn, g, wn_ref, g_ref)


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_cancelling_adapter_clamps_to_zero(dtype):
    """W = -s B A exactly: the factored sum is exactly zero, the clamp keeps the
    root real and g = m / eps (Chinese write-up section 1.2.2)."""
    d_out, d_in, r, s = 160, 192, 16, 2.0
    rng = np.random.default_rng(7)
    A = rng.integers(-2, 3, (r, d_in)).astype(np.float32)
    B = rng.integers(-2, 3, (d_out, r)).astype(np.float32)
    W = (-s * (B.astype(np.float64) @ A.astype(np.float64))).astype(np.float32)  # |W| <= 128
    m = np.full(d_out, 3.0, np.float32)
    x = {"W": W, "A": A, "B": B, "m": m}
    if dtype == configs.BF16:
        x = {k: gen.f32_to_bf16_bits(v) for k, v in x.items()}
    cfg = _custom("cancel", dtype, d_out, d_in, r, s)
    wn, g = _run(x, cfg)
    assert np.all(wn == 0.0)
    np.testing.assert_array_equal(g, np.full(d_out, np.float32(3.0 / np.float64(np.float32(1e-6))),
                                             np.float32))


def test_deterministic_across_calls():
    cfg = _custom("det", configs.BF16, 1024, 2048, 384, 1.0)
    x = gen.norm_inputs(cfg)
    a = _run(x, cfg)
    b = _run(x, cfg)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_deterministic_with_static_ranges():
    """20000 x 4096, r = 384 (static ranges): which CTA pair takes which
    range depends on the order in which the pairs start, which varies from
    call to call; the ranges, and so every sum, do not."""
    cfg = _custom("det-ranges", configs.BF16, 20000, 4096, 384, 1.0)
    x = gen.norm_inputs(cfg)
    runs = [_run(x, cfg) for _ in range(3)]
    for wn, g in runs[1:]:
        np.testing.assert_array_equal(wn, runs[0][0])
        np.testing.assert_array_equal(g, runs[0][1])


def test_one_workspace_across_schedules_and_leftover_words():
    """One workspace, filled with random bytes first, serves norms that plan
    their work differently -- a piece table (fewer pair tiles than pairs,
    control words zeroed by the Gram kernel), static ranges (more pair tiles
    than pairs, zeroing kernel), two accumulators per buffer (r <= 128) and
    the s = 0 path -- in an order where every call finds the previous call's
    control words (completion counters, work counter, status) left over.
    Every result must match the oracle, and repeating the sequence must give
    the same bits."""
    shapes = [(2048, 1024, 384, 1.0), (20000, 1024, 384, 1.0), (4096, 2048, 128, 2.0),
              (2048, 1024, 384, 0.0), (2048, 1024, 384, 1.0)]
    cfgs = [_custom(f"ws-{i}", configs.BF16, d_out, d_in, r, s) for i, (d_out, d_in, r, s)
            in enumerate(shapes)]
    xs = [gen.norm_inputs(c) for c in cfgs]
    size = max(api.workspace_size(d_out, d_in, r, torch.bfloat16) for d_out, d_in, r, _ in shapes)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    gen_t = torch.Generator(device="cuda")
    gen_t.manual_seed(11)
    ws.copy_(torch.randint(0, 256, (size,), dtype=torch.uint8, device="cuda", generator=gen_t))
    first = []
    for rep in range(2):
        for i, (cfg, x) in enumerate(zip(cfgs, xs)):
            dev = {k: to_dev(x[k], cfg.dtype) for k in ("W", "A", "B", "m")}
            wn, g = api.dora_factored_norm(dev["W"], dev["A"], dev["B"], cfg.s, dev["m"],
                                           cfg.eps, workspace=ws)
            assert api.dora_check_status(ws) == 0
            wn, g = wn.cpu().numpy(), g.cpu().numpy()
            if rep == 0:
                rows = np.arange(cfg.module.d_out)
                if cfg.module.d_out > 4096:
                    rows = np.sort(np.random.default_rng(i).choice(cfg.module.d_out, 512, False))
                wn_ref, g_ref = _oracle(x, cfg, rows=rows)
                _check(cfg, wn[rows], g[rows], wn_ref, g_ref)
                first.append((wn, g))
            else:
                np.testing.assert_array_equal(wn, first[i][0])
                np.testing.assert_array_equal(g, first[i][1])
