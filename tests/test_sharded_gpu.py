"""GPU parity of the d_in-sharded norm: dora_norm_partials on each column
slice, the slices' partials added in a fixed order on the device, then
dora_norm_finalize_partials -- against the float64 oracle of the whole module
(Chinese write-up, section 1.2.1: every term of the factored norm is a sum
over d_in).  All slices run on one GPU here; between GPUs the addition is one
all-reduce of the same buffer (tests/test_sharded_cpu.py covers that exchange
on CPU ranks)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import NORM_RTOL, rel_err, to_dev

pytestmark = pytest.mark.gpu

TORCH_DT = {configs.BF16: torch.bfloat16, configs.F32: torch.float32}


def _slices(x, dtype, parts):
    """Device copies of every slice's W and A columns (contiguous), and B, m."""
    d_in = x["W"].shape[1]
    out = []
    for i in range(parts):
        k0, k1 = api.slice_bounds(d_in, parts, i, TORCH_DT[dtype])
        out.append((k0, k1, to_dev(np.ascontiguousarray(x["W"][:, k0:k1]), dtype),
                    to_dev(np.ascontiguousarray(x["A"][:, k0:k1]), dtype)))
    return out, to_dev(x["B"], dtype), to_dev(x["m"], dtype)


def _sharded(x, dtype, parts, s, eps):
    slices, B, m = _slices(x, dtype, parts)
    parts_dev = [api.dora_norm_partials(W, A, B) for _, _, W, A in slices]
    total = parts_dev[0].clone()
    for p in parts_dev[1:]:
        total += p                      # in slice order
    wn, g = api.dora_norm_finalize_partials(total, B, s, m, eps)
    torch.cuda.synchronize()
    return slices, parts_dev, wn.cpu().numpy(), g.cpu().numpy()


def _check_slice_partials(x, dtype, slices, parts_dev, rows):
    """Each slice's partials against the oracle's shares, in the error bound of
    an fp32 sum of |terms| (products exact for bf16, 3xTF32 for fp32)."""
    Wf, Af, Bf = (oracle.decode(x[k], dtype) for k in ("W", "A", "B"))
    d_out, r = Bf.shape
    for (k0, k1, _, _), p in zip(slices, parts_dev):
        base, cross, G = (v.cpu().numpy().astype(np.float64)
                          for v in api.partials_views(p, d_out, r))
        rb, rc, rg = oracle.norm_partials(Wf[rows, k0:k1], Af[:, k0:k1], Bf[rows])
        ab, ac, ag = oracle.norm_partials(np.abs(Wf[rows, k0:k1]), np.abs(Af[:, k0:k1]),
                                          np.abs(Bf[rows]))
        tol = 2e-6
        assert np.all(np.abs(base[rows] - rb) <= tol * ab + 1e-30)
        assert np.all(np.abs(cross[rows] - rc) <= tol * ac + 1e-30)
        assert np.all(np.abs(G - rg) <= tol * ag + 1e-30)


CASES = [
    # (config, parts): the metric workload and its ragged / fp32 relatives
    (configs.get(1), 2),
    (configs.get(1), 4),
    (configs.Config("shard-ragged", 40, configs.BF16, (configs.Module("m", 1000, 2056),), r=40,
                    s=-0.75, eps=1e-6, tokens=4), 2),
    (configs.Config("shard-ragged", 40, configs.BF16, (configs.Module("m", 1000, 2056),), r=40,
                    s=-0.75, eps=1e-6, tokens=4), 4),
    (configs.get(0), 2),
    (configs.Config("shard-f32", 41, configs.F32, (configs.Module("m", 300, 1000),), r=24,
                    s=2.0, eps=1e-6, tokens=4), 4),
    (configs.Config("shard-f32-r512", 42, configs.F32, (configs.Module("m", 520, 2048),), r=512,
                    s=0.5, eps=1e-6, tokens=4), 2),
]


@pytest.mark.parametrize("cfg,parts", CASES, ids=[f"{c.name}-x{p}" for c, p in CASES])
def test_sharded_norm_matches_oracle(cfg, parts):
    x = gen.norm_inputs(cfg)
    d_out = x["W"].shape[0]
    slices, parts_dev, wn, g = _sharded(x, cfg.dtype, parts, cfg.s, cfg.eps)
    rng = np.random.default_rng(parts)
    rows = np.arange(d_out) if d_out <= 2048 else np.unique(
        np.concatenate([np.arange(64), np.arange(d_out - 64, d_out), rng.choice(d_out, 512, False)]))
    wn_ref, g_ref = oracle.norm_and_scale(x["W"][rows], x["A"], x["B"][rows], x["m"][rows], cfg.s,
                                          float(np.float32(cfg.eps)), cfg.dtype)
    tol = NORM_RTOL[cfg.dtype]
    assert rel_err(wn[rows], wn_ref).max() <= tol
    assert rel_err(g[rows], g_ref).max() <= tol
    _check_slice_partials(x, cfg.dtype, slices, parts_dev, rows)
    # the same as the one-device norm of the whole module, to fp32 rounding of the partials
    wn1, _ = api.dora_factored_norm(to_dev(x["W"], cfg.dtype), to_dev(x["A"], cfg.dtype),
                                    to_dev(x["B"], cfg.dtype), cfg.s, to_dev(x["m"], cfg.dtype),
                                    cfg.eps)
    assert rel_err(wn, wn1.cpu().numpy()).max() <= tol


@pytest.mark.parametrize("dtype", [configs.BF16, configs.F32])
def test_finalize_from_oracle_partials(dtype):
    """The finalize alone, fed the oracle's partials of the whole module
    (rounded once to fp32): wnorm and g against the oracle's norm from the
    same partials."""
    cfg = configs.Config("fin", 43, dtype, (configs.Module("m", 700, 512),), r=48, s=1.25,
                         eps=1e-6, tokens=4)
    x = gen.norm_inputs(cfg)
    Bf = oracle.decode(x["B"], dtype)
    base, cross, G = oracle.norm_partials(oracle.decode(x["W"], dtype),
                                          oracle.decode(x["A"], dtype), Bf)
    p32 = np.concatenate([base, cross, G.reshape(-1)]).astype(np.float32)
    wn, g = api.dora_norm_finalize_partials(torch.from_numpy(p32).cuda(), to_dev(x["B"], dtype),
                                            cfg.s, to_dev(x["m"], dtype), cfg.eps)
    torch.cuda.synchronize()
    d_out = Bf.shape[0]
    pf = p32.astype(np.float64)
    ref = oracle.norm_from_partials(pf[:d_out], pf[d_out:2 * d_out],
                                    pf[2 * d_out:].reshape(cfg.r, cfg.r), Bf, cfg.s)
    g_ref = oracle.magnitude_scale(oracle.decode(x["m"], dtype), ref, float(np.float32(cfg.eps)))
    tol = NORM_RTOL[dtype]
    assert rel_err(wn.cpu().numpy(), ref).max() <= tol
    assert rel_err(g.cpu().numpy(), g_ref).max() <= tol


def test_sharded_edge_cases():
    """Empty slices (more slices than K tiles), s = 0 and r = 0 at the
    finalize, a module without rows (G only), and bitwise-repeatable partials."""
    cfg = configs.Config("edge", 44, configs.BF16, (configs.Module("m", 260, 128),), r=16,
                         s=1.0, eps=1e-6, tokens=4)
    x = gen.norm_inputs(cfg)
    d_out = x["W"].shape[0]
    slices, parts_dev, wn, g = _sharded(x, cfg.dtype, 4, cfg.s, cfg.eps)
    assert any(k0 == k1 for k0, k1, _, _ in slices)
    for (k0, k1, _, _), p in zip(slices, parts_dev):
        if k0 == k1:
            assert not torch.any(p).item()
    wn_ref, _ = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s, 1e-6, cfg.dtype)
    assert rel_err(wn, wn_ref).max() <= NORM_RTOL[cfg.dtype]
    # s = 0: the base term alone
    _, _, wn0, _ = _sharded(x, cfg.dtype, 2, 0.0, cfg.eps)
    ref0, _ = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], 0.0, 1e-6, cfg.dtype)
    assert rel_err(wn0, ref0).max() <= NORM_RTOL[cfg.dtype]
    # r = 0: partials are base and a zero cross
    W = to_dev(x["W"], cfg.dtype)
    e = torch.empty((0, W.shape[1]), dtype=W.dtype, device="cuda")
    p0 = api.dora_norm_partials(W, e, torch.empty((d_out, 0), dtype=W.dtype, device="cuda"))
    wr, _ = api.dora_norm_finalize_partials(p0, torch.empty((d_out, 0), dtype=W.dtype,
                                                            device="cuda"),
                                            cfg.s, to_dev(x["m"], cfg.dtype), cfg.eps)
    torch.cuda.synchronize()
    assert not torch.any(p0[d_out:]).item()
    assert rel_err(wr.cpu().numpy(), ref0).max() <= NORM_RTOL[cfg.dtype]
    # no rows: only G = A A^T
    A = to_dev(x["A"], cfg.dtype)
    pg = api.dora_norm_partials(torch.empty((0, A.shape[1]), dtype=A.dtype, device="cuda"), A,
                                torch.empty((0, cfg.r), dtype=A.dtype, device="cuda"))
    torch.cuda.synchronize()
    Af = oracle.decode(x["A"], cfg.dtype)
    Gr = Af @ Af.T
    bound = 2e-6 * (np.abs(Af) @ np.abs(Af).T)      # fp32 sums of exact products
    assert np.all(np.abs(pg.cpu().numpy().reshape(cfg.r, cfg.r) - Gr) <= bound)
    # the partials of one slice are the same bits on every call
    W1, A1 = slices[1][2], slices[1][3]
    B = to_dev(x["B"], cfg.dtype)
    a = api.dora_norm_partials(W1, A1, B).cpu().numpy()
    b = api.dora_norm_partials(W1, A1, B).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
