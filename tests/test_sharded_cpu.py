"""The exchange of the d_in-sharded norm on CPU, with two and three gloo ranks.

Every term of the factored norm is a sum over d_in (Chinese write-up, section
1.2.1 and Algorithm 1 of section 5.1), so ranks that hold column slices of W
and A add their partials [base | cross | G] with one all-reduce and then
finish the norm locally.  Here each rank computes its slice's partials with
the float64 oracle (there is no GPU), hands them to the library's exchange
(``api.allreduce_partials``, through its layout helpers ``slice_bounds`` and
``partials_views``), and checks that every rank ends up with the partials of
the whole module and, through the oracle's identity, the dense norm.  The GPU
kernels behind the partials and the finalize are covered by
tests/test_sharded_gpu.py."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        import oracle
        from dora_parameter_efficient_gb300 import api
        from synthetic import configs, gen
        cfg = configs.Config("shard-cpu", 31, configs.BF16, (configs.Module("m", 96, 1000),),
                             r=24, s=1.5, eps=1e-6, tokens=4)
        x = gen.norm_inputs(cfg)                      # the same module on every rank
        d_out, d_in = x["W"].shape
        r = cfg.r
        k0, k1 = api.slice_bounds(d_in, world, rank, torch.bfloat16)
        W = oracle.decode(x["W"], cfg.dtype)[:, k0:k1]
        A = oracle.decode(x["A"], cfg.dtype)[:, k0:k1]
        B = oracle.decode(x["B"], cfg.dtype)
        base, cross, G = oracle.norm_partials(W, A, B)
        buf = torch.zeros(api.norm_partials_floats(d_out, r), dtype=torch.float32)
        vb, vc, vg = api.partials_views(buf, d_out, r)
        vb.copy_(torch.from_numpy(base))
        vc.copy_(torch.from_numpy(cross))
        vg.copy_(torch.from_numpy(G))
        api.allreduce_partials(buf)
        # a subgroup of all ranks behaves the same
        sub = dist.new_group(list(range(world)))
        buf2 = torch.zeros_like(buf)
        api.partials_views(buf2, d_out, r)[0].copy_(torch.from_numpy(base))
        api.allreduce_partials(buf2, group=sub)
        q.put((rank, (k0, k1), buf.numpy().copy(), buf2.numpy().copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_exchange_partials(world):
    import torch
    import torch.multiprocessing as mp

    import oracle
    from dora_parameter_efficient_gb300 import api
    from synthetic import configs, gen

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(world):
            rank, bounds, buf, buf2 = q.get(timeout=180)
            results[rank] = (bounds, buf, buf2)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert sorted(results) == list(range(world))

    cfg = configs.Config("shard-cpu", 31, configs.BF16, (configs.Module("m", 96, 1000),),
                         r=24, s=1.5, eps=1e-6, tokens=4)
    x = gen.norm_inputs(cfg)
    d_out, d_in = x["W"].shape
    # the slices tile d_in in order, on the 64-column grid
    bounds = [results[k][0] for k in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == d_in
    assert all(a[1] == b[0] for a, b in zip(bounds[:-1], bounds[1:]))
    assert all(k0 % 64 == 0 for k0, _ in bounds)
    W, A, B = (oracle.decode(x[k], cfg.dtype) for k in ("W", "A", "B"))
    whole = oracle.norm_partials(W, A, B)
    base_sum = sum(oracle.norm_partials(W[:, a:b], A[:, a:b], B)[0].astype(np.float32)
                   for a, b in bounds)
    for rank, (_, buf, buf2) in results.items():
        t = torch.from_numpy(buf)
        base, cross, G = (v.numpy().astype(np.float64) for v in api.partials_views(t, d_out, cfg.r))
        # every rank holds the whole module's partials (fp32 shares, summed in fp32)
        np.testing.assert_allclose(base, whole[0], rtol=1e-6)
        np.testing.assert_allclose(cross, whole[1], rtol=0, atol=1e-6 * np.abs(whole[1]).max())
        np.testing.assert_allclose(G, whole[2], rtol=0, atol=1e-6 * np.abs(whole[2]).max())
        # and from them the dense norm of the whole module
        wn = oracle.norm_from_partials(base, cross, G, B, cfg.s)
        ref, _ = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s, 1e-6, cfg.dtype)
        assert np.max(np.abs(wn - ref) / ref) < 1e-6
        # the subgroup exchange summed the base shares alone
        np.testing.assert_allclose(buf2[:d_out], base_sum, rtol=1e-6)
        assert not np.any(buf2[d_out:])


def test_slice_bounds_edges():
    import torch

    from dora_parameter_efficient_gb300 import api
    # more slices than K tiles: some slices are empty, the union is still d_in
    b = [api.slice_bounds(128, 4, i, torch.bfloat16) for i in range(4)]
    assert b[0][0] == 0 and b[-1][1] == 128
    assert all(x[1] == y[0] for x, y in zip(b[:-1], b[1:]))
    assert any(k0 == k1 for k0, k1 in b)
    # a ragged last slice keeps 16-byte rows
    k0, k1 = api.slice_bounds(1000, 3, 2, torch.float32)
    assert k1 == 1000 and ((k1 - k0) * 4) % 16 == 0
    with pytest.raises(ValueError):
        api.slice_bounds(100, 2, 0, torch.bfloat16)          # 200-byte rows
    with pytest.raises(ValueError):
        api.slice_bounds(128, 2, 2, torch.bfloat16)
