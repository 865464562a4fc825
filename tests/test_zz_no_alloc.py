"""The allocation-free norm entry point, dora_factored_norm_noalloc.

It serves callers that cannot allocate device memory (a plug-in inside a host
program whose allocator owns the device's free memory, or a path where
cudaMalloc/cudaFree are off limits because they synchronize the device and
can fail under memory pressure).  Instead of a caller workspace it uses the
library's own fixed 32 MiB device array.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes alone in a fresh
process.  The GPU test calls the new entry point through the C ABI twice in a
row, on two different modules, and compares each result with the existing
entry point (dora_factored_norm with a caller workspace) and with the float64
CPU oracle, within the parity tolerances of the other tests.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

from dora_parameter_efficient_gb300 import _lib
from synthetic import configs, gen


def _lib_loaded():
    if not os.path.exists(_lib.LIB_PATH):
        from dora_parameter_efficient_gb300 import build
        build.build()
    return _lib.load()


def test_oversized_shape_is_refused_before_any_launch():
    """A shape whose workspace exceeds the 32 MiB array is refused on the host."""
    lib = _lib_loaded()
    P = 1 << 20        # never dereferenced: the call returns before touching the device
    d_out, d_in, r = 300_000, 4096, 512
    assert lib.dora_norm_workspace_size(d_out, d_in, r, _lib.DORA_BF16) > (32 << 20)
    st = lib.dora_factored_norm_noalloc(P, 2 * P, 3 * P, _lib.DORA_BF16, d_out, d_in, r, 1.0,
                                        4 * P, 1e-6, 5 * P, 6 * P, None)
    assert st == _lib.DORA_ERR_WORKSPACE
    assert lib.dora_factored_norm_noalloc(P, 2 * P, 3 * P, 9, 64, 64, 8, 1.0, 4 * P, 1e-6,
                                          5 * P, 6 * P, None) == _lib.DORA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    import torch

    import oracle
    from dora_parameter_efficient_gb300 import api
    from tests.parity_util import NORM_RTOL, rel_err, to_dev

    _lib_loaded()
    cases = [
        configs.Config("noalloc-a", 0, configs.BF16, (configs.Module("a", 1000, 2048),), r=384,
                       s=1.0, eps=1e-6, tokens=4),
        configs.Config("noalloc-b", 1, configs.BF16, (configs.Module("b", 300, 520),), r=24,
                       s=-0.5, eps=1e-6, tokens=4),
    ]
    for cfg in cases:      # two calls in a row, different shapes, shared scratch
        x = gen.norm_inputs(cfg, seed=11)
        W, A, B, m = (to_dev(x[k], cfg.dtype) for k in ("W", "A", "B", "m"))
        d_out = W.shape[0]
        wn_ref, g_ref = api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps)
        wn = torch.full((d_out,), float("nan"), dtype=torch.float32, device="cuda")
        g = torch.full((d_out,), float("nan"), dtype=torch.float32, device="cuda")
        api.dora_factored_norm_noalloc(W, A, B, cfg.s, m, cfg.eps, wn, g)
        torch.cuda.synchronize()
        tol = NORM_RTOL[cfg.dtype]
        assert rel_err(wn.cpu().numpy(), wn_ref.cpu().numpy()).max() <= tol, cfg.name
        assert rel_err(g.cpu().numpy(), g_ref.cpu().numpy()).max() <= tol, cfg.name
        assert np.all(np.isfinite(wn.cpu().numpy()))
        # and against the float64 oracle on the same stored inputs
        wn_o, g_o = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s,
                                          float(np.float32(cfg.eps)), cfg.dtype)
        assert rel_err(wn.cpu().numpy(), wn_o).max() <= tol, cfg.name
        assert rel_err(g.cpu().numpy(), g_o).max() <= tol, cfg.name
