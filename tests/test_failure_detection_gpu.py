"""Device-side failure detection, without a GPU fault: a bounded wait that
nothing completes runs out, the kernel records DORA_ERR_TIMEOUT in the
workspace's status word and returns, the host reads it with
dora_check_status, and the same context -- and the same workspace -- then
runs a norm correctly."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from dora_parameter_efficient_gb300 import _lib, api
from synthetic import configs, gen
from tests.parity_util import NORM_RTOL, rel_err, to_dev

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_the_context_survives():
    cfg = configs.Config("after-timeout", 0, configs.BF16, (configs.Module("t", 300, 256),), r=32,
                         s=1.0, eps=1e-6, tokens=8)
    ws = api.alloc_workspace(300, 256, 32, torch.bfloat16)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.dora_selftest_timeout(ws, 50_000)            # 50 ms
    status = api.dora_check_status(ws)
    assert status == _lib.DORA_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.045         # the wait ran to its limit
    assert "ran out of time" in _lib.status_string(status)

    # the context is usable, and a norm on the same workspace starts from a
    # clean status word and is correct
    x = gen.norm_inputs(cfg)
    W, A, B, m = (to_dev(x[k], cfg.dtype) for k in ("W", "A", "B", "m"))
    wn, g = api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps, workspace=ws)
    assert api.dora_check_status(ws) == _lib.DORA_OK
    wn_ref, g_ref = oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s,
                                          float(np.float32(cfg.eps)), cfg.dtype)
    assert rel_err(wn.cpu().numpy(), wn_ref).max() <= NORM_RTOL[cfg.dtype]
    assert rel_err(g.cpu().numpy(), g_ref).max() <= NORM_RTOL[cfg.dtype]
