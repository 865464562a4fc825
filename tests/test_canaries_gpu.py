"""Guard bands around every output buffer and behind every workspace: the
bytes just before and after what a call may write must come back unchanged
(compute-sanitizer is not available here; this catches writes past the end
of an output or of the workspace on the shapes that stress the tile edges)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from dora_parameter_efficient_gb300 import api
from synthetic import configs, gen
from tests.parity_util import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096       # elements on each side (a multiple of 16 bytes for every dtype)


class Guarded:
    """A buffer of `shape` inside a larger one filled with random bytes; the
    view may start `offset` elements past a 16-byte boundary."""

    def __init__(self, shape, dtype, offset=0):
        self.n = int(np.prod(shape))
        self.start = GUARD + offset
        self.big = torch.empty(self.n + 2 * GUARD + offset, dtype=dtype, device="cuda")
        raw = self.big.view(torch.uint8)
        raw.copy_(torch.randint(0, 256, raw.shape, dtype=torch.uint8, device="cuda"))
        self.saved = self.big.clone()
        self.view = self.big[self.start:self.start + self.n].view(shape)

    def check(self, name):
        torch.cuda.synchronize()
        a, b = self.big.view(torch.uint8), self.saved.view(torch.uint8)
        esz = self.big.element_size()
        lo, hi = self.start * esz, (self.start + self.n) * esz
        assert torch.equal(a[:lo], b[:lo]), f"{name}: bytes before the buffer changed"
        assert torch.equal(a[hi:], b[hi:]), f"{name}: bytes after the buffer changed"


def _workspace(nbytes):
    """(workspace view of exactly nbytes, 256-byte aligned, guard object)."""
    g = Guarded((nbytes,), torch.uint8)
    assert g.view.data_ptr() % 256 == 0
    return g.view, g


def _module(dtype, d_out, d_in, r, s, index=40):
    cfg = configs.Config("canary", index, dtype, (configs.Module("c", d_out, d_in),), r=r, s=s,
                         eps=1e-6, tokens=8)
    x = gen.norm_inputs(cfg)
    return cfg, tuple(to_dev(x[k], dtype) for k in ("W", "A", "B", "m"))


@pytest.mark.parametrize("dtype,d_out,d_in,r,s", [
    (configs.BF16, 300, 520, 40, 1.0),
    (configs.BF16, 1000, 1024, 384, 1.0),
    (configs.BF16, 257, 64, 8, 0.0),          # s = 0: the base-only branch
    (configs.F32, 300, 260, 300, 1.0),
    (configs.F32, 70, 100, 512, 0.5),
])
def test_norm_writes_stay_inside(dtype, d_out, d_in, r, s):
    cfg, (W, A, B, m) = _module(dtype, d_out, d_in, r, s)
    tdt = torch.bfloat16 if dtype == configs.BF16 else torch.float32
    wn, g = Guarded((d_out,), torch.float32), Guarded((d_out,), torch.float32)
    ws, wsg = _workspace(api.workspace_size(d_out, d_in, r, tdt))
    api.dora_factored_norm(W, A, B, s, m, cfg.eps, wnorm=wn.view, g=g.view, workspace=ws)
    assert api.dora_check_status(ws) == 0
    wn.check("wnorm")
    g.check("g")
    wsg.check("workspace")
    assert torch.isfinite(wn.view).all()


def test_noalloc_norm_writes_stay_inside():
    cfg, (W, A, B, m) = _module(configs.BF16, 300, 520, 40, 1.0)
    wn, g = Guarded((300,), torch.float32), Guarded((300,), torch.float32)
    api.dora_factored_norm_noalloc(W, A, B, 1.0, m, cfg.eps, wn.view, g.view)
    wn.check("wnorm")
    g.check("g")


def test_grouped_plan_writes_stay_inside():
    mods, outs = [], []
    for i, (d_out, d_in) in enumerate(((300, 256), (64, 512), (520, 136))):
        _, mod = _module(configs.BF16, d_out, d_in, 24, 1.5, index=50 + i)
        mods.append(mod)
        outs.append((Guarded((d_out,), torch.float32), Guarded((d_out,), torch.float32)))
    ws, wsg = _workspace(api.norm_grouped_workspace_size(mods, torch.bfloat16))
    plan = api.dora_norm_grouped_plan_create(mods, wnorms=[w.view for w, _ in outs],
                                             gs=[g.view for _, g in outs], workspace=ws)
    plan.run(1.5, 1e-6)
    plan.run(0.0, 1e-6)          # the per-module path through the same workspace
    plan.run(1.5, 1e-6)
    torch.cuda.synchronize()
    for w, g in outs:
        w.check("grouped wnorm")
        g.check("grouped g")
    wsg.check("grouped workspace")
    plan.destroy()


@pytest.mark.parametrize("dtype,T,d_out,offset", [
    (configs.BF16, 37, 2048, 0),     # fixed-column vector path
    (configs.BF16, 37, 1000, 0),     # grid-stride vector path
    (configs.BF16, 9, 37, 1),        # unaligned: element-wise path
    (configs.F32, 21, 1024, 0),
    (configs.F32, 5, 33, 1),
])
def test_compose_and_training_writes_stay_inside(dtype, T, d_out, offset):
    tdt = torch.bfloat16 if dtype == configs.BF16 else torch.float32
    gen_t = torch.Generator(device="cuda")
    gen_t.manual_seed(T * d_out)
    base = torch.randn(T, d_out, device="cuda", generator=gen_t).to(tdt)
    lora = (torch.randn(T, d_out, device="cuda", generator=gen_t) * 0.05).to(tdt)
    grad = (torch.randn(T, d_out, device="cuda", generator=gen_t) * 0.01).to(tdt)
    g = 1 + 0.0015 * torch.randn(d_out, device="cuda", generator=gen_t)
    wnorm = 1 + torch.rand(d_out, device="cuda", generator=gen_t)

    out = Guarded((T, d_out), tdt, offset)
    api.dora_compose(base, lora, g, 1.0, out=out.view)
    out.check("out")

    out2, inner = Guarded((T, d_out), tdt, offset), Guarded((T, d_out), tdt, offset)
    api.dora_compose_train(base, lora, g, 1.0, out=out2.view, inner=inner.view)
    out2.check("train out")
    inner.check("inner")

    db, dl = Guarded((T, d_out), tdt, offset), Guarded((T, d_out), tdt, offset)
    dm = Guarded((d_out,), torch.float32)
    bws, bwsg = _workspace(max(16, api.compose_backward_workspace_size(T, d_out)))
    api.dora_compose_backward(grad, g, 1.0, inner=inner.view, wnorm=wnorm, eps=1e-6,
                              d_base=db.view, d_lora=dl.view, dmag=dm.view, workspace=bws)
    db.check("d_base")
    dl.check("d_lora")
    dm.check("dmag")
    bwsg.check("backward workspace")
