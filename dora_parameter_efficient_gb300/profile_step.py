"""Run the hot path (factored norm + compose) of one synthetic workload for a few
steps and print per-step CUDA-event times; meant as the target of profilers
(ncu), which want a short program with few launches.  With --training each
step also runs the training path of the compose (forward keeping inner,
backward with the magnitude gradient).

    python -m dora_parameter_efficient_gb300.profile_step --config 1 --steps 3 [--training]

With --grouped it runs every module of the config instead (the 196-module
stack: --config 4) as one grouped norm per step through a plan created once,
then one grouped compose, with inputs drawn on the device.

With --compose-pairs each step runs a second compose right after the first,
on a second set of activations (a copy) into a second output, so a profiler
that captures the second one sees the first one's output written back from
L2 to HBM during it, as it is in a running step.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dora_parameter_efficient_gb300 import api  # noqa: E402
from synthetic import configs, gen  # noqa: E402


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == configs.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def run_grouped(cfg, steps: int) -> int:
    gen_t = torch.Generator(device="cuda")
    gen_t.manual_seed(cfg.index)
    dt = torch.bfloat16 if cfg.dtype == configs.BF16 else torch.float32

    def rnd(*shape, std):
        return (torch.randn(*shape, device="cuda", generator=gen_t) * std).to(dt)

    norm_mods, comp_mods = [], []
    for mod in cfg.modules:
        norm_mods.append((rnd(mod.d_out, mod.d_in, std=cfg.std_w),
                          rnd(cfg.r, mod.d_in, std=cfg.std_a(mod.d_in)),
                          rnd(mod.d_out, cfg.r, std=cfg.std_b),
                          torch.ones(mod.d_out, dtype=dt, device="cuda")))
    plan = api.dora_norm_grouped_plan_create(norm_mods)
    for (W, *_), g in zip(norm_mods, plan.gs):
        comp_mods.append((rnd(cfg.tokens, W.shape[0], std=cfg.std_base),
                          rnd(cfg.tokens, W.shape[0], std=cfg.std_lora), g))
    outs = [torch.empty_like(b) for b, _, _ in comp_mods]
    for i in range(steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        plan.run(cfg.s, cfg.eps)
        e[1].record()
        api.dora_compose_grouped(comp_mods, cfg.s, outs=outs)
        e[2].record()
        torch.cuda.synchronize()
        print(f"step {i}: grouped norm {e[0].elapsed_time(e[1]) * 1e3:.1f} us, "
              f"grouped compose {e[1].elapsed_time(e[2]) * 1e3:.1f} us")
    plan.destroy()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--module", type=int, default=0)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--training", action="store_true")
    ap.add_argument("--grouped", action="store_true")
    ap.add_argument("--compose-pairs", action="store_true")
    args = ap.parse_args()
    cfg = configs.get(args.config)
    if args.grouped:
        return run_grouped(cfg, args.steps)
    x = gen.norm_inputs(cfg, module=args.module)
    c = gen.compose_inputs(cfg, module=args.module)
    W, A, B, m = (to_dev(x[k], cfg.dtype) for k in ("W", "A", "B", "m"))
    base, lora = to_dev(c["base"], cfg.dtype), to_dev(c["lora"], cfg.dtype)
    d_out, d_in = W.shape
    ws = api.alloc_workspace(d_out, d_in, A.shape[0], W.dtype)
    wn = torch.empty(d_out, dtype=torch.float32, device="cuda")
    g = torch.empty(d_out, dtype=torch.float32, device="cuda")
    out = torch.empty_like(base)
    if args.compose_pairs:
        base2, lora2, out2 = base.clone(), lora.clone(), torch.empty_like(base)
    if args.training:
        grad = to_dev(gen.grad_inputs(cfg, module=args.module), cfg.dtype)
        inner = torch.empty_like(base)
        d_base, d_lora = torch.empty_like(base), torch.empty_like(base)
        dmag = torch.empty(d_out, dtype=torch.float32, device="cuda")
        bws = torch.empty(max(16, api.compose_backward_workspace_size(base.shape[0], d_out)),
                          dtype=torch.uint8, device="cuda")
    for i in range(args.steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps, wnorm=wn, g=g, workspace=ws)
        e[1].record()
        api.dora_compose(base, lora, g, cfg.s, out=out)
        e[2].record()
        if args.compose_pairs:
            api.dora_compose(base2, lora2, g, cfg.s, out=out2)
        if args.training:
            api.dora_compose_train(base, lora, g, cfg.s, out=out, inner=inner)
            api.dora_compose_backward(grad, g, cfg.s, inner=inner, wnorm=wn, eps=cfg.eps,
                                      d_base=d_base, d_lora=d_lora, dmag=dmag, workspace=bws)
        torch.cuda.synchronize()
        print(f"step {i}: norm {e[0].elapsed_time(e[1]) * 1e3:.1f} us, "
              f"compose {e[1].elapsed_time(e[2]) * 1e3:.1f} us")
    status = api.dora_check_status(ws)
    print("status", status)
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
