"""Benchmark of the DoRA per-module hot path on one GB300 (or N, one process each).

One step = the whole hot path for one adapted module at d_out = d_in = 8192,
r = 384, bf16: dora_factored_norm (G = A A^T, the BA-norm term, the fused
U = W A^T main pass, finalize) followed by dora_compose on 2048 x 8192
activations with the g just computed.  Inputs are seeded synthetic tensors
resident in HBM; three input/output sets rotate so no step finds its operands
in the 129 MB L2.

Printed (rank 0, one JSON line):
  value      factored-norm TFLOP/s: algorithmic norm FLOPs of all ranks divided
             by the norm part of the step (CUDA events on the launching stream,
             averaged over the K timed steps, max over ranks)
  compose    compose GB/s over the compose part of the same steps
  back_to_back  the norm alone, the compose alone and the whole step in loops
             with one event pair around each loop (no events between launches)
  cuda_graph the same three loops captured as CUDA graphs and replayed
  roofline   the dominant kernel (the U = W A^T main pass) against the measured
             burst bf16 peak, its duration bounded by the period of back-to-back
             norms (and, as `isolated`, timed with events around its launch);
             roofline_compose the compose kernel against HBM copy BW
  e2e        the same metrics through the public API from pinned host buffers,
             host<->device copies inside the timed region
  cpu_baseline  the float64 CPU oracle on the host cores, bounded sample, with the
             BLAS thread count it ran on and a single-thread sample
  compose_training  the training forward (out, inner) and backward (d_base,
             d_lora, dmag) at the same shape, GB/s
  stack      the 196-module 7B-like stack at r = 128: grouped norm through a
             plan and grouped compose, modules per second
  fp32_norm  the fp32 norm at 8192 x 8192, r = 512 (3xTF32 tensor-core pass):
             per call with events and back to back, the pass alone against
             the derived TF32 peak and the counter's TF32 issue rate

--impl reference times the CPU oracle (the method's write-ups ship no code to
run) on the same metric, per step a bounded sample sized so the run ends in
minutes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import configs, gen  # noqa: E402

CFG_INDEX = 1
N_SETS = 3
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0, "tf32_tflops": 1100.0}


# ---------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def main_pass_flops(d_out, d_in, r):
    """Algorithmic FLOPs of the CTA-pair main pass: U = W A^T (2 d_out d_in r), B G (2 d_out r^2,
    counted once although the pass multiplies by the two bf16 terms of G'), the sum of squares
    of W (2 d_out d_in) and rowsum(B o (U + s/2 B G)) (2 d_out r)."""
    return 2 * d_out * d_in * r + 2 * d_out * r * r + 2 * d_out * d_in + 2 * d_out * r


def file_digest(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel_src, profile_name):
    """dram bytes per launch recorded in profiles/<profile_name>, if the kernel
    source it was measured on is unchanged."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_bytes or not m_src:
        return None
    if m_src.group(1) != file_digest(kernel_src):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((t, float(parts[2]), float(parts[3]), parts[6:10], parts[5]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        inside = [r for r in rows if self.t_start is not None and self.t_start <= r[0] <= self.t_end]
        use = inside if inside else rows[-3:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(cfg, norm_x, comp_x, g32, rows, tokens):
    """Time the float64 oracle on `rows` norm rows and `tokens` compose rows."""
    import oracle
    t0 = time.perf_counter()
    oracle.norm_and_scale(norm_x["W"][rows], norm_x["A"], norm_x["B"][rows], norm_x["m"][rows],
                          cfg.s, float(np.float32(cfg.eps)), cfg.dtype)
    t1 = time.perf_counter()
    oracle.compose_stored(comp_x["base"][tokens], comp_x["lora"][tokens], g32, cfg.s, cfg.dtype)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def blas_threads():
    """(threads, how): the thread count of the BLAS library numpy loaded, as
    that library reports it (threadpoolctl where installed, else the
    library's exported get_num_threads function found in this process's
    memory map), else the environment or the core count, saying which."""
    try:
        import threadpoolctl
        info = [d for d in threadpoolctl.threadpool_info() if d.get("user_api") == "blas"]
        if info:
            return int(info[0]["num_threads"]), f"reported by {info[0].get('internal_api', 'blas')}"
    except Exception:
        pass
    try:
        import ctypes
        libs = set()
        with open("/proc/self/maps") as f:
            for line in f:
                path = line.split()[-1] if len(line.split()) >= 6 else ""
                if "openblas" in os.path.basename(path).lower():
                    libs.add(path)
        for path in sorted(libs):
            lib = ctypes.CDLL(path)
            for name in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                         "openblas_get_num_threads64_", "openblas_get_num_threads"):
                fn = getattr(lib, name, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    return int(fn()), "reported by OpenBLAS"
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var]), f"from {var}"
    return os.cpu_count() or 1, "assumed: os.cpu_count()"


def cpu_threads():
    return blas_threads()[0]


SINGLE_THREAD_PROBE = r"""
import json, sys, time
import numpy as np
sys.path.insert(0, sys.argv[1])
from synthetic import configs, gen
import oracle
cfg = configs.get(int(sys.argv[2]))
mod = cfg.module
rows = np.arange(int(sys.argv[3]))
toks = np.arange(int(sys.argv[4]))
x = gen.norm_inputs(cfg, rows=rows)
c = gen.compose_inputs(cfg, tokens=len(toks))
g32 = np.full(mod.d_out, 1.0, np.float32)
tn = tc = 0.0
reps = 0
while reps < 1 or tn + tc < float(sys.argv[5]):
    t0 = time.perf_counter()
    oracle.norm_and_scale(x["W"], x["A"], x["B"], x["m"], cfg.s, float(np.float32(cfg.eps)), cfg.dtype)
    t1 = time.perf_counter()
    oracle.compose_stored(c["base"], c["lora"], g32, cfg.s, cfg.dtype)
    t2 = time.perf_counter()
    tn += t1 - t0
    tc += t2 - t1
    reps += 1
print(json.dumps({"norm_s": tn, "compose_s": tc, "reps": reps}))
"""


def single_thread_oracle(rows, toks, seconds=4.0):
    """The oracle on one host thread (BLAS and OpenMP limited to one thread in
    a fresh interpreter), on the first `rows` norm rows and `toks` compose
    token rows of the metric workload, repeated for about `seconds`."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    proc = subprocess.run([sys.executable, "-c", SINGLE_THREAD_PROBE, ROOT, str(CFG_INDEX),
                           str(rows), str(toks), str(seconds)],
                          env=env, capture_output=True, text=True, timeout=600)
    if proc.returncode != 0:
        return None
    return json.loads(proc.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cfg = configs.get(CFG_INDEX)
    mod = cfg.module
    norm_x = gen.norm_inputs(cfg)
    comp_x = gen.compose_inputs(cfg)
    g32 = np.full(mod.d_out, 1.0, np.float32)
    # calibrate: cost per norm row and per compose token row
    tn, tc = oracle_sample(cfg, norm_x, comp_x, g32, np.arange(64), np.arange(64))
    per_row, per_tok = tn / 64, tc / 64
    budget = 90.0 / max(1, args.steps + args.warmup)          # seconds per step
    rows = int(np.clip(budget * 0.8 / per_row, 1, mod.d_out))
    toks = int(np.clip(budget * 0.2 / per_tok, 1, cfg.tokens))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle_sample(cfg, norm_x, comp_x, g32, np.sort(rng.choice(mod.d_out, rows, False)),
                      np.sort(rng.choice(cfg.tokens, toks, False)))
    tn_tot = tc_tot = 0.0
    for _ in range(args.steps):
        a, b = oracle_sample(cfg, norm_x, comp_x, g32, np.sort(rng.choice(mod.d_out, rows, False)),
                             np.sort(rng.choice(cfg.tokens, toks, False)))
        tn_tot += a
        tc_tot += b
    norm_flops_row = configs.norm_flops(mod.d_out, mod.d_in, cfg.r) / mod.d_out
    value = norm_flops_row * rows * args.steps / tn_tot / 1e12
    comp_bytes_tok = configs.compose_bytes(1, mod.d_out, cfg.dtype)
    comp_gbs = comp_bytes_tok * toks * args.steps / tc_tot / 1e9
    sample = (f"per step: oracle norm on {rows} random rows of the {mod.d_out}x{mod.d_in} r={cfg.r} "
              f"module + compose on {toks} random token rows of {cfg.tokens}x{mod.d_out}; "
              f"scaled to TFLOP/s by the method's algorithmic FLOPs per row")
    line = {
        "impl": "reference", "metric": json.loads(BASELINE_METRIC), "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": (tn_tot + tc_tot) / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "d_out": mod.d_out, "d_in": mod.d_in, "r": cfg.r,
                   "tokens": cfg.tokens, "dtype_inputs": cfg.dtype},
        "compose": {"value": comp_gbs, "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(),
                         "cores_how": blas_threads()[1], "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


BASELINE_METRIC = json.dumps("factored-norm TFLOP/s + compose GB/s (% of GB300 peak) at 8192², r=384")


# ---------------------------------------------------------------- the stack workload
def run_stack(api, dev, peaks, steps=10):
    """Grouped norm + compose over the 196 modules of the 7B-like stack."""
    import torch
    cfg = configs.get(4)
    gen_t = torch.Generator(device=dev)
    gen_t.manual_seed(4)
    mods = []
    for m in cfg.modules:
        def rnd(*shape, std):
            return (torch.randn(*shape, device=dev, generator=gen_t) * std).to(torch.bfloat16)
        mods.append(dict(
            W=rnd(m.d_out, m.d_in, std=cfg.std_w), A=rnd(cfg.r, m.d_in, std=cfg.std_a(m.d_in)),
            B=rnd(m.d_out, cfg.r, std=cfg.std_b),
            m=torch.ones(m.d_out, dtype=torch.bfloat16, device=dev),
            base=rnd(cfg.tokens, m.d_out, std=cfg.std_base),
            lora=rnd(cfg.tokens, m.d_out, std=cfg.std_lora),
            wn=torch.empty(m.d_out, dtype=torch.float32, device=dev),
            g=torch.empty(m.d_out, dtype=torch.float32, device=dev), mod=m))
        mods[-1]["out"] = torch.empty_like(mods[-1]["base"])
    norm_mods = [(d["W"], d["A"], d["B"], d["m"]) for d in mods]
    comp_mods = [(d["base"], d["lora"], d["g"]) for d in mods]
    wns, gss, outs = [d["wn"] for d in mods], [d["g"] for d in mods], [d["out"] for d in mods]
    nws = torch.empty(api.norm_grouped_workspace_size(norm_mods, torch.bfloat16),
                      dtype=torch.uint8, device=dev)
    cws = torch.empty(65536, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # the weights keep their buffers from step to step: the grouped norm is
    # prepared once (tables and tensor maps) and each step only launches
    plan = api.dora_norm_grouped_plan_create(norm_mods, wnorms=wns, gs=gss, workspace=nws)

    def step(evs=None, oneshot=False):
        if oneshot:
            api.dora_factored_norm_grouped(norm_mods, cfg.s, cfg.eps, wnorms=wns, gs=gss,
                                           workspace=nws)
        else:
            plan.run(cfg.s, cfg.eps)
        if evs is not None:
            evs[1].record(stream)
        api.dora_compose_grouped(comp_mods, cfg.s, outs=outs, workspace=cws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in evs:
        e[0].record(stream)
        step(e)
        e[2].record(stream)
    torch.cuda.synchronize()
    norm_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in evs)
    comp_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in evs)
    for e in evs:
        e[0].record(stream)
        step(e, oneshot=True)
        e[2].record(stream)
    torch.cuda.synchronize()
    oneshot_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in evs)
    plan.destroy()
    nbytes = sum(configs.norm_bytes(d["mod"].d_out, d["mod"].d_in, cfg.r, cfg.dtype) for d in mods)
    nflops = sum(configs.norm_flops(d["mod"].d_out, d["mod"].d_in, cfg.r) for d in mods)
    cbytes = sum(configs.compose_bytes(cfg.tokens, d["mod"].d_out, cfg.dtype) for d in mods)
    out = {"workload": cfg.name, "modules": len(mods), "r": cfg.r, "tokens": cfg.tokens,
           "norm_ms": norm_ms, "norm_GB/s": nbytes / (norm_ms * 1e-3) / 1e9,
           "norm_frac_of_measured_hbm": nbytes / (norm_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "norm_TFLOP/s": nflops / (norm_ms * 1e-3) / 1e12,
           "compose_ms": comp_ms, "compose_GB/s": cbytes / (comp_ms * 1e-3) / 1e9,
           "compose_frac_of_measured_hbm": cbytes / (comp_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "modules_per_s": len(mods) / ((norm_ms + comp_ms) * 1e-3),
           "norm_unplanned_ms": oneshot_ms,
           "calls": "dora_norm_grouped_plan_run (plan created once, before timing) + "
                    "dora_compose_grouped, one launch sequence each for all 196 modules; "
                    "norm_unplanned_ms: dora_factored_norm_grouped, which encodes and copies "
                    "the module tables on every call",
           "data": "drawn on the device (torch.randn, seeded) with the config's distributions; "
                   "m = 1 (timing only)",
           "timing": f"CUDA events, mean over {steps} steps"}
    del mods, norm_mods, comp_mods, nws, plan
    torch.cuda.empty_cache()
    return out


def run_fp32(api, dev, peaks, calls=20):
    """The fp32 norm at 8192 x 8192, r = 512 (3xTF32 on the tensor cores)."""
    import torch
    cfg = configs.get(2)
    mod = cfg.module
    d_out, d_in, r = mod.d_out, mod.d_in, cfg.r
    gen_t = torch.Generator(device=dev)
    gen_t.manual_seed(2)
    W = torch.randn(d_out, d_in, device=dev, generator=gen_t) * cfg.std_w
    A = torch.randn(r, d_in, device=dev, generator=gen_t) * cfg.std_a(d_in)
    B = torch.randn(d_out, r, device=dev, generator=gen_t) * cfg.std_b
    m = torch.ones(d_out, device=dev)
    ws = api.alloc_workspace(d_out, d_in, r, torch.float32, device=dev)
    wn = torch.empty(d_out, device=dev)
    g = torch.empty(d_out, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(calls)]
    for e in evs:            # create the CUDA events (the library records e[1], e[2])
        for x in e:
            x.record()
    for _ in range(3):
        api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps, wnorm=wn, g=g, workspace=ws)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # whole calls first; then the main pass alone (events between launches
    # suspend the programmatic overlap, so they are kept out of the first loop)
    for e in evs:
        e[0].record(stream)
        api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps, wnorm=wn, g=g, workspace=ws)
        e[3].record(stream)
    for e in evs:
        api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps, wnorm=wn, g=g, workspace=ws,
                               main_events=(e[1], e[2]))
    torch.cuda.synchronize()
    norm_ms = statistics.fmean(e[0].elapsed_time(e[3]) for e in evs)
    main_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in evs)
    # the same calls back to back, one event pair around the loop (no event
    # between the calls suspends the programmatic chain)
    lp = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    lp[0].record(stream)
    for _ in range(calls):
        api.dora_factored_norm(W, A, B, cfg.s, m, cfg.eps, wnorm=wn, g=g, workspace=ws)
    lp[1].record(stream)
    torch.cuda.synchronize()
    b2b_ms = lp[0].elapsed_time(lp[1]) / calls
    flops = configs.norm_flops(d_out, d_in, r)
    rp = (r + 15) // 16 * 16
    # tensor-core work of the main pass: three TF32 products per fp32 product,
    # over the (W, A) and (B, G') K tiles
    mma_flops = 3 * 2 * d_out * (d_in + rp) * rp
    tf32_peak = peaks["bf16_tflops"] * NOMINAL["tf32_tflops"] / NOMINAL["bf16_tflops"]
    out = {"workload": cfg.name, "dtype": "f32 (3xTF32 tensor-core products, fp32 sums)",
           "norm_us": norm_ms * 1e3, "norm_TFLOP/s": flops / (norm_ms * 1e-3) / 1e12,
           "norm_back_to_back_us": b2b_ms * 1e3,
           "main_pass_us": main_ms * 1e3,
           "main_pass_tf32_TFLOP/s": mma_flops / (main_ms * 1e-3) / 1e12,
           "main_pass_frac_of_measured_derived_tf32": mma_flops / (main_ms * 1e-3) / 1e12 / tf32_peak,
           "tf32_peak_note": "measured bf16 burst x the nominal tf32 / bf16 ratio (1100 / 2250); "
                             "the bf16 figure is cuBLAS's achieved rate, so a kernel may read "
                             "a little above 1.0 against it",
           # against the issue rate the tensor counter implies for TF32 (4096
           # FLOP per clock per SM, half the bf16 rate) at the maximum SM clock
           "main_pass_frac_of_tf32_issue_rate": mma_flops / (main_ms * 1e-3) / 1e12
           / (4096 * 152 * 2.07e9 / 1e12),
           # W, A, B, G' once; the segment partials (at most 16 + 16 fp32 per row)
           "main_pass_algorithmic_bytes": 4 * (d_out * d_in + r * d_in + d_out * r + rp * rp),
           "main_pass_traffic": recorded_traffic(
               os.path.join(ROOT, "dora_parameter_efficient_gb300", "csrc", "gemm_tf32.cu"),
               "tf32_pass_8192x8192_r512_f32.md"),
           "data": "drawn on the device (torch.randn, seeded) with the config's distributions; "
                   "m = 1 (timing only)",
           "timing": f"CUDA events around each call, mean over {calls} calls; "
                     f"norm_back_to_back_us: {calls} calls inside one event pair "
                     f"(W is 256 MB, larger than L2)"}
    del W, A, B, m, ws, wn, g
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from dora_parameter_efficient_gb300 import _lib, api

    cfg = configs.get(CFG_INDEX)
    mod = cfg.module
    d_out, d_in, r, T = mod.d_out, mod.d_in, cfg.r, cfg.tokens
    peaks, peak_src = load_peaks()

    # ---- inputs: this rank's module (weak scaling: one independent module per rank)
    norm_x = gen.norm_inputs(cfg, seed=rank)
    comp_x = gen.compose_inputs(cfg, seed=rank)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    set0 = {k: to_dev(v) for k, v in {**norm_x, **comp_x}.items()}
    sets = [set0] + [{k: v.clone() for k, v in set0.items()} for _ in range(N_SETS - 1)]
    wn = [torch.empty(d_out, dtype=torch.float32, device=dev) for _ in range(N_SETS)]
    gg = [torch.empty(d_out, dtype=torch.float32, device=dev) for _ in range(N_SETS)]
    outs = [torch.empty((T, d_out), dtype=torch.bfloat16, device=dev) for _ in range(N_SETS)]
    ws = [api.alloc_workspace(d_out, d_in, r, torch.bfloat16, dev) for _ in range(N_SETS)]
    stream = torch.cuda.current_stream()
    set_bytes = sum(v.numel() * v.element_size() for v in set0.values())

    def step(i, evs=None, main=False):
        # main=True also records evs[1] / evs[2] right around the main-pass
        # launch; events between launches suspend the programmatic overlap of
        # that kernel with its neighbours, so the timed steps leave them out
        k = i % N_SETS
        s = sets[k]
        api.dora_factored_norm(s["W"], s["A"], s["B"], cfg.s, s["m"], cfg.eps, wnorm=wn[k],
                               g=gg[k], workspace=ws[k],
                               main_events=(evs[1], evs[2]) if (evs is not None and main) else None)
        if evs is not None:
            evs[3].record(stream)
        api.dora_compose(s["base"], s["lora"], gg[k], cfg.s, out=outs[k])

    # ---- warm-up (also starts the clock sampler so it is running by the timed region)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t_spin = time.time()
    i = args.warmup
    while time.time() - t_spin < 0.6:          # keep the GPU loaded until the sampler reports
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()
    for k in range(N_SETS):
        assert api.dora_check_status(ws[k]) == 0, "device pipeline reported a timeout"

    # ---- timed region: exactly K steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for e in evs:            # create the CUDA events before the timed region
        for x in e:
            x.record(stream)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    launches0 = _lib.load().dora_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    sampler.t_start = time.time()
    # two events per step: after the norm (e[3]) and after the compose (e[4]);
    # a step's norm runs from the previous step's e[4] (t_begin for the first)
    # to its e[3].  Every event recorded between two launches costs the step
    # a few microseconds of overlap, so no third one marks the step start.
    t_begin.record(stream)
    for i in range(args.steps):
        e = evs[i]
        step(i, e)
        e[4].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.t_end = time.time()
    barrier(world)
    launches = _lib.load().dora_launch_count() - launches0
    total_ms = t_begin.elapsed_time(t_end)
    starts = [t_begin] + [e[4] for e in evs[:-1]]
    norm_ms = [a.elapsed_time(e[3]) for a, e in zip(starts, evs)]
    comp_ms = [e[3].elapsed_time(e[4]) for e in evs]

    # ---- main-pass kernel timing: the same steps with events right around the
    # main-pass launch (its stand-alone duration, launch latency included)
    kern_steps = max(3, min(args.steps, 500))
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(kern_steps)]
    for e in kevs:
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for i in range(kern_steps):
        step(i, kevs[i], main=True)
    torch.cuda.synchronize()
    main_ms = [e[1].elapsed_time(e[2]) for e in kevs]

    # ---- back to back: the norm alone, the compose alone and the whole step,
    # each in a loop over the rotating sets with one event pair around the
    # loop and none between launches
    def norm_only(i):
        k = i % N_SETS
        s = sets[k]
        api.dora_factored_norm(s["W"], s["A"], s["B"], cfg.s, s["m"], cfg.eps, wnorm=wn[k],
                               g=gg[k], workspace=ws[k])

    def comp_only(i):
        k = i % N_SETS
        api.dora_compose(sets[k]["base"], sets[k]["lora"], gg[k], cfg.s, out=outs[k])

    def loop_ms(fn, n):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    b2b_n = max(3, min(args.steps, 2000))
    b2b = {"norm_ms": loop_ms(norm_only, b2b_n), "compose_ms": loop_ms(comp_only, b2b_n),
           "step_ms": loop_ms(step, b2b_n), "calls_per_loop": b2b_n}

    # ---- the same three loops captured once as CUDA graphs of 30 calls (ten
    # rounds of the rotating sets) and replayed: the launch chain without the
    # host's per-call enqueue work
    def graph_ms(fn, calls=30, replays=max(3, min(args.steps // 30, 100))):
        gr = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(gr):
            for i in range(calls):
                fn(i)
        for _ in range(3):
            gr.replay()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(replays):
            gr.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / (replays * calls)
        del gr
        return ms

    graphs = {"norm_ms": graph_ms(norm_only), "compose_ms": graph_ms(comp_only),
              "step_ms": graph_ms(step), "calls_per_graph": 30}
    sampler.stop()
    clocks = sampler.summary()

    mean = statistics.fmean
    ms_per_step = max_over_ranks(total_ms / args.steps, world, dev)
    norm_ms_m = max_over_ranks(mean(norm_ms), world, dev)
    main_ms_m = max_over_ranks(mean(main_ms), world, dev)
    comp_ms_m = max_over_ranks(mean(comp_ms), world, dev)

    nflops = configs.norm_flops(d_out, d_in, r)
    cbytes = configs.compose_bytes(T, d_out, cfg.dtype)
    value = nflops * world / (norm_ms_m * 1e-3) / 1e12
    comp_gbs = cbytes * world / (comp_ms_m * 1e-3) / 1e9
    mflops = main_pass_flops(d_out, d_in, r)
    main_tflops = mflops / (main_ms_m * 1e-3) / 1e12
    main_src = os.path.join(ROOT, "dora_parameter_efficient_gb300", "csrc", "gemm_pair.cu")
    comp_src = os.path.join(ROOT, "dora_parameter_efficient_gb300", "csrc", "compose.cu")
    # the dominant kernel's duration: the period of back-to-back norm calls.
    # Successive main passes never overlap (the next norm's Gram kernel, which
    # zeroes the control words, waits for this grid to complete before the
    # next main pass starts), so the period bounds the kernel's duration from above and the
    # rate below; the isolated figure times the same kernel with events right
    # around its launch, which removes the overlap with the Gram kernel it is
    # scheduled for and adds a launch.
    chain_ms = b2b["norm_ms"]
    main_tflops_chain = mflops / (chain_ms * 1e-3) / 1e12
    roofline = {"kernel": "k_gemm_pair main pass (U = W A^T, the folded B G' tiles, sum W^2, "
                          "rowsum(B o D), the fused finalize) on tcgen05 CTA pairs",
                "bound": "tensor", "achieved": main_tflops_chain,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": main_tflops_chain / peaks["bf16_tflops"],
                "peak_source": f"{peak_src} bf16 burst: the kernel runs about 45 us at a time "
                               f"inside loops of well under a second, at the clock sampled in "
                               f"`clocks` (the sustained figure was taken under the power cap "
                               f"at a lower clock)",
                "frac_of_measured_sustained": main_tflops_chain / peaks["bf16_tflops_sustained"],
                "frac_of_nominal": main_tflops_chain / NOMINAL["bf16_tflops"],
                "flops_per_launch": mflops, "ms_per_launch": chain_ms,
                "timing": f"upper bound of the kernel's duration: the period of {b2b_n} "
                          f"back-to-back norm calls over the rotating sets (Gram -> main pass, a "
                          f"programmatic chain, the Gram kernel zeroing the control words; one "
                          f"CUDA event pair on the launching stream around the loop, none between launches); "
                          f"successive main passes do not overlap, so the period includes the "
                          f"kernel's whole duration plus the gap to the next one",
                "isolated": {"ms_per_launch": main_ms_m, "achieved": main_tflops,
                             "frac": main_tflops / peaks["bf16_tflops"],
                             "timing": f"CUDA events right around the main-pass launch, mean "
                                       f"over {kern_steps} steps (the events suspend the overlap "
                                       f"with the Gram kernel and expose the launch latency)"},
                "traffic": recorded_traffic(main_src, "main_pass_8192x8192_r384.md"),
                # reads W, A, B, G'_hi, G'_lo, m once; writes one pair of fp32
                # partials per row and segment (counted once) and wnorm, g
                "algorithmic_bytes_per_launch": 2 * (d_out * d_in + r * d_in + d_out * r)
                + 2 * 2 * r * r + 2 * d_out + 8 * d_out + 8 * d_out}
    comp_chain_ms = b2b["compose_ms"]
    roofline_compose = {"kernel": "k_compose<bf16>", "bound": "hbm",
                        "achieved": cbytes / (comp_chain_ms * 1e-3) / 1e9,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": cbytes / (comp_chain_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        "frac_of_nominal": cbytes / (comp_chain_ms * 1e-3) / 1e9 / NOMINAL["hbm_gbs"],
                        "peak_source": f"{peak_src} HBM copy", "bytes_per_launch": cbytes,
                        "ms_per_launch": comp_chain_ms,
                        "timing": "period of back-to-back compose calls over the rotating sets "
                                  "(one event pair around the loop)",
                        "in_step": {"ms_per_launch": comp_ms_m,
                                    "achieved": cbytes / (comp_ms_m * 1e-3) / 1e9,
                                    "frac": cbytes / (comp_ms_m * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                    "timing": "compose part of the timed steps (events between "
                                              "the norm and the compose)"},
                        "traffic": recorded_traffic(comp_src, "compose_2048x8192_bf16.md")}

    # ---- training path of the compose (saved inner, dual-output backward,
    # magnitude gradient) on the same activations, timed like the step
    grad_x = gen.grad_inputs(cfg, seed=rank)
    d_outs = [to_dev(grad_x)] + [to_dev(grad_x).clone() for _ in range(N_SETS - 1)]
    inners = [torch.empty_like(outs[0]) for _ in range(N_SETS)]
    d_bases = [torch.empty_like(outs[0]) for _ in range(N_SETS)]
    d_loras = [torch.empty_like(outs[0]) for _ in range(N_SETS)]
    dmags = [torch.empty(d_out, dtype=torch.float32, device=dev) for _ in range(N_SETS)]
    bws = torch.empty(api.compose_backward_workspace_size(T, d_out), dtype=torch.uint8, device=dev)

    def train_fwd(k):
        api.dora_compose_train(sets[k]["base"], sets[k]["lora"], gg[k], cfg.s, out=outs[k],
                               inner=inners[k])

    def train_bwd(k):
        api.dora_compose_backward(d_outs[k], gg[k], cfg.s, inner=inners[k], wnorm=wn[k],
                                  eps=cfg.eps, d_base=d_bases[k], d_lora=d_loras[k],
                                  dmag=dmags[k], workspace=bws)

    train_steps = max(3, min(args.steps, 500))
    for i in range(max(3, args.warmup)):
        train_fwd(i % N_SETS)
        train_bwd(i % N_SETS)
    tevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(train_steps)]
    for e in tevs:
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for i in range(train_steps):
        e = tevs[i]
        e[0].record(stream)
        train_fwd(i % N_SETS)
        e[1].record(stream)
        train_bwd(i % N_SETS)
        e[2].record(stream)
    torch.cuda.synchronize()
    tf_ms = max_over_ranks(mean(e[0].elapsed_time(e[1]) for e in tevs), world, dev)
    tb_ms = max_over_ranks(mean(e[1].elapsed_time(e[2]) for e in tevs), world, dev)
    tf_bytes = configs.compose_train_bytes(T, d_out, cfg.dtype)
    tb_bytes = configs.compose_backward_bytes(T, d_out, cfg.dtype, dmag=True)
    compose_training = {
        "forward": {"kernel": "k_train_fwd_cols<bf16> (out and inner = base + s lora)",
                    "ms": tf_ms, "GB/s": tf_bytes / (tf_ms * 1e-3) / 1e9,
                    "bytes_per_launch": tf_bytes,
                    "frac_of_measured_hbm": tf_bytes / (tf_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "backward": {"kernel": "k_train_bwd_cols<bf16, dmag> + k_train_dm_finish "
                               "(d_base, d_lora, deterministic dmag column sums)",
                     "ms": tb_ms, "GB/s": tb_bytes / (tb_ms * 1e-3) / 1e9,
                     "bytes_per_call": tb_bytes,
                     "frac_of_measured_hbm": tb_bytes / (tb_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "timing": f"CUDA events around each call, mean over {train_steps} steps, "
                  f"{N_SETS} rotating input sets",
    }
    # the same kernels back to back: forward alone, and forward + backward
    # (one event pair around each loop, none between launches)
    tf_b2b = loop_ms(lambda i: train_fwd(i % N_SETS), train_steps)
    tfb_b2b = loop_ms(lambda i: (train_fwd(i % N_SETS), train_bwd(i % N_SETS)), train_steps)
    tb_b2b = tfb_b2b - tf_b2b
    compose_training["back_to_back"] = {
        "forward_ms": tf_b2b, "forward_GB/s": tf_bytes / (tf_b2b * 1e-3) / 1e9,
        "forward_frac_of_measured_hbm": tf_bytes / (tf_b2b * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "backward_ms": tb_b2b, "backward_GB/s": tb_bytes / (tb_b2b * 1e-3) / 1e9,
        "backward_frac_of_measured_hbm": tb_bytes / (tb_b2b * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "timing": f"loops of {train_steps} forwards and of {train_steps} forward + backward "
                  f"pairs over the rotating sets, one event pair around each loop; backward = "
                  f"the pair's time minus the forward's"}

    # ---- the 7B-like stack (196 modules, r = 128): grouped norm + compose,
    # one launch sequence per step for all modules; inputs drawn on the
    # device with the config's distributions (m = 1: timing only; the parity
    # of the grouped calls is in tests/test_grouped_gpu.py)
    stack = run_stack(api, dev, peaks) if not args.no_stack else None
    # ---- the fp32 norm (8192 x 8192, r = 512), outside the timed step
    fp32_norm = run_fp32(api, dev, peaks) if not args.no_stack else None

    # ---- end to end through the public API, from pinned host buffers
    e2e_steps = max(3, min(args.steps, 20))
    host = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).pin_memory()
            for k, v in {**norm_x, **comp_x}.items()}
    out_h = torch.empty((T, d_out), dtype=torch.bfloat16).pin_memory()
    g_h = torch.empty(d_out, dtype=torch.float32).pin_memory()
    wn_h = torch.empty(d_out, dtype=torch.float32).pin_memory()
    dbuf = sets[0]
    norm_keys = ("W", "A", "B", "m")
    comp_keys = ("base", "lora")

    def e2e_step(ev):
        ev[0].record(stream)
        for k in norm_keys:
            dbuf[k].copy_(host[k], non_blocking=True)
        api.dora_factored_norm(dbuf["W"], dbuf["A"], dbuf["B"], cfg.s, dbuf["m"], cfg.eps,
                               wnorm=wn[0], g=gg[0], workspace=ws[0])
        g_h.copy_(gg[0], non_blocking=True)
        wn_h.copy_(wn[0], non_blocking=True)
        ev[1].record(stream)
        for k in comp_keys:
            dbuf[k].copy_(host[k], non_blocking=True)
        api.dora_compose(dbuf["base"], dbuf["lora"], gg[0], cfg.s, out=outs[0])
        out_h.copy_(outs[0], non_blocking=True)
        ev[2].record(stream)

    for _ in range(2):
        e2e_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize()
    e2e_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(e2e_steps)]
    barrier(world)
    torch.cuda.synchronize()
    for ev in e2e_evs:
        e2e_step(ev)
    torch.cuda.synchronize()
    barrier(world)
    e2e_norm_ms = max_over_ranks(mean(e[0].elapsed_time(e[1]) for e in e2e_evs), world, dev)
    e2e_comp_ms = max_over_ranks(mean(e[1].elapsed_time(e[2]) for e in e2e_evs), world, dev)
    h2d = sum(host[k].numel() * host[k].element_size() for k in norm_keys + comp_keys)
    d2h = out_h.numel() * 2 + 8 * d_out
    e2e = {"value": nflops * world / (e2e_norm_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "ms_per_step": e2e_norm_ms + e2e_comp_ms,
           "compose": {"value": cbytes * world / (e2e_comp_ms * 1e-3) / 1e9, "unit": "GB/s"},
           "api": "dora_factored_norm + dora_compose (Python binding of the C ABI) with "
                  "pinned-host H2D of W, A, B, m, base, lora and D2H of wnorm, g, out"}

    # ---- CPU baseline: the oracle on this host, bounded sample (rank 0, N = 1 only)
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # whole passes of the workload (all rows, all token rows) until about
        # 10 s of CPU time has gone by
        rows = np.arange(d_out)
        toks = np.arange(T)
        g32 = gg[0].cpu().numpy()
        tn = tc = 0.0
        passes = 0
        while passes < 1 or tn + tc < 10.0:
            a, b = oracle_sample(cfg, norm_x, comp_x, g32, rows, toks)
            tn += a
            tc += b
            passes += 1
        cpu_value = nflops * passes / tn / 1e12
        threads, threads_how = blas_threads()
        st_rows, st_toks = 1024, 256
        st = single_thread_oracle(st_rows, st_toks)
        single = None
        if st is not None:
            single = {"value": nflops / d_out * st_rows * st["reps"] / st["norm_s"] / 1e12,
                      "unit": "TFLOP/s", "threads": 1,
                      "compose": {"value": configs.compose_bytes(st_toks, d_out, cfg.dtype)
                                  * st["reps"] / st["compose_s"] / 1e9, "unit": "GB/s"},
                      "sample": f"the first {st_rows} norm rows and {st_toks} compose token rows, "
                                f"{st['reps']} repetitions ({st['norm_s']:.1f} s norm, "
                                f"{st['compose_s']:.1f} s compose) in a fresh interpreter with "
                                f"OPENBLAS_NUM_THREADS = OMP_NUM_THREADS = 1"}
        cpu_baseline = {"value": cpu_value, "unit": "TFLOP/s", "cores": threads,
                        "cores_how": f"{threads_how}: the threads of the dense B A product; the "
                                     f"elementwise numpy steps run on one thread",
                        "host_cpus": os.cpu_count(),
                        "kind": "oracle",
                        "sample": f"float64 oracle (dense W+sBA row norms via numpy/OpenBLAS, "
                                  f"compose elementwise) on the whole workload, {passes} passes: "
                                  f"norm of all {d_out} rows ({tn:.1f} s in total), compose of all "
                                  f"{T} token rows ({tc:.1f} s in total); TFLOP/s uses the "
                                  f"method's algorithmic FLOPs",
                        "compose": {"value": cbytes * passes / tc / 1e9, "unit": "GB/s"},
                        "single_thread": single}

    if rank == 0:
        line = {
            "metric": json.loads(BASELINE_METRIC), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "d_out": d_out, "d_in": d_in, "r": r, "s": cfg.s,
                       "tokens": T, "modules_per_rank": 1,
                       "l2": f"{N_SETS} rotating input/output sets, {set_bytes / 1e6:.0f} MB "
                             f"of inputs each (> 129 MB L2)",
                       "parallelism": f"replicas x{world} (one independent module per rank)"},
            "value_definition": "algorithmic factored-norm FLOPs (2 d_out d_in r + 2 r^2 d_in + "
                                "2 d_out r^2 + 2 d_out d_in) / norm part of each timed step",
            "norm": {"tflops": value, "ms": norm_ms_m, "modules_per_s": world / (norm_ms_m * 1e-3),
                     "frac_of_measured_bf16": value / peaks["bf16_tflops"],
                     "frac_of_nominal_bf16": value / NOMINAL["bf16_tflops"]},
            "back_to_back": {
                **b2b,
                "norm_tflops": nflops / (b2b["norm_ms"] * 1e-3) / 1e12,
                "norm_frac_of_measured_bf16": nflops / (b2b["norm_ms"] * 1e-3) / 1e12 / peaks["bf16_tflops"],
                "compose_GB/s": cbytes / (b2b["compose_ms"] * 1e-3) / 1e9,
                "compose_frac_of_measured_hbm": cbytes / (b2b["compose_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "compose_frac_of_nominal_hbm": cbytes / (b2b["compose_ms"] * 1e-3) / 1e9 / NOMINAL["hbm_gbs"],
                "timing": "one CUDA event pair around a loop of calls over the rotating sets "
                          "(no event between launches); per call = loop time / calls"},
            "cuda_graph": {
                **graphs,
                "norm_tflops": nflops / (graphs["norm_ms"] * 1e-3) / 1e12,
                "norm_frac_of_measured_bf16": nflops / (graphs["norm_ms"] * 1e-3) / 1e12 / peaks["bf16_tflops"],
                "compose_GB/s": cbytes / (graphs["compose_ms"] * 1e-3) / 1e9,
                "compose_frac_of_measured_hbm": cbytes / (graphs["compose_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "compose_frac_of_nominal_hbm": cbytes / (graphs["compose_ms"] * 1e-3) / 1e9 / NOMINAL["hbm_gbs"],
                "timing": "each loop captured once as a CUDA graph of 30 calls over the rotating "
                          "sets, one event pair around the replays; per call = time / calls"},
            "compose": {"value": comp_gbs, "unit": "GB/s", "ms": comp_ms_m,
                        "elements_per_s": T * d_out * world / (comp_ms_m * 1e-3),
                        "frac_of_measured_hbm": comp_gbs / world / peaks["hbm_gbs"],
                        "frac_of_nominal_hbm": comp_gbs / world / NOMINAL["hbm_gbs"]},
            "roofline": roofline, "roofline_compose": roofline_compose,
            "compose_training": compose_training,
            "stack": stack,
            "fp32_norm": fp32_norm,
            "clocks": clocks, "e2e": e2e, "gpu_launches": int(launches),
            "cpu_baseline": cpu_baseline,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
