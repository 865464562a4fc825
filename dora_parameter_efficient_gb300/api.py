"""Python binding of the dora C ABI with the same names, for torch tensors.

Argument marshalling only: every step of the norm and the compose runs in the
CUDA kernels of ``libdora.so``.  torch supplies device memory, streams and
events; nothing here computes on tensor values.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import DORA_BF16, DORA_F32, DoraError, check

_DTYPES = {torch.bfloat16: DORA_BF16, torch.float32: DORA_F32}


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"dtype {t.dtype} is not supported (bfloat16 or float32)") from None


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def workspace_size(d_out: int, d_in: int, r: int, dtype: torch.dtype) -> int:
    return int(_lib.load().dora_norm_workspace_size(d_out, d_in, r, _DTYPES[dtype]))


def alloc_workspace(d_out: int, d_in: int, r: int, dtype: torch.dtype,
                    device="cuda") -> torch.Tensor:
    n = workspace_size(d_out, d_in, r, dtype)
    if n == 0:
        raise ValueError("invalid shape for dora_factored_norm")
    return torch.empty(n, dtype=torch.uint8, device=device)


def dora_factored_norm(W: torch.Tensor, A: torch.Tensor, B: torch.Tensor, s: float,
                       m: torch.Tensor, eps: float,
                       wnorm: Optional[torch.Tensor] = None, g: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None,
                       main_events: Optional[Tuple[torch.cuda.Event, torch.cuda.Event]] = None,
                       ) -> Tuple[torch.Tensor, torch.Tensor]:
    """wnorm = ||W + s B A||_row and g = m / max(wnorm, eps), both fp32 [d_out].

    W [d_out, d_in], A [r, d_in], B [d_out, r], m [d_out], all one dtype
    (bfloat16 or float32), contiguous, on the current CUDA device."""
    code = _dtype_code(W)
    for t, name in ((A, "A"), (B, "B"), (m, "m")):
        if t.dtype != W.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, W has {W.dtype}")
    d_out, d_in = W.shape
    r = A.shape[0]
    if A.shape != (r, d_in) or B.shape != (d_out, r) or m.shape != (d_out,):
        raise ValueError(f"shape mismatch: W{tuple(W.shape)} A{tuple(A.shape)} "
                         f"B{tuple(B.shape)} m{tuple(m.shape)}")
    if wnorm is None:
        wnorm = torch.empty(d_out, dtype=torch.float32, device=W.device)
    if g is None:
        g = torch.empty(d_out, dtype=torch.float32, device=W.device)
    if workspace is None:
        workspace = alloc_workspace(d_out, d_in, r, W.dtype, W.device)
    lib = _lib.load()
    args = (_dev(W, "W"), _dev(A, "A"), _dev(B, "B"), code, d_out, d_in, r, float(s),
            _dev(m, "m"), float(eps), _dev(wnorm, "wnorm"), _dev(g, "g"),
            _dev(workspace, "workspace"), workspace.numel(), _stream_handle(stream))
    if main_events is None:
        st = lib.dora_factored_norm(*args)
    else:
        st = lib.dora_factored_norm_timed(*args, main_events[0].cuda_event,
                                          main_events[1].cuda_event)
    check(st, "dora_factored_norm")
    return wnorm, g


# ---------------------------------------------------------------- d_in-sharded norm
def norm_partials_floats(d_out: int, r: int) -> int:
    """Length of the partials buffer: 2 d_out + r^2 float32 values."""
    return 2 * int(d_out) + int(r) * int(r)


def partials_views(partials: torch.Tensor, d_out: int, r: int):
    """(base [d_out], cross [d_out], G [r, r]) views of a partials buffer."""
    if partials.dim() != 1 or partials.numel() != norm_partials_floats(d_out, r):
        raise ValueError(f"partials must be 1-D with {norm_partials_floats(d_out, r)} values")
    return (partials[:d_out], partials[d_out:2 * d_out],
            partials[2 * d_out:].view(int(r), int(r)))


def slice_bounds(d_in: int, parts: int, index: int, dtype: torch.dtype) -> Tuple[int, int]:
    """Columns [k0, k1) of d_in held by slice `index` of `parts` when W and A
    are split along d_in: near-equal widths on a 64-column grid (the main
    pass's K tile), so every slice's rows stay 16-byte multiples; the last
    slice takes the remainder.  Host logic only."""
    if parts < 1 or not 0 <= index < parts or d_in < 0:
        raise ValueError("need parts >= 1, 0 <= index < parts and d_in >= 0")
    eb = torch.tensor([], dtype=dtype).element_size()
    if (d_in * eb) % 16 != 0:
        raise ValueError("d_in * element size must be a multiple of 16 bytes")
    tiles = -(-d_in // 64)
    k0 = min(d_in, (tiles * index // parts) * 64)
    k1 = d_in if index == parts - 1 else min(d_in, (tiles * (index + 1) // parts) * 64)
    return k0, k1


def dora_norm_partials(W: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                       partials: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The partials of one d_in slice: base = sum W^2, cross = rowsum(B o (W A^T))
    and G = A A^T over the slice's columns, as one float32 buffer
    [2 d_out + r^2] (W [d_out, d_in_slice], A [r, d_in_slice], B [d_out, r])."""
    code = _dtype_code(W)
    for t, name in ((A, "A"), (B, "B")):
        if t.dtype != W.dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, W has {W.dtype}")
    d_out, d_in = W.shape
    r = A.shape[0]
    if A.shape != (r, d_in) or B.shape != (d_out, r):
        raise ValueError(f"shape mismatch: W{tuple(W.shape)} A{tuple(A.shape)} B{tuple(B.shape)}")
    n = norm_partials_floats(d_out, r)
    if partials is None:
        partials = torch.empty(n, dtype=torch.float32, device=W.device)
    elif partials.dtype != torch.float32 or partials.numel() != n:
        raise ValueError(f"partials must be float32 with {n} values")
    if workspace is None:
        workspace = alloc_workspace(d_out, d_in, r, W.dtype, W.device)
    st = _lib.load().dora_norm_partials(_dev(W, "W"), _dev(A, "A"), _dev(B, "B"), code, d_out,
                                        d_in, r, _dev(partials, "partials"),
                                        _dev(workspace, "workspace"), workspace.numel(),
                                        _stream_handle(stream))
    check(st, "dora_norm_partials")
    return partials


def finalize_workspace_size(d_out: int, r: int, dtype: torch.dtype) -> int:
    return int(_lib.load().dora_norm_finalize_workspace_size(d_out, r, _DTYPES[dtype]))


def dora_norm_finalize_partials(partials: torch.Tensor, B: torch.Tensor, s: float,
                                m: torch.Tensor, eps: float,
                                wnorm: Optional[torch.Tensor] = None,
                                g: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                stream: Optional[torch.cuda.Stream] = None
                                ) -> Tuple[torch.Tensor, torch.Tensor]:
    """wnorm and g from partials summed over every d_in slice (B [d_out, r],
    m [d_out] in the inputs' dtype)."""
    code = _dtype_code(B)
    d_out, r = B.shape
    if m.dtype != B.dtype or m.shape != (d_out,):
        raise ValueError("m must match B's dtype and have d_out values")
    if partials.dtype != torch.float32 or partials.numel() != norm_partials_floats(d_out, r):
        raise ValueError("partials must be float32 [2 d_out + r^2]")
    if wnorm is None:
        wnorm = torch.empty(d_out, dtype=torch.float32, device=B.device)
    if g is None:
        g = torch.empty(d_out, dtype=torch.float32, device=B.device)
    if workspace is None:
        n = finalize_workspace_size(d_out, r, B.dtype)
        if n == 0:
            raise ValueError("invalid shape for dora_norm_finalize_partials")
        workspace = torch.empty(n, dtype=torch.uint8, device=B.device)
    st = _lib.load().dora_norm_finalize_partials(
        _dev(partials, "partials"), _dev(B, "B"), code, d_out, r, float(s), _dev(m, "m"),
        float(eps), _dev(wnorm, "wnorm"), _dev(g, "g"), _dev(workspace, "workspace"),
        workspace.numel(), _stream_handle(stream))
    check(st, "dora_norm_finalize_partials")
    return wnorm, g


def allreduce_partials(partials: torch.Tensor, group=None) -> torch.Tensor:
    """The one exchange of the d_in-sharded norm: the partials of every rank
    of `group` summed in place (torch.distributed all-reduce; NCCL between
    GPUs).  The sum's order is the collective's, so results agree with the
    single-device norm up to fp32 rounding of the partials."""
    import torch.distributed as dist
    dist.all_reduce(partials, op=dist.ReduceOp.SUM, group=group)
    return partials


def dora_factored_norm_sharded(W: torch.Tensor, A: torch.Tensor, B: torch.Tensor, s: float,
                               m: torch.Tensor, eps: float, group=None
                               ) -> Tuple[torch.Tensor, torch.Tensor]:
    """The norm of a module whose W and A are split along d_in over the ranks
    of `group` (this rank holds W [d_out, d_in_slice], A [r, d_in_slice] and
    all of B and m): the slice's partials, one all-reduce of 2 d_out + r^2
    floats, then wnorm and g for every row on every rank."""
    partials = dora_norm_partials(W, A, B)
    allreduce_partials(partials, group)
    return dora_norm_finalize_partials(partials, B, s, m, eps)


def dora_compose(base: torch.Tensor, lora: torch.Tensor, g: torch.Tensor, s: float,
                 out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out = (g - 1) * base + g * (s * lora); base/lora/out [T, d_out], g fp32 [d_out]."""
    code = _dtype_code(base)
    if lora.dtype != base.dtype or lora.shape != base.shape:
        raise ValueError("base and lora must have the same dtype and shape")
    if base.dim() != 2:
        raise ValueError("base must be 2-D [T, d_out]")
    T, d_out = base.shape
    if g.dtype != torch.float32 or g.shape != (d_out,):
        raise ValueError("g must be float32 [d_out]")
    if out is None:
        out = torch.empty_like(base)
    elif out.dtype != base.dtype or out.shape != base.shape:
        raise ValueError("out must match base")
    if T == 0 or d_out == 0:
        return out
    st = _lib.load().dora_compose(_dev(base, "base"), _dev(lora, "lora"), _dev(g, "g"),
                                  float(s), code, T, d_out, _dev(out, "out"),
                                  _stream_handle(stream))
    check(st, "dora_compose")
    return out


def _norm_table(modules, wnorms, gs):
    table = (_lib.NormModule * len(modules))()
    for i, (W, A, B, m) in enumerate(modules):
        d_out, d_in = W.shape
        table[i] = _lib.NormModule(_dev(W, "W"), _dev(A, "A"), _dev(B, "B"), _dev(m, "m"),
                                   _dev(wnorms[i], "wnorm"), _dev(gs[i], "g"), d_out, d_in)
    return table


def norm_grouped_workspace_size(modules, dtype: torch.dtype) -> int:
    r = modules[0][1].shape[0] if modules else 0
    table = (_lib.NormModule * len(modules))()
    for i, (W, A, B, m) in enumerate(modules):
        table[i] = _lib.NormModule(None, None, None, None, None, None, W.shape[0], W.shape[1])
    return int(_lib.load().dora_norm_grouped_workspace_size(table, len(modules), r, _DTYPES[dtype]))


def _grouped_norm_args(modules, wnorms, gs, workspace):
    """Checks a grouped norm's modules and allocates what the caller left out;
    returns (dtype code, r, wnorms, gs, workspace)."""
    W0, A0 = modules[0][0], modules[0][1]
    code = _dtype_code(W0)
    r = A0.shape[0]
    for W, A, B, m in modules:
        if any(t.dtype != W0.dtype for t in (W, A, B, m)):
            raise TypeError("every tensor of a grouped call must have one dtype")
        if A.shape[0] != r or A.shape[1] != W.shape[1] or B.shape != (W.shape[0], r) \
                or m.shape != (W.shape[0],):
            raise ValueError("shape mismatch in a grouped module (one rank for all modules)")
    dev = W0.device
    wnorms = [torch.empty(W.shape[0], dtype=torch.float32, device=dev) for W, *_ in modules] \
        if wnorms is None else list(wnorms)
    gs = [torch.empty(W.shape[0], dtype=torch.float32, device=dev) for W, *_ in modules] \
        if gs is None else list(gs)
    if workspace is None:
        workspace = torch.empty(max(256, norm_grouped_workspace_size(modules, W0.dtype)),
                                dtype=torch.uint8, device=dev)
    return code, r, wnorms, gs, workspace


def dora_factored_norm_grouped(modules, s: float, eps: float, wnorms=None, gs=None,
                               workspace: Optional[torch.Tensor] = None,
                               stream: Optional[torch.cuda.Stream] = None):
    """dora_factored_norm for a list of modules (W, A, B, m), all of one rank and
    dtype, in one launch sequence; returns the lists (wnorms, gs)."""
    modules = list(modules)
    if not modules:
        return [], []
    code, r, wnorms, gs, workspace = _grouped_norm_args(modules, wnorms, gs, workspace)
    table = _norm_table(modules, wnorms, gs)
    st = _lib.load().dora_factored_norm_grouped(table, len(modules), code, r, float(s),
                                                float(eps), _dev(workspace, "workspace"),
                                                workspace.numel(), _stream_handle(stream))
    check(st, "dora_factored_norm_grouped")
    return wnorms, gs


class NormGroupedPlan:
    """A dora_norm_grouped_plan: the grouped norm over fixed module buffers,
    prepared once.  It keeps every tensor it refers to (the modules, the
    outputs and the workspace) alive until destroy()."""

    def __init__(self, handle, modules, wnorms, gs, workspace):
        self._handle = handle
        self._keep = (modules, workspace)
        self.wnorms = wnorms
        self.gs = gs

    def run(self, s: float, eps: float, stream: Optional[torch.cuda.Stream] = None):
        """dora_norm_grouped_plan_run: writes (and returns) the lists (wnorms, gs)."""
        if self._handle is None:
            raise RuntimeError("dora_norm_grouped_plan_run on a destroyed plan")
        st = _lib.load().dora_norm_grouped_plan_run(self._handle, float(s), float(eps),
                                                    _stream_handle(stream))
        check(st, "dora_norm_grouped_plan_run")
        return self.wnorms, self.gs

    def destroy(self):
        """dora_norm_grouped_plan_destroy, after the device has finished every run."""
        if self._handle is not None:
            torch.cuda.synchronize(self._keep[1].device)
            _lib.load().dora_norm_grouped_plan_destroy(self._handle)
            self._handle = None
            self._keep = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def dora_norm_grouped_plan_create(modules, wnorms=None, gs=None,
                                  workspace: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None) -> NormGroupedPlan:
    """Prepares the grouped norm of `modules` (W, A, B, m) once; the returned
    plan's run(s, eps) is dora_factored_norm_grouped without the per-call
    host work.  The tensors must keep their storage (update them in place)."""
    modules = [tuple(m) for m in modules]
    if not modules:
        raise ValueError("a grouped norm plan needs at least one module")
    code, r, wnorms, gs, workspace = _grouped_norm_args(modules, wnorms, gs, workspace)
    table = _norm_table(modules, wnorms, gs)
    handle = ctypes.c_void_p()
    st = _lib.load().dora_norm_grouped_plan_create(table, len(modules), code, r,
                                                   _dev(workspace, "workspace"),
                                                   workspace.numel(), _stream_handle(stream),
                                                   ctypes.byref(handle))
    check(st, "dora_norm_grouped_plan_create")
    return NormGroupedPlan(handle, modules, wnorms, gs, workspace)


def dora_compose_grouped(modules, s: float, outs=None, workspace: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None):
    """dora_compose for a list of modules (base, lora, g) of one dtype, in one
    launch; returns the list of outputs."""
    modules = list(modules)
    if not modules:
        return []
    code = _dtype_code(modules[0][0])
    outs = [torch.empty_like(b) for b, _, _ in modules] if outs is None else outs
    table = (_lib.ComposeModule * len(modules))()
    for i, (base, lora, g) in enumerate(modules):
        if lora.shape != base.shape or base.dim() != 2 or g.shape != (base.shape[1],) \
                or g.dtype != torch.float32 or lora.dtype != base.dtype:
            raise ValueError("grouped compose module: base, lora [T, d_out] of one dtype, g fp32 [d_out]")
        table[i] = _lib.ComposeModule(_dev(base, "base"), _dev(lora, "lora"), _dev(g, "g"),
                                      _dev(outs[i], "out"), base.shape[0], base.shape[1])
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(max(256, lib.dora_compose_grouped_workspace_size(len(modules))),
                                dtype=torch.uint8, device=modules[0][0].device)
    st = lib.dora_compose_grouped(table, len(modules), float(s), code, _dev(workspace, "workspace"),
                                  workspace.numel(), _stream_handle(stream))
    check(st, "dora_compose_grouped")
    return outs


def dora_compose_train(base: torch.Tensor, lora: torch.Tensor, g: torch.Tensor, s: float,
                       out: Optional[torch.Tensor] = None, inner: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None
                       ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Training forward: out as dora_compose and inner = base + s * lora (the
    activation the magnitude gradient needs), written in one pass."""
    code = _dtype_code(base)
    if lora.dtype != base.dtype or lora.shape != base.shape or base.dim() != 2:
        raise ValueError("base and lora must be 2-D [T, d_out] of one dtype")
    T, d_out = base.shape
    if g.dtype != torch.float32 or g.shape != (d_out,):
        raise ValueError("g must be float32 [d_out]")
    out = torch.empty_like(base) if out is None else out
    inner = torch.empty_like(base) if inner is None else inner
    for t, name in ((out, "out"), (inner, "inner")):
        if t.dtype != base.dtype or t.shape != base.shape:
            raise ValueError(f"{name} must match base")
    if T == 0 or d_out == 0:
        return out, inner
    st = _lib.load().dora_compose_train(_dev(base, "base"), _dev(lora, "lora"), _dev(g, "g"),
                                        float(s), code, T, d_out, _dev(out, "out"),
                                        _dev(inner, "inner"), _stream_handle(stream))
    check(st, "dora_compose_train")
    return out, inner


def compose_backward_workspace_size(T: int, d_out: int) -> int:
    return int(_lib.load().dora_compose_backward_workspace_size(T, d_out))


def dora_compose_backward(d_out_grad: torch.Tensor, g: torch.Tensor, s: float,
                          inner: Optional[torch.Tensor] = None,
                          wnorm: Optional[torch.Tensor] = None, eps: float = 1e-6,
                          d_base: Optional[torch.Tensor] = None,
                          d_lora: Optional[torch.Tensor] = None,
                          dmag: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None):
    """Backward of the compose: (d_base, d_lora, dmag).  dmag is computed when
    inner and wnorm are given (a trainable magnitude), else it is None."""
    code = _dtype_code(d_out_grad)
    if d_out_grad.dim() != 2:
        raise ValueError("d_out_grad must be 2-D [T, d_out]")
    T, d_out = d_out_grad.shape
    if g.dtype != torch.float32 or g.shape != (d_out,):
        raise ValueError("g must be float32 [d_out]")
    d_base = torch.empty_like(d_out_grad) if d_base is None else d_base
    d_lora = torch.empty_like(d_out_grad) if d_lora is None else d_lora
    want_dm = inner is not None
    if want_dm:
        if wnorm is None or wnorm.dtype != torch.float32 or wnorm.shape != (d_out,):
            raise ValueError("wnorm must be float32 [d_out] when inner is given")
        if inner.dtype != d_out_grad.dtype or inner.shape != d_out_grad.shape:
            raise ValueError("inner must match d_out_grad")
        dmag = torch.empty(d_out, dtype=torch.float32, device=d_out_grad.device) \
            if dmag is None else dmag
        if workspace is None:
            workspace = torch.empty(max(16, compose_backward_workspace_size(T, d_out)),
                                    dtype=torch.uint8, device=d_out_grad.device)
    if T == 0 or d_out == 0:
        return d_base, d_lora, dmag if want_dm else None
    st = _lib.load().dora_compose_backward(
        _dev(d_out_grad, "d_out_grad"), _dev(inner, "inner") if want_dm else None, _dev(g, "g"),
        _dev(wnorm, "wnorm") if want_dm else None, float(eps), float(s), code, T, d_out,
        _dev(d_base, "d_base"), _dev(d_lora, "d_lora"), _dev(dmag, "dmag") if want_dm else None,
        _dev(workspace, "workspace") if want_dm else None,
        workspace.numel() if want_dm else 0, _stream_handle(stream))
    check(st, "dora_compose_backward")
    return d_base, d_lora, dmag if want_dm else None


def dora_check_status(workspace: torch.Tensor,
                      stream: Optional[torch.cuda.Stream] = None) -> int:
    """Device status word of the last dora_factored_norm on this workspace
    (waits for the stream)."""
    return int(_lib.load().dora_check_status(_dev(workspace, "workspace"),
                                             _stream_handle(stream)))


def dora_selftest_timeout(workspace: torch.Tensor, timeout_us: int,
                          stream: Optional[torch.cuda.Stream] = None) -> None:
    """Enqueues the failure-detection self-test on `workspace` (a wait that
    runs out after `timeout_us` and records DORA_ERR_TIMEOUT; read it with
    dora_check_status)."""
    st = _lib.load().dora_selftest_timeout(_dev(workspace, "workspace"), workspace.numel(),
                                           int(timeout_us), _stream_handle(stream))
    check(st, "dora_selftest_timeout")


def dora_selftest_schedule(d_out: int, d_in: int, r: int, clusters: int):
    """Host-only check of the main pass's work decomposition for a bf16
    d_out x d_in module at rank r on `clusters` CTA pairs: returns
    (schedule, most_pieces_of_one_tile, defects) with schedule one of
    SCHEDULE_SEGMENTS, SCHEDULE_RANGES, SCHEDULE_TABLE, SCHEDULE_WHOLE_TABLE;
    defects is 0 when
    every pair tile's K range is covered once, in order, by at most 16
    numbered pieces."""
    sc, mp, df = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    st = _lib.load().dora_selftest_schedule(int(d_out), int(d_in), int(r), int(clusters),
                                            ctypes.byref(sc), ctypes.byref(mp), ctypes.byref(df))
    check(st, "dora_selftest_schedule")
    return int(sc.value), int(mp.value), int(df.value)


SCHEDULE_SEGMENTS = 0   # K segments handed out one by one
SCHEDULE_RANGES = 1     # one static range of (pair tile, K tile) iterations per pair
SCHEDULE_TABLE = 2      # piece table: one K range of one pair tile per pair
SCHEDULE_WHOLE_TABLE = 3  # whole pair tiles per pair, then a piece table over the rest


def dora_selftest_grouped_schedule(shapes, r: int, clusters: int):
    """Host-only check of a grouped main pass's work items for bf16 modules
    of the given (d_out, d_in) shapes at rank r on `clusters` CTA pairs:
    returns (most_pieces_of_one_tile, defects); defects is 0 when the
    module order is longest-K first and every pair tile of every module is
    covered once, in order, by at most 16 numbered pieces."""
    n = len(shapes)
    d_out = (ctypes.c_int64 * max(n, 1))(*[int(a) for a, _ in shapes])
    d_in = (ctypes.c_int64 * max(n, 1))(*[int(b) for _, b in shapes])
    mp, df = ctypes.c_int(), ctypes.c_int64()
    st = _lib.load().dora_selftest_grouped_schedule(ctypes.addressof(d_out), ctypes.addressof(d_in),
                                                    n, int(r), int(clusters), ctypes.byref(mp),
                                                    ctypes.byref(df))
    check(st, "dora_selftest_grouped_schedule")
    return int(mp.value), int(df.value)


def dora_factored_norm_noalloc(W: torch.Tensor, A: torch.Tensor, B: torch.Tensor, s: float,
                               m: torch.Tensor, eps: float, wnorm: torch.Tensor,
                               g: torch.Tensor,
                               stream: Optional[torch.cuda.Stream] = None) -> None:
    """dora_factored_norm for callers that cannot allocate device memory.

    The caller passes every input and both fp32 [d_out] outputs; the library
    uses its own fixed 32 MiB device scratch (shared by all calls on a device,
    so calls must not overlap on the GPU) and allocates nothing."""
    code = _dtype_code(W)
    d_out, d_in = W.shape
    r = A.shape[0]
    st = _lib.load().dora_factored_norm_noalloc(
        _dev(W, "W"), _dev(A, "A"), _dev(B, "B"), code, d_out, d_in, r, float(s), _dev(m, "m"),
        float(eps), _dev(wnorm, "wnorm"), _dev(g, "g"), _stream_handle(stream))
    check(st, "dora_factored_norm_noalloc")


__all__ = ["dora_factored_norm", "dora_factored_norm_noalloc", "dora_compose",
           "dora_compose_train", "dora_compose_backward", "compose_backward_workspace_size",
           "dora_factored_norm_grouped", "dora_compose_grouped", "norm_grouped_workspace_size",
           "dora_check_status", "workspace_size", "alloc_workspace", "DoraError"]
