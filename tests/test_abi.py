"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU.

None of these calls reaches a CUDA launch: each argument set fails host-side
validation first (the pointers are never dereferenced)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from dora_parameter_efficient_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from dora_parameter_efficient_gb300 import build
        build.build()
    return _lib.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "dora.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dora_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = _declared_functions()
    assert "dora_factored_norm" in names and "dora_compose" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} missing from the Python binding"


def test_status_strings(lib):
    for code in range(7):
        s = _lib.status_string(code)
        assert s.startswith("DORA_")
    assert "unknown" in _lib.status_string(99)
    assert lib.dora_version() >> 16 == 1
    assert lib.dora_version() & 0xFFFF >= 1      # the schedule self-tests


def test_workspace_size(lib):
    n = lib.dora_norm_workspace_size(8192, 8192, 384, _lib.DORA_BF16)
    assert 0 < n < 32 << 20
    # fp32 at 8192^2, r=512: far below the 241 MB the write-up measured for the
    # reference implementation (Chinese write-up section 1.3); most of it is
    # the 24 K-segment partials of G (24 x 512 x 512 fp32), and it still fits
    # the allocation-free entry point's 32 MiB array
    n32 = lib.dora_norm_workspace_size(8192, 8192, 512, _lib.DORA_F32)
    assert 0 < n32 < 32 << 20
    assert lib.dora_norm_workspace_size(8192, 8192, 513, _lib.DORA_BF16) == 0
    assert lib.dora_norm_workspace_size(-1, 8, 8, _lib.DORA_BF16) == 0
    assert lib.dora_norm_workspace_size(8, 8, 8, 7) == 0
    # independent of d_in
    assert (lib.dora_norm_workspace_size(512, 64, 128, _lib.DORA_BF16)
            == lib.dora_norm_workspace_size(512, 1 << 20, 128, _lib.DORA_BF16))


P = 1 << 20      # fake, 256-aligned, never dereferenced


def _norm(lib, **kw):
    a = dict(W=P, A=2 * P, B=3 * P, dtype=_lib.DORA_BF16, d_out=256, d_in=512, r=64, s=1.0,
             m=4 * P, eps=1e-6, wnorm=5 * P, g=6 * P, ws=8 * P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.dora_factored_norm(a["W"], a["A"], a["B"], a["dtype"], a["d_out"], a["d_in"],
                                  a["r"], a["s"], a["m"], a["eps"], a["wnorm"], a["g"], a["ws"],
                                  a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=5), _lib.DORA_ERR_INVALID_ARG),
    (dict(d_out=-1), _lib.DORA_ERR_INVALID_ARG),
    (dict(d_in=-8), _lib.DORA_ERR_INVALID_ARG),
    (dict(r=513), _lib.DORA_ERR_UNSUPPORTED),
    (dict(eps=0.0), _lib.DORA_ERR_INVALID_ARG),
    (dict(eps=-1.0), _lib.DORA_ERR_INVALID_ARG),
    (dict(s=float("nan")), _lib.DORA_ERR_INVALID_ARG),
    (dict(W=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(A=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(m=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(g=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(g=5 * P), _lib.DORA_ERR_INVALID_ARG),              # wnorm == g
    (dict(g=5 * P + 64), _lib.DORA_ERR_INVALID_ARG),         # overlap
    (dict(wnorm=P + 128), _lib.DORA_ERR_INVALID_ARG),        # output inside W
    (dict(d_in=100), _lib.DORA_ERR_UNSUPPORTED),             # 200-byte rows
    (dict(r=60), _lib.DORA_ERR_UNSUPPORTED),                 # 120-byte B rows
    (dict(W=P + 8), _lib.DORA_ERR_UNSUPPORTED),              # misaligned
    (dict(ws=None), _lib.DORA_ERR_WORKSPACE),
    (dict(ws=8 * P + 64), _lib.DORA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), _lib.DORA_ERR_WORKSPACE),
    (dict(d_out=0), _lib.DORA_OK),                           # nothing to do
])
def test_norm_argument_checks(lib, kw, status):
    assert _norm(lib, **kw) == status


def test_norm_fp32_alignment_rule(lib):
    # fp32 rows need a multiple of 4 elements, bf16 a multiple of 8
    assert _norm(lib, dtype=_lib.DORA_F32, d_in=102) == _lib.DORA_ERR_UNSUPPORTED


def _compose(lib, **kw):
    a = dict(base=P, lora=2 * P, g=3 * P, s=1.0, dtype=_lib.DORA_BF16, T=16, d_out=64, out=4 * P,
             stream=None)
    a.update(kw)
    return lib.dora_compose(a["base"], a["lora"], a["g"], a["s"], a["dtype"], a["T"], a["d_out"],
                            a["out"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), _lib.DORA_ERR_INVALID_ARG),
    (dict(dtype=3), _lib.DORA_ERR_INVALID_ARG),
    (dict(s=float("inf")), _lib.DORA_ERR_INVALID_ARG),
    (dict(base=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(out=P + 2), _lib.DORA_ERR_INVALID_ARG),            # partial overlap with base
    (dict(g=4 * P + 8), _lib.DORA_ERR_INVALID_ARG),          # g inside out
    (dict(T=0), _lib.DORA_OK),
    (dict(d_out=0), _lib.DORA_OK),
])
def test_compose_argument_checks(lib, kw, status):
    assert _compose(lib, **kw) == status


def test_check_status_null(lib):
    assert lib.dora_check_status(None, None) == _lib.DORA_ERR_INVALID_ARG


def test_training_compose_rejects_bad_arguments(lib):
    P = 1 << 20
    T, d = 64, 128
    n = T * d * 2
    # forward: null inner, overlapping outputs, bad dtype
    assert lib.dora_compose_train(P, 2 * P, 3 * P, 1.0, _lib.DORA_BF16, T, d, 4 * P, None,
                                  None) == _lib.DORA_ERR_INVALID_ARG
    assert lib.dora_compose_train(P, 2 * P, 3 * P, 1.0, _lib.DORA_BF16, T, d, 4 * P,
                                  4 * P + n // 2, None) == _lib.DORA_ERR_INVALID_ARG
    assert lib.dora_compose_train(P, 2 * P, 3 * P, 1.0, 5, T, d, 4 * P, 5 * P,
                                  None) == _lib.DORA_ERR_INVALID_ARG
    assert lib.dora_compose_train(P, 2 * P, 3 * P, 1.0, _lib.DORA_BF16, 0, d, 4 * P, 5 * P,
                                  None) == _lib.DORA_OK
    # backward: dmag without inner / wnorm, workspace too small or misaligned, outputs overlap
    ws = lib.dora_compose_backward_workspace_size(T, d)
    assert ws == T * d * 4
    assert lib.dora_compose_backward_workspace_size(4096, d) == 256 * d * 4
    assert lib.dora_compose_backward(P, None, 3 * P, 4 * P, 1e-6, 1.0, _lib.DORA_BF16, T, d,
                                     5 * P, 6 * P, 7 * P, 8 * P, ws,
                                     None) == _lib.DORA_ERR_INVALID_ARG
    assert lib.dora_compose_backward(P, 2 * P, 3 * P, 4 * P, 1e-6, 1.0, _lib.DORA_BF16, T, d,
                                     5 * P, 6 * P, 7 * P, 8 * P, ws - 4,
                                     None) == _lib.DORA_ERR_WORKSPACE
    assert lib.dora_compose_backward(P, 2 * P, 3 * P, 4 * P, 1e-6, 1.0, _lib.DORA_BF16, T, d,
                                     5 * P, 6 * P, 7 * P, 8 * P + 4, ws,
                                     None) == _lib.DORA_ERR_WORKSPACE
    assert lib.dora_compose_backward(P, 2 * P, 3 * P, 4 * P, 1e-6, 1.0, _lib.DORA_BF16, T, d,
                                     5 * P, 5 * P + 16, None, None, 0,
                                     None) == _lib.DORA_ERR_INVALID_ARG
    assert lib.dora_compose_backward(P, 2 * P, 3 * P, 4 * P, 0.0, 1.0, _lib.DORA_BF16, T, d,
                                     5 * P, 6 * P, 7 * P, 8 * P, ws,
                                     None) == _lib.DORA_ERR_INVALID_ARG


def _plan_table(d_out=256, d_in=512):
    t = (_lib.NormModule * 1)()
    t[0] = _lib.NormModule(P, 2 * P, 3 * P, 4 * P, 5 * P, 6 * P, d_out, d_in)
    return t


def test_grouped_plan_rejects_before_the_gpu(lib):
    h = ctypes.c_void_p(12345)
    # no output handle
    assert lib.dora_norm_grouped_plan_create(_plan_table(), 1, _lib.DORA_BF16, 64, 8 * P, 1 << 30,
                                             None, None) == _lib.DORA_ERR_INVALID_ARG
    # an invalid module: the handle is cleared
    st = lib.dora_norm_grouped_plan_create(_plan_table(d_out=-1), 1, _lib.DORA_BF16, 64, 8 * P,
                                           1 << 30, None, ctypes.byref(h))
    assert st == _lib.DORA_ERR_INVALID_ARG and not h.value
    # a workspace that is too small or misaligned
    for ws, nbytes in ((8 * P, 256), (8 * P + 16, 1 << 30), (None, 1 << 30)):
        h = ctypes.c_void_p(12345)
        st = lib.dora_norm_grouped_plan_create(_plan_table(), 1, _lib.DORA_BF16, 64, ws, nbytes,
                                               None, ctypes.byref(h))
        assert st == _lib.DORA_ERR_WORKSPACE and not h.value
    assert lib.dora_norm_grouped_plan_run(None, 1.0, 1e-6, None) == _lib.DORA_ERR_INVALID_ARG
    lib.dora_norm_grouped_plan_destroy(None)


def test_selftest_timeout_rejects_before_the_gpu(lib):
    assert lib.dora_selftest_timeout(None, 1 << 20, 1000, None) == _lib.DORA_ERR_WORKSPACE
    assert lib.dora_selftest_timeout(8 * P + 16, 1 << 20, 1000, None) == _lib.DORA_ERR_WORKSPACE
    assert lib.dora_selftest_timeout(8 * P, 128, 1000, None) == _lib.DORA_ERR_WORKSPACE
    assert lib.dora_selftest_timeout(8 * P, 1 << 20, 0, None) == _lib.DORA_ERR_INVALID_ARG
    assert lib.dora_selftest_timeout(8 * P, 1 << 20, 2_000_000, None) == _lib.DORA_ERR_INVALID_ARG


# ---------------------------------------------------------------- d_in-sharded norm
def _partials(lib, **kw):
    a = dict(W=P, A=2 * P, B=3 * P, dtype=_lib.DORA_BF16, d_out=256, d_in=512, r=64,
             partials=4 * P, ws=8 * P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.dora_norm_partials(a["W"], a["A"], a["B"], a["dtype"], a["d_out"], a["d_in"],
                                  a["r"], a["partials"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=5), _lib.DORA_ERR_INVALID_ARG),
    (dict(d_out=-1), _lib.DORA_ERR_INVALID_ARG),
    (dict(r=513), _lib.DORA_ERR_UNSUPPORTED),
    (dict(partials=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(partials=4 * P + 2), _lib.DORA_ERR_INVALID_ARG),   # not 4-byte aligned
    (dict(partials=P + 64), _lib.DORA_ERR_INVALID_ARG),      # inside W
    (dict(W=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(A=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(B=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(d_in=100), _lib.DORA_ERR_UNSUPPORTED),             # 200-byte rows
    (dict(r=60), _lib.DORA_ERR_UNSUPPORTED),
    (dict(A=2 * P + 8), _lib.DORA_ERR_UNSUPPORTED),          # misaligned
    (dict(ws=None), _lib.DORA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), _lib.DORA_ERR_WORKSPACE),
    (dict(d_out=0, r=0), _lib.DORA_OK),                      # no partials at all
])
def test_partials_argument_checks(lib, kw, status):
    assert _partials(lib, **kw) == status


def _finalize(lib, **kw):
    a = dict(partials=4 * P, B=3 * P, dtype=_lib.DORA_BF16, d_out=256, r=64, s=1.0, m=5 * P,
             eps=1e-6, wnorm=6 * P, g=7 * P, ws=8 * P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.dora_norm_finalize_partials(a["partials"], a["B"], a["dtype"], a["d_out"], a["r"],
                                           a["s"], a["m"], a["eps"], a["wnorm"], a["g"], a["ws"],
                                           a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=5), _lib.DORA_ERR_INVALID_ARG),
    (dict(r=513), _lib.DORA_ERR_UNSUPPORTED),
    (dict(eps=0.0), _lib.DORA_ERR_INVALID_ARG),
    (dict(s=float("nan")), _lib.DORA_ERR_INVALID_ARG),
    (dict(partials=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(B=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(m=None), _lib.DORA_ERR_INVALID_ARG),
    (dict(g=6 * P), _lib.DORA_ERR_INVALID_ARG),              # wnorm == g
    (dict(wnorm=4 * P + 512), _lib.DORA_ERR_INVALID_ARG),    # output inside the partials
    (dict(r=60), _lib.DORA_ERR_UNSUPPORTED),                 # 120-byte B rows
    (dict(ws=None), _lib.DORA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), _lib.DORA_ERR_WORKSPACE),
    (dict(d_out=0), _lib.DORA_OK),
])
def test_finalize_partials_argument_checks(lib, kw, status):
    assert _finalize(lib, **kw) == status


def test_partials_sizes(lib):
    assert lib.dora_norm_partials_floats(8192, 384) == 2 * 8192 + 384 * 384
    assert lib.dora_norm_partials_floats(-1, 8) == 0
    assert lib.dora_norm_partials_floats(8, 513) == 0
    n = lib.dora_norm_finalize_workspace_size(8192, 384, _lib.DORA_BF16)
    assert n == lib.dora_norm_workspace_size(8192, 64, 384, _lib.DORA_BF16)
    assert lib.dora_norm_finalize_workspace_size(8, 513, _lib.DORA_BF16) == 0
    assert lib.dora_version() & 0xFFFF >= 2      # the d_in-sharded norm
