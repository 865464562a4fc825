"""DoRA per-module hot path on GB300: factored row norm + stable fused compose.

The compute lives in ``libdora.so`` (CUDA kernels for sm_103a behind the C ABI
of include/dora.h); this package is its Python binding.  Importing the package
does not load the library; the first call does, and raises if it is missing.
"""
from ._lib import DoraError, LIB_PATH, load  # noqa: F401


def __getattr__(name):
    if name in ("dora_factored_norm", "dora_compose", "dora_check_status", "workspace_size",
                "alloc_workspace"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
