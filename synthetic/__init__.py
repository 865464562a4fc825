"""Seeded synthetic workloads shared by the oracle-side and GPU-side tests and
the bench.  Holds shapes and random draws only, none of the DoRA arithmetic."""
from . import configs, gen  # noqa: F401
