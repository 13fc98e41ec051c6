"""Seeded synthetic restore workloads, shared by the tests, the oracle checks and
the benchmark.  Holds sizes, seeds and generators only -- no restore arithmetic."""
from . import configs, generate  # noqa: F401
from .configs import ModelShape, Workload, get, short_n  # noqa: F401
