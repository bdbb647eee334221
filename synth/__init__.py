"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests
and the benchmark.  Holds generators only: no attention arithmetic."""
from . import rng, formats, cases  # noqa: F401
from .cases import Case, make_case, config, CONFIG_NAMES  # noqa: F401
