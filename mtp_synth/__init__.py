"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

Holds shapes and random draws only; none of the drafter arithmetic lives here.
"""
from .configs import CONFIGS, Config, DrafterShape, Workload, config  # noqa: F401
from . import gen  # noqa: F401
