"""Seeded synthetic inputs shared by the oracle tests and the CUDA path.

Holds shapes, seeds and random draws only; no drafting arithmetic."""
from .configs import WORKLOADS, DrafterConfig, Workload  # noqa: F401
from . import gen  # noqa: F401
