"""Seeded synthetic workloads (shapes + random inputs) for the decode-step hot path.

Holds no part of the method's arithmetic; shared by the CUDA path's tests and
benchmark and by the fp64 oracle's checks.
"""
from . import configs, generate  # noqa: F401
