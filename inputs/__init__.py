"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This package holds input generation only (random numbers and the Plummer
sampling recipe). It contains none of the force evaluation's arithmetic, and
it imports neither the oracle nor the CUDA library.
"""
from .plummer import (  # noqa: F401
    PAGES_SEED,
    plummer,
    splitmix64,
    two_spheres,
    uniform01,
    uniform_cube,
    workload,
)
