"""Plummer-sphere particle sets from a SplitMix64 stream.

The pages measure on "a Plummer sphere, seed 20260811" (orrery:
docs/performance/sycl_tree.md, "The machine and the device" table) without
naming the generator. The reading taken here:

* Random stream: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014): the state advances by the
  golden-ratio increment and each output is the state passed through the
  published 64-bit finaliser. A uniform double in [0, 1) is the top 53 bits of
  an output times 2^-53.
* Per particle, three draws in order u1, u2, u3:
  X = 0.001 + 0.998 u1 (the mass fraction, kept away from 0 and 1),
  r = 1 / sqrt(X^(-2/3) - 1) (the inverse of the Plummer cumulative mass with
  scale radius 1), cos(polar) = 2 u2 - 1, azimuth = 2 pi u3.
  Positions are computed in float64 and rounded once to float32.
* Masses are equal: fl32(1 / N) for a single sphere of N particles.

Because float64 pow/sin/cos may differ by an ulp between hosts, generated
sets are compared only within one process; stored expected values never come
from these generators.
"""
from __future__ import annotations

import numpy as np

PAGES_SEED = 20260811

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MUL1 = np.uint64(0xBF58476D1CE4E5B9)
_MUL2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+count-1 of the SplitMix64 stream seeded with seed."""
    with np.errstate(over="ignore"):
        k = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MUL1
        z = (z ^ (z >> np.uint64(27))) * _MUL2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of each output."""
    z = splitmix64(seed, count, offset)
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def plummer(n: int, seed: int = PAGES_SEED, center=(0.0, 0.0, 0.0), mass: float | None = None,
            chunk: int = 1 << 20):
    """n particles of a Plummer sphere (scale radius 1). Returns (pos [n,3] f32, mass [n] f32)."""
    pos = np.empty((n, 3), np.float32)
    c = np.asarray(center, np.float64)
    for start in range(0, n, chunk):
        m = min(chunk, n - start)
        u = uniform01(seed, 3 * m, 3 * start).reshape(m, 3)
        X = 0.001 + 0.998 * u[:, 0]
        r = 1.0 / np.sqrt(X ** (-2.0 / 3.0) - 1.0)
        cos_t = 2.0 * u[:, 1] - 1.0
        sin_t = np.sqrt(np.maximum(0.0, 1.0 - cos_t * cos_t))
        phi = 2.0 * np.pi * u[:, 2]
        p = np.empty((m, 3), np.float64)
        p[:, 0] = r * sin_t * np.cos(phi) + c[0]
        p[:, 1] = r * sin_t * np.sin(phi) + c[1]
        p[:, 2] = r * cos_t + c[2]
        pos[start:start + m] = p.astype(np.float32)
    mval = np.float32(1.0 / n) if mass is None else np.float32(mass)
    return pos, np.full(n, mval, np.float32)


def two_spheres(n_each: int = 1048576, seeds=(1, 2), offset=(6.0, 0.0, 0.0)):
    """Sphere A (seeds[0], centre 0) followed by sphere B (seeds[1], centre offset).

    Every particle has mass 1/n_each, so each sphere has mass 1."""
    m = 1.0 / n_each
    pa, ma = plummer(n_each, seeds[0], (0.0, 0.0, 0.0), m)
    pb, mb = plummer(n_each, seeds[1], offset, m)
    return np.concatenate([pa, pb]), np.concatenate([ma, mb])


def uniform_cube(n: int, seed: int, lo: float = -1.0, hi: float = 1.0):
    """n particles uniform in a cube, equal masses 1/n (edge-case inputs)."""
    u = uniform01(seed, 3 * n).reshape(n, 3)
    pos = (lo + (hi - lo) * u).astype(np.float32)
    return pos, np.full(n, np.float32(1.0 / max(n, 1)), np.float32)


# The workloads of the benchmark and the parity tests, by name.
WORKLOADS = {
    "plummer_4096": dict(kind="plummer", n=4096, seed=PAGES_SEED, theta=0.5),
    "plummer_16384": dict(kind="plummer", n=16384, seed=PAGES_SEED, theta=0.5),
    "plummer_131072": dict(kind="plummer", n=131072, seed=PAGES_SEED, theta=0.5),
    "plummer_262144": dict(kind="plummer", n=262144, seed=PAGES_SEED, theta=0.5),
    "plummer_524288": dict(kind="plummer", n=524288, seed=PAGES_SEED, theta=0.5),
    "plummer_1048576": dict(kind="plummer", n=1048576, seed=PAGES_SEED, theta=0.5),
    "two_spheres_2x1048576": dict(kind="two_spheres", n=2 * 1048576, seed=(1, 2), theta=0.5),
}


def workload(name: str):
    """Returns (pos, mass, params) for a named workload (eps 0.05, leaf capacity 32)."""
    w = dict(WORKLOADS[name])
    if w["kind"] == "plummer":
        pos, mass = plummer(w["n"], w["seed"])
    else:
        pos, mass = two_spheres(w["n"] // 2, w["seed"])
    params = dict(theta=w["theta"], eps=0.05, leaf_cap=32)
    return pos, mass, params
