"""GB300-native Barnes-Hut monopole force evaluation.

A stackless depth-first octree with escape indices, walked either by one
thread per target or by whole warps that advance to the smallest node index
any lane still wants (the answer-preserving coherent walk). The work runs in
hand-written sm_103a CUDA kernels behind the C ABI of include/orrery_bh.h;
this package is the thin Python binding over that library.

    from tree_traversal_gb300 import bh_forces
    acc, interactions, visits = bh_forces(pos, mass, theta=0.5, eps=0.05,
                                          leaf_cap=32, traversal="coherent64")
"""
from .bh import (  # noqa: F401
    bh_forces,
    bh_forces_host,
    bh_tree,
    direct_forces,
    fp32_fma_rate,
    kernel_launches,
    last_timings,
    max_nodes,
    release,
    shard,
)
from ._lib import OrreryError, load  # noqa: F401
