"""bench.py's host-side bookkeeping, on the CPU: the walk's DRAM traffic is
taken from the committed ncu summary only while the profiled kernel code (the
source without its comments) is the current one."""
from __future__ import annotations

import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WALK_SRC = os.path.join(ROOT, "tree_traversal_gb300", "csrc", "bh_walk.cu")


def test_committed_traffic_matches_the_current_walk_source():
    # the summaries the bench lines read were captured on this source: the
    # default width-64 walk and the two walks the pages compare
    for kernel in ("k_walk_paired", "k_walk_coherent", "k_walk_independent"):
        traffic = bench.profile_traffic(WALK_SRC, kernel, True)
        assert traffic is not None and 40e6 < traffic < 120e6, kernel


def test_traffic_is_withheld_for_changed_code(tmp_path):
    # a comment changes nothing the kernel does: the summary still applies
    commented = tmp_path / "commented.cu"
    shutil.copy(WALK_SRC, commented)
    with open(commented, "a") as f:
        f.write("\n// a comment\n\n")
    assert bench.profile_traffic(str(commented), "k_walk_paired", True) is not None
    # a change to the code withholds it
    changed = tmp_path / "bh_walk.cu"
    shutil.copy(WALK_SRC, changed)
    with open(changed, "a") as f:
        f.write("\nstatic int changed_code = 1;\n")
    assert bench.profile_traffic(str(changed), "k_walk_paired", True) is None
    # and for a walk kernel with no summary of its own
    assert bench.profile_traffic(WALK_SRC, "k_walk_together", True) is None
