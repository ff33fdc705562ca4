"""The C-ABI library: it builds, loads, exports every declared symbol, and its
host-side argument checks answer before any CUDA call (no GPU needed)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from tree_traversal_gb300.build import build

    build()
    import tree_traversal_gb300._lib as L

    return L.load()


def declared_functions() -> list[str]:
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(orrery_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("orrery_bh_forces", "orrery_bh_forces_host", "orrery_bh_tree",
                 "orrery_direct_forces",
                 "orrery_bh_max_nodes", "orrery_bh_last_timings", "orrery_bh_kernel_launches",
                 "orrery_bh_strerror", "orrery_bh_release", "orrery_fp32_fma_rate"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from tree_traversal_gb300.build import LIB_PATH

    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_targets_sm103a_only():
    from tree_traversal_gb300.build import ARCH

    assert ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_argument_checks_answer_on_the_host(lib):
    import tree_traversal_gb300._lib as L

    P = None
    dummy = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    f = lib.orrery_bh_forces
    assert f(dummy, dummy, -1, 0.5, 0.05, 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, (1 << 30) + 1, 0.5, 0.05, 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, float("nan"), 0.05, 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, -0.1, 0.05, 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, float("nan"), 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, -1.0, 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 0, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 32, 7, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 32, 6, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 32, 0x201, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 32, 0x106, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 32, -1, dummy, P, P, P) == L.EINVAL
    assert f(P, dummy, 10, 0.5, 0.05, 32, 1, dummy, P, P, P) == L.EINVAL
    assert f(dummy, dummy, 10, 0.5, 0.05, 32, 1, P, P, P, P) == L.EINVAL
    # node bound beyond int32: 2^30 particles with leaf capacity 1
    assert f(dummy, dummy, 1 << 30, 0.5, 0.05, 1, 1, dummy, P, P, P) == L.ERANGE
    d = lib.orrery_direct_forces
    assert d(dummy, dummy, -1, 0.05, dummy, P) == L.EINVAL
    assert d(dummy, dummy, 10, float("nan"), dummy, P) == L.EINVAL
    assert d(P, dummy, 10, 0.05, dummy, P) == L.EINVAL
    assert d(P, P, 0, 0.05, P, P) == L.OK
    # the FMA-rate probe checks its outputs before touching the GPU
    x = ctypes.c_double(0.0)
    assert lib.orrery_fp32_fma_rate(None, ctypes.byref(x), None, None) == L.EINVAL
    assert lib.orrery_fp32_fma_rate(ctypes.byref(x), None, None, None) == L.EINVAL
    # n == 0 launches nothing and succeeds, whatever the pointers
    assert f(P, P, 0, 0.5, 0.05, 32, 0, P, P, P, P) == L.OK
    assert lib.orrery_bh_forces_host(P, P, 0, 0.5, 0.05, 32, 1, P, P, P, P) == L.OK
    nn = ctypes.c_int64(5)
    assert lib.orrery_bh_tree(P, P, 0, 32, P, P, P, P, P, 0, ctypes.byref(nn), P) == L.OK
    assert nn.value == 0
    assert lib.orrery_bh_tree(dummy, dummy, 10, 32, P, P, P, P, P, 0, None, P) == L.EINVAL
    # the target-slice entry: the same checks, plus 0 <= begin <= end <= n
    r = lib.orrery_bh_forces_range
    assert r(dummy, dummy, 10, 0.5, 0.05, 32, 3, -1, 5, dummy, P, P, P) == L.EINVAL
    assert r(dummy, dummy, 10, 0.5, 0.05, 32, 3, 6, 5, dummy, P, P, P) == L.EINVAL
    assert r(dummy, dummy, 10, 0.5, 0.05, 32, 3, 0, 11, dummy, P, P, P) == L.EINVAL
    assert r(dummy, dummy, 10, -0.5, 0.05, 32, 3, 0, 10, dummy, P, P, P) == L.EINVAL
    assert r(dummy, dummy, 10, 0.5, 0.05, 32, 9, 0, 10, dummy, P, P, P) == L.EINVAL
    assert r(P, dummy, 10, 0.5, 0.05, 32, 3, 0, 10, dummy, P, P, P) == L.EINVAL
    assert r(dummy, dummy, 10, 0.5, 0.05, 32, 3, 0, 10, P, P, P, P) == L.EINVAL
    assert r(dummy, dummy, 1 << 30, 0.5, 0.05, 1, 3, 0, 64, dummy, P, P, P) == L.ERANGE
    assert r(P, P, 0, 0.5, 0.05, 32, 3, 0, 0, P, P, P, P) == L.OK


def test_shard_tiles_the_targets():
    import tree_traversal_gb300 as tt

    for n in (0, 1, 63, 64, 65, 1000, 1048576, 1048577):
        for world in (1, 2, 3, 4, 7, 8):
            for align in (1, 32, 64):
                cuts = [tt.shard(n, r, world, align) for r in range(world)]
                assert cuts[0][0] == 0 and cuts[-1][1] == n
                for (b0, e0), (b1, e1) in zip(cuts, cuts[1:]):
                    assert e0 == b1
                for b, e in cuts:
                    assert 0 <= b <= e <= n
                    assert b % align == 0 and (e % align == 0 or e == n)
                sizes = [e - b for b, e in cuts]
                assert max(sizes) - min(sizes) <= align
    with pytest.raises(ValueError):
        tt.shard(10, 2, 2)


def test_node_bound(lib):
    import oracle
    from inputs import plummer, uniform_cube

    assert lib.orrery_bh_max_nodes(-1, 32) == -1 and lib.orrery_bh_max_nodes(10, 0) == -1
    assert lib.orrery_bh_max_nodes(0, 32) == 1
    # the bound holds on real trees, including leaf capacity 1 and duplicates
    dup = np.zeros((200, 3), np.float32)
    for pos, cap in ((plummer(5000, 3)[0], 32), (uniform_cube(3000, 4)[0], 1),
                     (plummer(4000, 5)[0], 2), (dup, 32)):
        T = oracle.Tree(pos, np.ones(len(pos), np.float32), cap)
        assert T.num_nodes <= lib.orrery_bh_max_nodes(len(pos), cap)


def test_strerror_and_counters(lib):
    import tree_traversal_gb300._lib as L

    for s in (L.OK, L.EINVAL, L.ENONFINITE, L.ERANGE, L.ECUDA, L.EWALK, L.ENOMEM, L.EINTERNAL,
              L.ESCRATCH):
        assert lib.orrery_bh_strerror(s).decode() not in ("", "unknown status")
    assert lib.orrery_bh_strerror(-99).decode() == "unknown status"
    t = L.Timings()
    if lib.orrery_bh_kernel_launches() == 0:
        assert lib.orrery_bh_last_timings(ctypes.byref(t)) == L.EINVAL
    assert lib.orrery_bh_last_timings(None) == L.EINVAL


def test_timings_struct_layout():
    import tree_traversal_gb300._lib as L

    # 11 floats, 2 int32, 2 int64, 1 uint64
    assert ctypes.sizeof(L.Timings) == 11 * 4 + 2 * 4 + 4 + 3 * 8
