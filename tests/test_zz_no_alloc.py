"""orrery_bh_forces_noalloc, the entry point for callers that cannot allocate
device memory during a call (their allocator or graph capture forbids it):
its results must equal the ordinary entry point's, call after call, although
its scratch is one fixed array shared by every call.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
REL_TOL = 1e-5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_traversal_gb300.build import build

    build()
    import tree_traversal_gb300._lib as L

    return L.load()


def _call(fn, pos, mass, theta, eps, cap, traversal):
    n = pos.shape[0]
    acc = torch.full((n, 3), float("nan"), device="cuda")
    inter = torch.full((n, 2), -1, dtype=torch.int32, device="cuda")
    vis = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = fn(p(pos), p(mass), n, theta, eps, cap, traversal, p(acc), p(inter), p(vis),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, acc, inter, vis


def test_noalloc_matches_the_allocating_entry_point(lib):
    import tree_traversal_gb300._lib as L
    from inputs import plummer, uniform_cube

    # two calls in a row on different inputs: a larger one, then a smaller
    # one that lands on scratch the first call left behind
    cases = [(plummer(65536, 3), 0.5, 0.05, 32, L.COHERENT),
             (uniform_cube(5003, 4), 0.7, 0.05, 7, L.INDEPENDENT),
             (plummer(40000, 5), 0.5, 0.05, 16, L.COHERENT)]
    for (pos_np, mass_np), theta, eps, cap, trav in cases:
        pos = torch.from_numpy(pos_np).cuda()
        mass = torch.from_numpy(mass_np).cuda()
        rc0, acc0, inter0, vis0 = _call(lib.orrery_bh_forces, pos, mass, theta, eps, cap, trav)
        assert rc0 == L.OK
        for _ in range(2):
            rc, acc, inter, vis = _call(lib.orrery_bh_forces_noalloc, pos, mass, theta, eps, cap,
                                        trav)
            assert rc == L.OK
            assert torch.equal(acc.view(torch.int32), acc0.view(torch.int32))
            assert torch.equal(inter, inter0) and torch.equal(vis, vis0)


def test_noalloc_every_traversal(lib):
    import tree_traversal_gb300._lib as L
    from inputs import plummer

    pos_np, mass_np = plummer(9001, 17)
    pos = torch.from_numpy(pos_np).cuda()
    mass = torch.from_numpy(mass_np).cuda()
    for trav in (L.INDEPENDENT, L.COHERENT, L.COHERENT_16, L.COHERENT_64, L.DESCEND_TOGETHER,
                 L.COHERENT_BALLOT):
        r0 = _call(lib.orrery_bh_forces, pos, mass, 0.5, 0.05, 32, trav)
        r1 = _call(lib.orrery_bh_forces_noalloc, pos, mass, 0.5, 0.05, 32, trav)
        assert r0[0] == r1[0] == L.OK
        for a, b in zip(r0[1:], r1[1:]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_noalloc_documented_sizes_fit(lib):
    """The header's promise: every n up to 65 536 fits at leaf_cap 16 and up to
    80 000 at leaf_cap 32 (the layout's limits are 79 030 and 99 197). At both
    limits the results are checked against the oracle itself: counts bit for
    bit, accelerations within 1e-5 relative error."""
    import oracle
    import tree_traversal_gb300._lib as L
    from inputs import plummer

    for n, cap in ((65536, 16), (80000, 32)):
        pos, mass = plummer(n, 41)
        p, m = torch.from_numpy(pos).cuda(), torch.from_numpy(mass).cuda()
        rc, acc, inter, vis = _call(lib.orrery_bh_forces_noalloc, p, m, 0.5, 0.05, cap, L.COHERENT)
        assert rc == L.OK, (n, cap, rc)
        r_acc, r_inter, r_vi, r_vc, _ = oracle.bh_forces(pos, mass, 0.5, 0.05, cap, True,
                                                         oracle.default_threads())
        assert np.array_equal(inter.cpu().numpy().view(np.uint32), r_inter)
        assert np.array_equal(vis.cpu().numpy().view(np.uint32), r_vc)
        rel = oracle.relative_error(acc.cpu().numpy(), r_acc).max()
        assert rel <= REL_TOL, (n, cap, rel)


_FRESH = r"""
import ctypes, sys
import torch
sys.path.insert(0, sys.argv[1])
import tree_traversal_gb300._lib as L
from inputs import plummer
lib = L.load()
sizes = [(65536, 32), (3000, 8), (40000, 16), (70000, 32)]
data = []
for n, cap in sizes:
    pos, mass = plummer(n, n)
    data.append((torch.from_numpy(pos).cuda(), torch.from_numpy(mass).cuda(),
                 torch.empty((n, 3), device="cuda"), torch.empty((n, 2), dtype=torch.int32, device="cuda"),
                 torch.empty((n,), dtype=torch.int32, device="cuda"), cap))
st = torch.cuda.Stream()
p = lambda t: ctypes.c_void_p(t.data_ptr())
def run(d, trav):
    pos, mass, acc, inter, vis, cap = d
    rc = lib.orrery_bh_forces_noalloc(p(pos), p(mass), pos.shape[0], 0.5, 0.05, cap, trav, p(acc),
                                      p(inter), p(vis), ctypes.c_void_p(st.cuda_stream))
    assert rc == L.OK, rc
travs = (L.COHERENT_64, L.COHERENT, L.INDEPENDENT)
for d in data:          # first calls: module load, kernel attributes
    for t in travs:
        run(d, t)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(3):
    for d in data:
        for t in travs:
            run(d, t)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
print("free", free0, free1)
assert free1 == free0, (free0, free1)
"""


def test_noalloc_allocates_nothing_in_a_fresh_process(lib, tmp_path):
    """A process that only ever calls the no-allocation entry point: after one
    round of calls (which may load the library's device code), further calls
    of several sizes and traversals leave the device's free memory exactly
    unchanged."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "fresh.py"
    script.write_text(_FRESH)
    r = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


def test_noalloc_rejects_what_does_not_fit(lib):
    import tree_traversal_gb300._lib as L

    dummy = ctypes.c_void_p(16)  # never dereferenced: the size check fails first
    assert lib.orrery_bh_forces_noalloc(dummy, dummy, 200000, 0.5, 0.05, 32, 1, dummy, None, None,
                                        None) == L.ESCRATCH
    assert lib.orrery_bh_forces_noalloc(dummy, dummy, 65536, 0.5, 0.05, 1, 1, dummy, None, None,
                                        None) == L.ESCRATCH
    assert lib.orrery_bh_forces_noalloc(dummy, dummy, 10, -1.0, 0.05, 32, 1, dummy, None, None,
                                        None) == L.EINVAL
    assert lib.orrery_bh_forces_noalloc(None, None, 0, 0.5, 0.05, 32, 1, None, None, None,
                                        None) == L.OK
