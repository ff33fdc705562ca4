"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every pin is a plain function (``pin_*``) so that ``test_planted_mistakes``
can run it against a copy of the oracle with one plausible mistake planted
and check that it fails. Sources of the expected values:

* hand derivations (tests/golden/morton_three_points.txt),
* library routines for special cases (numpy min/max, numpy stable argsort,
  numpy fp64 direct sums, math.fsum),
* an independent set-based formulation of the octree (cells of every level,
  a cell is a node iff its parent holds more than leaf_cap particles) and of
  the walk (a node is visited iff no strict ancestor was accepted),
* closed forms (two bodies, a far clump seen as one point mass, theta = 0
  equals direct summation, total momentum of a pairwise-antisymmetric sum),
* brute-force set unions for the coherent walk (ADR-0029, Decision),
* the orrery performance page's tables, as soft pins (their generator differs).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle
from inputs import plummer, splitmix64, two_spheres, uniform_cube

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS = 0.05


def read_golden(name: str) -> dict:
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                sections[cur] = []
            else:
                sections[cur].append(line.split())
    return sections


# ---------------------------------------------------------------------------
# independent formulations used by several pins
# ---------------------------------------------------------------------------
def brute_force_nodes(sorted_keys: np.ndarray, leaf_cap: int) -> np.ndarray:
    """All cells of every level by key prefix; a cell is a node iff it is the
    root or its parent cell holds more than leaf_cap particles. Depth-first
    preorder = sort by (first, level); escape = number of nodes whose first
    particle lies before the end of this node's range."""
    n = len(sorted_keys)
    if n == 0:
        return np.zeros((0, 4), np.int32)
    cells = {}
    for level in range(22):
        pre = sorted_keys >> np.uint64(3 * (21 - level))
        start = 0
        for j in range(1, n + 1):
            if j == n or pre[j] != pre[start]:
                cells[(level, int(pre[start]))] = (start, j - start)
                start = j
    nodes = []
    for (level, p), (first, count) in cells.items():
        if level == 0 or cells[(level - 1, p >> 3)][1] > leaf_cap:
            nodes.append((first, level, count))
    nodes.sort()
    firsts = np.array([a[0] for a in nodes])
    out = np.zeros((len(nodes), 4), np.int32)
    for k, (first, level, count) in enumerate(nodes):
        out[k] = (np.searchsorted(firsts, first + count, side="left"), first, count, level)
    return out


def parents_from_escape(nodes: np.ndarray) -> np.ndarray:
    par = np.full(len(nodes), -1, np.int64)
    stack = []
    for k in range(len(nodes)):
        while stack and nodes[stack[-1], 0] <= k:
            stack.pop()
        par[k] = stack[-1] if stack else -1
        stack.append(k)
    return par


def direct_numpy(pos, mass, eps):
    p = pos.astype(np.float64)
    d = p[None, :, :] - p[:, None, :]
    r2 = (d * d).sum(-1) + eps * eps
    f = mass.astype(np.float64)[None, :] / (r2 * np.sqrt(r2))
    np.fill_diagonal(f, 0.0)
    return (f[:, :, None] * d).sum(1)


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------
def test_splitmix64_reference_outputs():
    # First outputs of SplitMix64 seeded with 1234567, as published with the
    # generator's reference implementation and reproduced by its ports.
    g = read_golden("splitmix64_seed1234567.txt")
    want = [int(v[0]) for v in g["outputs"]]
    assert [int(v) for v in splitmix64(1234567, len(want))] == want


def test_plummer_recipe_properties():
    pos, m = plummer(20000, 7)
    r = np.linalg.norm(pos.astype(np.float64), axis=1)
    # X in [0.001, 0.999] maps to r in [1/sqrt(0.001^(-2/3)-1), 1/sqrt(0.999^(-2/3)-1)]
    assert r.min() >= 1.0 / math.sqrt(0.001 ** (-2 / 3) - 1) * (1 - 1e-6)
    assert r.max() <= 1.0 / math.sqrt(0.999 ** (-2 / 3) - 1) * (1 + 1e-6)
    # Plummer cumulative mass M(<r) = r^3 / (1 + r^2)^(3/2): the median radius
    # solves M = 0.5, i.e. r = 1/sqrt(0.5^(-2/3) - 1) ~ 1.305
    assert abs(np.median(r) - 1.0 / math.sqrt(0.5 ** (-2 / 3) - 1)) < 0.03
    assert m.dtype == np.float32 and np.all(m == np.float32(1 / 20000))


def ks_uniform(u, lo, hi):
    """Kolmogorov-Smirnov distance of a sample from the uniform law on [lo, hi]."""
    u = np.sort((np.asarray(u, np.float64) - lo) / (hi - lo))
    k = np.arange(1, len(u) + 1) / len(u)
    return max(np.max(k - u), np.max(u - (k - 1.0 / len(u))))


def test_plummer_recipe_distributions():
    # the mass fraction inside each particle's radius, X = r^3 / (1 + r^2)^1.5
    # (the Plummer cumulative mass), is uniform on [0.001, 0.999]; the
    # direction is isotropic: cos(polar) uniform on [-1, 1], azimuth uniform
    n = 40000
    pos, _ = plummer(n, 99)
    x = pos.astype(np.float64)
    r = np.linalg.norm(x, axis=1)
    X = r ** 3 / (1.0 + r * r) ** 1.5
    bound = 2.0 / math.sqrt(n)  # far above the 95 % KS quantile 1.36 / sqrt(n)
    assert ks_uniform(X, 0.001, 0.999) < bound
    assert ks_uniform(x[:, 2] / r, -1.0, 1.0) < bound
    assert ks_uniform(np.arctan2(x[:, 1], x[:, 0]) % (2 * math.pi), 0.0, 2 * math.pi) < bound
    # a generator that drew cos(polar) = u instead of 2u - 1 would fail
    assert ks_uniform(np.abs(x[:, 2] / r), -1.0, 1.0) > 10 * bound


# ---------------------------------------------------------------------------
# steps 1-3: cube, keys, sort
# ---------------------------------------------------------------------------
def pin_golden_three_points():
    g = read_golden("morton_three_points.txt")
    pts = np.array(g["points"], np.float32)
    lo, side, inv = oracle.cube(pts)
    c = [float(v) for v in g["cube"][0]]
    assert list(lo) == c[:3] and float(side) == c[3] and float(inv) == c[4]
    for p, q in zip(pts, g["quantised"]):
        assert [oracle.quantise(p[a], lo[a], inv) for a in range(3)] == [int(v) for v in q]
    k = oracle.keys(pts, lo, inv)
    assert [int(v) for v in k] == [int(v[0], 16) for v in g["keys"]]
    perm, sk = oracle.sort(k)
    assert list(perm) == [int(v) for v in g["perm"][0]]
    nodes = oracle.build_tree(sk, 1)
    assert nodes.tolist() == [[int(v) for v in row] for row in g["nodes leaf_cap=1"]]


def test_golden_three_points():
    pin_golden_three_points()


def pin_interleave_single_bits():
    rng = np.random.default_rng(1)
    for b in range(21):
        assert oracle.interleave(1 << b, 0, 0) == 1 << (3 * b + 2)
        assert oracle.interleave(0, 1 << b, 0) == 1 << (3 * b + 1)
        assert oracle.interleave(0, 0, 1 << b) == 1 << (3 * b)
    for _ in range(200):
        qx, qy, qz = (int(v) for v in rng.integers(0, 1 << 21, 3))
        k = oracle.interleave(qx, qy, qz)
        assert k == (oracle.interleave(qx, 0, 0) | oracle.interleave(0, qy, 0)
                     | oracle.interleave(0, 0, qz))
        assert k < (1 << 63)


def test_interleave_single_bits():
    pin_interleave_single_bits()


def pin_quantise():
    inv = np.float32(2 ** 21)  # side 1
    assert oracle.quantise(0.0, 0.0, inv) == 0
    assert oracle.quantise(1.0, 0.0, inv) == 2 ** 21 - 1  # clamped
    for j in (1, 3, 12345, 2 ** 20, 2 ** 21 - 1):
        x = j / 2 ** 21  # exact binary fractions: the product is exact
        assert oracle.quantise(x, 0.0, inv) == j
        assert oracle.quantise(np.nextafter(np.float32(x), np.float32(0)), 0.0, inv) == j - 1


def test_quantise_floor_and_clamp():
    pin_quantise()


def pin_cube():
    for n, seed in ((1, 1), (2, 2), (1000, 3)):
        pos, _ = uniform_cube(n, seed, -3.0, 5.0)
        lo, side, inv = oracle.cube(pos)
        assert np.array_equal(lo, pos.min(0))
        assert side == np.float32((pos.max(0) - pos.min(0)).max())
        if side > 0:
            assert inv == np.float32(2 ** 21) / side
    # the largest extent on each axis in turn: the side is the largest of the three
    for axis in range(3):
        pos, _ = uniform_cube(200, 10 + axis, -1.0, 1.0)
        pos[:, axis] *= 4.0
        lo, side, inv = oracle.cube(pos)
        assert side == np.float32((pos.max(0) - pos.min(0)).max())
    lo, side, inv = oracle.cube(np.ones((5, 3), np.float32))
    assert side == 0 and inv == 0
    assert np.all(oracle.keys(np.ones((5, 3), np.float32)) == 0)


def test_cube_is_numpy_min_max():
    pin_cube()


def pin_sort_stable():
    # many equal keys: the order among them is the original index order
    rng = np.random.default_rng(5)
    keys = rng.integers(0, 50, 5000).astype(np.uint64) << np.uint64(40)
    perm, sk = oracle.sort(keys)
    ref = np.argsort(keys, kind="stable")
    assert np.array_equal(perm, ref.astype(np.uint32))
    assert np.array_equal(sk, keys[ref])


def test_sort_is_stable_argsort():
    pin_sort_stable()


# ---------------------------------------------------------------------------
# step 4: tree
# ---------------------------------------------------------------------------
def _tree_inputs():
    dup = np.zeros((75, 3), np.float32)
    dup[65:] = uniform_cube(10, 9)[0]  # 65 identical points + 10 others
    clump, _ = uniform_cube(300, 4, 0.0, 1e-4)
    clump = np.concatenate([clump, uniform_cube(60, 5)[0]])
    return {
        "plummer300_cap4": (plummer(300, 11)[0], 4),
        "uniform500_cap1": (uniform_cube(500, 12)[0], 1),
        "uniform777_cap32": (uniform_cube(777, 13)[0], 32),
        "duplicates_cap32": (dup, 32),
        "clump_cap8": (clump, 8),
    }


def pin_tree_brute_force():
    for name, (pos, cap) in _tree_inputs().items():
        _, sk = oracle.sort(oracle.keys(pos))
        got = oracle.build_tree(sk, cap)
        want = brute_force_nodes(sk, cap)
        assert np.array_equal(got, want), name


def test_tree_brute_force():
    pin_tree_brute_force()


@pytest.mark.parametrize("n", [4096, 16384])
def test_tree_invariants(n):
    pos, m = plummer(n)
    T = oracle.Tree(pos, m, 32)
    nodes, cap = T.nodes, 32
    leaf = oracle.is_leaf(nodes, cap)
    assert nodes[0].tolist() == [T.num_nodes, 0, n, 0]
    # leaves partition the particles in order; leaves respect the capacity
    lf = nodes[leaf]
    assert lf[0, 1] == 0 and np.all(lf[1:, 1] == lf[:-1, 1] + lf[:-1, 2]) and lf[-1, 1] + lf[-1, 2] == n
    assert np.all((lf[:, 2] <= cap) | (lf[:, 3] == 21))
    # internal: over capacity, children partition the range in octant order
    par = parents_from_escape(nodes)
    for k in np.nonzero(~leaf)[0][:500]:
        assert nodes[k, 2] > cap
        kids = np.nonzero(par == k)[0]
        assert kids[0] == k + 1
        assert nodes[kids[0], 1] == nodes[k, 1]
        assert np.all(nodes[kids[1:], 1] == nodes[kids[:-1], 1] + nodes[kids[:-1], 2])
        assert nodes[kids].sum(0)[2] == nodes[k, 2]
        assert np.all(nodes[kids, 3] == nodes[k, 3] + 1)
        assert nodes[kids[-1], 0] == nodes[k, 0]
    # escape > k, and the last escape is the node count
    assert np.all(nodes[:, 0] > np.arange(T.num_nodes)) and nodes[:, 0].max() == T.num_nodes


def test_duplicates_make_a_depth21_leaf():
    pos = np.full((65, 3), 0.25, np.float32)
    pos = np.concatenate([pos, [[0.0, 0.0, 0.0], [1.0, 1.0, 1.0]]]).astype(np.float32)
    T = oracle.Tree(pos, np.full(67, 1 / 67, np.float32), 32)
    deep = T.nodes[T.nodes[:, 3] == 21]
    assert deep.tolist() == [[deep[0, 0], 1, 65, 21]]


def test_tree_soft_pins_against_pages():
    # orrery performance page, "Where one evaluation goes": 568 nodes / depth 8
    # at 4096 and 2171 / depth 9 at 16384 (their generator differs: +-25 %).
    for n, nodes_pages, depth_pages in ((4096, 568, 8), (16384, 2171, 9)):
        pos, m = plummer(n)
        T = oracle.Tree(pos, m, 32)
        assert abs(T.num_nodes / nodes_pages - 1) < 0.25
        assert abs(T.depth - depth_pages) <= 1


# ---------------------------------------------------------------------------
# step 5: moments
# ---------------------------------------------------------------------------
def pin_moments():
    # a symmetric pair with a power-of-two mass: the centre of mass is the
    # midpoint exactly and M = 2m
    pos = np.array([[-0.75, 0.5, 0.125], [0.75, 0.5, 0.125]], np.float32)
    m = np.full(2, 2.0 ** -4, np.float32)
    T = oracle.Tree(pos, m, 32)
    assert T.cm.tolist() == [[0.0, 0.5, 0.125, 0.125]]
    # a single leaf: M is the sequential fp32 sum of its masses
    rng = np.random.default_rng(3)
    pos = rng.random((20, 3)).astype(np.float32)
    m = rng.random(20).astype(np.float32)
    T = oracle.Tree(pos, m, 32)
    s = np.float32(0)
    for v in m[T.perm]:
        s = np.float32(s + v)
    assert T.cm[0, 3] == s
    # every node: M within rounding of fsum over its range, CoM within 1e-5
    # of the fp64 centre of mass of its range
    pos, m = plummer(3000, 21)
    m = (m * np.random.default_rng(2).uniform(0.5, 1.5, 3000)).astype(np.float32)
    T = oracle.Tree(pos, m, 8)
    for k in range(T.num_nodes):
        esc, first, count, level = T.nodes[k]
        ms = T.ps[first:first + count, 3].astype(np.float64)
        xs = T.ps[first:first + count, :3].astype(np.float64)
        M = math.fsum(ms)
        assert abs(T.cm[k, 3] - M) <= 1e-6 * M
        com = (ms[:, None] * xs).sum(0) / M
        scale = np.abs(xs).max() + 1e-30
        assert np.all(np.abs(T.cm[k, :3] - com) <= 2e-5 * scale), k


def test_moments():
    pin_moments()


# ---------------------------------------------------------------------------
# steps 6-8: walk, criterion and force term
# ---------------------------------------------------------------------------
def pin_two_body():
    for eps in (0.05, 0.0, 1.0):
        r = np.array([1.0, 0.5, -0.25])
        pos = np.array([[0.0, 0.0, 0.0], r], np.float32)
        m = np.array([0.25, 0.75], np.float32)
        acc, inter, vis, _, _ = oracle.bh_forces(pos, m, 0.5, eps, 32)
        d = np.linalg.norm(r) ** 2 + eps * eps
        a1 = 0.75 * r / d ** 1.5
        a2 = -0.25 * r / d ** 1.5
        assert np.allclose(acc[0], a1, rtol=1e-6, atol=0) and np.allclose(acc[1], a2, rtol=1e-6, atol=0)
        assert inter.tolist() == [[0, 1], [0, 1]] and vis.tolist() == [1, 1]


def test_two_body_closed_form():
    pin_two_body()


def pin_theta0_is_direct():
    for n, tol in ((64, 2e-6), (4096, 1e-4)):
        pos, m = plummer(n, 31) if n > 64 else uniform_cube(n, 31)
        T = oracle.Tree(pos, m, 8)
        acc, pc, pp, vis = T.walk(0.0, EPS, threads=oracle.default_threads())
        assert np.all(vis == T.num_nodes) and np.all(pc == 0) and np.all(pp == n - 1)
        ref = oracle.direct_f64(pos, m, EPS)[T.perm]
        assert oracle.relative_error(acc, ref).max() <= tol


def test_theta0_is_direct_sum():
    pin_theta0_is_direct()


def pin_direct_f32():
    # against the compensated fp64 sum (binary32 rounding only) ...
    pos, m = plummer(3000, 41)
    got = oracle.direct_f32(pos, m, EPS)
    assert oracle.relative_error(got, oracle.direct_f64(pos, m, EPS)).max() < 2e-5
    # ... and, on input already in Morton order with one leaf holding every
    # particle, equal bit for bit to the theta = 0 tree walk (same pairs, same order)
    pos, m = plummer(700, 42)
    perm, _ = oracle.sort(oracle.keys(pos))
    ps, ms = pos[perm], m[perm]
    acc, inter, _, _, _ = oracle.bh_forces(ps, ms, 0.0, EPS, 1000)
    assert np.array_equal(oracle.direct_f32(ps, ms, EPS).view(np.uint32), acc.view(np.uint32))
    tg = np.array([3, 0, 699])
    assert np.array_equal(oracle.direct_f32(ps, ms, EPS, tg), oracle.direct_f32(ps, ms, EPS)[tg])


def test_direct_f32():
    pin_direct_f32()


def pin_term_magnitude():
    """The tolerance scale of nearly cancelling sums: sum over j != i of
    |m_j (x_j - x_i)| / (r^2 + eps^2)^1.5, against numpy in fp64."""
    pos, m = uniform_cube(300, 13)
    m = (m * np.random.default_rng(13).uniform(0.5, 2.0, 300)).astype(np.float32)
    for eps in (0.05, 0.0):
        x = pos.astype(np.float64)
        d = x[None, :, :] - x[:, None, :]
        r2 = (d * d).sum(-1)
        np.fill_diagonal(r2, 1.0)  # the self pair is left out below
        w = m.astype(np.float64)[None, :] * np.sqrt(r2) / (r2 + eps * eps) ** 1.5
        np.fill_diagonal(w, 0.0)
        ref = w.sum(1)
        got = oracle.term_magnitude_f64(pos, m, eps)
        assert np.abs(got - ref).max() <= 1e-12 * ref.max()
        tg = np.array([7, 0, 299])
        assert np.array_equal(oracle.term_magnitude_f64(pos, m, eps, tg), got[tg])
        # never below the magnitude of the sum itself
        assert np.all(np.linalg.norm(oracle.direct_f64(pos, m, eps), axis=1) <= got * (1 + 1e-12))


def test_term_magnitude_against_numpy():
    pin_term_magnitude()


def test_direct_f64_against_numpy():
    pos, m = uniform_cube(200, 8)
    ref = direct_numpy(pos, m, EPS)
    got = oracle.direct_f64(pos, m, EPS)
    assert np.abs(got - ref).max() <= 1e-13 * np.abs(ref).max()
    tg = np.array([5, 0, 199])
    assert np.array_equal(oracle.direct_f64(pos, m, EPS, tg), got[tg])


def test_momentum_conservation():
    pos, m = plummer(2048, 17)
    ref = oracle.direct_f64(pos, m, EPS)
    w = m.astype(np.float64)[:, None]
    assert np.abs((w * ref).sum(0)).max() <= 1e-12 * (w * np.abs(ref)).sum()
    acc, _, _, _, _ = oracle.bh_forces(pos, m, 0.0, EPS, 32)
    assert np.abs((w * acc).sum(0)).max() <= 1e-5 * (w * np.abs(acc)).sum()


def pin_far_clump():
    # a clump of 8 particles far from a lone target: the clump's level-1 cell
    # passes the criterion and is summed as one point mass at its CoM
    rng = np.random.default_rng(4)
    clump = (10.0 + 1e-3 * rng.random((8, 3))).astype(np.float32)
    pos = np.concatenate([[[0.0, 0.0, 0.0]], clump]).astype(np.float32)
    m = np.full(9, 1 / 16, np.float32)
    acc, inter, vis, _, _ = oracle.bh_forces(pos, m, 0.5, EPS, 1)
    assert inter[0].tolist() == [1, 0]
    c = clump.astype(np.float64).mean(0)
    a = 0.5 * c / (c @ c + EPS * EPS) ** 1.5
    assert np.allclose(acc[0], a, rtol=2e-6, atol=0)


def test_far_clump_is_one_cell_term():
    pin_far_clump()


def test_huge_theta_accepts_the_root():
    pos, m = plummer(500, 3)
    acc, inter, vis, _, _ = oracle.bh_forces(pos, m, 1e30, EPS, 32)
    assert np.all(vis == 1) and np.all(inter[:, 0] == 1) and np.all(inter[:, 1] == 0)


def pin_criterion_set_formulation():
    """A node is visited iff no strict ancestor was accepted; the counts follow.
    Decisions here are taken in fp64 from the pages' criterion
    (side_L / d < theta, side_L = side / 2^L); targets with a near tie are skipped."""
    for theta, cap in ((0.5, 4), (0.3, 2), (0.8, 8)):
        pos, m = plummer(400, 5)
        T = oracle.Tree(pos, m, cap)
        acc, pc, pp, vis = T.walk(theta, EPS)
        par = parents_from_escape(T.nodes)
        leaf = oracle.is_leaf(T.nodes, cap)
        side_l = float(T.side) / 2.0 ** T.nodes[:, 3]
        checked = 0
        for i in range(T.n):
            d = np.linalg.norm(T.cm[:, :3].astype(np.float64) - T.ps[i, :3], axis=1)
            margin = side_l - theta * d
            if np.any(np.abs(margin) <= 1e-5 * side_l):
                continue
            acc_k = side_l < theta * d
            visited = np.zeros(T.num_nodes, bool)
            for k in range(T.num_nodes):
                visited[k] = par[k] < 0 or (visited[par[k]] and not acc_k[par[k]])
            want_pc = int((visited & acc_k).sum())
            opened = visited & ~acc_k & leaf
            want_pp = int(T.nodes[opened, 2].sum())
            own = np.nonzero(opened & (T.nodes[:, 1] <= i) & (i < T.nodes[:, 1] + T.nodes[:, 2]))[0]
            want_pp -= len(own)
            assert (pc[i], pp[i], vis[i]) == (want_pc, want_pp, int(visited.sum())), (theta, i)
            checked += 1
        assert checked > 300


def test_criterion_set_formulation():
    pin_criterion_set_formulation()


def pin_recursive_equals_escape():
    for theta, cap, n in ((0.5, 32, 4096), (0.7, 4, 2000), (0.0, 16, 700), (0.3, 1, 600)):
        pos, m = plummer(n, 100 + n)
        T = oracle.Tree(pos, m, cap)
        acc, pc, pp, vis = T.walk(theta, EPS, threads=oracle.default_threads())
        racc, rcnt = T.recursive(theta, EPS)
        assert np.array_equal(acc.view(np.uint32), racc.view(np.uint32))
        assert np.array_equal(np.stack([pc, pp, vis], 1), rcnt)


def test_recursive_equals_escape_walk():
    pin_recursive_equals_escape()


def test_permutation_invariance():
    pos, m = plummer(3000, 44)
    assert len(np.unique(oracle.keys(pos))) == 3000
    acc, inter, vis, vc, _ = oracle.bh_forces(pos, m, 0.5, EPS, 32, True)
    p = np.random.default_rng(0).permutation(3000)
    acc2, inter2, vis2, vc2, _ = oracle.bh_forces(pos[p], m[p], 0.5, EPS, 32, True)
    assert np.array_equal(acc2, acc[p]) and np.array_equal(inter2, inter[p])
    assert np.array_equal(vis2, vis[p]) and np.array_equal(vc2, vc[p])


def pin_degenerate():
    acc, inter, vis, _, nn = oracle.bh_forces(np.zeros((0, 3)), np.zeros(0), 0.5, EPS, 32)
    assert nn == 0 and acc.shape == (0, 3)
    # one particle: the root is its own leaf; d2 = 0 and side 0 tie at 0 < 0,
    # which the strict criterion rejects, so the leaf is opened and self skipped
    acc, inter, vis, vc, nn = oracle.bh_forces([[1.0, 2.0, 3.0]], [0.5], 0.5, EPS, 32, True)
    assert nn == 1 and acc.tolist() == [[0, 0, 0]] and inter.tolist() == [[0, 0]]
    assert vis.tolist() == [1] and vc.tolist() == [1]
    # two coincident particles: same tie; one particle-particle pair of zero force
    acc, inter, vis, vc, nn = oracle.bh_forces([[1.0, 2.0, 3.0]] * 2, [0.5, 0.5], 0.5, EPS, 32, True)
    assert inter.tolist() == [[0, 1], [0, 1]] and acc.tolist() == [[0, 0, 0]] * 2


def test_degenerate_inputs():
    pin_degenerate()


def test_accuracy_soft_pin_against_pages():
    # orrery performance page, "Accuracy": worst 2.03e-2 and RMS 2.03e-3 at 4096,
    # 1.34e-2 / 1.76e-3 at 16384 (theta 0.5). Their generator differs: factor 2.5.
    for n, worst, rms in ((4096, 2.03e-2, 2.03e-3), (16384, 1.34e-2, 1.76e-3)):
        pos, m = plummer(n)
        acc, _, _, _, _ = oracle.bh_forces(pos, m, 0.5, EPS, 32, threads=oracle.default_threads())
        e = oracle.relative_error(acc, oracle.direct_f64(pos, m, EPS))
        assert worst / 2.5 < e.max() < worst * 2.5
        assert rms / 2.5 < math.sqrt((e ** 2).mean()) < rms * 2.5


# ---------------------------------------------------------------------------
# step 9: coherent walk = union of the lanes' walks
# ---------------------------------------------------------------------------
def pin_group_union():
    pos, m = plummer(230, 9)
    T = oracle.Tree(pos, m, 4)
    # width 1: the union of one walk is that walk
    assert np.array_equal(T.group_visits(0.5, EPS, 1), T.walk(0.5, EPS)[3])
    for width in (2, 16, 32, 64):
        got = T.group_visits(0.5, EPS, width)
        for g in range(len(got)):
            u = np.zeros(T.num_nodes, bool)
            for i in range(g * width, min(T.n, (g + 1) * width)):
                u |= T.walk_marks(0.5, EPS, i)
            assert got[g] == u.sum(), (width, g)


def test_group_union_brute_force():
    pin_group_union()


def test_coherent_soft_pins():
    # orrery performance page, "The divergence mitigation": redundancy 1.25 at
    # 16384; coherent visits >= each lane's own; at theta 0 the union is all nodes
    pos, m = plummer(16384)
    acc, inter, vi, vc, nn = oracle.bh_forces(pos, m, 0.5, EPS, 32, True, oracle.default_threads())
    assert np.all(vc >= vi) and np.all(vc <= nn)
    red = vc.mean() / vi.mean()
    assert 1.1 < red < 1.4
    T = oracle.Tree(pos[:500], m[:500], 32)
    assert np.all(T.group_visits(0.0, EPS) == T.num_nodes)


def test_descend_together_contrast():
    # ADR-0029, Alternatives considered: descending with the group visits the
    # same nodes (the union), performs more interactions, and is more accurate;
    # at width 1 it is the independent walk itself
    pos, m = plummer(4096)
    T = oracle.Tree(pos, m, 32)
    a, pc, pp, v = T.walk(0.5, EPS)
    a1, pc1, pp1, v1 = T.descend_together(0.5, EPS, 1)
    assert np.array_equal(a1.view(np.uint32), a.view(np.uint32))
    assert np.array_equal(pc1, pc) and np.array_equal(pp1, pp) and np.array_equal(v1, v)
    ad, pcd, ppd, vd = T.descend_together(0.5, EPS, 32)
    assert np.array_equal(vd, np.repeat(T.group_visits(0.5, EPS, 32), 32)[: T.n])
    assert (pcd + ppd).sum() > 1.3 * (pc + pp).sum()
    ref = oracle.direct_f64(pos, m, EPS)[T.perm]
    rms = lambda e: math.sqrt((e ** 2).mean())
    assert rms(oracle.relative_error(ad, ref)) < 0.7 * rms(oracle.relative_error(a, ref))


def test_two_spheres_generator_layout():
    pos, m = two_spheres(1000)
    assert pos.shape == (2000, 3) and np.all(m == np.float32(1 / 1000))
    assert abs(pos[:1000, 0].mean()) < 1.0 and abs(pos[1000:, 0].mean() - 6.0) < 1.0


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
MISTAKES = [
    ("sign of dx", "float dx = xj - xi[0];", "float dx = xi[0] - xj;", pin_two_body),
    ("dropped softening", "float r2 = d2 + eps2;", "float r2 = d2;", pin_two_body),
    ("self not skipped", "if (j == i) continue;\n                const float *p",
     "const float *p", pin_theta0_is_direct),
    ("escape off by one", "st->nodes[4 * k + 0] = (int32_t)st->num_nodes;",
     "st->nodes[4 * k + 0] = (int32_t)st->num_nodes - 1;", pin_tree_brute_force),
    ("x and z transposed", "key |= xb << (3 * b + 2);", "key |= xb << (3 * b);",
     pin_golden_three_points),
    ("level scaling of the side", "ldexpf(side * side, -2 * level)", "ldexpf(side * side, -level)",
     pin_criterion_set_formulation),
    ("wrong axis in moments", "sx = fmaf(m, ps[4 * j + 0], sx);", "sx = fmaf(m, ps[4 * j + 1], sx);",
     pin_moments),
    ("non-strict criterion", "return cell_side_sq(side, level) < theta2 * d2;",
     "return cell_side_sq(side, level) <= theta2 * d2;", pin_degenerate),
    ("last lane dropped from the union", "i < (g + 1) * width && i < n",
     "i < (g + 1) * width - 1 && i < n", pin_group_union),
    ("the term's denominator r2^2 instead of r2^1.5", "float f = m / (r2 * sqrtf(r2));",
     "float f = m / (r2 * r2);", pin_two_body),
    ("the term's root taken of d2 instead of r2", "float f = m / (r2 * sqrtf(r2));",
     "float f = m / (r2 * sqrtf(d2));", pin_two_body),
    ("the term's mass left out", "float f = m / (r2 * sqrtf(r2));",
     "float f = 1.0f / (r2 * sqrtf(r2));", pin_two_body),
    ("cell term uses the target's mass", "add_term(xi, c[0], c[1], c[2], c[3], eps2, acc);",
     "add_term(xi, c[0], c[1], c[2], t->ps[4 * i + 3], eps2, acc);", pin_far_clump),
    ("equal keys in descending index order", "if (a->index != b->index) return (a->index < b->index) ? -1 : 1;",
     "if (a->index != b->index) return (a->index > b->index) ? -1 : 1;", pin_sort_stable),
    ("keys sorted descending", "if (a->key != b->key) return (a->key < b->key) ? -1 : 1;",
     "if (a->key != b->key) return (a->key > b->key) ? -1 : 1;", pin_sort_stable),
    ("a cell of exactly leaf_cap particles split", "int is_leaf = (count <= st->leaf_cap) || (level == ORACLE_LEVELS);",
     "int is_leaf = (count < st->leaf_cap) || (level == ORACLE_LEVELS);", pin_tree_brute_force),
    ("cube side from the first axis alone", "if (ext > s) s = ext;", "if (a == 0) s = ext;", pin_cube),
    ("quantise rounds instead of flooring", "return (uint32_t)floorf(t);", "return (uint32_t)roundf(t);",
     pin_quantise),
    ("no clamp at the top of the cube", "if (t >= 2097151.0f) return 2097151u;",
     "if (t >= 2097152.0f) return 2097152u;", pin_golden_three_points),
    ("an internal node's first child left out of its sums", "int64_t c = k + 1;\n        while (c < node[0]) {",
     "int64_t c = nodes[4 * (k + 1) + 0];\n        while (c < node[0]) {", pin_moments),
    ("the x sum used for the y coordinate of the CoM", "cm[4 * k + 1] = (M > 0.0f) ? sy / M : 0.0f;",
     "cm[4 * k + 1] = (M > 0.0f) ? sx / M : 0.0f;", pin_moments),
    ("the magnitude scale without the distance factor",
     "s += fabs((double)d->mass[j]) * sqrt(d2) / (r2 * sqrt(r2));",
     "s += fabs((double)d->mass[j]) / (r2 * sqrt(r2));", pin_term_magnitude),
    ("an opened leaf's last particle left out",
     "for (int64_t j = node[1]; j < (int64_t)node[1] + node[2]; ++j) {\n                if (j == i) continue;",
     "for (int64_t j = node[1]; j < (int64_t)node[1] + node[2] - 1; ++j) {\n                if (j == i) continue;",
     pin_theta0_is_direct),
]


@pytest.mark.parametrize("name,old,new,pin", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_planted_mistakes(name, old, new, pin, tmp_path):
    src = oracle.source_text()
    assert src.count(old) == 1, name
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / "variant.so"))
    with oracle.using(lib):
        with pytest.raises(AssertionError):
            pin()
