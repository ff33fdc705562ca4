"""CPU oracle of the Barnes-Hut monopole force evaluation (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library in
``tree_traversal_gb300``) never does, and this package imports nothing from it.

The arithmetic lives in ``orrery_oracle.c`` (plain C, binary32 IEEE operations,
compiled with ``-ffp-contract=off``); this module compiles it with gcc and
wraps it with ctypes and numpy. Each wrapper names the step it follows; the
step definitions and the pages they come from are in the C file's comments.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
facts that do not come from the oracle itself (hand-derived keys, a numpy
stable sort, a brute-force cell enumeration, closed forms, theta = 0 against a
compensated fp64 direct sum, a separately built pointer tree, brute-force set
unions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orrery_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liborrery_oracle.so")
_lock = threading.Lock()
_lib = None

LEVELS = 21


def build(force: bool = False) -> str:
    """Compiles the oracle library with gcc (no vendor flags, no -march)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


class using:
    """Context manager: run the wrappers against another build of the C file.

    The tests use it to plant a mistake in a copy of the oracle and check that
    a pin catches it."""

    def __init__(self, lib_path: str):
        self.path = lib_path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def compile_variant(src_text: str, out_path: str) -> str:
    """Compiles C source text (a modified copy of the oracle) with the oracle's flags."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-w", "-o", out_path, c_path, "-lm", "-lpthread"],
                   check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(lib):
    P = ctypes.c_void_p
    i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
    lib.oracle_cube.argtypes = [P, i64, P, P, P]
    lib.oracle_cube.restype = None
    lib.oracle_quantise.argtypes = [f32, f32, f32]
    lib.oracle_quantise.restype = ctypes.c_uint32
    lib.oracle_interleave.argtypes = [ctypes.c_uint32] * 3
    lib.oracle_interleave.restype = ctypes.c_uint64
    lib.oracle_keys.argtypes = [P, i64, P, f32, P]
    lib.oracle_keys.restype = None
    lib.oracle_sort.argtypes = [P, i64, P, P]
    lib.oracle_sort.restype = ctypes.c_int
    lib.oracle_build.argtypes = [P, i64, i32, P, i64]
    lib.oracle_build.restype = i64
    lib.oracle_moments.argtypes = [P, P, i64, i32, P]
    lib.oracle_moments.restype = ctypes.c_int
    lib.oracle_walk.argtypes = [P, P, P, i64, i32, f32, f32, f32, P, i64, P, P, P, P,
                                ctypes.c_int]
    lib.oracle_walk.restype = ctypes.c_int
    lib.oracle_walk_marks.argtypes = [P, P, P, i64, i32, f32, f32, f32, i64, P]
    lib.oracle_walk_marks.restype = None
    lib.oracle_group_visits.argtypes = [P, P, P, i64, i32, f32, f32, f32, i64, i32, P,
                                        i64, P]
    lib.oracle_group_visits.restype = ctypes.c_int
    lib.oracle_descend_together.argtypes = [P, P, P, i64, i32, f32, f32, f32, i64, i32, P, P,
                                            P, P]
    lib.oracle_descend_together.restype = ctypes.c_int
    lib.oracle_bh_forces.argtypes = [P, P, i64, f32, f32, i32, P, P, P, P, ctypes.c_int]
    lib.oracle_bh_forces.restype = i64
    lib.oracle_direct_f64.argtypes = [P, P, i64, f64, P, i64, P, ctypes.c_int]
    lib.oracle_direct_f64.restype = ctypes.c_int
    lib.oracle_term_magnitude_f64.argtypes = [P, P, i64, f64, P, i64, P, ctypes.c_int]
    lib.oracle_term_magnitude_f64.restype = ctypes.c_int
    lib.oracle_direct_f32.argtypes = [P, P, i64, f32, P, i64, P, ctypes.c_int]
    lib.oracle_direct_f32.restype = ctypes.c_int
    lib.oracle_bh_recursive.argtypes = [P, P, i64, i32, f32, f32, f32, P, P]
    lib.oracle_bh_recursive.restype = ctypes.c_int
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------
# Step 1: bounding cube
# --------------------------------------------------------------------------
def cube(pos) -> tuple[np.ndarray, np.float32, np.float32]:
    """Returns (lo[3], side, inv) of the bounding cube (step 1)."""
    pos = _f32(pos).reshape(-1, 3)
    lo = np.zeros(3, np.float32)
    side = np.zeros(1, np.float32)
    inv = np.zeros(1, np.float32)
    _load().oracle_cube(_ptr(pos), pos.shape[0], _ptr(lo), _ptr(side), _ptr(inv))
    return lo, side[0], inv[0]


# --------------------------------------------------------------------------
# Step 2: Morton keys
# --------------------------------------------------------------------------
def quantise(x: float, lo: float, inv: float) -> int:
    return int(_load().oracle_quantise(float(x), float(lo), float(inv)))


def interleave(qx: int, qy: int, qz: int) -> int:
    return int(_load().oracle_interleave(qx, qy, qz))


def keys(pos, lo=None, inv=None) -> np.ndarray:
    pos = _f32(pos).reshape(-1, 3)
    if lo is None:
        lo, _, inv = cube(pos)
    lo = _f32(lo)
    out = np.empty(pos.shape[0], np.uint64)
    _load().oracle_keys(_ptr(pos), pos.shape[0], _ptr(lo), float(inv), _ptr(out))
    return out


# --------------------------------------------------------------------------
# Step 3: sort
# --------------------------------------------------------------------------
def sort(keys_: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Returns (perm, sorted_keys): perm[k] = original index at sorted slot k."""
    keys_ = np.ascontiguousarray(keys_, dtype=np.uint64)
    n = keys_.shape[0]
    perm = np.empty(n, np.uint32)
    sk = np.empty(n, np.uint64)
    if _load().oracle_sort(_ptr(keys_), n, _ptr(perm), _ptr(sk)) != 0:
        raise MemoryError("oracle_sort")
    return perm, sk


# --------------------------------------------------------------------------
# Step 4: tree
# --------------------------------------------------------------------------
def build_tree(sorted_keys: np.ndarray, leaf_cap: int) -> np.ndarray:
    """Returns the node array [num_nodes, 4] int32 {escape, first, count, level}."""
    sorted_keys = np.ascontiguousarray(sorted_keys, dtype=np.uint64)
    n = sorted_keys.shape[0]
    max_nodes = 22 * n + 1
    nodes = np.empty((max_nodes, 4), np.int32)
    nn = _load().oracle_build(_ptr(sorted_keys), n, int(leaf_cap), _ptr(nodes), max_nodes)
    if nn < 0:
        raise RuntimeError("oracle_build overflow")
    return nodes[:nn].copy()


def is_leaf(nodes: np.ndarray, leaf_cap: int) -> np.ndarray:
    return (nodes[:, 2] <= leaf_cap) | (nodes[:, 3] == LEVELS)


# --------------------------------------------------------------------------
# Step 5: moments
# --------------------------------------------------------------------------
def moments(ps: np.ndarray, nodes: np.ndarray, leaf_cap: int) -> np.ndarray:
    """Returns [num_nodes, 4] float32 {CoM_x, CoM_y, CoM_z, M}."""
    ps = _f32(ps).reshape(-1, 4)
    nodes = np.ascontiguousarray(nodes, dtype=np.int32)
    cm = np.zeros((nodes.shape[0], 4), np.float32)
    if _load().oracle_moments(_ptr(ps), _ptr(nodes), nodes.shape[0], int(leaf_cap), _ptr(cm)) != 0:
        raise MemoryError("oracle_moments")
    return cm


class Tree:
    """Steps 1-5 on one input, with every intermediate kept."""

    def __init__(self, pos, mass, leaf_cap: int = 32):
        pos = _f32(pos).reshape(-1, 3)
        mass = _f32(mass).reshape(-1)
        self.n = pos.shape[0]
        self.leaf_cap = int(leaf_cap)
        self.lo, self.side, self.inv = cube(pos)
        self.keys = keys(pos, self.lo, self.inv)
        self.perm, self.sorted_keys = sort(self.keys)
        self.ps = np.empty((self.n, 4), np.float32)
        self.ps[:, :3] = pos[self.perm]
        self.ps[:, 3] = mass[self.perm]
        self.nodes = build_tree(self.sorted_keys, self.leaf_cap)
        self.cm = moments(self.ps, self.nodes, self.leaf_cap)

    @property
    def num_nodes(self) -> int:
        return int(self.nodes.shape[0])

    @property
    def depth(self) -> int:
        return int(self.nodes[:, 3].max()) if self.num_nodes else 0

    def _args(self, theta, eps):
        return (_ptr(self.ps), _ptr(self.nodes), _ptr(self.cm), self.num_nodes,
                self.leaf_cap, float(self.side), float(theta), float(eps))

    def walk(self, theta: float, eps: float, targets=None, threads: int = 1):
        """Independent walk (steps 6-8) of sorted targets; all if targets is None.

        Returns (acc [t,3] f32, pc [t] u32, pp [t] u32, visits [t] u32) in the
        order of ``targets``."""
        if targets is None:
            nt, tp, tgt = self.n, None, None
        else:
            tgt = np.ascontiguousarray(targets, dtype=np.int64)
            nt, tp = tgt.shape[0], _ptr(tgt)
        acc = np.zeros((nt, 3), np.float32)
        pc = np.zeros(nt, np.uint32)
        pp = np.zeros(nt, np.uint32)
        vis = np.zeros(nt, np.uint32)
        rc = _load().oracle_walk(*self._args(theta, eps), tp, nt, _ptr(acc), _ptr(pc), _ptr(pp),
                                 _ptr(vis), int(threads))
        if rc != 0:
            raise RuntimeError("oracle_walk")
        return acc, pc, pp, vis

    def walk_marks(self, theta: float, eps: float, i: int) -> np.ndarray:
        """Boolean array over nodes: visited by the walk of sorted target i."""
        mark = np.zeros(max(self.num_nodes, 1), np.uint8)
        _load().oracle_walk_marks(*self._args(theta, eps), int(i), _ptr(mark))
        return mark[: self.num_nodes].astype(bool)

    def group_visits(self, theta: float, eps: float, width: int = 32, groups=None) -> np.ndarray:
        """Step 9: union size of each width-wide group of sorted targets."""
        if groups is None:
            ng, gp = (self.n + width - 1) // width, None
        else:
            g = np.ascontiguousarray(groups, dtype=np.int64)
            ng, gp = g.shape[0], _ptr(g)
        out = np.zeros(ng, np.uint32)
        rc = _load().oracle_group_visits(*self._args(theta, eps), self.n, int(width), gp, ng,
                                         _ptr(out))
        if rc != 0:
            raise MemoryError("oracle_group_visits")
        return out

    def descend_together(self, theta: float, eps: float, width: int = 32):
        """The rejected group-descending scheme (sorted order): (acc, pc, pp, visits)."""
        acc = np.zeros((self.n, 3), np.float32)
        pc = np.zeros(self.n, np.uint32)
        pp = np.zeros(self.n, np.uint32)
        vis = np.zeros(self.n, np.uint32)
        _load().oracle_descend_together(*self._args(theta, eps), self.n, int(width), _ptr(acc),
                                        _ptr(pc), _ptr(pp), _ptr(vis))
        return acc, pc, pp, vis

    def recursive(self, theta: float, eps: float):
        """Cross-check: pointer tree + recursive walk, sorted order.

        Returns (acc [n,3], counts [n,3] {pc, pp, visits})."""
        acc = np.zeros((self.n, 3), np.float32)
        cnt = np.zeros((self.n, 3), np.uint32)
        rc = _load().oracle_bh_recursive(_ptr(self.sorted_keys), _ptr(self.ps), self.n,
                                         self.leaf_cap, float(self.side), float(theta),
                                         float(eps), _ptr(acc), _ptr(cnt))
        if rc != 0:
            raise MemoryError("oracle_bh_recursive")
        return acc, cnt


def bh_forces(pos, mass, theta: float = 0.5, eps: float = 0.05, leaf_cap: int = 32,
              coherent_visits: bool = False, threads: int | None = None):
    """Whole evaluation (step 10), caller order.

    Returns (acc [n,3] f32, interactions [n,2] u32, visits_ind [n] u32,
    visits_coh [n] u32 or None, num_nodes)."""
    pos = _f32(pos).reshape(-1, 3)
    mass = _f32(mass).reshape(-1)
    n = pos.shape[0]
    acc = np.zeros((n, 3), np.float32)
    inter = np.zeros((n, 2), np.uint32)
    vi = np.zeros(n, np.uint32)
    vc = np.zeros(n, np.uint32) if coherent_visits else None
    nn = _load().oracle_bh_forces(_ptr(pos), _ptr(mass), n, float(theta), float(eps),
                                  int(leaf_cap), _ptr(acc), _ptr(inter), _ptr(vi), _ptr(vc),
                                  int(threads or 1))
    if nn < 0:
        raise MemoryError("oracle_bh_forces")
    return acc, inter, vi, vc, int(nn)


def direct_f64(pos, mass, eps: float = 0.05, targets=None, threads: int | None = None) -> np.ndarray:
    """Compensated fp64 direct sum; targets are ORIGINAL indices. [t,3] float64."""
    pos = _f32(pos).reshape(-1, 3)
    mass = _f32(mass).reshape(-1)
    if targets is None:
        nt, tp = pos.shape[0], None
    else:
        tgt = np.ascontiguousarray(targets, dtype=np.int64)
        nt, tp = tgt.shape[0], _ptr(tgt)
    out = np.zeros((nt, 3), np.float64)
    rc = _load().oracle_direct_f64(_ptr(pos), _ptr(mass), pos.shape[0], float(eps), tp, nt,
                                   _ptr(out), int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_direct_f64")
    return out


def direct_f32(pos, mass, eps: float = 0.05, targets=None, threads: int | None = None) -> np.ndarray:
    """Direct sum in binary32 with the walk's particle term, j ascending in
    caller order; targets are original indices. [t,3] float32."""
    pos = _f32(pos).reshape(-1, 3)
    mass = _f32(mass).reshape(-1)
    if targets is None:
        nt, tp = pos.shape[0], None
    else:
        tgt = np.ascontiguousarray(targets, dtype=np.int64)
        nt, tp = tgt.shape[0], _ptr(tgt)
    out = np.zeros((nt, 3), np.float32)
    rc = _load().oracle_direct_f32(_ptr(pos), _ptr(mass), pos.shape[0], float(eps), tp, nt,
                                   _ptr(out), int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_direct_f32")
    return out


def term_magnitude_f64(pos, mass, eps: float = 0.05, targets=None,
                       threads: int | None = None) -> np.ndarray:
    """Per target, the fp64 sum over j != i of |m_j (x_j - x_i)| / (r^2 + eps^2)^1.5:
    the scale against which two fp32 evaluations of a nearly cancelling sum
    are compared. targets are ORIGINAL indices. [t] float64."""
    pos = _f32(pos).reshape(-1, 3)
    mass = _f32(mass).reshape(-1)
    if targets is None:
        nt, tp = pos.shape[0], None
    else:
        tgt = np.ascontiguousarray(targets, dtype=np.int64)
        nt, tp = tgt.shape[0], _ptr(tgt)
    out = np.zeros(nt, np.float64)
    rc = _load().oracle_term_magnitude_f64(_ptr(pos), _ptr(mass), pos.shape[0], float(eps), tp,
                                           nt, _ptr(out), int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_term_magnitude_f64")
    return out


def relative_error(acc, ref) -> np.ndarray:
    """Per-target relative error |a - a_ref| / |a_ref| (vector norms)."""
    acc = np.asarray(acc, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.linalg.norm(acc - ref, axis=1) / np.linalg.norm(ref, axis=1)
