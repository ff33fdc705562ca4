"""ctypes loader for liborrery_bh.so (argument marshalling only).

Loading fails loudly when the library has not been built: there is no
fallback path of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

_lock = threading.Lock()
_lib = None

OK = 0
EINVAL = -1
ENONFINITE = -2
ERANGE = -3
ECUDA = -4
EWALK = -5
ENOMEM = -6
EINTERNAL = -7
ESCRATCH = -8

INDEPENDENT = 0
COHERENT = 1
COHERENT_16 = 2
COHERENT_64 = 3
DESCEND_TOGETHER = 4
COHERENT_BALLOT = 5
FAST_TERM = 0x100
# coherence width of each traversal (targets sharing one node index)
WIDTH = {INDEPENDENT: 1, COHERENT: 32, COHERENT_16: 16, COHERENT_64: 64, DESCEND_TOGETHER: 32,
         COHERENT_BALLOT: 32}


class Timings(ctypes.Structure):
    """Mirror of orrery_bh_timings."""

    _fields_ = [
        ("h2d_ms", ctypes.c_float),
        ("bbox_ms", ctypes.c_float),
        ("morton_ms", ctypes.c_float),
        ("sort_ms", ctypes.c_float),
        ("gather_ms", ctypes.c_float),
        ("build_ms", ctypes.c_float),
        ("moments_ms", ctypes.c_float),
        ("walk_ms", ctypes.c_float),
        ("scatter_ms", ctypes.c_float),
        ("d2h_ms", ctypes.c_float),
        ("total_ms", ctypes.c_float),
        ("traversal", ctypes.c_int32),
        ("depth", ctypes.c_int32),
        ("n", ctypes.c_int64),
        ("num_nodes", ctypes.c_int64),
        ("launches", ctypes.c_uint64),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class OrreryError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, strerror(status), status))


def load(path: str | None = None):
    """Loads and binds the library (once per process)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(
                "liborrery_bh.so is not built (%s); run tree_traversal_gb300.build.build()" % p)
        lib = ctypes.CDLL(p)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.orrery_bh_forces.argtypes = [P, P, i64, f32, f32, i32, i32, P, P, P, P]
        lib.orrery_bh_forces.restype = ctypes.c_int
        lib.orrery_bh_forces_range.argtypes = [P, P, i64, f32, f32, i32, i32, i64, i64, P, P, P, P]
        lib.orrery_bh_forces_range.restype = ctypes.c_int
        lib.orrery_bh_forces_host.argtypes = [P, P, i64, f32, f32, i32, i32, P, P, P, P]
        lib.orrery_bh_forces_host.restype = ctypes.c_int
        lib.orrery_bh_forces_noalloc.argtypes = [P, P, i64, f32, f32, i32, i32, P, P, P, P]
        lib.orrery_bh_forces_noalloc.restype = ctypes.c_int
        lib.orrery_direct_forces.argtypes = [P, P, i64, f32, P, P]
        lib.orrery_direct_forces.restype = ctypes.c_int
        lib.orrery_bh_tree.argtypes = [P, P, i64, i32, P, P, P, P, P, i64,
                                       ctypes.POINTER(ctypes.c_int64), P]
        lib.orrery_bh_tree.restype = ctypes.c_int
        lib.orrery_bh_max_nodes.argtypes = [i64, i32]
        lib.orrery_bh_max_nodes.restype = i64
        lib.orrery_bh_last_timings.argtypes = [ctypes.POINTER(Timings)]
        lib.orrery_bh_last_timings.restype = ctypes.c_int
        lib.orrery_fp32_fma_rate.argtypes = [ctypes.POINTER(ctypes.c_double)] * 3 + [P]
        lib.orrery_fp32_fma_rate.restype = ctypes.c_int
        lib.orrery_bh_kernel_launches.argtypes = []
        lib.orrery_bh_kernel_launches.restype = ctypes.c_uint64
        lib.orrery_bh_strerror.argtypes = [ctypes.c_int]
        lib.orrery_bh_strerror.restype = ctypes.c_char_p
        lib.orrery_bh_release.argtypes = []
        lib.orrery_bh_release.restype = None
        _lib = lib
        return lib


def strerror(status: int) -> str:
    return load().orrery_bh_strerror(int(status)).decode()
