"""Python face of the C ABI: torch tensors in, torch tensors out.

Only argument checking and marshalling happen here; every step of the force
evaluation runs in the CUDA library. PyTorch provides device memory and the
current stream.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib

_TRAVERSALS = {"independent": _lib.INDEPENDENT, "coherent": _lib.COHERENT,
               "coherent16": _lib.COHERENT_16, "coherent64": _lib.COHERENT_64,
               "together": _lib.DESCEND_TOGETHER, "ballot": _lib.COHERENT_BALLOT}
_TRAVERSALS.update({v: v for v in list(_TRAVERSALS.values())})


def _traversal(t) -> int:
    try:
        return _TRAVERSALS[t]
    except KeyError:
        raise ValueError("traversal must be one of %s, got %r"
                         % (sorted(k for k in _TRAVERSALS if isinstance(k, str)), t)) from None


def _check_device(t: torch.Tensor, name: str, shape, dtype=torch.float32):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %s tensor of shape %s" % (name, dtype, shape))


def _stream_handle(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def bh_forces(pos: torch.Tensor, mass: torch.Tensor, theta: float = 0.5, eps: float = 0.05,
              leaf_cap: int = 32, traversal="coherent", counters: bool = True, out=None,
              fast_term: bool = False, targets=None):
    """Accelerations of n particles (caller order) on the current CUDA stream.

    pos [n, 3] float32, mass [n] float32, both CUDA and contiguous.
    Returns (acc [n, 3] float32, interactions [n, 2] int32 {particle-cell,
    particle-particle} or None, visits [n] int32 or None); the counters are
    uint32 values stored in int32 tensors (they never exceed 2^31).
    ``out`` may pass preallocated (acc, interactions, visits) tensors.
    ``fast_term`` selects the hardware approximate inverse square root
    (ORRERY_FAST_TERM) instead of the fixed Newton sequence: faster; both are
    within the same tolerance of the law, and the counts are identical.
    ``targets`` = (begin, end) walks only the sorted targets [begin, end)
    (orrery_bh_forces_range): only their entries of the outputs are written."""
    n = int(pos.shape[0]) if pos.dim() == 2 else -1
    _check_device(pos, "pos", (n, 3))
    _check_device(mass, "mass", (n,))
    if mass.device != pos.device:
        raise ValueError("pos and mass must be on the same device")
    dev = pos.device
    if out is not None:
        acc, inter, visits = out
    else:
        acc = torch.empty((n, 3), dtype=torch.float32, device=dev)
        inter = torch.empty((n, 2), dtype=torch.int32, device=dev) if counters else None
        visits = torch.empty((n,), dtype=torch.int32, device=dev) if counters else None
    _check_device(acc, "acc", (n, 3))
    if inter is not None:
        _check_device(inter, "interactions", (n, 2), torch.int32)
    if visits is not None:
        _check_device(visits, "visits", (n,), torch.int32)
    flags = _traversal(traversal) | (_lib.FAST_TERM if fast_term else 0)
    with torch.cuda.device(dev):
        if targets is None:
            rc = _lib.load().orrery_bh_forces(
                _ptr(pos), _ptr(mass), n, float(theta), float(eps), int(leaf_cap), flags,
                _ptr(acc), _ptr(inter), _ptr(visits), _stream_handle(dev))
            name = "orrery_bh_forces"
        else:
            begin, end = (int(v) for v in targets)
            rc = _lib.load().orrery_bh_forces_range(
                _ptr(pos), _ptr(mass), n, float(theta), float(eps), int(leaf_cap), flags,
                begin, end, _ptr(acc), _ptr(inter), _ptr(visits), _stream_handle(dev))
            name = "orrery_bh_forces_range"
    if rc != _lib.OK:
        raise _lib.OrreryError(rc, name)
    return acc, inter, visits


def shard(n: int, rank: int, world: int, align: int = 64) -> tuple[int, int]:
    """The sorted-target slice [begin, end) of rank ``rank`` of ``world`` when
    one evaluation is split into equal slices whose edges are multiples of
    ``align`` (the coherence width, so every rank reports the full
    evaluation's visit counts); the slices tile [0, n)."""
    if world < 1 or not 0 <= rank < world or n < 0 or align < 1:
        raise ValueError("invalid shard arguments")
    groups = -(-n // align)
    lo = groups * rank // world
    hi = groups * (rank + 1) // world
    return min(n, lo * align), min(n, hi * align)


def bh_forces_host(pos: np.ndarray, mass: np.ndarray, theta: float = 0.5, eps: float = 0.05,
                   leaf_cap: int = 32, traversal="coherent", out=None, device=None,
                   fast_term: bool = False):
    """The same evaluation from host arrays (numpy or CPU tensors, page-locked
    for the fastest copies) to host arrays; the copies run inside the call,
    and page-locked outputs are written by the walk directly.
    ``out`` = (acc [n,3] f32, interactions [n,2] u32 or None, visits [n] u32 or None);
    ``fast_term`` as for bh_forces."""
    def host_ptr(a, shape, dtype):
        if isinstance(a, torch.Tensor):
            if a.is_cuda or not a.is_contiguous() or tuple(a.shape) != shape or \
                    a.dtype != {np.float32: torch.float32, np.uint32: torch.int32}[dtype]:
                raise ValueError("host tensor of shape %s expected" % (shape,))
            return ctypes.c_void_p(a.data_ptr())
        if a.dtype != dtype or tuple(a.shape) != shape or not a.flags["C_CONTIGUOUS"]:
            raise ValueError("host array of shape %s and dtype %s expected" % (shape, dtype))
        return a.ctypes.data_as(ctypes.c_void_p)

    n = int(pos.shape[0])
    if out is None:
        out = (np.empty((n, 3), np.float32), np.empty((n, 2), np.uint32), np.empty(n, np.uint32))
    acc, inter, visits = out
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        rc = _lib.load().orrery_bh_forces_host(
            host_ptr(pos, (n, 3), np.float32), host_ptr(mass, (n,), np.float32), n, float(theta),
            float(eps), int(leaf_cap), _traversal(traversal) | (_lib.FAST_TERM if fast_term else 0),
            host_ptr(acc, (n, 3), np.float32),
            None if inter is None else host_ptr(inter, (n, 2), np.uint32),
            None if visits is None else host_ptr(visits, (n,), np.uint32), _stream_handle(dev))
    if rc != _lib.OK:
        raise _lib.OrreryError(rc, "orrery_bh_forces_host")
    return acc, inter, visits


def direct_forces(pos: torch.Tensor, mass: torch.Tensor, eps: float = 0.05, out=None):
    """Direct O(n^2) summation of the same softened law (every pair, caller
    order), on the current CUDA stream. Returns acc [n, 3] float32."""
    n = int(pos.shape[0]) if pos.dim() == 2 else -1
    _check_device(pos, "pos", (n, 3))
    _check_device(mass, "mass", (n,))
    dev = pos.device
    acc = torch.empty((n, 3), dtype=torch.float32, device=dev) if out is None else out
    _check_device(acc, "acc", (n, 3))
    with torch.cuda.device(dev):
        rc = _lib.load().orrery_direct_forces(_ptr(pos), _ptr(mass), n, float(eps), _ptr(acc),
                                              _stream_handle(dev))
    if rc != _lib.OK:
        raise _lib.OrreryError(rc, "orrery_direct_forces")
    return acc


def max_nodes(n: int, leaf_cap: int = 32) -> int:
    v = _lib.load().orrery_bh_max_nodes(int(n), int(leaf_cap))
    if v < 0:
        raise ValueError("invalid n or leaf_cap")
    return int(v)


def bh_tree(pos: torch.Tensor, mass: torch.Tensor, leaf_cap: int = 32) -> dict:
    """Cube, sorted keys, permutation, nodes and moments of one build.

    Returns a dict of CUDA tensors: cube [5] {lo_x, lo_y, lo_z, side, inv},
    keys [n] int64 (the uint64 key bits), perm [n] int32, nodes
    [num_nodes, 4] int32 {escape, first, count, level}, com [num_nodes, 4]
    float32 {CoM_x, CoM_y, CoM_z, M}."""
    n = int(pos.shape[0])
    _check_device(pos, "pos", (n, 3))
    _check_device(mass, "mass", (n,))
    dev = pos.device
    cap = max_nodes(n, leaf_cap)
    cube = torch.zeros(5, dtype=torch.float32, device=dev)
    keys = torch.empty(n, dtype=torch.int64, device=dev)
    perm = torch.empty(n, dtype=torch.int32, device=dev)
    nodes = torch.empty((max(cap, 1), 4), dtype=torch.int32, device=dev)
    com = torch.empty((max(cap, 1), 4), dtype=torch.float32, device=dev)
    nn = ctypes.c_int64(0)
    with torch.cuda.device(dev):
        rc = _lib.load().orrery_bh_tree(
            _ptr(pos), _ptr(mass), n, int(leaf_cap), _ptr(cube), _ptr(keys), _ptr(perm),
            _ptr(nodes), _ptr(com), cap, ctypes.byref(nn), _stream_handle(dev))
    if rc != _lib.OK:
        raise _lib.OrreryError(rc, "orrery_bh_tree")
    k = int(nn.value)
    return dict(cube=cube, keys=keys, perm=perm, nodes=nodes[:k], com=com[:k])


def last_timings() -> dict:
    t = _lib.Timings()
    rc = _lib.load().orrery_bh_last_timings(ctypes.byref(t))
    if rc != _lib.OK:
        raise _lib.OrreryError(rc, "orrery_bh_last_timings")
    return t.as_dict()


def fp32_fma_rate(device=None) -> dict:
    """Measured FP32 FMA rate of the GPU, long independent chains on every SM,
    on the current stream: {"scalar": TFLOP/s of FFMA, "packed": TFLOP/s of
    FFMA2, "sm_mhz": the SM clock during the scalar probe}."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    scalar, packed, mhz = ctypes.c_double(0.0), ctypes.c_double(0.0), ctypes.c_double(0.0)
    with torch.cuda.device(dev):
        rc = _lib.load().orrery_fp32_fma_rate(ctypes.byref(scalar), ctypes.byref(packed),
                                               ctypes.byref(mhz), _stream_handle(dev))
    if rc != _lib.OK:
        raise _lib.OrreryError(rc, "orrery_fp32_fma_rate")
    return {"scalar": float(scalar.value), "packed": float(packed.value), "sm_mhz": float(mhz.value)}


def kernel_launches() -> int:
    return int(_lib.load().orrery_bh_kernel_launches())


def release() -> None:
    _lib.load().orrery_bh_release()
