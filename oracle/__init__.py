"""ORACLE -- test infrastructure, not part of the product.

A plain float64 CPU implementation of the data-parallel step (oracle.c), a
message-passing ring simulator with traffic counters (ring.py) and pure
Python brute force for tiny inputs (brute.py).  Only tests/, the smoke check
of __graft_entry__ and bench.py's CPU-baseline leg may import this package.
It shares no code with the CUDA path and imports nothing from it.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

from . import build as _build

_LIB = None


class Problem(ctypes.Structure):
    _fields_ = [
        ("psi", ctypes.c_int64),
        ("n", ctypes.c_int32), ("a", ctypes.c_int32), ("stage", ctypes.c_int32), ("nseg", ctypes.c_int32),
        ("seg", ctypes.c_void_p),
        ("grads", ctypes.c_void_p),
        ("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("replicas", ctypes.c_void_p),
        ("gbar", ctypes.c_void_p),
        ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
        ("loss_scale", ctypes.c_float),
        ("t", ctypes.c_int32), ("found", ctypes.c_int32),
        ("nonfinite", ctypes.c_int64),
        ("nthreads", ctypes.c_int32), ("pad", ctypes.c_int32),
    ]


def lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        L.oracle_step.argtypes = [ctypes.POINTER(Problem)]
        L.oracle_step.restype = ctypes.c_int
        L.oracle_reduce.argtypes = [ctypes.POINTER(Problem)]
        L.oracle_reduce.restype = ctypes.c_int
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        _LIB = L
    return _LIB


def _ptrs(arrs: Sequence[np.ndarray], dtype) -> ctypes.Array:
    for x in arrs:
        assert x.dtype == dtype and x.flags.c_contiguous, (x.dtype, dtype)
    return (ctypes.c_void_p * max(1, len(arrs)))(*[x.ctypes.data for x in arrs])


def _seg_array(segs) -> np.ndarray:
    a = np.zeros((max(1, len(segs)), 4), dtype=np.int64)
    for k, s in enumerate(segs):
        a[k] = s
    return a


def _problem(psi, n, a, stage, segs, grads, master, m, v, replicas, lr, beta1, beta2, eps, loss_scale, t,
             gbar, threads, keep):
    seg = _seg_array(segs)
    keep.append(seg)
    gp = _ptrs(grads, np.uint16)
    mp, m1, v1 = _ptrs(master, np.float32), _ptrs(m, np.float32), _ptrs(v, np.float32)
    keep += [gp, mp, m1, v1]
    rp = None
    if replicas is not None:
        rp = _ptrs(replicas, np.uint16)
        keep.append(rp)
    P = Problem()
    P.psi, P.n, P.a, P.stage, P.nseg = psi, n, a, stage, len(segs)
    P.seg = seg.ctypes.data
    P.grads = ctypes.cast(gp, ctypes.c_void_p)
    P.master, P.m, P.v = (ctypes.cast(mp, ctypes.c_void_p), ctypes.cast(m1, ctypes.c_void_p),
                          ctypes.cast(v1, ctypes.c_void_p))
    P.replicas = ctypes.cast(rp, ctypes.c_void_p) if rp is not None else None
    if gbar is not None:
        assert gbar.dtype == np.float64 and gbar.size >= psi
    P.gbar = gbar.ctypes.data if gbar is not None else None
    P.lr, P.beta1, P.beta2, P.eps, P.loss_scale = lr, beta1, beta2, eps, loss_scale
    P.t = t
    P.nthreads = threads
    return P


def step(psi: int, n: int, a: int, stage: int, segs, grads: List[np.ndarray], master: List[np.ndarray],
         m: List[np.ndarray], v: List[np.ndarray], replicas: Optional[List[np.ndarray]], lr: float, beta1: float,
         beta2: float, eps: float, loss_scale: float, t: int, gbar: Optional[np.ndarray] = None,
         threads: int = 1) -> dict:
    """One step in place on the numpy arrays.  Returns found / nonfinite / t."""
    keep: list = []
    P = _problem(psi, n, a, stage, segs, grads, master, m, v, replicas, lr, beta1, beta2, eps, loss_scale, t,
                 gbar, threads, keep)
    rc = lib().oracle_step(ctypes.byref(P))
    if rc != 0:
        raise RuntimeError("oracle_step failed: %d" % rc)
    return {"found": int(P.found), "nonfinite": int(P.nonfinite), "t": int(P.t)}


def reduce(psi: int, n: int, a: int, grads: List[np.ndarray], loss_scale: float, threads: int = 1) -> dict:
    """The exact averaged gradient gbar (float64) and the non-finite decision."""
    keep: list = []
    gbar = np.zeros(max(1, psi), dtype=np.float64)
    dummy = [np.zeros(1, np.float32)] * n
    P = _problem(psi, n, a, 1, [], grads, dummy, dummy, dummy, None, 0.0, 0.0, 0.0, 0.0, loss_scale, 0, gbar,
                 threads, keep)
    rc = lib().oracle_reduce(ctypes.byref(P))
    if rc != 0:
        raise RuntimeError("oracle_reduce failed: %d" % rc)
    return {"gbar": gbar[:psi], "found": int(P.found), "nonfinite": int(P.nonfinite)}


def f32_to_bf16(x: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(np.float32(x))))


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    f = lib().oracle_f32_to_bf16
    return np.array([f(float(v)) for v in np.asarray(x, dtype=np.float32).ravel()], dtype=np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
