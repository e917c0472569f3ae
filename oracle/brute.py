"""ORACLE -- test infrastructure.  Pure-Python brute force for tiny inputs.

* exact_gbar: the averaged gradient with exact rational arithmetic
  (fractions.Fraction), rounded once to float64 -- the plain definition of
  gbar = (sum_r sum_k g_{r,k}) / (n S) with no rounding inside the sum.
* ring_gbar: the averaged gradient as the simulated ring actually computes
  it hop by hop (ring.py), after each rank has accumulated its micro-steps
  locally with no communication ("Distributed Training: Split along the Four
  Axes", worked example: accumulate locally, one all-reduce after the a-th
  micro-step), in float32 or float32 (hi, lo) pairs; or ("f32chain") with
  every rank folding its micro-steps one at a time into the (hi, lo) pair that
  arrives from its left neighbour.  This is the reduction
  order the GPU path promises, derived from message passing rather than from
  the GPU code.
* tree_gbar: the same local accumulation, then the ranks' sums added up the
  simulated binomial tree of tree.py (the second reduction order).
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence

import numpy as np

from .ring import Ring, two_sum32


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def exact_gbar(grads: Sequence[np.ndarray], n: int, a: int, loss_scale: float) -> np.ndarray:
    """grads: n*a bf16 bit arrays (rank-major).  Exact rational sum, one rounding to float64."""
    vals = [bf16_bits_to_f32(g).astype(np.float64) for g in grads]
    psi = vals[0].size if vals else 0
    den = Fraction(n) * Fraction(float(np.float32(loss_scale)))
    out = np.zeros(psi, dtype=np.float64)
    for i in range(psi):
        s = Fraction(0)
        for q in range(n * a):
            s += Fraction(float(vals[q][i]))
        out[i] = float(s / den)
    return out


def local_accumulate(grads: Sequence[np.ndarray], n: int, a: int, arith: str) -> List:
    """Rank-local accumulation of the a micro-steps, left to right, before any communication."""
    res = []
    for r in range(n):
        xs = [bf16_bits_to_f32(grads[r * a + k]) for k in range(a)]
        if arith == "f32pair":
            h = xs[0].copy()
            lo = np.zeros_like(h)
            for k in range(1, a):
                h, e = two_sum32(h, xs[k])
                lo = (lo + e).astype(np.float32)
            res.append((h, lo))
        elif arith == "f32":
            h = xs[0].copy()
            for k in range(1, a):
                h = (h + xs[k]).astype(np.float32)
            res.append(h)
        else:
            h = xs[0].astype(np.float64)
            for k in range(1, a):
                h = h + xs[k].astype(np.float64)
            res.append(h)
    return res


def ring_gbar(grads: Sequence[np.ndarray], n: int, a: int, segs, psi: int, loss_scale: float,
              arith: str = "f32") -> np.ndarray:
    """gbar as the ring computes it: float32 partials ("f32") or float32 (hi, lo) pairs ("f32pair") after
    rank-local accumulation, or a float32 (hi, lo) pair into which every rank folds its unsummed micro-steps
    ("f32chain"); then hi + lo, then one multiply by fl32(1 / (n S))."""
    if arith == "f32chain":
        loc = [[bf16_bits_to_f32(grads[r * a + k]) for k in range(a)] for r in range(n)]
    else:
        loc = local_accumulate(grads, n, a, arith)
    ring = Ring(n, segs, psi)
    red = ring.reduce_scatter(loc, arith=arith, wire_bytes=4)
    inv = np.float32(1.0 / (float(n) * float(np.float32(loss_scale))))
    out = np.zeros(psi, dtype=np.float32)
    for s in range(n):
        if arith in ("f32pair", "f32chain"):
            H, L = red[s]
            p = (H + L).astype(np.float32)
        else:
            p = np.asarray(red[s], dtype=np.float32)
        ring._put(out, s, (p * inv).astype(np.float32))
    return out


def tree_gbar(grads: Sequence[np.ndarray], n: int, a: int, segs, psi: int, loss_scale: float,
              arith: str = "f32") -> np.ndarray:
    """gbar as the binomial tree (tree.py) computes it after the same rank-local accumulation: float32
    partials ("f32") or float32 (hi, lo) pairs ("f32pair"), then hi + lo, then one multiply by
    fl32(1 / (n S)).  The tree's root holds the whole sum; the owner keeps its shard of it."""
    from .tree import Tree, combine
    loc = local_accumulate(grads, n, a, arith)
    tot = Tree(n).reduce(loc, combine(arith), elems=psi)
    p = (tot[0] + tot[1]).astype(np.float32) if arith == "f32pair" else np.asarray(tot, dtype=np.float32)
    inv = np.float32(1.0 / (float(n) * float(np.float32(loss_scale))))
    return (p * inv).astype(np.float32)


def micro_rs_gbar(grads: Sequence[np.ndarray], n: int, a: int, segs, psi: int, loss_scale: float,
                  arith: str = "f32") -> np.ndarray:
    """gbar as the per-micro-step reduce-scatter (the ZeRO-2 form) computes it: each micro-step's n gradients go
    round the simulated ring on their own (ring.py: the chunk of owner s starts at s+1), and every owner adds
    the arriving micro-step sum to its shard accumulator, A = ((p_0 + p_1) + ...) + p_{a-1}; float32 or float32
    (hi, lo) pairs ("f32pair": the accumulator adds (H, e) = TwoSum(A_H, p_H), A_L = (A_L + e) + p_L); then
    hi + lo and one multiply by fl32(1 / (n S))."""
    ring = Ring(n, segs, psi)
    acc = {}
    for k in range(a):
        xs = [bf16_bits_to_f32(grads[r * a + k]) for r in range(n)]
        loc = [(x, np.zeros_like(x)) for x in xs] if arith == "f32pair" else xs
        red = ring.reduce_scatter(loc, arith=arith, wire_bytes=4, phase="rs%d" % k)
        for s in range(n):
            p = red[s]
            if k == 0:
                acc[s] = p
            elif arith == "f32pair":
                H, e = two_sum32(acc[s][0], p[0])
                L = (acc[s][1] + e).astype(np.float32)
                L = (L + p[1]).astype(np.float32)
                acc[s] = (H, L)
            else:
                acc[s] = (acc[s] + p).astype(np.float32)
    inv = np.float32(1.0 / (float(n) * float(np.float32(loss_scale))))
    out = np.zeros(psi, dtype=np.float32)
    for s in range(n):
        v = acc[s]
        q = (v[0] + v[1]).astype(np.float32) if arith == "f32pair" else np.asarray(v, dtype=np.float32)
        ring._put(out, s, (q * inv).astype(np.float32))
    return out
