"""ORACLE -- test infrastructure.  A message-passing binomial tree among n simulated ranks.

The second reduction order: NCCL offers tree algorithms beside the ring
because a ring all-reduce takes 2(N-1) steps while a tree takes about
2 log2(N) ("Data vs Tensor vs Pipeline Parallelism", section "DP gradient
sync at scale").  The pages name the algorithm only; the reading used here is
the textbook binomial tree rooted at rank 0:

* reduce: at step l = 0, 1, ... every rank r with r mod 2^(l+1) == 0 receives
  the partial sum of rank r + 2^l (if that rank exists) and adds it to its
  own, own + received -- so the lower-index block is the left operand, and a
  block with no partner waits a level unchanged;
* broadcast: the same steps in reverse carry the total back down;
* every element uses the same tree, whoever owns its shard; the owner keeps
  its shard of the all-reduced result.

Arithmetic of a combine: "f64", "f32", or "f32pair" (hi, lo) with Knuth's
TwoSum on the hi parts and the errors added as (lo_left + e) + lo_right.
Traffic counters count elements per rank and steps per phase, like the ring's.
"""
from __future__ import annotations

from typing import Callable, List

import numpy as np

from .ring import Traffic, two_sum32


def combine(arith: str) -> Callable:
    def add(left, right):
        if arith == "f64":
            return left.astype(np.float64) + right.astype(np.float64)
        if arith == "f32":
            return (left.astype(np.float32) + right.astype(np.float32)).astype(np.float32)
        H, e = two_sum32(left[0], right[0])
        L = (left[1] + e).astype(np.float32)
        L = (L + right[1]).astype(np.float32)
        return (H, L)
    return add


class Tree:
    def __init__(self, n: int):
        self.n = n
        self.traffic = {}

    def levels(self) -> int:
        lv = 0
        while (1 << lv) < self.n:
            lv += 1
        return lv

    def reduce(self, local: List, add: Callable, elems: int, wire_bytes: int = 4, phase: str = "reduce"):
        """local[r]: rank r's contribution.  Returns rank 0's total after the binomial reduce."""
        n = self.n
        tr = self.traffic.setdefault(phase, Traffic(n))
        val = list(local)
        for lv in range(self.levels()):
            step = 1 << lv
            for r in range(0, n, 2 * step):
                src = r + step
                if src < n:
                    tr.add(src, r, elems, wire_bytes)
                    val[r] = add(val[r], val[src])
                    val[src] = None      # sent: the sender holds nothing more of this sum
            tr.steps += 1
        return val[0]

    def broadcast(self, total, elems: int, wire_bytes: int = 4, phase: str = "broadcast") -> List:
        n = self.n
        tr = self.traffic.setdefault(phase, Traffic(n))
        val = [None] * n
        val[0] = total
        for lv in reversed(range(self.levels())):
            step = 1 << lv
            for r in range(0, n, 2 * step):
                dst = r + step
                if dst < n:
                    tr.add(r, dst, elems, wire_bytes)
                    val[dst] = val[r]
            tr.steps += 1
        return val


def tree_expression(n: int) -> str:
    """The parenthesised sum the tree forms over symbols g0..g{n-1} (for pins against the definition)."""
    t = Tree(n)
    return t.reduce(["g%d" % r for r in range(n)], lambda x, y: "(%s+%s)" % (x, y), elems=0)
