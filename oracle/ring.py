"""ORACLE -- test infrastructure.  A message-passing ring among n simulated ranks.

Each rank holds its own arrays; at every step each rank sends one message to
its right neighbour, and the receiver combines it with its own data.  The
simulator counts, per rank and per phase, the elements and bytes sent and
received and the number of steps, so the communication volumes the pages
state can be checked against messages actually passed:

* ring all-reduce = reduce-scatter + all-gather, about 2(N-1)/N x the
  gradient bytes per GPU, in 2(N-1) steps ("Data vs Tensor vs Pipeline
  Parallelism", section "Data parallelism: split the batch"; section "DP
  gradient sync at scale");
* a reduce-scatter leaves each rank the sum of its own shard; ZeRO-3 / FSDP
  gathers the weights twice (forward and backward) and so moves 1.5x the
  bytes of plain DP, while stages 1 and 2 move the same bytes (same page,
  "Sharded data parallelism"; "Distributed Training: Split along the Four
  Axes", ZeRO/FSDP paragraphs).

Reduction order: the chunk owned by rank s starts at rank s+1, which sends
its own contribution; every later rank adds its contribution to what it
received (received + own) and forwards it, so the chunk arrives at s after
n-1 hops as ((g_{s+1} + g_{s+2}) + ...) + g_s.

Arithmetic of a hop, selectable: "f64" (float64 adds), "f32" (float32 adds)
or "f32pair" (the partial travels as a float32 (hi, lo) pair; the receiver
adds its own (hi, lo) with Knuth's TwoSum error-free transformation, TAOCP
vol. 2 section 4.2.2, and accumulates the error terms in lo).  "f32chain":
the partial travels as a float32 (hi, lo) pair too, but a rank's contribution
is its list of micro-step gradients, not yet summed, and the receiver folds
them into the pair one at a time (hi, e) = TwoSum(hi, x), lo = lo + e; the
first rank of a chunk starts the pair at (its first micro-step, 0).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


def two_sum32(a: np.ndarray, b: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """s = fl(a+b) and the exact rounding error e, s + e = a + b, in float32 (Knuth)."""
    a = a.astype(np.float32, copy=False)
    b = b.astype(np.float32, copy=False)
    s = (a + b).astype(np.float32)
    z = (s - a).astype(np.float32)
    e = ((a - (s - z).astype(np.float32)).astype(np.float32) + (b - z).astype(np.float32)).astype(np.float32)
    return s, e


class Traffic:
    def __init__(self, n: int):
        self.n = n
        self.sent_elems = [0] * n
        self.recv_elems = [0] * n
        self.sent_bytes = [0] * n
        self.recv_bytes = [0] * n
        self.steps = 0

    def add(self, src: int, dst: int, elems: int, wire_bytes: int) -> None:
        self.sent_elems[src] += elems
        self.recv_elems[dst] += elems
        self.sent_bytes[src] += elems * wire_bytes
        self.recv_bytes[dst] += elems * wire_bytes


class Ring:
    """Ring collectives over a shard layout of (global_off, len, owner, local_off) segments."""

    def __init__(self, n: int, segs: Sequence[Tuple[int, int, int, int]], psi: int):
        self.n = n
        self.psi = psi
        # chunk of rank s: its segments in global order (concatenated)
        self.ranges: Dict[int, List[Tuple[int, int]]] = {s: [] for s in range(n)}
        for g, ln, o, _ in sorted(segs):
            if ln > 0:
                self.ranges[o].append((g, ln))
        self.traffic: Dict[str, Traffic] = {}
        self.drop = None      # (phase, step, src) of a message to lose, for failure tests

    def chunk_len(self, s: int) -> int:
        return sum(ln for _, ln in self.ranges[s])

    def _take(self, full: np.ndarray, s: int) -> np.ndarray:
        if not self.ranges[s]:
            return full[:0].copy()
        return np.concatenate([full[g:g + ln] for g, ln in self.ranges[s]])

    def _put(self, full: np.ndarray, s: int, vals: np.ndarray) -> None:
        c = 0
        for g, ln in self.ranges[s]:
            full[g:g + ln] = vals[c:c + ln]
            c += ln

    def _send(self, phase: str, step: int, src: int, elems: int, wire_bytes: int, payload):
        tr = self.traffic.setdefault(phase, Traffic(self.n))
        tr.add(src, (src + 1) % self.n, elems, wire_bytes)
        if self.drop is not None and self.drop == (phase, step, src):
            return None
        return payload

    def reduce_scatter(self, local: List, arith: str = "f32", wire_bytes: int = 4, phase: str = "rs") -> Dict[int, object]:
        """local[r]: rank r's full-length contribution (array, or (hi, lo) pair for f32pair).
        Returns {owner s: its reduced chunk} in the ring order described in the module docstring."""
        n = self.n
        tr = self.traffic.setdefault(phase, Traffic(n))

        def own(r: int, s: int):
            if arith == "f32chain":
                return [self._take(x, s) for x in local[r]]
            if arith == "f32pair":
                return (self._take(local[r][0], s), self._take(local[r][1], s))
            return self._take(local[r], s)

        def fold(pair, xs):
            H, L = pair
            for x in xs:
                H, e = two_sum32(H, x)
                L = (L + e).astype(np.float32)
            return (H, L)

        def start(mine):
            if arith != "f32chain":
                return mine
            first = mine[0].astype(np.float32)
            return fold((first, np.zeros_like(first)), mine[1:])

        def combine(recv, mine):
            if arith == "f32chain":
                return fold(recv, mine)
            if arith == "f64":
                return recv.astype(np.float64) + mine.astype(np.float64)
            if arith == "f32":
                return (recv.astype(np.float32) + mine.astype(np.float32)).astype(np.float32)
            H, e = two_sum32(recv[0], mine[0])
            L = (recv[1] + e).astype(np.float32)
            L = (L + mine[1]).astype(np.float32)
            return (H, L)

        if n == 1:
            return {0: start(own(0, 0))}
        inbox: List = [None] * n
        for t in range(n - 1):
            out = []
            for r in range(n):
                s = (r - 1 - t) % n
                payload = start(own(r, s)) if t == 0 else inbox[r][1]
                if t > 0 and inbox[r][0] != s:
                    raise RuntimeError("ring schedule broken")
                elems = self.chunk_len(s)
                out.append((r, s, self._send(phase, t, r, elems, wire_bytes, payload)))
            new = [None] * n
            for r, s, payload in out:
                d = (r + 1) % n
                if payload is None:
                    raise RuntimeError("message lost: phase %s step %d from rank %d" % (phase, t, r))
                new[d] = (s, combine(payload, own(d, s)))
            inbox = new
            tr.steps += 1
        res = {}
        for r in range(n):
            s, val = inbox[r]
            assert s == r
            res[r] = val
        return res

    def all_gather(self, shards: Dict[int, np.ndarray], wire_bytes: int, phase: str = "ag") -> List[np.ndarray]:
        """shards[s]: rank s's finished chunk.  Returns every rank's full-length array."""
        n = self.n
        tr = self.traffic.setdefault(phase, Traffic(n))
        dtype = shards[0].dtype if n > 0 else np.float32
        full = [np.zeros(self.psi, dtype=dtype) for _ in range(n)]
        for s in range(n):
            self._put(full[s], s, shards[s])
        have = [{s: shards[s]} for s in range(n)]
        for t in range(n - 1):
            out = []
            for r in range(n):
                s = (r - t) % n
                payload = have[r][s]
                out.append((r, s, self._send(phase, t, r, self.chunk_len(s), wire_bytes, payload)))
            for r, s, payload in out:
                d = (r + 1) % n
                if payload is None:
                    raise RuntimeError("message lost: phase %s step %d from rank %d" % (phase, t, r))
                have[d][s] = payload
                self._put(full[d], s, payload)
            tr.steps += 1
        return full


def step_traffic(n: int, segs, psi: int, stage: int, wire_grad: int, wire_param: int) -> Dict[str, Traffic]:
    """Run the collectives one training step of a ZeRO stage needs, on zero data, and return the counters.
    stage 0: all-reduce of the gradient (RS + AG of gradients); stage 1/2: RS of gradients + AG of the updated
    parameters; stage 3: RS of gradients + AG of parameters for forward + AG again for backward."""
    ring = Ring(n, segs, psi)
    zeros = [np.zeros(psi, dtype=np.float32) for _ in range(n)]
    red = ring.reduce_scatter(zeros, arith="f32", wire_bytes=wire_grad, phase="rs_grad")
    if stage == 0:
        ring.all_gather(red, wire_grad, phase="ag_grad")
    elif stage in (1, 2):
        ring.all_gather(red, wire_param, phase="ag_param")
    else:
        ring.all_gather(red, wire_param, phase="ag_param_fwd")
        ring.all_gather(red, wire_param, phase="ag_param_bwd")
    return ring.traffic
