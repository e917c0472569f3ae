"""Seeded synthetic workloads for the fused data-parallel step.

This module is shared by the oracle side (tests, the CPU baseline) and the
GPU side (tests, bench).  It holds only input generation: workload shapes,
shard layouts and counter-based random values.  It computes nothing of the
step (no sums, no optimizer, no rounding of results), so neither side
borrows arithmetic from the other through it.

Workload shapes follow the parameter lists of the distributed-training
pages' workloads (GPT-2-small-like list, a 1.3B-parameter list, the first 16
decoder layers of a Llama-7B-like model) as flat parameter spaces; values are
N(0, sigma) samples rounded to bf16 (gradients) or fp32 (master weights).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field, replace
from typing import List, Sequence, Tuple

import numpy as np

from . import build as _build

# Stream roles (the key's second word carries role, rank and micro-step).
ROLE_GRAD = 1
ROLE_MASTER = 2
ROLE_LAYOUT = 6
ROLE_INJECT = 7

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, u64, u32, dbl, vp, ci = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double,
                                      ctypes.c_void_p, ctypes.c_int)
        L.synth_philox4x64_10.argtypes = [vp, vp, vp]
        L.synth_philox4x64_10.restype = None
        L.synth_bf16_normal.argtypes = [u64, u32, u32, u32, i64, i64, dbl, dbl, dbl, vp, ci]
        L.synth_bf16_normal_at.argtypes = [u64, u32, u32, u32, vp, i64, dbl, dbl, dbl, vp, ci]
        L.synth_f32_normal.argtypes = [u64, u32, u32, u32, i64, i64, dbl, vp, ci]
        L.synth_f32_normal_at.argtypes = [u64, u32, u32, u32, vp, i64, dbl, vp, ci]
        L.synth_f64_normal.argtypes = [u64, u32, u32, u32, i64, i64, vp, ci]
        L.synth_u64.argtypes = [u64, u32, u32, u32, i64, i64, vp]
        L.synth_f64_to_bf16.argtypes = [dbl]
        L.synth_f64_to_bf16.restype = ctypes.c_uint16
        for f in (L.synth_bf16_normal, L.synth_bf16_normal_at, L.synth_f32_normal, L.synth_f32_normal_at,
                  L.synth_f64_normal, L.synth_u64):
            f.restype = None
        _LIB = L
    return _LIB


def threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# --------------------------------------------------------------------------------------------
# Raw streams
# --------------------------------------------------------------------------------------------

def philox4x64_10(ctr: Sequence[int], key: Sequence[int]) -> List[int]:
    c = np.asarray(ctr, dtype=np.uint64)
    k = np.asarray(key, dtype=np.uint64)
    o = np.zeros(4, dtype=np.uint64)
    lib().synth_philox4x64_10(_ptr(c), _ptr(k), _ptr(o))
    return [int(x) for x in o]


def u64_stream(seed: int, role: int, rank: int, micro: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    lib().synth_u64(seed, role, rank, micro, start, count, _ptr(out))
    return out


def normal_f64(seed: int, role: int, rank: int, micro: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    lib().synth_f64_normal(seed, role, rank, micro, start, count, _ptr(out), threads())
    return out


def f64_to_bf16_bits(x: float) -> int:
    return int(lib().synth_f64_to_bf16(float(x)))


# --------------------------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------------------------

def gpt2_small_shapes() -> List[Tuple[int, ...]]:
    """Embedding 50257x768, then 12 x {768x2304, 768x768, 768x3072, 3072x768, 4 LayerNorm vectors of 768}."""
    shapes: List[Tuple[int, ...]] = [(50257, 768)]
    for _ in range(12):
        shapes += [(768, 2304), (768, 768), (768, 3072), (3072, 768), (768,), (768,), (768,), (768,)]
    return shapes


def gpt_1p3b_shapes() -> List[Tuple[int, ...]]:
    """24 layers, hidden 2048, FFN 8192, vocab 50257; the GPT-2 pattern at that width."""
    h, f = 2048, 8192
    shapes: List[Tuple[int, ...]] = [(50257, h)]
    for _ in range(24):
        shapes += [(h, 3 * h), (h, h), (h, f), (f, h), (h,), (h,), (h,), (h,)]
    return shapes


def llama7b_16l_shapes() -> List[Tuple[int, ...]]:
    """First 16 decoder layers: 4 attention 4096x4096, 3 SwiGLU 4096x11008, 2 RMSNorm vectors; no embedding."""
    h, f = 4096, 11008
    shapes: List[Tuple[int, ...]] = []
    for _ in range(16):
        shapes += [(h, h)] * 4 + [(h, f), (h, f), (f, h)] + [(h,), (h,)]
    return shapes


def numel(shapes: Sequence[Tuple[int, ...]]) -> int:
    total = 0
    for s in shapes:
        p = 1
        for d in s:
            p *= d
        total += p
    return total


def flatten_offsets(shapes: Sequence[Tuple[int, ...]]) -> List[int]:
    """Start offset of every tensor in the flat parameter space (list order, no padding)."""
    offs, cur = [], 0
    for s in shapes:
        offs.append(cur)
        p = 1
        for d in s:
            p *= d
        cur += p
    return offs


@dataclass(frozen=True)
class Workload:
    name: str
    psi: int
    n: int
    a: int
    stage: int
    layout: str = "even"          # even | buckets | ragged | random
    bucket: int = 0
    misalign: int = 0
    nseg: int = 0                 # random layouts: number of segments
    sigma_g: float = 1e-3
    tail_p: float = 0.0
    tail_mult: float = 1.0
    sigma_master: float = 0.02
    loss_scale: float = 1.0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    seed: int = 0
    warm: bool = False
    description: str = ""

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def grad_bytes(self) -> int:
        return 2 * self.n * self.a * self.psi


WORKLOADS = {
    "tiny": Workload(
        name="tiny", psi=1 << 20, n=2, a=1, stage=1, layout="even", sigma_g=1e-3, loss_scale=1.0, seed=0,
        description="single flat tensor of 2^20 params, n=2, a=1, ZeRO-1 even shards"),
    "gpt2_small": Workload(
        name="gpt2_small", psi=numel(gpt2_small_shapes()), n=8, a=4, stage=1, layout="even", sigma_g=1e-3,
        loss_scale=float(1 << 16), seed=1,
        description="GPT-2-small param list (123,568,896 params), n=8, a=4, ZeRO-1 even shards, S=2^16"),
    "gpt_1p3b": Workload(
        name="gpt_1p3b", psi=numel(gpt_1p3b_shapes()), n=8, a=1, stage=3, layout="buckets", bucket=25_000_000,
        misalign=3, sigma_g=1e-4, loss_scale=1.0, seed=2, warm=True,
        description="1.3B param list (1,311,082,496 params), n=8, a=1, ZeRO-3 25M-element buckets with "
                    "shard boundaries moved +3 elements, warm m/v"),
    "llama7b_16l": Workload(
        name="llama7b_16l", psi=numel(llama7b_16l_shapes()), n=4, a=2, stage=2, layout="even", sigma_g=1e-4,
        tail_p=0.01, tail_mult=100.0, loss_scale=1.0, seed=3,
        description="Llama-7B-shaped first 16 decoder layers (3,238,133,760 params), n=4, a=2, ZeRO-2 even, "
                    "1% heavy-tail x100 outliers"),
}

SWEEP_PSI = [1 << 20, (1 << 20) + 3, 1 << 24, 10 ** 8, (1 << 28) + 5, 10 ** 9]
SWEEP_N = [2, 4, 8]
SWEEP_A = [1, 8]
SWEEP_S = [float(1 << 8), float(1 << 12), float(1 << 16), float(1 << 20), float(1 << 24)]


def sweep_cases() -> List[Workload]:
    """The flat-buffer sweep: every (psi, n, a, even|ragged), loss scales cycled over the cases."""
    out = []
    i = 0
    for psi in SWEEP_PSI:
        for n in SWEEP_N:
            for a in SWEEP_A:
                for lay in ("even", "ragged"):
                    out.append(Workload(
                        name="sweep_%d_n%d_a%d_%s" % (psi, n, a, lay), psi=psi, n=n, a=a, stage=1 + (i % 3),
                        layout=lay, sigma_g=1e-3, loss_scale=SWEEP_S[i % len(SWEEP_S)], seed=4 + i,
                        description="flat sweep case"))
                    i += 1
    return out


# --------------------------------------------------------------------------------------------
# Layouts: lists of (global_off, len, owner, local_off)
# --------------------------------------------------------------------------------------------

Segment = Tuple[int, int, int, int]


def layout_even(psi: int, n: int) -> List[Segment]:
    """Contiguous shards in rank order; the first psi mod n shards are one element longer."""
    base, extra = divmod(psi, n)
    segs, g = [], 0
    for s in range(n):
        ln = base + (1 if s < extra else 0)
        segs.append((g, ln, s, 0))
        g += ln
    return segs


def layout_buckets(psi: int, n: int, bucket: int, misalign: int) -> List[Segment]:
    """Per-bucket shards: the flat space is cut into buckets, each bucket split n ways with every
    interior boundary moved by +misalign elements; each rank's pieces are concatenated locally."""
    segs: List[Segment] = []
    local = [0] * n
    b0 = 0
    while b0 < psi:
        L = min(bucket, psi - b0)
        base, extra = divmod(L, n)
        cuts = [k * base + min(k, extra) for k in range(n + 1)]
        for k in range(1, n):
            cuts[k] = min(L, cuts[k] + misalign)
        for k in range(1, n + 1):
            cuts[k] = max(cuts[k], cuts[k - 1])
        for s in range(n):
            ln = cuts[s + 1] - cuts[s]
            segs.append((b0 + cuts[s], ln, s, local[s]))
            local[s] += ln
        b0 += L
    return segs


def layout_ragged(psi: int, n: int, seed: int) -> List[Segment]:
    """One contiguous shard per rank with seeded random sizes; empty shards are possible."""
    if n == 1:
        return [(0, psi, 0, 0)]
    w = u64_stream(seed, ROLE_LAYOUT, n, 0, 0, n - 1)
    cuts = sorted(int(x % np.uint64(psi + 1)) for x in w)
    bounds = [0] + cuts + [psi]
    return [(bounds[s], bounds[s + 1] - bounds[s], s, 0) for s in range(n)]


def layout_random(psi: int, n: int, nseg: int, seed: int) -> List[Segment]:
    """nseg segments with seeded random cut points and random owners (not in rank order);
    every owner's local space is the concatenation of its segments in global order."""
    w = u64_stream(seed, ROLE_LAYOUT, n, 1, 0, 2 * nseg)
    cuts = sorted(int(x % np.uint64(psi + 1)) for x in w[: nseg - 1])
    bounds = [0] + cuts + [psi]
    local = [0] * n
    segs = []
    for k in range(nseg):
        owner = int(w[nseg + k] % np.uint64(n))
        ln = bounds[k + 1] - bounds[k]
        segs.append((bounds[k], ln, owner, local[owner]))
        local[owner] += ln
    return segs


def layout_of(wl: Workload) -> List[Segment]:
    if wl.layout == "even":
        return layout_even(wl.psi, wl.n)
    if wl.layout == "buckets":
        return layout_buckets(wl.psi, wl.n, wl.bucket, wl.misalign)
    if wl.layout == "ragged":
        return layout_ragged(wl.psi, wl.n, wl.seed)
    if wl.layout == "random":
        return layout_random(wl.psi, wl.n, wl.nseg, wl.seed)
    raise ValueError("unknown layout " + wl.layout)


def shard_lengths(segs: Sequence[Segment], n: int) -> List[int]:
    """Local length of every rank's shard (end of its furthest segment)."""
    out = [0] * n
    for g, ln, o, l in segs:
        if ln > 0:
            out[o] = max(out[o], l + ln)
    return out


# --------------------------------------------------------------------------------------------
# Values
# --------------------------------------------------------------------------------------------

def grad_seed(wl: Workload, prior: bool = False) -> int:
    return wl.seed + (1000 if prior else 0)


def grads_bf16(wl: Workload, r: int, k: int, start: int = 0, count: int = -1, out: np.ndarray = None,
               prior: bool = False) -> np.ndarray:
    """bf16 bit patterns of micro-step k's gradient on rank r, elements [start, start+count)."""
    if count < 0:
        count = wl.psi - start
    if out is None:
        out = np.empty(count, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size >= count and out.flags.c_contiguous
    lib().synth_bf16_normal(grad_seed(wl, prior), ROLE_GRAD, r, k, start, count, wl.sigma_g, wl.tail_p,
                            wl.tail_mult, _ptr(out), threads())
    return out


def grads_bf16_at(wl: Workload, r: int, k: int, idx: np.ndarray, prior: bool = False) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.size, dtype=np.uint16)
    lib().synth_bf16_normal_at(grad_seed(wl, prior), ROLE_GRAD, r, k, _ptr(idx), idx.size, wl.sigma_g, wl.tail_p,
                               wl.tail_mult, _ptr(out), threads())
    return out


def master_f32(wl: Workload, start: int = 0, count: int = -1, out: np.ndarray = None) -> np.ndarray:
    """fp32 master weights (identical on every replica), elements [start, start+count) of the flat space."""
    if count < 0:
        count = wl.psi - start
    if out is None:
        out = np.empty(count, dtype=np.float32)
    assert out.dtype == np.float32 and out.size >= count and out.flags.c_contiguous
    lib().synth_f32_normal(wl.seed, ROLE_MASTER, 0, 0, start, count, wl.sigma_master, _ptr(out), threads())
    return out


def master_f32_at(wl: Workload, idx: np.ndarray) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.size, dtype=np.float32)
    lib().synth_f32_normal_at(wl.seed, ROLE_MASTER, 0, 0, _ptr(idx), idx.size, wl.sigma_master, _ptr(out),
                              threads())
    return out


def inject_site(wl: Workload, case: int) -> Tuple[int, int, int, int]:
    """A seeded (rank, micro-step, element, kind) for one non-finite injection; kind 0:+inf 1:-inf 2:NaN."""
    w = u64_stream(wl.seed, ROLE_INJECT, case, 0, 0, 4)
    return (int(w[0] % np.uint64(wl.n)), int(w[1] % np.uint64(wl.a)), int(w[2] % np.uint64(max(1, wl.psi))),
            int(w[3] % np.uint64(3)))


BF16_POS_INF = 0x7F80
BF16_NEG_INF = 0xFF80
BF16_NAN = 0x7FC0
