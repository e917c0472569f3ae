"""Helpers of the -m gpu tests: set up one step on both sides from the same seeded inputs, compare."""
from __future__ import annotations

import struct
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
import synth
import zero_gradient_sync_gb300 as dp
from synth import device as sd
from zero_gradient_sync_gb300.buffers import StepBuffers

# fp32 master / m / v: |x - ref| <= ABS + REL |ref|; bf16 replicas within 1 ulp.
ABS, REL = 1e-9, 2e-6


def bf16_ord(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def state_bytes(t: int, beta1: float, beta2: float) -> bytes:
    """A host-built dp_step_state_t with t steps applied (beta powers as running products, like the device)."""
    b1t = b2t = 1.0
    for _ in range(t):
        b1t *= float(np.float32(beta1))
        b2t *= float(np.float32(beta2))
    return struct.pack("<iiiiQddQIIfI", t, 0, 0, 0, 0, b1t, b2t, 0, 0, 0, 0.0, 0)


@dataclass
class Case:
    wl: synth.Workload
    segs: list
    stage: int
    layout: dp.Layout
    grads: List[np.ndarray]
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    t: int


def make_case(wl: synth.Workload, stage: Optional[int] = None, segs=None, t: int = 0, m=None, v=None,
              master=None) -> Case:
    stage = wl.stage if stage is None else stage
    segs = synth.layout_of(wl) if segs is None else segs
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    master = synth.master_f32(wl) if master is None else master
    m = np.zeros(wl.psi, np.float32) if m is None else m
    v = np.zeros(wl.psi, np.float32) if v is None else v
    return Case(wl, segs, stage, dp.Layout(stage, wl.n, wl.psi, segs), grads, master, m, v, t)


def upload(c: Case, device="cuda", second_set: bool = False, micro_acc: bool = False) -> StepBuffers:
    b = StepBuffers(c.layout, c.wl.a, device, second_set=second_set, micro_acc=micro_acc)
    for q, g in enumerate(c.grads):
        b.grads[q].copy_(sd.bf16_from_bits(g))
    sd.place_full(b.master, c.master, c.segs, c.stage)
    sd.place_full(b.m, c.m, c.segs, c.stage)
    sd.place_full(b.v, c.v, c.segs, c.stage)
    for r in b.replicas:
        r.fill_(0)
    if c.t:
        b.state.copy_(torch.frombuffer(bytearray(state_bytes(c.t, c.wl.beta1, c.wl.beta2)), dtype=torch.uint8))
    return b


BAND = 256         # sentinel bytes on each side of a guarded buffer
SENTINEL = 0xA5


class Guarded:
    """Moves every device buffer of a StepBuffers into an allocation with BAND sentinel bytes before and after
    it (content kept), so that a kernel store outside any buffer lands in a band; check() finds it.  The
    interiors start BAND bytes into their allocation, so base pointers keep 256-byte alignment."""

    NAMES = ("grads", "replicas", "master", "m", "v", "gbar", "master1", "m1", "v1", "acc")

    def __init__(self, b: StepBuffers):
        self.outer = []
        for name in self.NAMES:
            setattr(b, name, [self._wrap(t) for t in getattr(b, name)])
        b.state = self._wrap(b.state)

    def _wrap(self, t: torch.Tensor) -> torch.Tensor:
        nb = t.numel() * t.element_size()
        o = torch.full((2 * BAND + nb,), SENTINEL, dtype=torch.uint8, device=t.device)
        inner = o[BAND:BAND + nb].view(t.dtype)
        inner.copy_(t)
        self.outer.append((o, nb))
        return inner

    def check(self, what: str = "") -> None:
        bands = torch.cat([x for o, nb in self.outer for x in (o[:BAND], o[BAND + nb:])])
        bad = int((bands != SENTINEL).sum().item())
        assert bad == 0, "%s: %d sentinel bytes overwritten outside the buffers" % (what, bad)


def run_oracle(c: Case, threads: int = 8):
    """The oracle's step on the same inputs: returns full-length master/m/v, replicas and the result dict."""
    wl = c.wl
    lens = [wl.psi] * wl.n if c.stage == 0 else synth.shard_lengths(c.segs, wl.n)
    M = [np.zeros(L, np.float32) for L in lens]
    Mm = [np.zeros(L, np.float32) for L in lens]
    Vv = [np.zeros(L, np.float32) for L in lens]
    for arrs, full in ((M, c.master), (Mm, c.m), (Vv, c.v)):
        if c.stage == 0:
            for x in arrs:
                x[:] = full
        else:
            for g, ln, o, lo in c.segs:
                arrs[o][lo:lo + ln] = full[g:g + ln]
    reps = [np.zeros(wl.psi, np.uint16) for _ in range(wl.n)]
    res = oracle.step(wl.psi, wl.n, wl.a, c.stage, c.segs, c.grads, M, Mm, Vv, reps, wl.lr, wl.beta1, wl.beta2,
                      wl.eps, wl.loss_scale, c.t, threads=threads)

    def full(arrs):
        if c.stage == 0:
            return arrs[0]
        out = np.zeros(wl.psi, np.float32)
        for g, ln, o, lo in c.segs:
            out[g:g + ln] = arrs[o][lo:lo + ln]
        return out

    return {"master": full(M), "m": full(Mm), "v": full(Vv), "replicas": reps, **res}


def gpu_result(c: Case, b: StepBuffers) -> dict:
    torch.cuda.synchronize()
    st = dp.read_state(b.state)
    out = {"master": sd.gather_full(b.master, c.segs, c.wl.psi, c.stage),
           "m": sd.gather_full(b.m, c.segs, c.wl.psi, c.stage),
           "v": sd.gather_full(b.v, c.segs, c.wl.psi, c.stage),
           "replicas": [sd.bits_of_bf16(r) for r in b.replicas],
           "found": st["found_inf"], "nonfinite": st["nonfinite"], "t": st["t"], "error": st["error"]}
    if c.stage == 0:
        out["all_master"] = [x.detach().cpu().numpy() for x in b.master]
    return out


def assert_close_f32(x: np.ndarray, ref: np.ndarray, name: str, scale: float = 1.0) -> None:
    d = np.abs(x.astype(np.float64) - ref.astype(np.float64))
    tol = scale * (ABS + REL * np.abs(ref.astype(np.float64)))
    bad = np.nonzero(~(d <= tol))[0]
    assert bad.size == 0, "%s: %d elements out of tolerance, first %s: gpu %r ref %r" % (
        name, bad.size, bad[:5], x[bad[:5]], ref[bad[:5]])


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_replicas(reps: List[np.ndarray], ref: List[np.ndarray], ulps: int = 1) -> None:
    """Within 1 bf16 ulp -- or, where the master's absolute tolerance term dominates (|theta| below ~5e-4), within
    that tolerance plus one bf16 ulp: a replica is bf16_rne of the master, so it can differ by no more than the
    master it rounds."""
    for r, (x, y) in enumerate(zip(reps, ref)):
        d = np.abs(bf16_ord(x) - bf16_ord(y))
        far = np.nonzero(d > ulps)[0]
        if far.size:
            xv, yv = bf16_value(x[far]), bf16_value(y[far])
            ulp = np.abs(bf16_value(y[far] ^ 1) - yv)
            ok = np.abs(xv - yv) <= ABS + REL * np.abs(yv) + ulp
            far = far[~ok]
        assert far.size == 0, "replica %d: %d elements beyond %d bf16 ulp, first %s" % (r, far.size, ulps, far[:5])
    for x in reps[1:]:
        assert np.array_equal(x, reps[0]), "replicas differ from each other"


def assert_matches_oracle(g: dict, o: dict, scale: float = 1.0) -> None:
    assert g["error"] == 0
    assert g["found"] == o["found"]
    assert g["nonfinite"] == o["nonfinite"]
    assert g["t"] == o["t"]
    assert_close_f32(g["master"], o["master"], "master", scale)
    assert_close_f32(g["m"], o["m"], "m", scale)
    assert_close_f32(g["v"], o["v"], "v", scale)
    assert_replicas(g["replicas"], o["replicas"])


def snapshot(b: StepBuffers) -> List[bytes]:
    torch.cuda.synchronize()
    ts = b.master + b.m + b.v + b.replicas
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in ts]


# ------------------------------------------------------------------ full-size runs checked on sampled elements

def sample_indices(wl, segs, count, seed):
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, wl.psi, count).tolist())
    for g, ln, o, lo in segs:
        if ln:
            idx.update([g, g + ln - 1, min(g + 1, g + ln - 1), max(g, g + ln - 2)])
    idx.update(range(max(0, wl.psi - 9), wl.psi))
    return np.array(sorted(idx), dtype=np.int64)


def owners_of(segs, idx):
    """Owner rank and local index of each global index."""
    goff = np.array([s[0] for s in segs if s[1]], dtype=np.int64)
    own = np.array([s[2] for s in segs if s[1]], dtype=np.int64)
    loff = np.array([s[3] for s in segs if s[1]], dtype=np.int64)
    k = np.searchsorted(goff, idx, side="right") - 1
    return own[k], loff[k] + (idx - goff[k])


def gather_state(arrs, segs, idx, stage):
    """Values of per-rank state arrays at global indices (rank 0's copy for plain data parallelism)."""
    if stage == 0:
        return arrs[0][torch.from_numpy(idx).to(arrs[0].device)].cpu().numpy()
    own, loc = owners_of(segs, idx)
    out = np.zeros(idx.size, np.float32)
    for r in np.unique(own):
        sel = np.nonzero(own == r)[0]
        t = torch.from_numpy(loc[sel]).to(arrs[int(r)].device)
        out[sel] = arrs[int(r)][t].cpu().numpy()
    return out


def oracle_at(wl, idx, t0=0, m=None, v=None, master=None, prior=False):
    """The oracle's step on the sampled elements only (the step is elementwise; found is per element)."""
    ns = idx.size
    contiguous = ns > 0 and idx[-1] - idx[0] == ns - 1
    if contiguous:   # a chunk of the space: the generator's contiguous path gives the same values, faster
        grads = [synth.grads_bf16(wl, r, k, int(idx[0]), ns, prior=prior) for r in range(wl.n) for k in range(wl.a)]
    else:
        grads = [synth.grads_bf16_at(wl, r, k, idx, prior=prior) for r in range(wl.n) for k in range(wl.a)]
    if master is None:
        master = synth.master_f32(wl, int(idx[0]), ns) if contiguous else synth.master_f32_at(wl, idx)
    M = [master.copy()]
    Mm = [m.copy() if m is not None else np.zeros(ns, np.float32)]
    Vv = [v.copy() if v is not None else np.zeros(ns, np.float32)]
    M += [np.zeros(0, np.float32)] * (wl.n - 1)
    Mm += [np.zeros(0, np.float32)] * (wl.n - 1)
    Vv += [np.zeros(0, np.float32)] * (wl.n - 1)
    reps = [np.zeros(ns, np.uint16) for _ in range(wl.n)]
    res = oracle.step(ns, wl.n, wl.a, 1, [(0, ns, 0, 0)], grads, M, Mm, Vv, reps, wl.lr, wl.beta1, wl.beta2,
                      wl.eps, wl.loss_scale, t0, threads=16)
    return {"master": M[0], "m": Mm[0], "v": Vv[0], "replicas": reps, **res}
