"""Upload seeded synthetic inputs into device tensors, chunk by chunk through pinned host memory.

Only input placement lives here: the values come from the counter-based generator in synth/__init__.py,
so the oracle side can regenerate any element on the host.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from . import Workload, grads_bf16, master_f32

CHUNK = 1 << 25   # elements per host chunk


class _Pinned:
    def __init__(self, nbytes: int):
        self.buf = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)

    def view(self, dtype: np.dtype, count: int) -> np.ndarray:
        nb = count * np.dtype(dtype).itemsize
        return self.buf[:nb].numpy().view(dtype)


def bf16_from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bits_of_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def fill_grads(grads: Sequence[torch.Tensor], wl: Workload, prior: bool = False, chunk: int = CHUNK) -> None:
    """grads[r*a + k][i] = the generator's bf16 value of rank r, micro-step k, element i."""
    pin = _Pinned(2 * min(chunk, max(1, wl.psi)))
    for r in range(wl.n):
        for k in range(wl.a):
            dst = grads[r * wl.a + k]
            for s in range(0, wl.psi, chunk):
                c = min(chunk, wl.psi - s)
                h = pin.view(np.uint16, c)
                grads_bf16(wl, r, k, s, c, out=h, prior=prior)
                dst[s:s + c].copy_(bf16_from_bits(h), non_blocking=False)


def fill_master(master: Sequence[torch.Tensor], wl: Workload, segs, stage: int, chunk: int = CHUNK) -> None:
    """Master weights: rank s's shard holds its segments' values (stage 1-3); every rank holds all (stage 0)."""
    pin = _Pinned(4 * min(chunk, max(1, wl.psi)))
    if stage == 0:
        for s in range(0, wl.psi, chunk):
            c = min(chunk, wl.psi - s)
            h = pin.view(np.float32, c)
            master_f32(wl, s, c, out=h)
            ht = torch.from_numpy(h)
            for r in range(wl.n):
                master[r][s:s + c].copy_(ht)
        return
    for g, ln, o, lo in segs:
        for s in range(0, ln, chunk):
            c = min(chunk, ln - s)
            h = pin.view(np.float32, c)
            master_f32(wl, g + s, c, out=h)
            master[o][lo + s:lo + s + c].copy_(torch.from_numpy(h))


def place_full(dst: Sequence[torch.Tensor], full: np.ndarray, segs, stage: int) -> None:
    """Put a full-length fp32 host array into per-rank state arrays (shards, or full copies for stage 0)."""
    if stage == 0:
        t = torch.from_numpy(np.ascontiguousarray(full, dtype=np.float32))
        for d in dst:
            d.copy_(t)
        return
    for g, ln, o, lo in segs:
        if ln:
            dst[o][lo:lo + ln].copy_(torch.from_numpy(np.ascontiguousarray(full[g:g + ln], dtype=np.float32)))


def gather_full(src: Sequence[torch.Tensor], segs, psi: int, stage: int, rank: int = 0) -> np.ndarray:
    """Full-length host array from per-rank state arrays."""
    if stage == 0:
        return src[rank].detach().cpu().numpy().copy()
    out = np.zeros(psi, dtype=np.float32)
    host = [t.detach().cpu().numpy() for t in src]
    for g, ln, o, lo in segs:
        out[g:g + ln] = host[o][lo:lo + ln]
    return out
