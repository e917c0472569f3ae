"""ORACLE -- test infrastructure, not part of the product.

What a sharded checkpoint holds and what a reshard must produce, written out
plainly ("Distributed Training: Split along the Four Axes", checkpoint
paragraphs: ZeRO/FSDP state is stored by rank as shards and reloads into a
different world size; the write goes through temporary artifacts and an
atomic manifest).

* to_full / from_full: the placement rule of a layout.  Element i of the flat
  parameter space lives in rank `owner`'s arrays at local_off + (i -
  global_off) of the segment that holds i (stages 1-3), or at i in every
  rank's full-length copy (stage 0).  A reshard is from_full(new, to_full(old)),
  so a loaded state must equal it bit for bit.
* fnv1a64_words: the checksum the manifest records -- FNV-1a 64 (Fowler, Noll,
  Vo) over little-endian 64-bit words, the last 0..7 bytes one at a time.  On
  inputs shorter than 8 bytes it is the byte-wise FNV-1a 64 of the published
  test vectors.
* read_checkpoint: an independent parser of the on-disk format, so a test can
  check what a save wrote without the library's loader.

Plain Python and numpy; shares nothing with the library.
"""
from __future__ import annotations

import os
import struct
from typing import Dict, List, Sequence, Tuple

import numpy as np

FNV_BASIS = 14695981039346656037
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1
SHARD_MAGIC = 0x48535044
LAYOUT_MAGIC = 0x4C535044


def shard_lengths(segs: Sequence[Tuple[int, int, int, int]], n: int) -> List[int]:
    lens = [0] * n
    for g, ln, o, lo in segs:
        if ln:
            lens[o] = max(lens[o], lo + ln)
    return lens


def to_full(arrays: Sequence[np.ndarray], segs, psi: int, stage: int, rank: int = 0) -> np.ndarray:
    """The full-length array that per-rank state arrays hold (stage 0: rank `rank`'s copy)."""
    if stage == 0:
        return np.array(arrays[rank][:psi], dtype=np.float32)
    out = np.zeros(psi, dtype=np.float32)
    for g, ln, o, lo in segs:
        out[g:g + ln] = arrays[o][lo:lo + ln]
    return out


def from_full(full: np.ndarray, segs, n: int, stage: int) -> List[np.ndarray]:
    """Per-rank state arrays of a layout holding `full` (holes of a local space are zero)."""
    psi = full.shape[0]
    if stage == 0:
        return [full.astype(np.float32, copy=True) for _ in range(n)]
    out = [np.zeros(L, dtype=np.float32) for L in shard_lengths(segs, n)]
    for g, ln, o, lo in segs:
        out[o][lo:lo + ln] = full[g:g + ln]
    assert sum(ln for _, ln, _, _ in segs) == psi
    return out


def fnv1a64_words(data: bytes) -> int:
    h = FNV_BASIS
    nw = len(data) // 8
    for w in struct.unpack_from("<%dQ" % nw, data):
        h = ((h ^ w) * FNV_PRIME) & MASK64
    for b in data[8 * nw:]:
        h = ((h ^ b) * FNV_PRIME) & MASK64
    return h


def read_manifest(d: str) -> Dict[str, Tuple[int, int]]:
    with open(os.path.join(d, "MANIFEST")) as f:
        lines = f.read().splitlines()
    assert lines[0] == "dpstep-checkpoint 1", lines[0]
    out = {}
    for ln in lines[1:]:
        kind, name, size, fnv = ln.split()
        assert kind == "file"
        out[name] = (int(size), int(fnv, 16))
    return out


def read_checkpoint(root: str, tag: str = None) -> dict:
    """Parses a checkpoint directory: the layout, the full-length master/m/v, the raw state and user bytes."""
    if tag is None:
        with open(os.path.join(root, "LATEST")) as f:
            tag = f.read().strip()
    d = os.path.join(root, tag)
    with open(os.path.join(d, "layout.bin"), "rb") as f:
        raw = f.read()
    magic, ver, stage, n = struct.unpack_from("<4I", raw, 0)
    psi, nseg = struct.unpack_from("<qq", raw, 16)
    assert magic == LAYOUT_MAGIC and ver == 1
    segs = []
    for k in range(nseg):
        g, ln, o, _res, lo = struct.unpack_from("<qqiiq", raw, 32 + 32 * k)
        segs.append((g, ln, o, lo))
    lens = shard_lengths(segs, n)
    per = {"master": [], "m": [], "v": []}
    for r in range(n):
        with open(os.path.join(d, "shard_%d.bin" % r), "rb") as f:
            b = f.read()
        mg, v1, rr, _z = struct.unpack_from("<4I", b, 0)
        (L,) = struct.unpack_from("<q", b, 16)
        assert (mg, v1, rr, L) == (SHARD_MAGIC, 1, r, lens[r])
        assert len(b) == 24 + 12 * L
        arr = np.frombuffer(b, dtype=np.float32, offset=24)
        for k, name in enumerate(("master", "m", "v")):
            per[name].append(arr[k * L:(k + 1) * L])
    full = {}
    for name, arrs in per.items():
        out = np.zeros(psi, dtype=np.float32)
        for g, ln, o, lo in segs:
            out[g:g + ln] = arrs[o][lo:lo + ln]
        full[name] = out
    with open(os.path.join(d, "state.bin"), "rb") as f:
        state = f.read()
    with open(os.path.join(d, "user.bin"), "rb") as f:
        user = f.read()
    return {"tag": tag, "stage": stage, "n": n, "psi": psi, "segs": segs, "state": state, "user": user,
            "manifest": read_manifest(d), **full}
