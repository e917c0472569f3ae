"""Sharded checkpoints and resharding (host buffers: the library's real save/load code, no GPU).

A reshard is a permutation, so every check is bit for bit: what a save wrote is parsed by the oracle's own
reader, a load into any other layout must equal the oracle's placement rule applied to the saved full
arrays, and the manifest's checksums are pinned to the published FNV-1a 64 test vectors.
"""
import ctypes
import importlib.util
import os
import struct
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import synth
from oracle import checkpoint as ock

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _built():
    spec = importlib.util.spec_from_file_location(
        "_dpstep_build", os.path.join(ROOT, "zero_gradient_sync_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import zero_gradient_sync_gb300 as z
    return z


dp = _built()


def full_bits(psi: int, seed: int) -> np.ndarray:
    """fp32 arrays of arbitrary bit patterns: NaN payloads, infinities, subnormals and -0 included."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=psi, dtype=np.uint64).astype(np.uint32)
    if psi >= 6:
        bits[:6] = [0x7FC00001, 0xFF800000, 0x00000001, 0x80000000, 0x7F800000, 0xFFBFFFFF]
    return bits.view(np.float32)


def state_blob(t=7, found=1, err=0, good=3, nonfinite=5, b1t=0.9 ** 7, b2t=0.999 ** 7, scale=1024.0, cur=1):
    return bytearray(struct.pack("<iiiiQddQIIfI", t, found, err, good, nonfinite, b1t, b2t, 9, 1, 2, scale, cur))


def decode_state(raw: bytes) -> tuple:
    return struct.unpack("<iiiiQddQIIfI", bytes(raw))


def arrays_for(layout, fulls, sentinel=None):
    """Host master/m/v lists of a layout holding the given full arrays (or filled with a sentinel)."""
    out = []
    for f in fulls:
        if sentinel is None:
            out.append(ock.from_full(f, layout.segs, layout.n, layout.stage))
        else:
            out.append([np.full(L, sentinel, np.uint32).view(np.float32) for L in layout.state_lens()])
    return out


def bits(x):
    return np.asarray(x).view(np.uint32)


def layouts(psi: int):
    """(name, Layout) cases: even, ragged with empty shards, per-bucket misaligned, random owners, holes
    in the local spaces, plain data parallelism, one rank, sixteen ranks."""
    holes = [(g, ln, o, lo + 5 * k) for k, (g, ln, o, lo) in enumerate(synth.layout_random(psi, 3, 9, 5))]
    return [
        ("even4", dp.Layout(1, 4, psi, synth.layout_even(psi, 4))),
        ("ragged5", dp.Layout(2, 5, psi, synth.layout_ragged(psi, 5, 11))),
        ("buckets8", dp.Layout(3, 8, psi, synth.layout_buckets(psi, 8, 7_001, 3))),
        ("random6", dp.Layout(1, 6, psi, synth.layout_random(psi, 6, 23, 4))),
        ("holes3", dp.Layout(2, 3, psi, holes)),
        ("dp2", dp.Layout(0, 2, psi, synth.layout_even(psi, 2))),
        ("one", dp.Layout(1, 1, psi, [(0, psi, 0, 0)])),
        ("sixteen", dp.Layout(1, 16, psi, synth.layout_ragged(psi, 16, 3))),
    ]


PSI = 30_011


@pytest.fixture
def saved(tmp_path):
    """A checkpoint of a ragged n=4 ZeRO-1 layout with known full arrays, state and user bytes."""
    lay = dp.Layout(1, 4, PSI, synth.layout_ragged(PSI, 4, 7))
    fulls = [full_bits(PSI, s) for s in (1, 2, 3)]
    M, Mm, V = arrays_for(lay, fulls)
    st = state_blob()
    root = str(tmp_path / "ck")
    dp.dp_checkpoint_save(root, "step7", lay, M, Mm, V, st, user_meta=b"cursor=4096\x00rng=\xff")
    return root, lay, fulls, st


def test_fnv_pins():
    """Inputs under 8 bytes take the byte path only: the published FNV-1a 64 vectors."""
    assert ock.fnv1a64_words(b"") == 0xCBF29CE484222325
    assert ock.fnv1a64_words(b"a") == 0xAF63DC4C8601EC8C
    assert ock.fnv1a64_words(b"foobar") == 0x85944171F73967E8
    # one full word: the xor takes the 8 bytes as a little-endian integer
    w = b"\x01\x02\x03\x04\x05\x06\x07\x08"
    assert ock.fnv1a64_words(w) == ((0xCBF29CE484222325 ^ 0x0807060504030201) * 0x100000001B3) % 2 ** 64


@pytest.mark.parametrize("case", range(8))
def test_oracle_placement_rule_brute(case):
    """from_full / to_full against a per-element search for the segment holding each index."""
    psi = 97
    name, lay = layouts(psi)[case]
    full = np.arange(1, psi + 1, dtype=np.float32)
    arrs = ock.from_full(full, lay.segs, lay.n, lay.stage)
    for i in range(psi):
        hits = [(g, ln, o, lo) for g, ln, o, lo in lay.segs if g <= i < g + ln]
        assert len(hits) == 1, (name, i)
        g, ln, o, lo = hits[0]
        if lay.stage == 0:
            assert all(a[i] == i + 1 for a in arrs), (name, i)
        else:
            assert arrs[o][lo + i - g] == i + 1, (name, i)
    assert sum(int(np.count_nonzero(a)) for a in arrs) == psi * (lay.n if lay.stage == 0 else 1)
    for r in range(lay.n if lay.stage == 0 else 1):
        assert np.array_equal(ock.to_full(arrs, lay.segs, psi, lay.stage, rank=r), full)


def test_library_checksum_matches_pins(tmp_path):
    lay = dp.Layout(1, 1, 3, [(0, 3, 0, 0)])
    arr = [np.zeros(3, np.float32)]
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "t", lay, arr, [np.zeros(3, np.float32)], [np.zeros(3, np.float32)],
                          bytearray(64), user_meta=b"foobar")
    man = ock.read_manifest(os.path.join(root, "t"))
    assert man["user.bin"] == (6, 0x85944171F73967E8)


def test_save_format_read_by_oracle(saved):
    root, lay, fulls, st = saved
    ck = ock.read_checkpoint(root)
    assert ck["tag"] == "step7" and (ck["stage"], ck["n"], ck["psi"]) == (1, 4, PSI)
    assert ck["segs"] == lay.segs
    for name, f in zip(("master", "m", "v"), fulls):
        assert np.array_equal(bits(ck[name]), bits(f)), name
    assert ck["user"] == b"cursor=4096\x00rng=\xff"
    d = os.path.join(root, "step7")
    assert set(ck["manifest"]) == {"shard_0.bin", "shard_1.bin", "shard_2.bin", "shard_3.bin", "state.bin",
                                   "layout.bin", "user.bin"}
    for name, (size, fnv) in ck["manifest"].items():
        data = open(os.path.join(d, name), "rb").read()
        assert (len(data), ock.fnv1a64_words(data)) == (size, fnv), name
    # saved: t, beta powers, error, good_steps, loss scale; cleared: the per-step and kernel fields, cur_set
    t, found, err, good, nonf, b1t, b2t, wc, wf, wt, scale, cur = decode_state(ck["state"])
    assert (t, found, err, good, nonf, wc, wf, wt, scale, cur) == (7, 0, 0, 3, 0, 0, 0, 0, 1024.0, 0)
    assert (b1t, b2t) == (0.9 ** 7, 0.999 ** 7)
    assert open(os.path.join(root, "LATEST")).read() == "step7\n"
    assert not os.path.exists(os.path.join(root, "step7.partial"))


@pytest.mark.parametrize("src", range(8))
@pytest.mark.parametrize("dst", range(8))
def test_reshard_is_the_placement_rule(tmp_path, src, dst):
    """Save in one layout, load into another: the loaded arrays hold every element at its new place, bit for
    bit, and nothing outside the new layout's segments is written."""
    psi = 12_007
    (sn, slay), (dn, dlay) = layouts(psi)[src], layouts(psi)[dst]
    fulls = [full_bits(psi, 100 + s) for s in range(3)]
    M, Mm, V = arrays_for(slay, fulls)
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "a", slay, M, Mm, V, state_blob())
    sentinel = 0x5A5A5A5A
    M2, Mm2, V2 = arrays_for(dlay, fulls, sentinel=sentinel)
    st2 = bytearray(64)
    meta = dp.dp_checkpoint_load(root, None, dlay, M2, Mm2, V2, st2)
    assert meta == b""
    covered = [np.zeros(L, bool) for L in dlay.state_lens()]
    for g, ln, o, lo in dlay.segs:
        if dlay.stage == 0:
            for c in covered:
                c[g:g + ln] = True
        else:
            covered[o][lo:lo + ln] = True
    for name, got, f in zip(("master", "m", "v"), (M2, Mm2, V2), fulls):
        want = ock.from_full(f, dlay.segs, dlay.n, dlay.stage)
        for r in range(dlay.n):
            c = covered[r]
            assert np.array_equal(bits(got[r])[c], bits(want[r])[c]), (sn, dn, name, r)
            assert np.all(bits(got[r])[~c] == sentinel), (sn, dn, name, r)
    assert decode_state(st2)[:4] == (7, 0, 0, 3)


def test_round_trip_through_another_layout(tmp_path):
    psi = 20_003
    ls = layouts(psi)
    a, b = ls[2][1], ls[3][1]
    fulls = [full_bits(psi, 9 + s) for s in range(3)]
    A = arrays_for(a, fulls)
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "a", a, *A, state_blob())
    B = arrays_for(b, fulls, sentinel=0)
    stb = bytearray(64)
    dp.dp_checkpoint_load(root, "a", b, *B, stb)
    dp.dp_checkpoint_save(root, "b", b, *B, stb)
    A2 = arrays_for(a, fulls, sentinel=0)
    dp.dp_checkpoint_load(root, "b", a, *A2, bytearray(64))
    for x, y in zip(A, A2):
        for r in range(a.n):
            assert np.array_equal(bits(x[r]), bits(y[r]))
    info = dp.dp_checkpoint_info(root)
    assert (info.stage, info.n, info.psi, info.segs) == (b.stage, b.n, b.psi, b.segs)


def test_latest_and_leftover_partial(saved):
    root, lay, fulls, _ = saved
    fulls2 = [full_bits(PSI, s) for s in (4, 5, 6)]
    dp.dp_checkpoint_save(root, "step8", lay, *arrays_for(lay, fulls2), state_blob(t=8))
    # a save that died before its rename leaves a directory nobody reads
    junk = os.path.join(root, "step9.partial")
    os.makedirs(junk)
    open(os.path.join(junk, "shard_0.bin"), "wb").write(b"\x00" * 100)
    got = arrays_for(lay, fulls, sentinel=0)
    st = bytearray(64)
    dp.dp_checkpoint_load(root, None, lay, *got, st)
    assert decode_state(st)[0] == 8
    assert np.array_equal(bits(ock.to_full(got[0], lay.segs, PSI, lay.stage)), bits(fulls2[0]))
    # the next save of that tag overwrites the leftover
    dp.dp_checkpoint_save(root, "step9", lay, *arrays_for(lay, fulls), state_blob(t=9))
    assert ock.read_checkpoint(root)["tag"] == "step9"
    # an older checkpoint stays loadable by tag
    dp.dp_checkpoint_load(root, "step7", lay, *got, st)
    assert decode_state(st)[0] == 7


def test_existing_tag_is_refused(saved):
    root, lay, fulls, st = saved
    with pytest.raises(dp.DPError) as e:
        dp.dp_checkpoint_save(root, "step7", lay, *arrays_for(lay, fulls), st)
    assert e.value.code == dp.DP_ERR_IO
    assert open(os.path.join(root, "LATEST")).read() == "step7\n"


@pytest.mark.parametrize("tag", ["", ".hidden", "../escape", "a/b", "x" * 201, "sp ace"])
def test_bad_tags(tmp_path, tag):
    lay = dp.Layout(1, 1, 4, [(0, 4, 0, 0)])
    z = [np.zeros(4, np.float32)]
    with pytest.raises(dp.DPError) as e:
        dp.dp_checkpoint_save(str(tmp_path), tag, lay, z, z, z, bytearray(64))
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    assert os.listdir(str(tmp_path)) == []


def flip_byte(path: str, off: int) -> None:
    with open(path, "r+b") as f:
        f.seek(off)
        b = f.read(1)
        f.seek(off)
        f.write(bytes([b[0] ^ 0x10]))


def test_corrupt_shard_detected(saved):
    root, lay, fulls, _ = saved
    shard = os.path.join(root, "step7", "shard_2.bin")
    flip_byte(shard, 24 + 4 * 123)
    got = arrays_for(lay, fulls, sentinel=0)
    with pytest.raises(dp.DPError) as e:
        dp.dp_checkpoint_load(root, None, lay, *got, bytearray(64))
    assert e.value.code == dp.DP_ERR_IO and "shard_2.bin" in str(e.value)
    # unverified, the flipped value loads: the checksum is what catches it
    dp.dp_checkpoint_load(root, None, lay, *got, bytearray(64), verify=False)
    assert not np.array_equal(bits(got[0][2][:200]), bits(ock.from_full(fulls[0], lay.segs, 4, 1)[2][:200]))


def test_truncated_or_unlisted_files_detected(saved):
    root, lay, fulls, _ = saved
    got = arrays_for(lay, fulls, sentinel=0)
    d = os.path.join(root, "step7")
    with open(os.path.join(d, "shard_1.bin"), "r+b") as f:
        f.truncate(os.path.getsize(os.path.join(d, "shard_1.bin")) - 4)
    with pytest.raises(dp.DPError) as e:      # the size check runs even unverified
        dp.dp_checkpoint_load(root, None, lay, *got, bytearray(64), verify=False)
    assert e.value.code == dp.DP_ERR_IO
    man = open(os.path.join(d, "MANIFEST")).read().splitlines()
    open(os.path.join(d, "MANIFEST"), "w").write("\n".join(l for l in man if "state.bin" not in l) + "\n")
    with pytest.raises(dp.DPError) as e:
        dp.dp_checkpoint_info(root)
    assert e.value.code == dp.DP_ERR_IO and "state.bin" in str(e.value)
    open(os.path.join(root, "LATEST"), "w").write("../elsewhere\n")
    with pytest.raises(dp.DPError):
        dp.dp_checkpoint_info(root)


def test_parameter_count_must_match(saved):
    root, lay, fulls, _ = saved
    other = dp.Layout(1, 2, PSI + 1, synth.layout_even(PSI + 1, 2))
    z = [[np.zeros(L, np.float32) for L in other.state_lens()] for _ in range(3)]
    with pytest.raises(dp.DPError) as e:
        dp.dp_checkpoint_load(root, None, other, *z, bytearray(64))
    assert e.value.code == dp.DP_ERR_INVALID_ARG


def test_user_meta_capacity_is_checked(saved):
    root, lay, fulls, _ = saved
    got = arrays_for(lay, fulls, sentinel=0)
    ptr = lambda arrs: (ctypes.c_void_p * lay.n)(*[a.ctypes.data for a in arrs])
    st = bytearray(64)
    stp = ctypes.addressof(ctypes.c_char.from_buffer(st))
    buf = ctypes.create_string_buffer(4)
    cap = ctypes.c_uint64(4)
    rc = dp.LIB.dp_checkpoint_load(root.encode(), None, ctypes.byref(lay.c), ptr(got[0]), ptr(got[1]), ptr(got[2]),
                                   stp, buf, ctypes.byref(cap), 1, 1, 0)
    assert rc == dp.DP_ERR_INVALID_ARG
    size = ctypes.c_uint64(0)
    rc = dp.LIB.dp_checkpoint_load(root.encode(), None, ctypes.byref(lay.c), ptr(got[0]), ptr(got[1]), ptr(got[2]),
                                   stp, None, ctypes.byref(size), 1, 0, 0)
    assert rc == dp.DP_OK and size.value == len(b"cursor=4096\x00rng=\xff")


def test_failed_save_leaves_previous_checkpoint(saved):
    """A save that fails part-way (the file-size limit makes a shard write fail with EFBIG) returns DP_ERR_IO,
    publishes nothing, and the previous checkpoint stays the one LATEST names."""
    root, lay, fulls, _ = saved
    child = textwrap.dedent("""
        import os, resource, signal, sys
        import numpy as np
        sys.path[:0] = [%r, os.path.join(%r, "tests")]
        import synth
        import zero_gradient_sync_gb300 as dp
        from oracle import checkpoint as ock
        signal.signal(signal.SIGXFSZ, signal.SIG_IGN)
        lay = dp.Layout(1, 4, %d, synth.layout_ragged(%d, 4, 7))
        arrs = [ock.from_full(np.ones(%d, np.float32), lay.segs, 4, 1) for _ in range(3)]
        resource.setrlimit(resource.RLIMIT_FSIZE, (20000, 20000))
        try:
            dp.dp_checkpoint_save(%r, "step8", lay, *arrs, bytearray(64))
        except dp.DPError as e:
            print("code", e.code, e)
            sys.exit(0 if e.code == dp.DP_ERR_IO else 3)
        sys.exit(4)
    """) % (ROOT, ROOT, PSI, PSI, PSI, root)
    r = subprocess.run([sys.executable, "-c", child], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "File too large" in r.stdout or "EFBIG" in r.stdout or "write" in r.stdout
    assert open(os.path.join(root, "LATEST")).read() == "step7\n"
    assert not os.path.exists(os.path.join(root, "step8"))
    got = arrays_for(lay, fulls, sentinel=0)
    dp.dp_checkpoint_load(root, None, lay, *got, bytearray(64))
    for x, f in zip(got, fulls):
        assert np.array_equal(bits(ock.to_full(x, lay.segs, PSI, 1)), bits(f))


def test_mixed_buffer_kinds_rejected(saved):
    root, lay, fulls, _ = saved
    torch = pytest.importorskip("torch")
    got = arrays_for(lay, fulls, sentinel=0)
    got[0][0] = torch.zeros(len(got[0][0]))          # a CPU tensor is a host buffer too: accepted
    dp.dp_checkpoint_load(root, None, lay, *got, bytearray(64))
    with pytest.raises(ValueError):
        dp.dp_checkpoint_load(root, None, lay, got[0][:3], got[1], got[2], bytearray(64))
