"""The C-ABI library on the CPU: it loads, exports every entry point the header declares, and its host-side
logic (layout checks, layout construction, models, argument errors) works without touching a GPU."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dpstep.h")


@pytest.fixture(scope="module")
def dp():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_dpstep_build", os.path.join(ROOT, "zero_gradient_sync_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import zero_gradient_sync_gb300 as z
    return z


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return sorted(set(re.findall(r"\b(dp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = header_functions()
    for must in ("dp_accumulate", "dp_reduce_scatter_avg", "dp_adam_shard", "dp_allgather_params", "dp_step"):
        assert must in names
    assert len(names) >= 24


def test_library_exports_every_declared_symbol(dp):
    lib = ctypes.CDLL(dp.LIB_PATH)
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_struct_sizes(dp):
    from zero_gradient_sync_gb300 import _lib
    assert ctypes.sizeof(_lib.dp_segment_t) == 32
    assert ctypes.sizeof(_lib.dp_layout_t) == 32
    assert ctypes.sizeof(_lib.dp_adam_t) == 16
    assert ctypes.sizeof(_lib.dp_step_state_t) == 64
    assert dp.LIB.dp_abi_version() == 2
    assert ctypes.sizeof(_lib.dp_scaler_t) == 20


@pytest.mark.parametrize("psi,n,bucket,mis", [(0, 2, 0, 0), (7, 8, 0, 0), ((1 << 20) + 3, 8, 0, 0),
                                                (10_000, 4, 3000, 3), (1_311_082_496, 8, 25_000_000, 3)])
def test_layout_even_matches_generator(dp, psi, n, bucket, mis):
    L = dp.Layout.even(psi, n, stage=3, bucket=bucket, misalign=mis)
    ref = synth.layout_buckets(psi, n, bucket, mis) if bucket else synth.layout_even(psi, n)
    if psi == 0:
        ref = []
    assert L.segs == [tuple(s) for s in ref]
    L.validate()
    assert L.shard_lens() == synth.shard_lengths(ref, n)


@pytest.mark.parametrize("kind", ["ragged", "random"])
def test_generated_layouts_validate(dp, kind):
    psi, n = 100_003, 5
    segs = synth.layout_ragged(psi, n, 3) if kind == "ragged" else synth.layout_random(psi, n, 17, 2)
    L = dp.Layout(2, n, psi, segs)
    L.validate()
    assert L.shard_lens() == synth.shard_lengths(segs, n)
    assert L.workspace_size() >= 4 * psi


def _bad(dp, stage, n, psi, segs):
    L = dp.Layout(stage, n, psi, segs)
    with pytest.raises(dp.DPError) as e:
        L.validate()
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    return str(e.value)


def test_layout_rejections(dp):
    assert "contiguous" in _bad(dp, 1, 2, 10, [(0, 5, 0, 0), (6, 4, 1, 0)])           # gap
    assert "cover" in _bad(dp, 1, 2, 10, [(0, 5, 0, 0), (5, 4, 1, 0)])                # short
    assert "owner" in _bad(dp, 1, 2, 10, [(0, 5, 0, 0), (5, 5, 2, 0)])                # owner >= n
    assert "overlap" in _bad(dp, 1, 2, 10, [(0, 5, 0, 0), (5, 5, 0, 3)])              # local overlap
    _bad(dp, 4, 2, 10, [(0, 10, 0, 0)])                                               # stage
    _bad(dp, 1, 0, 10, [(0, 10, 0, 0)])                                               # n = 0
    _bad(dp, 1, 17, 10, [(0, 10, 0, 0)])                                              # n > 16
    _bad(dp, 1, 2, 10, [(0, -1, 0, 0), (-1, 11, 1, 0)])                               # negative len


def test_step_argument_errors_launch_nothing(dp):
    """Invalid arguments are refused on the host before any CUDA call (this machine has no GPU)."""
    L = dp.Layout(1, 2, 16, [(0, 8, 0, 0), (8, 8, 1, 0)])
    before = dp.dp_kernel_launches()
    A = dp.adam()
    fake = [16 * (k + 1) for k in range(8)]     # aligned, never dereferenced
    with pytest.raises(dp.DPError) as e:        # a = 0
        dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 0, L, A, 1.0, state=256, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError) as e:        # misaligned grad pointer
        dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], [16, 17], 1, L, A, 1.0, gbar_shard=fake[:2], state=256, stream=0)
    assert e.value.code == dp.DP_ERR_ALIGNMENT
    with pytest.raises(dp.DPError) as e:        # loss scale 0
        dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 1, L, A, 0.0, gbar_shard=fake[:2], state=256, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError) as e:        # beta1 = 1
        dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 1, L, dp.adam(beta1=1.0), 1.0,
                   gbar_shard=fake[:2], state=256, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError) as e:        # no gbar and no workspace
        dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 1, L, A, 1.0, state=256, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError) as e:        # null state
        dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 1, L, A, 1.0, gbar_shard=fake[:2], state=0, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError) as e:        # n * a > 64
        L9 = dp.Layout(1, 9, 9, [(k, 1, k, 0) for k in range(9)])
        dp.dp_step([16] * 9, [16] * 9, [16] * 9, [16] * 9, [16] * 72, 8, L9, A, 1.0, gbar_shard=[16] * 9, state=256, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    with pytest.raises(dp.DPError) as e:
        dp.dp_accumulate([16, 32], [16, 32], 16, 2, True, sum_mode=7, stream=0)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    assert dp.dp_kernel_launches() == before


def test_step_from_host_argument_errors_queue_nothing(dp):
    """dp_step_from_host checks every argument before it queues a copy or a kernel (no GPU needed)."""
    import ctypes
    L = dp.Layout(1, 2, 16, [(0, 8, 0, 0), (8, 8, 1, 0)])
    arr = ctypes.c_void_p * 2
    fake, null = arr(16, 32), arr(0, 0)
    A = dp.adam()
    f = dp.LIB.dp_step_from_host
    before = dp.dp_kernel_launches()
    # a = 0
    assert f(fake, fake, fake, fake, fake, fake, 0, ctypes.byref(L.c), A, 1.0, 0, fake, None, 256, None,
             None) == dp.DP_ERR_INVALID_ARG
    # a host gradient buffer missing
    assert f(fake, fake, fake, fake, null, fake, 1, ctypes.byref(L.c), A, 1.0, 0, fake, None, 256, None,
             None) != dp.DP_OK
    # a misaligned device gradient buffer
    assert f(fake, fake, fake, fake, fake, arr(16, 17), 1, ctypes.byref(L.c), A, 1.0, 0, fake, None, 256, None,
             None) == dp.DP_ERR_ALIGNMENT
    # no state
    assert f(fake, fake, fake, fake, fake, fake, 1, ctypes.byref(L.c), A, 1.0, 0, fake, None, None, None,
             None) == dp.DP_ERR_INVALID_ARG
    assert dp.dp_kernel_launches() == before


def test_global_batch(dp):
    G = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_numbers.json")))["global_batch_example"]
    assert dp.dp_global_batch(G["b"], G["n"], G["a"]) == G["B_global"] == 256
    # 3D parallelism: TP and PP degrees are not multiplied in -- only b, a and the DP degree
    assert dp.dp_global_batch(4, 8, 8) == 4 * 8 * 8
    assert dp.dp_global_batch(-1, 8, 8) == -1
    assert dp.dp_global_batch(2 ** 40, 2 ** 30, 2 ** 30) == -1


def test_memory_model_page_numbers(dp):
    G = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_numbers.json")))
    e = G["model_state_7b"]
    assert dp.dp_memory_model(0, e["params"], 1)[3] == e["bytes"]              # 16 B/param, 7B -> 112 GB
    w = G["fp16_weights_7b"]
    assert dp.dp_memory_model(0, w["params"], 8)[0] == w["bytes"]              # 2 B/param weights -> 14 GB
    for n in (1, 2, 8, 64):
        assert dp.dp_memory_model(3, e["params"], n)[3] == pytest.approx(16 * e["params"] / n)  # 16 Psi / N
    rng = G["mixed_precision_state_range"]
    assert rng["low_bytes_per_param"] <= dp.dp_memory_model(0, 1, 1)[3] <= rng["high_bytes_per_param"]
    # sharding only ever lowers the per-rank footprint, stage by stage
    tot = [dp.dp_memory_model(s, 10 ** 9, 8)[3] for s in range(4)]
    assert tot[0] > tot[1] > tot[2] > tot[3]


def test_traffic_model_matches_ring_simulation(dp):
    from oracle import ring
    for n in (2, 4, 8):
        psi = 8 * 105
        segs = synth.layout_even(psi, n)
        for stage in range(4):
            tr = ring.step_traffic(n, segs, psi, stage, 2, 2)
            sim = tr[list(tr)[0]].sent_bytes[0] + sum(t.sent_bytes[0] for t in list(tr.values())[1:])
            steps = sum(t.steps for t in tr.values())
            per, nsteps, ratio = dp.dp_traffic_model(stage, psi, n, 2, 2)
            assert per == pytest.approx(sim)
            assert nsteps == steps
        assert dp.dp_traffic_model(3, psi, n, 2, 2)[2] == pytest.approx(1.5)
        assert dp.dp_traffic_model(1, psi, n, 2, 2)[2] == pytest.approx(1.0)
        assert dp.dp_traffic_model(0, psi, n, 2, 2)[0] == pytest.approx(2 * (n - 1) / n * psi * 2)


def test_status_strings_and_timeout_knob(dp):
    assert dp.LIB.dp_status_str(0) == b"DP_OK"
    assert dp.LIB.dp_status_str(4) == b"DP_ERR_TIMEOUT"
    old = dp.dp_get_wait_timeout_ns()
    dp.dp_set_wait_timeout_ns(12345)
    assert dp.dp_get_wait_timeout_ns() == 12345
    dp.dp_set_wait_timeout_ns(old)


@pytest.mark.parametrize("kind", ["even", "buckets", "ragged", "random"])
def test_layout_slice_maps_every_element(dp, kind):
    """dp_layout_slice: every element of [lo, hi) keeps its owner, and its local index in the slice plus the
    owner's local_base is its local index in the whole layout (checked element by element)."""
    import synth
    psi, n = 9_973, 5
    wl = synth.WORKLOADS["tiny"].with_(psi=psi, n=n, layout=kind, bucket=1_001, misalign=3, nseg=37, seed=5)
    segs = synth.layout_of(wl)
    L = dp.Layout(3, n, psi, segs)
    own = np.empty(psi, np.int64)
    loc = np.empty(psi, np.int64)
    for g, ln, o, lo in segs:
        own[g:g + ln] = o
        loc[g:g + ln] = lo + np.arange(ln)
    rng = np.random.default_rng(3)
    cuts = [(0, psi), (0, 0), (psi, psi), (1, 2), (17, 5_000), (4_999, psi)]
    cuts += [tuple(sorted(rng.integers(0, psi + 1, 2).tolist())) for _ in range(6)]
    for lo, hi in cuts:
        S, base = L.slice(lo, hi)
        S.validate()
        assert S.psi == hi - lo and S.n == n and S.stage == 3
        got_own = np.full(hi - lo, -1, np.int64)
        got_loc = np.full(hi - lo, -1, np.int64)
        for g, ln, o, l0 in S.segs:
            got_own[g:g + ln] = o
            got_loc[g:g + ln] = base[o] + l0 + np.arange(ln)
        assert np.array_equal(got_own, own[lo:hi])
        assert np.array_equal(got_loc, loc[lo:hi])
        for r in range(n):   # each slice shard starts at the owner's lowest local index in the slice
            mine = loc[lo:hi][own[lo:hi] == r]
            assert base[r] == (mine.min() if mine.size else 0)
    with pytest.raises(dp.DPError):
        L.slice(5, 3)
    with pytest.raises(dp.DPError):
        L.slice(0, psi + 1)


def test_step_flags_accepted_only_where_documented(dp):
    """DP_DEFER_COMMIT / DP_DEVICE_SCALE: the calls that cannot defer refuse them before any launch; the
    commit calls check their arguments on the host."""
    L = dp.Layout(1, 2, 16, [(0, 8, 0, 0), (8, 8, 1, 0)])
    A = dp.adam()
    fake = [16 * (k + 1) for k in range(8)]
    before = dp.dp_kernel_launches()
    for flag in (dp.DP_DEFER_COMMIT, dp.DP_DEVICE_SCALE):
        with pytest.raises(dp.DPError) as e:
            dp.dp_step(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 1, L, A, 1.0, sum_mode=flag,
                       gbar_shard=fake[:2], state=256, stream=0)
        assert e.value.code == dp.DP_ERR_INVALID_ARG and "not accepted" in str(e.value)
        with pytest.raises(dp.DPError):
            dp.dp_step_scaled(fake[:2], fake[:2], fake[:2], fake[:2], fake[:2], 1, L, A, dp.scaler(), sum_mode=flag,
                              gbar_shard=fake[:2], state=256, stream=0)
        with pytest.raises(dp.DPError):
            dp.dp_reduce_scatter_avg(fake[:2], fake[:2], L, 1.0, flag, 256, stream=0)
    with pytest.raises(dp.DPError):              # an unknown bit
        dp.dp_step_reduce(fake[:2], None, fake[:2], 1, L, A, 1.0, 128, 256, stream=0)
    with pytest.raises(dp.DPError):              # commit: null state
        dp.dp_commit_step(0, A, stream=0)
    with pytest.raises(dp.DPError):              # commit: bad scaler
        dp.dp_commit_step(256, A, dp.scaler(growth_factor=0.5), stream=0)
    with pytest.raises(dp.DPError):              # single-pass commit: stage 0
        dp.dp_commit_single_pass(fake[:2], fake[:4], dp.Layout(0, 2, 16, [(0, 8, 0, 0), (8, 8, 1, 0)]), A, 256,
                                 stream=0)
    assert dp.dp_kernel_launches() == before


def test_layouts_beyond_one_launch_table_validate(dp):
    """Layouts of more than DP_KERNEL_SEG segments are accepted on the host (each kernel then runs as several
    launches); shard lengths and the workspace follow the segments; more than DP_MAX_SEG is refused."""
    import synth
    psi, n = 1_000_003, 8
    segs = synth.layout_random(psi, n, 5000, seed=9)
    L = dp.Layout(2, n, psi, segs)
    L.validate()
    assert len([s for s in segs if s[1]]) > dp.DP_KERNEL_SEG
    assert L.shard_lens() == synth.shard_lengths(segs, n)
    assert L.workspace_size() == sum((4 * x + 255) // 256 * 256 for x in L.shard_lens())
    B = dp.Layout.even(psi, 4, stage=3, bucket=700, misalign=3)      # 1429 buckets x 4 = 5716 segments
    assert len(B.segs) == 4 * ((psi + 699) // 700)
    B.validate()
    with pytest.raises(dp.DPError):
        dp.Layout.even(dp.DP_MAX_SEG + 1, 2, bucket=1)


def test_single_pass_from_host_argument_errors_queue_nothing(dp):
    """dp_step_single_pass_from_host checks every argument before it queues a copy or a kernel (no GPU needed)."""
    import ctypes
    L = dp.Layout(1, 2, 16, [(0, 8, 0, 0), (8, 8, 1, 0)])
    two, four = ctypes.c_void_p * 2, ctypes.c_void_p * 4
    fake, null = two(16, 32), two(0, 0)
    st4 = four(16, 32, 48, 64)
    A = dp.adam()
    f = dp.LIB.dp_step_single_pass_from_host
    before = dp.dp_kernel_launches()
    assert f(fake, st4, st4, st4, fake, fake, 0, ctypes.byref(L.c), A, 1.0, 0, 256, None, None) == dp.DP_ERR_INVALID_ARG
    assert f(fake, st4, st4, st4, None, fake, 1, ctypes.byref(L.c), A, 1.0, 0, 256, None, None) == dp.DP_ERR_INVALID_ARG
    assert f(fake, st4, st4, st4, null, fake, 1, ctypes.byref(L.c), A, 1.0, 0, 256, None, None) != dp.DP_OK
    assert f(fake, st4, st4, st4, fake, two(16, 17), 1, ctypes.byref(L.c), A, 1.0, 0, 256, None,
             None) == dp.DP_ERR_ALIGNMENT
    assert f(fake, st4, st4, st4, fake, fake, 1, ctypes.byref(L.c), A, 1.0, 0, None, None, None) == dp.DP_ERR_INVALID_ARG
    assert f(fake, st4, st4, st4, fake, fake, 1, ctypes.byref(L.c), A, 1.0, dp.DP_ORDER_TREE | (1 << 10), 256, None,
             None) == dp.DP_ERR_INVALID_ARG
    assert dp.dp_kernel_launches() == before
