"""Sharded checkpoints of device state (-m gpu): save after GPU steps, reshard on load, resume.

A reshard is a permutation, so it is checked bit for bit against the oracle's placement rule and its reader
of the on-disk format; a resumed run is checked against the oracle's step from the loaded state, and, where
the reduction order is unchanged, bit for bit against the run that never stopped.
"""
import shutil

import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from oracle import checkpoint as ock
from synth import device as sd

import gpu_util as gu

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["tiny"].with_(psi=200_003, n=4, a=2, stage=1, layout="ragged", seed=301)


def adam_of(wl):
    return dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)


def feed(b, wl, seed):
    w = wl.with_(seed=seed)
    for q in range(wl.n * wl.a):
        b.grads[q].copy_(sd.bf16_from_bits(synth.grads_bf16(w, q // wl.a, q % wl.a)))


def full_state(b, segs, psi, stage):
    return [sd.gather_full(x, segs, psi, stage) for x in (b.master, b.m, b.v)]


def bits(x):
    return np.asarray(x).view(np.uint32)


def test_save_then_reshard_to_fewer_ranks_and_resume(dev, tmp_path):
    wl = BASE
    c = gu.make_case(wl)
    b = gu.upload(c)
    A = adam_of(wl)
    for s in range(2):
        feed(b, wl, wl.seed + s)
        b.step(A, wl.loss_scale)
    saved = full_state(b, c.segs, wl.psi, c.stage)
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "t2", c.layout, b.master, b.m, b.v, b.state, user_meta=b"lr-schedule:cosine")
    ck = ock.read_checkpoint(root)
    for name, x in zip(("master", "m", "v"), saved):
        assert np.array_equal(bits(ck[name]), bits(x)), name

    # n = 3, ZeRO-2, misaligned buckets: a different world size and layout of the same parameters
    wl3 = wl.with_(n=3, stage=2, layout="buckets", bucket=30_011, misalign=3, seed=wl.seed + 50)
    segs3 = synth.layout_of(wl3)
    c3 = gu.make_case(wl3, segs=segs3, t=2, master=saved[0], m=saved[1], v=saved[2])
    b3 = gu.upload(gu.make_case(wl3, segs=segs3))          # different contents, overwritten by the load
    meta = dp.dp_checkpoint_load(root, None, c3.layout, b3.master, b3.m, b3.v, b3.state)
    assert meta == b"lr-schedule:cosine"
    loaded = full_state(b3, segs3, wl.psi, c3.stage)
    for x, y in zip(loaded, saved):
        assert np.array_equal(bits(x), bits(y))
    st = dp.read_state(b3.state)
    assert (st["t"], st["found_inf"], st["error"]) == (2, 0, 0)

    # one more step at n = 3 against the oracle started from the same state
    for q, g in enumerate(c3.grads):
        b3.grads[q].copy_(sd.bf16_from_bits(g))
    b3.step(adam_of(wl3), wl3.loss_scale)
    gu.assert_matches_oracle(gu.gpu_result(c3, b3), gu.run_oracle(c3))


def test_resume_equals_uninterrupted_run(dev, tmp_path):
    """Same segments (so the same reduction order), stage 1 -> stage 0 through a checkpoint: the resumed run
    is bit-identical to the run that never stopped."""
    wl = BASE.with_(layout="random", nseg=13)
    c = gu.make_case(wl)
    A = adam_of(wl)
    ref = gu.upload(c)
    run = gu.upload(c)
    for s in range(2):
        feed(ref, wl, wl.seed + s)
        feed(run, wl, wl.seed + s)
        ref.step(A, wl.loss_scale)
        run.step(A, wl.loss_scale)
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "t2", c.layout, run.master, run.m, run.v, run.state)
    lay0 = dp.Layout(0, wl.n, wl.psi, c.segs)
    from zero_gradient_sync_gb300.buffers import StepBuffers
    res = StepBuffers(lay0, wl.a, "cuda")
    dp.dp_checkpoint_load(root, "t2", lay0, res.master, res.m, res.v, res.state)
    for s in (2, 3):
        feed(ref, wl, wl.seed + s)
        feed(res, wl, wl.seed + s)
        ref.step(A, wl.loss_scale)
        res.step(A, wl.loss_scale)
    torch.cuda.synchronize()
    for x, y in zip(full_state(ref, c.segs, wl.psi, 1), full_state(res, c.segs, wl.psi, 0)):
        assert np.array_equal(bits(x), bits(y))
    for r in range(wl.n):
        assert torch.equal(ref.replicas[r].view(torch.int16), res.replicas[r].view(torch.int16))
    assert dp.read_state(ref.state)["t"] == dp.read_state(res.state)["t"] == 4


def test_loss_scale_survives_checkpoint(dev, tmp_path):
    """The dynamic loss scale and its clean-step count are part of the saved state."""
    wl = BASE.with_(psi=50_021, sigma_g=1e-3)
    c = gu.make_case(wl)
    A = adam_of(wl)
    sc = dp.scaler(2.0, 0.5, 3, 2.0 ** 8, 2.0 ** 24)
    ref, run = gu.upload(c), gu.upload(c)
    for b in (ref, run):
        dp.dp_scaler_init(b.state, 2.0 ** 16)
    for s in range(4):
        for b in (ref, run):
            feed(b, wl, wl.seed + s)
            b.step_scaled(A, sc)
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "s4", c.layout, run.master, run.m, run.v, run.state)
    res = gu.upload(c)
    dp.dp_checkpoint_load(root, "s4", c.layout, res.master, res.m, res.v, res.state)
    a, b_ = dp.read_state(ref.state), dp.read_state(res.state)
    assert (a["loss_scale"], a["good_steps"], a["t"]) == (b_["loss_scale"], b_["good_steps"], b_["t"])
    assert a["loss_scale"] == 2.0 ** 17 and a["good_steps"] == 1
    for s in range(4, 7):
        for b in (ref, res):
            feed(b, wl, wl.seed + s)
            b.step_scaled(A, sc)
    sa, sb = gu.snapshot(ref), gu.snapshot(res)
    n_state = 3 * wl.n
    assert sa[:n_state] == sb[:n_state]
    assert dp.read_state(ref.state)["loss_scale"] == dp.read_state(res.state)["loss_scale"]


def test_single_pass_current_set_checkpoint(dev, tmp_path):
    """A single-pass run keeps two master/m/v sets; the current one is saved and loads as set 0."""
    wl = BASE.with_(psi=70_001)
    c = gu.make_case(wl)
    A = adam_of(wl)
    run = gu.upload(c, second_set=True)
    for s in range(3):
        feed(run, wl, wl.seed + s)
        run.step_single_pass(A, wl.loss_scale)
    cur = run.current()
    want = [sd.gather_full(x, c.segs, wl.psi, c.stage) for x in cur]
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "sp", c.layout, *cur, run.state)
    res = gu.upload(c, second_set=True)
    dp.dp_checkpoint_load(root, "sp", c.layout, res.master, res.m, res.v, res.state)
    st = dp.read_state(res.state)
    assert (st["cur_set"], st["t"]) == (0, 3)
    got = [sd.gather_full(x, c.segs, wl.psi, c.stage) for x in res.current()]
    for x, y in zip(got, want):
        assert np.array_equal(bits(x), bits(y))


def test_gpu_save_load_of_full_size_state(dev, tmp_path):
    """The 123,568,896-parameter, n = 8 ZeRO-1 state (1.5 GB) saves and reloads into n = 4 intact."""
    psi = synth.WORKLOADS["gpt2_small"].psi
    lay8 = dp.Layout.even(psi, 8, stage=1)
    lay4 = dp.Layout.even(psi, 4, stage=1)
    g = torch.Generator(device="cuda").manual_seed(5)
    src = [[torch.randn(L, device="cuda", generator=g) for L in lay8.state_lens()] for _ in range(3)]
    state = dp.new_state("cuda")
    root = str(tmp_path)
    dp.dp_checkpoint_save(root, "full", lay8, *src, state)
    dst = [[torch.empty(L, device="cuda") for L in lay4.state_lens()] for _ in range(3)]
    dp.dp_checkpoint_load(root, "full", lay4, *dst, state, verify=True)
    for a, b in zip(src, dst):
        assert torch.equal(torch.cat(a).view(torch.int32), torch.cat(b).view(torch.int32))
    shutil.rmtree(root, ignore_errors=True)   # 1.5 GB of shard files: not left behind in pytest's kept temp dirs
