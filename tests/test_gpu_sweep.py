"""The flat-buffer sweep at its own sizes (-m gpu): every case up to 10^8 parameters.

The sweep is the n x a axis of the data-parallel worked example in "Distributed Training: Split along the Four
Axes" (each of n ranks accumulates a micro-steps before one all-reduce), over flat buffers of 2^20, 2^20 + 3 (an
odd tail), 2^24 and 10^8 parameters, n in {2, 4, 8}, a in {1, 8}, even and seeded ragged shards (empty shards
possible), ZeRO stages and loss scales 2^8 ... 2^24 cycled over the cases.  Each case:

1. one step in the benchmark's launch configuration (dp_step_reduce, dp_step_update) at the case's fixed loss
   scale, checked against the float64 oracle on every element (up to 2^20 + 3) or on 10^5 random elements plus
   both ends of every shard and the end of the space;
2. one step with a non-finite value injected at the case's seeded site (+inf, -inf or NaN in one rank's
   micro-step) through dp_step_scaled with the device-resident scale set to the case's: the step is skipped,
   every master/m/v/replica byte and t are unchanged, and the scale backs off to half;
3. the injected value removed, one more dp_step_scaled step at the halved scale, checked against the oracle's
   own two-step chain (its step 1 feeds its step 2) at twice the single-step tolerance.
Cases of 2^28 + 5 and 10^9 parameters run in test_gpu_fullsize.py.
"""
import gc

import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from synth import device as sd
from zero_gradient_sync_gb300.buffers import StepBuffers

import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = [w for w in synth.sweep_cases() if w.psi <= 10 ** 8]
INJECT_BITS = {0: synth.BF16_POS_INF, 1: synth.BF16_NEG_INF, 2: synth.BF16_NAN}


def sampled(b, segs, idx, wl, gi):
    return {"master": gu.gather_state(b.master, segs, idx, wl.stage),
            "m": gu.gather_state(b.m, segs, idx, wl.stage),
            "v": gu.gather_state(b.v, segs, idx, wl.stage),
            "replicas": [sd.bits_of_bf16(r[gi]) for r in b.replicas]}


def check(g, o, scale=1.0):
    gu.assert_close_f32(g["master"], o["master"], "master", scale)
    gu.assert_close_f32(g["m"], o["m"], "m", scale)
    gu.assert_close_f32(g["v"], o["v"], "v", scale)
    gu.assert_replicas(g["replicas"], o["replicas"])


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_sweep_case(dev, wl):
    segs = synth.layout_of(wl)
    L = dp.Layout(wl.stage, wl.n, wl.psi, segs)
    b = StepBuffers(L, wl.a)
    sd.fill_grads(b.grads, wl)
    sd.fill_master(b.master, wl, segs, wl.stage)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    S = wl.loss_scale

    # 1. the benchmark's two launches at the case's fixed loss scale
    b.reduce(A, S)
    b.update(A)
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["error"], st["t"]) == (0, 0, 0, 1)
    if wl.psi <= (1 << 20) + 3:
        idx = np.arange(wl.psi, dtype=np.int64)
    else:
        idx = gu.sample_indices(wl, segs, 100_000, wl.seed + 17)
    gi = torch.from_numpy(idx).to(dev)
    o1 = gu.oracle_at(wl, idx)
    assert (o1["found"], o1["nonfinite"], o1["t"]) == (0, 0, 1)
    check(sampled(b, segs, idx, wl, gi), o1)

    # 2. a skipped step: one non-finite gradient value at the case's seeded site, dynamic scale set to S
    r, k, i, kind = synth.inject_site(wl, 0)
    keep = b.grad(r, k)[i:i + 1].clone()
    b.grad(r, k)[i:i + 1].view(torch.int16).fill_(np.array(INJECT_BITS[kind], np.uint16).view(np.int16).item())
    before = [x.clone() for x in b.master + b.m + b.v + b.replicas]
    dp.dp_scaler_init(b.state, S)
    sc = dp.scaler(2.0, 0.5, 1 << 30, 1.0, 2.0 ** 24)
    b.step_scaled(A, sc)
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["error"], st["t"]) == (1, 1, 0, 1)
    assert st["loss_scale"] == S / 2
    for x, y in zip(before, b.master + b.m + b.v + b.replicas):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    del before

    # 3. the same gradients, clean again, at the backed-off scale; the oracle chains its own two steps
    b.grad(r, k)[i:i + 1].copy_(keep)
    b.step_scaled(A, sc)
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["error"], st["t"]) == (0, 0, 0, 2)
    o2 = gu.oracle_at(wl.with_(loss_scale=S / 2), idx, t0=1, m=o1["m"], v=o1["v"], master=o1["master"])
    assert (o2["found"], o2["t"]) == (0, 2)
    check(sampled(b, segs, idx, wl, gi), o2, scale=2.0)
    del b
    gc.collect()
    torch.cuda.empty_cache()
