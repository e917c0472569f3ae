"""The per-micro-step reduce-scatter on the GPU (-m gpu): dp_reduce_scatter_micro for k = 0..a-1, then
dp_step_update.

Its averaged gradient must equal, bit for bit, the brute-force emulation in which each micro-step goes round
the simulated ring and is summed into the owner's accumulator (both arithmetics); the step must match the
float64 oracle within the usual tolerances; a non-finite value in any micro-step skips the whole step.
"""
import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from oracle import brute
from synth import device as sd

import gpu_util as gu

pytestmark = pytest.mark.gpu

COMP, PLAIN = dp.DP_SUM_COMPENSATED, dp.DP_SUM_PLAIN
BASE = synth.WORKLOADS["tiny"]


def adam_of(wl):
    return dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)


def upload_micro(c):
    from zero_gradient_sync_gb300.buffers import StepBuffers
    b = StepBuffers(c.layout, c.wl.a, "cuda", micro_acc=True)
    ref = gu.upload(c)
    for x, y in zip(b.grads, ref.grads):
        x.copy_(y)
    for dst, src in ((b.master, ref.master), (b.m, ref.m), (b.v, ref.v), (b.replicas, ref.replicas)):
        for x, y in zip(dst, src):
            x.copy_(y)
    b.state.copy_(ref.state)
    return b


CASES = [
    # psi, n, a, stage, layout, extra
    (1, 1, 1, 1, "even", {}),
    (13, 3, 2, 1, "even", {}),
    (4099, 2, 3, 2, "even", {}),
    (3 * 7680 + 5, 5, 4, 2, "ragged", {}),
    (65536 + 3, 7, 2, 3, "random", {"nseg": 29}),
    (100_003, 8, 4, 2, "buckets", {"bucket": 20_000, "misalign": 3}),
    (40_961, 16, 2, 2, "even", {}),
    (33_335, 4, 1, 2, "random", {"nseg": 9}),
    (20_000, 6, 8, 0, "ragged", {}),
]


@pytest.mark.parametrize("psi,n,a,stage,layout,extra", CASES)
@pytest.mark.parametrize("arith", [PLAIN, COMP])
def test_micro_gbar_equals_emulation(dev, psi, n, a, stage, layout, extra, arith):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=700 + n, sigma_g=1.0, tail_p=0.3,
                    tail_mult=float(2 ** 20), **extra)
    c = gu.make_case(wl)
    b = upload_micro(c)
    for k in range(a):
        b.reduce_micro(k, adam_of(wl), wl.loss_scale, arith)
    torch.cuda.synchronize()
    want = brute.micro_rs_gbar(c.grads, n, a, c.segs, psi, wl.loss_scale, "f32pair" if arith == COMP else "f32")
    got = sd.gather_full(b.gbar, c.segs, psi, 1)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["t"]) == (0, 1)


@pytest.mark.parametrize("psi,n,a,stage,layout,extra", CASES)
def test_micro_step_matches_oracle(dev, psi, n, a, stage, layout, extra):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=800 + n, **extra)
    c = gu.make_case(wl)
    b = upload_micro(c)
    b.step_micro(adam_of(wl), wl.loss_scale, COMP)
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


def test_micro_on_loss_scale_one_with_outliers(dev):
    wl = BASE.with_(psi=300_007, n=4, a=4, loss_scale=1.0, tail_p=0.01, tail_mult=100.0, seed=19, stage=2)
    c = gu.make_case(wl)
    b = upload_micro(c)
    b.step_micro(adam_of(wl), wl.loss_scale, COMP)
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


def test_micro_skip_and_determinism(dev):
    wl = BASE.with_(psi=2_000_003, n=8, a=4, stage=2, layout="ragged", seed=23)
    c = gu.make_case(wl)
    A = adam_of(wl)
    b = upload_micro(c)
    for k in range(wl.a):
        b.reduce_micro(k, A, wl.loss_scale, COMP)
    first = [x.clone() for x in b.gbar]
    for _ in range(2):
        for k in range(wl.a):
            b.reduce_micro(k, A, wl.loss_scale, COMP)
        torch.cuda.synchronize()
        for x, y in zip(first, b.gbar):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    # -inf in a middle micro-step of one rank: the whole step is skipped
    b2 = upload_micro(c)
    before = gu.snapshot(b2)
    b2.grad(3, 1)[12345:12346].view(torch.int16).fill_(synth.BF16_NEG_INF - 0x10000)   # as a signed 16-bit word
    b2.step_micro(A, wl.loss_scale, COMP)
    st = dp.read_state(b2.state)
    assert (st["found_inf"], st["nonfinite"], st["t"]) == (1, 1, 0)
    assert gu.snapshot(b2) == before


def test_micro_argument_checks(dev):
    wl = BASE.with_(psi=5000, n=2, a=2)
    c = gu.make_case(wl)
    b = upload_micro(c)
    A = adam_of(wl)
    g = [b.grad(r, 0) for r in range(wl.n)]
    with pytest.raises(dp.DPError):
        dp.dp_reduce_scatter_micro(b.acc, b.gbar, None, g, 2, 2, c.layout, A, 1.0, COMP, b.state)
    with pytest.raises(dp.DPError):
        dp.dp_reduce_scatter_micro(b.acc, b.gbar, None, g, 0, 2, c.layout, A, 1.0, COMP | dp.DP_ORDER_TREE, b.state)
    # a > 1 with no accumulator: refused before any launch
    rc = dp.LIB.dp_reduce_scatter_micro(None, None, None, dp._lib._ptr_array(g), 0, 2, dp._lib.ctypes.byref(c.layout.c),
                                        A, 1.0, COMP, b.state.data_ptr(), 0)
    assert rc == dp.DP_ERR_INVALID_ARG


@pytest.mark.parametrize("inject", [False, True])
def test_micro_deferred_commit_equals_direct(dev, inject):
    """The per-micro-step form with DP_DEFER_COMMIT on its calls (the step split across GPUs) and
    DP_DEVICE_SCALE: the last call publishes the decision without committing; dp_commit_step with the scaler then
    commits (or, with a NaN in one micro-step, skips and backs the scale off) and dp_step_update finishes.  The
    result equals, byte for byte, dp_step_scaled's -- the same order of ranks within each micro-step only when
    a = 1, so the comparison runs at a = 1 -- and the state words (t, scale, clean-step count) agree."""
    wl = BASE.with_(psi=250_003, n=4, a=1, stage=2, layout="ragged", seed=41, loss_scale=2.0 ** 12)
    c = gu.make_case(wl)
    A = adam_of(wl)
    sc = dp.scaler(2.0, 0.5, 2, 2.0 ** 8, 2.0 ** 24)
    ref = gu.upload(c)
    b = upload_micro(c)
    for x in (ref, b):
        dp.dp_scaler_init(x.state, wl.loss_scale)
        if inject:
            x.grad(2, 0)[777:778].view(torch.int16).fill_(synth.BF16_NAN)
    for _ in range(3):
        ref.step_scaled(A, sc)
        b.reduce_micro(0, A, 1.0, COMP | dp.DP_DEFER_COMMIT | dp.DP_DEVICE_SCALE)
        mid = dp.read_state(b.state)
        assert mid["found_inf"] == int(inject)
        dp.dp_commit_step(b.state, A, sc)
        b.update(A)
        r, g = dp.read_state(ref.state), dp.read_state(b.state)
        for key in ("t", "found_inf", "nonfinite", "loss_scale", "good_steps", "b1t", "b2t", "error"):
            assert g[key] == r[key], key
        assert gu.snapshot(b) == gu.snapshot(ref)
