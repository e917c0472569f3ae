"""The device-resident dynamic loss scale (dp_step_scaled, -m gpu).

The scale lives in the step state: the reduction unscales by it and its last CTA updates it once the skip
decision is known.  Checked against the oracle's policy (pinned to torch's own loss-scale update on the CPU)
step by step through a run with injected overflows, and bit for bit against dp_step at the same scale.
"""
import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from oracle import scaler as oscaler
from synth import device as sd

import gpu_util as gu

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["tiny"].with_(psi=60_013, n=4, a=2, stage=2, layout="ragged", seed=201)


def test_scaled_step_equals_fixed_scale_step(dev):
    S = 2.0 ** 12
    wl = BASE.with_(loss_scale=S)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    fixed = gu.upload(c)
    fixed.step(A, S)
    scaled = gu.upload(c)
    dp.dp_scaler_init(scaled.state, S)
    sc = dp.scaler(2.0, 0.5, 4, 2.0 ** 8, 2.0 ** 24)
    scaled.step_scaled(A, sc)
    assert gu.snapshot(fixed) == gu.snapshot(scaled)
    st = dp.read_state(scaled.state)
    assert (st["loss_scale"], st["good_steps"], st["t"], st["found_inf"]) == (S, 1, 1, 0)
    gu.assert_matches_oracle(gu.gpu_result(c, scaled), gu.run_oracle(c))


def test_scale_follows_policy_through_overflows(dev):
    """30 steps, growth every 3 clean steps, overflow injected at some steps: the device scale, its clean-step
    count and the skip flag follow the oracle's policy, and the state equals a fixed-scale run fed the
    oracle's scale sequence."""
    wl = BASE.with_(sigma_g=1e-3)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    growth, backoff, interval, lo, hi = 2.0, 0.5, 3, 2.0 ** 8, 2.0 ** 24
    sc = dp.scaler(growth, backoff, interval, lo, hi)
    scaled = gu.upload(c)
    ref = gu.upload(c)
    S0 = 2.0 ** 22
    dp.dp_scaler_init(scaled.state, S0)
    s_or, good = S0, 0
    inject_at = {4, 5, 11, 12, 13, 20}
    for step in range(30):
        wls = wl.with_(seed=wl.seed + step)
        for q in range(wl.n * wl.a):
            g = synth.grads_bf16(wls, q // wl.a, q % wl.a)
            if step in inject_at and q == 3:
                g[(step * 977) % wl.psi] = synth.BF16_NAN if step % 2 else synth.BF16_POS_INF
            t = sd.bf16_from_bits(g)
            scaled.grads[q].copy_(t)
            ref.grads[q].copy_(t)
        scaled.step_scaled(A, sc)
        ref.step(A, s_or)          # the same step at the oracle's current scale
        found = step in inject_at
        s_or, good = oscaler.update(s_or, good, found, growth, backoff, interval, lo, hi)
        st = dp.read_state(scaled.state)
        assert st["found_inf"] == int(found), step
        assert (st["loss_scale"], st["good_steps"]) == (np.float32(s_or), good), step
        assert gu.snapshot(scaled) == gu.snapshot(ref), step
    assert lo <= s_or <= hi


def test_scale_stays_in_range(dev):
    wl = BASE.with_(psi=5000)
    c = gu.make_case(wl)
    A = dp.adam()
    b = gu.upload(c)
    dp.dp_scaler_init(b.state, 2.0 ** 24)
    sc = dp.scaler(2.0, 0.5, 1, 2.0 ** 8, 2.0 ** 24)
    for _ in range(3):
        b.step_scaled(A, sc)
        assert dp.read_state(b.state)["loss_scale"] == 2.0 ** 24
    b.grads[0].view(torch.int16)[7] = synth.BF16_POS_INF
    dp.dp_scaler_init(b.state, 2.0 ** 9)
    for expect in (2.0 ** 8, 2.0 ** 8):
        b.step_scaled(A, sc)
        assert dp.read_state(b.state)["loss_scale"] == expect


def test_invalid_device_scale_records_error_and_skips(dev):
    wl = BASE.with_(psi=5000)
    c = gu.make_case(wl)
    b = gu.upload(c)
    before = gu.snapshot(b)
    raw = bytearray(b.state.cpu().numpy().tobytes())
    raw[56:60] = np.float32(0.0).tobytes()          # loss_scale = 0: 1 / (n S) is not finite
    b.state.copy_(torch.frombuffer(raw, dtype=torch.uint8))
    b.step_scaled(dp.adam(), dp.scaler())
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["error"], st["t"]) == (1, dp.DP_ERR_INVALID_ARG, 0)
    assert gu.snapshot(b) == before


def test_scaler_argument_checks(dev):
    wl = BASE.with_(psi=5000)
    b = gu.upload(gu.make_case(wl))
    with pytest.raises(dp.DPError):
        dp.dp_scaler_init(b.state, 0.0)
    with pytest.raises(dp.DPError):
        b.step_scaled(dp.adam(), dp.scaler(growth_factor=0.5))
    with pytest.raises(dp.DPError):
        b.step_scaled(dp.adam(), dp.scaler(min_scale=4.0, max_scale=2.0))


def test_single_pass_with_device_scale_equals_fixed_scale(dev):
    """dp_step_single_pass with DP_DEVICE_SCALE unscales by the device-resident scale: with that scale set to S it
    equals the single pass at the fixed loss scale S byte for byte, and without a deferred commit it leaves the
    scale as it was (the policy runs only in dp_step_scaled or a commit given a scaler)."""
    S = 2.0 ** 14
    wl = BASE.with_(loss_scale=S)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    fixed = gu.upload(c, second_set=True)
    dev_scale = gu.upload(c, second_set=True)
    dp.dp_scaler_init(dev_scale.state, S)
    for _ in range(2):
        fixed.step_single_pass(A, S)
        dev_scale.step_single_pass(A, 1.0, dp.DP_SUM_COMPENSATED | dp.DP_DEVICE_SCALE)
    a, b = dp.read_state(fixed.state), dp.read_state(dev_scale.state)
    assert (b["t"], b["cur_set"], b["loss_scale"], b["good_steps"]) == (a["t"], a["cur_set"], S, 0)

    def current(x):
        torch.cuda.synchronize()
        ms, mm, vv = x.current()
        return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in ms + mm + vv + x.replicas]
    assert current(fixed) == current(dev_scale)
