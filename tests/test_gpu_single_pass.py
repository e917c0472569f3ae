"""dp_step_single_pass: the fused step in one pass over memory with double-buffered optimizer state (-m gpu).

Checked bit for bit against the two-pass dp_step (itself checked against the oracle) over several steps, on
every layout kind and ZeRO stage 1-3 and both reduction modes, plus the skip semantics (replicas restored,
current set kept, t kept) and the oracle directly.
"""
import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from synth import device as sd

import gpu_util as gu

pytestmark = pytest.mark.gpu

COMP, PLAIN = dp.DP_SUM_COMPENSATED, dp.DP_SUM_PLAIN
BASE = synth.WORKLOADS["tiny"]


def snap_current(b):
    torch.cuda.synchronize()
    ms, mm, vv = b.current()
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in ms + mm + vv + b.replicas]


def snap_two_pass(b):
    torch.cuda.synchronize()
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in b.master + b.m + b.v + b.replicas]


CASES = [
    (7, 2, 1, 1, "even", {}),
    (7680 * 3 + 11, 4, 2, 2, "ragged", {}),
    (100_003, 8, 4, 1, "even", {}),
    (100_003, 8, 1, 3, "buckets", {"bucket": 23_456, "misalign": 3}),
    (300_007, 5, 3, 2, "random", {"nseg": 200}),
    (65_536, 16, 4, 3, "random", {"nseg": 21}),
    # shard offsets all multiples of 4 and >= 16 inputs a tile: the variant that keeps gbar in registers and
    # streams with four stages; shard edges fall inside tiles (12,480 = 7680 + 4800)
    (7680 * 13, 8, 2, 1, "even", {}),
    (131_072, 16, 1, 2, "even", {}),
    (7680 * 40, 4, 8, 3, "even", {}),
]


@pytest.mark.parametrize("mode", [COMP, PLAIN])
@pytest.mark.parametrize("psi,n,a,stage,layout,extra", CASES)
def test_single_pass_equals_two_pass(dev, psi, n, a, stage, layout, extra, mode):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=psi % 1000 + n, sigma_g=1e-4, **extra)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    two = gu.upload(c)
    one = gu.upload(c, second_set=True)
    for step in range(3):
        if step:
            w2 = wl.with_(seed=wl.seed + step)
            for q in range(n * a):
                g = sd.bf16_from_bits(synth.grads_bf16(w2, q // a, q % a))
                two.grads[q].copy_(g)
                one.grads[q].copy_(g)
        two.step(A, wl.loss_scale, mode)
        one.step_single_pass(A, wl.loss_scale, mode)
        assert snap_current(one) == snap_two_pass(two), step
        s1, s2 = dp.read_state(one.state), dp.read_state(two.state)
        assert (s1["t"], s1["found_inf"], s1["nonfinite"], s1["b1t"]) == (s2["t"], s2["found_inf"], s2["nonfinite"],
                                                                         s2["b1t"])
        assert s1["cur_set"] == (step + 1) % 2


def test_single_pass_matches_oracle(dev):
    wl = BASE.with_(psi=123_457, n=4, a=2, stage=2, layout="random", nseg=9, seed=11)
    c = gu.make_case(wl)
    b = gu.upload(c, second_set=True)
    b.step_single_pass(dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps), wl.loss_scale)
    torch.cuda.synchronize()
    ms, mm, vv = b.current()
    g = {"master": sd.gather_full(ms, c.segs, wl.psi, c.stage), "m": sd.gather_full(mm, c.segs, wl.psi, c.stage),
         "v": sd.gather_full(vv, c.segs, wl.psi, c.stage), "replicas": [sd.bits_of_bf16(r) for r in b.replicas]}
    st = dp.read_state(b.state)
    g.update(found=st["found_inf"], nonfinite=st["nonfinite"], t=st["t"], error=st["error"])
    gu.assert_matches_oracle(g, gu.run_oracle(c))


@pytest.mark.parametrize("kind", [synth.BF16_POS_INF, synth.BF16_NAN])
def test_single_pass_skip_keeps_state_and_restores_replicas(dev, kind):
    wl = BASE.with_(psi=50_001, n=4, a=2, stage=3, layout="buckets", bucket=9_000, misalign=3, seed=21)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    b = gu.upload(c, second_set=True)
    b.step_single_pass(A, wl.loss_scale)        # an applied step: replicas = bf16(master) from here on
    before = snap_current(b)
    st0 = dp.read_state(b.state)
    b.grads[5].view(torch.int16)[12_345] = kind
    b.step_single_pass(A, wl.loss_scale)
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["t"], st["cur_set"]) == (1, 1, st0["t"], st0["cur_set"])
    assert snap_current(b) == before
    # and the next clean step proceeds exactly like the two-pass path from the same state
    b.grads[5].copy_(sd.bf16_from_bits(c.grads[5]))
    b.step_single_pass(A, wl.loss_scale)
    assert dp.read_state(b.state)["t"] == st0["t"] + 1


def test_single_pass_launches_and_arguments(dev):
    wl = BASE.with_(psi=10_000, n=2, a=1, stage=1)
    c = gu.make_case(wl)
    b = gu.upload(c, second_set=True)
    before = dp.dp_kernel_launches()
    b.step_single_pass(dp.adam(), 1.0)
    assert dp.dp_kernel_launches() - before == 2
    L0 = dp.Layout(0, wl.n, wl.psi, c.segs)
    with pytest.raises(dp.DPError):
        dp.dp_step_single_pass(b.replicas, b.master + b.master1, b.m + b.m1, b.v + b.v1, b.grads, 1, L0, dp.adam(), 1.0,
                               state=b.state)
