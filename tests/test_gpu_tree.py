"""The tree reduction order on the GPU (-m gpu): DP_ORDER_TREE through the same entry points.

Its averaged gradient must equal, bit for bit, the simulated binomial tree of the oracle's brute force (both
arithmetics), and its step must match the float64 oracle within the same tolerances as the ring order.  The
fused kernel and the staged calls agree bit for bit, runs repeat exactly, and a non-finite input skips.
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

COMP, PLAIN, TREE = dp.DP_SUM_COMPENSATED, dp.DP_SUM_PLAIN, dp.DP_ORDER_TREE
BASE = synth.WORKLOADS["tiny"]


def adam_of(wl):
    return dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)


def gbar_full(b, c):
    torch.cuda.synchronize()
    return sd.gather_full(b.gbar, c.segs, c.wl.psi, 1)


CASES = [
    # psi, n, a, stage, layout, extra
    (1, 1, 1, 1, "even", {}),
    (9, 3, 1, 1, "even", {}),
    (4099, 2, 2, 1, "even", {}),
    (3 * 7680 + 5, 5, 3, 2, "ragged", {}),
    (65536 + 3, 7, 1, 3, "random", {"nseg": 29}),
    (100_003, 8, 4, 1, "buckets", {"bucket": 20_000, "misalign": 3}),
    (40_961, 16, 4, 2, "even", {}),
    (33_335, 13, 2, 0, "random", {"nseg": 9}),
    (20_000, 6, 8, 1, "ragged", {}),
    (2 * 7680 + 1919, 4, 3, 3, "random", {"nseg": 7}),
    (3 * 7680 + 961, 9, 1, 1, "ragged", {}),
    (50_001, 12, 2, 2, "buckets", {"bucket": 4_000, "misalign": 3}),
    (30_721, 15, 3, 3, "even", {}),
    # n = 9, 10: the second group's micro-steps packed eight and four to a stage (a = 7: one partial stage;
    # a = 6: a full and a partial one)
    (20_011, 9, 7, 1, "even", {}),
    (2 * 7680 + 9, 10, 6, 2, "ragged", {}),
]


@pytest.mark.parametrize("psi,n,a,stage,layout,extra", CASES)
@pytest.mark.parametrize("arith", [PLAIN, COMP])
def test_tree_gbar_equals_simulated_tree(dev, psi, n, a, stage, layout, extra, arith):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=500 + n, sigma_g=1.0, **extra)
    c = gu.make_case(wl)
    b = gu.upload(c)
    b.reduce(adam_of(wl), wl.loss_scale, arith | TREE)
    want = brute.tree_gbar(c.grads, n, a, c.segs, psi, wl.loss_scale, "f32pair" if arith == COMP else "f32")
    got = gbar_full(b, c)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("psi,n,a,stage,layout,extra", CASES)
def test_tree_step_matches_oracle(dev, psi, n, a, stage, layout, extra):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=600 + n, **extra)
    c = gu.make_case(wl)
    b = gu.upload(c)
    b.step(adam_of(wl), wl.loss_scale, COMP | TREE)
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


def test_tree_on_the_tiny_workload_and_loss_scale_one(dev):
    """The 2^20-parameter, n=2 workload, and a loss-scale-1 cold start with outliers, compensated tree."""
    for wl in (BASE, BASE.with_(psi=300_007, n=6, a=2, loss_scale=1.0, tail_p=0.01, tail_mult=100.0, seed=9)):
        c = gu.make_case(wl)
        b = gu.upload(c)
        b.step(adam_of(wl), wl.loss_scale, COMP | TREE)
        gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


@pytest.mark.parametrize("arith", [PLAIN, COMP])
def test_tree_fused_equals_staged(dev, arith):
    wl = BASE.with_(psi=70_001, n=5, a=3, stage=2, layout="random", nseg=17, seed=41, sigma_g=1.0)
    c = gu.make_case(wl)
    fused = gu.upload(c)
    fused.reduce(adam_of(wl), wl.loss_scale, arith | TREE)
    staged = gu.upload(c)
    acc_elems = wl.psi * (2 if arith == COMP else 1)
    acc = [torch.empty(acc_elems, dtype=torch.float32, device="cuda") for _ in range(wl.n)]
    for k in range(wl.a):
        dp.dp_accumulate(acc, [staged.grad(r, k) for r in range(wl.n)], wl.psi, wl.n, k == 0, arith | TREE)
    dp.dp_reduce_scatter_avg(staged.gbar, acc, c.layout, wl.loss_scale, arith | TREE, staged.state)
    assert np.array_equal(gbar_full(fused, c).view(np.uint32), gbar_full(staged, c).view(np.uint32))
    a_, b_ = dp.read_state(fused.state), dp.read_state(staged.state)
    assert (a_["found_inf"], a_["nonfinite"]) == (b_["found_inf"], b_["nonfinite"]) == (0, 0)


def test_tree_deterministic_and_skips(dev):
    wl = BASE.with_(psi=3_000_017, n=8, a=4, stage=1, layout="ragged", seed=77)
    c = gu.make_case(wl)
    b = gu.upload(c)
    A = adam_of(wl)
    b.reduce(A, wl.loss_scale, COMP | TREE)
    first = [x.clone() for x in b.gbar]
    for _ in range(3):
        b.reduce(A, wl.loss_scale, COMP | TREE)
        torch.cuda.synchronize()
        for x, y in zip(first, b.gbar):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    # a NaN in one micro-step of one rank: the whole step is skipped, state unchanged
    b2 = gu.upload(c)
    before = gu.snapshot(b2)
    b2.grad(5, 2)[wl.psi - 1:wl.psi].view(torch.int16).fill_(synth.BF16_NAN)
    b2.step(A, wl.loss_scale, COMP | TREE)
    st = dp.read_state(b2.state)
    assert (st["found_inf"], st["nonfinite"], st["t"]) == (1, 1, 0)
    assert gu.snapshot(b2) == before


def test_tree_with_device_loss_scale(dev):
    """dp_step_scaled with the tree order equals dp_step with the tree order at the same scale."""
    S = 2.0 ** 10
    wl = BASE.with_(psi=50_009, n=4, a=2, stage=2, layout="ragged", loss_scale=S, seed=88)
    c = gu.make_case(wl)
    A = adam_of(wl)
    fixed = gu.upload(c)
    fixed.step(A, S, COMP | TREE)
    scaled = gu.upload(c)
    dp.dp_scaler_init(scaled.state, S)
    scaled.step_scaled(A, dp.scaler(2.0, 0.5, 3, 1.0, 2.0 ** 20), COMP | TREE)
    assert gu.snapshot(fixed) == gu.snapshot(scaled)


def test_tree_rejected_where_unsupported(dev):
    """The per-micro-step reduce-scatter runs in ring order only, and dp_step takes no deferred commit."""
    wl = BASE.with_(psi=5000, n=2, a=2)
    c = gu.make_case(wl)
    b = gu.upload(c, micro_acc=True)
    with pytest.raises(dp.DPError):
        b.step_micro(adam_of(wl), 1.0, COMP | TREE)
    with pytest.raises(dp.DPError):
        b.step(adam_of(wl), 1.0, COMP | TREE | dp.DP_DEFER_COMMIT)


# ---------------------------------------------------------------- the tree order's single pass

SP_CASES = [
    # psi, n, a, stage, layout, extra -- every element class (n = 1: 16 elements a thread, n = 2: 8, n >= 3: 4)
    # and group count (n <= 4: one group of four, up to 16: four)
    (1, 1, 1, 1, "even", {}),
    (7, 2, 1, 1, "even", {}),
    (7680 * 3 + 11, 3, 2, 2, "ragged", {}),
    (7680 * 5 + 1, 4, 8, 3, "even", {}),
    (300_007, 5, 3, 2, "random", {"nseg": 200}),
    (30_000, 6, 1, 1, "random", {"nseg": 30}),
    (100_003, 8, 4, 1, "even", {}),
    (100_003, 8, 1, 3, "buckets", {"bucket": 23_456, "misalign": 3}),
    (50_001, 9, 2, 1, "ragged", {}),
    (70_001, 12, 3, 2, "buckets", {"bucket": 9_999, "misalign": 1}),
    (40_961, 13, 2, 3, "even", {}),
    (65_536, 16, 4, 3, "random", {"nseg": 21}),
]


def snap_current(b):
    torch.cuda.synchronize()
    ms, mm, vv = b.current()
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in ms + mm + vv + b.replicas]


def snap_two_pass(b):
    torch.cuda.synchronize()
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in b.master + b.m + b.v + b.replicas]


@pytest.mark.parametrize("arith", [COMP, PLAIN])
@pytest.mark.parametrize("psi,n,a,stage,layout,extra", SP_CASES)
def test_tree_single_pass_equals_two_pass_tree(dev, psi, n, a, stage, layout, extra, arith):
    """dp_step_single_pass in tree order gives exactly dp_step's tree-order results over three steps with new
    gradients each time: the same gbar feeds the same Adam, so master/m/v (the current set), the replicas and
    the step state agree bit for bit."""
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=700 + n + psi % 97, sigma_g=1e-3, **extra)
    c = gu.make_case(wl)
    A = adam_of(wl)
    two = gu.upload(c)
    one = gu.upload(c, second_set=True)
    for step in range(3):
        if step:
            w2 = wl.with_(seed=wl.seed + step)
            for q in range(n * a):
                g = sd.bf16_from_bits(synth.grads_bf16(w2, q // a, q % a))
                two.grads[q].copy_(g)
                one.grads[q].copy_(g)
        two.step(A, wl.loss_scale, arith | TREE)
        one.step_single_pass(A, wl.loss_scale, arith | TREE)
        assert snap_current(one) == snap_two_pass(two), step
        s1, s2 = dp.read_state(one.state), dp.read_state(two.state)
        assert (s1["t"], s1["found_inf"], s1["nonfinite"], s1["error"]) == (s2["t"], s2["found_inf"], s2["nonfinite"],
                                                                          s2["error"]) == (step + 1, 0, 0, 0)
        assert s1["cur_set"] == (step + 1) % 2


def test_tree_single_pass_matches_oracle(dev):
    wl = BASE.with_(psi=123_457, n=8, a=2, stage=2, layout="random", nseg=9, seed=12, loss_scale=2.0 ** 12)
    c = gu.make_case(wl)
    b = gu.upload(c, second_set=True)
    b.step_single_pass(adam_of(wl), wl.loss_scale, COMP | TREE)
    torch.cuda.synchronize()
    b.master, b.m, b.v = b.current()
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


@pytest.mark.parametrize("n", [3, 8, 11])
def test_tree_single_pass_skip_keeps_state_and_restores_replicas(dev, n):
    wl = BASE.with_(psi=50_001, n=n, a=2, stage=3, layout="buckets", bucket=9_000, misalign=3, seed=22)
    c = gu.make_case(wl)
    A = adam_of(wl)
    b = gu.upload(c, second_set=True)
    b.step_single_pass(A, wl.loss_scale, COMP | TREE)    # an applied step: replicas = bf16(master) from here on
    before = snap_current(b)
    st0 = dp.read_state(b.state)
    b.grads[2 * n - 1].view(torch.int16)[12_345] = synth.BF16_NAN
    b.step_single_pass(A, wl.loss_scale, COMP | TREE)
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["t"], st["cur_set"]) == (1, 1, st0["t"], st0["cur_set"])
    assert snap_current(b) == before
