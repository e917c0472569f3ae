"""Layouts with more segments than one launch's table holds (-m gpu).

A kernel receives its segment table by value, 1024 segments at most; a larger layout -- one piece per tensor
and rank, or small buckets, the FSDP units of "Data vs Tensor vs Pipeline Parallelism", "FSDP wrapping
granularity" -- runs every kernel as several launches over contiguous runs of 1024 segments.  The skip decision
then spans the launches: the first sets found_inf and the non-finite count, later ones OR and add into them,
and only the last commits.  Checked on every launch path:
  - plain arithmetic: gbar equals the message-passing ring simulation bit for bit (the per-element order does
    not depend on how the segments are grouped into launches), and every path matches the float64 oracle;
  - a non-finite value in the first, a middle or the last run of segments skips the whole step with the exact
    count, t unchanged and every byte of state unchanged;
  - the single pass (ring and tree order), the two-pass tree order, the per-micro-step reduce-scatter and the
    staged calls agree with the oracle on the same layouts.
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

BASE = synth.WORKLOADS["tiny"]
LAYOUTS = [
    # psi, n, a, stage, layout extra: 3000 random segments; 4 x 2200 small misaligned buckets
    (600_011, 8, 2, 3, {"layout": "random", "nseg": 3000}),
    (2_200_007, 4, 3, 2, {"layout": "buckets", "bucket": 1000, "misalign": 3}),
]


def case_of(psi, n, a, stage, extra, seed=71):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, seed=seed, loss_scale=4.0, **extra)
    c = gu.make_case(wl)
    assert len([s for s in c.segs if s[1] > 0]) > dp.DP_KERNEL_SEG
    return wl, c


@pytest.mark.parametrize("psi,n,a,stage,extra", LAYOUTS)
def test_ring_order_and_oracle_over_launches(dev, psi, n, a, stage, extra):
    wl, c = case_of(psi, n, a, stage, extra)
    b = gu.upload(c)
    before = dp.dp_kernel_launches()
    b.step(dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps), wl.loss_scale, dp.DP_SUM_PLAIN)
    torch.cuda.synchronize()
    assert dp.dp_kernel_launches() - before > 2          # several launches per kernel
    ref = brute.ring_gbar(c.grads, wl.n, wl.a, c.segs, wl.psi, wl.loss_scale, "f32")
    got = sd.gather_full(b.gbar, c.segs, wl.psi, 1)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


@pytest.mark.parametrize("path", ["two_pass", "tree", "single_pass", "single_pass_tree", "microstep", "staged"])
@pytest.mark.parametrize("psi,n,a,stage,extra", LAYOUTS)
def test_every_path_matches_the_oracle(dev, psi, n, a, stage, extra, path):
    wl, c = case_of(psi, n, a, stage, extra, seed=72)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    b = gu.upload(c, second_set=path.startswith("single_pass"), micro_acc=path == "microstep")
    S = wl.loss_scale
    if path == "two_pass":
        b.step(A, S)
    elif path == "tree":
        b.step(A, S, dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)
    elif path.startswith("single_pass"):
        b.step_single_pass(A, S, dp.DP_SUM_COMPENSATED | (dp.DP_ORDER_TREE if path.endswith("tree") else 0))
        b.master, b.m, b.v = b.current()
    elif path == "microstep":
        b.step_micro(A, S)
    else:
        acc = [torch.empty(2 * wl.psi, dtype=torch.float32, device=dev) for _ in range(wl.n)]
        for k in range(wl.a):
            dp.dp_accumulate(acc, [b.grad(r, k) for r in range(wl.n)], wl.psi, wl.n, k == 0)
        dp.dp_reduce_scatter_avg(b.gbar, acc, c.layout, S, dp.DP_SUM_COMPENSATED, b.state)
        dp.dp_adam_shard(b.master, b.m, b.v, b.gbar, c.layout, A, b.state)
        dp.dp_allgather_params(b.replicas, b.master, c.layout, b.state)
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


@pytest.mark.parametrize("where", ["first", "middle", "last", "spread"])
@pytest.mark.parametrize("single", [False, True])
def test_skip_spans_the_launches(dev, where, single):
    psi, n, a, stage, extra = LAYOUTS[1]
    wl, c = case_of(psi, n, a, stage, extra, seed=73)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    b = gu.upload(c, second_set=single)
    nz = [s for s in c.segs if s[1] > 0]
    K = dp.DP_KERNEL_SEG
    runs = {"first": [0], "middle": [K + 5], "last": [len(nz) - 1], "spread": [3, K + 1, len(nz) - 2]}[where]
    for j, sidx in enumerate(runs):
        g0, ln, _, _ = nz[sidx]
        b.grad(j % n, j % a)[g0 + ln // 2:g0 + ln // 2 + 1].view(torch.int16).fill_(synth.BF16_POS_INF)
    if single:   # replicas equal bf16(master) before the step, as after any applied step
        dp.dp_allgather_params(b.replicas, b.master, c.layout, b.state)
    before = gu.snapshot(b)
    if single:
        b.step_single_pass(A, wl.loss_scale)
    else:
        b.step(A, wl.loss_scale)
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["t"], st["error"], st["cur_set"]) == (1, len(runs), 0, 0, 0)
    assert gu.snapshot(b) == before
