"""Full-size parity (-m gpu): the workloads at their real parameter counts, in the launch configuration the
benchmark times (dp_step_reduce then dp_step_update), checked against the float64 oracle on sampled elements.

Inputs are generated on the host, chunk by chunk, from the counter-based generator, so the oracle can
regenerate exactly the inputs of any sampled element.  Samples: random elements plus the first and last
element of every segment (shard boundaries, misaligned cuts) and the last elements of the space.  Properties
that hold at any size are checked on the whole run: no skip, no non-finite value, t advanced, and (for one
workload) a full-size skip that leaves the sampled state bit-identical.
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

CHUNK = 1 << 26


def warm_state_by_oracle(b, wl, segs):
    """Warm moments from one prior step (seed + 1000) computed by the oracle for every element, chunk by
    chunk, written into the device shards; returns nothing (the device buffers hold master, m, v at t = 1)."""
    for s in range(0, wl.psi, CHUNK):
        c = min(CHUNK, wl.psi - s)
        idx = np.arange(s, s + c, dtype=np.int64)
        o = gu.oracle_at(wl, idx, prior=True)
        assert o["found"] == 0
        for arr, vals in ((b.master, o["master"]), (b.m, o["m"]), (b.v, o["v"])):
            for g, ln, own, lo in segs:
                a0, a1 = max(g, s), min(g + ln, s + c)
                if a0 < a1:
                    arr[own][lo + (a0 - g):lo + (a1 - g)].copy_(torch.from_numpy(vals[a0 - s:a1 - s]))
    b.state.copy_(torch.frombuffer(bytearray(gu.state_bytes(1, wl.beta1, wl.beta2)), dtype=torch.uint8))


def run_fullsize(wl, samples=200_000, warm=False, inject=False, repeat=0, mode=dp.DP_SUM_COMPENSATED,
                 single=False):
    """single: dp_step_single_pass (two state sets, the step's results in the set it makes current)."""
    segs = synth.layout_of(wl)
    L = dp.Layout(wl.stage, wl.n, wl.psi, segs)
    b = StepBuffers(L, wl.a, second_set=single)
    sd.fill_grads(b.grads, wl)
    t0 = 0
    if warm:
        warm_state_by_oracle(b, wl, segs)
        t0 = 1
    else:
        sd.fill_master(b.master, wl, segs, wl.stage)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)

    def step():
        if single:
            b.step_single_pass(A, wl.loss_scale, mode)
        else:
            b.reduce(A, wl.loss_scale, mode)
            b.update(A)

    step()
    torch.cuda.synchronize()
    st = dp.read_state(b.state)
    assert (st["found_inf"], st["nonfinite"], st["error"], st["t"]) == (0, 0, 0, t0 + 1)

    idx = gu.sample_indices(wl, segs, samples, wl.seed + 17)
    if warm:
        pr = gu.oracle_at(wl, idx, prior=True)
        o = gu.oracle_at(wl, idx, t0=1, m=pr["m"], v=pr["v"], master=pr["master"])
    else:
        o = gu.oracle_at(wl, idx)
    assert (o["found"], o["nonfinite"], o["t"]) == (0, 0, t0 + 1)
    gi = torch.from_numpy(idx).to(b.grads[0].device)
    cm, cmm, cv = b.current() if single else (b.master, b.m, b.v)
    g = {"master": gu.gather_state(cm, segs, idx, wl.stage), "m": gu.gather_state(cmm, segs, idx, wl.stage),
         "v": gu.gather_state(cv, segs, idx, wl.stage),
         "replicas": [sd.bits_of_bf16(r[gi]) for r in b.replicas]}
    gu.assert_close_f32(g["master"], o["master"], "master")
    gu.assert_close_f32(g["m"], o["m"], "m")
    gu.assert_close_f32(g["v"], o["v"], "v")
    gu.assert_replicas(g["replicas"], o["replicas"])

    if repeat and not single:
        # the fixed-order reduction is bit-identical run to run over the whole parameter space
        first = [x.clone() for x in b.gbar]
        for _ in range(repeat):
            b.reduce(A, wl.loss_scale, mode)
            torch.cuda.synchronize()
            for x, y in zip(first, b.gbar):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        del first

    if inject:
        # one +inf in one rank's micro-step at a seeded element: the whole step is skipped
        r, k, i, _ = synth.inject_site(wl, 0)
        b.grad(r, k)[i:i + 1].view(torch.int16).fill_(synth.BF16_POS_INF)
        before = [gu.gather_state(x, segs, idx, wl.stage) for x in (b.current() if single else (b.master, b.m, b.v))]
        reps_before = [sd.bits_of_bf16(x[gi]) for x in b.replicas]
        step()
        torch.cuda.synchronize()
        st2 = dp.read_state(b.state)
        assert (st2["found_inf"], st2["nonfinite"], st2["t"]) == (1, 1, t0 + 1 + (0 if single else repeat))
        after = [gu.gather_state(x, segs, idx, wl.stage) for x in (b.current() if single else (b.master, b.m, b.v))]
        for x, y in zip(before, after):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
        for x, rep in zip(reps_before, b.replicas):
            assert np.array_equal(x, sd.bits_of_bf16(rep[gi]))
    del b
    gc.collect()
    torch.cuda.empty_cache()


def test_fullsize_gpt2_small(dev):
    """123,568,896 params, n=8, a=4, ZeRO-1 even, loss scale 2^16: the benchmark's workload."""
    run_fullsize(synth.WORKLOADS["gpt2_small"], inject=True, repeat=3)


def test_fullsize_gpt2_small_tree_order(dev):
    """The benchmark's workload with the ranks' sums added up the binomial tree instead of the ring."""
    run_fullsize(synth.WORKLOADS["gpt2_small"], inject=True, repeat=2,
                 mode=dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)


def test_fullsize_gpt_1p3b(dev):
    """1,311,082,496 params, n=8, a=1, ZeRO-3 25M buckets with +3-misaligned cuts, warm m/v, t = 2."""
    run_fullsize(synth.WORKLOADS["gpt_1p3b"], warm=True, repeat=3)


def test_fullsize_llama7b_16l(dev):
    """3,238,133,760 params, n=4, a=2, ZeRO-2 even, 1% x100 outliers, loss scale 1 (cold start)."""
    run_fullsize(synth.WORKLOADS["llama7b_16l"])


def test_fullsize_gpt2_small_single_pass(dev):
    """The benchmark's workload through dp_step_single_pass, and a skipped step after it."""
    run_fullsize(synth.WORKLOADS["gpt2_small"], inject=True, single=True)


def test_fullsize_gpt2_small_single_pass_tree_order(dev):
    """The benchmark's workload through dp_step_single_pass in tree order, and a skipped step after it."""
    run_fullsize(synth.WORKLOADS["gpt2_small"], inject=True, single=True,
                 mode=dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)


def test_fullsize_gpt_1p3b_tree_order(dev):
    """The 1.3B list's +3-misaligned 25M-bucket ZeRO-3 layout, warm m/v, with the tree order's two-pass step."""
    run_fullsize(synth.WORKLOADS["gpt_1p3b"], warm=True, mode=dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)


def test_fullsize_llama7b_16l_single_pass_tree_order(dev):
    """The Llama-16L list (n = 4, a = 2, outliers, loss scale 1) through the tree order's single pass."""
    run_fullsize(synth.WORKLOADS["llama7b_16l"], single=True, mode=dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)


def test_fullsize_gpt_1p3b_single_pass(dev):
    """The 1.3B list's +3-misaligned 25M-bucket ZeRO-3 layout through the single pass, warm m/v."""
    run_fullsize(synth.WORKLOADS["gpt_1p3b"], warm=True, single=True)


def test_fullsize_llama7b_16l_single_pass(dev):
    """Llama-16L (3.2B params, heavy-tailed gradients, cold start) through the single pass."""
    run_fullsize(synth.WORKLOADS["llama7b_16l"], single=True)


@pytest.mark.parametrize("psi,n,a,layout", [((1 << 28) + 5, 4, 8, "ragged"), (10 ** 9, 8, 8, "even")])
def test_fullsize_sweep_extremes(dev, psi, n, a, layout):
    """The flat sweep's large cases, including its largest: 10^9 params x 8 ranks x 8 micro-steps."""
    wl = [w for w in synth.sweep_cases() if w.psi == psi and w.n == n and w.a == a and w.layout == layout][0]
    free, _ = torch.cuda.mem_get_info()
    need = 2 * n * a * psi + 2 * n * psi + 16 * psi + (1 << 30)
    assert free > need, "device memory: need %.1f GB, free %.1f GB" % (need / 1e9, free / 1e9)
    run_fullsize(wl, samples=100_000)
