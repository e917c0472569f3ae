"""GPU path vs the float64 oracle, element by element, through the C ABI (-m gpu).

Sizes span several 7680-element tiles with ragged tails; layouts cover even, ragged, random multi-segment,
bucketed +3-misaligned and empty shards; every ZeRO stage; both reduction modes; skip injection; staged vs
fused; determinism; the bounded-wait self-test; CUDA graph capture.
"""
import numpy as np
import pytest
import torch

import oracle
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


def step_and_compare(c, mode=COMP, scale=1.0):
    b = gu.upload(c)
    b.step(adam_of(c.wl), c.wl.loss_scale, mode)
    g = gu.gpu_result(c, b)
    o = gu.run_oracle(c)
    gu.assert_matches_oracle(g, o, scale)
    return b, g, o


@pytest.mark.parametrize("mode", [COMP, PLAIN])
def test_tiny_workload(dev, mode):
    """The 2^20-parameter, n=2, a=1, ZeRO-1 workload at its full size."""
    step_and_compare(gu.make_case(BASE), mode)


CASES = [
    # psi, n, a, stage, layout, extra
    (1, 1, 1, 1, "even", {}),
    (7, 2, 1, 1, "even", {}),
    (4096, 2, 2, 1, "even", {}),
    (4097, 3, 2, 2, "even", {}),
    (3 * 4096 + 5, 4, 4, 3, "ragged", {}),
    (65536 + 3, 8, 1, 1, "random", {"nseg": 37}),
    (100_003, 8, 4, 2, "buckets", {"bucket": 20_000, "misalign": 3}),
    (50_001, 5, 3, 3, "random", {"nseg": 11}),
    (40_960, 16, 4, 1, "even", {}),
    (33_333, 2, 8, 2, "ragged", {}),
    (8 * 4096, 8, 8, 1, "even", {}),
    (123_457, 4, 2, 0, "random", {"nseg": 9}),
]


@pytest.mark.parametrize("mode", [COMP, PLAIN])
@pytest.mark.parametrize("psi,n,a,stage,layout,extra", CASES)
def test_small_cases(dev, psi, n, a, stage, layout, extra, mode):
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=psi + n, sigma_g=1e-4,
                    loss_scale=float(1 << (n % 5)), **extra)
    step_and_compare(gu.make_case(wl), mode)


def test_ragged_layout_with_empty_shards(dev):
    psi, n = 20_000, 6
    segs = [(0, 0, 0, 0), (0, 9_000, 1, 0), (9_000, 0, 2, 0), (9_000, 11_000, 3, 0), (20_000, 0, 4, 0),
            (20_000, 0, 5, 0)]
    wl = BASE.with_(psi=psi, n=n, a=2, stage=2, seed=77)
    step_and_compare(gu.make_case(wl, segs=segs))


def test_many_segments_large_table(dev):
    """More than 32 segments selects the large segment-table kernels."""
    wl = BASE.with_(psi=400_000, n=8, a=2, stage=3, layout="random", nseg=1000, seed=5)
    step_and_compare(gu.make_case(wl))


@pytest.mark.parametrize("S", [2.0 ** 8, 2.0 ** 12, 2.0 ** 16, 2.0 ** 20, 2.0 ** 24, 3.0])
def test_loss_scales(dev, S):
    wl = BASE.with_(psi=30_000, n=3 if S == 3.0 else 4, a=2, loss_scale=S, sigma_g=1e-3 * S / 2 ** 16, seed=int(S) % 97)
    step_and_compare(gu.make_case(wl))


def test_heavy_tail_outliers(dev):
    wl = synth.WORKLOADS["llama7b_16l"].with_(psi=200_003)
    step_and_compare(gu.make_case(wl))


def test_warm_state_misaligned_buckets(dev):
    """The 1.3B workload's layout pattern at reduced size: 25M buckets scaled down, +3-misaligned cuts, warm
    m/v from one prior step computed by the oracle, measured step t = 2."""
    wl = synth.WORKLOADS["gpt_1p3b"].with_(psi=1_000_003, bucket=120_000)
    segs = synth.layout_of(wl)
    prior = gu.make_case(wl.with_(seed=wl.seed + 1000), segs=segs)
    po = gu.run_oracle(prior)
    c = gu.make_case(wl, segs=segs, t=1, m=po["m"], v=po["v"], master=po["master"])
    step_and_compare(c)


def test_two_chained_steps(dev):
    wl = BASE.with_(psi=77_777, n=4, a=2, stage=1, layout="ragged", seed=3)
    c = gu.make_case(wl)
    b = gu.upload(c)
    A = adam_of(wl)
    b.step(A, wl.loss_scale)
    wl2 = wl.with_(seed=4)
    c2grads = [synth.grads_bf16(wl2, r, k) for r in range(wl.n) for k in range(wl.a)]
    for q, g in enumerate(c2grads):
        b.grads[q].copy_(sd.bf16_from_bits(g))
    b.step(A, wl.loss_scale)
    g = gu.gpu_result(c, b)
    o1 = gu.run_oracle(c)
    c2 = gu.Case(wl, c.segs, c.stage, c.layout, c2grads, o1["master"], o1["m"], o1["v"], 1)
    o2 = gu.run_oracle(c2)
    gu.assert_matches_oracle(g, o2, scale=2.0)


@pytest.mark.parametrize("mode,arith", [(PLAIN, "f32"), (COMP, "f32chain")])
def test_reduction_order_matches_ring_simulation(dev, mode, arith):
    """gbar equals, bit for bit, what the message-passing ring computes as every chunk travels s+1 -> ... -> s:
    plain, each rank adds the sum of its micro-steps; compensated, each rank folds its micro-steps one at a time
    into the travelling (hi, lo) pair."""
    wl = BASE.with_(psi=20_011, n=5, a=3, stage=1, layout="random", nseg=7, seed=21, sigma_g=1e-2,
                    tail_p=0.05, tail_mult=1e4, loss_scale=8.0)
    c = gu.make_case(wl)
    b = gu.upload(c)
    b.step(adam_of(wl), wl.loss_scale, mode)
    torch.cuda.synchronize()
    ref = brute.ring_gbar(c.grads, wl.n, wl.a, c.segs, wl.psi, wl.loss_scale, arith)
    got = np.zeros(wl.psi, np.float32)
    host = [t.cpu().numpy() for t in b.gbar]
    for g0, ln, o, lo in c.segs:
        got[g0:g0 + ln] = host[o][lo:lo + ln]
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("mode,arith", [(PLAIN, "f32"), (COMP, "f32chain")])
@pytest.mark.parametrize("n,a,layout", [(3, 3, "even"), (3, 1, "ragged"), (1, 1, "even"), (7, 1, "random")])
def test_odd_input_count_matches_ring_simulation(dev, mode, arith, n, a, layout):
    """Pass A streams two inputs a stage; with n*a odd the last stage of every tile carries one.  Many whole
    tiles (the guard-free loop) plus segment edges and a ragged buffer tail (the general loop): gbar equals the
    simulated ring bit for bit, and the step matches the oracle."""
    wl = BASE.with_(psi=7680 * 23 + 13, n=n, a=a, stage=1, layout=layout, nseg=5, seed=61 + n + a, sigma_g=1e-2,
                    tail_p=0.02, tail_mult=1e3, loss_scale=4.0)
    c = gu.make_case(wl)
    b = gu.upload(c)
    b.step(adam_of(wl), wl.loss_scale, mode)
    torch.cuda.synchronize()
    ref = brute.ring_gbar(c.grads, wl.n, wl.a, c.segs, wl.psi, wl.loss_scale, arith)
    got = sd.gather_full(b.gbar, c.segs, wl.psi, 1)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


def test_compensated_gbar_is_nearly_exact(dev):
    """Compensated reduction: gbar within 1 ulp of the exactly rounded average (n S a power of two)."""
    wl = synth.WORKLOADS["llama7b_16l"].with_(psi=300_000, a=8, seed=8)
    c = gu.make_case(wl)
    b = gu.upload(c)
    b.step(adam_of(wl), wl.loss_scale, COMP)
    torch.cuda.synchronize()
    ex = oracle.reduce(wl.psi, wl.n, wl.a, c.grads, wl.loss_scale, threads=8)["gbar"]
    got = np.zeros(wl.psi, np.float32)
    host = [t.cpu().numpy() for t in b.gbar]
    for g0, ln, o, lo in c.segs:
        got[g0:g0 + ln] = host[o][lo:lo + ln]
    # Sum2 bound (Ogita, Rump, Oishi 2005): one ulp of the result plus gamma_{na}^2 times the sum of |x|.
    ulp = np.spacing(np.abs(ex.astype(np.float32))).astype(np.float64)
    absum = np.sum([np.abs(brute.bf16_bits_to_f32(x).astype(np.float64)) for x in c.grads], axis=0)
    gamma = wl.n * wl.a * 2.0 ** -24
    tol = ulp + 2 * gamma * gamma * absum / (wl.n * wl.loss_scale)
    assert np.all(np.abs(got.astype(np.float64) - ex) <= tol)


@pytest.mark.parametrize("mode", [COMP, PLAIN])
def test_fused_equals_staged(dev, mode):
    """The staged calls (accumulate per micro-step, reduce-scatter, Adam, all-gather) against dp_step.  Plain: the
    same fp32 operations in the same order, so identical bits.  Compensated: the staged form keeps one (hi, lo)
    accumulator per rank and combines the ranks' pairs, the fused one carries a single pair through all inputs,
    so they may differ by rounding; each step matches the oracle."""
    wl = BASE.with_(psi=90_001, n=4, a=3, stage=2, layout="random", nseg=13, seed=31)
    c = gu.make_case(wl)
    A = adam_of(wl)
    fused = gu.upload(c)
    fused.step(A, wl.loss_scale, mode)
    staged = gu.upload(c)
    acc = [torch.empty(int(dp.LIB.dp_acc_elems(wl.psi, mode)), dtype=torch.float32, device=dev)
           for _ in range(wl.n)]
    for k in range(wl.a):
        dp.dp_accumulate(acc, [staged.grad(r, k) for r in range(wl.n)], wl.psi, wl.n, k == 0, mode)
    dp.dp_reduce_scatter_avg(staged.gbar, acc, c.layout, wl.loss_scale, mode, staged.state)
    dp.dp_adam_shard(staged.master, staged.m, staged.v, staged.gbar, c.layout, A, staged.state)
    dp.dp_allgather_params(staged.replicas, staged.master, c.layout, staged.state)
    if mode == PLAIN:
        assert gu.snapshot(fused) == gu.snapshot(staged)
        for x, y in zip(fused.gbar, staged.gbar):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    else:
        gu.assert_matches_oracle(gu.gpu_result(c, fused), gu.run_oracle(c))
    sf, ss = dp.read_state(fused.state), dp.read_state(staged.state)
    assert (sf["t"], sf["found_inf"], sf["nonfinite"], sf["b1t"], sf["b2t"]) == \
           (ss["t"], ss["found_inf"], ss["nonfinite"], ss["b1t"], ss["b2t"])
    gu.assert_matches_oracle(gu.gpu_result(c, staged), gu.run_oracle(c))


def test_stages_bitwise_equal(dev):
    """Sharding changes the storage layout, not the update: stage 0 (full replicas of the state) and stages
    1, 2, 3 produce identical bits."""
    wl = BASE.with_(psi=60_013, n=4, a=2, layout="random", nseg=9, seed=41)
    segs = synth.layout_of(wl)
    outs = []
    for stage in range(4):
        c = gu.make_case(wl, stage=stage, segs=segs)
        b = gu.upload(c)
        b.step(adam_of(wl), wl.loss_scale)
        g = gu.gpu_result(c, b)
        if stage == 0:
            for x in g["all_master"][1:]:
                assert np.array_equal(x.view(np.uint32), g["all_master"][0].view(np.uint32))
        outs.append((g["master"].tobytes(), g["m"].tobytes(), g["v"].tobytes(),
                     b"".join(r.tobytes() for r in g["replicas"])))
    assert all(o == outs[0] for o in outs[1:])


@pytest.mark.parametrize("mode", [COMP, PLAIN])
def test_deterministic_runs(dev, mode):
    wl = BASE.with_(psi=250_007, n=8, a=4, stage=1, layout="ragged", seed=51, loss_scale=65536.0)
    c = gu.make_case(wl)
    ref = None
    for _ in range(10):
        b = gu.upload(c)
        b.step(adam_of(wl), wl.loss_scale, mode)
        snap = gu.snapshot(b) + [t.cpu().numpy().tobytes() for t in b.gbar]
        if ref is None:
            ref = snap
        assert snap == ref


@pytest.mark.parametrize("where", ["first", "last", "boundary", "misaligned_tail", "other_rank_tile"])
@pytest.mark.parametrize("kind", [synth.BF16_POS_INF, synth.BF16_NEG_INF, synth.BF16_NAN])
def test_skip_on_injected_nonfinite(dev, where, kind):
    wl = BASE.with_(psi=3 * 4096 + 13, n=4, a=2, stage=3, layout="buckets", bucket=5000, misalign=3, seed=61)
    c = gu.make_case(wl, t=3, m=np.full(wl.psi, 1e-5, np.float32), v=np.full(wl.psi, 1e-9, np.float32))
    segs = c.segs
    idx = {"first": 0, "last": wl.psi - 1, "boundary": segs[1][0], "misaligned_tail": wl.psi - 5,
           "other_rank_tile": segs[5][0] + 1}[where]
    r, k = (2, 1) if where != "first" else (0, 0)
    c.grads[r * wl.a + k][idx] = kind
    b = gu.upload(c)
    for rep in b.replicas:
        rep.view(torch.int16).fill_(0x1234)
    before = gu.snapshot(b)
    st0 = dp.read_state(b.state)
    b.step(adam_of(wl), wl.loss_scale)
    assert b.status() == (1, 0)
    st = dp.read_state(b.state)
    assert st["t"] == st0["t"] == 3 and st["nonfinite"] == 1 and st["b1t"] == st0["b1t"]
    assert gu.snapshot(b) == before
    o = gu.run_oracle(c)
    assert o["found"] == 1 and o["nonfinite"] == 1
    # a clean step afterwards still matches the oracle
    c.grads[r * wl.a + k][idx] = synth.grads_bf16(wl, r, k, idx, 1)[0]
    b.grads[r * wl.a + k].copy_(sd.bf16_from_bits(c.grads[r * wl.a + k]))
    b.step(adam_of(wl), wl.loss_scale)
    gu.assert_matches_oracle(gu.gpu_result(c, b), gu.run_oracle(c))


def test_overflow_of_finite_inputs_skips(dev):
    wl = BASE.with_(psi=10_000, n=2, a=1, seed=71)
    c = gu.make_case(wl)
    c.grads[0][1234] = 0x7F62
    c.grads[1][1234] = 0x7F62
    b = gu.upload(c)
    before = gu.snapshot(b)
    b.step(adam_of(wl), wl.loss_scale)
    assert b.status() == (1, 0)
    assert gu.snapshot(b) == before
    assert gu.run_oracle(c)["found"] == 1


def test_workspace_equals_caller_shards(dev):
    wl = BASE.with_(psi=70_001, n=3, a=2, stage=2, layout="random", nseg=8, seed=81)
    c = gu.make_case(wl)
    b1 = gu.upload(c)
    b1.step(adam_of(wl), wl.loss_scale)
    b2 = gu.upload(c)
    ws = torch.empty(c.layout.workspace_size(), dtype=torch.uint8, device=dev)
    dp.dp_step(b2.replicas, b2.master, b2.m, b2.v, b2.grads, wl.a, c.layout, adam_of(wl), wl.loss_scale,
               ws=ws, state=b2.state)
    assert gu.snapshot(b1) == gu.snapshot(b2)


def test_empty_parameter_space(dev):
    L = dp.Layout(1, 2, 0, [])
    st = dp.new_state(dev)
    dummy = [torch.empty(8, dtype=torch.float32, device=dev) for _ in range(2)]
    reps = [torch.empty(8, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    grads = [torch.empty(8, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dp.dp_step(reps, dummy, dummy, dummy, grads, 1, L, dp.adam(), 1.0, gbar_shard=dummy, state=st)
    s = dp.read_state(st)
    assert (s["t"], s["found_inf"], s["nonfinite"], s["error"]) == (1, 0, 0, 0)


def test_bounded_wait_times_out_and_context_survives(dev):
    st = dp.new_state(dev)
    dp.dp_selftest_wait_timeout(st, 20_000_000)
    assert dp.dp_read_status(st) == (0, dp.DP_ERR_TIMEOUT)
    # a step on a state with a recorded error is skipped, and nothing is written
    wl = BASE.with_(psi=5000, n=2, a=1, seed=91)
    c = gu.make_case(wl)
    b = gu.upload(c)
    before = gu.snapshot(b)
    dp.dp_selftest_wait_timeout(b.state, 1_000_000)
    b.step(adam_of(wl), wl.loss_scale)
    assert b.status() == (1, dp.DP_ERR_TIMEOUT)
    assert gu.snapshot(b) == before
    # the context is still usable: a fresh state steps normally
    b2 = gu.upload(c)
    b2.step(adam_of(wl), wl.loss_scale)
    gu.assert_matches_oracle(gu.gpu_result(c, b2), gu.run_oracle(c))


def test_cuda_graph_capture_replays_the_step(dev):
    wl = BASE.with_(psi=50_000, n=4, a=2, stage=1, seed=101)
    c = gu.make_case(wl)
    A = adam_of(wl)
    direct = gu.upload(c)
    graphed = gu.upload(c)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        graphed.step(A, wl.loss_scale, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        direct.step(A, wl.loss_scale)
        g.replay()
    torch.cuda.synchronize()
    assert gu.snapshot(direct) == gu.snapshot(graphed)
    assert dp.read_state(direct.state)["t"] == dp.read_state(graphed.state)["t"] == 3


def test_kernel_launch_count(dev):
    wl = BASE.with_(psi=10_000, n=2, a=1)
    b = gu.upload(gu.make_case(wl))
    before = dp.dp_kernel_launches()
    b.step(adam_of(wl), 1.0)
    assert dp.dp_kernel_launches() - before == 2
