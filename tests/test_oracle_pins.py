"""Pins of the float64 oracle against things other than itself (CPU only).

Each test ties one part of the oracle to a library routine, a closed form, an
invariant the distributed-training pages state, or brute force, so that a
dropped term, a wrong sign or index, or a transposed operand fails one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from oracle import brute, ring

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


def f32(x):
    return float(np.float32(x))


def bits_of(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def bf16_bits(vals):
    """bf16 bit patterns of values that are exactly representable in bf16."""
    a = np.asarray(vals, dtype=np.float32)
    b = a.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def make_state(psi, n, stage, segs, master_full, m_full=None, v_full=None):
    """Shard arrays (stage 1-3) or full per-rank arrays (stage 0) from full-length values."""
    if stage == 0:
        lens = [psi] * n
    else:
        lens = synth.shard_lengths(segs, n)
    M = [np.zeros(L, np.float32) for L in lens]
    Mm = [np.zeros(L, np.float32) for L in lens]
    Vv = [np.zeros(L, np.float32) for L in lens]
    for r in range(n):
        if stage == 0:
            M[r][:] = master_full
            if m_full is not None:
                Mm[r][:] = m_full
                Vv[r][:] = v_full
    if stage != 0:
        for g, ln, o, lo in segs:
            M[o][lo:lo + ln] = master_full[g:g + ln]
            if m_full is not None:
                Mm[o][lo:lo + ln] = m_full[g:g + ln]
                Vv[o][lo:lo + ln] = v_full[g:g + ln]
    return M, Mm, Vv


def gather_full(arrs, segs, psi, stage, rank=0):
    if stage == 0:
        return arrs[rank].copy()
    out = np.zeros(psi, np.float32)
    for g, ln, o, lo in segs:
        out[g:g + ln] = arrs[o][lo:lo + ln]
    return out


def run_oracle(psi, n, a, stage, segs, grads, master_full, m_full=None, v_full=None, t=0, S=1.0,
               lr=LR, b1=B1, b2=B2, eps=EPS):
    M, Mm, Vv = make_state(psi, n, stage, segs, master_full, m_full, v_full)
    reps = [np.zeros(psi, np.uint16) for _ in range(n)]
    res = oracle.step(psi, n, a, stage, segs, grads, M, Mm, Vv, reps, lr, b1, b2, eps, S, t)
    return res, M, Mm, Vv, reps


# ---------------------------------------------------------------- reduction

def test_sum_matches_fsum_library():
    """The float64 reduction equals math.fsum (correctly rounded) on generated bf16 gradients."""
    wl = synth.WORKLOADS["gpt2_small"].with_(psi=3000)
    grads = [synth.grads_bf16(wl, r, k, 0, wl.psi) for r in range(wl.n) for k in range(wl.a)]
    red = oracle.reduce(wl.psi, wl.n, wl.a, grads, wl.loss_scale)
    vals = np.stack([brute.bf16_bits_to_f32(g).astype(np.float64) for g in grads])
    nS = wl.n * wl.loss_scale
    ref = np.array([math.fsum(vals[:, i]) / nS for i in range(wl.psi)])
    assert np.array_equal(red["gbar"], ref)


def test_sum_matches_exact_rational():
    """Brute force with exact rationals on tiny inputs, including a non-power-of-two n."""
    wl = synth.WORKLOADS["tiny"].with_(psi=97, n=3, a=3, loss_scale=8.0, tail_p=0.2, tail_mult=1e4)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    red = oracle.reduce(wl.psi, wl.n, wl.a, grads, wl.loss_scale)
    ex = brute.exact_gbar(grads, wl.n, wl.a, wl.loss_scale)
    assert np.array_equal(red["gbar"], ex)


def test_global_batch_example_256_samples():
    """b=4 samples per micro-step, a=8 micro-steps, n=8 replicas: one update consumes 4 x 8 x 8 = 256
    samples ("Distributed Training", worked example).  Integer-valued per-sample gradients make every
    sum exact, so the oracle's gbar times n must equal the plain sum of all 256 sample gradients."""
    b, n, a, psi = 4, 8, 8, 33
    rng = np.random.default_rng(7)
    samples = rng.integers(-20, 21, size=(n, a, b, psi)).astype(np.float32)   # 256 sample gradients
    grads = [bf16_bits(samples[r, k].sum(axis=0)) for r in range(n) for k in range(a)]
    red = oracle.reduce(psi, n, a, grads, 1.0)
    total = samples.reshape(-1, psi).sum(axis=0).astype(np.float64)
    assert samples.reshape(-1, psi).shape[0] == 256
    assert np.array_equal(red["gbar"] * n, total)


def test_ring_f64_matches_oracle_sum():
    """The message-passing ring (float64 hops) reduces to the same values the oracle sums directly."""
    wl = synth.WORKLOADS["tiny"].with_(psi=1500, n=5, a=2, loss_scale=2.0)
    segs = synth.layout_random(wl.psi, wl.n, 11, 2)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    red = oracle.reduce(wl.psi, wl.n, wl.a, grads, wl.loss_scale)
    loc = brute.local_accumulate(grads, wl.n, wl.a, "f64")
    rg = ring.Ring(wl.n, segs, wl.psi)
    out = rg.reduce_scatter(loc, arith="f64")
    full = np.zeros(wl.psi)
    for s in range(wl.n):
        rg._put(full, s, out[s])
    assert np.array_equal(full / (wl.n * wl.loss_scale), red["gbar"])


def test_ring_order_is_owner_plus_one_first():
    """Order matters in fp32 (page: floating-point addition is not associative).  With contributions
    2^24 on rank s+1, then 1 on each other rank and -2^24 on the owner... the float32 ring must absorb
    the ones (2^24 + 1 rounds to 2^24), which only happens if the chunk starts at rank s+1."""
    n, psi = 4, 4
    segs = synth.layout_even(psi, n)                  # element s owned by rank s
    big = np.float32(2 ** 24)
    loc = []
    for r in range(n):
        x = np.ones(psi, np.float32)
        for s in range(n):
            if r == (s + 1) % n:
                x[s] = big
            if r == s:
                x[s] = -big
        loc.append(x)
    rg = ring.Ring(n, segs, psi)
    out = rg.reduce_scatter(loc, arith="f32")
    for s in range(n):
        assert out[s][0] == 0.0                        # ((2^24 + 1) + 1) - 2^24 in fp32
    ex = rg.reduce_scatter(loc, arith="f64", phase="x")
    for s in range(n):
        assert ex[s][0] == 2.0                         # exact


# ---------------------------------------------------------------- Adam

def _torch_adam_step(theta, m, v, g, t, lr=LR, b1=B1, b2=B2, eps=EPS):
    torch = pytest.importorskip("torch")
    p = torch.nn.Parameter(torch.tensor(theta, dtype=torch.float64))
    opt = torch.optim.Adam([p], lr=f32(lr), betas=(f32(b1), f32(b2)), eps=f32(eps), foreach=False,
                           fused=False)
    p.grad = torch.tensor(g, dtype=torch.float64)
    if t > 0:
        opt.state[p] = {"step": torch.tensor(float(t), dtype=torch.float64),
                        "exp_avg": torch.tensor(m, dtype=torch.float64),
                        "exp_avg_sq": torch.tensor(v, dtype=torch.float64)}
    opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def _assert_f32_close_ulps(a, ref64, ulps):
    ref = ref64.astype(np.float32)
    d = np.abs(a.astype(np.float64) - ref.astype(np.float64))
    sp = np.spacing(np.abs(ref)).astype(np.float64)
    assert np.all(d <= ulps * sp + 1e-45), np.max(d / sp)


@pytest.mark.parametrize("t", [0, 1, 7, 1000])
def test_adam_matches_torch_optim_adam(t):
    """One oracle step equals torch.optim.Adam (float64, library) from the same state, rounded to fp32."""
    wl = synth.WORKLOADS["tiny"].with_(psi=4000, n=2, a=2, loss_scale=1.0)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    theta = synth.master_f32(wl)
    rng = np.random.default_rng(t)
    m0 = (rng.standard_normal(wl.psi) * 1e-4).astype(np.float32) if t else np.zeros(wl.psi, np.float32)
    v0 = (rng.random(wl.psi) * 1e-8).astype(np.float32) if t else np.zeros(wl.psi, np.float32)
    segs = synth.layout_even(wl.psi, wl.n)
    res, M, Mm, Vv, reps = run_oracle(wl.psi, wl.n, wl.a, 1, segs, grads, theta, m0, v0, t=t)
    assert res == {"found": 0, "nonfinite": 0, "t": t + 1}
    gbar = oracle.reduce(wl.psi, wl.n, wl.a, grads, 1.0)["gbar"]
    th, mm, vv = _torch_adam_step(theta.astype(np.float64), m0.astype(np.float64), v0.astype(np.float64), gbar, t)
    _assert_f32_close_ulps(gather_full(M, segs, wl.psi, 1), th, 1)
    _assert_f32_close_ulps(gather_full(Mm, segs, wl.psi, 1), mm, 1)
    _assert_f32_close_ulps(gather_full(Vv, segs, wl.psi, 1), vv, 1)


def test_adam_cold_start_closed_form():
    """m = v = 0 at t = 0: mhat = gbar and vhat = gbar^2, so th' = th - lr gbar / (|gbar| + eps)."""
    psi, n, a = 6, 2, 1
    # gbar = (g0 + g1) / 2 = +1, -1, +0.5, 0, 1e-8-ish, -3
    g0 = bf16_bits([1.0, -1.0, 0.5, 0.0, 2 ** -27, -3.0])
    g1 = bf16_bits([1.0, -1.0, 0.5, 0.0, 2 ** -27, -3.0])
    theta = np.array([0.5, -0.25, 0.0, 0.125, 1.0, 2.0], np.float32)
    segs = synth.layout_even(psi, n)
    res, M, Mm, Vv, reps = run_oracle(psi, n, a, 1, segs, [g0, g1], theta)
    th = gather_full(M, segs, psi, 1)
    gb = np.array([1.0, -1.0, 0.5, 0.0, 2 ** -27, -3.0])
    lr, eps = f32(LR), f32(EPS)
    ref = theta.astype(np.float64) - lr * gb / (np.abs(gb) + eps)
    _assert_f32_close_ulps(th, ref, 1)
    # the hand values: gbar = +-1 moves theta by -+lr / (1 + eps)
    assert th[0] == np.float32(0.5 - lr / (1 + eps))
    assert th[1] == np.float32(-0.25 + lr / (1 + eps))
    # gbar = 0: theta unchanged, moments stay zero
    assert th[3] == theta[3]
    assert gather_full(Mm, segs, psi, 1)[3] == 0.0 and gather_full(Vv, segs, psi, 1)[3] == 0.0
    # first moment after one step is (1 - beta1) gbar, second (1 - beta2) gbar^2
    _assert_f32_close_ulps(gather_full(Mm, segs, psi, 1), (1 - f32(B1)) * gb, 1)
    _assert_f32_close_ulps(gather_full(Vv, segs, psi, 1), (1 - f32(B2)) * gb * gb, 1)


def test_adam_constant_gradient_closed_form():
    """With the same gbar every step, bias correction makes mhat = gbar and vhat = gbar^2 at every t,
    so each step moves theta by exactly -lr gbar / (|gbar| + eps).  A wrong power of beta, a t counted
    from 0, or a missing correction breaks this after the first step."""
    psi, n, a = 5, 1, 1
    gv = [0.75, -2.0, 1.0 / 64, -1.0 / 1024, 3.0]
    g = bf16_bits(gv)
    segs = synth.layout_even(psi, n)
    theta = np.array([0.1, 0.2, -0.3, 0.4, -0.5], np.float32)
    M, Mm, Vv = make_state(psi, n, 1, segs, theta)
    reps = [np.zeros(psi, np.uint16)]
    t = 0
    lr, eps = f32(LR), f32(EPS)
    gb = np.array(gv)
    cur = theta.astype(np.float64)
    for step in range(1, 9):
        res = oracle.step(psi, n, a, 1, segs, [g], M, Mm, Vv, reps, LR, B1, B2, EPS, 1.0, t)
        t = res["t"]
        assert t == step
        cur = cur - lr * gb / (np.abs(gb) + eps)
        # each stored step rounds to fp32 once; allow a few ulps of drift over 8 steps
        d = np.abs(M[0].astype(np.float64) - cur)
        assert np.all(d <= 8 * np.spacing(np.abs(cur.astype(np.float32))).astype(np.float64))


def test_ones_gradient_first_step_hand_value():
    """Hand-computed: gbar = 1 at t = 1 from zero moments gives m = 0.1, v = 0.001 (in fp32 arithmetic of
    the constants) and theta - 1e-3 / (1 + 1e-8)."""
    g = bf16_bits([1.0])
    segs = [(0, 1, 0, 0)]
    res, M, Mm, Vv, reps = run_oracle(1, 1, 1, 1, segs, [g], np.array([1.0], np.float32))
    assert Mm[0][0] == np.float32(1.0 - f32(B1))
    assert Vv[0][0] == np.float32(1.0 - f32(B2))
    assert M[0][0] == np.float32(1.0 - f32(LR) / (1.0 + f32(EPS)))


# ---------------------------------------------------------------- skip, replicas, sharding

@pytest.mark.parametrize("where", ["first", "last", "boundary", "middle"])
@pytest.mark.parametrize("kind", [0x7F80, 0xFF80, 0x7FC0])
def test_skip_on_nonfinite_leaves_state(where, kind):
    wl = synth.WORKLOADS["tiny"].with_(psi=1003, n=4, a=2)
    segs = synth.layout_even(wl.psi, wl.n)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    idx = {"first": 0, "last": wl.psi - 1, "boundary": segs[2][0], "middle": 517}[where]
    grads[5][idx] = kind
    theta = synth.master_f32(wl)
    m0 = np.full(wl.psi, 1e-5, np.float32)
    v0 = np.full(wl.psi, 1e-9, np.float32)
    M, Mm, Vv = make_state(wl.psi, wl.n, 1, segs, theta, m0, v0)
    before = [x.copy() for x in M + Mm + Vv]
    reps = [np.full(wl.psi, 0x1234, np.uint16) for _ in range(wl.n)]
    res = oracle.step(wl.psi, wl.n, wl.a, 1, segs, grads, M, Mm, Vv, reps, LR, B1, B2, EPS, 1.0, 5)
    assert res == {"found": 1, "nonfinite": 1, "t": 5}
    for x, y in zip(M + Mm + Vv, before):
        assert np.array_equal(bits_of(x), bits_of(y))
    assert all(np.all(r == 0x1234) for r in reps)


def test_overflow_of_finite_inputs_is_found():
    """Two bf16 values of 3e38 on one element sum past the fp32 range: the step is skipped."""
    big = np.uint16(0x7F62)   # about 3.0e38 in bf16
    assert oracle.lib().oracle_bf16_to_double(int(big)) > 2.9e38
    psi = 8
    g0 = np.zeros(psi, np.uint16)
    g1 = np.zeros(psi, np.uint16)
    g0[3] = big
    g1[3] = big
    res = oracle.reduce(psi, 2, 1, [g0, g1], 1.0)
    assert res["found"] == 1 and res["nonfinite"] == 1


def test_replicas_identical_and_equal_bf16_of_master():
    """After the step every replica holds the same parameters (page: replicas stay consistent), each the
    round-to-nearest-even bf16 image of the fp32 master (checked against torch's conversion)."""
    torch = pytest.importorskip("torch")
    wl = synth.WORKLOADS["tiny"].with_(psi=2048 + 5, n=4, a=2)
    segs = synth.layout_random(wl.psi, wl.n, 6, 1)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    res, M, Mm, Vv, reps = run_oracle(wl.psi, wl.n, wl.a, 2, segs, grads, synth.master_f32(wl))
    for r in reps[1:]:
        assert np.array_equal(r, reps[0])
    full = gather_full(M, segs, wl.psi, 2)
    ref = torch.tensor(full).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(reps[0], ref)


def test_bf16_rounding_vs_torch_library():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 100000, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, np.array([0x3F808000, 0x3F818000, 0x3F808001, 0x00008000, 0x00018000,
                                           0x7F7F8000, 0x7F7FFFFF, 0x80000000], np.uint32)])
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    mine = oracle.f32_to_bf16_array(x)
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("layout", ["even", "ragged", "random", "buckets"])
def test_sharded_equals_unsharded(layout):
    """ZeRO-1/2/3 shards give exactly the plain data-parallel result (page: sharding changes the storage
    layout and communication pattern, not the update semantics)."""
    wl = synth.WORKLOADS["tiny"].with_(psi=3001, n=4, a=2, layout=layout, nseg=9, bucket=700, misalign=3, seed=9)
    segs = synth.layout_of(wl)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    theta = synth.master_f32(wl)
    rng = np.random.default_rng(3)
    m0 = (rng.standard_normal(wl.psi) * 1e-5).astype(np.float32)
    v0 = (rng.random(wl.psi) * 1e-9).astype(np.float32)
    r0, M0, Mm0, Vv0, reps0 = run_oracle(wl.psi, wl.n, wl.a, 0, segs, grads, theta, m0, v0, t=3)
    for r in range(1, wl.n):
        assert np.array_equal(M0[r], M0[0])
    for stage in (1, 2, 3):
        r1, M1, Mm1, Vv1, reps1 = run_oracle(wl.psi, wl.n, wl.a, stage, segs, grads, theta, m0, v0, t=3)
        assert r1 == r0
        assert np.array_equal(bits_of(gather_full(M1, segs, wl.psi, stage)), bits_of(M0[0]))
        assert np.array_equal(bits_of(gather_full(Mm1, segs, wl.psi, stage)), bits_of(Mm0[0]))
        assert np.array_equal(bits_of(gather_full(Vv1, segs, wl.psi, stage)), bits_of(Vv0[0]))
        for r in range(wl.n):
            assert np.array_equal(reps1[r], reps0[r])


def test_threads_do_not_change_results():
    wl = synth.WORKLOADS["tiny"].with_(psi=50001, n=2, a=3)
    segs = synth.layout_ragged(wl.psi, wl.n, 1)
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    theta = synth.master_f32(wl)
    outs = []
    for th in (1, 7):
        M, Mm, Vv = make_state(wl.psi, wl.n, 1, segs, theta)
        reps = [np.zeros(wl.psi, np.uint16) for _ in range(wl.n)]
        oracle.step(wl.psi, wl.n, wl.a, 1, segs, grads, M, Mm, Vv, reps, LR, B1, B2, EPS, 1.0, 0, threads=th)
        outs.append(np.concatenate([bits_of(x) for x in M + Mm + Vv]))
    assert np.array_equal(outs[0], outs[1])


def test_empty_problem_advances_t():
    res = oracle.step(0, 2, 1, 1, [], [np.zeros(0, np.uint16)] * 2, [np.zeros(0, np.float32)] * 2,
                      [np.zeros(0, np.float32)] * 2, [np.zeros(0, np.float32)] * 2, None, LR, B1, B2, EPS, 1.0, 4)
    assert res == {"found": 0, "nonfinite": 0, "t": 5}


# ---------------------------------------------------------------- ring traffic

@pytest.mark.parametrize("n", [2, 3, 4, 8])
def test_ring_allreduce_traffic_even(n):
    """Ring all-reduce: each rank sends and receives 2(N-1)/N x the gradient bytes, in 2(N-1) steps."""
    psi = 840
    tr = ring.step_traffic(n, synth.layout_even(psi, n), psi, 0, 2, 2)
    sent = [tr["rs_grad"].sent_bytes[r] + tr["ag_grad"].sent_bytes[r] for r in range(n)]
    recv = [tr["rs_grad"].recv_bytes[r] + tr["ag_grad"].recv_bytes[r] for r in range(n)]
    want = Fraction(2 * (n - 1), n) * psi * 2
    assert all(Fraction(s) == want for s in sent)
    assert all(Fraction(x) == want for x in recv)
    assert tr["rs_grad"].steps + tr["ag_grad"].steps == 2 * (n - 1)


def test_ring_traffic_ragged():
    n, psi = 5, 1009
    segs = synth.layout_ragged(psi, n, 2)
    lens = [ln for _, ln, _, _ in segs]
    tr = ring.step_traffic(n, segs, psi, 1, 4, 2)
    assert sum(tr["rs_grad"].sent_elems) + sum(tr["ag_param"].sent_elems) == 2 * (n - 1) * psi
    for r in range(n):
        assert tr["rs_grad"].sent_elems[r] == psi - lens[r]
        assert tr["ag_param"].sent_elems[r] == psi - lens[(r + 1) % n]


def test_zero_stage_traffic_ratios():
    """Stages 1 and 2 move the same bytes as plain DP; stage 3 gathers the weights twice: 1.5x."""
    n, psi = 8, 8000
    segs = synth.layout_even(psi, n)
    tot = {}
    for stage in range(4):
        tr = ring.step_traffic(n, segs, psi, stage, 2, 2)
        tot[stage] = sum(sum(t.sent_bytes) for t in tr.values())
    assert tot[1] == tot[0] and tot[2] == tot[0]
    assert Fraction(tot[3], tot[0]) == Fraction(3, 2)


def test_ring_detects_lost_message():
    n, psi = 4, 40
    rg = ring.Ring(n, synth.layout_even(psi, n), psi)
    rg.drop = ("rs", 1, 2)
    with pytest.raises(RuntimeError, match="message lost"):
        rg.reduce_scatter([np.ones(psi, np.float32)] * n)


# ---------------------------------------------------------------- dynamic loss scale

def test_scaler_policy_matches_torch_amp_update():
    """With no clamping, the oracle's scale policy equals torch's own loss-scale update (library)."""
    torch = pytest.importorskip("torch")
    from oracle import scaler
    rng = np.random.default_rng(5)
    for growth, backoff, interval in ((2.0, 0.5, 3), (2.0, 0.25, 1), (1.5, 0.5, 7)):
        s_t = torch.tensor([2.0 ** 16])
        g_t = torch.tensor([0], dtype=torch.int32)
        f_t = torch.tensor([0.0])
        s, g = 2.0 ** 16, 0
        for step in range(200):
            found = bool(rng.random() < 0.15)
            f_t.fill_(1.0 if found else 0.0)
            torch._amp_update_scale_(s_t, g_t, f_t, growth, backoff, interval)
            s, g = scaler.update(s, g, found, growth, backoff, interval, 0.0, float(np.finfo(np.float32).max))
            assert s == s_t.item() and g == g_t.item()


def test_scaler_clamps_to_range():
    from oracle import scaler
    s, g = 2.0 ** 24, 0
    s, g = scaler.update(s, 1, False, 2.0, 0.5, 2, 2.0 ** 8, 2.0 ** 24)
    assert (s, g) == (2.0 ** 24, 0)
    s, g = 2.0 ** 8, 0
    s, g = scaler.update(s, g, True, 2.0, 0.5, 2, 2.0 ** 8, 2.0 ** 24)
    assert (s, g) == (2.0 ** 8, 0)
