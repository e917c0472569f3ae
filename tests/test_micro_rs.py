"""The per-micro-step reduce-scatter order on the CPU: the brute-force emulation (each micro-step round the
simulated ring, then summed in the owner's accumulator) pinned to hand-written sums and special cases."""
import numpy as np
import pytest

import synth
from oracle import brute


def grads(n, a, psi, seed, wide=False):
    wl = synth.WORKLOADS["tiny"].with_(psi=psi, n=n, a=a, seed=seed, sigma_g=1.0,
                                       tail_p=0.3 if wide else 0.0, tail_mult=float(2 ** 20) if wide else 1.0)
    return [synth.grads_bf16(wl, r, k) for r in range(n) for k in range(a)]


def f32(bits):
    return brute.bf16_bits_to_f32(bits)


@pytest.mark.parametrize("arith", ["f32", "f32pair"])
def test_one_micro_step_is_the_ring(arith):
    """With a = 1 there is nothing to accumulate: the per-micro-step form is the ring order itself."""
    n, psi = 5, 3001
    g = grads(n, 1, psi, 3, wide=True)
    segs = synth.layout_ragged(psi, n, 4)
    x = brute.micro_rs_gbar(g, n, 1, segs, psi, 1.0, arith)
    y = brute.ring_gbar(g, n, 1, segs, psi, 1.0, arith)
    assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_one_rank_sums_micro_steps_left_to_right():
    n, a, psi = 1, 4, 777
    g = grads(n, a, psi, 5, wide=True)
    want = f32(g[0])
    for k in range(1, a):
        want = (want + f32(g[k])).astype(np.float32)
    x = brute.micro_rs_gbar(g, n, a, [(0, psi, 0, 0)], psi, 1.0, "f32")
    assert np.array_equal(x.view(np.uint32), want.view(np.uint32))


def test_two_ranks_two_micro_steps_by_hand():
    """n = 2, a = 2, owner 0's chunk: p_k = g_{1,k} + g_{0,k}, A = p_0 + p_1; owner 1's: p_k = g_{0,k} + g_{1,k}."""
    n, a, psi = 2, 2, 1000
    g = grads(n, a, psi, 7, wide=True)
    segs = synth.layout_even(psi, n)
    G = lambda r, k: f32(g[r * a + k])
    add = lambda x, y: (x + y).astype(np.float32)
    own0 = add(add(G(1, 0), G(0, 0)), add(G(1, 1), G(0, 1)))
    own1 = add(add(G(0, 0), G(1, 0)), add(G(0, 1), G(1, 1)))
    want = np.concatenate([own0[:500], own1[500:]]) * np.float32(0.5)
    x = brute.micro_rs_gbar(g, n, a, segs, psi, 1.0, "f32")
    assert np.array_equal(x.view(np.uint32), want.astype(np.float32).view(np.uint32))


def test_order_differs_from_the_step_order_but_compensated_agrees():
    n, a, psi = 4, 4, 20_000
    g = grads(n, a, psi, 9, wide=True)
    segs = synth.layout_even(psi, n)
    mp = brute.micro_rs_gbar(g, n, a, segs, psi, 1.0, "f32")
    rp = brute.ring_gbar(g, n, a, segs, psi, 1.0, "f32")
    assert not np.array_equal(mp, rp)            # the order is observable in plain fp32 on wide-range inputs
    mc = brute.micro_rs_gbar(g, n, a, segs, psi, 1.0, "f32pair")
    exact = np.zeros(psi)
    for q in range(n * a):
        exact += f32(g[q]).astype(np.float64)
    want = (exact.astype(np.float32) * np.float32(1.0 / n)).astype(np.float32)
    ulps = np.abs(mc.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    assert np.abs(mp.astype(np.float64) - exact / n).max() > np.abs(mc.astype(np.float64) - exact / n).max()
