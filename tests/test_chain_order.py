"""The compensated ring order of the fused step on the CPU: every rank folds its unsummed micro-step gradients,
one at a time, into the float32 (hi, lo) pair that travels round the simulated ring ("f32chain").  Pinned to
the pair arithmetic of the rank-local form where the two coincide (one micro-step), to hand values where plain
float32 loses the answer, and to the correctly rounded sum."""
import math

import numpy as np
import pytest

import synth
from oracle import brute
from oracle.ring import Ring


def grads(n, a, psi, seed, wide=False):
    wl = synth.WORKLOADS["tiny"].with_(psi=psi, n=n, a=a, seed=seed, sigma_g=1.0,
                                       tail_p=0.3 if wide else 0.0, tail_mult=float(2 ** 20) if wide else 1.0)
    return [synth.grads_bf16(wl, r, k) for r in range(n) for k in range(a)]


def bf16_bits(values):
    """Exact bf16 bit patterns of float values that bf16 represents (checked)."""
    f = np.asarray(values, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(brute.bf16_bits_to_f32(bits), f)
    return bits


@pytest.mark.parametrize("n", [1, 2, 5])
def test_one_micro_step_equals_the_pair_ring(n):
    """With a = 1 a rank folds a single value: (H, e) = TwoSum(H, x), L = L + e -- the pair ring's combine with a
    zero low word, so both arithmetics give the same bits."""
    psi = 4001
    g = grads(n, 1, psi, 11, wide=True)
    segs = synth.layout_ragged(psi, n, 5)
    x = brute.ring_gbar(g, n, 1, segs, psi, 2.0, "f32chain")
    y = brute.ring_gbar(g, n, 1, segs, psi, 2.0, "f32pair")
    assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_cancellation_kept_where_plain_float32_loses_it():
    """Owner 0 of n = 3, a = 2 receives rank 1's [2^30, 1], then rank 2's [-2^30, 2^-10], then its own [0, 0]:
    the exact sum is 1 + 2^-10.  Plain float32 rounds each rank's local sum to +-2^30 and returns 0."""
    n, a = 3, 2
    vals = {(0, 0): 0.0, (0, 1): 0.0, (1, 0): 2.0 ** 30, (1, 1): 1.0, (2, 0): -(2.0 ** 30), (2, 1): 2.0 ** -10}
    g = [bf16_bits([vals[(r, k)]]) for r in range(n) for k in range(a)]
    segs = [(0, 1, 0, 0)]
    chain = brute.ring_gbar(g, n, a, segs, 1, 1.0, "f32chain")
    plain = brute.ring_gbar(g, n, a, segs, 1, 1.0, "f32")
    inv = np.float32(1.0 / 3.0)
    assert chain[0] == np.float32(np.float32(1.0 + 2.0 ** -10) * inv)
    assert plain[0] == np.float32(0.0)


def test_close_to_the_correctly_rounded_sum_on_wide_inputs():
    """n S a power of two: gbar within one ulp of fl32(exact sum) / (n S) (the Sum2 bound of Ogita, Rump and
    Oishi, 2005, on inputs spanning 2^20), and closer to the exact value than plain float32 at its worst."""
    n, a, psi = 4, 4, 3000
    g = grads(n, a, psi, 13, wide=True)
    segs = synth.layout_ragged(psi, n, 6)
    chain = brute.ring_gbar(g, n, a, segs, psi, 1.0, "f32chain")
    plain = brute.ring_gbar(g, n, a, segs, psi, 1.0, "f32")
    vals = [brute.bf16_bits_to_f32(x).astype(np.float64) for x in g]
    exact = np.array([math.fsum(v[i] for v in vals) for i in range(psi)])
    want = (exact.astype(np.float32) * np.float32(1.0 / n)).astype(np.float32)
    ulps = np.abs(chain.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    err_chain = np.abs(chain.astype(np.float64) - exact / n).max()
    err_plain = np.abs(plain.astype(np.float64) - exact / n).max()
    assert err_chain < err_plain


def test_same_messages_as_the_other_arithmetics():
    """The arithmetic of a hop changes no message: elements, bytes and steps per rank are those of the f32 ring."""
    n, a, psi = 5, 3, 2003
    g = grads(n, a, psi, 17)
    segs = synth.layout_ragged(psi, n, 4)
    counts = []
    for arith in ("f32", "f32chain"):
        ring = Ring(n, segs, psi)
        if arith == "f32chain":
            loc = [[brute.bf16_bits_to_f32(g[r * a + k]) for k in range(a)] for r in range(n)]
        else:
            loc = brute.local_accumulate(g, n, a, arith)
        ring.reduce_scatter(loc, arith=arith, wire_bytes=4)
        tr = ring.traffic["rs"]
        counts.append((tr.sent_elems, tr.recv_elems, tr.sent_bytes, tr.steps))
    assert counts[0] == counts[1]
