"""Fixed values the pages print (tests/golden/pages_numbers.json), checked against the oracle side (CPU)."""
import json
import os
from fractions import Fraction

import numpy as np

import oracle
import synth
from oracle import ring

HERE = os.path.dirname(os.path.abspath(__file__))
G = json.load(open(os.path.join(HERE, "golden", "pages_numbers.json")))


def test_ring_allreduce_numbers():
    for n in (2, 4, 8, 16):
        psi = 16 * 27
        tr = ring.step_traffic(n, synth.layout_even(psi, n), psi, 0, 2, 2)
        per_rank = tr["rs_grad"].sent_bytes[0] + tr["ag_grad"].sent_bytes[0]
        assert Fraction(per_rank, psi * 2) == Fraction(2 * (n - 1), n)
        assert tr["rs_grad"].steps + tr["ag_grad"].steps == 2 * (n - 1)


def test_zero_traffic_numbers():
    n, psi = 4, 4000
    segs = synth.layout_even(psi, n)
    tot = [sum(sum(t.sent_bytes) for t in ring.step_traffic(n, segs, psi, s, 2, 2).values()) for s in range(4)]
    z = G["zero_traffic"]
    assert Fraction(tot[1], tot[0]) == Fraction(z["stage1_vs_dp"]).limit_denominator()
    assert Fraction(tot[2], tot[0]) == Fraction(z["stage2_vs_dp"]).limit_denominator()
    assert Fraction(tot[3], tot[0]) == Fraction(z["stage3_vs_dp"]).limit_denominator()


def test_cold_start_unit_gradient_example():
    ex = G["adam_cold_start_unit_gradient"]
    g = np.array([0x3F80], np.uint16)                 # bf16 1.0
    M = [np.array([0.0], np.float32)]
    Z = [np.zeros(1, np.float32)]
    Z2 = [np.zeros(1, np.float32)]
    oracle.step(1, 1, 1, 1, [(0, 1, 0, 0)], [g], M, Z, Z2, None, ex["lr"], 0.9, 0.999, ex["eps"], 1.0, 0)
    assert abs(float(M[0][0]) - ex["delta_theta"]) <= 1e-12 + 1e-6 * abs(ex["delta_theta"])


def test_global_batch_example_is_product():
    e = G["global_batch_example"]
    assert e["b"] * e["n"] * e["a"] == e["B_global"]
