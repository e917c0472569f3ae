"""The tree reduction order on the CPU: the simulated binomial tree pinned to its definition, to hand-written
sums, to the step counts that motivate it, and the forms the kernels use -- the incremental binary counter and
the grouped rank-major form -- checked against it."""
import math

import numpy as np
import pytest

import synth
from oracle import brute
from oracle.ring import Ring, two_sum32
from oracle.tree import Tree, combine, tree_expression


def definition(n: int) -> str:
    """Top-down: the block [lo, lo + size) of a power-of-two size is its lower half plus its upper half; an upper
    half that starts at or past n does not exist and the lower half stands alone."""
    def rec(lo: int, size: int) -> str:
        if size == 1:
            return "g%d" % lo
        half = size // 2
        if lo + half >= n:
            return rec(lo, half)
        return "(%s+%s)" % (rec(lo, half), rec(lo + half, half))
    return rec(0, 1 << math.ceil(math.log2(n)) if n > 1 else 1)


def counter_form(n: int) -> str:
    """The kernels' incremental form: a binary counter of pending block sums, merged when a rank completes,
    the leftovers joined smallest first at the end."""
    slot = [None] * 5
    for r in range(n):
        v = "g%d" % r
        top = (~r & (r + 1)).bit_length() - 1          # lowest clear bit of r
        for lv in range(5):
            if lv < top:
                v = "(%s+%s)" % (slot[lv], v)
            elif lv == top:
                slot[lv] = v
    tot, have = None, False
    for lv in range(5):
        if (n >> lv) & 1:
            tot = "(%s+%s)" % (slot[lv], tot) if have else slot[lv]
            have = True
    return tot


def grouped_form(n: int, group: int) -> str:
    """The rank-major kernels' form: the ranks in aligned groups of `group` (a power of two), each group summed
    up its own binomial tree, then the group totals added up the binomial tree over groups -- the two-pass
    kernel with groups of eight, the single pass with groups of four."""
    def tree_of(items):
        val = list(items)
        step = 1
        while step < len(val):
            for r in range(0, len(val), 2 * step):
                if r + step < len(val):
                    val[r] = "(%s+%s)" % (val[r], val[r + step])
            step *= 2
        return val[0]
    groups = [tree_of(["g%d" % r for r in range(lo, min(n, lo + group))]) for lo in range(0, n, group)]
    return tree_of(groups)


HAND = {
    1: "g0",
    2: "(g0+g1)",
    3: "((g0+g1)+g2)",
    4: "((g0+g1)+(g2+g3))",
    5: "(((g0+g1)+(g2+g3))+g4)",
    6: "(((g0+g1)+(g2+g3))+(g4+g5))",
    7: "(((g0+g1)+(g2+g3))+((g4+g5)+g6))",
    8: "(((g0+g1)+(g2+g3))+((g4+g5)+(g6+g7)))",
}


@pytest.mark.parametrize("n", sorted(HAND))
def test_tree_by_hand(n):
    assert tree_expression(n) == HAND[n]


@pytest.mark.parametrize("n", range(1, 17))
def test_tree_matches_definition_and_kernel_form(n):
    e = tree_expression(n)
    assert e == definition(n)
    assert e == counter_form(n)
    assert sorted(int(x) for x in e.replace("(", " ").replace(")", " ").replace("+", " ").replace("g", " ").split()) \
        == list(range(n))


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("n", range(1, 17))
def test_grouped_form_is_the_tree(n, group):
    """Groups aligned to a power of two, each summed up its own tree, then the totals up the tree over groups,
    parenthesise exactly as the binomial tree: its levels below log2(group) pair ranks only inside an aligned
    block of `group`, and the levels above pair whole blocks."""
    assert grouped_form(n, group) == tree_expression(n)


@pytest.mark.parametrize("n", [2, 3, 4, 5, 8, 9, 16])
def test_step_counts_and_traffic(n):
    """A tree all-reduce takes 2 ceil(log2 n) steps against the ring's 2(n-1): the page's reason for trees."""
    psi = 1000
    t = Tree(n)
    local = [np.full(psi, r + 1.0) for r in range(n)]
    tot = t.reduce(local, combine("f64"), elems=psi)
    out = t.broadcast(tot, elems=psi)
    assert np.all(tot == n * (n + 1) / 2)
    assert all(np.array_equal(o, tot) for o in out)
    lv = math.ceil(math.log2(n))
    assert t.traffic["reduce"].steps == lv and t.traffic["broadcast"].steps == lv
    assert 2 * lv <= 2 * (n - 1) and (n < 4 or 2 * lv < 2 * (n - 1))
    # reduce: every rank but the root sends its block sum exactly once; broadcast: every rank but the root
    # receives the total exactly once
    assert t.traffic["reduce"].sent_elems == [0] + [psi] * (n - 1)
    assert t.traffic["broadcast"].recv_elems == [0] + [psi] * (n - 1)


def random_grads(n, a, psi, seed):
    wl = synth.WORKLOADS["tiny"].with_(psi=psi, n=n, a=a, seed=seed, sigma_g=1.0)
    return [synth.grads_bf16(wl, r, k) for r in range(n) for k in range(a)]


@pytest.mark.parametrize("n", [3, 5, 7, 8, 13])
def test_tree_gbar_f32_written_out(n):
    """Plain fp32: the simulated tree equals the hand-parenthesised fp32 sum, evaluated directly."""
    psi, a = 257, 1
    grads = random_grads(n, a, psi, 40 + n)
    g = [brute.bf16_bits_to_f32(x) for x in grads]
    f = lambda x, y: (x + y).astype(np.float32)
    if n == 3:
        want = f(f(g[0], g[1]), g[2])
    elif n == 5:
        want = f(f(f(g[0], g[1]), f(g[2], g[3])), g[4])
    elif n == 7:
        want = f(f(f(g[0], g[1]), f(g[2], g[3])), f(f(g[4], g[5]), g[6]))
    elif n == 8:
        want = f(f(f(g[0], g[1]), f(g[2], g[3])), f(f(g[4], g[5]), f(g[6], g[7])))
    else:   # 13 = 8 + 4 + 1
        b8 = f(f(f(g[0], g[1]), f(g[2], g[3])), f(f(g[4], g[5]), f(g[6], g[7])))
        b4 = f(f(g[8], g[9]), f(g[10], g[11]))
        want = f(b8, f(b4, g[12]))
    inv = np.float32(1.0 / n)
    got = brute.tree_gbar(grads, n, a, None, psi, 1.0, arith="f32")
    assert np.array_equal(got.view(np.uint32), (want * inv).astype(np.float32).view(np.uint32))


def test_tree_and_ring_orders_differ_but_agree_within_rounding():
    n, a, psi = 8, 2, 4000
    grads = random_grads(n, a, psi, 77)
    segs = synth.layout_even(psi, n)
    tree = brute.tree_gbar(grads, n, a, segs, psi, 1.0, arith="f32")
    ring = brute.ring_gbar(grads, n, a, segs, psi, 1.0, arith="f32")
    assert not np.array_equal(tree, ring)          # the order is observable in plain fp32
    treep = brute.tree_gbar(grads, n, a, segs, psi, 1.0, arith="f32pair")
    ringp = brute.ring_gbar(grads, n, a, segs, psi, 1.0, arith="f32pair")
    # compensated, both orders give the correctly rounded sum here, so they agree bit for bit
    exact = np.zeros(psi)
    for q in range(n * a):
        exact = exact + brute.bf16_bits_to_f32(grads[q]).astype(np.float64)
    want = (exact.astype(np.float32) * np.float32(1.0 / n)).astype(np.float32)
    assert np.array_equal(treep.view(np.uint32), ringp.view(np.uint32))
    assert np.array_equal(treep.view(np.uint32), want.view(np.uint32))


def test_compensated_merge_rule():
    """(H, e) = TwoSum(H_left, H_right); L = (L_left + e) + L_right, in that order."""
    add = combine("f32pair")
    hl = (np.float32([1.0]), np.float32([2 ** -30]))
    hr = (np.float32([2 ** -24]), np.float32([2 ** -31]))
    H, L = add(hl, hr)
    s, e = two_sum32(hl[0], hr[0])
    assert H == s and L == np.float32(np.float32(hl[1] + e) + hr[1])
