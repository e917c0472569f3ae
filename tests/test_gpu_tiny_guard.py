"""Every head, tail and ragged path at tiny sizes, with sentinel bands around every device buffer (-m gpu).

compute-sanitizer is not available to these tests, so out-of-bounds stores are looked for directly: every
buffer a step touches (gradients, replicas, master/m/v and the single pass's second set, gbar shards, the
per-micro-step accumulators, the step state) sits inside an allocation with 256 sentinel bytes on each side,
and the bands are checked after every step.  Sizes psi = 1 ... 67 with n in {1, 2, 3, 5, 8} and a in {1, 2, 3}
run through the five launch paths -- dp_step in ring order and in tree order, dp_step_single_pass in both
orders, and the per-micro-step reduce-scatter + dp_step_update -- and every element is compared with the
float64 oracle.  The tree order also runs n in {9, 10, 12, 16}, where its ranks form more than one group of eight
(two-pass) or four (single pass).

Layouts cycle over four kinds, so the misaligned cases reach the kernels' ragged branches:
  - 3-element-misaligned buckets of about psi / 3 elements and 1-misaligned buckets of 5 elements: shard
    offsets that are not multiples of 4 or 8, so every tile has ragged local ends (the update's <= 3-element
    scalar ends, the single pass's element-by-element groups), odd staging offsets (the 1- and 2-element
    branches of the bf16 staging store) and global ends shorter than 8 (the replicas' plain stores);
  - seeded random segments with random owners (local spaces with several pieces per rank);
  - seeded ragged shards, some of them empty.
psi not a multiple of 8 puts the buffer's last partial 8-group on the reduction's plain-load path.  Shapes that
need more than 67 elements (a whole misaligned warp's shuffle store, whole-cell tiles) are covered at larger
sizes in test_gpu_parity.py and test_gpu_single_pass.py.
"""
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp

import gpu_util as gu

pytestmark = pytest.mark.gpu

PATHS = ["two_pass", "tree", "single_pass", "single_pass_tree", "microstep"]
NS = [1, 2, 3, 5, 8]
BASE = synth.WORKLOADS["tiny"]


def layout_kind(i: int, psi: int) -> dict:
    k = i % 4
    if k == 0:
        return {"layout": "buckets", "bucket": max(1, (psi + 2) // 3), "misalign": 3}
    if k == 1:
        return {"layout": "random", "nseg": 1 + i % 7}
    if k == 2:
        return {"layout": "ragged"}
    return {"layout": "buckets", "bucket": 5, "misalign": 1}


def run_case(path: str, psi: int, n: int, a: int, i: int) -> None:
    single = path in ("single_pass", "single_pass_tree")
    stage = 1 + i % 3 if single else i % 4
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, seed=9000 + i, loss_scale=float(2 ** (i % 9)),
                    **layout_kind(i, psi))
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    b = gu.upload(c, second_set=single, micro_acc=path == "microstep")
    guard = gu.Guarded(b)
    S = wl.loss_scale
    if path == "two_pass":
        b.step(A, S)
    elif path == "tree":
        b.step(A, S, dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)
    elif path == "single_pass":
        b.step_single_pass(A, S)
    elif path == "single_pass_tree":
        b.step_single_pass(A, S, dp.DP_SUM_COMPENSATED | dp.DP_ORDER_TREE)
    else:
        b.step_micro(A, S)
    torch.cuda.synchronize()
    what = "%s psi=%d n=%d a=%d stage=%d %s" % (path, psi, n, a, stage, wl.layout)
    guard.check(what)
    if single:
        b.master, b.m, b.v = b.current()
    g = gu.gpu_result(c, b)
    o = gu.run_oracle(c, threads=1)
    try:
        gu.assert_matches_oracle(g, o)
    except AssertionError as e:
        raise AssertionError("%s: %s" % (what, e)) from None


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("path", PATHS)
def test_tiny_sizes_guarded(dev, path, n):
    i = 0
    for psi in range(1, 68):
        for a in (1, 2, 3):
            run_case(path, psi, n, a, i)
            i += 1


@pytest.mark.parametrize("path", ["tree", "single_pass_tree"])
@pytest.mark.parametrize("n", [9, 10, 12, 16])
def test_tiny_sizes_guarded_tree_groups(dev, n, path):
    i = 0
    for psi in range(1, 68):
        for a in (1, 2, 3):
            run_case(path, psi, n, a, i)
            i += 1
