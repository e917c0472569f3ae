"""The step split into slices of the parameter space, on one GPU (-m gpu).

Each slice gets buffers of its own holding its part of every gradient, replica and shard (Layout.slice), and
runs the sliced protocol of zero_gradient_sync_gb300.sliced: the reduction with DP_DEFER_COMMIT, found_inf
combined over the slices with a maximum (here a max over the slices' state words on the one device, standing
in for the 4-byte all-reduce between GPUs), then the commit and the update.  The per-element arithmetic does
not depend on the slicing, so over three steps -- the second with a non-finite value in the last slice only --
the slices' results put back together must equal the whole-space step bit for bit: the same t, skip flag,
master/m/v, replicas (and, with the device-resident loss scale, the same scale).  Two-pass steps in ring and
tree order, single-pass steps, fixed and dynamic loss scale.
"""
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from zero_gradient_sync_gb300 import sliced
from zero_gradient_sync_gb300.buffers import StepBuffers

import gpu_util as gu

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["tiny"]
CASES = [
    # psi, n, a, stage, layout, extra, slices
    (300_007, 4, 2, 3, "buckets", {"bucket": 70_001, "misalign": 3}, 2),
    (123_457, 8, 1, 1, "even", {}, 3),
    (200_003, 5, 3, 2, "random", {"nseg": 40}, 2),
    (100_001, 3, 2, 0, "ragged", {}, 2),
]


def slice_buffers(whole, L, lo, hi, single):
    """Buffers of the slice [lo, hi) holding whole's data for it."""
    S, base = L.slice(lo, hi)
    b = StepBuffers(S, whole.a, second_set=single)
    for x, y in zip(b.grads, whole.grads):
        x.copy_(y[lo:hi])
    for x, y in zip(b.replicas, whole.replicas):
        x.copy_(y[lo:hi])
    pairs = [(b.master, whole.master), (b.m, whole.m), (b.v, whole.v)]
    if single:
        pairs += [(b.master1, whole.master1), (b.m1, whole.m1), (b.v1, whole.v1)]
    for dst, src in pairs:
        if L.stage == 0:
            for x, y in zip(dst, src):
                x.copy_(y[lo:hi])
        else:
            for g, ln, o, loc in S.segs:
                dst[o][loc:loc + ln].copy_(src[o][base[o] + loc:base[o] + loc + ln])
    b.state.copy_(whole.state)
    return b, S, base


def snap_current(b, single):
    """Bytes of the current optimizer-state set and the replicas."""
    torch.cuda.synchronize()
    ms, mm, vv = b.current() if single else (b.master, b.m, b.v)
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in ms + mm + vv + b.replicas]


def assert_slices_equal_whole(whole, parts, L, single):
    torch.cuda.synchronize()
    ws = dp.read_state(whole.state)
    for b, S, base, lo, hi in parts:
        st = dp.read_state(b.state)
        for key in ("t", "found_inf", "error", "loss_scale", "good_steps", "cur_set", "b1t", "b2t"):
            assert st[key] == ws[key], key
        for x, y in zip(b.replicas, whole.replicas):
            assert torch.equal(x.view(torch.int16), y[lo:hi].view(torch.int16))
        sets = [(b.master, whole.master), (b.m, whole.m), (b.v, whole.v)]
        if single:
            sets += [(b.master1, whole.master1), (b.m1, whole.m1), (b.v1, whole.v1)]
        for dst, src in sets:
            if L.stage == 0:
                for x, y in zip(dst, src):
                    assert torch.equal(x.view(torch.int32), y[lo:hi].view(torch.int32))
            else:
                for g, ln, o, loc in S.segs:
                    assert torch.equal(dst[o][loc:loc + ln].view(torch.int32),
                                       src[o][base[o] + loc:base[o] + loc + ln].view(torch.int32))


@pytest.mark.parametrize("scaled", [False, True])
@pytest.mark.parametrize("single,order", [(False, 0), (True, 0), (False, dp.DP_ORDER_TREE), (True, dp.DP_ORDER_TREE)])
@pytest.mark.parametrize("psi,n,a,stage,layout,extra,G", CASES)
def test_slices_equal_whole_space_step(dev, psi, n, a, stage, layout, extra, G, single, order, scaled):
    if single and stage == 0:
        pytest.skip("the single pass takes stages 1-3")
    mode = dp.DP_SUM_COMPENSATED | order
    wl = BASE.with_(psi=psi, n=n, a=a, stage=stage, layout=layout, seed=500 + psi % 97, loss_scale=2.0 ** 10,
                    **extra)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    whole = gu.upload(c, second_set=single)
    if single:
        for x, y in zip(whole.master1 + whole.m1 + whole.v1, whole.master + whole.m + whole.v):
            x.copy_(y)
    sc = dp.scaler(2.0, 0.5, 2, 2.0 ** 8, 2.0 ** 24) if scaled else None
    if scaled:
        dp.dp_scaler_init(whole.state, wl.loss_scale)
    parts = []
    for j in range(G):
        lo, hi = sliced.slice_bounds(psi, G, j)
        b, S, base = slice_buffers(whole, c.layout, lo, hi, single)
        parts.append((b, S, base, lo, hi))
    ops = sliced.LibraryOps()
    for step in range(3):
        if step == 1:   # a NaN in the last slice only: every slice must skip
            b, S, base, lo, hi = parts[-1]
            i = (hi - lo) // 3
            whole.grad(n - 1, a - 1)[lo + i:lo + i + 1].view(torch.int16).fill_(synth.BF16_NAN)
            b.grad(n - 1, a - 1)[i:i + 1].view(torch.int16).fill_(synth.BF16_NAN)
            before = snap_current(whole, single)
        if step == 2:   # clean again
            b, S, base, lo, hi = parts[-1]
            i = (hi - lo) // 3
            src = synth.grads_bf16(wl, n - 1, a - 1, lo + i, 1)
            val = int(src.view("int16")[0])
            whole.grad(n - 1, a - 1)[lo + i:lo + i + 1].view(torch.int16).fill_(val)
            b.grad(n - 1, a - 1)[i:i + 1].view(torch.int16).fill_(val)
        # the whole space in one call
        if scaled and single:
            whole.step_single_pass(A, 1.0, mode | dp.DP_DEFER_COMMIT | dp.DP_DEVICE_SCALE)
            dp.dp_commit_single_pass(whole.replicas, whole.master + whole.master1, c.layout, A, whole.state, sc)
        elif scaled:
            whole.step_scaled(A, sc, mode)
        elif single:
            whole.step_single_pass(A, wl.loss_scale, mode)
        else:
            whole.step(A, wl.loss_scale, mode)
        # the slices: reduce each with the commit deferred, combine the flags, commit and update each
        for b, *_ in parts:
            sliced.reduce_deferred(b, A, wl.loss_scale, mode, single_pass=single, scaler_=sc)
        flags = [ops.found_flag(b) for b, *_ in parts]
        f = torch.stack(flags).max()
        for x in flags:
            x.copy_(f.view(1))
        for b, *_ in parts:
            sliced.commit_and_update(b, A, single_pass=single, scaler_=sc)
        st = dp.read_state(whole.state)
        assert st["found_inf"] == (1 if step == 1 else 0)
        assert st["t"] == (1 if step < 2 else 2)
        if step == 1:
            assert snap_current(whole, single) == before
        assert_slices_equal_whole(whole, parts, c.layout, single)
