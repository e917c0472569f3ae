"""The step split across processes by slices of the parameter space, on CPU (gloo, world size 2).

Each process holds one contiguous slice of the space with all n ranks' data for it (slice_bounds,
Layout.slice -- the library's own host code) and runs step_sliced: the reduction with the commit deferred,
a real 4-byte MAX all-reduce of found_inf over the gloo group, then the commit and the update.  The
per-slice arithmetic comes from an ops object backed by the float64 oracle (this machine has no GPU), so
what is tested is the slicing and the commit protocol:
  - clean step: both processes commit, t = 1 on both, and the slices' results put back together equal the
    whole-space oracle step bit for bit (slicing maps every element to its owner's shard correctly);
  - a +inf in one micro-step of rank-1's slice: process 0's own slice is clean, yet both processes skip,
    t stays 0 on both and every array is unchanged.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _workload():
    import synth
    return synth.WORKLOADS["tiny"].with_(psi=20_011, n=4, a=2, stage=3, layout="buckets", bucket=3001, misalign=3,
                                         seed=77)


class SliceState:
    """One process's slice on the host: inputs, shard pieces, replicas and the commit state."""

    def __init__(self, wl, layout, lo, hi, inject: bool):
        import synth
        S, base = layout.slice(lo, hi)
        self.wl, self.layout, self.lo, self.hi, self.base = wl, S, lo, hi, base
        self.grads = [synth.grads_bf16(wl, r, k, lo, hi - lo) for r in range(wl.n) for k in range(wl.a)]
        if inject:
            self.grads[1 * wl.a + 1][(hi - lo) // 2] = synth.BF16_POS_INF
        full = synth.master_f32(wl)
        lens = S.shard_lens()
        self.master = [np.zeros(L, np.float32) for L in lens]
        for g, ln, o, loc in S.segs:
            self.master[o][loc:loc + ln] = full[lo + g:lo + g + ln]
        self.m = [np.zeros(L, np.float32) for L in lens]
        self.v = [np.zeros(L, np.float32) for L in lens]
        self.replicas = [np.zeros(hi - lo, np.uint16) for _ in range(wl.n)]
        self.t = 0
        self.flag = torch.zeros(1, dtype=torch.int32)
        self.pending = None


class OracleOps:
    """The phases of step_sliced with the oracle's arithmetic on a SliceState (host memory)."""

    def reduce(self, b, adam_, loss_scale, sum_mode, single_pass):
        import oracle
        from zero_gradient_sync_gb300 import DP_DEFER_COMMIT
        assert sum_mode & DP_DEFER_COMMIT, "a sliced step defers its commit"
        wl = b.wl
        res = [[x.copy() for x in arrs] for arrs in (b.master, b.m, b.v, b.replicas)]
        out = oracle.step(b.hi - b.lo, wl.n, wl.a, wl.stage, b.layout.segs, b.grads, *res, wl.lr, wl.beta1,
                          wl.beta2, wl.eps, loss_scale, b.t)
        b.flag[0] = out["found"]
        b.pending = (res, out["t"])

    def found_flag(self, b):
        return b.flag

    def commit(self, b, adam_, scaler_, single_pass):
        if int(b.flag[0]) == 0:
            (b.master, b.m, b.v, b.replicas), b.t = b.pending
        b.pending = None

    def update(self, b, adam_, single_pass):
        pass


def _worker(rank, world, port, inject_rank, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import synth
    import zero_gradient_sync_gb300 as dp
    from zero_gradient_sync_gb300 import sliced
    wl = _workload()
    L = dp.Layout(wl.stage, wl.n, wl.psi, synth.layout_of(wl))
    lo, hi = sliced.slice_bounds(wl.psi, world, rank)
    b = SliceState(wl, L, lo, hi, inject=(rank == inject_rank))
    before = [x.copy() for arrs in (b.master, b.m, b.v, b.replicas) for x in arrs]
    sliced.step_sliced(b, dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps), wl.loss_scale,
                       lambda f: tdist.all_reduce(f, op=tdist.ReduceOp.MAX), ops=OracleOps())
    after = [x.copy() for arrs in (b.master, b.m, b.v, b.replicas) for x in arrs]
    unchanged = all(np.array_equal(x.view(np.uint8), y.view(np.uint8)) for x, y in zip(before, after))
    out.put((rank, lo, hi, b.base, b.layout.segs, b.t, int(b.flag[0]), unchanged, b.master, b.m, b.v,
             b.replicas))
    tdist.barrier()
    tdist.destroy_process_group()


def _run(inject_rank):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, inject_rank, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=180) for _ in range(2)], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return res


def test_two_slices_equal_the_whole_space_step():
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    wl = _workload()
    res = _run(inject_rank=-1)
    assert [r[5] for r in res] == [1, 1] and [r[6] for r in res] == [0, 0]
    assert res[0][1] == 0 and res[0][2] == res[1][1] and res[1][2] == wl.psi
    # the whole-space step, and the slices' results put back into whole shard arrays
    segs = synth.layout_of(wl)
    lens = synth.shard_lengths(segs, wl.n)
    full = synth.master_f32(wl)
    M = [np.zeros(L, np.float32) for L in lens]
    for g, ln, o, loc in segs:
        M[o][loc:loc + ln] = full[g:g + ln]
    Mm = [np.zeros(L, np.float32) for L in lens]
    Vv = [np.zeros(L, np.float32) for L in lens]
    reps = [np.zeros(wl.psi, np.uint16) for _ in range(wl.n)]
    grads = [synth.grads_bf16(wl, r, k) for r in range(wl.n) for k in range(wl.a)]
    out = oracle.step(wl.psi, wl.n, wl.a, wl.stage, segs, grads, M, Mm, Vv, reps, wl.lr, wl.beta1, wl.beta2,
                      wl.eps, wl.loss_scale, 0)
    assert (out["found"], out["t"]) == (0, 1)
    got = [[np.full(L, np.nan, np.float32) for L in lens] for _ in range(3)]
    got_reps = [np.zeros(wl.psi, np.uint16) for _ in range(wl.n)]
    for rank, lo, hi, base, ssegs, t, flag, unchanged, sm, smm, sv, sreps in res:
        for g, ln, o, loc in ssegs:
            for dst, src in zip(got, (sm, smm, sv)):
                dst[o][base[o] + loc:base[o] + loc + ln] = src[o][loc:loc + ln]
        for r in range(wl.n):
            got_reps[r][lo:hi] = sreps[r]
    for dst, ref in zip(got, (M, Mm, Vv)):
        for x, y in zip(dst, ref):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    for x, y in zip(got_reps, reps):
        assert np.array_equal(x, y)


def test_inf_in_one_slice_skips_every_slice():
    res = _run(inject_rank=1)
    for rank, lo, hi, base, ssegs, t, flag, unchanged, *_ in res:
        assert flag == 1, rank        # process 0's own slice was clean; the all-reduce brought rank 1's flag
        assert t == 0, rank
        assert unchanged, rank


def test_slice_bounds_cover_the_space():
    sys.path.insert(0, ROOT)
    from zero_gradient_sync_gb300.sliced import slice_bounds
    for psi, G in ((0, 1), (7, 3), (10 ** 9 + 7, 8), (5, 8)):
        b = [slice_bounds(psi, G, j) for j in range(G)]
        assert b[0][0] == 0 and b[-1][1] == psi
        assert all(x[1] == y[0] for x, y in zip(b, b[1:]))
        assert max(h - l for l, h in b) - min(h - l for l, h in b) <= 1
    with pytest.raises(ValueError):
        slice_bounds(10, 0, 0)
