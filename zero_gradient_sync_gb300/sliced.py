"""The step split across G GPUs by contiguous slices of the flat parameter space, with one global skip decision.

GPU j holds slice j = [lo_j, hi_j) of the space with all n ranks' data for it: the n*a gradient pieces, the n
replica pieces, and each rank's optimizer-state pieces (Layout.slice gives the slice's own layout and where its
shard pieces start in the ranks' whole shards).  Every step of the path is elementwise over the space, so each
GPU runs the step on its slice alone, with no data exchange.  One thing crosses slices: the skip decision.  A
non-finite value anywhere must skip the step everywhere ("Distributed Training: Split along the Four Axes",
data-parallel paragraph: every rank applies the same update, so the replicas stay identical), so a sliced step
is

    1. the reduction of this slice with DP_DEFER_COMMIT (found_inf published, nothing committed);
    2. found_inf combined over all slices with a maximum -- one 4-byte all-reduce;
    3. the commit (t, beta powers, state set, loss scale: all or nothing) and the update of this slice.

The calls of each phase come from an ops object (LibraryOps: the C ABI on a StepBuffers); a multi-process test
without GPUs substitutes its own.
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple

from . import _lib
from ._lib import DP_DEFER_COMMIT, DP_DEVICE_SCALE, DP_SUM_COMPENSATED


def slice_bounds(psi: int, slices: int, j: int) -> Tuple[int, int]:
    """Slice j of `slices` contiguous slices of [0, psi): the first psi mod slices slices one element longer."""
    if slices < 1 or not 0 <= j < slices or psi < 0:
        raise ValueError("slice %d of %d over psi = %d" % (j, slices, psi))
    base, extra = divmod(psi, slices)
    lo = j * base + min(j, extra)
    return lo, lo + base + (1 if j < extra else 0)


class LibraryOps:
    """The phases of a sliced step as calls of the library on one slice's StepBuffers."""

    def reduce(self, b, adam_, loss_scale: float, sum_mode: int, single_pass: bool) -> None:
        if single_pass:
            b.step_single_pass(adam_, loss_scale, sum_mode)
        else:
            b.reduce(adam_, loss_scale, sum_mode)

    def found_flag(self, b):
        """found_inf of the slice's step state, as a one-element int32 tensor viewing the state (byte offset 4):
        the operand of the all-reduce."""
        import torch
        return b.state[4:8].view(torch.int32)

    def commit(self, b, adam_, scaler_, single_pass: bool) -> None:
        if single_pass:
            _lib.dp_commit_single_pass(b.replicas, b.master + b.master1, b.layout, adam_, b.state, scaler_)
        else:
            _lib.dp_commit_step(b.state, adam_, scaler_)

    def update(self, b, adam_, single_pass: bool) -> None:
        if not single_pass:
            b.update(adam_)


def reduce_deferred(b, adam_, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED, single_pass: bool = False,
                    scaler_: Optional[_lib.dp_scaler_t] = None, ops=None) -> None:
    """Phase 1 on one slice.  With a scaler the reduction unscales by the device-resident scale (DP_DEVICE_SCALE)
    and loss_scale is not used."""
    ops = ops or LibraryOps()
    mode = sum_mode | DP_DEFER_COMMIT | (DP_DEVICE_SCALE if scaler_ is not None else 0)
    ops.reduce(b, adam_, loss_scale, mode, single_pass)


def commit_and_update(b, adam_, single_pass: bool = False, scaler_: Optional[_lib.dp_scaler_t] = None,
                      ops=None) -> None:
    """Phase 3 on one slice, once its found_inf holds the maximum over all slices."""
    ops = ops or LibraryOps()
    ops.commit(b, adam_, scaler_, single_pass)
    ops.update(b, adam_, single_pass)


def step_sliced(b, adam_, loss_scale: float, combine_max: Callable, sum_mode: int = DP_SUM_COMPENSATED,
                single_pass: bool = False, scaler_: Optional[_lib.dp_scaler_t] = None, ops=None) -> None:
    """One step of this process's slice.  combine_max(flag) must turn the one-element int32 flag, in place, into
    its maximum over every slice's process -- e.g. torch.distributed.all_reduce(flag, op=ReduceOp.MAX)."""
    ops = ops or LibraryOps()
    reduce_deferred(b, adam_, loss_scale, sum_mode, single_pass, scaler_, ops)
    combine_max(ops.found_flag(b))
    commit_and_update(b, adam_, single_pass, scaler_, ops)
