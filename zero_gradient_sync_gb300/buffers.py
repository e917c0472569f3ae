"""Device buffers of one data-parallel step, allocated with PyTorch (memory and streams only).

StepBuffers holds, for a layout of n replicas and a micro-steps: the n*a bf16 gradient buffers (rank-major),
the n bf16 parameter replicas, each rank's fp32 master/m/v arrays (its shard, or full length for plain data
parallelism), the n fp32 averaged-gradient shards and the 64-byte device step state.  Every tensor is a
separate allocation, so every base pointer is 256-byte aligned.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import _lib
from ._lib import DP_SUM_COMPENSATED, Layout


class StepBuffers:
    def __init__(self, layout: Layout, a: int, device=None, with_grads: bool = True, second_set: bool = False,
                 micro_acc: bool = False):
        self.layout = layout
        self.n, self.a, self.psi = layout.n, int(a), layout.psi
        self.device = torch.device(device or "cuda")
        dev = self.device
        lens = layout.state_lens()
        shard = layout.shard_lens()
        self.grads: List[torch.Tensor] = (
            [torch.empty(self.psi, dtype=torch.bfloat16, device=dev) for _ in range(self.n * self.a)]
            if with_grads else [])
        self.replicas = [torch.empty(self.psi, dtype=torch.bfloat16, device=dev) for _ in range(self.n)]
        self.master = [torch.empty(L, dtype=torch.float32, device=dev) for L in lens]
        self.m = [torch.zeros(L, dtype=torch.float32, device=dev) for L in lens]
        self.v = [torch.zeros(L, dtype=torch.float32, device=dev) for L in lens]
        self.gbar = [torch.empty(L, dtype=torch.float32, device=dev) for L in shard]
        self.state = _lib.new_state(dev)
        # Single pass: a second master/m/v set; set 0 is master/m/v above.
        self.master1 = [torch.empty(L, dtype=torch.float32, device=dev) for L in lens] if second_set else []
        self.m1 = [torch.zeros(L, dtype=torch.float32, device=dev) for L in lens] if second_set else []
        self.v1 = [torch.zeros(L, dtype=torch.float32, device=dev) for L in lens] if second_set else []
        # Per-micro-step reduce-scatter: the owner shard accumulators, (hi, lo) pairs (enough for either mode).
        self.acc = [torch.empty(2 * L, dtype=torch.float32, device=dev) for L in shard] if micro_acc else []

    def step_micro(self, adam_: _lib.dp_adam_t, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED,
                   stream=None) -> None:
        """The step with a per-micro-step reduce-scatter (one call per micro-step), then the update."""
        for k in range(self.a):
            self.reduce_micro(k, adam_, loss_scale, sum_mode, stream)
        self.update(adam_, stream=stream)

    def reduce_micro(self, k: int, adam_: _lib.dp_adam_t, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED,
                     stream=None) -> None:
        _lib.dp_reduce_scatter_micro(self.acc, self.gbar, None, [self.grad(r, k) for r in range(self.n)], k, self.a,
                                     self.layout, adam_, loss_scale, sum_mode, self.state, stream=stream)

    def step_single_pass(self, adam_: _lib.dp_adam_t, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED,
                         stream=None) -> None:
        _lib.dp_step_single_pass(self.replicas, self.master + self.master1, self.m + self.m1, self.v + self.v1,
                                 self.grads, self.a, self.layout, adam_, loss_scale, sum_mode, state=self.state,
                                 stream=stream)

    def step_single_pass_from_host(self, host_grads, adam_: _lib.dp_adam_t, loss_scale: float,
                                   sum_mode: int = DP_SUM_COMPENSATED, host_state=None, stream=None) -> None:
        """One single-pass step with this step's gradients in host memory (copied into self.grads first)."""
        _lib.dp_step_single_pass_from_host(self.replicas, self.master + self.master1, self.m + self.m1,
                                           self.v + self.v1, host_grads, self.grads, self.a, self.layout, adam_,
                                           loss_scale, sum_mode, state=self.state, host_state=host_state,
                                           stream=stream)

    def current(self):
        """The current (master, m, v) set of a single-pass run."""
        cur = _lib.read_state(self.state)["cur_set"]
        return (self.master, self.m, self.v) if cur == 0 else (self.master1, self.m1, self.v1)

    def grad(self, r: int, k: int) -> torch.Tensor:
        return self.grads[r * self.a + k]

    def step(self, adam_: _lib.dp_adam_t, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED,
             stream=None) -> None:
        _lib.dp_step(self.replicas, self.master, self.m, self.v, self.grads, self.a, self.layout, adam_,
                     loss_scale, sum_mode, gbar_shard=self.gbar, state=self.state, stream=stream)

    def step_from_host(self, host_grads, adam_: _lib.dp_adam_t, loss_scale: float,
                       sum_mode: int = DP_SUM_COMPENSATED, host_state=None, stream=None) -> None:
        """One step with this step's gradients in host memory (copied into self.grads first)."""
        _lib.dp_step_from_host(self.replicas, self.master, self.m, self.v, host_grads, self.grads, self.a,
                               self.layout, adam_, loss_scale, sum_mode, gbar_shard=self.gbar, state=self.state,
                               host_state=host_state, stream=stream)

    def step_scaled(self, adam_: _lib.dp_adam_t, scaler_: _lib.dp_scaler_t, sum_mode: int = DP_SUM_COMPENSATED,
                    stream=None) -> None:
        _lib.dp_step_scaled(self.replicas, self.master, self.m, self.v, self.grads, self.a, self.layout, adam_,
                            scaler_, sum_mode, gbar_shard=self.gbar, state=self.state, stream=stream)

    def reduce(self, adam_: _lib.dp_adam_t, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED,
               stream=None) -> None:
        _lib.dp_step_reduce(self.gbar, None, self.grads, self.a, self.layout, adam_, loss_scale, sum_mode,
                            self.state, stream=stream)

    def update(self, adam_: _lib.dp_adam_t, stream=None) -> None:
        _lib.dp_step_update(self.replicas, self.master, self.m, self.v, self.gbar, None, self.layout, adam_,
                            self.state, stream=stream)

    def status(self, stream=None):
        return _lib.dp_read_status(self.state, stream=stream)

    def nbytes(self) -> int:
        ts = self.grads + self.replicas + self.master + self.m + self.v + self.gbar
        return sum(t.numel() * t.element_size() for t in ts) + _lib.STATE_BYTES
