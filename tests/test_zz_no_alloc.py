"""dp_step_static: the fused step for callers that cannot allocate device memory (-m gpu).

Some callers cannot call cudaMalloc themselves -- for example a plugin inside a runtime that owns and
pre-plans all device memory, or a training loop that must not allocate once it is running.  For them
dp_step_static keeps dp_step's scratch (the averaged-gradient shards) in a fixed array inside the library,
so they pass only inputs and outputs.  These tests call it through the C ABI and check it against dp_step
on two steps in a row, with the parity tolerance of the other GPU tests, check that a call allocates no
device memory, and check that a layout too large for the array is refused before anything is launched.
"""
import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp
from synth import device as sd

import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_static_scratch_step_matches_dp_step_on_two_calls(dev):
    wl = synth.WORKLOADS["tiny"].with_(psi=1_000_003, n=4, a=2, stage=2, layout="ragged", seed=123)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    ref = gu.upload(c)     # dp_step with caller-allocated gradient shards
    got = gu.upload(c)     # dp_step_static, no scratch from the caller
    for call in range(2):
        if call == 1:      # the second step sees new gradients
            wl2 = wl.with_(seed=wl.seed + 1)
            for q in range(wl.n * wl.a):
                g = sd.bf16_from_bits(synth.grads_bf16(wl2, q // wl.a, q % wl.a))
                ref.grads[q].copy_(g)
                got.grads[q].copy_(g)
        dp.dp_step(ref.replicas, ref.master, ref.m, ref.v, ref.grads, wl.a, c.layout, A, wl.loss_scale,
                   gbar_shard=ref.gbar, state=ref.state)
        torch.cuda.synchronize()
        free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
        dp.dp_step_static(got.replicas, got.master, got.m, got.v, got.grads, wl.a, c.layout, A, wl.loss_scale,
                          state=got.state)
        torch.cuda.synchronize()
        # No call allocates: the device's free memory and torch's pool are unchanged by the call.  (The first
        # call on a device may load the library's module that holds the array; later calls change nothing.)
        assert torch.cuda.memory_reserved() == reserved0
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free0
        r, g = gu.gpu_result(c, ref), gu.gpu_result(c, got)
        assert (g["found"], g["nonfinite"], g["t"], g["error"]) == (r["found"], r["nonfinite"], r["t"], r["error"])
        assert g["t"] == call + 1
        gu.assert_close_f32(g["master"], r["master"], "master")
        gu.assert_close_f32(g["m"], r["m"], "m")
        gu.assert_close_f32(g["v"], r["v"], "v")
        gu.assert_replicas(g["replicas"], r["replicas"])


def test_static_scratch_refuses_a_layout_too_large(dev):
    psi, n = 20_000_000, 4           # 80 MB of gradient shards: more than the 64 MiB array
    L = dp.Layout(1, n, psi, synth.layout_even(psi, n))
    assert L.workspace_size() > dp._lib.STATIC_SCRATCH_BYTES
    fake = [256 * (k + 1) for k in range(n * 2)]   # never dereferenced: the size check comes first
    before = dp.dp_kernel_launches()
    with pytest.raises(dp.DPError) as e:
        dp.dp_step_static(fake[:n], fake[:n], fake[:n], fake[:n], fake[:n * 1], 1, L, dp.adam(), 1.0, state=256)
    assert e.value.code == dp.DP_ERR_INVALID_ARG
    assert "static scratch" in str(e.value)
    assert dp.dp_kernel_launches() == before
