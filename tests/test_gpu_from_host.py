"""dp_step_from_host: the step with its gradients in (pinned) host memory, through the C ABI (-m gpu).

It must give exactly dp_step's results on the same gradients -- the copies change where the bytes come from,
not the arithmetic -- over consecutive steps with new gradients each time, and return the step state in the
caller's host buffer."""
import numpy as np
import pytest
import torch

import synth
import zero_gradient_sync_gb300 as dp

import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [dp.DP_SUM_COMPENSATED, dp.DP_SUM_PLAIN])
def test_from_host_equals_device_step(dev, mode):
    wl = synth.WORKLOADS["tiny"].with_(psi=200_003, n=4, a=2, stage=3, layout="ragged", seed=77)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    ref, got = gu.upload(c), gu.upload(c)
    host_state = torch.empty(dp.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
    for step in range(3):
        w = wl.with_(seed=wl.seed + step)
        host = [torch.from_numpy(synth.grads_bf16(w, q // wl.a, q % wl.a).view(np.int16)).pin_memory()
                for q in range(wl.n * wl.a)]
        for q, h in enumerate(host):
            ref.grads[q].view(torch.int16).copy_(h)
        for g in got.grads:          # stale device gradients: the call must overwrite them
            g.zero_()
        ref.step(A, wl.loss_scale, mode)
        got.step_from_host(host, A, wl.loss_scale, mode, host_state=host_state)
        torch.cuda.synchronize()
        assert gu.snapshot(got) == gu.snapshot(ref)
        st = dp.read_state(got.state)
        hs = np.frombuffer(host_state.numpy().tobytes(), dtype=np.uint8)
        assert hs.tobytes() == got.state.cpu().numpy().tobytes()
        assert st["t"] == step + 1 and st["found_inf"] == 0


def test_from_host_skip_leaves_state(dev):
    """A non-finite value in the host gradients skips the step exactly as on the device path."""
    wl = synth.WORKLOADS["tiny"].with_(psi=50_001, n=2, a=1, stage=1, layout="even", seed=78)
    c = gu.make_case(wl)
    b = gu.upload(c)
    before = gu.snapshot(b)
    host = [torch.from_numpy(synth.grads_bf16(wl, r, 0).view(np.int16)).pin_memory() for r in range(wl.n)]
    host[1][12345] = 0x7F80          # +inf in bf16
    host_state = torch.empty(dp.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
    b.step_from_host(host, dp.adam(), wl.loss_scale, host_state=host_state)
    torch.cuda.synchronize()
    st = dp.read_state(b.state)
    assert st["found_inf"] == 1 and st["t"] == 0 and st["nonfinite"] >= 1
    assert gu.snapshot(b) == before   # master, m, v and replicas bit for bit


def _current(b):
    torch.cuda.synchronize()
    ms, mm, vv = b.current()
    return [t.detach().cpu().view(torch.uint8).numpy().tobytes() for t in ms + mm + vv + b.replicas]


@pytest.mark.parametrize("mode", [dp.DP_SUM_COMPENSATED, dp.DP_SUM_PLAIN])
def test_single_pass_from_host_equals_device_single_pass(dev, mode):
    """dp_step_single_pass_from_host (the benchmark's end-to-end call) gives exactly dp_step_single_pass's results
    on the same gradients over consecutive steps, the third with a NaN (skipped: the current set, the replicas
    and t kept), and returns the step state in the caller's host buffer."""
    wl = synth.WORKLOADS["tiny"].with_(psi=200_003, n=4, a=2, stage=2, layout="buckets", bucket=50_000,
                                       misalign=3, seed=79)
    c = gu.make_case(wl)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)
    ref, got = gu.upload(c, second_set=True), gu.upload(c, second_set=True)
    host_state = torch.empty(dp.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
    for step in range(3):
        w = wl.with_(seed=wl.seed + step)
        host = [torch.from_numpy(synth.grads_bf16(w, q // wl.a, q % wl.a).view(np.int16)).pin_memory()
                for q in range(wl.n * wl.a)]
        if step == 2:
            host[5][4321] = synth.BF16_NAN
        for q, h in enumerate(host):
            ref.grads[q].view(torch.int16).copy_(h)
        for g in got.grads:          # stale device gradients: the call must overwrite them
            g.zero_()
        ref.step_single_pass(A, wl.loss_scale, mode)
        got.step_single_pass_from_host(host, A, wl.loss_scale, mode, host_state=host_state)
        torch.cuda.synchronize()
        assert _current(got) == _current(ref)
        st = dp.read_state(got.state)
        assert np.frombuffer(host_state.numpy().tobytes(), dtype=np.uint8).tobytes() == got.state.cpu().numpy().tobytes()
        assert (st["t"], st["found_inf"]) == ((2, 1) if step == 2 else (step + 1, 0))
