"""ctypes binding of libdpstep.so: the C entry points under the same names.

Argument marshalling only -- tensors become device pointers, streams become
cudaStream_t handles, layouts become dp_layout_t structs.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback: if the
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdpstep.so")

DP_OK, DP_ERR_INVALID_ARG, DP_ERR_ALIGNMENT, DP_ERR_CUDA, DP_ERR_TIMEOUT, DP_ERR_IO = 0, 1, 2, 3, 4, 5
DP_SUM_COMPENSATED, DP_SUM_PLAIN = 0, 1
DP_ORDER_RING, DP_ORDER_TREE = 0, 16   # OR'd into sum_mode
DP_DEFER_COMMIT, DP_DEVICE_SCALE = 32, 64   # step flags, OR'd into sum_mode
DP_MAX_N, DP_MAX_NA, DP_MAX_SEG, DP_KERNEL_SEG = 16, 64, 1 << 20, 1024
STATE_BYTES = 64

c_i32, c_i64, c_u64, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p


class dp_segment_t(ctypes.Structure):
    _fields_ = [("global_off", c_i64), ("len", c_i64), ("owner", c_i32), ("reserved", c_i32), ("local_off", c_i64)]


class dp_layout_t(ctypes.Structure):
    _fields_ = [("stage", c_i32), ("n", c_i32), ("psi", c_i64), ("nseg", c_i32), ("reserved", c_i32),
                ("seg", ctypes.POINTER(dp_segment_t))]


class dp_adam_t(ctypes.Structure):
    _fields_ = [("lr", c_f32), ("beta1", c_f32), ("beta2", c_f32), ("eps", c_f32)]


class dp_step_state_t(ctypes.Structure):
    _fields_ = [("t", c_i32), ("found_inf", c_i32), ("error", c_i32), ("good_steps", c_i32), ("nonfinite", c_u64),
                ("b1t", ctypes.c_double), ("b2t", ctypes.c_double), ("work_count", c_u64),
                ("work_found", ctypes.c_uint32), ("work_ticket", ctypes.c_uint32), ("loss_scale", c_f32),
                ("cur_set", ctypes.c_uint32)]


class dp_scaler_t(ctypes.Structure):
    _fields_ = [("growth_factor", c_f32), ("backoff_factor", c_f32), ("growth_interval", c_i32),
                ("min_scale", c_f32), ("max_scale", c_f32)]


assert ctypes.sizeof(dp_step_state_t) == STATE_BYTES
assert ctypes.sizeof(dp_segment_t) == 32


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libdpstep.so is not built (run zero_gradient_sync_gb300.build.build()); "
                          "there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "dp_abi_version": (c_i32, []),
        "dp_status_str": (ctypes.c_char_p, [c_i32]),
        "dp_last_error": (ctypes.c_char_p, []),
        "dp_layout_validate": (c_i32, [P(dp_layout_t)]),
        "dp_layout_even": (c_i32, [c_i64, c_i32, c_i64, c_i32, P(dp_segment_t), P(c_i32)]),
        "dp_layout_slice": (c_i32, [P(dp_layout_t), c_i64, c_i64, P(dp_segment_t), P(c_i32), P(c_i64)]),
        "dp_commit_step": (c_i32, [c_vp, dp_adam_t, P(dp_scaler_t), c_vp]),
        "dp_commit_single_pass": (c_i32, [c_vp, c_vp, P(dp_layout_t), dp_adam_t, P(dp_scaler_t), c_vp, c_vp]),
        "dp_step_single_pass_from_host": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t,
                                                  c_f32, c_i32, c_vp, c_vp, c_vp]),
        "dp_shard_len": (c_i64, [P(dp_layout_t), c_i32]),
        "dp_workspace_size": (ctypes.c_size_t, [P(dp_layout_t)]),
        "dp_acc_elems": (ctypes.c_size_t, [c_i64, c_i32]),
        "dp_global_batch": (c_i64, [c_i64, c_i32, c_i32]),
        "dp_memory_model": (c_i32, [c_i32, c_i64, c_i32, P(ctypes.c_double)]),
        "dp_traffic_model": (c_i32, [c_i32, c_i64, c_i32, c_i32, c_i32, P(ctypes.c_double)]),
        "dp_set_wait_timeout_ns": (None, [c_u64]),
        "dp_get_wait_timeout_ns": (c_u64, []),
        "dp_kernel_launches": (c_u64, []),
        "dp_state_init": (c_i32, [c_vp, c_vp]),
        "dp_accumulate": (c_i32, [c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_vp]),
        "dp_reduce_scatter_avg": (c_i32, [c_vp, c_vp, P(dp_layout_t), c_f32, c_i32, c_vp, c_vp]),
        "dp_adam_shard": (c_i32, [c_vp, c_vp, c_vp, c_vp, P(dp_layout_t), dp_adam_t, c_vp, c_vp]),
        "dp_allgather_params": (c_i32, [c_vp, c_vp, P(dp_layout_t), c_vp, c_vp]),
        "dp_step": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t, c_f32, c_i32, c_vp,
                            c_vp, c_vp, c_vp]),
        "dp_step_from_host": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t, c_f32,
                                      c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
        "dp_step_reduce": (c_i32, [c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t, c_f32, c_i32, c_vp, c_vp]),
        "dp_step_update": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, P(dp_layout_t), dp_adam_t, c_vp, c_vp]),
        "dp_read_status": (c_i32, [c_vp, P(c_i32), P(c_i32), c_vp]),
        "dp_selftest_wait_timeout": (c_i32, [c_vp, c_u64, c_vp]),
        "dp_scaler_init": (c_i32, [c_vp, c_f32, c_vp]),
        "dp_step_scaled": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t, P(dp_scaler_t), c_i32,
                                   c_vp, c_vp, c_vp, c_vp]),
        "dp_step_single_pass": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t, c_f32, c_i32,
                                        c_vp, c_vp]),
        "dp_step_static": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, P(dp_layout_t), dp_adam_t, c_f32, c_i32,
                                   c_vp, c_vp]),
        "dp_reduce_scatter_micro": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, P(dp_layout_t), dp_adam_t, c_f32,
                                            c_i32, c_vp, c_vp]),
        "dp_checkpoint_save": (c_i32, [ctypes.c_char_p, ctypes.c_char_p, P(dp_layout_t), c_vp, c_vp, c_vp, c_vp, c_vp,
                                       c_u64, c_i32, c_vp]),
        "dp_checkpoint_load": (c_i32, [ctypes.c_char_p, ctypes.c_char_p, P(dp_layout_t), c_vp, c_vp, c_vp, c_vp, c_vp,
                                       P(c_u64), c_i32, c_i32, c_vp]),
        "dp_checkpoint_info": (c_i32, [ctypes.c_char_p, ctypes.c_char_p, c_i32, P(c_i32), P(c_i32), P(c_i64),
                                       P(c_i32), P(dp_segment_t), c_i32, P(c_u64)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


LIB = _load()


class DPError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = LIB.dp_last_error().decode(errors="replace")
        super().__init__("%s: %s (%s)" % (where, LIB.dp_status_str(code).decode(), msg))


def _check(rc: int, where: str) -> None:
    if rc != DP_OK:
        raise DPError(rc, where)


# ------------------------------------------------------------------------------------------- marshalling

def _ptr(t) -> int:
    """Device address of a tensor (or an int address, or None -> NULL)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ptr_array(ts: Optional[Sequence]):
    if ts is None:
        return None
    arr = (c_vp * max(1, len(ts)))(*[_ptr(t) for t in ts])
    return arr


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_tensors(ts: Sequence, itemsize: int, min_numel: Sequence[int], name: str) -> None:
    for i, t in enumerate(ts):
        if isinstance(t, int):
            continue
        if not t.is_cuda:
            raise ValueError("%s[%d] must be a CUDA tensor" % (name, i))
        if not t.is_contiguous():
            raise ValueError("%s[%d] must be contiguous" % (name, i))
        if t.element_size() != itemsize:
            raise ValueError("%s[%d]: element size %d, expected %d" % (name, i, t.element_size(), itemsize))
        if t.numel() < min_numel[i]:
            raise ValueError("%s[%d]: %d elements, need %d" % (name, i, t.numel(), min_numel[i]))


class Layout:
    """A dp_layout_t plus the segment array it points to (kept alive with it)."""

    def __init__(self, stage: int, n: int, psi: int, segs: Sequence[Tuple[int, int, int, int]]):
        self.stage, self.n, self.psi = int(stage), int(n), int(psi)
        self.segs = [tuple(int(x) for x in s) for s in segs]
        self._arr = (dp_segment_t * max(1, len(self.segs)))()
        for k, (g, ln, o, lo) in enumerate(self.segs):
            self._arr[k] = dp_segment_t(g, ln, o, 0, lo)
        self.c = dp_layout_t(self.stage, self.n, self.psi, len(self.segs), 0,
                             ctypes.cast(self._arr, ctypes.POINTER(dp_segment_t)))

    @classmethod
    def even(cls, psi: int, n: int, stage: int = 1, bucket: int = 0, misalign: int = 0) -> "Layout":
        cnt = c_i32(0)
        _check(LIB.dp_layout_even(psi, n, bucket, misalign, None, ctypes.byref(cnt)), "dp_layout_even")
        arr = (dp_segment_t * max(1, cnt.value))()
        _check(LIB.dp_layout_even(psi, n, bucket, misalign, arr, ctypes.byref(cnt)), "dp_layout_even")
        return cls(stage, n, psi, [(arr[k].global_off, arr[k].len, arr[k].owner, arr[k].local_off)
                                   for k in range(cnt.value)])

    def validate(self) -> None:
        _check(LIB.dp_layout_validate(ctypes.byref(self.c)), "dp_layout_validate")

    def shard_len(self, rank: int) -> int:
        v = LIB.dp_shard_len(ctypes.byref(self.c), rank)
        if v < 0:
            raise DPError(DP_ERR_INVALID_ARG, "dp_shard_len")
        return int(v)

    def shard_lens(self) -> List[int]:
        return [self.shard_len(r) for r in range(self.n)]

    def state_lens(self) -> List[int]:
        """Length of each rank's master/m/v arrays: its shard, or psi for plain data parallelism."""
        return [self.psi] * self.n if self.stage == 0 else self.shard_lens()

    def workspace_size(self) -> int:
        return int(LIB.dp_workspace_size(ctypes.byref(self.c)))

    def slice(self, lo: int, hi: int) -> Tuple["Layout", List[int]]:
        """The part of this layout inside global [lo, hi) as a layout of its own (dp_layout_slice), and each
        rank's local_base: where the slice's shard array starts in that rank's whole shard array."""
        cnt = c_i32(0)
        _check(LIB.dp_layout_slice(ctypes.byref(self.c), lo, hi, None, ctypes.byref(cnt), None), "dp_layout_slice")
        arr = (dp_segment_t * max(1, cnt.value))()
        base = (c_i64 * max(1, self.n))()
        _check(LIB.dp_layout_slice(ctypes.byref(self.c), lo, hi, arr, ctypes.byref(cnt), base), "dp_layout_slice")
        segs = [(arr[k].global_off, arr[k].len, arr[k].owner, arr[k].local_off) for k in range(cnt.value)]
        return Layout(self.stage, self.n, hi - lo, segs), [int(base[r]) for r in range(self.n)]


def adam(lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8) -> dp_adam_t:
    return dp_adam_t(lr, beta1, beta2, eps)


# ------------------------------------------------------------------------------------------- entry points

def dp_state_init(state, stream=None) -> None:
    _check(LIB.dp_state_init(_ptr(state), _stream(stream)), "dp_state_init")


def dp_accumulate(acc, g, psi: int, n: int, first: bool, sum_mode: int = DP_SUM_COMPENSATED, stream=None) -> None:
    _check_tensors(acc, 4, [int(LIB.dp_acc_elems(psi, sum_mode))] * n, "acc")
    _check_tensors(g, 2, [psi] * n, "g")
    _check(LIB.dp_accumulate(_ptr_array(acc), _ptr_array(g), psi, n, 1 if first else 0, sum_mode, _stream(stream)),
           "dp_accumulate")


def dp_reduce_scatter_avg(gbar_shard, acc, layout: Layout, loss_scale: float, sum_mode: int, state,
                          stream=None) -> None:
    _check_tensors(gbar_shard, 4, layout.shard_lens(), "gbar_shard")
    _check_tensors(acc, 4, [int(LIB.dp_acc_elems(layout.psi, sum_mode))] * layout.n, "acc")
    _check(LIB.dp_reduce_scatter_avg(_ptr_array(gbar_shard), _ptr_array(acc), ctypes.byref(layout.c), loss_scale,
                                     sum_mode, _ptr(state), _stream(stream)), "dp_reduce_scatter_avg")


def dp_adam_shard(master, m, v, gbar_shard, layout: Layout, adam_: dp_adam_t, state, stream=None) -> None:
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        _check_tensors(ts, 4, lens, name)
    _check_tensors(gbar_shard, 4, layout.shard_lens(), "gbar_shard")
    _check(LIB.dp_adam_shard(_ptr_array(master), _ptr_array(m), _ptr_array(v), _ptr_array(gbar_shard),
                             ctypes.byref(layout.c), adam_, _ptr(state), _stream(stream)), "dp_adam_shard")


def dp_allgather_params(replicas, master, layout: Layout, state, stream=None) -> None:
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(master, 4, layout.state_lens(), "master")
    _check(LIB.dp_allgather_params(_ptr_array(replicas), _ptr_array(master), ctypes.byref(layout.c), _ptr(state),
                                   _stream(stream)), "dp_allgather_params")


def _gbar_args(layout: Layout, gbar_shard, ws):
    if gbar_shard is not None:
        _check_tensors(gbar_shard, 4, layout.shard_lens(), "gbar_shard")
    if ws is not None and not isinstance(ws, int) and ws.numel() * ws.element_size() < layout.workspace_size():
        raise ValueError("workspace smaller than dp_workspace_size")
    return _ptr_array(gbar_shard), _ptr(ws)


def dp_step(replicas, master, m, v, grads, a: int, layout: Layout, adam_: dp_adam_t, loss_scale: float,
            sum_mode: int = DP_SUM_COMPENSATED, gbar_shard=None, ws=None, state=None, stream=None) -> None:
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    gb, w = _gbar_args(layout, gbar_shard, ws)
    _check(LIB.dp_step(_ptr_array(replicas), _ptr_array(master), _ptr_array(m), _ptr_array(v), _ptr_array(grads), a,
                       ctypes.byref(layout.c), adam_, loss_scale, sum_mode, gb, w, _ptr(state), _stream(stream)),
           "dp_step")


def _host_args(layout: Layout, host_grads, grads, host_state):
    """Host gradient pointer array and host state address of the *_from_host calls."""
    if len(host_grads) != len(grads):
        raise ValueError("host_grads: %d buffers for %d device buffers" % (len(host_grads), len(grads)))
    for i, h in enumerate(host_grads):
        if h.is_cuda or h.element_size() != 2 or not h.is_contiguous() or h.numel() < layout.psi:
            raise ValueError("host_grads[%d] must be a contiguous CPU tensor of >= psi 2-byte elements" % i)
    hs = 0
    if host_state is not None:
        if host_state.is_cuda or host_state.numel() * host_state.element_size() < STATE_BYTES:
            raise ValueError("host_state must be a CPU tensor of at least %d bytes" % STATE_BYTES)
        hs = host_state.data_ptr()
    return (c_vp * max(1, len(host_grads)))(*[h.data_ptr() for h in host_grads]), hs


def dp_step_from_host(replicas, master, m, v, host_grads, grads, a: int, layout: Layout, adam_: dp_adam_t,
                      loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED, gbar_shard=None, ws=None, state=None,
                      host_state=None, stream=None) -> None:
    """dp_step with the gradients in host memory: host_grads (CPU tensors, pinned for asynchronous copies, 2-byte
    elements) are copied into the device buffers grads on the stream, then the step runs; host_state (a CPU
    uint8 tensor of STATE_BYTES, or None) receives the step state afterwards."""
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    hp, hs = _host_args(layout, host_grads, grads, host_state)
    gb, w = _gbar_args(layout, gbar_shard, ws)
    _check(LIB.dp_step_from_host(_ptr_array(replicas), _ptr_array(master), _ptr_array(m), _ptr_array(v), hp,
                                 _ptr_array(grads), a, ctypes.byref(layout.c), adam_, loss_scale, sum_mode, gb, w,
                                 _ptr(state), hs, _stream(stream)), "dp_step_from_host")


def dp_step_reduce(gbar_shard, ws, grads, a: int, layout: Layout, adam_: dp_adam_t, loss_scale: float,
                   sum_mode: int, state, stream=None) -> None:
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    gb, w = _gbar_args(layout, gbar_shard, ws)
    _check(LIB.dp_step_reduce(gb, w, _ptr_array(grads), a, ctypes.byref(layout.c), adam_, loss_scale, sum_mode,
                              _ptr(state), _stream(stream)), "dp_step_reduce")


def dp_reduce_scatter_micro(acc_shard, gbar_shard, ws, g, k: int, a: int, layout: Layout, adam_: dp_adam_t,
                            loss_scale: float, sum_mode: int, state, stream=None) -> None:
    """Micro-step k of a: its n gradients (one per rank) reduce-scattered into the owner shard accumulators;
    the last micro-step writes gbar and publishes the skip decision."""
    _check_tensors(g, 2, [layout.psi] * len(g), "g")
    if a > 1:
        per = 2 if (sum_mode & 0xF) == DP_SUM_COMPENSATED else 1
        _check_tensors(acc_shard, 4, [per * L for L in layout.shard_lens()], "acc_shard")
    gb, w = _gbar_args(layout, gbar_shard, ws) if k == a - 1 else (None, None)
    _check(LIB.dp_reduce_scatter_micro(_ptr_array(acc_shard) if a > 1 else None, gb, w, _ptr_array(g), k, a,
                                       ctypes.byref(layout.c), adam_, loss_scale, sum_mode, _ptr(state),
                                       _stream(stream)), "dp_reduce_scatter_micro")


def dp_step_update(replicas, master, m, v, gbar_shard, ws, layout: Layout, adam_: dp_adam_t, state,
                   stream=None) -> None:
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    gb, w = _gbar_args(layout, gbar_shard, ws)
    _check(LIB.dp_step_update(_ptr_array(replicas), _ptr_array(master), _ptr_array(m), _ptr_array(v), gb, w,
                              ctypes.byref(layout.c), adam_, _ptr(state), _stream(stream)), "dp_step_update")


def dp_step_single_pass(replicas, master2, m2, v2, grads, a: int, layout: Layout, adam_: dp_adam_t,
                        loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED, state=None, stream=None) -> None:
    """One-pass step with double-buffered optimizer state: master2, m2, v2 are lists of 2n tensors (set 0, then
    set 1); the state's cur_set names the current set."""
    lens = layout.shard_lens() * 2
    for name, ts in (("master", master2), ("m", m2), ("v", v2)):
        if len(ts) != 2 * layout.n:
            raise ValueError("%s: need 2n = %d tensors" % (name, 2 * layout.n))
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    _check(LIB.dp_step_single_pass(_ptr_array(replicas), _ptr_array(master2), _ptr_array(m2), _ptr_array(v2),
                                   _ptr_array(grads), a, ctypes.byref(layout.c), adam_, loss_scale, sum_mode,
                                   _ptr(state), _stream(stream)), "dp_step_single_pass")


def dp_step_single_pass_from_host(replicas, master2, m2, v2, host_grads, grads, a: int, layout: Layout,
                                  adam_: dp_adam_t, loss_scale: float, sum_mode: int = DP_SUM_COMPENSATED,
                                  state=None, host_state=None, stream=None) -> None:
    """dp_step_single_pass with the gradients in host memory (see dp_step_from_host for host_grads and
    host_state)."""
    lens = layout.shard_lens() * 2
    for name, ts in (("master", master2), ("m", m2), ("v", v2)):
        if len(ts) != 2 * layout.n:
            raise ValueError("%s: need 2n = %d tensors" % (name, 2 * layout.n))
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    hp, hs = _host_args(layout, host_grads, grads, host_state)
    _check(LIB.dp_step_single_pass_from_host(_ptr_array(replicas), _ptr_array(master2), _ptr_array(m2),
                                             _ptr_array(v2), hp, _ptr_array(grads), a, ctypes.byref(layout.c), adam_,
                                             loss_scale, sum_mode, _ptr(state), hs, _stream(stream)),
           "dp_step_single_pass_from_host")


def dp_commit_step(state, adam_: dp_adam_t, scaler_: Optional[dp_scaler_t] = None, stream=None) -> None:
    """Commits a step reduced with DP_DEFER_COMMIT once found_inf holds every slice's decision."""
    _check(LIB.dp_commit_step(_ptr(state), adam_, ctypes.byref(scaler_) if scaler_ is not None else None,
                              _stream(stream)), "dp_commit_step")


def dp_commit_single_pass(replicas, master2, layout: Layout, adam_: dp_adam_t, state,
                          scaler_: Optional[dp_scaler_t] = None, stream=None) -> None:
    """dp_commit_step for a single pass run with DP_DEFER_COMMIT: flips the state set unless skipped, and
    repairs the replicas on a skipped step."""
    if len(master2) != 2 * layout.n:
        raise ValueError("master: need 2n = %d tensors" % (2 * layout.n))
    _check_tensors(master2, 4, layout.shard_lens() * 2, "master")
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check(LIB.dp_commit_single_pass(_ptr_array(replicas), _ptr_array(master2), ctypes.byref(layout.c), adam_,
                                     ctypes.byref(scaler_) if scaler_ is not None else None, _ptr(state),
                                     _stream(stream)), "dp_commit_single_pass")


STATIC_SCRATCH_BYTES = 64 * 1024 * 1024


def dp_step_static(replicas, master, m, v, grads, a: int, layout: Layout, adam_: dp_adam_t, loss_scale: float,
                   sum_mode: int = DP_SUM_COMPENSATED, state=None, stream=None) -> None:
    """dp_step with its gradient-shard scratch inside the library (for callers that cannot allocate device
    memory); the layout's workspace must fit STATIC_SCRATCH_BYTES."""
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    _check(LIB.dp_step_static(_ptr_array(replicas), _ptr_array(master), _ptr_array(m), _ptr_array(v),
                              _ptr_array(grads), a, ctypes.byref(layout.c), adam_, loss_scale, sum_mode,
                              _ptr(state), _stream(stream)), "dp_step_static")


def scaler(growth_factor: float = 2.0, backoff_factor: float = 0.5, growth_interval: int = 2000,
           min_scale: float = 2.0 ** 8, max_scale: float = 2.0 ** 24) -> dp_scaler_t:
    return dp_scaler_t(growth_factor, backoff_factor, growth_interval, min_scale, max_scale)


def dp_scaler_init(state, scale: float, stream=None) -> None:
    _check(LIB.dp_scaler_init(_ptr(state), scale, _stream(stream)), "dp_scaler_init")


def dp_step_scaled(replicas, master, m, v, grads, a: int, layout: Layout, adam_: dp_adam_t, scaler_: dp_scaler_t,
                   sum_mode: int = DP_SUM_COMPENSATED, gbar_shard=None, ws=None, state=None, stream=None) -> None:
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        _check_tensors(ts, 4, lens, name)
    _check_tensors(replicas, 2, [layout.psi] * layout.n, "replicas")
    _check_tensors(grads, 2, [layout.psi] * len(grads), "grads")
    gb, w = _gbar_args(layout, gbar_shard, ws)
    _check(LIB.dp_step_scaled(_ptr_array(replicas), _ptr_array(master), _ptr_array(m), _ptr_array(v),
                              _ptr_array(grads), a, ctypes.byref(layout.c), adam_, ctypes.byref(scaler_), sum_mode,
                              gb, w, _ptr(state), _stream(stream)), "dp_step_scaled")


def dp_read_status(state, stream=None) -> Tuple[int, int]:
    sk, er = c_i32(0), c_i32(0)
    _check(LIB.dp_read_status(_ptr(state), ctypes.byref(sk), ctypes.byref(er), _stream(stream)), "dp_read_status")
    return int(sk.value), int(er.value)


def dp_selftest_wait_timeout(state, timeout_ns: int, stream=None) -> None:
    _check(LIB.dp_selftest_wait_timeout(_ptr(state), timeout_ns, _stream(stream)), "dp_selftest_wait_timeout")


def dp_global_batch(b: int, n: int, a: int) -> int:
    return int(LIB.dp_global_batch(b, n, a))


def dp_memory_model(stage: int, psi: int, n: int) -> List[float]:
    out = (ctypes.c_double * 4)()
    _check(LIB.dp_memory_model(stage, psi, n, out), "dp_memory_model")
    return list(out)


def dp_traffic_model(stage: int, psi: int, n: int, wire_bytes_grad: int, wire_bytes_param: int) -> List[float]:
    out = (ctypes.c_double * 3)()
    _check(LIB.dp_traffic_model(stage, psi, n, wire_bytes_grad, wire_bytes_param, out), "dp_traffic_model")
    return list(out)


def dp_kernel_launches() -> int:
    return int(LIB.dp_kernel_launches())


def dp_set_wait_timeout_ns(ns: int) -> None:
    LIB.dp_set_wait_timeout_ns(ns)


def dp_get_wait_timeout_ns() -> int:
    return int(LIB.dp_get_wait_timeout_ns())


def new_state(device=None):
    """A 64-byte device state buffer, initialised (t = 0)."""
    import torch
    st = torch.zeros(STATE_BYTES, dtype=torch.uint8, device=device or "cuda")
    dp_state_init(st)
    return st


def read_state(state) -> dict:
    """Decodes a device state buffer (copies it to the host)."""
    raw = bytes(state.detach().cpu().numpy().tobytes())
    s = dp_step_state_t.from_buffer_copy(raw)
    return {"t": s.t, "found_inf": s.found_inf, "error": s.error, "nonfinite": s.nonfinite, "b1t": s.b1t,
            "b2t": s.b2t, "work_count": s.work_count, "work_found": s.work_found, "work_ticket": s.work_ticket,
            "good_steps": s.good_steps, "loss_scale": s.loss_scale, "cur_set": s.cur_set}


# ------------------------------------------------------------------------------------------- checkpoints

def _host_addr(x) -> Optional[int]:
    """Host address of a numpy array / CPU tensor / bytearray, or None if x is a CUDA tensor."""
    if x is None:
        return 0
    if hasattr(x, "is_cuda"):
        if x.is_cuda:
            return None
        if not x.is_contiguous():
            raise ValueError("checkpoint buffers must be contiguous")
        return x.data_ptr()
    if isinstance(x, bytearray):
        return ctypes.addressof(ctypes.c_char.from_buffer(x))
    if not x.flags["C_CONTIGUOUS"] or not x.flags["WRITEABLE"]:
        raise ValueError("checkpoint buffers must be contiguous and writable")
    return x.ctypes.data


def _ckpt_buffers(layout: Layout, master, m, v, state):
    """Pointer arrays and the host_buffers flag: every buffer on the host, or every buffer a CUDA tensor."""
    lens = layout.state_lens()
    for name, ts in (("master", master), ("m", m), ("v", v)):
        if len(ts) != layout.n:
            raise ValueError("%s: %d arrays for n = %d" % (name, len(ts), layout.n))
    items = list(master) + list(m) + list(v) + [state]
    host = [_host_addr(x) for x in items]
    if all(h is None for h in host):
        for name, ts in (("master", master), ("m", m), ("v", v)):
            _check_tensors(ts, 4, lens, name)
        return _ptr_array(master), _ptr_array(m), _ptr_array(v), _ptr(state), 0
    if any(h is None for h in host):
        raise ValueError("checkpoint buffers must be all on the host or all CUDA tensors")
    for name, ts in (("master", master), ("m", m), ("v", v)):
        for r, x in enumerate(ts):
            nbytes = x.numel() * x.element_size() if hasattr(x, "numel") else x.nbytes
            if nbytes < 4 * lens[r]:
                raise ValueError("%s[%d]: %d bytes, need %d" % (name, r, nbytes, 4 * lens[r]))
    k = layout.n
    mk = lambda hs: (c_vp * max(1, k))(*hs)
    return mk(host[:k]), mk(host[k:2 * k]), mk(host[2 * k:3 * k]), host[3 * k], 1


def dp_checkpoint_save(root: str, tag: str, layout: Layout, master, m, v, state, user_meta: bytes = b"",
                       stream=None) -> None:
    """Saves master/m/v (CUDA tensors, or host arrays: numpy / CPU tensors) and the state by shard."""
    pm, pmm, pv, ps, host = _ckpt_buffers(layout, master, m, v, state)
    meta = bytes(user_meta)
    buf = ctypes.create_string_buffer(meta, max(1, len(meta)))
    _check(LIB.dp_checkpoint_save(os.fsencode(root), tag.encode(), ctypes.byref(layout.c), pm, pmm, pv, ps,
                                  buf if meta else None, len(meta), host, 0 if host else _stream(stream)),
           "dp_checkpoint_save")


def dp_checkpoint_load(root: str, tag: Optional[str], layout: Layout, master, m, v, state, verify: bool = True,
                       stream=None) -> bytes:
    """Loads checkpoint `tag` (None: LATEST) into `layout`, resharding; returns the saved user bytes."""
    pm, pmm, pv, ps, host = _ckpt_buffers(layout, master, m, v, state)
    tb = tag.encode() if tag is not None else None
    size = c_u64(0)
    _check(LIB.dp_checkpoint_info(os.fsencode(root), tb, 0, None, None, None, None, None, 0, ctypes.byref(size)),
           "dp_checkpoint_load")
    buf = ctypes.create_string_buffer(max(1, size.value))
    cap = c_u64(size.value)
    _check(LIB.dp_checkpoint_load(os.fsencode(root), tb, ctypes.byref(layout.c), pm, pmm, pv, ps, buf,
                                  ctypes.byref(cap), host, int(verify), 0 if host else _stream(stream)),
           "dp_checkpoint_load")
    return buf.raw[:cap.value]


def dp_checkpoint_info(root: str, tag: Optional[str] = None, verify: bool = False) -> Layout:
    """The layout checkpoint `tag` (None: LATEST) was saved with."""
    tb = tag.encode() if tag is not None else None
    stage, n, nseg, psi = c_i32(0), c_i32(0), c_i32(0), c_i64(0)
    _check(LIB.dp_checkpoint_info(os.fsencode(root), tb, int(verify), ctypes.byref(stage), ctypes.byref(n),
                                  ctypes.byref(psi), ctypes.byref(nseg), None, 0, None), "dp_checkpoint_info")
    arr = (dp_segment_t * max(1, nseg.value))()
    _check(LIB.dp_checkpoint_info(os.fsencode(root), tb, 0, None, None, None, None, arr, nseg.value, None),
           "dp_checkpoint_info")
    return Layout(stage.value, n.value, psi.value,
                  [(arr[k].global_off, arr[k].len, arr[k].owner, arr[k].local_off) for k in range(nseg.value)])
