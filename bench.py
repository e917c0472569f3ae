"""Benchmark of the fused data-parallel step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--workload NAME]

One step = the whole hot path over one batch of synthetic inputs: n*a bf16 micro-step gradients accumulated,
reduced in ring order, averaged, unscaled and finite-checked, partitioned Adam on the fp32 shards, and the bf16
all-gather into the n replicas.  By default the step is dp_step_single_pass (one reduce-and-update pass over
double-buffered optimizer state, the fastest path); --path two-pass times dp_step's two kernels
(dp_step_reduce + dp_step_update), --path microstep the per-micro-step reduce-scatter + dp_step_update.  The
default workload is the GPT-2-small parameter list (123,568,896 params), n=8, a=4, ZeRO-1 even shards, loss scale
2^16.  hbm_gbs counts the single-pass algorithmic minimum B1 = 2na + 24 + 2n bytes per parameter for every
path; hbm_gbs_path_bytes counts the bytes the timed path's own design moves (B1 + 8 for the two-pass step).

The end-to-end leg ("e2e") times the same step through one C-ABI call with the gradients in host memory
(dp_step_single_pass_from_host, or dp_step_from_host for --path two-pass): every step's gradients copied from
pinned host memory, the step, and the 64-byte step state read back.  --order tree times the binomial-tree order
(dp_step by default, --path single-pass for its single pass); --workload also takes the flat sweep's case names
(sweep_<psi>_n<n>_a<a>_<even|ragged>).

Multi-GPU (torchrun): every rank holds one workload-sized slice of an N-times-larger parameter space (weak
scaling) and runs the sliced step: its reduction with the commit deferred, one 4-byte NCCL all-reduce (MAX) of
the skip flag, then the commit and the update -- the one collective of a step split across GPUs.  Barrier and
max-over-ranks timing.

Rank 0 prints one JSON line.  --impl reference times the float64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused DP grad-reduce+Adam step: Gparams/s and achieved HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", default="gpt2_small")
    p.add_argument("--sum", choices=["compensated", "plain"], default="compensated")
    p.add_argument("--e2e-steps", type=int, default=0, help="steps of the end-to-end leg (0: same as --steps, max 20)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample", type=int, default=1 << 21, help="elements of the oracle's CPU sample")
    p.add_argument("--psi", type=int, default=0, help="override the parameter count (small profiling cases)")
    p.add_argument("--checkpoint", default="",
                   help="time sharded checkpoint save / reshard-load of the workload's optimizer state under this "
                        "directory instead of the step (prints its own JSON line)")
    p.add_argument("--order", choices=["ring", "tree"], default="ring",
                   help="order of the ranks' sums: the ring reduce-scatter's, or a binomial tree's")
    p.add_argument("--path", choices=["two-pass", "single-pass", "microstep"], default=None,
                   help="dp_step_single_pass (one pass, two state sets; the default), dp_step (reduce + update "
                        "kernels; the default with --order tree) or dp_reduce_scatter_micro per micro-step + "
                        "dp_step_update (the ZeRO-2 form)")
    p.add_argument("--stage", type=int, default=-1, choices=[-1, 0, 1, 2, 3],
                   help="override the workload's ZeRO stage (0: plain data parallelism, two-pass path)")
    args = p.parse_args()
    if args.path is None:
        # the tree order's two-pass step outruns its single pass on the GPT-2 list (57.7 against 47 Gparams/s)
        args.path = "two-pass" if args.stage == 0 or args.order == "tree" else "single-pass"
    return args


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (one all-reduce of 8 bytes); x itself when not distributed."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(psi: int, world_size: int, ms_per_step: float) -> float:
    """Whole-job Gparams/s: every rank processes its own replica of psi parameters per step (weak scaling)."""
    return psi * world_size / (ms_per_step * 1e-3) / 1e9


def barrier() -> None:
    import torch.distributed as tdist
    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        tdist.barrier()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(wl):
    """Algorithmic bytes per parameter: single-pass minimum B1 = 2na + 24 + 2n; the two-pass design adds the
    fp32 gbar shard written by the reduce kernel and read back by the update kernel (B2 = B1 + 8).  Plain data
    parallelism (stage 0) keeps n full copies of master/m/v, so its update reads gbar once and reads and writes
    every rank's state: B1 = 2na + 26n."""
    if wl.stage == 0:
        b1 = 2 * wl.n * wl.a + 26 * wl.n
        return b1, b1 + 8, 2 * wl.n * wl.a + 4, 4 + 26 * wl.n
    b1 = 2 * wl.n * wl.a + 24 + 2 * wl.n
    return b1, b1 + 8, 2 * wl.n * wl.a + 4, 4 + 24 + 2 * wl.n


KERNEL_SOURCES = {"reduce": ("dp_kernels.cu", "dp_single.cuh", "dp_device.cuh", "dp_launch.h"),
                  "update": ("dp_kernels.cu", "dp_single.cuh", "dp_device.cuh", "dp_launch.h"),
                  "single_pass": ("dp_kernels.cu", "dp_single.cuh", "dp_device.cuh", "dp_launch.h"),
                  "single_pass_tree": ("dp_tree_sp.cu", "dp_single.cuh", "dp_device.cuh", "dp_launch.h"),
                  "reduce_tree": ("dp_tree.cu", "dp_device.cuh", "dp_launch.h"),
                  "rs_micro": ("dp_micro.cu", "dp_device.cuh", "dp_launch.h")}


def micro_bytes(wl, comp: bool) -> int:
    """Algorithmic bytes per parameter of the a per-micro-step launches: every gradient read once (2na), the
    shard accumulator written at k = 0, read and written in between, read at k = a-1 (8 B an access
    compensated, 4 plain), and gbar written once (4)."""
    acc = 8 if comp else 4
    if wl.a == 1:
        return 2 * wl.n + 4
    return 2 * wl.n * wl.a + acc + 2 * acc * (wl.a - 2) + acc + 4


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and blank space, so that a comment edit does not mark a kernel as
    changed."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel="reduce"):
    """sha256 prefix of the code (comments and spacing removed) of the files that make up a kernel."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "zero_gradient_sync_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
        e = j[workload][kernel]
        if e.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if self.t0 is not None and self.t0 - 0.06 <= ts <= (self.t1 or ts) + 0.06]
        use = inside if inside else rows
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        smax = [num(p[2]) for p in use if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in use:
            for nm, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_region": len(inside)}


# ----------------------------------------------------------------------------------------------- oracle leg

def oracle_sample(wl, host_grads, master_full, sample):
    """A bounded sample of the workload for the CPU oracle: its first `sample` parameters with the same n, a,
    stage and an even layout over the sample."""
    import numpy as np
    import synth
    ps = min(sample, wl.psi)
    segs = synth.layout_even(ps, wl.n)
    grads = [np.ascontiguousarray(g[:ps]) for g in host_grads]
    lens = [ps] * wl.n if wl.stage == 0 else synth.shard_lengths(segs, wl.n)
    master = [np.zeros(L, np.float32) for L in lens]
    for g, ln, o, lo in segs:
        master[o][lo:lo + ln] = master_full[g:g + ln]
    m = [np.zeros(L, np.float32) for L in lens]
    v = [np.zeros(L, np.float32) for L in lens]
    reps = [np.zeros(ps, np.uint16) for _ in range(wl.n)]
    return ps, segs, grads, master, m, v, reps


def run_oracle_steps(wl, sample_data, steps, threads):
    import oracle
    ps, segs, grads, master, m, v, reps = sample_data
    t = 0
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        res = oracle.step(ps, wl.n, wl.a, wl.stage, segs, grads, master, m, v, reps, wl.lr, wl.beta1, wl.beta2,
                          wl.eps, wl.loss_scale, t, threads=threads)
        times.append(time.perf_counter() - t0)
        t = res["t"]
    return times


def host_inputs_small(wl, ps):
    import numpy as np
    import synth
    grads = [synth.grads_bf16(wl, r, k, 0, ps) for r in range(wl.n) for k in range(wl.a)]
    return grads, synth.master_f32(wl, 0, ps)


def reference_main(args, wl):
    ws, rank, local = dist_env()
    if ws > 1 and rank != 0:
        return 0
    threads = os.cpu_count() or 1
    ps = min(args.cpu_sample, wl.psi)
    grads, mfull = host_inputs_small(wl, ps)
    data = oracle_sample(wl, grads, mfull, ps)
    run_oracle_steps(wl, data, max(0, args.warmup), threads)
    times = run_oracle_steps(wl, data, args.steps, threads)
    tot = sum(times)
    per = tot / max(1, len(times))
    val = ps / per / 1e9
    sample = "first %d of %d parameters of the workload per step (even layout over the sample), n=%d, a=%d" % (
        ps, wl.psi, wl.n, wl.a)
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": "Gparams/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config_of(wl, args),
           "cpu_baseline": {"value": val, "unit": "Gparams/s", "cores": threads, "kind": "oracle", "sample": sample},
           "e2e": {"value": val, "unit": "Gparams/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def config_of(wl, args):
    b1, b2, _, _ = step_bytes(wl)
    return {"workload": wl.description, "psi": wl.psi, "n": wl.n, "a": wl.a, "zero_stage": wl.stage,
            "layout": wl.layout, "loss_scale": wl.loss_scale, "sum_mode": args.sum, "order": args.order,
            "path": args.path,
            "grad_dtype": "bf16",
            "state_dtype": "fp32", "bytes_per_param_single_pass": b1, "bytes_per_param_two_pass": b2,
            "l2": "inputs larger than L2: %.1f GB streamed per step vs 129 MB L2, no flush" % (
                (b1 if args.path == "single-pass" else b2) * wl.psi / 1e9)}


# ----------------------------------------------------------------------------------------------- native leg

def native_main(args, wl):
    import numpy as np
    import torch

    import synth
    import zero_gradient_sync_gb300 as dp
    from synth import device as sd
    from zero_gradient_sync_gb300 import sliced
    from zero_gradient_sync_gb300.buffers import StepBuffers

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    # N > 1: this rank's workload is its slice of an N-times-larger space; the slices share one skip decision.
    split = ws > 1

    def combine_max(flag):
        import torch.distributed as tdist
        tdist.all_reduce(flag, op=tdist.ReduceOp.MAX)

    dev = torch.device("cuda", torch.cuda.current_device())
    mode = dp.DP_SUM_COMPENSATED if args.sum == "compensated" else dp.DP_SUM_PLAIN
    tree = args.order == "tree"
    if tree:
        mode |= dp.DP_ORDER_TREE
    segs = synth.layout_of(wl)
    layout = dp.Layout(wl.stage, wl.n, wl.psi, segs)
    single = args.path == "single-pass"
    micro = args.path == "microstep"
    if micro and tree:
        raise SystemExit("--path microstep runs in ring order only")
    if micro and split:
        raise SystemExit("--path microstep runs on one GPU")
    if single and wl.stage == 0:
        raise SystemExit("the single pass takes ZeRO stages 1-3; use --path two-pass for stage 0")
    bufs = StepBuffers(layout, wl.a, dev, second_set=single, micro_acc=micro)
    A = dp.adam(wl.lr, wl.beta1, wl.beta2, wl.eps)

    # Inputs: generated on the host into pinned buffers (kept for the end-to-end leg), then copied to HBM.
    t_gen = time.time()
    host_grads = []
    for r in range(wl.n):
        for k in range(wl.a):
            h = torch.empty(wl.psi, dtype=torch.int16, pin_memory=True)
            synth.grads_bf16(wl, r, k, 0, wl.psi, out=h.numpy().view(np.uint16))
            host_grads.append(h)
            bufs.grad(r, k).view(torch.int16).copy_(h)
    sd.fill_master(bufs.master, wl, segs, wl.stage)
    if single:
        for x, y in zip(bufs.master1, bufs.master):
            x.copy_(y)
    torch.cuda.synchronize()
    t_gen = time.time() - t_gen

    stream = torch.cuda.current_stream()

    flag_ops = sliced.LibraryOps()

    def first_half():
        """The timed kernel of the roofline: the single pass, the a per-micro-step launches, or pass A."""
        if split:
            sliced.reduce_deferred(bufs, A, wl.loss_scale, mode, single_pass=single)
        elif single:
            bufs.step_single_pass(A, wl.loss_scale, mode)
        elif micro:
            for kk in range(wl.a):
                bufs.reduce_micro(kk, A, wl.loss_scale, mode)
        else:
            bufs.reduce(A, wl.loss_scale, mode)

    def second_half():
        if split:
            combine_max(flag_ops.found_flag(bufs))
            sliced.commit_and_update(bufs, A, single_pass=single)
        elif not single:
            bufs.update(A)

    def one_step():
        first_half()
        second_half()

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    end = torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(("GPU-" + str(uuid)) if uuid is not None else str(torch.cuda.current_device()))
    clocks.start()
    time.sleep(0.15)
    barrier()
    torch.cuda.synchronize()
    l0 = dp.dp_kernel_launches()
    clocks.mark(0)
    for k in range(K):
        ev[k][0].record(stream)
        first_half()
        ev[k][1].record(stream)
        second_half()
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(1)
    barrier()
    launches = dp.dp_kernel_launches() - l0
    total_ms = ev[0][0].elapsed_time(end)
    red_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    upd_ms = [ev[k][1].elapsed_time(ev[k + 1][0] if k + 1 < K else end) for k in range(K)]
    step_ms = sorted(ev[k][0].elapsed_time(ev[k + 1][0] if k + 1 < K else end) for k in range(K))
    clk = clocks.stop()
    skipped, err = bufs.status()
    total_ms = max_over_ranks(total_ms, dev)
    ms = total_ms / K
    psi_all = wl.psi * ws
    value = job_throughput(wl.psi, ws, ms)

    b1, b2, red_bytes, upd_bytes = step_bytes(wl)
    if single:
        red_bytes, upd_bytes = b1, 0     # one kernel streams the single-pass minimum; the repair kernel is idle
    if micro:
        red_bytes = micro_bytes(wl, args.sum == "compensated")
    peak, peak_kind = measured_peak()
    red_avg = sum(red_ms) / K
    upd_avg = sum(upd_ms) / K
    red_ach = red_bytes * wl.psi / (red_avg * 1e-3) / 1e9
    upd_ach = upd_bytes * wl.psi / max(1e-9, upd_avg * 1e-3) / 1e9
    path_bytes = b1 if single else (red_bytes + upd_bytes) if micro else b2
    step_gbs = b1 * wl.psi / (ms * 1e-3) / 1e9           # the single-pass algorithmic minimum, every path
    path_gbs = path_bytes * wl.psi / (ms * 1e-3) / 1e9    # what the timed path's own design moves
    traffic = recorded_traffic(wl.name, ("single_pass_tree" if tree else "single_pass") if single else
                               "rs_micro" if micro else ("reduce_tree" if tree else "reduce"))

    # End to end through the public call with host buffers: the step's gradients copied from pinned host
    # memory, the step, and the step's status read back, every step -- one C-ABI call does all three
    # (dp_step_single_pass_from_host, or dp_step_from_host for the two-pass step).
    e2e = None
    if not args.no_e2e:
        KE = args.e2e_steps or min(K, 20)
        host_state = torch.empty(dp.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)

        def e2e_step():
            if split:
                for q, h in enumerate(host_grads):
                    bufs.grads[q].view(torch.int16).copy_(h, non_blocking=True)
                one_step()
                host_state.copy_(bufs.state, non_blocking=True)
            elif single:
                bufs.step_single_pass_from_host(host_grads, A, wl.loss_scale, mode, host_state=host_state)
            elif micro:
                for q, h in enumerate(host_grads):
                    bufs.grads[q].view(torch.int16).copy_(h, non_blocking=True)
                bufs.step_micro(A, wl.loss_scale, mode)
                host_state.copy_(bufs.state, non_blocking=True)
            else:
                bufs.step_from_host(host_grads, A, wl.loss_scale, mode, host_state=host_state)

        # Untimed warm-up of this leg too: the first host-to-device copy from freshly pinned pages has measured
        # ~250 ms on its own for the 7.9 GB of the GPT-2 workload (a one-time mapping cost), against 37.5 ms after.
        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        barrier()
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(KE):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e_ms = max_over_ranks(s0.elapsed_time(s1) / KE, dev)
        e2e = {"value": job_throughput(wl.psi, ws, e_ms), "unit": "Gparams/s",
               "h2d_bytes_per_step": 2 * wl.n * wl.a * wl.psi, "d2h_bytes_per_step": dp.STATE_BYTES,
               "ms_per_step": e_ms, "steps": KE}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        ps = min(args.cpu_sample, wl.psi)
        host_np = [h[:ps].numpy().view(np.uint16) for h in host_grads]
        data = oracle_sample(wl, host_np, synth.master_f32(wl, 0, ps), ps)
        run_oracle_steps(wl, data, 1, threads)
        reps = 1
        t_one = sum(run_oracle_steps(wl, data, 1, threads))
        # about 10-30 s of CPU work (thread-seconds), at most ~12 s of wall time
        target = max(1, min(int(15.0 / max(1e-6, t_one * threads)), int(12.0 / max(1e-6, t_one))))
        times = run_oracle_steps(wl, data, target, threads)
        per = sum(times) / len(times)
        # one step of the same sample on a single thread, for the per-core rate
        one = run_oracle_steps(wl, data, 1, 1)[0]
        cpu = {"value": ps / per / 1e9, "unit": "Gparams/s", "cores": threads, "kind": "oracle",
               "value_1_thread": ps / one / 1e9,
               "sample": "first %d of %d parameters (even layout over the sample), n=%d, a=%d; %d timed steps, "
                         "%.1f s wall on %d threads; one step on 1 thread"
                         % (ps, wl.psi, wl.n, wl.a, len(times), sum(times), threads)}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "Gparams/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms, "ms_per_step_median": statistics.median(step_ms), "ms_per_step_min": step_ms[0],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Philox4x64 N(0, sigma) bf16 gradients, fp32 master; no dataset)",
            "config": config_of(wl, args),
            "hbm_gbs": step_gbs, "hbm_frac_of_peak": step_gbs / peak, "hbm_frac_of_nominal_7900": step_gbs / 7900.0,
            "hbm_bytes_per_param": b1, "hbm_gbs_path_bytes": path_gbs, "path_bytes_per_param": path_bytes,
            "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
            "split": ({"slices": ws, "collective": "4-byte NCCL all-reduce (MAX) of found_inf per step"}
                      if split else None),
            "roofline": {"bound": "hbm",
                         "kernel": ("single-pass reduce (tree order) + Adam + all-gather" if single and tree else
                                    "single-pass reduce + Adam + all-gather" if single else
                                    "per-micro-step reduce-scatter (a launches per step, summed)" if micro else
                                    "reduce (accumulate + tree reduce + average + check)" if tree else
                                    "reduce (accumulate + ring reduce-scatter + average + check)"),
                         "achieved": red_ach, "peak": peak, "unit": "GB/s", "frac": red_ach / peak,
                         "traffic": traffic, "bytes_per_launch": red_bytes * wl.psi, "avg_ms": red_avg,
                         "peak_kind": peak_kind},
            "kernels": ({"single_pass": {"avg_ms": red_avg, "gbs": red_ach, "bytes_per_param": red_bytes,
                                         "note": "events bracket the fused kernel and the repair launch, which "
                                                 "returns at once on an applied step"},
                         "after": {"avg_ms": upd_avg}} if single else
                        {("rs_micro" if micro else "reduce"): {"avg_ms": red_avg, "gbs": red_ach,
                                                                "bytes_per_param": red_bytes},
                         "update": {"avg_ms": upd_avg, "gbs": upd_ach, "bytes_per_param": upd_bytes}}),
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "status": {"skipped_last_step": skipped, "error": err}, "setup_s": t_gen,
        }
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()
    return 0


def checkpoint_main(args, wl):
    """Sharded checkpoint of the workload's fp32 master/m/v (12 bytes a parameter): --steps saves, each
    followed by a load into a layout of n/2 ranks (a reshard), wall-clock timed (the calls are host-synchronous).
    Bounds measured on the same box: the pinned device-to-host / host-to-device copy rate and the file system's
    multi-threaded write / read rate for the same bytes."""
    import shutil
    from concurrent.futures import ThreadPoolExecutor

    import torch

    import synth
    import zero_gradient_sync_gb300 as dp

    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    lay = dp.Layout(wl.stage, wl.n, wl.psi, synth.layout_of(wl))
    n2 = max(1, wl.n // 2)
    lay2 = dp.Layout.even(wl.psi, n2, stage=max(1, wl.stage))
    g = torch.Generator(device=dev).manual_seed(11)
    src = [[torch.randn(L, device=dev, generator=g) for L in lay.state_lens()] for _ in range(3)]
    dst = [[torch.empty(L, device=dev) for L in lay2.state_lens()] for _ in range(3)]
    state = dp.new_state(dev)
    nbytes = 12 * wl.psi
    root = os.path.abspath(args.checkpoint)
    os.makedirs(root, exist_ok=True)

    def fresh(tag):
        d = os.path.join(root, tag)
        if os.path.isdir(d):
            shutil.rmtree(d)

    saves, loads = [], []
    for k in range(args.warmup + args.steps):
        tag = "bench%d" % (k % 2)
        fresh(tag)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dp.dp_checkpoint_save(root, tag, lay, *src, state)
        t1 = time.perf_counter()
        dp.dp_checkpoint_load(root, tag, lay2, *dst, state, verify=False)
        t2 = time.perf_counter()
        if k >= args.warmup:
            saves.append(t1 - t0)
            loads.append(t2 - t1)
    t0 = time.perf_counter()
    dp.dp_checkpoint_load(root, None, lay2, *dst, state, verify=True)
    t_verify = time.perf_counter() - t0
    ok = all(torch.equal(torch.cat(a).view(torch.int32), torch.cat(b).view(torch.int32)) for a, b in zip(src, dst))

    # bounds: pinned host<->device copies, and plain multi-threaded file writes / reads of the same bytes
    chunk = 1 << 24
    pin = torch.empty(nbytes // 4, dtype=torch.float32, pin_memory=True)
    flat = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pin.copy_(flat, non_blocking=True)
    torch.cuda.synchronize()
    d2h = nbytes / (time.perf_counter() - t0) / 1e9
    t0 = time.perf_counter()
    flat.copy_(pin, non_blocking=True)
    torch.cuda.synchronize()
    h2d = nbytes / (time.perf_counter() - t0) / 1e9
    view = memoryview(pin.numpy()).cast("B")
    workers = min(8, os.cpu_count() or 1)
    part = -(-nbytes // workers)
    rawdir = os.path.join(root, "raw")
    os.makedirs(rawdir, exist_ok=True)

    def write_part(i):
        path = os.path.join(rawdir, "p%d" % i)
        fd = os.open(path, os.O_WRONLY | os.O_CREAT | os.O_TRUNC, 0o644)
        try:
            lo, hi = i * part, min(nbytes, (i + 1) * part)
            for o in range(lo, hi, chunk):
                os.write(fd, view[o:min(hi, o + chunk)])
            os.fsync(fd)
        finally:
            os.close(fd)

    def read_part(i):
        path = os.path.join(rawdir, "p%d" % i)
        with open(path, "rb", buffering=0) as f:
            while f.read(chunk):
                pass

    with ThreadPoolExecutor(workers) as ex:
        t0 = time.perf_counter()
        list(ex.map(write_part, range(workers)))
        fs_w = nbytes / (time.perf_counter() - t0) / 1e9
        t0 = time.perf_counter()
        list(ex.map(read_part, range(workers)))
        fs_r = nbytes / (time.perf_counter() - t0) / 1e9
    shutil.rmtree(rawdir)
    for tag in ("bench0", "bench1"):
        fresh(tag)

    save_s, load_s = statistics.median(saves), statistics.median(loads)
    out = {
        "metric": "sharded checkpoint of fp32 master/m/v: save and reshard-load GB/s",
        "value": round(nbytes / save_s / 1e9, 3), "unit": "GB/s (save)", "higher_is_better": True,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * save_s, 2),
        "load_gbs": round(nbytes / load_s / 1e9, 3), "load_verified_gbs": round(nbytes / t_verify / 1e9, 3),
        "bytes": nbytes, "bit_exact": ok,
        "bounds": {"d2h_gbs": round(d2h, 2), "h2d_gbs": round(h2d, 2), "fs_write_fsync_gbs": round(fs_w, 3),
                   "fs_read_gbs": round(fs_r, 3), "threads": workers},
        "config": {"workload": wl.name, "psi": wl.psi, "n": wl.n, "stage": wl.stage, "layout": wl.layout,
                   "reshard_to_n": n2, "dir_fs": _fs_type(root)},
        "data": "synthetic", "dtype": "f32",
    }
    print(json.dumps(out), flush=True)
    return 0


def _fs_type(path: str) -> str:
    try:
        best, kind = "", "unknown"
        with open("/proc/mounts") as f:
            for line in f:
                parts = line.split()
                if len(parts) > 2 and path.startswith(parts[1]) and len(parts[1]) > len(best):
                    best, kind = parts[1], parts[2]
        return kind
    except OSError:
        return "unknown"


def main():
    args = parse()
    import synth
    known = dict(synth.WORKLOADS)
    known.update({w.name: w for w in synth.sweep_cases()})   # the flat sweep's cases, e.g. sweep_1000000000_n8_a8_even
    if args.workload not in known:
        raise SystemExit("unknown workload %s (have %s, and the sweep_* cases)" %
                         (args.workload, ", ".join(synth.WORKLOADS)))
    wl = known[args.workload]
    if args.psi > 0:
        wl = wl.with_(psi=args.psi, description=wl.description + " [psi overridden to %d]" % args.psi)
    if args.stage >= 0 and args.stage != wl.stage:
        wl = wl.with_(stage=args.stage, description=wl.description + " [ZeRO stage overridden to %d]" % args.stage)
    if args.impl == "reference":
        return reference_main(args, wl)
    if args.checkpoint:
        return checkpoint_main(args, wl)
    return native_main(args, wl)


if __name__ == "__main__":
    sys.exit(main())
