"""Benchmark of sparse embedding weight-gradient accumulation on one GB300 per rank.

Workload: large vocabulary, V = 129280, H = 7168, 8192 Zipf(1.1) token ids, bf16 grad,
fp32 main_grad (seeded synthetic inputs, see workloads.py).  A step is one call of the
whole path (plan: validate + sort + run listing; apply: partial sums + combine + add).

Prints one JSON line:
  value       mean device microseconds per accumulate_embedding_wgrad call, inputs
              resident in HBM, L2 flushed (a 256 MiB memset) before every call;
  e2e         the host-input call (ewg_accumulate_host: ids and grad in pinned host memory,
              copied in by the library) and the device status word read back, all
              inside the timing;
  roofline    the apply kernel: algorithmic bytes (grad rows read + touched main_grad
              rows read and written) per launch / its CUDA-event duration, against the
              measured HBM copy bandwidth;
  cpu_baseline  the CPU oracle on the same workload, on this host's cores.
With --impl reference the CPU oracle is the timed arm.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "wgrad-accumulate µs/call & HBM GB/s vs ~8 TB/s at 129280x7168, 8192 tokens"
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="large_vocab")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU work budget of the oracle baseline")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the CPU baseline, the dense comparison and the clock sampler")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world, device):
    """Element-wise maximum of `values` over the ranks (one all_reduce; the identity on
    one rank).  Every rank runs its own replica, so the job takes as long as its slowest
    rank."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def host_inputs(w):
    """Seeded inputs: ids on the host; grad drawn on the host too (it is a per-step input)."""
    ids = workloads.make_ids(w).reshape(-1)
    grad = workloads.make_grad(w).reshape(ids.size, w.hidden)
    return ids, grad


def algorithmic_bytes(w, ids):
    n, H = ids.size, w.hidden
    U = int(np.unique(ids).size)
    gs = torch.finfo(w.grad_dtype).bits // 8
    ms = torch.finfo(w.mg_dtype).bits // 8
    apply_bytes = n * H * gs + 2 * U * H * ms
    return U, apply_bytes, apply_bytes + n * ids.itemsize


# --- clocks during the timed region ----------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines or len(self.marks) < 2:
            return None
        t0, t1 = self.marks[0], self.marks[-1]
        rows = [l for (t, l) in self.lines if t0 - 0.06 <= t <= t1 + 0.06] or \
            [l for (_, l) in self.lines]
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# --- our arm ---------------------------------------------------------------------------

def traffic_from_profile(kernel_src_hash: str, workload: str):
    """DRAM bytes per apply launch from the committed ncu summary, if it was taken on
    the current kernel source and the same workload; None otherwise."""
    if workload != "large_vocab":
        return None
    path = os.path.join(ROOT, "profiles", "apply_kernel_large_vocab.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256") != kernel_src_hash:
        return None
    return d.get("dram_bytes_per_launch")


# the files the apply kernel is compiled from
APPLY_SOURCES = ("embedding_weight_grad_gb300/csrc/ewg_apply.cu",
                 "embedding_weight_grad_gb300/csrc/ewg_internal.cuh",
                 "embedding_weight_grad_gb300/csrc/ewg_ptx.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    for f in APPLY_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def kernel_launches_per_call(n, V):
    """Kernels one accumulate call launches: the plan (one hashed kernel up to 8192
    tokens; otherwise pack, a digit histogram, one sweep per radix pass of at most 9 id
    bits, and the listing) and the apply kernel."""
    if n <= 8192:
        return 1 + 1
    id_bits = max(0, int(V - 1).bit_length())
    passes = -(-id_bits // 9)
    return 1 + (1 if passes else 0) + passes + 1 + 1


def time_events(fn, steps, stream, flush):
    """Runs fn() `steps` times with an L2 flush before each; returns per-call ms lists
    from CUDA events recorded on `stream` around each call."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s, e in evs:
        flush()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def run_ours(args, w, world, rank, local):
    import embedding_weight_grad_gb300 as ewg
    from embedding_weight_grad_gb300 import build as cuda_build

    cuda_build.build()
    ewg.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    ids_h, grad_h = host_inputs(w)
    n, H, V = ids_h.size, w.hidden, w.num_embeddings
    U, apply_bytes, call_bytes = algorithmic_bytes(w, ids_h)
    ids_d = torch.from_numpy(ids_h).to(dev)
    grad_d = grad_h.to(dev)
    mg = workloads.make_main_grad(w, dev)
    ws = ewg.new_workspace(n, H, dev)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    read_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_clean():   # the memset, then a read that leaves L2 holding clean lines
        flush_buf.fill_(1)
        read_buf.sum()

    def call():
        ewg.accumulate_embedding_wgrad(ids_d, grad_d, mg, workspace=ws)

    def call_plan():
        ewg.plan(ids_d, V, H, ws)

    def call_apply():
        ewg.apply(grad_d, mg, n, ws)

    for _ in range(args.warmup):
        flush()
        call()
    ewg.raise_on_device_status(ws)

    sampler = ClockSampler(local)
    if not args.no_extras:
        sampler.start()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark()
    t_wall = time.perf_counter()
    per_call = time_events(call, args.steps, stream, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    region_s = time.perf_counter() - t_wall

    # the same call after a flush that leaves L2 clean: the memset's dirty lines are not
    # written back inside the timed call
    per_call_clean = time_events(call, args.steps, stream, flush_clean)

    # calls enqueued back to back (no flush, no host synchronisation in between): the GPU
    # never idles, and each call finds L2 as the previous call left it
    per_call_b2b = time_events(call, args.steps, stream, lambda: None)

    # calls made after the GPU has sat idle: the host synchronises and waits 1 ms before
    # each call.  An idle GB300 runs the next few tens of microseconds slower (a GPU-side
    # sleep kernel of 50 us or more before the call, which touches no memory, removes the
    # difference), so this is a property of the idle GPU, not of the call.
    def idle():
        torch.cuda.synchronize()
        time.sleep(1e-3)

    idle_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(max(10, args.steps // 10))]
    for s_ev, e_ev in idle_evs:
        idle()
        s_ev.record(stream)
        call()
        e_ev.record(stream)
    torch.cuda.synchronize()
    per_call_idle = [s_ev.elapsed_time(e_ev) for s_ev, e_ev in idle_evs]

    # the same call split into its two C-ABI halves, to time the apply kernel alone
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for e0, e1, e2 in ev:
        flush()
        e0.record(stream)
        call_plan()
        e1.record(stream)
        call_apply()
        e2.record(stream)
    torch.cuda.synchronize()
    plan_ms = [a.elapsed_time(b) for a, b, _ in ev]
    apply_ms = [b.elapsed_time(c) for _, b, c in ev]

    # end to end: the host-input call (ids and grad in pinned host memory, copied in by the
    # library, the grad copy overlapping the plan), status read back, every step
    ids_pin = torch.from_numpy(ids_h).pin_memory()
    grad_pin = grad_h.pin_memory()
    status_pin = torch.empty(1, dtype=torch.int32).pin_memory()
    ws_host = ewg.new_host_workspace(n, H, ids_pin.dtype, grad_pin.dtype, dev)
    status_word = ws_host[:4].view(torch.int32)

    def e2e_call():
        ewg.accumulate_embedding_wgrad_from_host(ids_pin, grad_pin, mg, workspace=ws_host)
        status_pin.copy_(status_word, non_blocking=True)

    for _ in range(3):
        flush()
        e2e_call()
    e2e_ms = time_events(e2e_call, max(10, args.steps // 10), stream, flush)
    assert int(status_pin.item()) == 0
    sampler.mark()
    sampler.stop()

    mean_ms, median_ms, plan_mean, apply_mean, e2e_mean, clean_ms, b2b_ms, idle_ms = reduce_max(
        [statistics.fmean(per_call), statistics.median(per_call), statistics.fmean(plan_ms),
         statistics.fmean(apply_ms), statistics.fmean(e2e_ms), statistics.fmean(per_call_clean),
         statistics.fmean(per_call_b2b), statistics.fmean(per_call_idle)],
        world, dev)

    out = None
    if rank == 0:
        hbm_peak, peak_kind = peaks()
        achieved = apply_bytes / (apply_mean * 1e-3) / 1e9
        traffic = traffic_from_profile(kernel_source_hash(), w.name)
        launches_per_call = kernel_launches_per_call(n, V)
        us = mean_ms * 1e3
        out = {
            "metric": METRIC,
            "value": round(us, 3),
            "unit": "us/call",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(mean_ms, 5),
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded Zipf ids, N(0, sigma) grad / main_grad)",
            "config": {
                "workload": w.name, "num_embeddings": V, "hidden": H, "num_tokens": n,
                "ids": f"zipf(s={w.zipf_s})" if w.ids_dist == "zipf" else w.ids_dist,
                "grad_dtype": str(w.grad_dtype).replace("torch.", ""),
                "main_grad_dtype": str(w.mg_dtype).replace("torch.", ""),
                "unique_ids": U, "l2": "256 MiB memset before every timed call",
                "parallelism": f"replicas x{world}",
            },
            "median_us": round(median_ms * 1e3, 3),
            "hbm_gbs": round(call_bytes / (mean_ms * 1e-3) / 1e9, 1),
            "job_hbm_gbs": round(world * call_bytes / (mean_ms * 1e-3) / 1e9, 1),
            "frac_of_8tbs": round(call_bytes / (mean_ms * 1e-3) / 8e12, 4),
            "algorithmic_bytes_per_call": call_bytes,
            "plan_us": round(plan_mean * 1e3, 3),
            "clean_l2": {"value": round(clean_ms * 1e3, 3), "unit": "us/call",
                         "flush": "256 MiB memset then a 256 MiB read before every call"},
            "back_to_back": {"value": round(b2b_ms * 1e3, 3), "unit": "us/call",
                             "what": "calls enqueued with no flush and no host sync in between"},
            "after_idle": {"value": round(idle_ms * 1e3, 3), "unit": "us/call",
                           "what": "host sync and 1 ms of GPU idle before every call"},
            "apply_us": round(apply_mean * 1e3, 3),
            "roofline": {
                "kernel": "apply_kernel (one ewg_apply call)",
                "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": apply_bytes,
                "traffic": traffic,
            },
            "e2e": {
                "value": round(e2e_mean * 1e3, 3), "unit": "us/call",
                "h2d_bytes_per_step": ids_h.nbytes + grad_h.numel() * grad_h.element_size(),
                "d2h_bytes_per_step": 4,
            },
            "gpu_launches": launches_per_call * args.steps if launches_per_call else None,
            "timed_region_s": round(region_s, 4),
        }
        clk = sampler.summary()
        if clk:
            out["clocks"] = clk
        if not args.no_extras:
            out["dense_path"] = dense_path(w, ids_d, grad_d, mg, args, stream, flush)
            out["shards"] = shard_path(w, ids_d, grad_d, mg, args, stream, flush, ws)
    return out


def shard_path(w, ids_d, grad_d, mg, args, stream, flush, ws):
    """The table split in two row halves, one ewg_accumulate_shard call each (on a
    vocabulary-parallel setup each GPU runs one of them)."""
    import embedding_weight_grad_gb300 as ewg

    V = w.num_embeddings
    half = V // 2
    out = {}
    for name, b0, b1 in (("rows_0_to_half", 0, half), ("rows_half_to_end", half, V)):
        part = mg[b0:b1]

        def call():
            ewg.accumulate_embedding_wgrad_shard(ids_d, grad_d, part, b0, V, workspace=ws)

        for _ in range(3):
            flush()
            call()
        ms = time_events(call, 20, stream, flush)
        out[name] = round(statistics.fmean(ms) * 1e3, 2)
    out["unit"] = "us/call"
    return out


def dense_path(w, ids_d, grad_d, mg, args, stream, flush):
    """PyTorch's dense path on the same GPU: embedding_dense_backward then main_grad.add_
    over every row (the comparison the page's 'about 1 ms per embedding use' describes)."""
    V = w.num_embeddings

    def call():
        dense = torch.ops.aten.embedding_dense_backward(grad_d, ids_d, V, -1, False)
        mg.add_(dense)

    for _ in range(3):
        flush()
        call()
    ms = time_events(call, 20, stream, flush)
    return {"us_per_call": round(statistics.fmean(ms) * 1e3, 2), "calls": 20,
            "what": "torch embedding_dense_backward + main_grad.add_ (whole [V, H])"}


# --- CPU oracle (baseline and reference arm) -------------------------------------------

def oracle_sample(w):
    """The oracle's inputs for one call: the full token list and grad, and the touched
    main_grad rows (ids renumbered densely in the same order, which leaves every run and
    its order unchanged, so the arithmetic work is the call's)."""
    ids, grad = host_inputs(w)
    touched = np.unique(ids)
    dense = np.searchsorted(touched, ids)
    g = grad.view(torch.int16).numpy().view(np.uint16) if grad.dtype == torch.bfloat16 \
        else grad.numpy()
    mg = workloads.make_main_grad(workloads.scaled(w, num_embeddings=touched.size))
    mg = mg.view(torch.int16).numpy().view(np.uint16) if mg.dtype == torch.bfloat16 else mg.numpy()
    return dense, g, mg


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(w, budget_s, max_calls=None, threads=None):
    import oracle
    oracle.build()
    dense, g, mg = oracle_sample(w)
    c = threads or cores()
    times = []
    t_all = time.perf_counter()
    while True:
        work = mg.copy()
        t0 = time.perf_counter()
        oracle.accumulate(dense, g, work, num_threads=c)
        times.append(time.perf_counter() - t0)
        if max_calls and len(times) >= max_calls:
            break
        if time.perf_counter() - t_all >= budget_s:
            break
    return times, c


def cpu_baseline(w, budget_s):
    """The oracle on every host core (the reported value) and on one core."""
    times, c = time_oracle(w, 0.7 * budget_s)
    one, _ = time_oracle(w, 0.3 * budget_s, threads=1)
    return {"value": round(statistics.fmean(times) * 1e6, 1), "unit": "us/call", "cores": c,
            "kind": "oracle",
            "single_thread_us": round(statistics.fmean(one) * 1e6, 1),
            "sample": f"{len(times)} full calls of the {w.name} workload (all {w.num_tokens} "
                      f"tokens x {w.hidden} columns, touched main_grad rows) on {c} threads, "
                      f"{sum(times):.1f} s wall; {len(one)} calls on one thread"}


def run_reference(args, w, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    dense, g, mg = oracle_sample(w)
    c = cores()
    for _ in range(args.warmup):
        oracle.accumulate(dense, g, mg.copy(), num_threads=c)
    # each step is one full oracle call; bound the whole run to a few minutes
    steps = args.steps
    t_probe = time.perf_counter()
    oracle.accumulate(dense, g, mg.copy(), num_threads=c)
    one = time.perf_counter() - t_probe
    steps = max(1, min(steps, int(120.0 / max(one, 1e-6))))
    times = []
    for _ in range(steps):
        work = mg.copy()
        t0 = time.perf_counter()
        oracle.accumulate(dense, g, work, num_threads=c)
        times.append(time.perf_counter() - t0)
    us = statistics.fmean(times) * 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/call",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, same recipe)",
        "config": {"workload": w.name, "num_embeddings": w.num_embeddings, "hidden": w.hidden,
                   "num_tokens": w.num_tokens},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": c, "kind": "oracle",
                         "sample": f"{steps} full calls of the {w.name} workload"},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world, rank, local = dist_env()
    w = workloads.BY_NAME[args.workload]
    if args.impl == "reference":
        out = run_reference(args, w, rank)
        if out:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    out = run_ours(args, w, world, rank, local)
    if rank == 0 and out is not None:
        if not args.no_extras:
            out["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
