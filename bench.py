"""Benchmark of the paged-MLA decode hot path on GB300 (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the whole path (split-KV attention kernel + combine kernel)
over one batch of the named synthetic workload, inputs resident in HBM.  Between
timed steps L2 is flushed by writing a 256 MiB buffer; each step is timed with
CUDA events on the launching stream.  ``value`` is microseconds per call.
``e2e`` times the same call from pinned host buffers: host->device copies of every
input, the call, and the device->host copy of out and lse.

--impl reference times the float64 CPU oracle on the host cores instead (bounded
samples of the same workload, scaled to a whole call).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA paged decode µs/call, KV TB/s & TFLOP/s as % of GB300 roofline"
DEFAULT_WORKLOAD = "decode_b64_h128_ps64"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_work(w):
    """Bytes and flops the operator must move / do (per call), per unit:
    1152 B + 4 B index per cached key of a request (a prefill request's query rows share
    its keys, so each is read once); 1152 B q + 1024 B out + 4 B lse per (row, head);
    2 * (576 + 512) flops per (visible key, head), a visible key being a (query row, key)
    pair that the causal mask keeps."""
    keys = w.visible_keys()
    rows_heads = w.rows * w.num_qo_heads
    nbytes = sum(w.kv_lens()) * (1152 + 4) + rows_heads * (1152 + 1024 + 4)
    flops = keys * w.num_qo_heads * 2 * (576 + 512)
    return nbytes, flops, keys


# The sources that define the attention kernel; the recorded DRAM traffic is valid only
# while these are unchanged.
KERNEL_SOURCES = ("mla_tc.cu", "tc_kernel.h", "ptx.cuh", "plan.cuh", "common.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_head_latent_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if it
    was taken on the current kernel sources and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] and self.uuid not in parts[1] and parts[1] not in self.uuid:
                    continue
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[4]) for r in rows if r[4].replace(".", "").isdigit())
                if any(r[4].replace(".", "").isdigit() for r in rows) else None}


# ------------------------------------------------------------------ reference arm

def time_oracle(w, budget_s, max_rows=None):
    """Run the oracle on whole query rows of ``w`` (all heads) until ``budget_s`` of CPU
    wall time has passed; returns (seconds, visible keys processed, rows processed)."""
    import numpy as np
    import oracle
    ckv = w.ckv_cache.view(-1, 512)
    kpe = w.kpe_cache.view(-1, 64)
    kp = w.kv_indptr.tolist()
    qo = w.qo_indptr.tolist() if w.qo_indptr is not None else list(range(w.batch + 1))
    rows = []
    for b in range(w.batch):
        for i in range(qo[b + 1] - qo[b]):
            n = (kp[b + 1] - kp[b]) - (qo[b + 1] - qo[b]) + i + 1
            rows.append((qo[b] + i, kp[b], n))
    order = np.random.default_rng(0).permutation(len(rows))
    t0 = time.perf_counter()
    keys = 0
    done = 0
    for k in order:
        r, k0, n = rows[k]
        slots = w.kv_indices[k0:k0 + max(n, 0)].long()
        oracle.attend(w.q_nope[r].float().numpy(), w.q_pe[r].float().numpy(), ckv[slots].float().numpy(),
                      kpe[slots].float().numpy(), w.sm_scale)
        keys += max(n, 0)
        done += 1
        if time.perf_counter() - t0 >= budget_s or (max_rows and done >= max_rows):
            break
    return time.perf_counter() - t0, keys, done


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def max_over_ranks(value, world, device=None):
    """The largest value over all ranks (every rank gets it); the value itself at N = 1."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reference_arm(args, rank, world):
    from paged_head_latent_gb300 import workloads as wl
    if rank != 0:
        return
    w = wl.by_name(args.workload)
    total_keys = w.visible_keys()
    per_step = max(0.02, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(w, per_step)
    secs, keys = 0.0, 0
    for _ in range(args.steps):
        s, k, _ = time_oracle(w, per_step)
        secs += s
        keys += k
    us_per_call = secs / keys * total_keys * 1e6
    nbytes, flops, _ = algorithmic_work(w)
    sample = (f"{args.steps} steps, each whole query rows (all {w.num_qo_heads} heads) of {w.name} for "
              f"~{per_step:.2f} s; {keys} visible keys in total, scaled to the call's {total_keys} keys")
    line = {
        "impl": "reference", "metric": METRIC, "value": us_per_call, "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us_per_call / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "batch": w.batch, "num_qo_heads": w.num_qo_heads,
                                        "page_size": w.page_size, "visible_keys": total_keys},
        "kv_tbs": nbytes / (us_per_call * 1e-6) / 1e12, "tflops": flops / (us_per_call * 1e-6) / 1e12,
        "cpu_baseline": {"value": us_per_call, "unit": "us/call", "cores": cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": us_per_call, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ our arm

def our_arm(args, rank, world, local_rank):
    import torch
    import paged_head_latent_gb300 as mla
    from paged_head_latent_gb300 import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w_cpu = wl.by_name(args.workload)
    w = w_cpu.to(dev)
    nbytes, flops, keys = algorithmic_work(w_cpu)
    stream = torch.cuda.Stream(dev)
    out = torch.empty(w.rows, w.num_qo_heads, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.rows, w.num_qo_heads, dtype=torch.float32, device=dev)
    ws = None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    with torch.cuda.stream(stream):
        ws = torch.zeros(mla.workload_workspace_bytes(w), dtype=torch.uint8, device=dev)
        # The C-ABI call with its arguments checked and marshalled once.
        call = mla.bind_workload(w, out, lse, ws, stream)
        for _ in range(max(args.warmup, 3)):
            flush.fill_(1)
            call()
    stream.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    with ClockSampler(uuid) as clocks:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                starts[i].record(stream)
                call()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        # keep sampling long enough for a few readings when the timed loop was short
        while not args.quick and time.perf_counter() - wall0 < 1.0:
            with torch.cuda.stream(stream):
                for _ in range(20):
                    call()
            stream.synchronize()
    wall_timed = time.perf_counter() - wall0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_per_step = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    # Per-kernel durations: the same K steps again with the library's CUDA events around
    # each kernel on the launching stream (kept out of the first pass, whose step time
    # they would lengthen by separating the two kernels).
    torch.cuda.synchronize(dev)
    mla.profile_enable(True)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            call()
    torch.cuda.synchronize(dev)
    main_ms, comb_ms, ncalls = mla.profile_read()
    mla.profile_enable(False)
    main_avg_ms = main_ms / max(ncalls, 1)
    comb_avg_ms = comb_ms / max(ncalls, 1)

    # ---- end to end through the C ABI from pinned host buffers
    host = {k: v.pin_memory() for k, v in w_cpu.tensors().items()}
    dev_in = w.tensors()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    e2e_steps = 0 if args.quick else max(3, min(args.steps, 30))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for it in range(e2e_steps + 2 if e2e_steps else 0):
            if it == 2:
                e0.record(stream)
            for k, t in host.items():
                dev_in[k].copy_(t, non_blocking=True)
            call()
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        if e2e_steps:
            e1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps if e2e_steps else float("nan"), world, dev)

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])
    us = ms_per_step * 1e3
    # Dominant kernel: the attention kernel.  Its algorithmic bytes per launch are the
    # whole call's (the combine only re-reads split-KV partials, which are not algorithmic).
    ach_gbs = nbytes / (main_avg_ms * 1e-3) / 1e9
    ach_tflops = flops / (main_avg_ms * 1e-3) / 1e12
    roof_time_us = max(nbytes / (hbm * 1e9), flops / (tc * 1e12)) * 1e6
    # The bound of the dominant kernel: HBM for decode at these head counts, the tensor
    # pipe for long causal prefill.  A kernel that runs for milliseconds is compared with
    # the sustained bf16 figure, a short one with the burst figure.
    tensor_bound = flops / (tc * 1e12) > nbytes / (hbm * 1e9)
    common = {"peak_kind": peak_kind, "kernel": "attention (main) kernel", "kernel_us": main_avg_ms * 1e3,
              "combine_us": comb_avg_ms * 1e3, "hbm_gbs": ach_gbs, "hbm_frac": ach_gbs / hbm,
              "tensor_tflops": ach_tflops, "tensor_frac": ach_tflops / tc}
    if tensor_bound:
        tc_peak = float(peaks.get("bf16_tflops_sustained", tc)) if main_avg_ms > 1.0 else tc
        roofline = {"bound": "tensor", "achieved": ach_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": ach_tflops / tc_peak, "traffic": recorded_traffic(w_cpu.name),
                    "peak_figure": "sustained" if main_avg_ms > 1.0 else "burst", **common}
    else:
        roofline = {"bound": "hbm", "achieved": ach_gbs, "peak": hbm, "unit": "GB/s", "frac": ach_gbs / hbm,
                    "traffic": recorded_traffic(w_cpu.name), **common}
    cpu = None
    if world == 1 and not args.no_cpu_baseline and not args.quick:
        secs, ck, cr = time_oracle(w_cpu, args.cpu_seconds)
        cpu_us = secs / max(ck, 1) * keys * 1e6
        cpu = {"value": cpu_us, "unit": "us/call", "cores": cores_used(), "kind": "oracle",
               "sample": f"{cr} of {w_cpu.rows} query rows (all heads), {ck} of {keys} visible keys, "
                         f"{secs:.1f} s, scaled to the whole call"}
    line = {
        "metric": METRIC, "value": us, "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w_cpu.name, "batch": w_cpu.batch, "num_qo_heads": w_cpu.num_qo_heads,
                   "page_size": w_cpu.page_size, "visible_keys": keys, "replicas": world,
                   "l2": "flushed between steps (256 MiB write)", "accumulate": "fp32"},
        "kv_tbs": nbytes / (us * 1e-6) / 1e12,
        "tflops": flops / (us * 1e-6) / 1e12,
        "roofline_time_us": roof_time_us,
        "roofline_frac_call": roof_time_us / us,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_ms * 1e3, "unit": "us/call", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_loop": wall_timed,
        "kernel_timing": "attention and merge kernels timed with CUDA events in a second pass of the same steps",
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no clock soak, no end-to-end leg, no CPU baseline")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    from paged_head_latent_gb300 import _build
    _build.build_library()
    our_arm(args, rank, world, local_rank)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
