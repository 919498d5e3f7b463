"""Benchmark of the paged-MLA hot path on GB300 (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the whole path (split-KV attention kernel + merge kernel) over one
batch of a named synthetic workload, inputs resident in HBM.  Before every timed step
L2 is flushed by writing a 256 MiB buffer; each step is timed with CUDA events on the
launching stream.  ``value`` is the median microseconds per call of the headline
workload (decode, batch 128, 128 heads, page size 1, 4096 keys each: the largest
single-GPU decode configuration); p10/p90 and the mean are reported beside it.
``configs`` holds the same measurements for the other named workloads (the small
decode, the page-64 decode, the skewed decode, the causal prefill, the packed
multi-token decode and the sparse top-k decode).  ``e2e`` times the
headline call from pinned host buffers: host->device copies of every input, the call,
and the device->host copy of out and lse.

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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA paged decode µs/call, KV TB/s & TFLOP/s as % of GB300 roofline"
HEADLINE = "decode_b128_h128_ps1"
SUB_WORKLOADS = ("decode_b4_h16_ps64", "decode_b64_h128_ps64", "decode_b32_h128_skew", "prefill_causal_h128",
                 "mtp_b64_h16_q4_ps64", "sparse_b64_h128_topk2048", "fp8_b64_h128_ps64")
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
    pair that the causal mask keeps.  Sparse decode: 1152 B per valid entry (padding
    entries read only their 4 B index).  An FP8 cache holds 656 B per key instead of 1152."""
    keys = w.visible_keys()
    rows_heads = w.rows * w.num_qo_heads
    kv_bytes = 656 if w.kind.endswith("_fp8") else 1152
    if w.kind.startswith("sparse"):
        nbytes = keys * kv_bytes + w.num_kv_indices * 4 + rows_heads * (1152 + 1024 + 4)
    else:
        nbytes = sum(w.kv_lens()) * (kv_bytes + 4) + rows_heads * (1152 + 1024 + 4)
    flops = keys * w.num_qo_heads * 2 * (576 + 512)
    return nbytes, flops, keys


def config_of(w):
    """The workload description both arms print (identical keys and values)."""
    c = {"workload": w.name, "batch": w.batch, "num_qo_heads": w.num_qo_heads, "page_size": w.page_size,
         "visible_keys": w.visible_keys()}
    if w.kv_fp8 is not None:
        c["kv_cache"] = "fp8 e4m3 latent + fp32 tile scales + bf16 rope, 656 B/token"
    return c


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


def percentiles(vals):
    v = sorted(vals)
    q = lambda f: v[min(len(v) - 1, max(0, int(round(f * (len(v) - 1)))))]
    return {"median": statistics.median(v), "p10": q(0.10), "p90": q(0.90), "mean": sum(v) / len(v)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"mla_clocks_{os.getpid()}.csv")

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


# ------------------------------------------------------------------ CPU oracle legs

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
        slots = slots[(slots >= 0) & (slots < ckv.shape[0])]  # sparse decode: padding entries are skipped
        if w.kv_fp8 is not None:  # the FP8 oracle reads the row's tokens back to BF16 first
            k_ckv, k_kpe = oracle.dequantize_fp8_cache(w.kv_fp8.view(-1, 656)[slots].numpy())
        else:
            k_ckv, k_kpe = ckv[slots].float().numpy(), kpe[slots].float().numpy()
        oracle.attend(w.q_nope[r].float().numpy(), w.q_pe[r].float().numpy(), k_ckv, k_kpe, w.sm_scale)
        keys += slots.numel()
        done += 1
        if time.perf_counter() - t0 >= budget_s or (max_rows and done >= max_rows):
            break
    return time.perf_counter() - t0, keys, done


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(w, budget_s):
    keys = w.visible_keys()
    secs, ck, cr = time_oracle(w, budget_s)
    return {"value": secs / max(ck, 1) * keys * 1e6, "unit": "us/call", "cores": cores_used(), "kind": "oracle",
            "sample": f"{cr} of {w.rows} query rows (all heads) of {w.name}, {ck} of {keys} visible keys, "
                      f"{secs:.1f} s, scaled to the whole call"}


_SINGLE_THREAD = r"""
import json, sys, time
import numpy as np
sys.path.insert(0, sys.argv[2])
import oracle
d = np.load(sys.argv[1])
best = None
for _ in range(3):
    t0 = time.perf_counter()
    oracle.mla_decode(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], d["indptr"], d["indices"], float(d["scale"]))
    t = time.perf_counter() - t0
    best = t if best is None or t < best else best
print(json.dumps({"us": best * 1e6}))
"""


def single_thread_oracle_us(w):
    """The whole call of a (small) decode workload on one host thread: the oracle runs in
    a child process whose BLAS is limited to one thread; min of three runs."""
    import numpy as np
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "inputs.npz")
        np.savez(path, q_nope=w.q_nope.float().numpy(), q_pe=w.q_pe.float().numpy(),
                 ckv=w.ckv_cache.float().numpy(), kpe=w.kpe_cache.float().numpy(),
                 indptr=w.kv_indptr.numpy(), indices=w.kv_indices.numpy(), scale=w.sm_scale)
        env = dict(os.environ)
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[k] = "1"
        r = subprocess.run([sys.executable, "-c", _SINGLE_THREAD, path, ROOT], capture_output=True, text=True,
                           env=env, timeout=300)
        if r.returncode != 0:
            return None
        return json.loads(r.stdout.strip().splitlines()[-1])["us"]


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
        "data": "synthetic", "config": config_of(w),
        "kv_tbs": nbytes / (us_per_call * 1e-6) / 1e12, "tflops": flops / (us_per_call * 1e-6) / 1e12,
        "cpu_baseline": {"value": us_per_call, "unit": "us/call", "cores": cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": us_per_call, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ our arm

def roofline_of(w_cpu, kernel_ms, peaks, peak_kind):
    """Roofline of the dominant (attention) kernel: algorithmic bytes or flops per launch
    over its CUDA-event duration, against the measured HBM copy bandwidth or bf16 GEMM
    rate, whichever bound the operator's work has (a kernel that runs for milliseconds
    is compared with the sustained bf16 figure, a short one with the burst figure)."""
    nbytes, flops, _ = algorithmic_work(w_cpu)
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])
    ach_gbs = nbytes / (kernel_ms * 1e-3) / 1e9
    ach_tflops = flops / (kernel_ms * 1e-3) / 1e12
    tensor_bound = flops / (tc * 1e12) > nbytes / (hbm * 1e9)
    common = {"peak_kind": peak_kind, "kernel": "attention kernel (mla_tc_kernel)", "kernel_us": kernel_ms * 1e3,
              "hbm_gbs": ach_gbs, "hbm_frac": ach_gbs / hbm, "tensor_tflops": ach_tflops, "tensor_frac": ach_tflops / tc,
              "algorithmic_bytes": nbytes, "algorithmic_flops": flops}
    if tensor_bound:
        tc_peak = float(peaks.get("bf16_tflops_sustained", tc)) if kernel_ms > 1.0 else tc
        return {"bound": "tensor", "achieved": ach_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ach_tflops / tc_peak, "traffic": recorded_traffic(w_cpu.name),
                "peak_figure": "sustained" if kernel_ms > 1.0 else "burst", **common}
    return {"bound": "hbm", "achieved": ach_gbs, "peak": hbm, "unit": "GB/s", "frac": ach_gbs / hbm,
            "traffic": recorded_traffic(w_cpu.name), **common}


def measure(mla, w_cpu, dev, stream, flush, steps, warmup, world, clocks_uuid=None, e2e=False, quick=False):
    """Time `steps` calls of the path on `w_cpu` (inputs resident on `dev`, L2 flushed
    before every call); returns per-call statistics, per-kernel times and, with e2e,
    the end-to-end time from pinned host buffers."""
    import torch
    w = w_cpu.to(dev)
    out = torch.empty(w.rows, w.num_qo_heads, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.rows, w.num_qo_heads, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        ws = torch.zeros(mla.workload_workspace_bytes(w), dtype=torch.uint8, device=dev)
        call = mla.bind_workload(w, out, lse, ws, stream)  # arguments checked and marshalled once
        for _ in range(max(warmup, 3)):
            flush.fill_(1)
            call()
    stream.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    res = {}
    clocks = ClockSampler(clocks_uuid) if clocks_uuid is not False else None
    wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push(f"timed {w.name}")
    if clocks:
        clocks.__enter__()
    try:
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush.fill_(i & 0xFF)
                starts[i].record(stream)
                call()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        # keep sampling clocks long enough for a few readings when the timed loop was short
        while clocks and not quick and time.perf_counter() - wall0 < 1.0:
            with torch.cuda.stream(stream):
                for _ in range(20):
                    call()
            stream.synchronize()
    finally:
        if clocks:
            clocks.__exit__()
        torch.cuda.nvtx.range_pop()
    res["wall_s_timed_loop"] = time.perf_counter() - wall0
    step_us = [s.elapsed_time(e) * 1e3 for s, e in zip(starts, ends)]
    res["us"] = percentiles(step_us)
    res["us"]["median"] = max_over_ranks(res["us"]["median"], world, dev)
    if clocks:
        res["clocks"] = clocks.summary()
    # Per-kernel durations: the same steps again with the library's CUDA events around
    # each kernel on the launching stream (kept out of the first pass, whose call time
    # they would lengthen by separating the two kernels).
    torch.cuda.synchronize(dev)
    mla.profile_enable(True)
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(i & 0xFF)
            call()
    torch.cuda.synchronize(dev)
    main_ms, comb_ms, ncalls = mla.profile_read()
    mla.profile_enable(False)
    res["kernel_ms"] = main_ms / max(ncalls, 1)
    res["combine_ms"] = comb_ms / max(ncalls, 1)
    if e2e:
        host = {k: v.pin_memory() for k, v in w_cpu.tensors().items()}
        dev_in = w.tensors()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        res["h2d"] = sum(t.numel() * t.element_size() for t in host.values())
        res["d2h"] = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
        e2e_steps = 0 if quick else max(3, min(steps, 30))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push(f"e2e {w.name}")
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
        torch.cuda.nvtx.range_pop()
        res["e2e_us"] = max_over_ranks(e0.elapsed_time(e1) / e2e_steps * 1e3 if e2e_steps else float("nan"),
                                       world, dev)
    del ws, out, lse, w
    return res


def our_arm(args, rank, world, local_rank):
    import torch
    import paged_head_latent_gb300 as mla
    from paged_head_latent_gb300 import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks, peak_kind = load_peaks()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass

    w_cpu = wl.by_name(args.workload)
    m = measure(mla, w_cpu, dev, stream, flush, args.steps, args.warmup, world, clocks_uuid=uuid,
                e2e=True, quick=args.quick)
    subs = []
    if world == 1 and not args.no_sub:
        for name in SUB_WORKLOADS:
            if name == args.workload:
                continue
            ws_cpu = wl.by_name(name)
            steps = min(args.steps, 20 if ws_cpu.kind == "prefill" else 100)
            sm = measure(mla, ws_cpu, dev, stream, flush, steps, args.warmup, 1, clocks_uuid=False, quick=True)
            nb, fl, _ = algorithmic_work(ws_cpu)
            hbm, tc = float(peaks["hbm_gbs"]), float(peaks["bf16_tflops"])
            roof_us = max(nb / (hbm * 1e9), fl / (tc * 1e12)) * 1e6
            sub = {"workload": name, "config": config_of(ws_cpu), "steps": steps,
                   "us_median": sm["us"]["median"], "us_p10": sm["us"]["p10"], "us_p90": sm["us"]["p90"],
                   "us_mean": sm["us"]["mean"], "kernel_us": sm["kernel_ms"] * 1e3,
                   "combine_us": sm["combine_ms"] * 1e3, "roofline_time_us": roof_us,
                   "roofline_frac_call": roof_us / sm["us"]["median"],
                   "roofline": roofline_of(ws_cpu, sm["kernel_ms"], peaks, peak_kind)}
            if not args.no_cpu_baseline and not args.quick:
                sub["cpu_baseline"] = cpu_baseline(ws_cpu, 3.0 if ws_cpu.kind == "prefill" else 2.0)
                if name == "decode_b4_h16_ps64":
                    st = single_thread_oracle_us(ws_cpu)
                    sub["cpu_baseline_single_thread_us"] = st
            subs.append(sub)
    if rank != 0:
        return
    nbytes, flops, keys = algorithmic_work(w_cpu)
    hbm, tc = float(peaks["hbm_gbs"]), float(peaks["bf16_tflops"])
    us = m["us"]["median"]
    roof_time_us = max(nbytes / (hbm * 1e9), flops / (tc * 1e12)) * 1e6
    cpu = None
    if world == 1 and not args.no_cpu_baseline and not args.quick:
        cpu = cpu_baseline(w_cpu, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": us, "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w_cpu),
        "timing": {"us_median": us, "us_p10": m["us"]["p10"], "us_p90": m["us"]["p90"], "us_mean": m["us"]["mean"],
                   "statistic": "value is the median of the per-step CUDA-event times",
                   "l2": "flushed before every step (256 MiB write)", "accumulate": "fp32", "replicas": world,
                   "kernel_timing": "attention and merge kernels timed with CUDA events in a second pass"},
        "kv_tbs": nbytes / (us * 1e-6) / 1e12,
        "tflops": flops / (us * 1e-6) / 1e12,
        "roofline_time_us": roof_time_us,
        "roofline_frac_call": roof_time_us / us,
        "roofline": dict(roofline_of(w_cpu, m["kernel_ms"], peaks, peak_kind), combine_us=m["combine_ms"] * 1e3),
        "cpu_baseline": cpu,
        "e2e": {"value": m.get("e2e_us"), "unit": "us/call", "h2d_bytes_per_step": m.get("h2d"),
                "d2h_bytes_per_step": m.get("d2h")},
        "gpu_launches": 2 * args.steps,
        "clocks": m.get("clocks"),
        "wall_s_timed_loop": m["wall_s_timed_loop"],
        "configs": subs,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="measure only the named workload")
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
