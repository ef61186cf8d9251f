"""Benchmark of paged verify attention on GB300 (one JSON line on rank 0).

A step is one call of the whole path (split-KV kernel + log-sum-exp combine)
over one batch of the MTP-5 bf16 verify workload: 8 sequences, 6 verify
tokens each, 32 q / 4 KV heads, head_dim 128, context lengths uniform in
[4096, 32768], 16-token pages scattered in the pool, q/K/V ~ N(0, 1).
`value` is KV GB/s (algorithmic K+V bytes read once, divided by the median
call time), `ms_per_step` the median call time. `roofline.frac` is the split
kernel's own fraction of the HBM peak (its bytes over its event time);
`roofline.frac_call` is the same bytes over the whole call. The other
long-context workloads (MTP-5 FP8, the mixed FP8 batch, the 1 Mi-token
context, head_dim 256 FP8 at batch 8) are measured the same way and reported
under `other_configs`. Under torchrun each rank runs its own batch (weak
scaling, no data exchange); rank 0 prints the job aggregate.

`--impl reference` times the CPU fp64 oracle on the same workload instead
(a bounded sample per step, on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_speculative_gb300 import synth  # noqa: E402

METRIC = "verify-attention µs/call and KV GB/s vs GB300 HBM peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_DESC = {
    "tiny": "tiny: B=2 q=[1,6] ctx=[37,100] Hq=4 Hkv=1 D=64 bf16 KV, 32-page pool, seed 0",
    "mtp5_bf16": "MTP-5 verify bf16 KV: B=8 q=6 Hq=32 Hkv=4 D=128 page 16, ctx U[4096,32768] (seed 2), scattered pages",
    "mtp5_fp8": "MTP-5 verify FP8 E4M3 KV + per-token fp32 scales: B=4 q=6 Hq=32 Hkv=4 D=128, ctx 131072 each (seed 3)",
    "mixed_fp8": "mixed FP8 batch: B=64 q U{1..8} Hq=16 Hkv=2 D=128, ctx lognormal(median 8192, sigma 1, cap 131072) (seed 4)",
    "ctx1mi_bf16": "1Mi-token verify bf16 KV: B=1 q=6 Hq=8 Hkv=1 D=128, ctx 1048576, 65536-entry table, random page order (seed 5)",
}
for _bs in (1, 2, 4, 8):
    WORKLOAD_DESC[f"d256_fp8_bs{_bs}"] = (f"head_dim 256 FP8 E4M3 KV + per-token fp32 scales: B={_bs} q=6 Hq=8 Hkv=1 "
                                          "(48 rows), ctx 150000 each, scattered pages (seed 6)")
WORKLOAD_DESC["d256_bf16_bs8"] = ("head_dim 256 bf16 KV: B=8 q=6 Hq=8 Hkv=1 (48 rows), ctx 150000 each, scattered pages "
                                  "(seed 6)")


_C_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(src: str) -> str:
    """C/C++/CUDA source without comments, whitespace runs collapsed (string literals kept)."""
    no_comments = _C_TOKENS.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", src)
    return " ".join(no_comments.split())


def kernel_source_hash() -> str:
    """Identifies the library's code: comments and layout do not count, so a counter capture stays valid
    across edits that change neither."""
    csrc = os.path.join(ROOT, "paged_kv_speculative_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return None, "fallback"


def hbm_peak(peaks):
    if peaks:
        for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs", "hbm"):
            v = peaks.get(k)
            if isinstance(v, (int, float)) and v > 0:
                return float(v), "of measured"
            if isinstance(v, dict):
                for kk in ("gbs", "value", "burst"):
                    if isinstance(v.get(kk), (int, float)):
                        return float(v[kk]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


def traffic_for(workload: str):
    """DRAM bytes per split-kernel launch from a committed ncu summary, if the
    kernel sources still match the ones the counters were taken on."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(prob, budget_s: float, sample_note_prefix: str):
    """Times the oracle on whole sequences of `prob` (all their rows) until
    about `budget_s` seconds of wall time have been spent."""
    import oracle
    threads = os.cpu_count() or 1
    off = prob.q_offsets()
    order = np.argsort(prob.context_lens)  # short sequences first keeps the first sample small
    done_bytes, elapsed, seqs = 0, 0.0, 0
    per_th = 2 * prob.head_dim * (2 if prob.kv_dtype == synth.KV_BF16 else 1) + (8 if prob.kv_dtype == synth.KV_FP8 else 0)
    for b in order:
        rows = np.array([(t, h) for t in range(off[b], off[b + 1]) for h in range(prob.num_q_heads)], dtype=np.int64)
        t0 = time.perf_counter()
        oracle.verify_attention(prob, rows=rows, threads=threads)
        elapsed += time.perf_counter() - t0
        done_bytes += int(prob.context_lens[b]) * prob.num_kv_heads * per_th
        seqs += 1
        if elapsed >= budget_s:
            break
    gbs = done_bytes / elapsed / 1e9
    note = (f"{sample_note_prefix}: {seqs} of {prob.num_seqs} sequences (all rows), {done_bytes / 1e6:.1f} MB of KV, "
            f"{elapsed:.2f} s, fp64 C oracle, {threads} threads")
    return gbs, threads, note, elapsed


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    prob = synth.make_config(args.config, poison=False)
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        cpu_oracle_sample(prob, 0.0, "warmup")
    vals, times = [], []
    note, threads = "", 1
    for _ in range(args.steps):
        gbs, threads, note, el = cpu_oracle_sample(prob, args.ref_budget, "sample")
        vals.append(gbs)
        times.append(el)
    value = float(statistics.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(statistics.median(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD_DESC[args.config], "name": args.config},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": note},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class L2Flush:
    """Evicts the call's inputs from L2 between steps, outside the timed events:
    writes one 256 MiB buffer (> 129 MB L2), then reads another, so the timed
    call starts with L2 holding clean lines only, as under ncu's cache control
    (with dirty lines left behind, their write-back would compete with the
    call's reads)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def _timed(fn, steps, warmup, flush, dev):
    import torch
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    return ms


def run_side_op(args):
    """Measures the paged KV write (FP8 quantising) or the greedy verdict."""
    import torch
    from paged_kv_speculative_gb300 import _build, pa_verify as pv
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    flush = L2Flush(dev)
    g = torch.Generator(device="cpu").manual_seed(7)
    peaks, _ = load_peaks()
    peak, peak_note = hbm_peak(peaks)
    if args.op == "kv_write":
        # bulk write: 8192 new tokens x 8 KV heads x head_dim 128, bf16 in -> E4M3 + fp32 scales
        n, hkv, d, n_pg = 8192, 8, 128, 8192 // 16 + 64
        k_new = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16).to(dev)
        v_new = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16).to(dev)
        slots = torch.randperm(n_pg * 16, generator=g)[:n].to(torch.int64).to(dev)
        kc = torch.zeros((n_pg, hkv, 16, d), dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.zeros((n_pg, hkv, 16), dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        fn = lambda: pv.kv_write(k_new, v_new, slots, kc, vc, ks, vs, pv.KV_FP8_E4M3)
        nbytes = 2 * n * hkv * d * 2 + n * 8 + 2 * n * hkv * (d + 4)
        workload = "paged KV write, FP8 per-token quantisation: 8192 tokens x 8 KV heads x D=128, random slots"
        metric, launches = "paged KV write GB/s (bf16 in, E4M3 + fp32 scales out)", 1
    else:
        # greedy verdict over the MTP-5 verify positions of 8 sequences, vocab 151936
        B, q, V = 8, 6, 151936
        T = B * q
        logits = (torch.randn((T, V), generator=g) * 3).to(torch.bfloat16).to(dev)
        ids = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).to(dev)
        ql = torch.full((B,), q, dtype=torch.int32, device=dev)
        ws = torch.zeros(pv.lib().pa_greedy_verdict_workspace_bytes(T, V), dtype=torch.uint8, device=dev)
        fn = lambda: pv.greedy_verdict(logits, ids, ql, workspace=ws)
        nbytes = T * V * 2
        workload = "greedy verify verdict: 8 sequences x 6 verify positions, vocab 151936, bf16 logits"
        metric, launches = "greedy verdict GB/s (logits read once)", 2
    ms = _timed(fn, args.steps, args.warmup, flush, dev)
    mean = float(np.mean(ms))
    gbs = nbytes / (mean * 1e-3) / 1e9
    line = {"op": args.op, "metric": metric, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean, "us_per_call": 1e3 * mean, "higher_is_better": True,
            "dtype": "bf16 in", "data": "synthetic",
            "config": {"workload": workload, "bytes_per_call": nbytes,
                       "l2": "flushed between steps (256 MiB write, then 256 MiB read: L2 left clean; outside the events)"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": peak_note},
            "gpu_launches": args.steps * launches}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mtp5_bf16", choices=list(synth.ALL_NAMES))
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=3.0, help="seconds of oracle time per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--also", default="mtp5_fp8,mixed_fp8,ctx1mi_bf16,d256_fp8_bs8,d256_bf16_bs8",
                    help="comma-separated extra workloads to report under 'other_configs' ('' for none)")
    ap.add_argument("--also-cpu-budget", type=float, default=3.0,
                    help="seconds of oracle time for each extra workload's cpu_baseline")
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "tc"],
                    help="split kernel: automatic choice, warp-MMA, or tcgen05")
    ap.add_argument("--op", default="verify", choices=["verify", "kv_write", "verdict"],
                    help="verify attention (the path), or the paged KV write / greedy verdict steps around it")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.op != "verify":
        return run_side_op(args)

    import torch
    import torch.distributed as dist
    from paged_kv_speculative_gb300 import _build, pa_verify as pv, replicas
    from paged_kv_speculative_gb300.device_inputs import host_tensors

    world, rank, local = dist_setup()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    _build.build()

    def barrier():
        if world > 1:
            dist.barrier()

    flush = L2Flush(dev)

    def measure(name, steps, warmup, seed_offset):
        ctx, ql, hq, hkv, d, kvd, seed = synth.config_lengths(name)
        kw = {"pool_pages": 32} if name == "tiny" else {}
        prob = synth.make_problem(ctx, ql, hq, hkv, d, kv_dtype=kvd, seed=seed + 1000 * seed_offset, poison=False,
                                  name=name, **kw)
        host = host_tensors(prob, pin=True)
        dv = [None if x is None else x.to(dev) for x in host.args()]
        kern = {"auto": pv.KERNEL_AUTO, "mma": pv.KERNEL_WARP_MMA, "tc": pv.KERNEL_TCGEN05}[args.kernel]
        va = pv.VerifyAttention(hq, hkv, d, kvd, prob.num_pages, prob.block_table.shape[1], ctx, ql,
                                out_dtype=pv.OUT_BF16, device=dev, kernel=kern)
        out = va.new_out()
        stream = torch.cuda.current_stream(dev)
        for _ in range(warmup):
            flush()
            va(*dv, prob.softmax_scale, out=out)
        torch.cuda.synchronize(dev)
        # timed steps: events only around the call, nothing recorded inside it
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for k in range(steps):
            flush()
            evs[k][0].record(stream)
            va(*dv, prob.softmax_scale, out=out)
            evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        wall = time.perf_counter() - wall0
        step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
        # the same number of steps again with the library's per-kernel events (split kernel, combine)
        pv.profile_enable(va.plan, True)
        split_ms, comb_ms = [], []
        for k in range(steps):
            flush()
            va(*dv, prob.softmax_scale, out=out)
            a, c = pv.profile_read(va.plan)
            split_ms.append(a)
            comb_ms.append(c)
        pv.profile_enable(va.plan, False)
        errs = va.device_errors()
        info = va.info
        res = {"prob": prob, "host": host, "va": va, "dv": dv, "out": out, "step_ms": step_ms,
               "split_ms": split_ms, "comb_ms": comb_ms, "wall": wall, "info": info, "errs": errs}
        return res

    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        r = measure(args.config, args.steps, args.warmup, rank)
    clocks = clk.summary()
    prob, info = r["prob"], r["info"]
    med_ms = float(np.median(r["step_ms"]))
    mean_ms = float(np.mean(r["step_ms"]))
    step_ms_job = replicas.max_over_ranks(med_ms, device=dev)  # the slowest rank's median call
    kv_bytes_rank = int(info["kv_bytes"])
    kv_bytes_all = replicas.sum_over_ranks(kv_bytes_rank, device=dev)
    value = replicas.job_throughput(kv_bytes_all, 1, step_ms_job)
    split_avg = float(np.mean(r["split_ms"]))
    comb_avg = float(np.mean(r["comb_ms"]))

    # ---- end to end through the public API with host buffers
    host, va = r["host"], r["va"]
    out_host = torch.empty(r["out"].shape, dtype=r["out"].dtype, pin_memory=True)
    dv = r["dv"]
    h2d = sum(x.numel() * x.element_size() for x in host.args() if x is not None)
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.current_stream(dev)
    e2e_ms = []
    for k in range(args.e2e_steps + 2):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for dst, src in zip(dv, host.args()):
            if src is not None:
                dst.copy_(src, non_blocking=True)
        va(*dv, prob.softmax_scale, out=r["out"])
        out_host.copy_(r["out"], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if k >= 2:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_val = replicas.job_throughput(kv_bytes_all, 1, replicas.max_over_ranks(float(np.mean(e2e_ms)), device=dev))

    peaks, _ = load_peaks()
    peak, peak_note = hbm_peak(peaks)
    others = {}
    for name in [x for x in args.also.split(",") if x and x != args.config]:
        o = measure(name, max(10, args.steps // 2), args.warmup, rank)
        oms = float(np.median(o["step_ms"]))
        osplit = float(np.mean(o["split_ms"]))
        ocomb = float(np.mean(o["comb_ms"]))
        ob = o["info"]["kv_bytes"]
        others[name] = {"workload": WORKLOAD_DESC[name], "us_per_call": 1e3 * oms,
                        "kv_gbs": ob / (oms * 1e-3) / 1e9, "frac_call": ob / (oms * 1e-3) / 1e9 / peak,
                        "split_kernel_us": 1e3 * osplit, "combine_kernel_us": 1e3 * ocomb,
                        "split_kernel_gbs": ob / (osplit * 1e-3) / 1e9,
                        "frac_split": ob / (osplit * 1e-3) / 1e9 / peak, "peak_source": peak_note,
                        "kv_bytes_per_call": ob, "steps": len(o["step_ms"]),
                        "traffic": traffic_for(name),
                        "units": o["info"]["num_units"], "chunk": o["info"]["chunk_tokens"],
                        "splits_max": o["info"]["max_splits"],
                        "kernel": "tcgen05" if o["info"]["kernel"] == pv.KERNEL_TCGEN05 else "warp-mma",
                        "device_errors": o["errs"]}
        if rank == 0 and not args.no_cpu_baseline:
            gbs, threads, note, _ = cpu_oracle_sample(o["prob"], args.also_cpu_budget, "sample")
            others[name]["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                            "sample": note}
        del o

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    achieved = kv_bytes_rank / (split_avg * 1e-3) / 1e9
    call_gbs = kv_bytes_rank / (med_ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        gbs, threads, note, _ = cpu_oracle_sample(prob, args.cpu_budget, "sample")
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": note}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms_job, "us_per_call": 1e3 * med_ms,
        "us_per_call_mean": 1e3 * mean_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if prob.kv_dtype == 0 else "fp8-e4m3 KV, bf16 q",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.config], "name": args.config,
                   "kv_bytes_per_call": kv_bytes_rank, "l2": "flushed between steps (256 MiB write, then 256 MiB read: L2 left clean; outside the events)",
                   "units": info["num_units"], "chunk_tokens": info["chunk_tokens"], "splits_max": info["max_splits"],
                   "kernel": "tcgen05" if info["kernel"] == pv.KERNEL_TCGEN05 else "warp-mma",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_note, "traffic": traffic_for(args.config),
                     "frac_call": call_gbs / peak, "call_gbs": call_gbs,
                     "kernel": "pa_tc_split_kernel" if info["kernel"] == pv.KERNEL_TCGEN05 else "pa_split_kernel",
                     "split_kernel_us": 1e3 * split_avg, "combine_kernel_us": 1e3 * comb_avg},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": float(np.mean(e2e_ms))},
        "gpu_launches": args.steps * (1 + int(info["needs_combine"])),
        "clocks": clocks,
        "device_errors": r["errs"],
    }
    if cpu:
        line["cpu_baseline"] = cpu
    if others:
        line["other_configs"] = others
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
