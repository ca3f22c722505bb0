"""Benchmark of the exact attention forward (BF16) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

A step is one attention forward over one batch of the chosen workload (all of
the hot path: loads, QKᵀ, online softmax, P·V, epilogue — one kernel launch).
Throughput is counted as 4·B·H·Sq·Sk·d FLOPs per step, halved when causal,
divided by the kernel time measured with CUDA events on the launching stream.
Inputs are resident in device memory before timing starts; L2 is flushed
(a 256 MiB write) between timed steps.  ``e2e`` repeats the measurement
through the host-buffer C-ABI entry point, with the host↔device copies of
every step inside the timed region.

Multi-GPU (torchrun, one process per GPU): every rank runs the same workload
on its own independently seeded batch — attention heads are independent, so
nothing is exchanged on the data path (weak scaling).  ``--shard heads``
splits the B·H heads of one problem across the ranks instead (strong
scaling; each rank computes its contiguous share of the heads, again with no
exchange).  Only the timing uses a barrier and a max-reduction.

``--impl reference`` times the CPU fp64 oracle (the reference arm of this
comparison) on a bounded sample of the same workload.

Variants of the workload (each its own JSON line, the metric unchanged):
``--kv-heads H_kv`` grouped-query K/V heads; ``--causal-align bottom-right``;
``--varlen N`` N sequences of seeded lengths packed along the rows (FLOPs
counted per sequence); ``--backward`` a step is the backward instead — the
preparation kernel and the dK/dV and dQ passes, three launches — with FLOPs
counted as 2.5× the forward's (S, dP, dV, dK, dQ); ``--fp8`` the FP8 (E4M3)
forward on the workload's E4M3 inputs (head dim 128; FLOPs counted as for
bf16, against twice the measured bf16 peak — the nominal FP8/BF16 ratio of
the tensor core).  The variants report no
``e2e`` (the host-buffer entry point takes the dense forward only), and
``roofline.traffic`` is given only for workloads whose ncu counters are in
``profiles/traffic.json`` for the current kernel sources (else null).
"""

from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (BF16, causal & non-causal) and % of GB300 tensor peak"
CONTRACT_PEAK_TFLOPS = 2250.0  # BF16 dense figure the pages give for the Blackwell tensor core
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ["exact_attention_63_gb300/csrc/attn_fwd_kernel.cuh", "exact_attention_63_gb300/csrc/attn_fwd_rows.cuh",
                  "exact_attention_63_gb300/csrc/attn_fwd_fp8.cuh", "exact_attention_63_gb300/csrc/attn_fwd_fp8_rows.cuh",
                  "exact_attention_63_gb300/csrc/attn_device.cuh"]


def kernel_source_hash():
    import hashlib

    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_profile_traffic(workload_name):
    """Per-launch DRAM bytes from the committed ncu summary, if it covers this
    workload and was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
        if data.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return data.get(workload_name)
    except (OSError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def mark(self, which):
        setattr(self, which, time.time())

    def summary(self):
        """Median SM clock and throttle reasons over the samples taken inside
        [t_start, t_end] (marked around the timed region); if the region was
        shorter than the sampling interval, the sample nearest to it."""
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        continue
                    rows.append((ts, parts[1:]))
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        t0, t1 = getattr(self, "t_start", rows[0][0]), getattr(self, "t_end", rows[-1][0])
        inside = [r for ts, r in rows if t0 <= ts <= t1]
        window = "timed region"
        if not inside:
            mid = 0.5 * (t0 + t1)
            inside = [min(rows, key=lambda x: abs(x[0] - mid))[1]]
            window = "nearest sample to the timed region"
        rows = inside

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "window": window}


def cpu_oracle_rate(w, budget_s: float, start_chunk: int = 0):
    """Time the fp64 oracle on 128-row chunks of one head shaped like workload
    ``w`` (same Sq, Sk, d, mask and value distribution) for about ``budget_s``
    seconds.  FLOPs are counted per row with the same convention as the GPU
    (4·d per visible key), so causal rows count what they see.
    Returns (TFLOP/s, sample description, cores, seconds, chunks)."""
    import numpy as np

    import oracle
    from exact_attention_63_gb300 import inputs

    small = inputs.Workload(w.name, 1, 1, w.Sq, w.Sk, w.d, w.causal, w.sigma_qk, w.sigma_v, w.seed)
    q, k, v = (oracle.to_f64(t)[0, :, 0, :] for t in inputs.make_inputs(small))
    nch = (w.Sq + 127) // 128
    n, t, flops = 0, 0.0, 0.0
    while n == 0 or t < budget_s:
        c = (start_chunk + 37 * n) % nch
        rows = np.arange(c * 128, min(w.Sq, c * 128 + 128))
        t0 = time.perf_counter()
        oracle.attention_head(q, k, v, w.scale, w.causal, rows=rows)
        t += time.perf_counter() - t0
        vis = np.minimum(w.Sk, rows + 1) if w.causal else np.full(rows.shape, w.Sk)
        flops += 4.0 * w.d * float(vis.sum())
        n += 1
    cores = len(os.sched_getaffinity(0))
    sample = (f"{n} chunks of 128 query rows of one {w.Sq}x{w.Sk} d={w.d}{' causal' if w.causal else ''} head "
              f"(same shape and distribution as the workload), fp64 numpy, {t:.1f} s")
    return flops / t / 1e12, sample, cores, t, n


def host_link_bound(h2d_bytes, d2h_bytes, kernel_ms, flops, dev, stream, reps=5):
    """The roofline of the host-buffer call: one pinned host->device copy of a
    step's upload bytes, one device->host copy of its download bytes (one
    cudaMemcpyAsync each), and the two issued together on two streams, timed
    with CUDA events, best of ``reps``.  With uploads, downloads and the kernel
    fully overlapped, a step takes at least the longest of the single copies,
    the concurrent pair (the link may share its bandwidth between the two
    directions) and the kernel, which bounds the end-to-end throughput."""
    import torch

    up_h = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    up_d = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dn_d = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    dn_h = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    side = torch.cuda.Stream(device=dev)

    def best(fn):
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            t.append(a.elapsed_time(b))
        return min(t)

    def both():
        go, done = torch.cuda.Event(), torch.cuda.Event()
        go.record(stream)
        side.wait_event(go)
        with torch.cuda.stream(stream):
            up_d.copy_(up_h, non_blocking=True)
        with torch.cuda.stream(side):
            dn_h.copy_(dn_d, non_blocking=True)
        done.record(side)
        stream.wait_event(done)

    with torch.cuda.stream(stream):
        t_up = best(lambda: up_d.copy_(up_h, non_blocking=True))
        t_dn = best(lambda: dn_h.copy_(dn_d, non_blocking=True))
    t_both = best(both)
    t_min = max(t_up, t_dn, t_both, kernel_ms)
    return {"link_h2d_gbs": h2d_bytes / (t_up * 1e-3) / 1e9, "link_d2h_gbs": d2h_bytes / (t_dn * 1e-3) / 1e9,
            "link_both_gbs": (h2d_bytes + d2h_bytes) / (t_both * 1e-3) / 1e9,
            "bound_tflops": flops / (t_min * 1e-3) / 1e12,
            "bound": "max(one pinned upload copy, one pinned download copy, the two together, the kernel) per step"}


def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle, on rank 0 only."""
    if rank != 0:
        return
    # Whole run bounded to about two minutes of CPU time.
    budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    chunk = 0
    for _ in range(args.warmup):
        *_, n = cpu_oracle_rate(w, budget, chunk)
        chunk += n
    rates, total_t = [], 0.0
    for _ in range(args.steps):
        r, sample, cores, t, n = cpu_oracle_rate(w, budget, chunk)
        chunk += n
        rates.append(r)
        total_t += t
    value = statistics.mean(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{k_: getattr(w, k_) for k_ in ("B", "H", "Sq", "Sk", "d", "causal")}},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 500 steps of the default workload time about half a second of kernel work
    # (five or more clock samples); longer runs reach the GPU's power cap and
    # the SM clock drops by a few percent (both recorded in the clocks field).
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=4,
                    help="workload index 1-5 (default 4: B8 H32 S4096 d64, the longest non-causal workload)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--poly-mask", type=lambda x: int(x, 0), default=0, help="override the exp2 split (tuning)")
    ap.add_argument("--tau", type=float, default=0.0, help="override the rescale threshold (tuning; 0 = default)")
    ap.add_argument("--diag", action="store_true", help="report the rescale rate of one extra launch")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="grouped-query variant of the workload: K/V heads (H must be a multiple); 0 = H")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (dQ, dK, dV) instead; FLOPs counted as 2.5x the forward's "
                         "(the five products S, dP, dV, dK, dQ), halved when causal")
    ap.add_argument("--deterministic", action="store_true",
                    help="with --backward: the two-pass, bit-reproducible schedule instead of the one-pass default")
    ap.add_argument("--varlen", type=int, default=0,
                    help="packed-sequence variant: this many sequences with a seeded mix of lengths up to the "
                         "workload's S (same H, d, mask); FLOPs counted per sequence")
    ap.add_argument("--fp8", action="store_true",
                    help="the FP8 (E4M3) forward on the workload's E4M3 inputs (head dim 128 workloads)")
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="N > 1: every rank its own batch (weak scaling, default) or one problem's heads split "
                         "across the ranks (strong scaling)")
    ap.add_argument("--causal-align", choices=["top-left", "bottom-right"], default="top-left",
                    help="causal alignment when Sq != Sk (only the square workloads ship, where both agree)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from exact_attention_63_gb300 import inputs

    w = inputs.WORKLOADS[args.config]
    if args.backward and (args.kv_heads or args.varlen or args.causal_align != "top-left"):
        ap.error("--backward takes the plain workloads")
    if args.fp8 and (w.d != 128 or args.backward or args.varlen or args.kv_heads or args.shard != "replicas"
                     or args.causal_align != "top-left"):
        ap.error("--fp8 takes the plain head-dim-128 workloads (--config 2, 3 or 5)")
    if args.shard == "heads" and (args.backward or args.varlen or args.kv_heads):
        ap.error("--shard heads takes the plain forward workloads")
    if args.kv_heads or args.causal_align != "top-left" or args.varlen:
        import dataclasses

        if args.kv_heads and w.H % args.kv_heads:
            ap.error(f"H = {w.H} is not a multiple of --kv-heads {args.kv_heads}")
        tag = (f"_hkv{args.kv_heads}" if args.kv_heads else "") + \
            ("_br" if args.causal_align == "bottom-right" else "") + (f"_varlen{args.varlen}" if args.varlen else "")
        w = dataclasses.replace(w, name=w.name + tag, H_kv=args.kv_heads, causal_align=args.causal_align)
        args.no_e2e = True  # the host-buffer entry point takes dense, unpacked multi-head tensors only
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import torch.distributed as dist

    from exact_attention_63_gb300 import attn
    from exact_attention_63_gb300 import dist as adist

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    attn.lib()  # fails loudly if the library is missing

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    seed = adist.rank_seed(w.seed, rank)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    opts = (attn.make_options(poly_exp2_mask=args.poly_mask, rescale_threshold=args.tau)
            if (args.poly_mask or args.tau) else None)
    stream = torch.cuda.current_stream()
    lens = None
    if args.varlen:
        # Packed sequences: lengths from the seeded mix; FLOPs per sequence.
        lens = inputs.varlen_lengths(args.varlen, w.Sq, seed)
        q, kk, vv, cu_q, cu_k = inputs.make_varlen_inputs(lens, lens, w.H, w.kv_heads, w.d, seed,
                                                          sigma_qk=w.sigma_qk)
        qd, kd, vd, cqd, ckd = (t_.to(dev) for t_ in (q, kk, vv, cu_q, cu_k))
        od = torch.empty_like(qd)
        ld = torch.empty((w.H, qd.shape[0]), dtype=torch.float32, device=dev)
        per_seq = [4.0 * w.H * w.d * n * n for n in lens]
        varlen_flops = sum(f / 2 if w.causal else f for f in per_seq)

        def step():
            attn.attn_fwd_varlen(qd, kd, vd, cqd, ckd, max(lens), causal=w.causal, scale=w.scale, out=od, lse=ld,
                                 options=opts, causal_align=w.causal_align)
    elif args.fp8:
        q8, k8, v8, dq8, dk8, dv8 = inputs.make_fp8_inputs(w, seed=seed)
        qd, kd, vd = q8.to(dev), k8.to(dev), v8.to(dev)
        od = torch.empty(q8.shape, dtype=torch.bfloat16, device=dev)
        ld = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)

        def step():
            attn.attn_fwd_fp8(qd, kd, vd, dq8, dk8, dv8, causal=w.causal, scale=w.scale, out=od, lse=ld)
        args.no_e2e = True
    elif args.shard == "heads":
        # One problem (the workload's own seed on every rank); this rank's
        # contiguous share of its B·H heads, as (batch, head) units.
        units = adist.shard_heads(w.B, w.H, world, rank)
        q, k, v = inputs.make_inputs(w)
        sel = lambda t: torch.stack([t[b_, :, h_, :] for b_, h_ in units], dim=1).unsqueeze(0).contiguous()
        q, k, v = sel(q), sel(k), sel(v)  # [1, S, n_units, d]
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        od = torch.empty_like(qd)
        ld = torch.empty((1, len(units), w.Sq), dtype=torch.float32, device=dev)
        shard_flops = w.flops * len(units) / (w.B * w.H)

        def step():
            attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld, options=opts,
                          causal_align=w.causal_align)
        args.no_e2e = True
    else:
        q, k, v = inputs.make_inputs(w, seed=seed)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        od = torch.empty_like(qd)
        ld = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)

        def step():
            attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld, options=opts,
                          causal_align=w.causal_align)

        if args.backward:
            step()  # O and LSE for the backward
            gen = torch.Generator().manual_seed(seed + 7)
            gd = torch.randn(q.shape, generator=gen).to(torch.bfloat16).to(dev)
            dqd, dkd, dvd = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
            wsd = torch.empty(attn.lib().attn_bwd_workspace_size(w.B, w.H, w.Sq), dtype=torch.uint8, device=dev)

            def step():
                attn.attn_bwd(qd, kd, vd, od, ld, gd, causal=w.causal, scale=w.scale, dq=dqd, dk=dkd, dv=dvd,
                              workspace=wsd, deterministic=args.deterministic)
            args.no_e2e = True

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        clk.mark("t_start")
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
        clk.mark("t_end")
    if attn.get_status() != 0:
        raise RuntimeError("kernel reported a device-side error")
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = adist.max_over_ranks(sum(times_ms), device=dev)
    ms_per_step = total_ms / args.steps
    flops = varlen_flops if lens is not None else w.flops
    if args.backward:
        flops *= 2.5
    if args.shard == "heads":
        # strong scaling: the whole problem's FLOPs over the slowest rank's time
        value = flops * args.steps / (total_ms * 1e-3) / 1e12
        achieved = shard_flops / (statistics.mean(times_ms) * 1e-3) / 1e12
    else:
        value = flops * world * args.steps / (total_ms * 1e-3) / 1e12
        achieved = flops / (statistics.mean(times_ms) * 1e-3) / 1e12

    # ---- end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t_.pin_memory() for t_ in (q, k, v))
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32).pin_memory()
        ws = torch.empty(attn.workspace_size(w.B, w.H, w.Sq, w.Sk, w.d), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            attn.attn_fwd_host(qh, kh, vh, oh, lh, w.causal, w.scale, ws)
        barrier()
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            e_s[i].record(stream)
            attn.attn_fwd_host(qh, kh, vh, oh, lh, w.causal, w.scale, ws)
            e_e[i].record(stream)
        barrier()
        e_ms = adist.max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)), device=dev)
        h2d = int(3 * q.numel() * 2)
        d2h = int(q.numel() * 2 + w.B * w.H * w.Sq * 4)
        e2e = {"value": flops * world * args.steps / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
               **host_link_bound(h2d, d2h, statistics.mean(times_ms), flops, dev, stream)}
        e2e["frac_of_bound"] = e2e["value"] / world / e2e["bound_tflops"]
        del ws

    diag = None
    if args.diag and lens is None:
        cnt = torch.zeros(2, dtype=torch.int64, device=dev)
        attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld,
                      options=attn.make_options(poly_exp2_mask=args.poly_mask, rescale_threshold=args.tau,
                                                counters=cnt))
        torch.cuda.synchronize()
        c = cnt.cpu().tolist()
        # d = 64 runs the full-row kernel (one running maximum per row); the
        # d = 128 kernel keeps one per 64-key half of each row.
        parts = 1 if w.d == 64 else 2
        diag = {"rescales": c[0], "row_block_updates": c[1], "tau": args.tau or 32.0,
                "rescale_unit": "row x 128-key block" if parts == 1 else "row x 64-key half block",
                "rescales_per_unit": c[0] / max(1, parts * c[1])}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"]) * (2.0 if args.fp8 else 1.0)
    # (forward kernels only: the backward's sources are not in the recorded hash)
    traffic = None if args.backward else load_profile_traffic(w.name + ("_fp8" if args.fp8 else ""))
    cpu = None
    if args.cpu_budget > 0 and world == 1:  # the CPU baseline is taken at N = 1 only
        rate, sample, cores, _, _ = cpu_oracle_rate(w, args.cpu_budget)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "strong" if args.shard == "heads" else "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name + ("_backward" if args.backward else "") + ("_two_pass" if args.deterministic else "") + ("_fp8" if args.fp8 else ""), "B": w.B, "H": w.H, "H_kv": w.kv_heads, "Sq": w.Sq, "Sk": w.Sk, "d": w.d,
                   "causal": w.causal, "causal_align": w.causal_align, "sigma_qk": w.sigma_qk, "seed": w.seed,
                   **({"varlen_lengths": lens} if lens is not None else {}),
                   "l2": "flushed between timed steps (256 MiB write)",
                   "parallelism": (f"heads{world}" if args.shard == "heads" else f"replicas{world}")
                   if world > 1 else "single"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} bf16_tflops (burst cuBLAS)"
                     + (" x 2 (nominal FP8/BF16 tensor ratio)" if args.fp8 else ""),
                     **({"frac_of_nominal_fp8_4500": achieved / (2 * CONTRACT_PEAK_TFLOPS)} if args.fp8 else
                        {"frac_of_contract_2250": achieved / CONTRACT_PEAK_TFLOPS})},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (3 if args.backward else 1),
        "clocks": clk.summary(),
    }
    if diag is not None:
        line["diag"] = diag
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
