"""Benchmark: one step = one forward + one backward pass of exact attention over
one batch of synthetic bf16 input (every stage of the path: forward kernel,
backward pre / main / post kernels), on the mid-length workload
B=4, H=16, N=8192, d=128, non-causal (32k tokens, hidden 2048).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. ``value`` is whole-job attention TFLOP/s (forward
4*N^2*d per head plus backward 2.5x that), inputs resident in device memory;
``e2e`` is the same metric through the public binding with host buffers, the
host->device copies of q, k, v, dO and the device->host copies of o, lse, dq,
dk, dv of every step inside the timed region (copies overlapped with the
neighbouring steps' compute; the serial figure is reported beside it). ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "mid"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    help="named workload (tiny, short, short_causal, mid, mid_causal, long, varlen_gqa)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size (small cases for profiling)")
    ap.add_argument("--causal", action="store_true", help="causal variant of the workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fwd-variant", default="one_cta", choices=["one_cta", "pair"],
                    help="forward kernel at d = 128 (the CTA-pair kernel is kept for measurement)")
    ap.add_argument("--bwd-variant", default="one_cta", choices=["one_cta", "pair"],
                    help="backward main kernel at d = 128 (the CTA-pair kernel is kept for measurement)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward with ordered (bit-reproducible) dQ accumulation")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """Largest value of x over all ranks (the slowest rank decides the time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(step_flops_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Weak scaling: every rank runs its own replica of the workload; the job's
    throughput is all ranks' work over the slowest rank's time (TFLOP/s)."""
    return world * step_flops_per_rank * steps / (max_ms * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


SUSTAINED_AFTER_S = 2.0


def roof_peak(timed_s: float, burst: float, sustained: float):
    """Tensor peak a kernel's fraction is taken against: the burst bf16 rate
    while the timed region is short (the GPU has not yet reached its power cap),
    the sustained rate once it lasts seconds."""
    if timed_s >= SUSTAINED_AFTER_S:
        return "bf16_tflops_sustained", sustained
    return "bf16_tflops", burst


class ClockSampler:
    """Samples nvidia-smi every 50 ms; only the samples after mark() (taken
    while the timed region runs) are summarised."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self):
        self.first = len(self.lines)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[getattr(self, "first", 0):]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "exact_attention_15_gb300", "csrc", rec["source"])
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    if sha != rec.get("source_sha256_16"):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ shared description of the step

def step_metric(fwd_only):
    return ("attention fwd TFLOP/s (bf16, 1xGB300)" if fwd_only
            else "attention fwd+bwd TFLOP/s (bf16, 1xGB300)")


def step_config(w, B, N, H, H_kv, d, d_v, fwd_only, world, bwd_variant, l2_note, fwd_variant="one_cta"):
    return {"workload": f"{w.name}: " + (w.note or f"B{B} H{H} N{N} d{d}") +
                        (", fwd only" if fwd_only else ", fwd+bwd"),
            "global_batch": B * world, "seq_len": N, "heads": H, "kv_heads": H_kv,
            "head_dim": d, "head_dim_v": d_v, "fwd_variant": fwd_variant, "bwd_variant": bwd_variant,
            "parallelism": f"replicas x{world}", "l2": l2_note}


# ------------------------------------------------------------------ reference arm (oracle)

def workload_name(args, W):
    """The named workload both arms run (``--workload``, ``--causal``)."""
    name = args.workload
    if args.causal and not name.endswith("_causal") and name + "_causal" in W.WORKLOADS:
        name += "_causal"
    return name


def oracle_unit_shapes(w, inp=None):
    """Units of oracle work of a workload: one (batch entry or packed sequence,
    query head) each, as (query rows, key rows). Packed workloads take their
    lengths from the generated inputs."""
    if w.varlen is None:
        B = w.B if inp is None else inp.B
        return [(w.N, w.N)] * (B * w.H_q)
    return [(int(L), int(L)) for L in inp.seqlens() for _ in range(w.H_q)]


def oracle_step(oracle, q, k, v, do, w, fwd_only):
    if fwd_only:
        oracle.head_forward(q, k, v, w.scale, w.causal)
    else:
        oracle.head_backward(q, k, v, do, w.scale, w.causal)


def unit_flops(W, w, L_q, L_k, fwd_only):
    d_v = w.d_v or w.d
    f = W.fwd_flops(1, 1, L_q, L_k, w.d, w.causal, d_v=d_v)
    return f if fwd_only else 3.5 * f


def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np
    import oracle
    from exact_attention_15_gb300 import workloads as W

    w = W.WORKLOADS[workload_name(args, W)]
    fwd_only = False
    # bounded sample: one (batch entry or sequence, head) unit per step, every
    # query row; packed workloads take a unit of the median sequence length
    if w.varlen is None:
        L = w.N
    else:
        L = int(np.median(W.generate(w.name, parts=("q",)).seqlens()))
    inp = W.custom(1, 1, 1, L, L, w.d, w.scale, w.causal, seed=w.seed, d_v=w.d_v)
    f64 = W.bf16_bits_to_f64
    q, k, v, do = (f64(x[0, :, 0, :]) for x in (inp.q, inp.k, inp.v, inp.do))
    flops = unit_flops(W, w, L, L, fwd_only)
    for _ in range(args.warmup):
        oracle_step(oracle, q, k, v, do, w, fwd_only)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(oracle, q, k, v, do, w, fwd_only)
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = flops / sec / 1e12
    cores = os.cpu_count()
    config = step_config(w, w.B, w.N, w.H_q, w.H_kv, w.d, w.d_v or w.d, fwd_only, world,
                         args.bwd_variant, "host memory (oracle)", args.fwd_variant)
    unit = "(sequence, head) unit of median length" if w.varlen else "(batch, head) pair"
    config["step_sample"] = f"1 {unit} of the workload per step, all {L} query rows"
    passes = "fwd" if fwd_only else "fwd+bwd"
    line = {
        "impl": "reference", "metric": step_metric(fwd_only), "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"one {unit} of the workload per step ({L} query rows, "
                                   f"d={w.d}), {passes}, numpy fp64 BLAS on all host cores"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_sample(name, inp, fwd_only, min_seconds=10.0, max_units=32):
    """The oracle as it stands on a bounded sample of the workload's own inputs:
    whole (batch entry or sequence, head) units in a seeded order, forward (and
    backward unless the step is forward only), until at least `min_seconds` of
    host time; the full-workload time is extrapolated from the measured rate."""
    import numpy as np
    import oracle
    from exact_attention_15_gb300 import workloads as W
    w = W.WORKLOADS[name]
    f64 = W.bf16_bits_to_f64
    g = inp.H_q // inp.H_kv
    if inp.cu_seqlens is None:
        units = [(b, h, None) for b in range(inp.B) for h in range(inp.H_q)]
    else:
        cu = inp.cu_seqlens
        units = [(s, h, (int(cu[s]), int(cu[s + 1]))) for s in range(len(cu) - 1)
                 for h in range(inp.H_q)]
    order = np.random.default_rng(w.seed).permutation(len(units))

    def slices(u):
        b, h, span = u
        if span is None:
            return (f64(inp.q[b, :, h, :]), f64(inp.k[b, :, h // g, :]), f64(inp.v[b, :, h // g, :]),
                    f64(inp.do[b, :, h, :]))
        a, e = span
        return (f64(inp.q[a:e, h, :]), f64(inp.k[a:e, h // g, :]), f64(inp.v[a:e, h // g, :]),
                f64(inp.do[a:e, h, :]))

    q0, k0, v0, do0 = slices(units[order[0]])
    oracle_step(oracle, q0[:512], k0, v0, do0[:512], w, fwd_only)  # warm BLAS
    t0 = time.perf_counter()
    n, flops = 0, 0.0
    for idx in order[:max_units]:
        q, k, v, do = slices(units[idx])
        oracle_step(oracle, q, k, v, do, w, fwd_only)
        flops += unit_flops(W, w, q.shape[0], k.shape[0], fwd_only)
        n += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    sec = time.perf_counter() - t0
    rate = flops / sec
    total = sum(unit_flops(W, w, a, b, fwd_only) for a, b in oracle_unit_shapes(w, inp))
    kind = "(sequence, head) units" if inp.cu_seqlens is not None else "(batch, head) pairs"
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} seeded {kind} of the workload (d={w.d}), "
                      f"{'fwd' if fwd_only else 'fwd+bwd'} in {sec:.1f} s, numpy fp64 BLAS on all "
                      f"host cores",
            "seconds_per_unit": sec / n,
            "extrapolated_step_s": total / rate,
            "extrapolated_note": f"extrapolated: the whole workload ({len(units)} units) at the "
                                 f"measured rate, not measured"}


# ------------------------------------------------------------------ our arm

def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import numpy as np
    import torch
    from exact_attention_15_gb300 import binding, workloads as W

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    binding.load()
    if args.bwd_variant == "pair":
        binding.attn_set_bwd_variant(binding.BWD_CTA_PAIR)
    if args.fwd_variant == "pair":
        binding.attn_set_fwd_variant(binding.FWD_CTA_PAIR)

    name = workload_name(args, W)
    w = W.WORKLOADS[name]
    if args.batch is not None and w.varlen is None:
        inp = W.custom(args.batch, w.H_q, w.H_kv, w.N, w.N, w.d, w.scale, w.causal, seed=w.seed,
                       boost_frac=w.boost_frac, boost=w.boost, d_v=w.d_v)
        w = W.Workload(w.name, args.batch, w.H_q, w.H_kv, w.N, w.d, w.scale, w.causal, w.seed,
                       d_v=w.d_v)
    else:
        inp = W.generate(w.name)
    fwd_only = False  # every workload's step is one forward and one backward pass
    dev = lambda bits: torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    q, k, v, do = dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.do)
    varlen = inp.cu_seqlens is not None
    B, H, H_kv, d, d_v = inp.B, inp.H_q, inp.H_kv, inp.d, inp.d_v
    N = inp.N_q
    cu = torch.from_numpy(inp.cu_seqlens).cuda() if varlen else None
    cu_ptr = cu.data_ptr() if varlen else None
    o = torch.empty(q.shape[:-1] + (d_v,), dtype=q.dtype, device="cuda")
    lse = torch.empty((H, N) if varlen else (B, H, N), dtype=torch.float32, device="cuda")
    det = 1 if args.deterministic else 0
    if fwd_only:
        dq = dk = dv = None
        ws_bytes, ws = 0, None
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws_bytes = binding.attn_bwd_dims_workspace_bytes(B, H, H_kv, N, N, d, d_v, varlen, det)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def step():
        st = binding.attn_fwd_dims(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, H_kv, N, N, d, d_v, w.causal, cu_ptr,
                                   w.scale, sp)
        assert st == 0, st
        if fwd_only:
            return
        st = binding.attn_bwd_dims(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, H_kv, N, N, d, d_v, w.causal, cu_ptr,
                                   w.scale, det, ws.data_ptr(), ws_bytes, sp)
        assert st == 0, st

    fwd_flops = W.fwd_flops(B, H, N, N, d, w.causal, seqlens=inp.seqlens() if varlen else None,
                            d_v=d_v)
    step_flops = fwd_flops * (1.0 if fwd_only else 3.5)  # forward + 2.5x backward

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert binding.attn_check(sp) == 0

    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    binding.attn_profile_enable(True)
    binding.attn_profile_read()
    sampler.start()
    time.sleep(0.3)
    sampler.mark()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    binding.attn_profile_enable(False)
    recs = binding.attn_profile_read()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world)
    if world > 1:
        torch.distributed.barrier()
    assert binding.attn_check(sp) == 0
    ms_step = ms_total / args.steps
    value = whole_job_value(step_flops, args.steps, world, ms_total)

    per_kernel = {}
    for kname, ms in recs:
        per_kernel.setdefault(kname, []).append(ms)
    if "attn_bwd_main_kernel_pass2" in per_kernel:
        # query/key head dimension 192: the backward main kernel runs in two
        # passes; the roofline takes them together (one launch of each per step)
        p1, p2 = per_kernel["attn_bwd_main_kernel"], per_kernel["attn_bwd_main_kernel_pass2"]
        per_kernel["attn_bwd_main_kernel (both passes)"] = [a + b for a, b in zip(p1, p2)]
    kt = {n: {"launches": len(v_), "avg_ms": sum(v_) / len(v_), "total_ms": sum(v_)} for n, v_ in per_kernel.items()}
    tot = sum(x["total_ms"] for n, x in kt.items() if not n.endswith("(both passes)")) or 1.0
    for x in kt.values():
        x["share"] = x["total_ms"] / tot
    peaks, peak_src = measured_peaks()
    sustained = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    burst = float(peaks.get("bf16_tflops"))
    timed_s = ms_total * 1e-3
    peak_kind, peak = roof_peak(timed_s, burst, sustained)

    def roof(kernel, flops_per_launch):
        if kernel not in kt:
            return None
        ach = flops_per_launch / (kt[kernel]["avg_ms"] * 1e-3) / 1e12
        tr = traffic_for(kernel, w.name if args.batch is None else None)
        return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": tr, "kernel": kernel,
                "peak_kind": f"{peak_kind} ({peak_src}; timed region {timed_s:.2f} s)",
                "timed_region_s": timed_s,
                "frac_of_burst": ach / burst, "frac_of_sustained": ach / sustained,
                "frac_of_2250": ach / 2250.0}

    dominant = max(kt, key=lambda n: kt[n]["total_ms"]) if kt else None
    flops_of = {"attn_fwd_kernel": fwd_flops, "attn_fwd_pair_kernel": fwd_flops,
                "attn_bwd_main_kernel": 2.5 * fwd_flops,
                "attn_bwd_main_kernel (both passes)": 2.5 * fwd_flops}
    if "attn_bwd_main_kernel_pass2" in kt:
        flops_of.pop("attn_bwd_main_kernel")
    fwd_kernel = "attn_fwd_pair_kernel" if args.fwd_variant == "pair" else "attn_fwd_kernel"
    roofline = roof(dominant, flops_of.get(dominant, 0.0)) if dominant in flops_of else None
    roofline_fwd = roof(fwd_kernel, fwd_flops)

    # end to end through the public binding with host buffers: every step copies
    # its inputs (q, k, v, dO) from pinned host memory and its results (o, lse,
    # dq, dk, dv) back. Timed two ways: serial (copy in, compute, copy out on one
    # stream) and pipelined (three device buffer sets: step s+1's inputs and step
    # s-1's results move while step s computes, on two copy streams at once or on
    # one; e2e reports the faster of the two copy schedules, both are listed).
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "k", "v") if fwd_only else ("q", "k", "v", "do")
        names_out = ("o", "lse") if fwd_only else ("o", "lse", "dq", "dk", "dv")
        host_in = dict(q=inp.q, k=inp.k, v=inp.v, do=inp.do)
        hq = [torch.from_numpy(host_in[n].view(np.int16)).view(torch.bfloat16).pin_memory()
              for n in names_in]
        sets = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)]
        sets[0] = {n: t for n, t in sets[0].items() if t is not None}
        n_sets = 3
        for _ in range(n_sets - 1):
            sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
        hout = [[torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype).pin_memory() for n in names_out]
                for _ in range(n_sets)]
        h2d = sum(t.numel() * t.element_size() for t in hq)
        d2h = sum(t.numel() * t.element_size() for t in hout[0])

        def run_step(st_, sp_):
            r = binding.attn_fwd_dims(st_["q"].data_ptr(), st_["k"].data_ptr(), st_["v"].data_ptr(),
                                      st_["o"].data_ptr(), st_["lse"].data_ptr(), B, H, H_kv, N, N,
                                      d, d_v, w.causal, cu_ptr, w.scale, sp_)
            assert r == 0, r
            if fwd_only:
                return
            r = binding.attn_bwd_dims(st_["q"].data_ptr(), st_["k"].data_ptr(), st_["v"].data_ptr(),
                                      st_["o"].data_ptr(), st_["lse"].data_ptr(),
                                      st_["do"].data_ptr(), st_["dq"].data_ptr(),
                                      st_["dk"].data_ptr(), st_["dv"].data_ptr(), B, H, H_kv, N, N,
                                      d, d_v, w.causal, cu_ptr, w.scale, det, ws.data_ptr(),
                                      ws_bytes, sp_)
            assert r == 0, r

        def copy_in(st_):
            for hsrc, n in zip(hq, names_in):
                st_[n].copy_(hsrc, non_blocking=True)

        def copy_out(st_, hset):
            for n, hdst in zip(names_out, hset):
                hdst.copy_(st_[n], non_blocking=True)

        def serial_step():
            copy_in(sets[0])
            run_step(sets[0], sp)
            copy_out(sets[0], hout[0])

        s_in, s_out0 = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(n_sets)]
        done = [torch.cuda.Event() for _ in range(n_sets)]
        freed = [torch.cuda.Event() for _ in range(n_sets)]

        def pipelined(n_steps, one_stream):
            # step i's inputs are copied in during step i-1; its results are
            # copied out during step i+1 (on s_in as well with one_stream)
            s_o = s_in if one_stream else s_out0

            def enqueue_in(i):
                b_ = i % n_sets
                with torch.cuda.stream(s_in):
                    if i >= n_sets:
                        s_in.wait_event(freed[b_])  # that set's earlier results have left it
                    copy_in(sets[b_])
                    in_ready[b_].record(s_in)

            enqueue_in(0)
            for i in range(n_steps):
                b_ = i % n_sets
                if i + 1 < n_steps:
                    enqueue_in(i + 1)
                stream.wait_event(in_ready[b_])
                run_step(sets[b_], sp)
                done[b_].record(stream)
                with torch.cuda.stream(s_o):
                    s_o.wait_event(done[b_])
                    copy_out(sets[b_], hout[b_])
                    freed[b_].record(s_o)
            stream.wait_stream(s_in)
            stream.wait_stream(s_o)

        for _ in range(2):
            serial_step()
        pipelined(n_sets, False)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            serial_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms_serial = max_over_ranks(ev0.elapsed_time(ev1), world)
        # Two copy schedules: outgoing and incoming copies on separate streams
        # (both directions at once), or on one stream (one direction at a time).
        # Which is faster depends on the host link; both are timed and reported.
        ms_sched = {}
        for sched in ("both_directions", "one_direction"):
            one = sched == "one_direction"
            pipelined(n_sets, one)
            torch.cuda.synchronize()
            s_in.wait_stream(stream)
            ev0.record(s_in)
            pipelined(args.steps, one)
            ev1.record(stream)
            torch.cuda.synchronize()
            ms_sched[sched] = max_over_ranks(ev0.elapsed_time(ev1), world)
        best = min(ms_sched, key=ms_sched.get)
        ms_pipe = ms_sched[best]
        assert binding.attn_check(sp) == 0
        e2e = {"value": whole_job_value(step_flops, args.steps, world, ms_pipe), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms_pipe / args.steps,
               "mode": "pipelined: three device buffer sets, copies on their own streams; "
                       f"faster copy schedule: {best}",
               "ms_per_step_by_schedule": {k: v / args.steps for k, v in ms_sched.items()},
               "serial": {"value": whole_job_value(step_flops, args.steps, world, ms_serial),
                          "ms_per_step": ms_serial / args.steps}}

    if rank == 0:
        cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline_sample(w.name, inp, fwd_only)
        fwd_ms = kt.get(fwd_kernel, {}).get("avg_ms")
        line = {
            "metric": step_metric(fwd_only), "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": step_config(w, B, N, H, H_kv, d, d_v, fwd_only, world, args.bwd_variant,
                                  f"inputs larger than L2 (q, k, v, o, dO: {q.numel() * 2 / 2**20:.0f} MiB each)"
                                  if q.numel() * 2 * 5 > 129e6 else "inputs smaller than L2 (L2 not flushed)",
                                  fwd_variant=args.fwd_variant),
            "deterministic_bwd": bool(det),
            "fwd_tflops": (fwd_flops / (fwd_ms * 1e-3) / 1e12) if fwd_ms else None,
            "kernels": kt,
            "roofline": roofline,
            "roofline_fwd": roofline_fwd,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": sum(x["launches"] for x in kt.values()),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
