"""Benchmark of the smoothed INT8/FP8 quantized attention forward on GB300.

One step = the whole hot path over one batch: the quantisation prologue
(K smoothing, INT8 Q/K, FP8 V) followed by the fused attention kernel, for
the workload B=2, H=24, L=4096, D=128, fp16, HND, non-causal (the shape of the
pages' RTX 5070 measurement).  Inputs are seeded synthetic tensors already
resident in HBM; L2 is flushed (256 MiB write) between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload NAME]

Prints one JSON line.  `--impl reference` times the plain CPU oracle (the
reference arm) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_attention_smooth_gb300 import workloads as wl  # noqa: E402

METRIC = "attention TOPS (4*B*H*Lq*Lk*D / device time)"
DEFAULT_WORKLOAD = "b2_h24_l4096_d128"
L2_FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) per attention-kernel launch on the default
# workload, from the ncu capture of the attention kernel (None where no
# capture of the current kernel exists).
ATTN_NCU_DRAM_BYTES = {"b2_h24_l4096_d128": 126.744320e6 + 63.198208e6}
# the same for the FP16-PV variant's attention kernel (fp16 V and P~)
ATTN16_NCU_DRAM_BYTES = {"b2_h24_l4096_d128": 152.014592e6 + 63.843584e6}
# (query row, key) pairs of attention in the oracle's bounded sample (one
# head of the 4096 x 4096 workload; a whole small workload)
ORACLE_PAIR_BUDGET = 4096 * 4096
# flops of one M=128 N=128 tcgen05 MMA of each kind (sage_debug_tc_rate)
TC_FLOP = {0: 2.0 * 128 * 128 * 16, 1: 2.0 * 128 * 128 * 32}


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_ops(w: wl.Workload, dim=None) -> float:
    return w.ops(dim=dim)


def prologue_bytes(w: wl.Workload, v_bytes: int = 1) -> float:
    """Algorithmic HBM bytes of the prologue: read q, k, v (2 B each); write
    the fp16 code copies of Q and K (2 B each) and V (e4m3: 1 B, or fp16 for
    the FP16-PV variant: 2 B) per padded element; the second pass over K and
    V is an L2 re-read and counts 0."""
    Dp = 64 if w.D <= 64 else 128
    nq = nk = 0
    for lq, lk in w.seg_lengths():
        nq += lq
        nk += lk
    read = 2 * w.D * (nq * w.Hq + 2 * nk * w.Hkv)
    write = Dp * (2 * nq * w.Hq + (2 + v_bytes) * nk * w.Hkv)
    scales = 4 * (nq * w.Hq + nk * w.Hkv // 128 + 2 * w.Hkv * Dp * w.nseg)
    return float(read + write + scales)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- GPU arm
def count_launches(torch, fn) -> int:
    """Kernels of this library launched by one call of fn (the library's own
    host-side launch counter)."""
    from quantized_attention_smooth_gb300 import sage
    before = sage.launch_count()
    fn()
    torch.cuda.synchronize()
    return sage.launch_count() - before


def to_device(torch, bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == wl.F16 else torch.bfloat16)


def run_gpu(args, w: wl.Workload, rank: int, world: int):
    import torch
    import torch.distributed as dist
    from quantized_attention_smooth_gb300 import sage

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(w)
    host = {k: to_device(torch, inp[k], w.dtype).pin_memory() for k in ("q", "k", "v")}
    d = {k: host[k].to(dev) for k in host}
    if w.varlen:
        d["cu_q"] = torch.from_numpy(inp["cu_q"]).to(dev)
        d["cu_k"] = torch.from_numpy(inp["cu_k"]).to(dev)
        nbytes = sage.workspace_bytes_varlen(w.nseg, sum(w.seqlens_q), sum(w.seqlens_k),
                                             w.Hq, w.Hkv, w.D)
    else:
        nbytes = sage.workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D)
    ws = sage.alloc_workspace(nbytes, dev)
    out = torch.empty(d["q"].shape, dtype=torch.float32, device=dev)
    out_host = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    scale = wl.default_sm_scale(w)

    pv16 = args.variant == "pv16"

    def fwd():
        if w.varlen:
            sage.attn_fwd_varlen(d["q"], d["k"], d["v"], out, d["cu_q"], d["cu_k"],
                                 max(w.seqlens_q), max(w.seqlens_k), w.causal, scale, ws=ws)
        elif pv16:
            sage.attn_fwd_pv16(d["q"], d["k"], d["v"], out, w.layout, w.causal, scale, ws=ws)
        else:
            sage.attn_fwd(d["q"], d["k"], d["v"], out, w.layout, w.causal, scale, ws=ws)

    def prologue():
        if pv16:
            return sage.quant_prologue_pv16(d["q"], d["k"], d["v"], w.layout, ws=ws)
        if w.varlen:
            return sage.quant_prologue_varlen(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"],
                                              max(w.seqlens_q), max(w.seqlens_k), ws=ws)
        return sage.quant_prologue(d["q"], d["k"], d["v"], w.layout, ws=ws)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def step():
        """One step through the two-call API (the same kernels as fwd()), with
        events around the prologue and around the attention kernel."""
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        qt = prologue()
        b.record(stream)
        sage.attn_quantized(qt, out, w.layout, w.causal, scale)
        c.record(stream)
        return a, b, c

    for _ in range(args.warmup):
        fwd()
        flush.zero_()
        step()
        flush.zero_()
    torch.cuda.synchronize()
    assert sage.device_status(ws) == sage.OK, sage.last_error()
    launches_per_step = count_launches(torch, fwd)

    # ---- timed region: K steps (prologue + attention), device events
    clocks = ClockSampler(dev.index)
    clocks.start()
    t_end = time.perf_counter() + 0.4          # keep the GPU busy while the sampler starts
    while time.perf_counter() < t_end:
        fwd()
        flush.zero_()
        torch.cuda.synchronize()
    barrier()
    ev = []
    launches0 = sage.launch_count()
    for i in range(args.steps):
        flush.zero_()                          # L2 flush between timed steps
        ev.append(step())
    barrier()
    launches = sage.launch_count() - launches0
    clock_info = clocks.stop()
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    total_ms = sum(step_ms)
    pro_ms = statistics.mean(a.elapsed_time(b) for a, b, c in ev)
    att_ms = statistics.mean(b.elapsed_time(c) for a, b, c in ev)
    assert sage.device_status(ws) == sage.OK, sage.last_error()

    # ---- end to end: host buffers, copies inside the timed region, through
    # the library's host-buffer calls, which pipeline chunk copies with
    # compute (the FP16-PV variant has no packed-sequence call: there the
    # step copies in, computes and copies back).
    host_call = not (w.varlen and pv16)
    cu_host = {}
    if host_call and w.varlen:
        cu_host = {k: torch.from_numpy(inp[k]) for k in ("cu_q", "cu_k")}
        ws_host = sage.alloc_workspace(sage.workspace_bytes_varlen_host(
            w.nseg, sum(w.seqlens_q), sum(w.seqlens_k), w.Hq, w.Hkv, w.D), dev)
    elif host_call:
        ws_host = sage.alloc_workspace(sage.workspace_bytes_host(
            w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D), dev)
    e2e_ev = []
    n_e2e = max(5, min(args.steps, 50))
    for i in range(max(3, args.warmup) + n_e2e):      # the first ones are warm-up
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if host_call and w.varlen:
            sage.attn_fwd_varlen_host(host["q"], host["k"], host["v"], out_host,
                                      cu_host["cu_q"], cu_host["cu_k"], max(w.seqlens_q),
                                      max(w.seqlens_k), w.causal, scale, ws=ws_host,
                                      stream=stream)
        elif host_call:
            sage.attn_fwd_host(host["q"], host["k"], host["v"], out_host, w.layout, w.causal,
                               scale, ws=ws_host, stream=stream, pv16=pv16)
        else:
            for k in ("q", "k", "v"):
                d[k].copy_(host[k], non_blocking=True)
            fwd()
            out_host.copy_(out, non_blocking=True)
        b.record(stream)
        e2e_ev.append((a, b))
    torch.cuda.synchronize()
    # query head 0 of segment 0 of the last output, for the parity sample
    out_rows = np.array(wl.out_segment(w, out_host.numpy(), 0, inp.get("cu_q"))[0])
    e2e_ev = e2e_ev[-n_e2e:]
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_ev)
    h2d = (sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v")) +
           sum(t.numel() * 4 for t in cu_host.values()))
    d2h = out_host.numel() * 4

    # the tensor pipe's rate for the kernel's two MMA kinds, measured now, at
    # the clock the GPU runs under this load (sage_debug_tc_rate)
    tc = tensor_rates(torch, sage, stream, dev)

    Dp = 64 if w.D <= 64 else 128
    r = dict(tc=tc, total_ms=total_ms, step_ms=step_ms, pro_ms=pro_ms, att_ms=att_ms,
             launches_per_step=launches_per_step, launches=launches,
             e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, ops=workload_ops(w), out_rows=out_rows,
             e2e_api=(("sage_attn_fwd_varlen_host" if w.varlen else
                       "sage_attn_fwd_host_pv16" if pv16 else "sage_attn_fwd_host") +
                      " (chunks of kv heads, copies pipelined with compute)"
                      if host_call else "copies, then the one-call entry point, then a copy back"),
             ops_padded=workload_ops(w, Dp),
             ops_effective=w.ops(causal_effective=True),
             ops_padded_effective=w.ops(dim=Dp, causal_effective=True),
             clocks=clock_info)
    return reduce_over_ranks(r, world, dev)


def tensor_rates(torch, sage, stream, dev, n_mma: int = 1 << 15, reps: int = 5):
    """TFLOP/s of back-to-back M=128 N=128 tcgen05 MMAs on every SM, per kind
    (0: fp16 K=16, 1: e4m3 K=32): best of `reps` event-timed launches."""
    status = torch.zeros(64, dtype=torch.int32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for kind in (0, 1):
        sage.debug_tc_rate(kind, 1024, status, stream)          # warm-up
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sage.debug_tc_rate(kind, n_mma, status, stream)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        assert sage.device_status(status) == sage.OK, sage.last_error()
        out[kind] = TC_FLOP[kind] * n_mma * sms / (best * 1e-3) / 1e12
    return out


# ---------------------------------------------------------- rank aggregation
TIME_KEYS = ("total_ms", "pro_ms", "att_ms", "e2e_ms")


def reduce_over_ranks(r: dict, world: int, device=None) -> dict:
    """Max over ranks of every time-like figure: the job's step ends when its
    slowest rank's does.  Rank counts and op totals stay per rank (every rank
    runs the same workload on its own GPU, replicas with no collective in the
    data path).  Called by every rank; one all-reduce."""
    if world <= 1:
        return r
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(r[k]) for k in TIME_KEYS], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    out = dict(r)
    out.update(zip(TIME_KEYS, t.tolist()))
    return out


def job_figures(r: dict, world: int, steps: int) -> dict:
    """Whole-job throughputs in TOPS: the ops all `world` ranks processed
    divided by the max-over-ranks time.  `value` counts 4*Lq*Lk*D literally;
    the padded figures use the head dimension the tensor cores see, and the
    effective ones drop the causally masked half."""
    def tops(ops, ms):
        return ops * world / (ms * 1e-3) / 1e12
    step_ms = r["total_ms"] / steps
    return {
        "value": tops(r["ops"], step_ms),
        "value_padded_d": tops(r["ops_padded"], step_ms),
        "value_causal_effective": tops(r["ops_effective"], step_ms),
        "e2e": tops(r["ops"], r["e2e_ms"]),
        "attention_tflops_padded": r["ops_padded"] / (r["att_ms"] * 1e-3) / 1e12,
        "attention_tflops_padded_effective":
            r["ops_padded_effective"] / (r["att_ms"] * 1e-3) / 1e12,
    }


# ---------------------------------------------------------- CPU oracle arm
def oracle_sample_plan(w: wl.Workload, budget: int = ORACLE_PAIR_BUDGET):
    """The oracle's bounded sample of a workload, the same in both arms:
    segment 0, query rows [0, rows) of query heads [0, heads), with
    rows * Lk <= budget (row, key) pairs per head and as many heads as fit
    the budget (whole groups of the heads that share a kv head).  Returns
    (heads, kv_heads, rows)."""
    lq, lk = w.seg_lengths()[0]
    rows = max(1, min(lq, budget // max(lk, 1)))
    group = w.Hq // w.Hkv
    fit = max(1, budget // max(rows * max(lk, 1), 1))
    heads = min(w.Hq, fit)
    if heads >= group:
        heads = heads // group * group
        return heads, heads // group, rows
    return 1, 1, rows            # query head 0 alone reads kv head 0


def oracle_sample(w: wl.Workload, inp: dict, pv16: bool = False,
                  budget: int = ORACLE_PAIR_BUDGET):
    """Times the oracle (prologue + attention; the FP16-PV variant's when pv16)
    on the sample of oracle_sample_plan; returns (ops, seconds, threads,
    output rows [rows, D] of query head 0, description)."""
    import oracle
    heads, kv_heads, rows = oracle_sample_plan(w, budget)
    q, k, v = wl.segment(w, inp, 0)
    qs = np.ascontiguousarray(q[:heads])
    ks = np.ascontiguousarray(k[:kv_heads])
    vs = np.ascontiguousarray(v[:kv_heads])
    lq, lk = w.seg_lengths()[0]
    t0 = time.perf_counter()
    pro = oracle.prologue(qs, ks, vs, w.dtype)
    if pv16:
        ref = oracle.attn_pv16(pro, oracle.v16(vs, w.dtype), w.causal, wl.default_sm_scale(w),
                               rows=(0, rows))
    else:
        ref = oracle.attn(pro, w.causal, wl.default_sm_scale(w), rows=(0, rows))
    dt = time.perf_counter() - t0
    if w.causal:
        # the sample's unmasked work, restated in the metric's literal count
        # (the workload's literal/effective ratio): a linear extrapolation
        pairs = sum(min(i + 1, lk) for i in range(rows))
        pairs *= w.ops() / w.ops(causal_effective=True)
    else:
        pairs = rows * lk
    ops = 4.0 * heads * pairs * w.D
    whole = heads == w.Hq and rows == lq and w.nseg == 1
    desc = (f"segment 0, query heads [0,{heads}), rows [0,{rows}) of each"
            f"{' (the whole workload)' if whole else ''}: the prologue of those heads plus "
            f"attention, scaled to the workload's op count by the sample's (row, key) pairs")
    return ops, dt, os.cpu_count(), ref[0, :rows], desc


def reference_arm(args, w: wl.Workload, rank: int, world: int):
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = wl.make_inputs(w)
    pv16 = args.variant == "pv16"
    for _ in range(args.warmup):
        oracle_sample(w, inp, pv16=pv16, budget=max(args.oracle_pairs // 16, 1))
    tot_ops, tot_s, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        ops, dt, cores, _, desc = oracle_sample(w, inp, pv16=pv16, budget=args.oracle_pairs)
        tot_ops += ops
        tot_s += dt
    tops = tot_ops / tot_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int8+fp16 (fp32 softmax)" if pv16 else "int8+e4m3 (fp32 softmax)",
        "data": "synthetic", "config": dict(config_of(w), variant=args.variant),
        "cpu_baseline": {"value": tops, "unit": "TOPS", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc + ", per step"},
        "e2e": {"value": tops, "unit": "TOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w: wl.Workload) -> dict:
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Lq": w.Lq, "Lk": w.Lk,
         "D": w.D, "input_dtype": "fp16" if w.dtype == wl.F16 else "bf16",
         "layout": "HND" if w.layout == wl.HND else "NHD", "causal": w.causal,
         "l2": "flushed between timed steps (256 MiB write)"}
    if w.varlen:
        c["seqlens"] = list(w.seqlens_q)
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="sage", choices=["sage", "reference"])
    ap.add_argument("--variant", default="fp8", choices=["fp8", "pv16"],
                    help="fp8: INT8 QK^T + FP8 PV (default); pv16: INT8 QK^T + FP16 PV")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--oracle-pairs", type=int, default=ORACLE_PAIR_BUDGET,
                    help="(query row, key) pairs per head of the oracle's sample, both arms")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    w = wl.WORKLOADS[args.workload]

    if args.impl == "reference":
        reference_arm(args, w, rank, world)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_gpu(args, w, rank, world)
    if rank != 0:
        return
    peaks, src = load_peaks()
    # attention kernel roofline: QK^T on the 16-bit tensor pipe (exact int8
    # emulation) and PV on the FP8 pipe (2x rate) => ceiling 4/3 x bf16 peak
    bf16 = peaks["bf16_tflops"]
    pv16 = args.variant == "pv16"
    # the FP16-PV variant runs both products on the 16-bit pipe
    mix_peak = bf16 if pv16 else bf16 * 4.0 / 3.0
    fp8_peak = bf16 * 2.0
    fig = job_figures(r, world, args.steps)
    # the kernel's algorithmic work: padded head dimension, masked tiles of a
    # causal problem not counted (the kernel skips them)
    att_tflops = fig["attention_tflops_padded_effective"]
    tops = fig["value"]
    pro_gbs = prologue_bytes(w, 2 if pv16 else 1) / (r["pro_ms"] * 1e-3) / 1e9
    inp = wl.make_inputs(w)
    cpu_ops, cpu_s, cores, ref_rows, cpu_desc = oracle_sample(w, inp, pv16=pv16,
                                                               budget=args.oracle_pairs)
    # the bench's own output on the oracle's sample (segment 0, query head 0)
    got_rows = r["out_rows"][:ref_rows.shape[0]]
    # the tensor ceiling measured live (same clock as the timed region):
    # QK^T at the fp16 rate and PV at the e4m3 rate, equal flops each, or
    # both products at the fp16 rate for the FP16-PV variant
    r16, r8 = r["tc"][0], r["tc"][1]
    live_peak = r16 if pv16 else 2.0 / (1.0 / r16 + 1.0 / r8)
    parity = float(np.max(np.abs(got_rows.astype(np.float64) - ref_rows)))
    line = {
        "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["total_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("int8+fp16 (fp32 softmax/accumulate)" if pv16 else
                  "int8+e4m3 (fp32 softmax/accumulate)"), "data": "synthetic",
        "config": dict(config_of(w), variant=args.variant),
        "roofline": {"bound": "tensor", "achieved": att_tflops, "peak": mix_peak,
                     "unit": "TFLOP/s", "frac": att_tflops / mix_peak,
                     "traffic": (ATTN16_NCU_DRAM_BYTES if pv16 else
                                 ATTN_NCU_DRAM_BYTES).get(w.name),
                     "kernel": "attn_kernel (fused QK^T/softmax/PV)",
                     "peak_note": (f"{src} bf16 burst {bf16} (QK^T and the fp16 PV at the "
                                   "16-bit rate)" if pv16 else
                                   f"4/3 x {src} bf16 burst {bf16} (QK^T at the 16-bit "
                                   "rate, PV at the FP8 rate)"),
                     "fp8_peak": fp8_peak, "frac_of_fp8_peak": att_tflops / fp8_peak,
                     "live_tensor_tflops": {"fp16_k16": r16, "e4m3_k32": r8},
                     "live_peak": live_peak, "frac_of_live_peak": att_tflops / live_peak,
                     "live_peak_note": ("back-to-back M=128 N=128 tcgen05 MMAs on every SM, "
                                        "measured right after the timed region (sage_debug_"
                                        "tc_rate); the mix ceiling at the clock the kernel "
                                        "ran at")},
        "ops_per_step": {"literal": r["ops"], "padded_d": r["ops_padded"],
                         "causal_effective": r["ops_effective"],
                         "padded_d_causal_effective": r["ops_padded_effective"]},
        "value_padded_d": fig["value_padded_d"],
        "value_causal_effective": fig["value_causal_effective"],
        "attention_ms": r["att_ms"], "attention_tops": att_tflops,
        "attention_tops_literal": r["ops"] / (r["att_ms"] * 1e-3) / 1e12,
        "prologue_ms": r["pro_ms"], "prologue_gbs": pro_gbs,
        "prologue_hbm_frac": pro_gbs / peaks["hbm_gbs"],
        "e2e": {"value": fig["e2e"], "unit": "TOPS",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "api": r["e2e_api"]},
        "parity_sample": {"max_abs_vs_oracle": parity, "tolerance": 2e-3,
                          "rows": f"segment 0, query head 0, rows [0,{ref_rows.shape[0]}) "
                                  "of the last e2e output"},
        "gpu_launches": r["launches"],
        "launches_per_step": r["launches_per_step"],
        "clocks": r["clocks"],
        "cpu_baseline": {"value": cpu_ops / cpu_s / 1e12, "unit": "TOPS", "cores": cores,
                         "kind": "oracle", "sample": cpu_desc},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
