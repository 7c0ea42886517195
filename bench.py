#!/usr/bin/env python
"""Benchmark of the KDA operator's hot path on one GB300 (or N replicas).

One step = one packed-sequence prefill of 131072 + 65536 + 32768 + 8192
tokens at H=96, dk=dv=128, bf16 inputs / fp32 state (kda_chunk_fwd), then one
decode step of 256 sequences at H=96, d=128 with the 1.6 GB fp32 state
(kda_decode_step).  Inputs are seeded synthetic tensors resident in HBM
before the timed region; both working sets exceed the 129 MB L2 (29 GB of
prefill inputs, 1.6 GB of decode state), so no L2 flush is needed.

value      : prefill tokens/s (token positions, all 96 heads each), timed over
             the prefill launches with CUDA events on the launching stream.
decode     : state GB/s of the decode step (2 * N*H*dk*dv*4 bytes per step).
prep / post: the passes around the operator on the same 237,568 tokens x 96
             heads: kda_qkv_prep (ShortConv + Swish + L2Norm of q, k, v and
             Sigmoid of beta) and kda_output_gate (Sigmoid(gate) * RMSNorm(o)),
             each timed after the main region: HBM GB/s of the bytes each
             pass must move.
gate_variants: the 8192-token x 96-head prefill under Kimi Linear's
             unbounded negative-softplus gate and under one bounded gate per
             head (gated delta), both on the tensor-core prefill (tiles past
             fp32's range for e^{-b} take its position-pair path), timed
             after the main region.
spec_replay: speculative replay (kda_decode_steps) of 256 sequences x 8
             verified tokens with 1..8 accepted, timed after the main region:
             algorithmic GB/s (state once in and out + the applied tokens'
             inputs and outputs) and applied tokens/s.
roofline   : the dominant kernel's algorithmic bytes / launch time vs the
             measured HBM copy bandwidth.
e2e        : prefill tokens/s through the same API with pinned host buffers:
             host->device copies of the step's inputs, the call and the
             device->host read of out and final_state, all inside the timing.
cpu_baseline / --impl reference : the fp64 CPU oracle on a bounded sample of
             the same workload, on the host's cores.

Multi-GPU (torchrun): the (sequence, head) chains share nothing, so no
collective is on the data path; the barrier and a max-over-ranks of the
timings are the only communication.  --partition replicas (default): every
rank runs an independent replica of the workload (weak scaling), value = all
ranks' tokens / the slowest rank's time.  --partition heads: the ranks split
the one workload's 96 heads ([h0, h1) per rank, partition.head_range; the
decode state likewise), value = the workload's tokens / the slowest rank's
time (strong scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_11_gb300 import inputs as kin  # noqa: E402

METRIC = "KDA prefill tokens/s (H=96,d=128) + % TC peak; decode step state GB/s vs HBM"
PREFILL = kin.WORKLOADS["varlen_bf16_H96_237568"]
DECODE = kin.WORKLOADS["decode_bf16_N256_H96"]
SPEC = kin.WORKLOADS["spec_bf16_N256_H96_K8"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# Algorithmic work per token and head, d = dk = dv = 128, 16-token tiles:
# flops 6 d^2 (state products) + 2*16*(3d + 2d) (intra-tile products);
# bytes: q, k, v, g_raw (4 d bf16) + beta (bf16) + out (d bf16).
D = 128
FLOPS_PER_TOKEN_HEAD = 6 * D * D + 2 * 16 * (3 * D + 2 * D)
BYTES_PER_TOKEN_HEAD = 4 * D * 2 + 2 + D * 2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--partition", choices=["replicas", "heads"], default="replicas",
                    help="multi-GPU: independent replicas, or the ranks split one workload by heads")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--only", choices=["all", "prefill", "split", "decode", "spec", "prep", "post"],
                    default="all",
                    help="run one leg only (for profiling captures; the JSON line needs 'all')")
    ap.add_argument("--prep-tokens", type=int, default=0,
                    help="--only prep/post: the first N tokens of the workload (profiling captures); 0 = all")
    ap.add_argument("--prefill-workload", default="varlen_bf16_H96_237568",
                    choices=[k for k, w in kin.WORKLOADS.items() if w.kind == "prefill" and w.dtype == "bf16"],
                    help="prefill workload (profiling captures use the smaller layer-shaped one)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(*names):
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "gated_delta_rule_11_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(kernel_key, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel source as it is now (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha1") != src_hash:
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


def time_region(fn, steps, stream):
    """CUDA-event time of each call of fn on `stream`, in ms (list)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        evs[i][0].record(stream)
        fn(i)
        evs[i][1].record(stream)
    return evs


def run_cpu_oracle_sample(seconds_target, nthreads=None):
    """Time the fp64 oracle on a bounded sample of the prefill workload: the
    32768-token sequence, successive heads, until about `seconds_target` of
    wall time.  Returns (tokens/s expressed at H=96, sample description, threads)."""
    import oracle
    w = PREFILL
    T, dk, dv = 32768, w.dk, w.dv
    nt = oracle.default_threads() if nthreads is None else nthreads
    per_round = max(1, nt)
    g = torch.Generator(device="cpu")
    g.manual_seed(1234)
    done_heads, elapsed = 0, 0.0
    while elapsed < seconds_target and done_heads < w.H:
        nh = min(per_round, w.H - done_heads)
        sample = kin.make_prefill_inputs(w, device="cpu", seed=w.seed + 100 + done_heads,
                                         B=1, T=T, seqlens=(), H=nh)
        args = [sample[n] for n in ("q", "k", "v", "g_raw", "beta")]
        t0 = time.perf_counter()
        oracle.kda_oracle_fwd(*args, None, None, nthreads=nt)
        elapsed += time.perf_counter() - t0
        done_heads += nh
    token_heads = done_heads * T
    rate = token_heads / elapsed / w.H
    desc = (f"oracle (fp64, C, {nt} threads) on the 32768-token sequence of the packed "
            f"workload, {done_heads} of 96 heads ({token_heads} token-heads) in {elapsed:.1f} s; "
            f"tokens/s = token-heads/s / 96")
    return rate, desc, nt


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local)


def reduce_max(x, world):
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, rank, world):
    """The oracle arm: each step runs the fp64 CPU oracle on a bounded sample
    (16 heads of the 8192-token sequence) of the same workload."""
    if rank != 0:
        return 0
    import oracle
    w = PREFILL
    T, nh = 8192, 16
    sample = kin.make_prefill_inputs(w, device="cpu", seed=w.seed + 77, B=1, T=T, seqlens=(), H=nh)
    a = [sample[n] for n in ("q", "k", "v", "g_raw", "beta")]
    nt = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.kda_oracle_fwd(*a, None, None, nthreads=nt)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kda_oracle_fwd(*a, None, None, nthreads=nt)
    dt = time.perf_counter() - t0
    tok_per_s = args.steps * T * nh / dt / w.H
    desc = (f"oracle (fp64, C, {nt} threads): per step 16 of 96 heads of the 8192-token "
            f"sequence ({T * nh} token-heads); tokens/s = token-heads/s / 96")
    line = {"impl": "reference", "metric": METRIC, "value": tok_per_s, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "varlen_bf16_H96_237568 (sampled)", "H": 96, "dk": 128,
                       "dv": 128, "sample": "16 heads x 8192 tokens per step"},
            "cpu_baseline": {"value": tok_per_s, "unit": "tokens/s", "cores": nt,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": tok_per_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_single_leg(args, kda, dev):
    """--only prefill|decode: warm-up then timed launches of one kernel, for
    profiler captures; prints per-launch CUDA-event times, no JSON line."""
    if args.only == "prefill":
        w = kin.WORKLOADS[args.prefill_workload]
        inp = kin.make_prefill_inputs(w, device=dev)
        a = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
        out, fin = kda.kda_chunk_fwd(*a, inp["init_state"], inp["cu_seqlens"])
        fn = lambda i: kda.kda_chunk_fwd(*a, inp["init_state"], inp["cu_seqlens"], out=out, final_state=fin)
    elif args.only == "split":
        w = kin.WORKLOADS["tp8_bf16_H12_T131072"]
        inp = kin.make_prefill_inputs(w, device=dev)
        a = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
        tau = kda.split_segment_tokens(w.B, w.T, w.H, w.B, False,
                                       torch.cuda.get_device_properties(dev).multi_processor_count)
        ws = torch.empty(kda.split_workspace_bytes(w.B, w.T, w.H, w.dk, w.dv, w.B, tau),
                         dtype=torch.uint8, device=dev)
        out, fin = kda.kda_chunk_fwd_split(*a, None, None, segment_tokens=tau, workspace=ws)
        fn = lambda i: kda.kda_chunk_fwd_split(*a, None, None, segment_tokens=tau, workspace=ws,
                                               out=out, final_state=fin)
    elif args.only == "decode":
        w = DECODE
        S = kin.make_decode_state(w, device=dev)
        t = kin.make_decode_token(w, 0, device=dev)
        fn = lambda i: kda.kda_decode_step(t["q"], t["k"], t["v"], t["g_raw"], t["beta"], S)
    elif args.only == "prep":
        w = PREFILL
        ntok = min(args.prep_tokens or w.total_tokens, w.total_tokens)
        pi = kin.make_prep_inputs(ntok, w.H, w.dk, "bf16", device=dev)
        bounds = [min(b, ntok) for b in itertools.accumulate(w.seqlens)]
        cu = torch.tensor([0] + bounds, dtype=torch.int32, device=dev)
        fn = lambda i: kda.kda_qkv_prep(pi["x_qkv"], pi["conv_w"], pi["beta_logit"], cu)
    elif args.only == "post":
        w = PREFILL
        po = kin.make_post_inputs(w.total_tokens * w.H, w.dv, "bf16", device=dev)
        fn = lambda i: kda.kda_output_gate(po["o"], po["gate"], po["norm_w"])
    else:
        w = SPEC
        S = kin.make_decode_state(w, device=dev)
        t = kin.make_decode_drafts(w, 0, device=dev)
        fn = lambda i: kda.kda_decode_steps(t["q"], t["k"], t["v"], t["g_raw"], t["beta"], S,
                                            t["accepted"])
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    for i in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(i)
        e1.record()
        torch.cuda.synchronize()
        print(f"{args.only} {w.name}: {e0.elapsed_time(e1):.3f} ms", flush=True)
    kda.check_device_status()
    return 0


def run_ours(args, rank, world, local):
    from gated_delta_rule_11_gb300 import kda
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.load_library()
    if args.only != "all":
        return run_single_leg(args, kda, dev)
    peaks, peak_src = load_peaks()

    # ---- inputs, resident in HBM
    pw = kin.WORKLOADS[args.prefill_workload]
    by_heads = args.partition == "heads" and world > 1
    if by_heads:      # this rank's heads of the one workload (same shapes per head)
        from gated_delta_rule_11_gb300.partition import head_range
        h0, h1 = head_range(rank, world, pw.H)
        inp = kin.make_prefill_inputs(pw, device=dev, seed=pw.seed + h0, H=h1 - h0)
    else:
        h0, h1 = 0, pw.H
        inp = kin.make_prefill_inputs(pw, device=dev, seed=pw.seed + 1000 * rank)
    H_rank = h1 - h0
    q, k, v, g, b = (inp[n] for n in ("q", "k", "v", "g_raw", "beta"))
    cu = inp["cu_seqlens"]
    N = pw.n_seqs
    T_total = pw.total_tokens
    out = torch.empty_like(v)
    fin = torch.empty((N, H_rank, pw.dk, pw.dv), dtype=torch.float32, device=dev)

    dw = DECODE
    dH = H_rank if by_heads else dw.H
    dseed = dw.seed + (h0 if by_heads else 1000 * rank)
    S = kin.make_decode_state(dw, device=dev, seed=dseed, H=dH)
    toks = [kin.make_decode_token(dw, i, device=dev, seed=dseed, H=dH) for i in range(4)]
    dout = torch.empty((dw.N, dH, dw.dv), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)

    def prefill(_i):
        kda.kda_chunk_fwd(q, k, v, g, b, None, cu, out=out, final_state=fin)

    def decode(i):
        t = toks[i % len(toks)]
        kda.kda_decode_step(t["q"], t["k"], t["v"], t["g_raw"], t["beta"], S, out=dout)

    for i in range(args.warmup):
        prefill(i)
        decode(i)
    torch.cuda.synchronize()

    # ---- timed region: K steps of (prefill, decode)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.1)
    launches0 = kda.launch_count()
    t_wall0 = time.perf_counter()
    ev_all0 = torch.cuda.Event(enable_timing=True)
    ev_all1 = torch.cuda.Event(enable_timing=True)
    pev, dev_ev = [], []
    ev_all0.record(stream)
    for i in range(args.steps):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        prefill(i)
        e1.record(stream)
        decode(i)
        e2.record(stream)
        pev.append((e0, e1))
        dev_ev.append((e1, e2))
    ev_all1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = kda.launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()

    prefill_ms = [a.elapsed_time(c) for a, c in pev]
    decode_ms = [a.elapsed_time(c) for a, c in dev_ev]
    total_ms = ev_all0.elapsed_time(ev_all1)
    p_mean = reduce_max(statistics.fmean(prefill_ms), world)
    d_mean = reduce_max(statistics.fmean(decode_ms), world)
    step_ms = reduce_max(total_ms / args.steps, world)

    # whole job: every rank's tokens (replicas), or the one workload's tokens
    # with its heads split over the ranks
    tokens = T_total if by_heads else T_total * world
    value = tokens / (p_mean * 1e-3)
    token_heads = T_total * H_rank            # one rank's launch (the roofline is per GPU)
    alg_bytes = token_heads * BYTES_PER_TOKEN_HEAD + N * H_rank * pw.dk * pw.dv * 4
    alg_flops = token_heads * FLOPS_PER_TOKEN_HEAD
    p_gbs = alg_bytes / (p_mean * 1e-3) / 1e9
    tc_tflops = alg_flops / (p_mean * 1e-3) / 1e12
    dec_bytes = 2 * dw.N * dH * dw.dk * dw.dv * 4
    d_gbs = dec_bytes / (d_mean * 1e-3) / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    # the prefill launch is timed on its own (CUDA events around it), so the
    # burst cuBLAS figure is its denominator, not the seconds-long sustained one
    tc_peak = float(peaks["bf16_tflops"])
    kernel_name = kda.chunk_fwd_kernel(torch.bfloat16, pw.dk, pw.dv)
    prefill_src = (source_hash("kda_prefill_tc.cu", "kda_internal.cuh", "kda_sm100.cuh", "kda_tc_util.cuh")
                   if kernel_name == "prefill_tc_kernel"
                   else source_hash("kda_prefill_simt.cu", "kda_internal.cuh", "kda_sm100.cuh"))
    decode_src = source_hash("kda_decode.cu", "kda_internal.cuh")
    p_traffic = recorded_traffic("prefill", prefill_src)
    d_traffic = recorded_traffic("decode", decode_src)

    layer = run_layer_prefill(kda, dev, rank, world, min(args.steps, 10), args.warmup, hbm_peak,
                              float(peaks["bf16_tflops"]), peak_src)
    split = run_split_prefill(kda, dev, rank, world, min(args.steps, 10), args.warmup, hbm_peak,
                              peak_src)
    spec = run_spec(kda, dev, rank, world, args.steps, args.warmup, hbm_peak, peak_src)
    prep, post = run_prepost(kda, dev, world, min(args.steps, 10), args.warmup, hbm_peak, peak_src)
    gates = run_gate_variants(kda, dev, world, min(args.steps, 5), args.warmup, hbm_peak, peak_src)

    e2e = None
    if not args.no_e2e:   # every rank: the timing is reduced over ranks
        e2e = run_e2e(kda, q, k, v, g, b, cu, out, fin, args.e2e_steps, world,
                      T_total if by_heads else T_total * world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, nt = run_cpu_oracle_sample(args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": nt, "kind": "oracle", "sample": desc}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "strong" if by_heads else "weak", "vs_baseline": None,
        "dtype": ("f16 tensor-core operands (bf16 inputs; fp32 state, gates and accumulation)"
                  if kernel_name == "prefill_tc_kernel" else "f32 (bf16 inputs)"),
        "data": "synthetic",
        "config": {
            "workload": f"{pw.name} prefill + decode_bf16_N256_H96 step",
            "prefill_seqlens": list(pw.seqlens) or [pw.T] * pw.B, "H": pw.H, "dk": pw.dk, "dv": pw.dv,
            "decode_N": dw.N, "l2": "inputs larger than L2 (29 GB prefill inputs, 1.6 GB decode state); no flush",
            "value_counts": "prefill launches only (decode reported under 'decode')",
            "parallelism": (f"heads split over {world} ranks ({H_rank} on rank 0)" if by_heads
                            else f"replicas x{world}"),
        },
        "prefill_ms": p_mean, "decode_ms": d_mean,
        "roofline": {"kernel": kernel_name, "bound": "hbm", "achieved": p_gbs,
                     "peak": hbm_peak, "unit": "GB/s", "frac": p_gbs / hbm_peak,
                     "traffic": p_traffic, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": alg_bytes},
        "tensor": {"achieved_tflops": tc_tflops, "peak_tflops": tc_peak,
                   "frac": tc_tflops / tc_peak, "algorithmic_flops_per_launch": alg_flops,
                   "peak_source": peak_src + " (burst bf16: the launch is timed alone)"},
        "decode": {"metric": "decode step state GB/s", "value": d_gbs, "unit": "GB/s",
                   "ms": d_mean, "state_bytes_per_step": dec_bytes,
                   "roofline": {"kernel": "decode1_kernel", "bound": "hbm", "achieved": d_gbs,
                                "peak": hbm_peak, "unit": "GB/s", "frac": d_gbs / hbm_peak,
                                "traffic": d_traffic, "peak_source": peak_src}},
        "layer_prefill": layer,
        "split_prefill": split,
        "spec_replay": spec, "prep": prep, "post": post, "gate_variants": gates,
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches,
        "clocks": clocks, "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_layer_prefill(kda, dev, rank, world, steps, warmup, hbm_peak, tc_peak, peak_src):
    """The model's layer shape, one 8192-token sequence x 96 heads (fewer
    chains than SMs), default gate: its own roofline line."""
    w = kin.WORKLOADS["layer_bf16_H96_T8192"]
    inp = kin.make_prefill_inputs(w, device=dev, seed=w.seed + 1000 * rank)
    a = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    out = torch.empty_like(inp["v"])
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fn = lambda i: kda.kda_chunk_fwd(*a, None, None, out=out, final_state=fin)
    for i in range(warmup):
        fn(i)
    barrier(world)
    torch.cuda.synchronize()
    evs = time_region(fn, steps, stream)
    torch.cuda.synchronize()
    ms = reduce_max(statistics.fmean(a.elapsed_time(b) for a, b in evs), world)
    th = w.B * w.T * w.H
    nbytes = th * BYTES_PER_TOKEN_HEAD + w.B * w.H * w.dk * w.dv * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    tfl = th * FLOPS_PER_TOKEN_HEAD / (ms * 1e-3) / 1e12
    res = {"workload": w.name, "ms": ms, "tokens_per_s": w.B * w.T * world / (ms * 1e-3),
           "chains": w.B * w.H,
           "roofline": {"kernel": kda.chunk_fwd_kernel(torch.bfloat16, w.dk, w.dv), "bound": "hbm",
                        "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                        "algorithmic_bytes_per_launch": nbytes, "peak_source": peak_src},
           "tensor": {"achieved_tflops": tfl, "peak_tflops": tc_peak, "frac": tfl / tc_peak,
                      "peak_source": peak_src + " (burst bf16)"}}
    del inp, a, out, fin
    torch.cuda.empty_cache()
    return res


def run_split_prefill(kda, dev, rank, world, steps, warmup, hbm_peak, peak_src):
    """One 131,072-token sequence x 12 heads (the 96-head layer sharded 8
    ways by head): 12 chains on the whole GPU, unsplit and with the segment
    split (kda_chunk_fwd_split, automatic segment length).  The roofline
    counts the operator's own bytes (inputs, outputs, final states); the
    split's workspace traffic is reported beside it."""
    w = kin.WORKLOADS["tp8_bf16_H12_T131072"]
    inp = kin.make_prefill_inputs(w, device=dev, seed=w.seed + 1000 * rank)
    a = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    out = torch.empty_like(inp["v"])
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tau = kda.split_segment_tokens(w.B, w.T, w.H, w.B, False, sms)
    ws = torch.empty(max(kda.split_workspace_bytes(w.B, w.T, w.H, w.dk, w.dv, w.B, tau), 1),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    th = w.B * w.T * w.H
    nbytes = th * BYTES_PER_TOKEN_HEAD + w.B * w.H * w.dk * w.dv * 4
    res = {"workload": w.name, "chains": w.B * w.H, "sms": sms, "segment_tokens": tau}
    legs = (("unsplit", lambda i: kda.kda_chunk_fwd(*a, None, None, out=out, final_state=fin)),
            ("split", lambda i: kda.kda_chunk_fwd_split(*a, None, None, segment_tokens=tau,
                                                        workspace=ws, out=out, final_state=fin)))
    for name, fn in legs:
        for i in range(warmup):
            fn(i)
        barrier(world)
        torch.cuda.synchronize()
        l0 = kda.launch_count()
        evs = time_region(fn, steps, stream)
        torch.cuda.synchronize()
        ms = reduce_max(statistics.fmean(x.elapsed_time(y) for x, y in evs), world)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "tokens_per_s": w.B * w.T * world / (ms * 1e-3),
                     "launches_per_call": (kda.launch_count() - l0) // max(steps, 1),
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                                  "frac": gbs / hbm_peak, "algorithmic_bytes_per_launch": nbytes,
                                  "peak_source": peak_src}}
    P = -(-w.T // tau) if tau else 1
    # the split's workspace traffic per token and head of segments 1..: the
    # transition run's q, k, g_raw, beta reads, its fp32 rows written and
    # read, the zero-state run's fp32 rows (instead of bf16) written and
    # read; plus the virtual chains' states (written, read, composed)
    later = w.T - min(tau, w.T) if tau else 0
    per_tok = (3 * w.dk * 2 + 2) + 2 * w.dk * 4 + (w.dv * 4 - w.dv * 2) + w.dv * 4
    res["split"]["extra_bytes"] = (w.H * later * per_tok
                                   + w.H * (2 * P - 1) * w.dk * w.dv * 4 * 3) if tau else 0
    res["speedup"] = res["unsplit"]["ms"] / res["split"]["ms"]
    del inp, a, out, fin, ws
    torch.cuda.empty_cache()
    return res


def run_spec(kda, dev, rank, world, steps, warmup, hbm_peak, peak_src):
    """Speculative replay on the spec workload: `steps` launches, each with its
    own drafts and accepted counts (a few batches cycled), the state carried
    from launch to launch.  Returns the report object."""
    w = SPEC
    S = kin.make_decode_state(w, device=dev, seed=w.seed + 1000 * rank)
    batches = [kin.make_decode_drafts(w, i, device=dev, seed=w.seed + 1000 * rank) for i in range(4)]
    out = torch.empty((w.N, w.drafts, w.H, w.dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fn(i):
        t = batches[i % len(batches)]
        kda.kda_decode_steps(t["q"], t["k"], t["v"], t["g_raw"], t["beta"], S, t["accepted"],
                             out=out)

    for i in range(warmup):
        fn(i)
    barrier(world)
    torch.cuda.synchronize()
    evs = time_region(fn, steps, stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    applied = [int(batches[i % len(batches)]["accepted"].sum()) for i in range(steps)]
    mean_ms = reduce_max(statistics.fmean(ms), world)
    state_bytes = 2 * w.N * w.H * w.dk * w.dv * 4
    tok_bytes = w.H * (3 * w.dk * 2 + w.dv * 2 + 2 + w.dv * 2)   # q, k, g_raw, v, beta in; out
    mean_applied = statistics.fmean(applied)
    alg = state_bytes + mean_applied * tok_bytes
    gbs = alg / (mean_ms * 1e-3) / 1e9
    return {"workload": w.name, "N": w.N, "K": w.drafts, "H": w.H,
            "mean_accepted_per_seq": mean_applied / w.N, "ms": mean_ms,
            "applied_tokens_per_s": mean_applied * world / (mean_ms * 1e-3),
            "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": gbs,
                         "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "algorithmic_bytes_per_launch": alg, "peak_source": peak_src}}


def run_gate_variants(kda, dev, world, steps, warmup, hbm_peak, peak_src):
    """Prefill of the layer-shaped workload under two non-default gates."""
    w = kin.WORKLOADS["layer_bf16_H96_T8192"]
    inp = kin.make_prefill_inputs(w, device=dev)
    args = [inp[n] for n in ("q", "k", "v")]
    out = torch.empty_like(inp["v"])
    fin = torch.empty((1, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    g_head = inp["g_raw"][..., 0].contiguous()          # one gate per (token, head)
    res = {"workload": w.name}
    for name, g, mode, per_head in (("neg_softplus", inp["g_raw"], "neg_softplus", False),
                                    ("gated_delta_per_head", g_head, "bounded", True)):
        fn = lambda i: kda.kda_chunk_fwd(*args, g, inp["beta"], None, None, out=out, final_state=fin,
                                         gate_mode=mode, gate_per_head=per_head)
        for i in range(warmup):
            fn(i)
        barrier(world)
        torch.cuda.synchronize()
        evs = time_region(fn, steps, stream)
        torch.cuda.synchronize()
        ms = reduce_max(statistics.fmean(a.elapsed_time(b) for a, b in evs), world)
        th = w.T * w.H
        gate_bytes = (w.dk if not per_head else 1) * 2
        nbytes = th * (BYTES_PER_TOKEN_HEAD - D * 2 + gate_bytes) + w.H * w.dk * w.dv * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "tokens_per_s": w.T / (ms * 1e-3),
                     "kernel": kda.chunk_fwd_kernel(torch.bfloat16, w.dk, w.dv),
                     "achieved_gbs": gbs, "frac": gbs / hbm_peak,
                     "peak_source": peak_src}
    del inp, out, fin
    torch.cuda.empty_cache()
    return res


def run_prepost(kda, dev, world, steps, warmup, hbm_peak, peak_src):
    """The pre/post passes on the varlen workload's tokens and heads."""
    w = PREFILL
    T, H, d = w.total_tokens, w.H, w.dk
    stream = torch.cuda.current_stream(dev)
    cu = torch.tensor([0] + list(itertools.accumulate(w.seqlens)), dtype=torch.int32, device=dev)

    def measure(fn, nbytes, kernel):
        for i in range(warmup):
            fn(i)
        barrier(world)
        torch.cuda.synchronize()
        evs = time_region(fn, steps, stream)
        torch.cuda.synchronize()
        ms = reduce_max(statistics.fmean(a.elapsed_time(b) for a, b in evs), world)
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"ms": ms, "roofline": {"kernel": kernel, "bound": "hbm", "achieved": gbs,
                                       "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                                       "algorithmic_bytes_per_launch": nbytes,
                                       "peak_source": peak_src}}

    pi = kin.make_prep_inputs(T, H, d, "bf16", device=dev)
    outs = [torch.empty((1, T, H, d), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    beta = torch.empty((1, T, H), dtype=torch.bfloat16, device=dev)
    fn = lambda i: kda.kda_qkv_prep(pi["x_qkv"], pi["conv_w"], pi["beta_logit"], cu,
                                    out=(*outs, beta))
    prep_bytes = 2 * (3 * T * H * d * 2) + 2 * T * H * 2 + 3 * H * d * 16
    prep = measure(fn, prep_bytes, "prep_kernel")
    prep.update({"tokens": T, "H": H, "d": d})
    del pi, outs, beta
    po = kin.make_post_inputs(T * H, d, "bf16", device=dev)
    y = torch.empty_like(po["o"])
    fn = lambda i: kda.kda_output_gate(po["o"], po["gate"], po["norm_w"], out=y)
    post = measure(fn, 3 * T * H * d * 2 + d * 4, "output_gate_kernel")
    post.update({"rows": T * H, "d": d})
    del po, y
    torch.cuda.empty_cache()
    return prep, post


def run_e2e(kda, q, k, v, g, b, cu, out, fin, steps, world, job_tokens):
    """Prefill through the public API from pinned host buffers, pipelined:
    every step copies its inputs host->device and its out and final_state
    device->host; step i+1's upload runs while step i computes and downloads
    (two device buffer sets; three streams ordered by events)."""
    def pinned_copy(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    # Allocate first, then agree over the ranks: a host that cannot pin every
    # rank's buffers (or a device out of memory) skips the leg on all ranks
    # alike, so no rank waits in a collective that another never reaches.
    failure = None
    try:
        hin = [pinned_copy(t) for t in (q, k, v, g, b)]
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        hfin = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
        din = [[q, k, v, g, b], [torch.empty_like(t) for t in (q, k, v, g, b)]]
        dout = [[out, fin], [torch.empty_like(out), torch.empty_like(fin)]]
    except RuntimeError as exc:
        failure = str(exc).splitlines()[0][:200]
    if reduce_max(1.0 if failure else 0.0, world) > 0.0:
        hin = hout = hfin = din = dout = None
        torch.cuda.empty_cache()
        return {"unavailable": "end-to-end buffers could not be allocated on "
                               + ("this rank: " + failure if failure else "another rank")}
    up, comp, down = torch.cuda.Stream(), torch.cuda.current_stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    uploaded, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in computed + downloaded:
        e.record(comp)

    def step(i):
        sl = i % 2
        up.wait_event(computed[sl])                 # the kernel two steps back read this input set
        with torch.cuda.stream(up):
            for d, h in zip(din[sl], hin):
                d.copy_(h, non_blocking=True)
        uploaded[sl].record(up)
        comp.wait_event(uploaded[sl])
        comp.wait_event(downloaded[sl])             # this output set was downloaded two steps back
        kda.kda_chunk_fwd(*din[sl], None, cu, out=dout[sl][0], final_state=dout[sl][1])
        computed[sl].record(comp)
        down.wait_event(computed[sl])
        with torch.cuda.stream(down):
            hout.copy_(dout[sl][0], non_blocking=True)
            hfin.copy_(dout[sl][1], non_blocking=True)
        downloaded[sl].record(down)

    step(0)
    step(1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    ms = reduce_max((time.perf_counter() - t0) * 1e3 / steps, world)
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = hout.numel() * hout.element_size() + hfin.numel() * hfin.element_size()
    del din[1], dout[1]
    torch.cuda.empty_cache()
    return {"value": job_tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "host wall clock over the steps, device synchronised on both sides",
            "pipelined": "step i+1's host->device copy overlaps step i's kernel and device->host copy"}


if __name__ == "__main__":
    sys.exit(main())
