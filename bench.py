#!/usr/bin/env python
"""Bench of the packed lookahead call on one GB300 (or N independent replicas).

Workload (one bench step = one request): Llama-7B-shape random-init bf16
model (32 layers, d 4096, 32 heads of 128, FFN 11008, vocab 32000, weights
N(0, 0.02) seed 0), batch 1, a 512-token prompt from a seeded order-2 Markov
chain with Zipf(1.1) next-token ranks (seed 2), greedy, 256 new tokens,
W=15, N=5, G=15.

Reported (one JSON line on rank 0):
  value        committed tokens/s of the decode phase: tokens produced by the
               packed calls / their device time (CUDA events on the library's
               stream), summed over the timed requests and all ranks
  e2e          tokens/s of the same requests through la_generate with host
               prompt and host output (prompt H2D, prefill, decode, D2H)
  roofline     the packed call against HBM: algorithmic bytes per call
               (weights read once + committed K/V read + temporary K/V
               written) / measured call time, peak = measured copy bandwidth
  cpu_baseline the CPU oracle on this host's cores on a bounded sample
Inputs are larger than L2 (13 GB of weights stream every call), so no L2
flush is needed between steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

W_, N_, G_ = 15, 5, 15
PROMPT_LEN, MAX_NEW = 512, 256


def algorithmic_bytes_per_call(cfg, K_in: float, Q: float) -> float:
    """Weights read once + committed K/V read + temporary K/V written, bf16."""
    d, F, V, L = cfg.d_model, cfg.d_ffn, cfg.vocab, cfg.n_layers
    HD = cfg.n_heads * cfg.head_dim
    weights = L * (d * 3 * HD + HD * d + 3 * d * F) * 2 + V * d * 2 + (2 * L + 1) * d * 2
    kv_read = K_in * L * 2 * HD * 2
    kv_write = Q * L * 2 * HD * 2
    return weights + kv_read + kv_write


def gemm_bytes_per_call(cfg, Q: float, need_rows: float) -> float:
    """Algorithmic bytes of the tensor-core GEMMs of one packed call (bf16
    weights read once, bf16 activations read once, outputs written once;
    the residual GEMMs read and write the fp32 residual rows)."""
    d, F, V, L = cfg.d_model, cfg.d_ffn, cfg.vocab, cfg.n_layers
    HD = cfg.n_heads * cfg.head_dim
    per_layer = ((3 * HD * d) * 2 + Q * d * 2 + Q * 3 * HD * 2          # QKV: store bf16
                 + (d * HD) * 2 + Q * HD * 2 + Q * d * 8                # O: residual fp32 read + write
                 + (2 * F * d) * 2 + Q * d * 2 + Q * F * 2              # gate/up + SwiGLU: store bf16
                 + (d * F) * 2 + Q * F * 2 + Q * d * 8)                 # down: residual
    head = V * d * 2 + need_rows * d * 2 + need_rows * (V // 128) * 8   # argmax partials (value, id)
    return L * per_layer + head


# DRAM bytes (read + write) of the GEMM launches of one packed call (32 layers
# x (QKV + O + gate/up + down) + LM head), from the ncu capture of the current
# kernel's launches in a decode call summarised in profiles/; None once the
# kernel changes.
GEMM_TRAFFIC_PER_CALL = 13.608e9


def aggregate_replicas(new_tokens: float, decode_s: float, wall: float, device: str = "cpu"):
    """Whole-job figures of independent replicas (one request per rank): tokens
    summed over the ranks, decode and wall-clock times the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(new_tokens), float(decode_s), float(wall)
    t = torch.tensor([new_tokens, decode_s, wall], dtype=torch.float64, device=device)
    g = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(g, t)
    return sum(float(x[0]) for x in g), max(float(x[1]) for x in g), max(float(x[2]) for x in g)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        return parse_clocks(self.path)


def parse_clocks(path: str):
    """Median SM clock, its maximum and the throttle reasons seen, from the
    nvidia-smi samples (csv, no header, no units; columns as ClockSampler.Q)."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(cfg, weights, min_s: float = 10.0, max_calls: int = 64, prompt_len: int = 24):
    """The oracle (as it stands) on the host cores: a bounded sample of the same
    workload — prefill of a short Markov prompt (not timed), then packed
    lookahead calls at W=15, N=5, G=15 until `min_s` seconds of them have run
    (at most `max_calls`); returns committed tokens/s of those calls."""
    import numpy as np
    import synth
    from oracle import lookahead as la
    from oracle.model import OracleModel, argmax_lowest
    m = OracleModel(cfg, weights, compute_dtype=np.float32, store="bf16", cache_weights=True)
    p = synth.markov_zipf_prompt(cfg.vocab, prompt_len, 2).tolist()
    cache, lg = m.prefill(p)                    # also converts and caches the weights (not timed)
    st = la.LookaheadState(p, argmax_lowest(lg[-1]), W_, N_, G_)
    run = la.make_runner(m, cache, "meta")
    t0 = time.perf_counter()
    toks = 0
    n_calls = 0
    while n_calls < max_calls and (n_calls == 0 or time.perf_counter() - t0 < min_s):
        rows, g = st.plan()
        out = run.run(rows)
        info = st.publish(rows, g, [argmax_lowest(x) for x in out])
        run.commit(rows, info.commit_rows)
        toks += len(info.emitted)
        n_calls += 1
    dt = time.perf_counter() - t0
    return {"value": toks / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"oracle fp32 arithmetic, bf16 storage emulation; {n_calls} packed calls (W=15,N=5,G=15) "
                      f"after a {prompt_len}-token prompt on the 7B shape; {toks} tokens in {dt:.1f} s"}


def batch_prompts(vocab: int, B: int):
    """B different 512-token Markov/Zipf prompts (seeds 2, 3, ..)."""
    import synth
    return [synth.markov_zipf_prompt(vocab, PROMPT_LEN, 2 + b).tolist() for b in range(B)]


SWEEP_W, SWEEP_N, SWEEP_PROMPT = (1, 3, 7, 15, 31), (3, 5, 7), 1024


def run_sweep(args, cfg, rank: int, local: int) -> None:
    """Per sweep point (W, N, G = W) on a 1024-token Markov prompt: packed-call
    latency, committed tokens per call, the call's roofline fraction and the
    autoregressive step latency on the same kernels; one context per point."""
    if rank != 0:
        return
    import torch
    import synth
    torch.cuda.set_device(local)
    from lookahead_decoding_gb300 import build
    build()
    from lookahead_decoding_gb300 import lib
    L = lib()
    w = synth.llama_weights(cfg, 0, device=f"cuda:{local}")
    prompt = synth.markov_zipf_prompt(cfg.vocab, SWEEP_PROMPT, 2).tolist()
    peaks, src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    max_ctx = SWEEP_PROMPT + args.max_new + 64
    ar_ms, ar_out = None, None
    points = []
    for W in SWEEP_W:
        for N in SWEEP_N:
            try:
                ctx = L.Context(cfg, w, max_ctx=max_ctx, max_W=W, max_N=N, max_G=W)
            except L.LaError as e:
                points.append({"W": W, "N": N, "G": W, "unsupported": str(e)})
                continue
            if ar_ms is None:
                st = L.la_stats()
                ar_out = L.la_generate_ar(ctx.ctx, prompt, args.max_new, stats=st)
                ar_ms = st.decode_ns * 1e-6 / st.steps
            L.la_generate(ctx.ctx, prompt, args.max_new, W, N, W)          # warm-up (graph capture)
            st = L.la_stats()
            out = L.la_generate(ctx.ctx, prompt, args.max_new, W, N, W, stats=st)
            call_ms = st.decode_ns * 1e-6 / st.steps
            K_mean = SWEEP_PROMPT + args.max_new / 2.0
            bytes_call = algorithmic_bytes_per_call(cfg, K_mean, st.mean_rows)
            points.append({"W": W, "N": N, "G": W, "call_ms": call_ms, "tokens_per_call": (st.tokens - 1) / st.steps,
                           "tokens_per_s": (st.tokens - 1) / (st.decode_ns * 1e-9), "mean_rows": st.mean_rows,
                           "step_roofline_frac": bytes_call / (call_ms * 1e-3) / 1e9 / peak,
                           "equals_ar": out == ar_out})
            ctx.close()
    line = {"metric": "W x N sweep (7B-shape bf16, greedy)", "unit": "ms per packed call", "n_gpus": 1,
            "config": {"workload": f"llama-7b-shape bf16, batch 1, prompt {SWEEP_PROMPT} Markov/Zipf(1.1), "
                                   f"{args.max_new} new tokens, greedy, G = W", "model": "llama-7b-shape (random init)"},
            "ar_ms_per_token": ar_ms, "peak_gbs": peak, "peak_source": src, "points": points}
    print(json.dumps(line))


def run_batch(args, cfg, rank: int, local: int) -> None:
    """Several requests per packed call on one GPU: committed tokens/s of all
    requests (decode device time), each request checked against its AR output."""
    if rank != 0:
        return
    import torch
    import synth
    torch.cuda.set_device(local)
    from lookahead_decoding_gb300 import build
    build()
    from lookahead_decoding_gb300 import lib
    L = lib()
    B = args.batch
    w = synth.llama_weights(cfg, 0, device=f"cuda:{local}")
    ctx = L.Context(cfg, w, max_ctx=1024, max_W=W_, max_N=N_, max_G=G_, max_batch=B)
    prompts = batch_prompts(cfg.vocab, B)
    for _ in range(args.warmup):
        L.la_generate_batch(ctx.ctx, prompts, args.max_new, W_, N_, G_)
    os.makedirs(os.path.join(ROOT, "gpurun_out"), exist_ok=True)
    clocks = ClockSampler(local, os.path.join(ROOT, "gpurun_out", f"clocks_rank{rank}.csv"))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    stats, outs = [], []
    for _ in range(args.steps):
        st = L.la_stats()
        outs.append(L.la_generate_batch(ctx.ctx, prompts, args.max_new, W_, N_, G_, stats=st))
        stats.append(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    decode_s = sum(s.decode_ns for s in stats) * 1e-9
    calls = sum(s.steps for s in stats)
    new_tokens = sum(B * (args.max_new - 1) for _ in stats)
    ar = [L.la_generate_ar(ctx.ctx, p, args.max_new) for p in prompts]
    config = {"workload": f"llama-7b-shape bf16, {B} requests per packed call, prompts 512 Markov/Zipf(1.1), "
                          f"{args.max_new} new tokens each, greedy, W=15 N=5 G=15",
              "model": "llama-7b-shape (random init)", "global_batch": B, "seq_len": PROMPT_LEN + args.max_new,
              "parallelism": "one GPU", "l2": "inputs larger than L2 (13 GB weights per call); no flush"}
    line = {"metric": f"committed tokens/s @ batch {B} (7B-shape bf16)", "value": new_tokens / decode_s,
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
            "call_latency_ms": decode_s / calls * 1e3, "calls_per_request": calls / args.steps,
            "batched_equals_ar": all(o == ar for o in outs),
            "e2e": {"value": B * args.max_new * args.steps / wall, "unit": "tokens/s",
                    "h2d_bytes_per_step": B * PROMPT_LEN * 4, "d2h_bytes_per_step": B * args.max_new * 4},
            "clocks": clk}
    ctx.close()
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ar-steps", type=int, default=1)
    ap.add_argument("--max-new", type=int, default=MAX_NEW, help="new tokens per request (profiling runs)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling runs: a model with this many layers of the same shapes (0 = all 32)")
    ap.add_argument("--batch", type=int, default=1,
                    help="requests per packed call (la_generate_batch); 1 = the headline single-request bench")
    ap.add_argument("--sweep", action="store_true",
                    help="the W x N sweep on the 7B shape (W in 1,3,7,15,31; N in 3,5,7; G=W): one JSON line")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import torch
    import synth
    cfg = synth.LLAMA_7B
    if args.layers:
        import dataclasses
        cfg = dataclasses.replace(cfg, n_layers=args.layers)
    config = {"workload": "llama-7b-shape bf16, batch 1, prompt 512 Markov/Zipf(1.1), 256 new tokens, greedy, "
                          "W=15 N=5 G=15", "model": "llama-7b-shape (random init)", "global_batch": world,
              "seq_len": PROMPT_LEN + MAX_NEW, "parallelism": f"replicas{world}",
              "l2": "inputs larger than L2 (13 GB weights per call); no flush"}

    if args.impl == "reference":
        if rank != 0:
            return
        dev = "cuda:0" if torch.cuda.is_available() else "cpu"
        w = synth.llama_weights(cfg, 0, device=dev)
        vals = []
        for _ in range(max(1, args.warmup)):
            pass          # the oracle has no warm-up state; warm-up runs would only repeat the sample
        samples = [cpu_oracle_sample(cfg, w, min_s=8.0) for _ in range(max(1, args.steps))]
        v = statistics.mean(s["value"] for s in samples)
        line = {"impl": "reference", "metric": "committed tokens/s", "value": v, "unit": "tokens/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
                "cpu_baseline": dict(samples[-1], value=v),
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.sweep:
        return run_sweep(args, cfg, rank, local)
    if args.batch > 1:
        return run_batch(args, cfg, rank, local)

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from lookahead_decoding_gb300 import build
    build()
    from lookahead_decoding_gb300 import lib
    L = lib()
    w = synth.llama_weights(cfg, 0, device=f"cuda:{local}")
    ctx = L.Context(cfg, w, max_ctx=1024, max_W=W_, max_N=N_, max_G=G_)
    prompt = synth.markov_zipf_prompt(cfg.vocab, PROMPT_LEN, 2).tolist()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        L.la_generate(ctx.ctx, prompt, args.max_new, W_, N_, G_)
    os.makedirs(os.path.join(ROOT, "gpurun_out"), exist_ok=True)
    clocks = ClockSampler(local, os.path.join(ROOT, "gpurun_out", f"clocks_rank{rank}.csv"))
    barrier()
    t0 = time.perf_counter()
    stats = []
    outs = []
    for _ in range(args.steps):
        st = L.la_stats()
        outs.append(L.la_generate(ctx.ctx, prompt, args.max_new, W_, N_, G_, stats=st))
        stats.append(st)
    barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop()

    decode_s = sum(s.decode_ns for s in stats) * 1e-9
    calls = sum(s.steps for s in stats)
    new_tokens = sum(s.tokens - 1 for s in stats)      # tokens of the packed calls (the first comes from the prefill)
    tps = new_tokens / decode_s
    call_ms = decode_s / calls * 1e3
    # aggregate over ranks: total tokens / max time
    if world > 1:
        tot_tok, max_dec, wall = aggregate_replicas(new_tokens, decode_s, wall, f"cuda:{local}")
        tps = tot_tok / max_dec

    # autoregressive decode on the same kernels
    ar_stats = []
    for _ in range(args.ar_steps):
        st = L.la_stats()
        ar = L.la_generate_ar(ctx.ctx, prompt, args.max_new, stats=st)
        ar_stats.append(st)
    ar_tps = (sum(s.tokens - 1 for s in ar_stats) / (sum(s.decode_ns for s in ar_stats) * 1e-9)) if ar_stats else None
    same = all(o == ar for o in outs) if ar_stats else None

    # Live kernel timing of the same workload (one more request, with the
    # step graph bracketing every launch by CUDA events on the library's
    # stream): the GEMM family is the dominant kernel.
    L.la_set_debug(ctx.ctx, 4)
    st_prof = L.la_stats()
    L.la_generate(ctx.ctx, prompt, args.max_new, W_, N_, G_, stats=st_prof)
    prof = L.la_profile_read(ctx.ctx)
    L.la_set_debug(ctx.ctx, 0)

    # kernels of ours launched in the timed region: per request the prefill
    # (2 chunks x (rows + embed + 8 per layer) + need + head 3 + finish), begin,
    # and per packed call pack + embed + 7 per layer (RoPE folded into the
    # attention; 8 with LA_FUSE_ROPE=0) + head 3 + publish + commit
    chunks = (PROMPT_LEN + 255) // 256
    per_layer_call = 8 if os.environ.get("LA_FUSE_ROPE", "1").startswith("0") else 7
    per_call = 2 + per_layer_call * cfg.n_layers + 3 + 2
    per_request = chunks * (2 + 8 * cfg.n_layers) + 1 + 3 + 1 + 1
    launches = args.steps * per_request + calls * per_call
    peaks, src = measured_peaks()
    mean_K = PROMPT_LEN + args.max_new / 2.0
    mean_Q = statistics.mean(s.mean_rows for s in stats)
    mean_ct = statistics.mean(s.mean_candidates for s in stats)
    bytes_call = algorithmic_bytes_per_call(cfg, mean_K, mean_Q)
    step_achieved = bytes_call / (call_ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    samples = max(1, prof["samples"])
    gemm_ms_call = prof["ms"]["gemm"] / samples
    gemm_launches_call = prof["launches"]["gemm"] / samples
    gemm_bytes = gemm_bytes_per_call(cfg, mean_Q, 1 + W_ + mean_ct * (N_ - 1))
    gemm_achieved = gemm_bytes / (gemm_ms_call * 1e-3) / 1e9 if gemm_ms_call > 0 else None
    kernel_ms_call = {k: v / samples for k, v in prof["ms"].items()}
    line = {
        "metric": "committed tokens/s @ batch 1 (7B-shape bf16)",
        "value": tps * (1 if world == 1 else 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config,
        "tokens_per_call": new_tokens / calls,
        "call_latency_ms": call_ms,
        "prefill_ms": statistics.mean(s.prefill_ns for s in stats) * 1e-6,
        "mean_rows_per_call": mean_Q,
        "ar_tokens_per_s": ar_tps,
        "speedup_vs_ar": tps / ar_tps if (world == 1 and ar_tps) else None,
        "lookahead_equals_ar": same,
        "e2e": {"value": (args.max_new * args.steps * world) / wall, "unit": "tokens/s",
                "h2d_bytes_per_step": PROMPT_LEN * 4, "d2h_bytes_per_step": args.max_new * 4},
        "roofline": {"bound": "hbm", "achieved": gemm_achieved, "peak": peak, "unit": "GB/s",
                     "frac": (gemm_achieved / peak) if gemm_achieved else None,
                     "traffic": GEMM_TRAFFIC_PER_CALL,
                     "kernel": "k_gemm_tc (tcgen05 GEMMs: QKV, O, gate/up, down per layer + LM head), "
                               "per call: algorithmic bytes / summed launch time",
                     "launches_per_call": gemm_launches_call, "ms_per_call": gemm_ms_call,
                     "algorithmic_bytes_per_call": gemm_bytes, "peak_source": src + " (copy bandwidth)",
                     "timing": f"CUDA events around each launch in the step graph, {prof['samples']} sampled steps"},
        "step_roofline": {"achieved": step_achieved, "frac": step_achieved / peak,
                          "algorithmic_bytes_per_call": bytes_call,
                          "what": "whole packed call: weights once + committed K/V read + temporary K/V written"},
        "kernel_ms_per_call": kernel_ms_call,
        "clocks": clk,
        "gpu_launches": launches,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(cfg, w)
    ctx.close()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
