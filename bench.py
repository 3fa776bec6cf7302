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
# the headline metric, printed identically by both arms
METRIC = "committed tokens/s @ batch 1 (7B-shape bf16), tokens/step, % step roofline"


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


def kernel_source_digest(files) -> str:
    """sha256 (first 16 hex digits) of the named CUDA sources, concatenated in
    order: identifies the kernel build a DRAM-traffic capture belongs to."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "lookahead_decoding_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(profile: str, files):
    """DRAM bytes per call of the dominant kernel from the committed ncu summary
    `profiles/<profile>`: its line `traffic_bytes_per_call: <bytes> source_digest:
    <digest>`.  None when the file is missing or the kernel sources have changed
    since the capture (the digest no longer matches)."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None, None
    want = kernel_source_digest(files)
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and parts[0] == "traffic_bytes_per_call:" and parts[2] == "source_digest:":
            return (float(parts[1]) if parts[3] == want else None), parts[3]
    return None, None


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

    def __init__(self, index: int):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="la_clocks_", suffix=".csv")
        os.close(fd)
        self.proc = None
        try:
            self.f = open(self.path, "w")
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
        out = parse_clocks(self.path)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        return out


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


def oracle_model(cfg, weights):
    """The oracle transformer in the configuration the CPU baseline times
    (fp32 arithmetic, bf16 storage emulation, weights converted once)."""
    import numpy as np
    from oracle.model import OracleModel
    return OracleModel(cfg, weights, compute_dtype=np.float32, store="bf16", cache_weights=True)


def cpu_oracle_sample(cfg, weights, min_s: float = 10.0, max_calls: int = 64, prompt_len: int = 24, model=None):
    """The oracle (as it stands) on the host cores: a bounded sample of the same
    workload — prefill of a short Markov prompt (not timed), then packed
    lookahead calls at W=15, N=5, G=15 until `min_s` seconds of them have run
    (at most `max_calls`); returns committed tokens/s of those calls."""
    import synth
    from oracle import lookahead as la
    from oracle.model import argmax_lowest
    m = model if model is not None else oracle_model(cfg, weights)
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
            # AR on the same context: the attention's key split is fixed per
            # context by its largest path length, so outputs are compared
            # within one context
            st = L.la_stats()
            ar_out = L.la_generate_ar(ctx.ctx, prompt, args.max_new, stats=st)
            if ar_ms is None:
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
                           "mean_candidates": st.mean_candidates, "emitted_hist": list(st.emitted_hist)[:N],
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
    clocks = ClockSampler(local)
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
    tl = batch_timeline_per_call(L, ctx, prompts, W_, N_, G_)
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
            "gpu_launches": sum(s.kernel_launches for s in stats),
            "e2e": {"value": B * args.max_new * args.steps / wall, "unit": "tokens/s",
                    "h2d_bytes_per_step": B * PROMPT_LEN * 4, "d2h_bytes_per_step": B * args.max_new * 4},
            "kernel_ms_per_call": tl["ms"], "kernel_ms_per_call_by_kernel": tl["by_kernel_ms"],
            "kernel_timing": tl["what"], "clocks": clk}
    ctx.close()
    print(json.dumps(line))


# The single-request workloads: the headline (the pages' plain configuration
# on the 7B shape); pool seeding on the same prompt and the copy-heavy 13B
# prompt, where a trained model would accept the pool's candidates (a
# random-init one does not continue the prompt's n-grams); a 7B-shape
# model whose greedy next token is nearly a function of the current token,
# where the collected n-grams come true and calls commit several tokens; and
# sampled decoding of 16 prompts (the verifier's exact rejection scheme).
WORKLOADS = {
    "headline": {"desc": "llama-7b-shape bf16, batch 1, prompt 512 Markov/Zipf(1.1), 256 new tokens, greedy, "
                         "W=15 N=5 G=15", "model": "llama-7b-shape (random init)", "prompt": "markov",
                 "prompt_len": PROMPT_LEN, "max_new": MAX_NEW, "seed": 2, "knobs": (W_, N_, G_), "options": 0,
                 "cfg": "LLAMA_7B"},
    "pool-seeded": {"desc": "llama-7b-shape bf16, batch 1, prompt 512 Markov/Zipf(1.1), 256 new tokens, greedy, "
                            "W=15 N=5 G=15, pool seeded from the prompt and every output token",
                    "model": "llama-7b-shape (random init)", "prompt": "markov", "prompt_len": PROMPT_LEN,
                    "max_new": MAX_NEW, "seed": 2, "knobs": (W_, N_, G_), "options": 3, "cfg": "LLAMA_7B"},
    "code-13b": {"desc": "llama-13b-shape bf16, batch 1, code-like prompt 2048 (30% copied 8-32-token spans), "
                         "512 new tokens, greedy, W=10 N=5 G=10", "model": "llama-13b-shape (random init)",
                 "prompt": "code", "prompt_len": 2048, "max_new": 512, "seed": 4, "knobs": (10, 5, 10),
                 "options": 0, "cfg": "LLAMA_13B"},
    "predictable-7b": {"desc": "llama-7b-shape bf16 with attention output projections scaled by 2^-10 (next token "
                               "nearly a function of the current one), batch 1, prompt 512 Markov/Zipf(1.1), "
                               "256 new tokens, greedy, W=15 N=5 G=15",
                       "model": "llama-7b-shape (random init, wo x 2^-10)", "prompt": "markov",
                       "prompt_len": PROMPT_LEN, "max_new": MAX_NEW, "seed": 2, "knobs": (W_, N_, G_), "options": 0,
                       "cfg": "LLAMA_7B", "wo_scale": 2.0 ** -10},
    "sampled-7b": {"desc": "llama-7b-shape bf16, sampling (temperature 0.8, top-p 0.9, exact verification of the "
                           "candidates), 16 prompts of 256 Markov/Zipf(1.1) tokens one after another, 256 new "
                           "tokens each, W=15 N=5 G=15",
                   "model": "llama-7b-shape (random init)", "prompt": "markov", "prompt_len": 256, "max_new": 256,
                   "seed": 40, "knobs": (W_, N_, G_), "options": 0, "cfg": "LLAMA_7B", "n_prompts": 16,
                   "sampling": (0.8, 0.9)},
}
# the nominal HBM3e bandwidth the step roofline is also quoted against
SPEC_HBM_GBS = 8000.0
# the dominant kernel of a packed call: its kind in the kernel-timing totals,
# the committed ncu summary holding its DRAM traffic, and the sources that
# summary's digest covers
DOMINANT = {"kind": "gemm", "profile": "k_gemm_tc_llama7b_decode_call.md",
            "sources": ["la_gemm_tc.cu", "la_tc.cuh", "la_common.cuh", "la_kernels.h", "la_timeline.cuh"],
            "what": "k_gemm_tc (tcgen05 GEMMs: QKV, O, gate/up, down per layer + LM head), per call: "
                    "algorithmic bytes / summed launch time"}


def timeline_per_call(L, ctx, prompt, W: int, N: int, G: int, calls: int = 16, sampling=None):
    """Per-kind device time of a packed call from the library's kernel
    timeline (global-timer stamps per CTA, no events in the graph): one more
    request, prefill untimed, then `calls` packed calls one by one; every
    instant is charged to the running CTA that finishes next, so the kinds
    add up to the calls' device time (host gaps between calls are left out)."""
    import numpy as np
    cap = 120_000 * calls
    L.la_prefill(ctx.ctx, prompt, sampling=sampling)
    L.la_timeline_start(cap)
    try:
        for _ in range(calls):
            L.la_step(ctx.ctx, W, N, G, sampling=sampling)
    finally:
        rec = L.la_timeline_stop(cap)
    split = L.timeline_split(rec)
    ms = {k: v * 1e-6 / calls for k, v in split["ns"].items() if v}
    return {"ms": ms, "by_kernel_ms": {k: v * 1e-6 / calls for k, v in split["by_kernel_ns"].items()},
            "launches_per_call": float(np.sum(1.0 / rec[:, 4])) / calls if len(rec) else 0.0,
            "what": ("split of %d packed calls' device time from per-CTA global-timer stamps (every instant "
                     "charged to the running CTA that finishes next); the kinds add up to the calls' device "
                     "time, host gaps between the calls left out" % calls)}


def split_difference(long_split, short_split, calls: int):
    """Per-call device time of the calls that separate two kernel timelines of
    the same work (`timeline_split` results): the longer run's charges minus
    the shorter run's, per kind and per kernel, over `calls` calls.  Kernels
    whose charge does not grow between the runs (the prefill's, which both
    runs share up to the timer's jitter) are left out."""
    def diff(a, b):
        return {k: (v - b.get(k, 0)) * 1e-6 / calls for k, v in a.items() if v > b.get(k, 0)}
    return {"ms": diff(long_split["ns"], short_split["ns"]),
            "by_kernel_ms": diff(long_split["by_kernel_ns"], short_split["by_kernel_ns"])}


def batch_timeline_per_call(L, ctx, prompts, W: int, N: int, G: int, short: int = 2, long: int = 18):
    """Per-kind device time of a batched packed call: the kernel timeline of
    the request set generated to `long` tokens minus the same set generated
    to `short` (the prefills and first calls are the same and cancel), over
    the calls between them."""
    splits, steps = {}, {}
    for mn in (short, long):
        cap = 200_000 * (mn + 8) * len(prompts)
        st = L.la_stats()
        L.la_timeline_start(cap)
        try:
            L.la_generate_batch(ctx.ctx, prompts, mn, W, N, G, stats=st)
        finally:
            rec = L.la_timeline_stop(cap)
        splits[mn], steps[mn] = L.timeline_split(rec), st.steps
    calls = steps[long] - steps[short]
    out = split_difference(splits[long], splits[short], calls)
    out["what"] = ("split of %d batched calls' device time from per-CTA global-timer stamps (a run to %d "
                   "tokens minus a run to %d, prefills cancelling); every instant charged to the running "
                   "CTA that finishes next" % (calls, long, short))
    return out


def run_single(args, cfg, config, wl, rank: int, local: int, world: int):
    """One request at a time through la_generate (graph per packed call):
    committed tokens/s of the decode calls, acceptance, the step roofline, AR
    on the same kernels, per-kind kernel times and the end-to-end rate."""
    import torch
    import synth
    from lookahead_decoding_gb300 import lib
    L = lib()
    W, N, G = wl["knobs"]
    max_new = args.max_new if args.workload == "headline" else wl["max_new"]
    plen = wl["prompt_len"]
    w = synth.llama_weights(cfg, 0, device=f"cuda:{local}", wo_scale=wl.get("wo_scale", 1.0))
    ctx = L.Context(cfg, w, max_ctx=max(1024, plen + max_new + 64), max_W=W, max_N=N, max_G=G)
    if wl["options"]:
        L.la_set_options(ctx.ctx, wl["options"])
    n_prompts = wl.get("n_prompts", 1)
    if wl["prompt"] == "markov":
        prompts = [synth.markov_zipf_prompt(cfg.vocab, plen, wl["seed"] + i).tolist() for i in range(n_prompts)]
    else:
        prompts = [synth.code_like_prompt(cfg.vocab, plen, wl["seed"] + i).tolist() for i in range(n_prompts)]
    prompt = prompts[0]
    temp_top_p = wl.get("sampling")       # (temperature, top_p): request i of step k draws with seed 1000 k + i

    def samp(step: int, i: int):
        return None if temp_top_p is None else (temp_top_p[0], temp_top_p[1], 1000 * step + i)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()

    for k in range(args.warmup):
        L.la_generate(ctx.ctx, prompt, max_new, W, N, G, sampling=samp(k + 100, 0))
    clocks = ClockSampler(local)
    barrier()
    t0 = time.perf_counter()
    stats = []
    outs = []
    for k in range(args.steps):
        for i, pr in enumerate(prompts):
            st = L.la_stats()
            outs.append(L.la_generate(ctx.ctx, pr, max_new, W, N, G, sampling=samp(k, i), stats=st))
            stats.append(st)
    barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop()

    decode_s = sum(s.decode_ns for s in stats) * 1e-9
    calls = sum(s.steps for s in stats)
    new_tokens = sum(s.tokens - 1 for s in stats)      # tokens of the packed calls (the first comes from the prefill)
    tps = new_tokens / decode_s
    call_ms = decode_s / calls * 1e3
    if world > 1:
        tot_tok, max_dec, wall = aggregate_replicas(new_tokens, decode_s, wall, f"cuda:{local}")
        tps = tot_tok / max_dec

    # autoregressive decode on the same kernels and context
    ar_stats = []
    ars = []
    for k in range(args.ar_steps):
        for i, pr in enumerate(prompts):
            st = L.la_stats()
            ars.append(L.la_generate_ar(ctx.ctx, pr, max_new, sampling=samp(k, i), stats=st))
            ar_stats.append(st)
    ar_tps = (sum(s.tokens - 1 for s in ar_stats) / (sum(s.decode_ns for s in ar_stats) * 1e-9)) if ar_stats else None
    ar_ms = (sum(s.decode_ns for s in ar_stats) * 1e-6 / sum(s.steps for s in ar_stats)) if ar_stats else None
    # greedy: every request's lookahead output equals its AR output (sampled
    # outputs draw differently; the verifier's law is checked by the tests)
    same = (all(outs[k * n_prompts + i] == ars[i] for k in range(args.steps) for i in range(n_prompts))
            if ar_stats and temp_top_p is None else None)

    # Live kernel timing of the same workload (one more request, with the
    # step graph bracketing every launch by CUDA events on the library's
    # stream).  The brackets serialise launches that otherwise overlap, so
    # the per-kind figures are upper bounds that need not add up to a call.
    L.la_set_debug(ctx.ctx, 4)
    st_prof = L.la_stats()
    L.la_generate(ctx.ctx, prompt, max_new, W, N, G, sampling=samp(200, 0), stats=st_prof)
    prof = L.la_profile_read(ctx.ctx)
    L.la_set_debug(ctx.ctx, 0)
    tl = timeline_per_call(L, ctx, prompt, W, N, G, sampling=samp(300, 0))

    launches = sum(s.kernel_launches for s in stats)        # counted by the library
    peaks, src = measured_peaks()
    mean_K = plen + max_new / 2.0
    mean_Q = statistics.mean(s.mean_rows for s in stats)
    mean_ct = statistics.mean(s.mean_candidates for s in stats)
    hist = [sum(s.emitted_hist[i] for s in stats) for i in range(16)]
    bytes_call = algorithmic_bytes_per_call(cfg, mean_K, mean_Q)
    step_achieved = bytes_call / (call_ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    samples = max(1, prof["samples"])
    dom = DOMINANT
    dom_ms_call = prof["ms"][dom["kind"]] / samples
    dom_launches_call = prof["launches"][dom["kind"]] / samples
    dom_bytes = gemm_bytes_per_call(cfg, mean_Q, 1 + W + mean_ct * (N - 1))
    dom_achieved = dom_bytes / (dom_ms_call * 1e-3) / 1e9 if dom_ms_call > 0 else None
    # the capture is of the full headline model's calls
    full = args.workload == "headline" and not args.layers
    traffic, digest = captured_traffic(dom["profile"], dom["sources"]) if full else (None, None)
    line = {
        "metric": METRIC if args.workload == "headline" else f"{METRIC} [{args.workload}]",
        "value": tps,
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
        "accepted_tokens_per_step": new_tokens / calls,
        "mean_candidates": mean_ct,
        "emitted_hist": hist[:N],
        "call_latency_ms": call_ms,
        "prefill_ms": statistics.mean(s.prefill_ns for s in stats) * 1e-6,
        "mean_rows_per_call": mean_Q,
        "ar_tokens_per_s": ar_tps,
        "ar_call_latency_ms": ar_ms,
        "speedup_vs_ar": tps / ar_tps if (world == 1 and ar_tps) else None,
        "lookahead_equals_ar": same,
        "e2e": {"value": (max_new * n_prompts * args.steps * world) / wall, "unit": "tokens/s",
                "h2d_bytes_per_step": n_prompts * plen * 4, "d2h_bytes_per_step": n_prompts * max_new * 4},
        "roofline": {"bound": "hbm", "achieved": dom_achieved, "peak": peak, "unit": "GB/s",
                     "frac": (dom_achieved / peak) if dom_achieved else None,
                     "traffic": traffic,
                     "traffic_source": (f"ncu capture in profiles/{dom['profile']} (kernel sources {digest})"
                                        if traffic else "no capture of this kernel build"),
                     "kernel": dom["what"],
                     "launches_per_call": dom_launches_call, "ms_per_call": dom_ms_call,
                     "algorithmic_bytes_per_call": dom_bytes, "peak_source": src + " (copy bandwidth)",
                     "timing": f"CUDA events around each launch in the step graph, {prof['samples']} sampled steps"},
        "step_roofline": {"achieved": step_achieved, "frac": step_achieved / peak,
                          "frac_of_spec_8tbs": step_achieved / SPEC_HBM_GBS,
                          "algorithmic_bytes_per_call": bytes_call,
                          "what": "whole packed call: weights once + committed K/V read + temporary K/V written"},
        "kernel_ms_per_call": tl["ms"],
        "kernel_timing": tl["what"],
        "kernel_ms_per_call_by_kernel": tl["by_kernel_ms"],
        "kernel_ms_per_call_sum": sum(tl["ms"].values()),
        "kernel_ms_bracketed_per_call": {k: v / samples for k, v in prof["ms"].items()},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if rank == 0 and not args.no_cpu_baseline and args.workload == "headline":
        line["cpu_baseline"] = cpu_oracle_sample(cfg, w)
    ctx.close()
    return line


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
    ap.add_argument("--workload", default="headline", choices=sorted(WORKLOADS),
                    help="single-request workload: the headline, or one where the pool retrieves accepted candidates")
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
        m = oracle_model(cfg, w)
        # warm-up steps: one packed call each (weights converted, caches warm)
        for _ in range(args.warmup):
            cpu_oracle_sample(cfg, w, min_s=0.0, max_calls=1, model=m)
        samples = [cpu_oracle_sample(cfg, w, min_s=8.0, model=m) for _ in range(max(1, args.steps))]
        v = statistics.mean(s["value"] for s in samples)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
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
    wl = WORKLOADS[args.workload]
    if args.workload != "headline":
        cfg = getattr(synth, wl["cfg"])
        if args.layers:
            import dataclasses
            cfg = dataclasses.replace(cfg, n_layers=args.layers)
        config = dict(config, workload=wl["desc"], model=wl["model"], seq_len=wl["prompt_len"] + wl["max_new"])
    line = run_single(args, cfg, config, wl, rank, local, world)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
