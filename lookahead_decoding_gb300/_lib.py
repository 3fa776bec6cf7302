"""ctypes binding of liblookahead (argument marshalling only).

Every function named ``la_*`` here calls the C entry point of the same name
declared in include/lookahead.h; all computation happens in the library's
CUDA kernels.  Importing this module loads ``liblookahead.so`` from the
package directory and raises if it is missing — there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblookahead.so")

LA_OK, LA_EINVAL, LA_ECAPACITY, LA_ESTATE, LA_ECUDA, LA_EDEVICE, LA_ETIMEOUT, LA_ENOTSUP = range(8)
LA_F32, LA_BF16 = 0, 1

EXPORTS = ["la_init", "la_prefill", "la_step", "la_generate", "la_generate_ar", "la_set_debug", "la_debug_logits",
           "la_debug_state", "la_debug_pool", "la_step_inject", "la_query", "la_free", "la_strerror",
           "la_last_cuda_error", "la_debug_sample_verify", "la_debug_gemm", "la_bench_gemm",
           "la_gemm_noalloc", "la_profile_read", "la_set_options", "la_init_batch", "la_generate_batch",
           "la_debug_layer", "la_debug_batch_logits", "la_debug_batch_state", "la_timeline_start",
           "la_timeline_stop"]

# pool seeding options (la_set_options)
LA_OPT_POOL_FROM_PROMPT, LA_OPT_POOL_FROM_OUTPUT, LA_OPT_SLICE_WINDOW = 1, 2, 4


class la_model_cfg(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ffn", C.c_int32), ("vocab", C.c_int32), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("dtype", C.c_int32)]


_PP = C.POINTER(C.c_void_p)


class la_weights(C.Structure):
    _fields_ = [("tok_emb", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("attn_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP), ("wo", _PP),
                ("mlp_norm", _PP), ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP)]


class la_sampling(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_p", C.c_float), ("seed", C.c_uint64)]


class la_stats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("tokens", C.c_int64), ("prefill_ns", C.c_int64), ("decode_ns", C.c_int64),
                ("emitted_hist", C.c_int32 * 16), ("mean_candidates", C.c_double), ("mean_rows", C.c_double),
                ("kernel_launches", C.c_int64)]


class LaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {code} ({strerror(code)})")
        self.code = code


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with lookahead_decoding_gb300.build.build()")
    lib = C.CDLL(LIB_PATH)
    i32p = C.POINTER(C.c_int32)
    f32p = C.POINTER(C.c_float)
    vp = C.c_void_p
    sig = {
        "la_init": (C.c_int, [C.POINTER(la_model_cfg), C.POINTER(la_weights), C.c_int, C.c_int, C.c_int, C.c_int, vp,
                              C.POINTER(vp)]),
        "la_init_batch": (C.c_int, [C.POINTER(la_model_cfg), C.POINTER(la_weights), C.c_int, C.c_int, C.c_int,
                                    C.c_int, C.c_int, vp, C.POINTER(vp)]),
        "la_generate_batch": (C.c_int, [vp, C.c_int, i32p, i32p, C.c_int, C.c_int, C.c_int, C.c_int,
                                        C.POINTER(la_sampling), i32p, C.POINTER(la_stats)]),
        "la_prefill": (C.c_int, [vp, i32p, C.c_int, C.POINTER(la_sampling), i32p]),
        "la_step": (C.c_int, [vp, C.c_int, C.c_int, C.c_int, C.POINTER(la_sampling), i32p, C.POINTER(C.c_int)]),
        "la_generate": (C.c_int, [vp, i32p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(la_sampling), i32p,
                                  C.POINTER(C.c_int), C.POINTER(la_stats)]),
        "la_generate_ar": (C.c_int, [vp, i32p, C.c_int, C.c_int, C.POINTER(la_sampling), i32p, C.POINTER(C.c_int),
                                     C.POINTER(la_stats)]),
        "la_set_debug": (C.c_int, [vp, C.c_int]),
        "la_set_options": (C.c_int, [vp, C.c_uint32]),
        "la_profile_read": (C.c_int, [vp, C.POINTER(C.c_double), C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
        "la_timeline_start": (C.c_int, [C.c_int64]),
        "la_timeline_stop": (C.c_int, [C.POINTER(C.c_int64), C.c_int64, C.POINTER(C.c_int64)]),
        "la_debug_logits": (C.c_int, [vp, f32p, i32p, C.c_int, C.POINTER(C.c_int)]),
        "la_debug_layer": (C.c_int, [vp, C.c_int, C.c_int, vp, C.c_int]),
        "la_debug_batch_logits": (C.c_int, [vp, C.c_int, f32p, i32p, C.c_int, C.POINTER(C.c_int)]),
        "la_debug_state": (C.c_int, [vp, i32p, i32p, i32p, i32p, i32p, i32p]),
        "la_debug_batch_state": (C.c_int, [vp, C.c_int, i32p, i32p, i32p, i32p, i32p, i32p]),
        "la_debug_pool": (C.c_int, [vp, C.c_int, i32p, C.POINTER(C.c_int)]),
        "la_step_inject": (C.c_int, [vp, C.c_int, C.c_int, C.c_int, C.POINTER(la_sampling), C.c_int, i32p, f32p, i32p,
                                     C.POINTER(C.c_int)]),
        "la_query": (C.c_int, [vp, i32p]),
        "la_bench_gemm": (C.c_int, [C.c_int] * 8 + [f32p]),
        "la_gemm_noalloc": (C.c_int, [C.c_int, vp, vp, C.c_int, C.c_int, vp, C.c_int, vp, vp]),
        "la_debug_gemm": (C.c_int, [C.c_int, C.POINTER(C.c_uint16), C.POINTER(C.c_uint16), C.c_int, C.c_int, C.c_int,
                                    C.POINTER(C.c_uint16), C.c_int, C.c_int, f32p]),
        "la_debug_sample_verify": (C.c_int, [f32p, C.c_int, C.c_int, i32p, C.c_int, C.c_int, C.POINTER(la_sampling),
                                             C.c_int, i32p]),
        "la_free": (None, [vp]),
        "la_strerror": (C.c_char_p, [C.c_int]),
        "la_last_cuda_error": (C.c_char_p, [vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()


def strerror(code: int) -> str:
    return LIB.la_strerror(code).decode()


def _i32(a) -> Tuple[np.ndarray, C.POINTER(C.c_int32)]:
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data_as(C.POINTER(C.c_int32))


def _check(code: int, what: str, ctx=None) -> None:
    if code != LA_OK:
        msg = what
        if ctx is not None and code == LA_ECUDA:
            msg += " [" + LIB.la_last_cuda_error(ctx).decode() + "]"
        raise LaError(code, msg)


def _sampling(s) -> Optional[la_sampling]:
    if s is None:
        return None
    if isinstance(s, la_sampling):
        return s
    t, p, seed = s
    return la_sampling(float(t), float(p), int(seed))


# ---------------------------------------------------------------------------
# entry points with the C names
# ---------------------------------------------------------------------------

def la_init(cfg: la_model_cfg, weights: la_weights, max_ctx: int, max_W: int, max_N: int, max_G: int,
            stream: int = 0, max_batch: int = 1):
    ctx = C.c_void_p()
    if max_batch == 1:
        code = LIB.la_init(C.byref(cfg), C.byref(weights), max_ctx, max_W, max_N, max_G, C.c_void_p(stream or None),
                           C.byref(ctx))
    else:
        code = LIB.la_init_batch(C.byref(cfg), C.byref(weights), max_ctx, max_W, max_N, max_G, max_batch,
                                 C.c_void_p(stream or None), C.byref(ctx))
    _check(code, "la_init")
    return ctx


def la_generate_batch(ctx, prompts: Sequence[Sequence[int]], max_new: int, W: int, N: int, G: int,
                      sampling=None, stats: Optional[la_stats] = None) -> List[List[int]]:
    """Lookahead of several prompts in batched packed calls (request b samples with seed + b)."""
    B = len(prompts)
    flat = np.ascontiguousarray(np.concatenate([np.asarray(p, dtype=np.int32) for p in prompts]))
    lengths = np.ascontiguousarray(np.asarray([len(p) for p in prompts], dtype=np.int32))
    out = np.zeros(B * max_new, dtype=np.int32)
    i32 = C.POINTER(C.c_int32)
    s = _sampling(sampling)
    _check(LIB.la_generate_batch(ctx, B, flat.ctypes.data_as(i32), lengths.ctypes.data_as(i32), max_new, W, N, G,
                                 C.byref(s) if s else None, out.ctypes.data_as(i32),
                                 C.byref(stats) if stats is not None else None),
           "la_generate_batch", ctx)
    return [out[b * max_new:(b + 1) * max_new].tolist() for b in range(B)]


def la_set_options(ctx, flags: int) -> None:
    """Pool seeding and window schedule (LA_OPT_* bits) for requests started after this call."""
    _check(LIB.la_set_options(ctx, flags), "la_set_options", ctx)


def la_prefill(ctx, prompt: Sequence[int], sampling=None) -> int:
    arr, p = _i32(prompt)
    tok = C.c_int32()
    s = _sampling(sampling)
    _check(LIB.la_prefill(ctx, p, len(arr), C.byref(s) if s else None, C.byref(tok)), "la_prefill", ctx)
    return int(tok.value)


def la_step(ctx, W: int, N: int, G: int, sampling=None) -> List[int]:
    out = (C.c_int32 * 16)()
    n = C.c_int()
    s = _sampling(sampling)
    _check(LIB.la_step(ctx, W, N, G, C.byref(s) if s else None, out, C.byref(n)), "la_step", ctx)
    return [int(out[i]) for i in range(n.value)]


def la_generate(ctx, prompt, max_new: int, W: int, N: int, G: int, sampling=None, stats: Optional[la_stats] = None):
    arr, p = _i32(prompt)
    out = np.zeros(max_new, dtype=np.int32)
    n = C.c_int()
    s = _sampling(sampling)
    _check(LIB.la_generate(ctx, p, len(arr), max_new, W, N, G, C.byref(s) if s else None,
                           out.ctypes.data_as(C.POINTER(C.c_int32)), C.byref(n),
                           C.byref(stats) if stats is not None else None), "la_generate", ctx)
    return out[: n.value].tolist()


def la_generate_ar(ctx, prompt, max_new: int, sampling=None, stats: Optional[la_stats] = None):
    arr, p = _i32(prompt)
    out = np.zeros(max_new, dtype=np.int32)
    n = C.c_int()
    s = _sampling(sampling)
    _check(LIB.la_generate_ar(ctx, p, len(arr), max_new, C.byref(s) if s else None,
                              out.ctypes.data_as(C.POINTER(C.c_int32)), C.byref(n),
                              C.byref(stats) if stats is not None else None), "la_generate_ar", ctx)
    return out[: n.value].tolist()


def la_query(ctx) -> Dict[str, int]:
    v = (C.c_int32 * 8)()
    _check(LIB.la_query(ctx, v), "la_query")
    keys = ["Qmax", "max_W", "max_N", "max_G", "max_ctx", "vocab", "LMAX", "PMAX"]
    return {k: int(v[i]) for i, k in enumerate(keys)}


def la_set_debug(ctx, flags: int) -> None:
    _check(LIB.la_set_debug(ctx, flags), "la_set_debug")


PROFILE_KINDS = ("gemm", "attention", "rowwise", "state")


def la_profile_read(ctx) -> Dict[str, object]:
    """Kernel-timing totals since the last read (see la_set_debug bit 2)."""
    ms = (C.c_double * 4)()
    n = (C.c_int64 * 4)()
    samples = C.c_int64()
    _check(LIB.la_profile_read(ctx, ms, n, C.byref(samples)), "la_profile_read", ctx)
    return {"ms": dict(zip(PROFILE_KINDS, list(ms))), "launches": dict(zip(PROFILE_KINDS, list(n))),
            "samples": int(samples.value)}


TIMELINE_KINDS = ("gemm", "attention", "rowwise", "state", "chain")
# kernel ids of the timeline records and the kind of each
TIMELINE_IDS = (("k_gemm_tc", "gemm"), ("k_gemm_ffma", "gemm"), ("k_attn_fused", "attention"),
                ("k_attention", "attention"), ("k_embed", "rowwise"), ("k_rmsnorm", "rowwise"),
                ("k_rope_kv", "rowwise"), ("k_rope_kv4", "rowwise"), ("k_swiglu_split", "rowwise"),
                ("k_argmax_rows", "rowwise"), ("k_argmax_reduce", "rowwise"), ("k_sample_verify", "state"),
                ("k_begin", "state"), ("k_pack", "state"), ("k_pool_seed", "state"), ("k_publish", "state"),
                ("k_commit_kv", "state"), ("k_inject_map", "state"), ("k_prefill_rows", "state"),
                ("k_prefill_need", "state"), ("k_prefill_finish", "state"), ("k_mega", "chain"))


def la_timeline_start(max_ctas: int) -> None:
    """Opens the process-wide kernel timeline for up to max_ctas CTA records."""
    _check(LIB.la_timeline_start(int(max_ctas)), "la_timeline_start")


def la_timeline_stop(cap: int) -> np.ndarray:
    """Closes the timeline: int64 [CTAs, 5] = (start ns, end ns, kernel id,
    CTA, CTAs of the grid), in start order.  Raises if records were lost."""
    rec = np.zeros((max(1, cap), 5), dtype=np.int64)
    n = C.c_int64()
    _check(LIB.la_timeline_stop(rec.ctypes.data_as(C.POINTER(C.c_int64)), int(cap), C.byref(n)), "la_timeline_stop")
    if n.value > cap:
        raise RuntimeError(f"la_timeline_stop: {n.value} CTAs recorded, room for {cap}")
    return rec[:n.value]


def timeline_split(rec: np.ndarray) -> Dict[str, object]:
    """Splits the device time of a timeline (rows in start order) by kernel:
    every instant at which some CTA runs is charged to the running CTA that
    finishes next; instants with none running are idle.  The charges plus
    idle add up to the span from the first start to the last end."""
    import heapq
    by_id = {name: 0 for name, _ in TIMELINE_IDS}
    ctas = {name: 0 for name, _ in TIMELINE_IDS}
    idle = 0
    rows = [(int(a), max(int(a), int(b)), int(k)) for a, b, k in rec[:, :3].tolist()] if len(rec) else []
    heap: List[tuple] = []
    i, n = 0, len(rows)
    t = rows[0][0] if n else 0
    while i < n or heap:
        if not heap:
            if rows[i][0] > t:
                idle += rows[i][0] - t
                t = rows[i][0]
        while i < n and rows[i][0] <= t:
            heapq.heappush(heap, (rows[i][1], rows[i][2]))
            ctas[TIMELINE_IDS[rows[i][2]][0]] += 1
            i += 1
        if not heap:
            continue
        end, k = heap[0]
        nxt = rows[i][0] if i < n else None
        if nxt is not None and nxt < end:
            by_id[TIMELINE_IDS[k][0]] += nxt - t
            t = nxt
        else:
            by_id[TIMELINE_IDS[k][0]] += end - t
            t = end
            heapq.heappop(heap)
            while heap and heap[0][0] <= t:
                heapq.heappop(heap)
    ns = {k: 0 for k in TIMELINE_KINDS}
    for name, kind in TIMELINE_IDS:
        ns[kind] += by_id[name]
    span = (max(r[1] for r in rows) - rows[0][0]) if n else 0
    return {"ns": ns, "by_kernel_ns": {k: v for k, v in by_id.items() if ctas[k]},
            "ctas": {k: v for k, v in ctas.items() if v}, "idle_ns": idle, "span_ns": span}


def la_debug_logits(ctx, cap_rows: int, vocab: int):
    logits = np.zeros((cap_rows, vocab), dtype=np.float32)
    rows = np.zeros(cap_rows, dtype=np.int32)
    n = C.c_int()
    _check(LIB.la_debug_logits(ctx, logits.ctypes.data_as(C.POINTER(C.c_float)),
                               rows.ctypes.data_as(C.POINTER(C.c_int32)), cap_rows, C.byref(n)), "la_debug_logits", ctx)
    return logits[: n.value], rows[: n.value]


def la_debug_batch_logits(ctx, b: int, cap_rows: int, vocab: int):
    """Request b's needed-row logits of the last batched call and their packed
    indices within the request (needs debug bit 0)."""
    logits = np.zeros((cap_rows, vocab), dtype=np.float32)
    rows = np.zeros(cap_rows, dtype=np.int32)
    n = C.c_int()
    _check(LIB.la_debug_batch_logits(ctx, b, logits.ctypes.data_as(C.POINTER(C.c_float)),
                                     rows.ctypes.data_as(C.POINTER(C.c_int32)), cap_rows, C.byref(n)),
           "la_debug_batch_logits", ctx)
    return logits[: n.value], rows[: n.value]


def la_debug_layer(ctx, layer: int, what: int, rows: int, width: int, bf16: bool = True):
    """Rows of one storage point of `layer` in the last pass (see the header):
    what 0 the fp32 residual input (float32 array), 1 the attention output,
    2 the normalised MLP input, 3 the SwiGLU output (float64 arrays of the
    stored bf16 values, or float32 for an fp32 model); needs debug bit 3."""
    if what == 0:
        x = np.zeros((rows, width), dtype=np.float32)
    else:
        x = np.zeros((rows, width), dtype=np.uint16 if bf16 else np.float32)
    _check(LIB.la_debug_layer(ctx, layer, what, x.ctypes.data, rows), "la_debug_layer", ctx)
    if what != 0 and bf16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x


def la_debug_hidden(ctx, layer: int, rows: int, d_model: int):
    """fp32 residual rows [rows][d_model] at the input of `layer` (debug bit 3)."""
    return la_debug_layer(ctx, layer, 0, rows, d_model)


HDR_KEYS = ["K", "x_t", "W", "N", "G", "n_levels", "step", "Q", "C_t", "a", "winner", "n_out", "err", "steady",
            "n_need", "n_deep"]


def la_debug_state(ctx, b: Optional[int] = None):
    """Header, window levels and the last call's rows (tokens, positions,
    metadata); b: request b of a batched context."""
    q = la_query(ctx)
    R = q["max_N"] - 1
    hdr = np.zeros(16, dtype=np.int32)
    levels = np.zeros((R, q["LMAX"]), dtype=np.int32)
    lens = np.zeros(R, dtype=np.int32)
    tok = np.zeros(q["Qmax"], dtype=np.int32)
    pos = np.zeros(q["Qmax"], dtype=np.int32)
    meta = np.zeros(q["Qmax"], dtype=np.int32)
    P = lambda a: a.ctypes.data_as(C.POINTER(C.c_int32))
    if b is None:
        _check(LIB.la_debug_state(ctx, P(hdr), P(levels), P(lens), P(tok), P(pos), P(meta)), "la_debug_state", ctx)
    else:
        _check(LIB.la_debug_batch_state(ctx, b, P(hdr), P(levels), P(lens), P(tok), P(pos), P(meta)),
               "la_debug_batch_state", ctx)
    h = dict(zip(HDR_KEYS, hdr.tolist()))
    lv = [levels[r, : lens[r]].tolist() if r < h["n_levels"] else None for r in range(R)]
    Q = h["Q"]
    return h, lv, tok[:Q].tolist(), pos[:Q].tolist(), meta[:Q].tolist()


def la_debug_pool(ctx, key: int):
    """The bucket of `key`, oldest first, as tuples of the request's N-1 ids."""
    q = la_query(ctx)
    G, S = max(1, q["max_G"]), q["max_N"] - 1
    h = la_debug_state(ctx)[0]
    s_req = h["N"] - 1 if h["N"] >= 3 else S
    buf = np.zeros((G, S), dtype=np.int32)
    n = C.c_int()
    _check(LIB.la_debug_pool(ctx, key, buf.ctypes.data_as(C.POINTER(C.c_int32)), C.byref(n)), "la_debug_pool", ctx)
    return [tuple(r[:s_req]) for r in buf[: n.value].tolist()]


def la_step_inject(ctx, W: int, N: int, G: int, argmax: Sequence[int], sampling=None, logits=None) -> List[int]:
    arr, p = _i32(argmax)
    out = (C.c_int32 * 16)()
    n = C.c_int()
    s = _sampling(sampling)
    lp = None
    if logits is not None:
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        lp = lg.ctypes.data_as(C.POINTER(C.c_float))
    _check(LIB.la_step_inject(ctx, W, N, G, C.byref(s) if s else None, len(arr), p, lp, out, C.byref(n)),
           "la_step_inject", ctx)
    return [int(out[i]) for i in range(n.value)]


def la_debug_sample_verify(logits, cands, sampling, n_trials: int):
    """n_trials verifications of the same rows; returns an int32 array [n_trials][S+3]
    of (E, a, emitted ids padded with -1)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    rows, V = lg.shape
    c = np.ascontiguousarray(np.asarray(cands, dtype=np.int32).reshape(len(cands), -1)) if len(cands) else \
        np.zeros((0, 1), dtype=np.int32)
    Ct, S = c.shape[0], (c.shape[1] if len(cands) else 1)
    out = np.zeros((n_trials, S + 3), dtype=np.int32)
    s = _sampling(sampling)
    _check(LIB.la_debug_sample_verify(lg.ctypes.data_as(C.POINTER(C.c_float)), rows, V,
                                      c.ctypes.data_as(C.POINTER(C.c_int32)), Ct, S, C.byref(s), n_trials,
                                      out.ctypes.data_as(C.POINTER(C.c_int32))), "la_debug_sample_verify")
    return out


def _bf16_bits(a):
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(a.contiguous().view(torch.int16).numpy().view(np.uint16))
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint16))


GEMM_STORE, GEMM_RESID, GEMM_SWIGLU, GEMM_LOGITS = 0, 1, 2, 3


def la_debug_gemm(w_bf16, x_bf16, n_cta: int = 0, mode: int = GEMM_LOGITS, w2_bf16=None, n_seg: int = 1,
                  y_in=None):
    """The tensor-core GEMM with one epilogue on bf16 CPU tensors (see the header);
    n_cta persistent CTAs (0 = one per SM)."""
    wb, xb = _bf16_bits(w_bf16), _bf16_bits(x_bf16)
    n_out, K = wb.shape
    rows = xb.shape[0]
    y = np.zeros((rows, n_out), dtype=np.float32) if y_in is None else np.array(y_in, dtype=np.float32, order="C")
    w2b = _bf16_bits(w2_bf16) if w2_bf16 is not None else None
    P16 = C.POINTER(C.c_uint16)
    _check(LIB.la_debug_gemm(mode, wb.ctypes.data_as(P16), w2b.ctypes.data_as(P16) if w2b is not None else None,
                             n_seg, n_out, K, xb.ctypes.data_as(P16), rows, n_cta,
                             y.ctypes.data_as(C.POINTER(C.c_float))), "la_debug_gemm")
    return y


def la_bench_gemm(mode: int, n_out: int, K: int, rows: int, n_cta: int = 0, n_copies: int = 8,
                  reps: int = 20, packed: int = 1) -> float:
    """Mean device microseconds of one tensor-core GEMM launch (see the header)."""
    us = C.c_float()
    _check(LIB.la_bench_gemm(mode, n_out, K, rows, n_cta, n_copies, reps, packed, C.byref(us)), "la_bench_gemm")
    return float(us.value)


def la_gemm_noalloc(mode: int, w_ptr: int, w2_ptr: Optional[int], n_out: int, K: int, x_ptr: int, rows: int,
                    y_ptr: int, stream: Optional[int] = None) -> None:
    """The tensor-core GEMM on caller-owned device buffers (raw device
    addresses), with no device allocation (see the header)."""
    _check(LIB.la_gemm_noalloc(mode, w_ptr, w2_ptr, n_out, K, x_ptr, rows, y_ptr, stream), "la_gemm_noalloc")


def la_free(ctx) -> None:
    LIB.la_free(ctx)


# ---------------------------------------------------------------------------
# convenience: a context built from a dict of torch weight tensors
# ---------------------------------------------------------------------------

class Context:
    """Owns one la_ctx; ``weights`` maps the tensor names tok_emb, lm_head,
    final_norm and l{i}.{attn_norm,wq,wk,wv,wo,mlp_norm,w_gate,w_up,w_down} to
    CUDA tensors in the model dtype (kept referenced for the context's life)."""

    def __init__(self, cfg, weights: Dict[str, "object"], max_ctx: int, max_W: int, max_N: int, max_G: int,
                 stream: int = 0, max_batch: int = 1):
        dt = LA_F32 if cfg.dtype == "f32" else LA_BF16
        self.cfg = la_model_cfg(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn,
                                cfg.vocab, cfg.rms_eps, cfg.rope_theta, dt)
        self._keep = weights
        L = cfg.n_layers

        def ptrs(name):
            arr = (C.c_void_p * L)(*[weights[f"l{l}.{name}"].data_ptr() for l in range(L)])
            self._arrays.append(arr)
            return C.cast(arr, _PP)

        self._arrays = []
        self.w = la_weights(weights["tok_emb"].data_ptr(), weights["lm_head"].data_ptr(),
                            weights["final_norm"].data_ptr(), ptrs("attn_norm"), ptrs("wq"), ptrs("wk"), ptrs("wv"),
                            ptrs("wo"), ptrs("mlp_norm"), ptrs("w_gate"), ptrs("w_up"), ptrs("w_down"))
        self.ctx = la_init(self.cfg, self.w, max_ctx, max_W, max_N, max_G, stream, max_batch)
        self.vocab = cfg.vocab

    def close(self):
        if self.ctx:
            la_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
