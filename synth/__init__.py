"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the bench.

This module draws random numbers and nothing else: it holds none of the
lookahead method's arithmetic (no model, no window, no pool, no verifier).
Both sides of every parity check receive the *same bytes* from it.

Generators
----------
* ``hash32`` — a counter-based 32-bit hash (two rounds of the MurmurHash3
  32-bit finaliser over a keyed counter).  It is written with int64 tensor
  arithmetic whose intermediate values never exceed 2**50, so it gives the
  same integers on any torch device.
* ``uniform53`` / ``normal`` — 53-bit uniforms in (0,1) from two hashes, and
  standard normals by the Box–Muller transform (cosine branch) in float64.
* ``llama_weights`` — random-init Llama-style weights, N(0, std) for every
  matrix, ones for the RMSNorm gains, generated in float64 and rounded once to
  the storage dtype (fp32 or bf16, round-to-nearest-even by torch).
* ``uniform_prompt`` / ``markov_zipf_prompt`` / ``code_like_prompt`` — token
  sequences with the statistics of the workloads (uniform ids; an order-2
  Markov chain whose next-token rank follows a Zipf(s) law truncated at V;
  the same chain with copied earlier spans).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List

import numpy as np
import torch

_M32 = 0xFFFFFFFF


def _mul32(a: torch.Tensor, c: int) -> torch.Tensor:
    """(a * c) mod 2**32 for int64 tensors a in [0, 2**32) without overflow."""
    c_lo = c & 0xFFFF
    c_hi = (c >> 16) & 0xFFFF
    lo = a * c_lo                       # < 2**48
    hi = (a * c_hi) & 0xFFFF            # only the low 16 bits survive the shift
    return (lo + (hi << 16)) & _M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def _key(seed: int, stream: int) -> int:
    """Python-int key for (seed, stream); mixes with the same finaliser."""
    k = (seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x27D4EB2F) & _M32
    t = torch.tensor([k], dtype=torch.int64)
    return int(_fmix32(t)[0])


def hash32(seed: int, stream: int, counter: torch.Tensor) -> torch.Tensor:
    """Counter-based hash: int64 tensor of values in [0, 2**32).

    ``counter`` is an int64 tensor of non-negative values below 2**48.
    """
    k1 = _key(seed, stream)
    k2 = _key(seed ^ 0x5BD1E995, stream + 0x3C6EF372)
    lo = counter & _M32
    hi = counter >> 32
    h = _fmix32(lo ^ k1)
    h = _fmix32(h ^ hi ^ k2)
    return h


def uniform53(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """n float64 uniforms in (0,1) for counters start .. start+n-1."""
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    h1 = hash32(seed, stream, 2 * i)
    h2 = hash32(seed, stream, 2 * i + 1)
    num = (h1 >> 5).to(torch.float64) * 67108864.0 + (h2 >> 6).to(torch.float64) + 0.5
    return num * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """n float64 standard normals (Box–Muller, cosine branch)."""
    u1 = uniform53(seed, stream, 2 * start, 2 * n, device)
    a = u1[0::2]
    b = u1[1::2]
    return torch.sqrt(-2.0 * torch.log(a)) * torch.cos((2.0 * math.pi) * b)


# --------------------------------------------------------------------------
# model shapes and weights
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    d_model: int
    n_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    dtype: str = "bf16"          # storage dtype of weights: "f32" or "bf16"
    init_std: float = 0.02

    @property
    def n_kv_heads(self) -> int:
        return self.n_heads


TINY = ModelConfig(n_layers=2, d_model=128, n_heads=4, head_dim=32, d_ffn=512, vocab=512, dtype="f32")
LLAMA_7B = ModelConfig(n_layers=32, d_model=4096, n_heads=32, head_dim=128, d_ffn=11008, vocab=32000)
LLAMA_13B = ModelConfig(n_layers=40, d_model=5120, n_heads=40, head_dim=128, d_ffn=13824, vocab=32000)


def weight_names(cfg: ModelConfig) -> List[str]:
    """Fixed tensor order; the i-th name uses hash stream 1000+i."""
    names = ["tok_emb"]
    for l in range(cfg.n_layers):
        names += [f"l{l}.attn_norm", f"l{l}.wq", f"l{l}.wk", f"l{l}.wv", f"l{l}.wo",
                  f"l{l}.mlp_norm", f"l{l}.w_gate", f"l{l}.w_up", f"l{l}.w_down"]
    names += ["final_norm", "lm_head"]
    return names


def weight_shape(cfg: ModelConfig, name: str):
    d, f, v = cfg.d_model, cfg.d_ffn, cfg.vocab
    hd = cfg.n_heads * cfg.head_dim
    base = name.split(".")[-1]
    return {
        "tok_emb": (v, d), "lm_head": (v, d), "final_norm": (d,),
        "attn_norm": (d,), "mlp_norm": (d,),
        "wq": (hd, d), "wk": (hd, d), "wv": (hd, d), "wo": (d, hd),
        "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f),
    }[base]


def _torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_weight(cfg: ModelConfig, name: str, seed: int = 0, device="cpu",
                chunk: int = 1 << 24) -> torch.Tensor:
    """One weight tensor in storage dtype on ``device``."""
    shape = weight_shape(cfg, name)
    dt = _torch_dtype(cfg.dtype)
    if name.endswith("norm"):
        return torch.ones(shape, dtype=dt, device=device)
    stream = 1000 + weight_names(cfg).index(name)
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=dt, device=device)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        out[s:s + m] = (normal(seed, stream, s, m, device) * cfg.init_std).to(dt)
    return out.view(shape)


def llama_weights(cfg: ModelConfig, seed: int = 0, device="cpu", wo_scale: float = 1.0) -> Dict[str, torch.Tensor]:
    """Every weight of the model.  ``wo_scale`` (a power of two, so the
    stored values are the unscaled ones scaled exactly) multiplies the
    attention output projections: at 2**-10 the attention adds almost
    nothing to the residual stream, and the greedy next token becomes nearly
    a function of the current token alone -- a random map whose walks run
    into cycles, so the n-grams a lookahead window collects come true."""
    m, e = math.frexp(wo_scale)
    assert m == 0.5 and -40 < e <= 1, "wo_scale must be a power of two"
    w = {n: make_weight(cfg, n, seed, device) for n in weight_names(cfg)}
    if wo_scale != 1.0:
        for n in w:
            if n.endswith(".wo"):
                w[n].mul_(wo_scale)
    return w


# --------------------------------------------------------------------------
# prompts
# --------------------------------------------------------------------------

def _hash_np(seed: int, stream: int, counters) -> np.ndarray:
    c = torch.as_tensor(np.asarray(counters, dtype=np.int64))
    return hash32(seed, stream, c).numpy().astype(np.uint64)


def uniform_prompt(vocab: int, n: int, seed: int) -> np.ndarray:
    """n token ids uniform over [0, vocab)."""
    u = uniform53(seed, 1, 0, n).numpy()
    return np.minimum((u * vocab).astype(np.int64), vocab - 1).astype(np.int32)


class MarkovZipf:
    """Order-2 Markov chain: rank r ~ Zipf(s) on 1..V, token = (r*A + h(a,b)) mod V."""

    def __init__(self, vocab: int, seed: int, s: float = 1.1, A: int = 7919):
        assert math.gcd(A, vocab) == 1
        self.V, self.seed, self.A = vocab, seed, A
        w = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
        self.cdf = np.cumsum(w) / w.sum()
        self.ctr = 0

    def _u(self) -> float:
        u = float(uniform53(self.seed, 2, self.ctr, 1)[0])
        self.ctr += 1
        return u

    def first_two(self):
        return [min(int(self._u() * self.V), self.V - 1) for _ in range(2)]

    def next(self, a: int, b: int) -> int:
        r = int(np.searchsorted(self.cdf, self._u(), side="left")) + 1
        r = min(r, self.V)
        h = int(_hash_np(self.seed, 3, [a * self.V + b])[0])
        return int((r * self.A + h) % self.V)


def markov_zipf_prompt(vocab: int, n: int, seed: int, s: float = 1.1) -> np.ndarray:
    mc = MarkovZipf(vocab, seed, s)
    toks = mc.first_two()[:n]
    while len(toks) < n:
        toks.append(mc.next(toks[-2], toks[-1]))
    return np.asarray(toks, dtype=np.int32)


def code_like_prompt(vocab: int, n: int, seed: int, copy_frac: float = 0.3,
                     span_lo: int = 8, span_hi: int = 32) -> np.ndarray:
    """Markov text where a fraction ``copy_frac`` of tokens is copied from earlier spans.

    At each point a copy starts with probability q = f / ((1-f) E[L] + f), which
    makes the expected copied fraction f for span length L ~ U{lo..hi}.
    """
    mc = MarkovZipf(vocab, seed)
    EL = 0.5 * (span_lo + span_hi)
    q = copy_frac / ((1.0 - copy_frac) * EL + copy_frac)
    toks = mc.first_two()[:n]
    copied = 0
    while len(toks) < n:
        t = len(toks)
        if mc._u() < q:
            L = span_lo + min(int(mc._u() * (span_hi - span_lo + 1)), span_hi - span_lo)
            if t >= L:
                s0 = min(int(mc._u() * (t - L + 1)), t - L)
                span = toks[s0:s0 + L][: n - t]
                toks.extend(span)
                copied += len(span)
                continue
        toks.append(mc.next(toks[-2], toks[-1]))
    arr = np.asarray(toks, dtype=np.int32)
    code_like_prompt.last_copied_fraction = copied / max(1, n)
    return arr
