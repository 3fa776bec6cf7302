"""Plain decoder-only Llama-style forward on the CPU (oracle; test infrastructure).

The pages run one unchanged causal target model; they do not print its
equations, so the textbook Llama block is taken (reading recorded with the
design notes):

    x   = E[tok]
    h   = x + Wo . Attn(RoPE(Wq . rms(x)), RoPE(Wk . rms(x)), Wv . rms(x))
    x'  = h + Wdown . (silu(Wgate . rms(h)) * (Wup . rms(h)))
    logits = Whead . rms(x_final)

RMSNorm: y = x / sqrt(mean(x^2) + eps) * g.
RoPE: rotate-half pairing (i, i + d_h/2), angle = pos * theta^(-2i/d_h).
Attention: softmax(q.k / sqrt(d_h)) over the keys a row may see.

The visibility of the new rows is an explicit boolean relation (prefix keys
are always visible), so the same forward serves the autoregressive step,
the packed lookahead call with a dense mask (M7.3 §0x07A, dense packed
mask), the packed call with a metadata predicate, the separate-forwards
schedule (§0x07A, separate forwards) and, through ``forward_many``, several
requests in one call (each request's rows against its own cache and rows).

Arithmetic is float64 unless ``compute_dtype`` says otherwise.  With
``store="bf16"`` values are rounded to bf16 (round-to-nearest-even through
float32) at the points where the CUDA path stores bf16: the normalised
GEMM inputs, q/k/v before and after RoPE, the attention output and the
SwiGLU product.  The residual stream and the logits are never rounded.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np

try:  # torch is only used to read tensors handed in by the caller
    import torch
except Exception:  # pragma: no cover
    torch = None


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even) via float32 bits."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(x.dtype if hasattr(x, "dtype") else np.float64)


def _to_numpy(t, dtype) -> np.ndarray:
    if torch is not None and isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64 if dtype == np.float64 else torch.float32).numpy()
    return np.asarray(t, dtype=dtype)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half pairing.  x: [n, H, dh], pos: [n]."""
    dh = x.shape[-1]
    half = dh // 2
    i = np.arange(half, dtype=np.float64)
    inv = theta ** (-2.0 * i / dh)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]       # [n, half]
    c = np.cos(ang)[:, None, :].astype(x.dtype)
    s = np.sin(ang)[:, None, :].astype(x.dtype)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


class KVCache:
    """Committed K/V rows per layer, indexed by logical position 0..len-1."""

    def __init__(self, n_layers: int):
        self.k: List[Optional[np.ndarray]] = [None] * n_layers
        self.v: List[Optional[np.ndarray]] = [None] * n_layers

    def __len__(self) -> int:
        return 0 if self.k[0] is None else self.k[0].shape[0]

    def append(self, layer_k: List[np.ndarray], layer_v: List[np.ndarray]) -> None:
        for l in range(len(self.k)):
            if self.k[l] is None:
                self.k[l], self.v[l] = layer_k[l].copy(), layer_v[l].copy()
            else:
                self.k[l] = np.concatenate([self.k[l], layer_k[l]], axis=0)
                self.v[l] = np.concatenate([self.v[l], layer_v[l]], axis=0)

    def copy(self) -> "KVCache":
        c = KVCache(len(self.k))
        c.k = [None if a is None else a.copy() for a in self.k]
        c.v = [None if a is None else a.copy() for a in self.v]
        return c


class OracleModel:
    """Llama-style decoder with weights from a name -> tensor mapping.

    ``weights`` holds the names produced by ``synth.weight_names``; values may
    be numpy arrays or torch tensors on any device (read once per use, so very
    large models are converted layer by layer and never held in float64 at
    once unless ``cache_weights`` is set).
    """

    def __init__(self, cfg, weights: Dict[str, object], compute_dtype=np.float64,
                 store: Optional[str] = None, cache_weights: Optional[bool] = None):
        self.cfg = cfg
        self.dt = compute_dtype
        self.store = store
        self._src = weights
        if cache_weights is None:
            cache_weights = cfg.d_model * cfg.d_model * cfg.n_layers <= (1 << 24)
        self._cache: Optional[Dict[str, np.ndarray]] = {} if cache_weights else None

    # -- helpers -----------------------------------------------------------
    def w(self, name: str) -> np.ndarray:
        if self._cache is not None:
            if name not in self._cache:
                self._cache[name] = _to_numpy(self._src[name], self.dt)
            return self._cache[name]
        return _to_numpy(self._src[name], self.dt)

    def _st(self, x: np.ndarray) -> np.ndarray:
        return bf16_round(x).astype(self.dt) if self.store == "bf16" else x

    # -- forward -----------------------------------------------------------
    def forward(self, tokens, positions, cache: KVCache, allowed_new: np.ndarray):
        """Run new rows against committed ``cache``.

        tokens, positions: length-Q sequences.  allowed_new[i, j] says whether
        new row i may see new row j (every row sees all committed rows).
        Returns (logits [Q, V], new_k [L][Q,H,dh], new_v [L][Q,H,dh]).
        """
        return self.forward_many([(tokens, positions, cache, allowed_new)])[0]

    def forward_many(self, calls):
        """One forward over the rows of several independent requests.

        ``calls`` is a list of (tokens, positions, cache, allowed_new), one per
        request, each as in ``forward``.  The row-wise work (embedding, norms,
        projections, SwiGLU, head) runs on the requests' rows stacked in call
        order; attention runs per request, its rows against its own committed
        cache and its own new rows only (no row sees another request).  With
        one call this is exactly ``forward``.  Returns a list of
        (logits, new_k, new_v) in call order.
        """
        cfg = self.cfg
        toks = [np.asarray(c[0], dtype=np.int64) for c in calls]
        offs = np.cumsum([0] + [len(t) for t in toks])
        tokens = np.concatenate(toks)
        positions = np.concatenate([np.asarray(c[1], dtype=np.int64) for c in calls])
        groups = []
        for (_, _, cache, allowed_new), b in zip(calls, range(len(calls))):
            Qb = int(offs[b + 1] - offs[b])
            allowed = np.concatenate([np.ones((Qb, len(cache)), dtype=bool),
                                      np.asarray(allowed_new, dtype=bool)], axis=1)
            groups.append((slice(int(offs[b]), int(offs[b + 1])), cache, allowed))
        emb = self.w("tok_emb")
        x = emb[tokens].astype(self.dt)
        new_k = [[] for _ in calls]
        new_v = [[] for _ in calls]
        for l in range(cfg.n_layers):
            x, kl, vl = self.block(l, x, positions, groups)
            for b in range(len(calls)):
                new_k[b].append(kl[b])
                new_v[b].append(vl[b])
        logits = self.head(x)
        return [(logits[int(offs[b]):int(offs[b + 1])], new_k[b], new_v[b]) for b in range(len(calls))]

    def block(self, l: int, x: np.ndarray, positions, groups):
        """Decoder layer ``l`` on the residual rows ``x`` [Q, d] at ``positions``.

        ``groups`` lists, per request, (row slice, committed cache, visibility
        [Q_b, len(cache) + Q_b]); a request's rows attend to its own cache at
        layer ``l`` and its own new rows only.  Returns (x after the layer,
        per-request new K rows [Q_b, H, dh], per-request new V rows).  The
        stages below, in order, are the whole layer.
        """
        o, ks, vs = self.attention(l, x, positions, groups)
        x = self.o_residual(l, x, o)
        a = self.mlp_act(l, self.mlp_input(l, x))
        return self.down_residual(l, x, a), ks, vs

    def attention(self, l: int, x: np.ndarray, positions, groups):
        """RMSNorm, Q/K/V projections, RoPE and masked attention of layer l:
        (attention output [Q, H*dh] as stored, new K rows, new V rows)."""
        cfg = self.cfg
        H, dh = cfg.n_heads, cfg.head_dim
        Q = x.shape[0]
        scale = 1.0 / math.sqrt(dh)
        xn = self._st(rmsnorm(x, self.w(f"l{l}.attn_norm"), cfg.rms_eps))
        q = self._st(xn @ self.w(f"l{l}.wq").T).reshape(Q, H, dh)
        k = self._st(xn @ self.w(f"l{l}.wk").T).reshape(Q, H, dh)
        v = self._st(xn @ self.w(f"l{l}.wv").T).reshape(Q, H, dh)
        q = self._st(rope(q, positions, cfg.rope_theta))
        k = self._st(rope(k, positions, cfg.rope_theta))
        o = np.empty((Q, H, dh), dtype=self.dt)
        ks, vs = [], []
        for rows, cache, allowed in groups:
            kb, vb = k[rows], v[rows]
            ks.append(kb)
            vs.append(vb)
            K = kb if len(cache) == 0 else np.concatenate([cache.k[l], kb], axis=0)
            V = vb if len(cache) == 0 else np.concatenate([cache.v[l], vb], axis=0)
            for h in range(H):
                s = (q[rows, h, :] @ K[:, h, :].T) * scale             # [Q_b, K_b+Q_b]
                s = np.where(allowed, s, -np.inf)
                o[rows, h, :] = softmax_rows(s) @ V[:, h, :]
        return self._st(o.reshape(Q, H * dh)), ks, vs

    def o_residual(self, l: int, x: np.ndarray, o: np.ndarray) -> np.ndarray:
        """The residual after the attention: x + Wo . o."""
        return x + o @ self.w(f"l{l}.wo").T

    def mlp_input(self, l: int, x: np.ndarray) -> np.ndarray:
        """RMSNorm of the residual before the MLP, as stored."""
        return self._st(rmsnorm(x, self.w(f"l{l}.mlp_norm"), self.cfg.rms_eps))

    def mlp_act(self, l: int, hn: np.ndarray) -> np.ndarray:
        """SwiGLU of the normalised rows, as stored: silu(Wgate . hn) * (Wup . hn)."""
        return self._st(silu(hn @ self.w(f"l{l}.w_gate").T) * (hn @ self.w(f"l{l}.w_up").T))

    def down_residual(self, l: int, x: np.ndarray, a: np.ndarray) -> np.ndarray:
        """The residual after the MLP: x + Wdown . a."""
        return x + a @ self.w(f"l{l}.w_down").T

    def head(self, x: np.ndarray) -> np.ndarray:
        """Final RMSNorm and LM head of residual rows ``x`` [Q, d]: logits [Q, V]."""
        cfg = self.cfg
        xf = self._st(rmsnorm(x, self.w("final_norm"), cfg.rms_eps))
        return xf @ self.w("lm_head").T

    def causal(self, tokens, start_pos: int, cache: KVCache):
        """Plain causal forward of a token run at positions start_pos.."""
        Q = len(tokens)
        pos = np.arange(start_pos, start_pos + Q)
        return self.forward(tokens, pos, cache, np.tril(np.ones((Q, Q), dtype=bool)))

    def prefill(self, prompt):
        """Causal prefill of the prompt; returns (cache, logits of all rows)."""
        cache = KVCache(self.cfg.n_layers)
        logits, k, v = self.causal(prompt, 0, cache)
        cache.append(k, v)
        return cache, logits


def argmax_lowest(logits: np.ndarray) -> int:
    """Greedy selector with a fixed tie rule: the lowest token id among maxima."""
    return int(np.argmax(logits))   # numpy returns the first maximal index
