"""Pins of the oracle transformer and of the whole greedy lookahead loop."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import jacobi
from oracle import lookahead as la
from oracle.model import KVCache, OracleModel, bf16_round, rmsnorm, rope, argmax_lowest

MICRO = synth.ModelConfig(n_layers=1, d_model=16, n_heads=2, head_dim=8, d_ffn=32, vocab=6,
                          dtype="f32", init_std=0.5)
SMALL = synth.ModelConfig(n_layers=2, d_model=32, n_heads=4, head_dim=8, d_ffn=64, vocab=16,
                          dtype="f32", init_std=0.3)


def model_for(cfg, seed=0, **kw):
    return OracleModel(cfg, synth.llama_weights(cfg, seed), **kw)


# ---- textbook definitions -----------------------------------------------------

def test_rmsnorm_closed_form():
    x = np.array([[3.0, 4.0]])
    y = rmsnorm(x, np.array([1.0, 2.0]), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(y, [[3 / r, 8 / r]], rtol=0, atol=1e-15)
    z = np.random.default_rng(0).normal(size=(3, 8))
    assert np.allclose(rmsnorm(z, np.ones(8), 0.0), rmsnorm(7.5 * z, np.ones(8), 0.0))


def test_rope_properties():
    rnd = np.random.default_rng(1)
    x = rnd.normal(size=(5, 3, 8))
    assert np.allclose(rope(x, np.zeros(5, dtype=int), 10000.0), x)       # position 0: identity
    # dh = 2: a plain rotation by pos radians
    v = np.array([[[1.0, 2.0]]])
    c, s = math.cos(3.0), math.sin(3.0)
    assert np.allclose(rope(v, np.array([3]), 10000.0), [[[c - 2 * s, 2 * c + s]]])
    # the pair (i, i + dh/2) turns by pos * theta^(-2i/dh): norms kept per pair
    y = rope(x, np.arange(5) * 7, 10000.0)
    assert np.allclose(x[..., :4] ** 2 + x[..., 4:] ** 2, y[..., :4] ** 2 + y[..., 4:] ** 2)
    # q(m).k(n) depends only on m - n
    q, k = rnd.normal(size=(1, 1, 8)), rnd.normal(size=(1, 1, 8))
    d1 = (rope(q, np.array([9]), 100.0) * rope(k, np.array([4]), 100.0)).sum()
    d2 = (rope(q, np.array([25]), 100.0) * rope(k, np.array([20]), 100.0)).sum()
    assert abs(d1 - d2) < 1e-12


@pytest.mark.parametrize("dh,anchors", [
    # dh = 8, theta = 1e4: the pair-i frequency theta^(-2i/dh) = 10^(-i), i = 0..3
    (8, {0: 1.0, 1: 0.1, 2: 0.01, 3: 0.001}),
    # dh = 128, theta = 1e4: 10^(-i/16); the decades fall at i = 16, 32, 48
    (128, {0: 1.0, 1: 10 ** (-1 / 16), 2: 10 ** (-2 / 16), 3: 10 ** (-3 / 16),
           16: 0.1, 32: 0.01, 48: 0.001, 63: 10 ** (-63 / 16)}),
])
@pytest.mark.parametrize("pos", [1, 5, 517])
def test_rope_frequency_schedule_hand_values(dh, anchors, pos):
    """RoFormer's rotary embedding (Su et al., eq. 15, rotate-half pairing as in
    Llama): the unit vector on dimension i (< dh/2) at position pos becomes
    cos(pos*f_i) on dimension i and sin(pos*f_i) on its partner i + dh/2, with
    f_i = theta^(-2i/dh).  The frequencies are written out by hand above (for
    theta = 10^4 they are powers of ten), so a wrong exponent such as -i/dh or
    -2i/(dh-2), a swapped pair or a flipped sign fails here at every pos >= 1."""
    half = dh // 2
    for i, f in anchors.items():
        e = np.zeros((1, 1, dh))
        e[0, 0, i] = 1.0
        y = rope(e, np.array([pos]), 10000.0)[0, 0]
        want = np.zeros(dh)
        want[i] = math.cos(pos * f)
        want[i + half] = math.sin(pos * f)
        assert np.allclose(y, want, rtol=0, atol=1e-12), (dh, i, pos)
        # the partner dimension turns the other way: e_{i+half} -> (-sin, cos)
        e2 = np.zeros((1, 1, dh))
        e2[0, 0, i + half] = 1.0
        y2 = rope(e2, np.array([pos]), 10000.0)[0, 0]
        assert abs(y2[i] + math.sin(pos * f)) < 1e-12 and abs(y2[i + half] - math.cos(pos * f)) < 1e-12


def test_bf16_round_matches_torch():
    x = np.random.default_rng(2).normal(size=4096) * 10.0 ** np.random.default_rng(3).integers(-8, 8, 4096)
    ours = bf16_round(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_forward_equals_library_composition_at_position_zero():
    """With every position 0, RoPE is the identity and one causal forward reduces to
    torch's rms_norm / linear / scaled_dot_product_attention / silu composition."""
    cfg = SMALL
    W = synth.llama_weights(cfg, 4)
    m = OracleModel(cfg, W)
    toks = [3, 1, 4, 1, 5, 9, 2]
    Q = len(toks)
    logits, _, _ = m.forward(toks, [0] * Q, KVCache(cfg.n_layers), np.tril(np.ones((Q, Q), bool)))
    F = torch.nn.functional
    d = {k: v.double() for k, v in W.items()}
    x = d["tok_emb"][torch.tensor(toks)]
    for l in range(cfg.n_layers):
        xn = F.rms_norm(x, (cfg.d_model,), d[f"l{l}.attn_norm"], cfg.rms_eps)
        sh = lambda t: t.view(Q, cfg.n_heads, cfg.head_dim).transpose(0, 1)
        q, k, v = (sh(F.linear(xn, d[f"l{l}.{n}"])) for n in ("wq", "wk", "wv"))
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(0, 1).reshape(Q, -1)
        x = x + F.linear(o, d[f"l{l}.wo"])
        hn = F.rms_norm(x, (cfg.d_model,), d[f"l{l}.mlp_norm"], cfg.rms_eps)
        x = x + F.linear(F.silu(F.linear(hn, d[f"l{l}.w_gate"])) * F.linear(hn, d[f"l{l}.w_up"]), d[f"l{l}.w_down"])
    ref = F.linear(F.rms_norm(x, (cfg.d_model,), d["final_norm"], cfg.rms_eps), d["lm_head"])
    assert np.allclose(logits, ref.numpy(), rtol=0, atol=1e-10)


def test_cached_incremental_equals_one_call():
    m = model_for(SMALL, 5)
    toks = [2, 7, 1, 8, 2, 8, 1, 8]
    cache, full = m.prefill(toks)
    c2 = KVCache(SMALL.n_layers)
    rows = []
    for i, t in enumerate(toks):
        lg, k, v = m.causal([t], i, c2)
        c2.append(k, v)
        rows.append(lg[0])
    assert np.allclose(np.stack(rows), full, rtol=0, atol=1e-12)
    for l in range(SMALL.n_layers):
        assert np.allclose(cache.k[l], c2.k[l], atol=1e-12) and np.allclose(cache.v[l], c2.v[l], atol=1e-12)


def test_mlp_and_attention_off_reduce_to_head_of_embedding():
    cfg = SMALL
    W = synth.llama_weights(cfg, 6)
    for l in range(cfg.n_layers):
        W[f"l{l}.wo"] = torch.zeros_like(W[f"l{l}.wo"])
        W[f"l{l}.w_down"] = torch.zeros_like(W[f"l{l}.w_down"])
    m = OracleModel(cfg, W)
    cache, lg = m.prefill([4, 2, 9])
    e = W["tok_emb"].double().numpy()[[4, 2, 9]]
    ref = rmsnorm(e, np.ones(cfg.d_model), cfg.rms_eps) @ W["lm_head"].double().numpy().T
    assert np.allclose(lg, ref, atol=1e-12)


# ---- T12: schedules agree -----------------------------------------------------------

@pytest.mark.parametrize("W,N,G", [(5, 4, 2), (3, 3, 3), (1, 3, 1), (4, 5, 2)])
def test_schedules_agree(W, N, G):
    m = model_for(SMALL, 8)
    prompt = [1, 2, 3, 4, 5, 1, 2, 3]
    cache, lg = m.prefill(prompt)
    st = la.LookaheadState(prompt, argmax_lowest(lg[-1]), W, N, G)
    # fill a pool so verification rows exist
    for key in range(SMALL.vocab):
        for c in range(G):
            la.upsert_suffix_lru(st.pool, key, tuple((key + c + i) % SMALL.vocab for i in range(N - 1)), G)
    runners = {s: la.make_runner(m, cache.copy(), s) for s in ("separate", "dense", "meta")}
    for step in range(N + 1):
        rows, guesses = st.plan()
        out = {s: r.run(rows) for s, r in runners.items()}
        assert np.allclose(out["dense"], out["separate"], rtol=0, atol=1e-10)
        assert np.array_equal(out["dense"], out["meta"])
        argmax = [argmax_lowest(x) for x in out["dense"]]
        info = st.publish(rows, guesses, argmax)
        for r in runners.values():
            r.commit(rows, info.commit_rows)


# ---- whole loop: lookahead == autoregressive (greedy) ----------------------------------

def test_jacobi_on_model_reaches_ar_within_m_sweeps():
    m = model_for(MICRO, 1)
    prompt = [1, 4, 2]

    def T(i, y):
        lg, _, _ = m.causal(list(prompt) + list(y), 0, KVCache(1))
        return argmax_lowest(lg[-1])

    ar = la.ar_generate(m, prompt, 6)
    fp, n = jacobi.solve(T, [0] * 6)
    assert fp == ar and n <= 6


@pytest.mark.parametrize("W,N,G", [(3, 3, 3), (5, 4, 2), (2, 5, 4), (1, 3, 1), (6, 3, 6)])
def test_lookahead_equals_ar_tiny_vocab_many_seeds(W, N, G):
    hits = 0
    for seed in range(12):
        m = model_for(MICRO, seed)
        prompt = list(synth.uniform_prompt(MICRO.vocab, 5, 100 + seed))
        ar = la.ar_generate(m, prompt, 24)
        tr = []
        lk = la.lookahead_generate(m, prompt, 24, W, N, G, trace=tr)
        assert lk == ar, (seed, lk, ar)
        hits += sum(i.a for i in tr)
    assert hits > 0          # verification accepted candidates somewhere


def test_lookahead_separate_and_dense_schedules_equal_ar():
    for seed in range(3):
        m = model_for(MICRO, 40 + seed)
        prompt = [0, 1, 2, 3]
        ar = la.ar_generate(m, prompt, 16)
        for sch in ("separate", "dense"):
            assert la.lookahead_generate(m, prompt, 16, 3, 4, 3, schedule=sch) == ar


def test_tiny_llama_config_lookahead_equals_ar():
    cfg = synth.TINY
    m = model_for(cfg, 0)
    prompt = list(synth.uniform_prompt(cfg.vocab, 32, 1))
    ar = la.ar_generate(m, prompt, 64)
    assert la.lookahead_generate(m, prompt, 64, 5, 3, 5) == ar


def test_wrong_commit_row_breaks_equality():
    """Planted mistake on the CPU: committing the row after each accepted one
    changes later logits, so the AR-equality pin detects commit errors."""
    class OffByOne(la.LookaheadState):
        def publish(self, rows, guesses, argmax, verdict=None):
            info = super().publish(rows, guesses, argmax, verdict)
            S = self.S
            if info.a and info.a < S:
                info.commit_rows = [0] + [r + 1 for r in info.commit_rows[1:]]
            return info

    diverged = 0
    for seed in range(12):
        m = model_for(MICRO, seed)
        prompt = list(synth.uniform_prompt(MICRO.vocab, 5, 100 + seed))
        ar = la.ar_generate(m, prompt, 24)
        cache, lg = m.prefill(prompt)
        out = [argmax_lowest(lg[-1])]
        st = OffByOne(prompt, out[0], 3, 4, 3)
        run = la.make_runner(m, cache, "meta")
        while len(out) < 24:
            rows, g = st.plan()
            L = run.run(rows)
            info = st.publish(rows, g, [argmax_lowest(x) for x in L])
            run.commit(rows, info.commit_rows)
            out.extend(info.emitted)
        diverged += out[:24] != ar
    assert diverged > 0


@pytest.mark.parametrize("W,N,G", [(3, 3, 3), (5, 4, 2), (2, 5, 4)])
def test_seeded_pool_lookahead_equals_ar(W, N, G):
    """Seeding only changes which candidates are tried: the output stays the
    greedy AR output, and a copy-heavy prompt gets candidates from the first
    steady call on."""
    offered = 0
    for seed in range(8):
        m = model_for(MICRO, 60 + seed)
        base = list(synth.uniform_prompt(MICRO.vocab, 6, 200 + seed))
        prompt = base + base + base
        ar = la.ar_generate(m, prompt, 24)
        tr = []
        lk = la.lookahead_generate(m, prompt, 24, W, N, G, trace=tr, pool_from_prompt=True, pool_from_output=True)
        assert lk == ar, (seed, lk, ar)
        first_steady = next(i for i in tr if i.steady)
        offered += first_steady.C_t
    assert offered > 0


@pytest.mark.parametrize("W,N,G", [(3, 3, 3), (5, 4, 2), (2, 5, 4), (1, 3, 1)])
def test_sliced_window_lookahead_equals_ar(W, N, G):
    """The ALWAYS_FWD_ONE=False schedule only changes the proposals: the
    output stays the greedy AR output, while the calls made differ from the
    pinned schedule's on some seed."""
    changed = 0
    for seed in range(12):
        m = model_for(MICRO, seed)
        prompt = list(synth.uniform_prompt(MICRO.vocab, 5, 100 + seed))
        ar = la.ar_generate(m, prompt, 24)
        tr, tr0 = [], []
        lk = la.lookahead_generate(m, prompt, 24, W, N, G, trace=tr, slice_window=True)
        assert lk == ar, (seed, lk, ar)
        la.lookahead_generate(m, prompt, 24, W, N, G, trace=tr0)
        changed += [(i.Q, i.a) for i in tr] != [(i.Q, i.a) for i in tr0]
    assert changed > 0
