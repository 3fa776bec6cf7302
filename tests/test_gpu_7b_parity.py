"""Parity of the full-depth Llama-7B-shape bf16 path (32 layers, d 4096, 32
heads of 128, FFN 11008, vocab 32000) with the oracle at the stated 3e-2.

Stacked bf16 layers amplify rounding-order noise (two correct GPU GEMM paths
differ by ~0.14 in the logits after 32 layers), so depth is handled by
teacher forcing instead of a wider bound:

* every layer, stage by stage (la_debug_layer): from the GPU's values at the
  previous bf16 storage point, the oracle (fp64, bf16 storage emulation)
  reproduces the attention output, the RMSNorm output entering the MLP and
  the SwiGLU output up to one-ulp rounding flips, and both residual updates
  to fp32 rounding; the committed K/V the oracle's attention reads is its
  own, computed from the GPU's layer inputs of the committed rows.  Covered:
  a 24-token prefill and the first packed calls of a request (warm-up fills
  and steady calls with verification rows), each call's rows and visibility
  from the oracle's own row compiler;
* the final RMSNorm and LM head on the GPU's final residual: logits within
  3e-2, and the GPU's token equal to the oracle's argmax unless the oracle's
  top-2 gap is below 1e-2;
* the headline workload's calls that produce the first 64 tokens, teacher
  forced at the last layer: logits within 3e-2 and the GPU's argmax equal to
  the oracle's unless the oracle's top-2 gap is below 1e-2;
* the same 64 tokens against the whole oracle without teacher forcing inside
  the model (reported; near-ties wider than 1e-2 may flip at full depth).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import lookahead as la
from oracle.model import KVCache, OracleModel
from tests.gpu_util import context, top2_gap

pytestmark = pytest.mark.gpu

LOGIT_TOL = 3e-2     # bf16 configs: max-abs difference (logits, and every layer's residual rows)
TIE = 1e-2           # the oracle's top-2 gap under which a token may legitimately differ
W, N, G = 15, 5, 15


@pytest.fixture(scope="module")
def big7b():
    from lookahead_decoding_gb300 import lib
    cfg = synth.LLAMA_7B
    w = synth.llama_weights(cfg, 0, device="cuda:0")
    ctx = context(cfg, w, max_ctx=1024, W=W, N=N, G=G)
    yield lib(), ctx, cfg, w
    ctx.close()
    del w
    torch.cuda.empty_cache()


def layer_model(cfg, w, l):
    """The oracle restricted to layer l's weights, converted to fp64 once."""
    names = [f"l{l}.{n}" for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")]
    return OracleModel(cfg, {n: w[n].to("cpu", torch.float64).numpy() for n in names},
                       compute_dtype=np.float64, store="bf16", cache_weights=False)


def one_layer_cache(cfg, l, k, v):
    """A committed cache holding layer l's K/V (every layer slot names the
    same arrays, so the cache's length is theirs)."""
    c = KVCache(cfg.n_layers)
    c.k = [k] * cfg.n_layers
    c.v = [v] * cfg.n_layers
    return c


ULP = 2.0 ** -7           # one bf16 unit in the last place, relative to the larger value
FLIP_FRAC = 0.02          # most elements of a stored stage agree exactly
RESID_TOL = 1e-3          # fp32 sums of the residual updates against fp64


def check_stored(name, gpu, ref, carry=0.0, frac=FLIP_FRAC):
    """A stage stored in bf16: equal except where the two sides' pre-rounding
    values straddle a rounding boundary, so a differing element is one ulp of
    the larger value apart, plus `carry`, the most an input the two sides
    rounded apart can move it, plus a floor of 2^-8 of the stage's rms for
    values near zero; and at most `frac` of the elements differ at all."""
    diff = np.abs(gpu - ref)
    big = np.maximum(np.abs(gpu), np.abs(ref))
    floor = 2.0 ** -8 * float(np.sqrt(np.mean(ref ** 2)))
    excess = diff - (ULP * big + carry + floor)
    assert np.all(excess <= 0), (name, float(np.max(diff)), float(np.max(excess)))
    assert float(np.mean(diff > 0)) <= frac, (name, float(np.mean(diff > 0)))


def test_7b_every_layer_teacher_forced(big7b):
    """All 32 layers of the 7B shape, stage by stage, each from the GPU's own
    values at the previous storage point (a bf16 rounding that falls
    differently on the two sides would otherwise be amplified through the
    following layers, ~0.3 % of the residual per layer at this width): the
    attention output, the RMSNorm output entering the MLP and the SwiGLU
    output equal the oracle's except for one-ulp rounding flips; the two
    residual updates equal the oracle's to fp32 rounding; the final logits
    are within 3e-2.  Rows: a 24-token prefill and the first 12 packed calls
    of a request whose pool retrieves candidates."""
    L, ctx, cfg, w = big7b
    d, HD, F = cfg.d_model, cfg.n_heads * cfg.head_dim, cfg.d_ffn
    opts = L.LA_OPT_POOL_FROM_PROMPT | L.LA_OPT_POOL_FROM_OUTPUT
    # a short prompt whose first calls retrieve a candidate from the seeded
    # pool (checked on the GPU alone: C_t of the first 12 calls)
    p = None
    L.la_set_options(ctx.ctx, opts)
    for seed in range(11, 41):
        base = synth.markov_zipf_prompt(cfg.vocab, 8, seed).tolist()
        cand = base + base + base
        L.la_prefill(ctx.ctx, cand)
        hits = 0
        for _ in range(12):
            L.la_step(ctx.ctx, W, N, G)
            hits += L.la_debug_state(ctx.ctx)[0]["C_t"] > 0
        if hits:
            p = cand
            break
    assert p is not None, "no prompt of 30 retrieved a candidate"
    n = len(p)

    def grab(rows):
        return ([L.la_debug_layer(ctx.ctx, l, 0, rows, d) for l in range(cfg.n_layers + 1)],
                [L.la_debug_layer(ctx.ctx, l, 1, rows, HD) for l in range(cfg.n_layers)],
                [L.la_debug_layer(ctx.ctx, l, 2, rows, d) for l in range(cfg.n_layers)],
                [L.la_debug_layer(ctx.ctx, l, 3, rows, F) for l in range(cfg.n_layers)])

    L.la_set_debug(ctx.ctx, 1 | 8)
    try:
        first = L.la_prefill(ctx.ctx, p)
        pf = grab(n)
        lg_pf, _ = L.la_debug_logits(ctx.ctx, 2, cfg.vocab)
        # GPU calls, the oracle's state machine in lockstep on the GPU's tokens
        st = la.LookaheadState(p, first, W, N, G, pool_from_prompt=True, pool_from_output=True)
        calls = []
        for _ in range(12):
            rows, guesses = st.plan()
            em = L.la_step(ctx.ctx, W, N, G)
            hdr, _, tok, pos, _ = L.la_debug_state(ctx.ctx)
            Q = len(rows)
            assert hdr["Q"] == Q and hdr["C_t"] == len(guesses)
            assert tok == [r.token for r in rows] and pos == [r.position for r in rows]
            stages = grab(Q)
            lg, need = L.la_debug_logits(ctx.ctx, 1024, cfg.vocab)
            assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
            argmax = [0] * Q
            for i, r in enumerate(need):
                argmax[r] = int(np.argmax(lg[i]))
            info = st.publish(rows, guesses, argmax)
            assert em == info.emitted
            calls.append((rows, stages, lg, need, list(info.commit_rows)))
        assert any(any(r.role == la.VERIFY for r in c[0]) for c in calls), "no steady call verified a candidate"
    finally:
        L.la_set_debug(ctx.ctx, 0)
        L.la_set_options(ctx.ctx, 0)

    def check_layer(m, l, stages, positions, group, chk):
        xs, att, hn, act = stages
        o, ks, vs = m.attention(l, xs[l].astype(np.float64), positions, [group])
        # The oracle's q, k, v come from the GPU's layer input; a few elements
        # round one ulp apart from the GPU's, and an output element is a
        # softmax-weighted average of v, so it can move by up to one ulp of the
        # largest |v| and every element of an affected (row, head) may round
        # differently.
        vmax = max(float(np.max(np.abs(v))) for v in vs + [group[1].v[l]] if v is not None and v.size)
        check_stored(("attention", l), att[l], o, carry=ULP * vmax, frac=0.10)
        x_mid = m.o_residual(l, xs[l].astype(np.float64), att[l])
        check_stored(("mlp input", l), hn[l], m.mlp_input(l, x_mid))
        check_stored(("swiglu", l), act[l], m.mlp_act(l, hn[l]))
        x_next = m.down_residual(l, x_mid, act[l])
        err = float(np.max(np.abs(x_next[chk] - xs[l + 1][chk])))
        assert err < RESID_TOL, ("residual", l, err)
        # the whole layer from the GPU's input alone: the roundings that fall
        # apart cascade through the layer's bf16 storage points; measured
        # about 0.3 % of the residual's rms at this width
        whole, _, _ = m.block(l, xs[l].astype(np.float64), positions, [group])
        rel = float(np.sqrt(np.mean((whole[chk] - xs[l + 1][chk]) ** 2)) / np.sqrt(np.mean(xs[l + 1][chk] ** 2)))
        assert rel < 0.01, ("whole layer", l, rel)
        worst[0] = max(worst[0], float(np.max(np.abs(whole[chk] - xs[l + 1][chk]))))
        return ks[0], vs[0]

    worst = [0.0]
    for l in range(cfg.n_layers):
        m = layer_model(cfg, w, l)
        last = l + 1 == cfg.n_layers
        ck, cv = check_layer(m, l, pf, np.arange(n),
                             (slice(0, n), KVCache(cfg.n_layers), np.tril(np.ones((n, n), dtype=bool))),
                             [n - 1] if last else slice(None))
        for rows, stages, _, need, commit in calls:
            Q = len(rows)
            vis = np.concatenate([np.ones((Q, ck.shape[0]), dtype=bool), la.meta_mask(rows)], axis=1)
            k, v = check_layer(m, l, stages, np.array([r.position for r in rows]),
                               (slice(0, Q), one_layer_cache(cfg, l, ck, cv), vis), list(need) if last else slice(None))
            ck = np.concatenate([ck, k[commit]], axis=0)
            cv = np.concatenate([cv, v[commit]], axis=0)
        del m
    # final norm + LM head on the GPU's final residual
    head = OracleModel(cfg, {n_: w[n_].to("cpu", torch.float64).numpy() for n_ in ("final_norm", "lm_head")},
                       compute_dtype=np.float64, store="bf16", cache_weights=False)
    ref = head.head(pf[0][cfg.n_layers][[n - 1]])
    assert np.max(np.abs(lg_pf[0] - ref[0])) < LOGIT_TOL
    assert int(np.argmax(lg_pf[0])) == int(np.argmax(ref[0])) or top2_gap(ref[0]) < TIE
    for rows, stages, lg, need, _ in calls:
        ref = head.head(stages[0][cfg.n_layers][list(need)])
        assert np.max(np.abs(lg - ref)) < LOGIT_TOL
        for i in range(len(need)):
            assert int(np.argmax(lg[i])) == int(np.argmax(ref[i])) or top2_gap(ref[i]) < TIE
    print(f"whole-layer teacher-forced residual deviation, max-abs over 32 layers: {worst[0]:.4f}")


def test_7b_first_64_tokens_against_oracle(big7b):
    """Headline workload (prompt 512, W=15, N=5, G=15), the calls that produce
    the first 64 tokens.  Teacher-forced at the last layer: for every call, the
    oracle's final RMSNorm and LM head on the GPU's final residual of each
    needed row give logits within 3e-2 and the same argmax unless the oracle's
    top-2 gap is below 1e-2.  The emitted stream equals the GPU's AR stream."""
    L, ctx, cfg, w = big7b
    p = synth.markov_zipf_prompt(cfg.vocab, 512, 2).tolist()
    ar = L.la_generate_ar(ctx.ctx, p, 64)
    head = OracleModel(cfg, {n_: w[n_].to("cpu", torch.float64).numpy() for n_ in ("final_norm", "lm_head")},
                       compute_dtype=np.float64, store="bf16", cache_weights=False)
    L.la_set_debug(ctx.ctx, 1 | 8)
    try:
        out = [L.la_prefill(ctx.ctx, p)]
        worst = 0.0
        while len(out) < 64:
            out += L.la_step(ctx.ctx, W, N, G)
            Q = L.la_debug_state(ctx.ctx)[0]["Q"]
            lg, need = L.la_debug_logits(ctx.ctx, 1024, cfg.vocab)
            xf = L.la_debug_hidden(ctx.ctx, cfg.n_layers, Q, cfg.d_model)
            ref = head.head(xf[list(need)])
            worst = max(worst, float(np.max(np.abs(lg - ref))))
            for i in range(len(need)):
                assert int(np.argmax(lg[i])) == int(np.argmax(ref[i])) or top2_gap(ref[i]) < TIE
        assert worst < LOGIT_TOL, worst
        assert out[:64] == ar
    finally:
        L.la_set_debug(ctx.ctx, 0)


def test_7b_full_depth_token_stream_reported(big7b):
    """Without teacher forcing inside the model: the oracle runs all 32 layers
    over the prompt followed by the GPU's first 64 tokens and its argmax at
    each generated position is compared with the GPU's token.  Rounding-order
    differences grow through 32 random-init bf16 layers (the two GPU GEMM paths
    already differ by ~0.14 in the logits), so near-ties wider than 1e-2 can
    flip; the flips and the oracle's gaps there are printed, and the stream
    must agree on at least 56 of the 64 positions."""
    L, ctx, cfg, w = big7b
    p = synth.markov_zipf_prompt(cfg.vocab, 512, 2).tolist()
    got = L.la_generate(ctx.ctx, p, 64, W, N, G)
    oracle = OracleModel(cfg, w, compute_dtype=np.float64, store="bf16", cache_weights=False)
    _, logits = oracle.prefill(p + got[:-1])
    ref = logits[len(p) - 1:]                     # the rows that predict got[0 .. 63]
    mism = [(i, round(float(top2_gap(ref[i])), 4)) for i in range(64) if int(np.argmax(ref[i])) != got[i]]
    print(f"full-depth stream: {64 - len(mism)} of 64 tokens equal the oracle's argmax; flips (position, gap): {mism}")
    assert len(mism) <= 8, mism
