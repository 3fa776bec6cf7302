"""GPU parity of the bf16 tensor-core path (tcgen05 GEMMs) against the oracle.

* a small bf16 Llama (2 layers, d 512, 4 heads of 128, FFN 1408, vocab 4096):
  logits within 3e-2 of the oracle with bf16 storage emulation, every packed
  call's rows/logits/state, lookahead == autoregressive bit-exact;
* the 7B shape of the headline workload (32 layers, d 4096, 32 heads, FFN
  11008, vocab 32000; prompt 512 order-2 Markov/Zipf(1.1) tokens; W=15, N=5,
  G=15; 256 new tokens) in the launch configuration the bench times:
  lookahead == autoregressive token for token, and one layer of the 7B
  shapes against the oracle (full depth: test_gpu_7b_parity.py).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import lookahead as la
from oracle.model import KVCache, OracleModel, argmax_lowest
from tests.gpu_util import context, top2_gap

pytestmark = pytest.mark.gpu

MID = synth.ModelConfig(n_layers=2, d_model=512, n_heads=4, head_dim=128, d_ffn=1408, vocab=4096, dtype="bf16")
LOGIT_TOL = 3e-2          # bf16 configs: max-abs logit difference
TIE = 1e-2                # the oracle's top-2 gap under which a token may legitimately differ


@pytest.fixture(scope="module")
def mid():
    from lookahead_decoding_gb300 import lib
    w = synth.llama_weights(MID, 0, device="cuda:0")
    ctx = context(MID, w, max_ctx=640, W=15, N=5, G=15)
    oracle = OracleModel(MID, {k: v.cpu() for k, v in w.items()}, store="bf16")
    yield lib(), ctx, oracle
    ctx.close()


def test_prefill_logits_mid(mid):
    L, ctx, oracle = mid
    L.la_set_debug(ctx.ctx, 1)
    plain = OracleModel(MID, oracle._src)
    for n, seed in ((7, 1), (300, 2)):       # one chunk, two chunks with a ragged tail
        p = synth.markov_zipf_prompt(MID.vocab, n, seed).tolist()
        tok = L.la_prefill(ctx.ctx, p)
        lg, _ = L.la_debug_logits(ctx.ctx, 2, MID.vocab)
        _, ref = oracle.prefill(p)
        err = np.max(np.abs(lg[0] - ref[-1]))
        assert err < LOGIT_TOL, err
        _, ref2 = plain.prefill(p)               # without the storage emulation
        assert np.max(np.abs(lg[0] - ref2[-1])) < 2 * LOGIT_TOL
        assert tok == argmax_lowest(ref[-1]) or top2_gap(ref[-1]) < TIE
    L.la_set_debug(ctx.ctx, 0)


@pytest.mark.parametrize("W,N,G", [(15, 5, 15), (4, 3, 4), (1, 3, 1)])
def test_step_by_step_mid(mid, W, N, G):
    L, ctx, oracle = mid
    p = synth.markov_zipf_prompt(MID.vocab, 64, 5).tolist()
    L.la_set_debug(ctx.ctx, 1)
    first = L.la_prefill(ctx.ctx, p)
    cache, lg0 = oracle.prefill(p)
    st = la.LookaheadState(p, first, W, N, G)
    run = la.make_runner(oracle, cache, "meta")
    for step in range(12):
        rows, guesses = st.plan()
        ref = run.run(rows)
        em = L.la_step(ctx.ctx, W, N, G)
        h, _, tok, pos, _ = L.la_debug_state(ctx.ctx)
        assert tok == [r.token for r in rows] and pos == [r.position for r in rows]
        lg, need = L.la_debug_logits(ctx.ctx, 1024, MID.vocab)
        assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
        err = np.max(np.abs(lg - ref[need]))
        assert err < LOGIT_TOL, (step, err)
        # follow the GPU's selections; each must be the oracle's unless near a tie
        argmax = [argmax_lowest(x) for x in ref]
        for i, r in enumerate(need):
            g = int(np.argmax(lg[i]))
            assert g == argmax[r] or top2_gap(ref[r]) < TIE
            argmax[r] = g
        info = st.publish(rows, guesses, argmax)
        run.commit(rows, info.commit_rows)
        assert em == info.emitted
    L.la_set_debug(ctx.ctx, 0)


@pytest.fixture(scope="module")
def mid_pred():
    """MID with the attention output projections scaled by 2**-10: the greedy
    next token is nearly a function of the current one, so the pool's
    n-grams come true and calls accept candidates on real logits."""
    from lookahead_decoding_gb300 import lib
    w = synth.llama_weights(MID, 0, device="cuda:0", wo_scale=2.0 ** -10)
    ctx = context(MID, w, max_ctx=640, W=15, N=5, G=15)
    oracle = OracleModel(MID, {k: v.cpu() for k, v in w.items()}, store="bf16")
    yield lib(), ctx, oracle
    ctx.close()


def test_accepting_calls_against_oracle_mid(mid_pred):
    """Call by call against the oracle on a model whose candidates are
    accepted: rows, needed-row logits within 3e-2, the verdict and the
    emitted tokens (the GPU's argmax followed where the oracle's top-2 gap is
    under TIE); the run must include calls that commit several tokens (the
    accepted rows' K/V then feed every later call's logits)."""
    L, ctx, oracle = mid_pred
    W, N, G = 15, 5, 15
    p = synth.markov_zipf_prompt(MID.vocab, 64, 5).tolist()
    L.la_set_debug(ctx.ctx, 1)
    first = L.la_prefill(ctx.ctx, p)
    cache, _ = oracle.prefill(p)
    st = la.LookaheadState(p, first, W, N, G)
    run = la.make_runner(oracle, cache, "meta")
    multi = 0
    for step in range(60):
        rows, guesses = st.plan()
        ref = run.run(rows)
        em = L.la_step(ctx.ctx, W, N, G)
        h, _, tok, pos, _ = L.la_debug_state(ctx.ctx)
        assert tok == [r.token for r in rows] and pos == [r.position for r in rows]
        lg, need = L.la_debug_logits(ctx.ctx, 1024, MID.vocab)
        assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
        err = np.max(np.abs(lg - ref[need]))
        assert err < LOGIT_TOL, (step, err)
        argmax = [argmax_lowest(x) for x in ref]
        for i, r in enumerate(need):
            g = int(np.argmax(lg[i]))
            assert g == argmax[r] or top2_gap(ref[r]) < TIE
            argmax[r] = g
        info = st.publish(rows, guesses, argmax)
        run.commit(rows, info.commit_rows)
        assert em == info.emitted, step
        multi += len(em) > 1
    L.la_set_debug(ctx.ctx, 0)
    assert multi >= 5, multi


def test_accepting_generate_equals_ar_mid(mid_pred):
    """Whole requests with accepted candidates: lookahead == AR token for
    token, more than one token per call, and the oracle's greedy choice
    given the GPU's prefix (teacher forced)."""
    L, ctx, oracle = mid_pred
    p = synth.markov_zipf_prompt(MID.vocab, 96, 7).tolist()
    ar = L.la_generate_ar(ctx.ctx, p, 160)
    for W, N, G in [(15, 5, 15), (7, 4, 7)]:
        st = L.la_stats()
        got = L.la_generate(ctx.ctx, p, 160, W, N, G, stats=st)
        assert got == ar, (W, N, G)
        assert (st.tokens - 1) / st.steps > 1.2, (W, N, G, st.tokens, st.steps)
        assert sum(st.emitted_hist[1:]) > 0
    teacher_forced_check(oracle, p, ar)


def teacher_forced_check(oracle, prompt, tokens):
    """Every GPU token equals the oracle's greedy choice given the GPU's own prefix,
    except where the oracle's top-2 gap is below TIE.  Returns the number of ties."""
    cache, lg = oracle.prefill(prompt)
    ties = 0
    last = lg[-1]
    for t, tok in enumerate(tokens):
        if tok != argmax_lowest(last):
            assert top2_gap(last) < TIE, (t, tok, argmax_lowest(last), top2_gap(last))
            ties += 1
        if t + 1 < len(tokens):
            out, k, v = oracle.causal([tok], len(cache), cache)
            cache.append(k, v)
            last = out[0]
    return ties


def test_generate_equals_ar_mid(mid):
    L, ctx, oracle = mid
    p = synth.markov_zipf_prompt(MID.vocab, 96, 7).tolist()
    ar = L.la_generate_ar(ctx.ctx, p, 96)
    for W, N, G in [(15, 5, 15), (4, 3, 4), (1, 3, 1), (7, 5, 7), (8, 4, 0)]:
        st = L.la_stats()
        got = L.la_generate(ctx.ctx, p, 96, W, N, G, stats=st)
        assert got == ar, (W, N, G)
    teacher_forced_check(oracle, p, ar)


@pytest.mark.parametrize("opts", ["seed", "seed+slice", "slice"])
def test_generate_with_pool_seeding_equals_ar_mid(mid, opts):
    L, ctx, oracle = mid
    p = synth.markov_zipf_prompt(MID.vocab, 96, 8).tolist()
    ar = L.la_generate_ar(ctx.ctx, p, 96)
    flags = 0
    if "seed" in opts:
        flags |= L.LA_OPT_POOL_FROM_PROMPT | L.LA_OPT_POOL_FROM_OUTPUT
    if "slice" in opts:
        flags |= L.LA_OPT_SLICE_WINDOW
    L.la_set_options(ctx.ctx, flags)
    try:
        for W, N, G in [(15, 5, 15), (4, 3, 4)]:
            got = L.la_generate(ctx.ctx, p, 96, W, N, G)
            assert got == ar, (W, N, G)
    finally:
        L.la_set_options(ctx.ctx, 0)


@pytest.mark.parametrize("W,N,G", [(15, 5, 15), (7, 4, 7)])
def test_attention_layouts_bitwise_equal_mid(monkeypatch, W, N, G):
    """The attention's two shared-memory layouts (in-call keys staged after
    the committed blocks in the ring, or during them in a region of their
    own) compute the same bits: every call's needed-row logits and every
    layer's attention output (W=15: including calls that accept)."""
    from lookahead_decoding_gb300 import lib
    L = lib()
    w = synth.llama_weights(MID, 0, device="cuda:0", wo_scale=2.0 ** -10)
    p = synth.markov_zipf_prompt(MID.vocab, 64, 5).tolist()
    runs = []
    for sep in ("0", "1"):
        monkeypatch.setenv("LA_ATTN_SEP", sep)
        ctx = context(MID, w, max_ctx=640, W=15, N=5, G=15)
        L.la_set_debug(ctx.ctx, 1 | 8)
        L.la_prefill(ctx.ctx, p)
        calls = []
        for _ in range(24):
            em = L.la_step(ctx.ctx, W, N, G)
            lg, need = L.la_debug_logits(ctx.ctx, 1024, MID.vocab)
            h = L.la_debug_state(ctx.ctx)[0]
            Q = int(h["Q"])
            attn = [L.la_debug_layer(ctx.ctx, l, 1, Q, MID.n_heads * MID.head_dim) for l in range(MID.n_layers)]
            calls.append((em, lg.copy(), need.copy(), attn))
        ctx.close()
        runs.append(calls)
    for (e0, l0, n0, a0), (e1, l1, n1, a1) in zip(*runs):
        assert e0 == e1 and np.array_equal(n0, n1)
        assert np.array_equal(l0.view(np.uint32), l1.view(np.uint32))
        for x, y in zip(a0, a1):
            assert np.array_equal(x, y)
    if W == 15:
        assert any(len(c[0]) > 1 for c in runs[1]), "no accepting call"


def test_row_invariance_probe_mid(mid):
    L, ctx, oracle = mid
    p = synth.markov_zipf_prompt(MID.vocab, 200, 9).tolist()
    L.la_set_debug(ctx.ctx, 1)
    L.la_generate_ar(ctx.ctx, p, 2)
    alone, _ = L.la_debug_logits(ctx.ctx, 4, MID.vocab)
    L.la_prefill(ctx.ctx, p)
    L.la_step(ctx.ctx, 15, 5, 15)
    packed, need = L.la_debug_logits(ctx.ctx, 1024, MID.vocab)
    assert np.array_equal(alone[0].view(np.uint32), packed[0].view(np.uint32))
    L.la_set_debug(ctx.ctx, 0)


# ---------------------------------------------------------------------------
# the 7B shape (headline workload)
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def big():
    from lookahead_decoding_gb300 import lib
    cfg = synth.LLAMA_7B
    w = synth.llama_weights(cfg, 0, device="cuda:0")
    ctx = context(cfg, w, max_ctx=1024, W=15, N=5, G=15)
    yield lib(), ctx, cfg, w
    ctx.close()
    del w
    torch.cuda.empty_cache()


def test_7b_lookahead_equals_ar(big):
    L, ctx, cfg, w = big
    p = synth.markov_zipf_prompt(cfg.vocab, 512, 2).tolist()
    ar = L.la_generate_ar(ctx.ctx, p, 256)
    st = L.la_stats()
    got = L.la_generate(ctx.ctx, p, 256, 15, 5, 15, stats=st)
    assert got == ar
    # the call statistics account for every token: calls that emitted k+1
    # tokens, summed, give the 255 tokens after the prefill's
    hist = list(st.emitted_hist)
    assert st.steps == sum(hist) and sum((k + 1) * c for k, c in enumerate(hist)) == 255, (st.steps, hist)
    assert st.tokens == 256 and 0.0 <= st.mean_candidates <= 15.0


@pytest.fixture(scope="module")
def shallow():
    """One layer of the 7B shapes (d 4096, 32 heads of 128, FFN 11008, vocab
    32000): every kernel at full size and in its launch configuration.  Depth
    is left out because stacked bf16 layers amplify rounding-order noise: two
    correct GPU GEMM paths already differ by ~0.03 after two such layers."""
    from lookahead_decoding_gb300 import lib
    cfg = synth.ModelConfig(n_layers=1, d_model=4096, n_heads=32, head_dim=128, d_ffn=11008, vocab=32000)
    w = synth.llama_weights(cfg, 0, device="cuda:0")
    ctx = context(cfg, w, max_ctx=1024, W=15, N=5, G=15)
    yield lib(), ctx, cfg, w
    ctx.close()


def test_7b_shapes_logits_against_oracle(shallow):
    """Full-size rows at 3e-2: the prefill row and every needed row of the first
    packed calls (warm-up and steady, with verification rows)."""
    L, ctx, cfg, w = shallow
    oracle = OracleModel(cfg, w, compute_dtype=np.float64, store="bf16")
    p = synth.markov_zipf_prompt(cfg.vocab, 40, 11).tolist()
    L.la_set_debug(ctx.ctx, 1)
    first = L.la_prefill(ctx.ctx, p)
    lg, _ = L.la_debug_logits(ctx.ctx, 2, cfg.vocab)
    cache, ref = oracle.prefill(p)
    assert np.max(np.abs(lg[0] - ref[-1])) < LOGIT_TOL
    st = la.LookaheadState(p, first, 15, 5, 15)
    run = la.make_runner(oracle, cache, "meta")
    for step in range(6):
        rows, guesses = st.plan()
        refl = run.run(rows)
        em = L.la_step(ctx.ctx, 15, 5, 15)
        lg, need = L.la_debug_logits(ctx.ctx, 1024, cfg.vocab)
        assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
        err = np.max(np.abs(lg - refl[need]))
        assert err < LOGIT_TOL, (step, err)
        argmax = [int(np.argmax(x)) for x in refl]
        for i, r in enumerate(need):
            argmax[r] = int(np.argmax(lg[i]))
        info = st.publish(rows, guesses, argmax)
        run.commit(rows, info.commit_rows)
        assert em == info.emitted
    L.la_set_debug(ctx.ctx, 0)


# ---- the W x N sweep (W in {1, 3, 7, 15, 31}, N in {3, 5, 7}, G = W) ----------

@pytest.fixture(scope="module")
def sweep():
    """The small bf16 model in a context sized for the largest sweep point
    (W = 31, N = 7, G = 31: up to 388 rows per call)."""
    from lookahead_decoding_gb300 import lib
    w = {k: v.to("cuda:0") for k, v in synth.llama_weights(MID, 0).items()}
    ctx = context(MID, w, max_ctx=1400, W=31, N=7, G=31)
    yield lib(), ctx
    ctx.close()


def test_sweep_points_equal_ar(sweep):
    """Every sweep point on a 1024-token Markov prompt, 256 new tokens: the
    lookahead output is the AR output."""
    L, ctx = sweep
    p = synth.markov_zipf_prompt(MID.vocab, 1024, 5).tolist()
    ar = L.la_generate_ar(ctx.ctx, p, 256)
    for W in (1, 3, 7, 15, 31):
        for N in (3, 5, 7):
            assert L.la_generate(ctx.ctx, p, 256, W, N, W) == ar, (W, N)


# ---- the 13B shapes and the code-like workload -----------------------------

@pytest.fixture(scope="module")
def shallow13():
    """One layer of the 13B shapes (d 5120, 40 heads of 128, FFN 13824, vocab 32000)."""
    from lookahead_decoding_gb300 import lib
    cfg = synth.ModelConfig(n_layers=1, d_model=5120, n_heads=40, head_dim=128, d_ffn=13824, vocab=32000)
    w = synth.llama_weights(cfg, 0, device="cuda:0")
    ctx = context(cfg, w, max_ctx=512, W=10, N=5, G=10)
    yield lib(), ctx, cfg, w
    ctx.close()
    del w
    torch.cuda.empty_cache()


def test_13b_shapes_logits_against_oracle(shallow13):
    """Full-size 13B rows at 3e-2: the prefill row and every needed row of the
    first packed calls of a code-like prompt (W=10, N=5, G=10)."""
    L, ctx, cfg, w = shallow13
    oracle = OracleModel(cfg, w, compute_dtype=np.float64, store="bf16")
    p = synth.code_like_prompt(cfg.vocab, 48, 13).tolist()
    L.la_set_debug(ctx.ctx, 1)
    first = L.la_prefill(ctx.ctx, p)
    lg, _ = L.la_debug_logits(ctx.ctx, 2, cfg.vocab)
    cache, ref = oracle.prefill(p)
    assert np.max(np.abs(lg[0] - ref[-1])) < LOGIT_TOL
    st = la.LookaheadState(p, first, 10, 5, 10)
    run = la.make_runner(oracle, cache, "meta")
    for step in range(5):
        rows, guesses = st.plan()
        refl = run.run(rows)
        em = L.la_step(ctx.ctx, 10, 5, 10)
        lg, need = L.la_debug_logits(ctx.ctx, 1024, cfg.vocab)
        assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
        err = np.max(np.abs(lg - refl[need]))
        assert err < LOGIT_TOL, (step, err)
        argmax = [int(np.argmax(x)) for x in refl]
        for i, r in enumerate(need):
            argmax[r] = int(np.argmax(lg[i]))
        info = st.publish(rows, guesses, argmax)
        run.commit(rows, info.commit_rows)
        assert em == info.emitted
    L.la_set_debug(ctx.ctx, 0)


def test_13b_code_like_lookahead_equals_ar():
    """The 13B code-like workload at full size: 40 layers, a 2048-token prompt
    with 30 % copied spans, 512 new tokens, W=10, N=5, G=10."""
    from lookahead_decoding_gb300 import lib
    L = lib()
    cfg = synth.LLAMA_13B
    w = synth.llama_weights(cfg, 0, device="cuda:0")
    ctx = context(cfg, w, max_ctx=2600, W=10, N=5, G=10)
    try:
        p = synth.code_like_prompt(cfg.vocab, 2048, 3).tolist()
        ar = L.la_generate_ar(ctx.ctx, p, 512)
        st = L.la_stats()
        assert L.la_generate(ctx.ctx, p, 512, 10, 5, 10, stats=st) == ar
        assert st.steps < 512
    finally:
        ctx.close()
        del w
        torch.cuda.empty_cache()
