"""GPU exact-sampling verifier against the oracle and against the target law.

* the 3-token toy p = (0.5, 0.3, 0.2) of the speculative-decoding lesson
  (Ch. 1) with one-hot candidates B, B, C: the emitted token's law over 1e6
  verifier runs equals p (chi-square, df 2, alpha 0.001);
* a two-offset candidate set with shared first tokens: the joint law of the
  first two output tokens over 1e6 runs equals autoregressive sampling;
* the same rows and Philox counters give the oracle's decisions exactly;
* the whole state machine in sampling mode with injected logits follows the
  oracle call by call.
"""
import numpy as np
import pytest

import synth
from oracle import lookahead as la
from oracle import philox
from oracle import sampling as smp
from tests.gpu_util import context, top2_gap

pytestmark = pytest.mark.gpu

CHI2_DF2_001 = 13.816
CHI2_DF8_001 = 26.124


def L():
    from lookahead_decoding_gb300 import lib
    return lib()


def test_toy_three_token_law_1e6():
    p = np.array([0.5, 0.3, 0.2])
    logits = np.zeros((4, 3), dtype=np.float32)
    logits[:] = np.log(p).astype(np.float32)
    cands = [[1], [1], [2]]                       # B, B, C
    n = 1_000_000
    out = L().la_debug_sample_verify(logits, cands, (1.0, 1.0, 20240), n)
    first = out[:, 2]
    counts = np.bincount(first, minlength=3)[:3]
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < CHI2_DF2_001, (counts, chi2)
    # accepted candidate tokens carry their own mass, the residual the rest
    acc = out[:, 1] == 1
    assert abs(acc.mean() - 0.5) < 0.005          # P(accept B or C) = p(B) + p(C)


def test_two_offset_joint_law_1e6():
    V = 3
    rng = np.random.default_rng(4)
    p0 = np.array([0.45, 0.35, 0.2])
    cond = {t: rng.dirichlet(np.ones(V)) for t in range(V)}      # law of the 2nd token after token t
    cands = [[0, 1], [0, 2], [1, 1]]
    S = 2
    rows = np.zeros((1 + 3 * S, V), dtype=np.float32)
    rows[0] = np.log(p0)
    for c, g in enumerate(cands):
        rows[1 + c * S + 0] = np.log(cond[g[0]])
        rows[1 + c * S + 1] = np.log(np.ones(V) / V)             # bonus rows (not tested here)
    n = 1_000_000
    out = L().la_debug_sample_verify(rows, cands, (1.0, 1.0, 777), n)
    t1 = out[:, 2]
    t2 = out[:, 3].copy()
    # when the call stopped after one token, the next call would read cond[t1]
    short = out[:, 0] == 1
    for t in range(V):
        m = short & (t1 == t)
        t2[m] = rng.choice(V, size=int(m.sum()), p=cond[t])
    joint = np.zeros((V, V))
    np.add.at(joint, (t1, t2), 1)
    exp = n * np.array([[p0[a] * cond[a][b] for b in range(V)] for a in range(V)], dtype=np.float64)
    chi2 = float(((joint - exp) ** 2 / exp).sum())
    assert chi2 < CHI2_DF8_001, (joint, exp, chi2)


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.8, 0.9), (0.5, 0.6)])
def test_decisions_match_oracle(T, top_p):
    V, S = 16, 3
    rng = np.random.default_rng(9)
    cands = [[3, 5, 1], [3, 5, 2], [7, 1, 1], [3, 4, 4], [0, 0, 0]]
    rows = rng.normal(size=(1 + len(cands) * S, V)).astype(np.float32) * 1.5
    # survivors with one accepted prefix must read identical rows
    for c, g in enumerate(cands):
        for c2, g2 in enumerate(cands):
            for s in range(S):
                if list(g[: s + 1]) == list(g2[: s + 1]):
                    rows[1 + c2 * S + s] = rows[1 + c * S + s]
    seed, n = 31337, 3000
    out = L().la_debug_sample_verify(rows, cands, (T, top_p, seed), n)
    lg = rows.astype(np.float64)
    mism = 0
    for i in range(n):
        ch = smp.PhiloxChooser(seed, i)
        em, a, w = smp.sample_verify(cands, smp.warp(lg[0], T, top_p),
                                     lambda c, s: smp.warp(lg[1 + c * S + s], T, top_p), ch)
        got = [int(x) for x in out[i, 2: 2 + out[i, 0]]]
        if got != em or int(out[i, 1]) != a:
            mism += 1
    assert mism <= 1, mism


def fake_logits(rows, V, seed=5):
    """A stand-in model for the sampling state machine: each row's logits are a
    fixed random vector chosen by the last two tokens of its visible path,
    peaked on a few tokens so that pool hits and acceptances are frequent."""
    sets = la.vis_sets(rows)
    out = np.zeros((len(rows), V), dtype=np.float32)
    for i, (rw, s) in enumerate(zip(rows, sets)):
        path = [rows[j].token for j in sorted(s, key=lambda j: rows[j].position)]
        a = path[-1]
        b = path[-2] if len(path) > 1 else 0
        r = np.random.default_rng(seed * 1000003 + a * 1009 + b)
        v = np.full(V, -8.0, dtype=np.float32)
        hot = r.choice(8, size=3, replace=False)
        v[hot] = r.normal(size=3).astype(np.float32) * 0.7 + 2.0
        out[i] = v
    return out


@pytest.mark.parametrize("opts", [0, 4])
@pytest.mark.parametrize("W,N,G", [(5, 3, 5), (3, 4, 2), (6, 5, 6)])
def test_sampling_state_machine_with_injected_logits(W, N, G, opts):
    """Sampling verdicts, frontier and window against the oracle, with the
    pinned window schedule (opts 0) and ALWAYS_FWD_ONE=False (opts 4)."""
    cfg = synth.TINY
    w = {k: v.to("cuda:0") for k, v in synth.llama_weights(cfg, 0).items()}
    ctx = context(cfg, w, max_ctx=512, W=8, N=5, G=8)
    Lb = L()
    try:
        Lb.la_set_options(ctx.ctx, opts)
        T, top_p, seed = 0.9, 0.95, 4242
        p = [1, 2, 3, 4, 5, 6, 7, 0]
        first = Lb.la_prefill(ctx.ctx, p, sampling=(T, top_p, seed))
        st = la.LookaheadState(p, first, W, N, G, slice_window=bool(opts & 4))
        samp = la.Sampling(T, top_p, seed)
        mism = 0
        total_a = 0
        for step in range(40):
            rows, guesses = st.plan()
            lg = fake_logits(rows, cfg.vocab)
            argmax = [int(np.argmax(x)) for x in lg]
            em = Lb.la_step_inject(ctx.ctx, W, N, G, argmax, sampling=(T, top_p, seed), logits=lg)
            verdict = la.sample_step(lg.astype(np.float64), rows, guesses, st, samp)
            if em != verdict[0]:
                mism += 1
                # follow the GPU (a decision within rounding of a boundary)
                h = Lb.la_debug_state(ctx.ctx)[0]
                verdict = (em, h["a"], h["winner"])
            info = st.publish(rows, guesses, argmax, verdict)
            total_a += info.a
            h, lv, _, _, _ = Lb.la_debug_state(ctx.ctx)
            assert h["K"] == st.p and h["x_t"] == st.x_t
            assert lv[: N - 1] == [None if l is None else list(l) for l in st.levels]
        assert mism <= 1
        assert total_a > 0
    finally:
        ctx.close()


def test_generate_sampling_runs_and_is_seeded():
    cfg = synth.TINY
    w = {k: v.to("cuda:0") for k, v in synth.llama_weights(cfg, 0).items()}
    ctx = context(cfg, w, max_ctx=256, W=5, N=3, G=5)
    Lb = L()
    try:
        p = synth.uniform_prompt(cfg.vocab, 32, 1).tolist()
        a = Lb.la_generate(ctx.ctx, p, 48, 5, 3, 5, sampling=(0.8, 0.9, 1))
        b = Lb.la_generate(ctx.ctx, p, 48, 5, 3, 5, sampling=(0.8, 0.9, 1))
        c = Lb.la_generate(ctx.ctx, p, 48, 5, 3, 5, sampling=(0.8, 0.9, 2))
        assert a == b and a != c
        assert all(0 <= t < cfg.vocab for t in a)
        ar = Lb.la_generate_ar(ctx.ctx, p, 48, sampling=(0.8, 0.9, 1))
        assert len(ar) == 48
    finally:
        ctx.close()


def test_sampling_on_a_large_vocabulary_after_a_small_one():
    """The sampling verifier holds one fp32 row of the vocabulary in shared
    memory: after the 512-token model, a 32000-token one (128 KB) still
    samples, in range and reproducibly per seed."""
    Lb = L()
    small = synth.TINY
    ws = {k: v.to("cuda:0") for k, v in synth.llama_weights(small, 0).items()}
    c0 = context(small, ws, max_ctx=128, W=4, N=3, G=4)
    try:
        p = synth.uniform_prompt(small.vocab, 8, 3).tolist()
        assert len(Lb.la_generate(c0.ctx, p, 8, 4, 3, 4, sampling=(0.8, 0.9, 7))) == 8
    finally:
        c0.close()
    big = synth.ModelConfig(n_layers=1, d_model=512, n_heads=4, head_dim=128, d_ffn=1408, vocab=32000, dtype="bf16")
    wb = {k: v.to("cuda:0") for k, v in synth.llama_weights(big, 1).items()}
    c1 = context(big, wb, max_ctx=128, W=4, N=3, G=4)
    try:
        p = synth.uniform_prompt(big.vocab, 8, 4).tolist()
        a = Lb.la_generate(c1.ctx, p, 24, 4, 3, 4, sampling=(0.8, 0.9, 11))
        b = Lb.la_generate(c1.ctx, p, 24, 4, 3, 4, sampling=(0.8, 0.9, 11))
        c = Lb.la_generate(c1.ctx, p, 24, 4, 3, 4, sampling=(0.8, 0.9, 12))
        assert a == b and a != c and len(a) == 24
        assert all(0 <= t < big.vocab for t in a)
    finally:
        c1.close()


MID = synth.ModelConfig(n_layers=2, d_model=512, n_heads=4, head_dim=128, d_ffn=1408, vocab=4096, dtype="bf16")


@pytest.mark.parametrize("T,top_p", [(0.8, 0.9), (0.1, 0.9)])
def test_sampled_steps_with_real_logits_against_oracle(T, top_p):
    """The whole sampled packed call on a real bf16 model (2 layers, d 512,
    vocabulary 4096), call by call: every needed row's logits are within 3e-2
    of the oracle's (fp64, bf16 storage emulation), and the call's verdict
    (emitted tokens, accepted count, winner) is the oracle's exact sampling
    verifier applied to the GPU's own logits with the same Philox counters,
    except at most one decision that a uniform within rounding of a
    probability boundary may flip.  (Against the oracle's logits instead,
    decisions on a nearly flat 4096-token law move whenever a 3e-2 logit
    difference shifts a boundary past the uniform, so the verifier is checked
    on identical inputs.)  The oracle's state takes the GPU's decisions, so both
    follow one trajectory."""
    from oracle.model import OracleModel
    w = synth.llama_weights(MID, 0, device="cuda:0")
    ctx = context(MID, w, max_ctx=512, W=8, N=4, G=8)
    Lb = L()
    W, N, G = 8, 4, 8
    seed = 90210
    try:
        Lb.la_set_options(ctx.ctx, Lb.LA_OPT_POOL_FROM_PROMPT | Lb.LA_OPT_POOL_FROM_OUTPUT)
        Lb.la_set_debug(ctx.ctx, 1)
        oracle = OracleModel(MID, {k: v.cpu() for k, v in w.items()}, store="bf16")
        base = synth.markov_zipf_prompt(MID.vocab, 20, 3).tolist()
        p = base + base + base                      # recurring n-grams: the pool retrieves candidates
        samp = la.Sampling(T, top_p, seed)
        first = Lb.la_prefill(ctx.ctx, p, sampling=(T, top_p, seed))
        lg0, _ = Lb.la_debug_logits(ctx.ctx, 2, MID.vocab)
        cache, ref0 = oracle.prefill(p)
        assert np.max(np.abs(lg0[0] - ref0[-1])) < 3e-2
        mism = int(la._first_token(lg0[0].astype(np.float64), samp) != first)
        st = la.LookaheadState(p, first, W, N, G, pool_from_prompt=True, pool_from_output=True)
        run = la.make_runner(oracle, cache, "meta")
        verified = accepted = 0
        for step in range(30):
            rows, guesses = st.plan()
            refl = run.run(rows)
            em = Lb.la_step(ctx.ctx, W, N, G, sampling=(T, top_p, seed))
            h = Lb.la_debug_state(ctx.ctx)[0]
            assert h["Q"] == len(rows) and h["C_t"] == len(guesses)
            lg, need = Lb.la_debug_logits(ctx.ctx, 1024, MID.vocab)
            assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
            assert np.max(np.abs(lg - refl[need])) < 3e-2, step
            full = np.zeros_like(refl)
            full[need] = lg.astype(np.float64)
            verdict = la.sample_step(full, rows, guesses, st, samp)
            gpu = (em, h["a"], h["winner"])
            if (verdict[0], verdict[1]) != (em, h["a"]) or (h["a"] > 0 and verdict[2] != h["winner"]):
                mism += 1
            verified += bool(guesses)
            accepted += h["a"] > 0
            # the state follows the GPU's call: its verdict and its argmax of the
            # needed rows (equal to the oracle's unless the oracle nearly ties)
            argmax = [0] * len(rows)
            for i, r in enumerate(need):
                argmax[r] = int(np.argmax(lg[i]))
                assert argmax[r] == int(np.argmax(refl[r])) or top2_gap(refl[r]) < 1e-2
            info = st.publish(rows, guesses, argmax, gpu)
            run.commit(rows, info.commit_rows)
            assert h["K"] == st.p and h["x_t"] == st.x_t
        assert mism <= 1, mism
        assert verified > 0
        if T < 0.5:
            assert accepted > 0
    finally:
        ctx.close()
