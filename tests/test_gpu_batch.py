"""Several requests in one packed call on the GPU: every request's output is
bit-exact with its own la_generate run and its autoregressive output (the
definition the oracle's batched call writes out), with requests of different
prompt lengths that finish after different numbers of calls; and the batched
calls against the oracle's batched forward (oracle/batch.py): per request,
the needed rows, their logits within 3e-2 and the tokens, call by call."""
import numpy as np
import pytest

import synth
from lookahead_decoding_gb300._lib import LaError
from oracle.batch import BatchedLookahead
from oracle.model import OracleModel
from tests.gpu_util import top2_gap, weights

LOGIT_TOL = 3e-2
TIE = 1e-2

pytestmark = pytest.mark.gpu

MID = synth.ModelConfig(n_layers=2, d_model=512, n_heads=4, head_dim=128, d_ffn=1408, vocab=4096, dtype="bf16")


@pytest.fixture(scope="module")
def batched():
    from lookahead_decoding_gb300 import lib
    L = lib()
    w = weights(MID, 0)
    ctx = L.Context(MID, w, max_ctx=512, max_W=8, max_N=5, max_G=8, max_batch=3)
    yield L, ctx, w
    ctx.close()


def prompts(seed):
    base = synth.markov_zipf_prompt(MID.vocab, 24, seed).tolist()
    return [synth.markov_zipf_prompt(MID.vocab, 40, seed + 1).tolist(),
            base + base + base,
            synth.markov_zipf_prompt(MID.vocab, 96, seed + 2).tolist()]


@pytest.mark.parametrize("W,N,G", [(8, 5, 8), (4, 3, 4), (1, 3, 1)])
def test_batch_equals_solo_and_ar(batched, W, N, G):
    L, ctx, _ = batched
    ps = prompts(11)
    ar = [L.la_generate_ar(ctx.ctx, p, 48) for p in ps]
    solo_steps = []
    for p, a in zip(ps, ar):
        st = L.la_stats()
        assert L.la_generate(ctx.ctx, p, 48, W, N, G, stats=st) == a
        solo_steps.append(st.steps)
    st = L.la_stats()
    got = L.la_generate_batch(ctx.ctx, ps, 48, W, N, G, stats=st)
    assert got == ar, (W, N, G)
    assert st.steps == max(solo_steps) and st.tokens == 3 * 48


def test_batch_with_pool_seeding_equals_ar(batched):
    """Seeded pools make the requests accept different numbers of tokens, so
    they leave the batch after different numbers of calls."""
    L, ctx, _ = batched
    ps = prompts(21)
    ar = [L.la_generate_ar(ctx.ctx, p, 64) for p in ps]
    L.la_set_options(ctx.ctx, L.LA_OPT_POOL_FROM_PROMPT | L.LA_OPT_POOL_FROM_OUTPUT)
    try:
        assert L.la_generate_batch(ctx.ctx, ps, 64, 8, 5, 8) == ar
        assert L.la_generate_batch(ctx.ctx, ps[:2], 64, 8, 5, 8) == ar[:2]
    finally:
        L.la_set_options(ctx.ctx, 0)


def test_batch_of_one_and_single_request_after_a_batch(batched):
    L, ctx, _ = batched
    p = prompts(31)[2]
    ar = L.la_generate_ar(ctx.ctx, p, 32)
    assert L.la_generate_batch(ctx.ctx, [p], 32, 4, 4, 4) == [ar]
    assert L.la_generate(ctx.ctx, p, 32, 4, 4, 4) == ar


def test_batch_errors(batched):
    L, ctx, _ = batched
    p = prompts(41)[0]
    with pytest.raises(LaError):
        L.la_generate_batch(ctx.ctx, [p] * 4, 16, 4, 3, 4)           # more requests than the context holds
    with pytest.raises(LaError):
        L.la_generate_batch(ctx.ctx, [p, [1] * 500], 16, 4, 3, 4)    # prompt + max_new above max_ctx


def test_batch_sampling_equals_each_request_alone(batched):
    """Sampling in a batch: request b, drawing with seed + b, emits exactly its
    solo sampled la_generate output with that seed (same logits rows, same
    Philox counters)."""
    L, ctx, _ = batched
    ps = prompts(51)
    T, top_p, seed = 0.8, 0.9, 700
    solo = [L.la_generate(ctx.ctx, p, 40, 8, 5, 8, sampling=(T, top_p, seed + b)) for b, p in enumerate(ps)]
    got = L.la_generate_batch(ctx.ctx, ps, 40, 8, 5, 8, sampling=(T, top_p, seed))
    assert got == solo
    again = L.la_generate_batch(ctx.ctx, ps, 40, 8, 5, 8, sampling=(T, top_p, seed))
    assert again == got


@pytest.mark.parametrize("W,N,G", [(8, 5, 8), (4, 3, 4)])
def test_batched_calls_against_oracle(batched, W, N, G):
    """Calls 1 .. 6 of a batch of three requests against the oracle's batched
    forward (oracle/batch.py).  la_generate_batch stopped after k calls keeps
    the k-th call's needed-row logits per request; per request they must be
    within 3e-2 of the oracle's, on the same rows (tokens, positions), with the
    same argmax unless the oracle's top-2 gap is below 1e-2.  The oracle's
    state machine then takes the GPU's argmax, so both follow one trajectory
    (a near-tie resolved differently would otherwise part the windows)."""
    L, ctx, w = batched
    ps = prompts(61)
    oracle = OracleModel(MID, {k: v.cpu() for k, v in w.items()}, store="bf16")
    bl = BatchedLookahead(oracle, ps, W, N, G)
    first = L.la_generate_batch(ctx.ctx, ps, 1, W, N, G)
    for b in range(3):
        if first[b][0] != bl.out[b][0]:
            assert top2_gap(oracle.prefill(ps[b])[1][-1]) < TIE
            bl.out[b][0] = first[b][0]
            bl.states[b].x_t = first[b][0]
            bl.states[b].seq[-1] = first[b][0]
    L.la_set_debug(ctx.ctx, 1)
    try:
        for k in range(1, 7):
            got = L.la_generate_batch(ctx.ctx, ps, k + 1, W, N, G)
            gpu = []
            for b in range(3):
                _, _, tok, pos, _ = L.la_debug_state(ctx.ctx, b)
                lg, need = L.la_debug_batch_logits(ctx.ctx, b, 1024, MID.vocab)
                gpu.append((tok, pos, lg, need.tolist()))

            def choose(b, logits, need):
                tok, pos, lg, gneed = gpu[b]
                assert gneed == need, (k, b)
                ref = logits[need]
                err = float(np.max(np.abs(lg - ref)))
                assert err < LOGIT_TOL, (k, b, err)
                am = [0] * len(logits)
                for i, r in enumerate(need):
                    am[r] = int(np.argmax(lg[i]))
                    assert am[r] == int(np.argmax(ref[i])) or top2_gap(ref[i]) < TIE, (k, b, r)
                return am

            step = bl.step(10 ** 6, choose)
            for b in range(3):
                assert gpu[b][0] == step.tokens[b] and gpu[b][1] == step.positions[b], (k, b)
                assert got[b] == bl.out[b][: k + 1], (k, b)
            # the k-th call's logits are the last call's only while every request
            # emits one token per call (then all three run exactly k calls)
            if any(len(o) != k + 1 for o in bl.out):
                break
    finally:
        L.la_set_debug(ctx.ctx, 0)
