"""Several requests in one packed call on the GPU: every request's output is
bit-exact with its own la_generate run and its autoregressive output (the
definition the oracle's batched call writes out), with requests of different
prompt lengths that finish after different numbers of calls."""
import pytest

import synth
from lookahead_decoding_gb300._lib import LaError
from tests.gpu_util import weights

pytestmark = pytest.mark.gpu

MID = synth.ModelConfig(n_layers=2, d_model=512, n_heads=4, head_dim=128, d_ffn=1408, vocab=4096, dtype="bf16")


@pytest.fixture(scope="module")
def batched():
    from lookahead_decoding_gb300 import lib
    L = lib()
    w = weights(MID, 0)
    ctx = L.Context(MID, w, max_ctx=512, max_W=8, max_N=5, max_G=8, max_batch=3)
    yield L, ctx
    ctx.close()


def prompts(seed):
    base = synth.markov_zipf_prompt(MID.vocab, 24, seed).tolist()
    return [synth.markov_zipf_prompt(MID.vocab, 40, seed + 1).tolist(),
            base + base + base,
            synth.markov_zipf_prompt(MID.vocab, 96, seed + 2).tolist()]


@pytest.mark.parametrize("W,N,G", [(8, 5, 8), (4, 3, 4), (1, 3, 1)])
def test_batch_equals_solo_and_ar(batched, W, N, G):
    L, ctx = batched
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
    L, ctx = batched
    ps = prompts(21)
    ar = [L.la_generate_ar(ctx.ctx, p, 64) for p in ps]
    L.la_set_options(ctx.ctx, L.LA_OPT_POOL_FROM_PROMPT | L.LA_OPT_POOL_FROM_OUTPUT)
    try:
        assert L.la_generate_batch(ctx.ctx, ps, 64, 8, 5, 8) == ar
        assert L.la_generate_batch(ctx.ctx, ps[:2], 64, 8, 5, 8) == ar[:2]
    finally:
        L.la_set_options(ctx.ctx, 0)


def test_batch_of_one_and_single_request_after_a_batch(batched):
    L, ctx = batched
    p = prompts(31)[2]
    ar = L.la_generate_ar(ctx.ctx, p, 32)
    assert L.la_generate_batch(ctx.ctx, [p], 32, 4, 4, 4) == [ar]
    assert L.la_generate(ctx.ctx, p, 32, 4, 4, 4) == ar


def test_batch_errors(batched):
    L, ctx = batched
    p = prompts(41)[0]
    with pytest.raises(LaError):
        L.la_generate_batch(ctx.ctx, [p] * 4, 16, 4, 3, 4)           # more requests than the context holds
    with pytest.raises(LaError):
        L.la_generate_batch(ctx.ctx, [p, [1] * 500], 16, 4, 3, 4)    # prompt + max_new above max_ctx


def test_batch_sampling_equals_each_request_alone(batched):
    """Sampling in a batch: request b, drawing with seed + b, emits exactly its
    solo sampled la_generate output with that seed (same logits rows, same
    Philox counters)."""
    L, ctx = batched
    ps = prompts(51)
    T, top_p, seed = 0.8, 0.9, 700
    solo = [L.la_generate(ctx.ctx, p, 40, 8, 5, 8, sampling=(T, top_p, seed + b)) for b, p in enumerate(ps)]
    got = L.la_generate_batch(ctx.ctx, ps, 40, 8, 5, 8, sampling=(T, top_p, seed))
    assert got == solo
    again = L.la_generate_batch(ctx.ctx, ps, 40, 8, 5, 8, sampling=(T, top_p, seed))
    assert again == got
