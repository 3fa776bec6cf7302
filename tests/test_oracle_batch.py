"""Pins of the batched packed call (several requests in one forward): every
request's rows, logits, K/V and trajectory equal those of the request run
alone, and each request's output is its autoregressive output."""
import numpy as np
import pytest

import synth
from oracle import batch as ob
from oracle import lookahead as la
from oracle.model import OracleModel, argmax_lowest

MICRO = synth.ModelConfig(n_layers=1, d_model=16, n_heads=2, head_dim=8, d_ffn=32, vocab=6,
                          dtype="f32", init_std=0.5)
SMALL = synth.ModelConfig(n_layers=2, d_model=32, n_heads=4, head_dim=8, d_ffn=64, vocab=16,
                          dtype="f32", init_std=0.3)


def model_for(cfg, seed=0):
    return OracleModel(cfg, synth.llama_weights(cfg, seed))


def _call_of(m, prompt, W, N, G, fills):
    """(tokens, positions, cache, visibility) of a request after ``fills`` calls."""
    cache, lg = m.prefill(prompt)
    st = la.LookaheadState(prompt, argmax_lowest(lg[-1]), W, N, G)
    run = la.make_runner(m, cache, "meta")
    for _ in range(fills):
        rows, g = st.plan()
        L = run.run(rows)
        info = st.publish(rows, g, [argmax_lowest(x) for x in L])
        run.commit(rows, info.commit_rows)
    rows, _ = st.plan()
    return [r.token for r in rows], [r.position for r in rows], cache, la.meta_mask(rows)


def test_forward_many_rows_equal_each_request_alone():
    """Three requests with different prefixes, phases (warm-up and steady) and
    row counts in one forward: each request's logits and new K/V equal its
    own forward's (up to the rounding order of the stacked row-wise products)."""
    m = model_for(SMALL, 3)
    calls = [_call_of(m, [1, 2, 3], 4, 4, 2, 0),
             _call_of(m, [5, 6, 7, 8, 9, 10, 11], 3, 3, 3, 3),
             _call_of(m, [2, 4, 6, 8, 10], 5, 4, 2, 4)]
    assert len({len(c[0]) for c in calls}) > 1
    many = m.forward_many(calls)
    for c, (lg, k, v) in zip(calls, many):
        lg1, k1, v1 = m.forward(*c)
        assert lg.shape == lg1.shape
        np.testing.assert_allclose(lg, lg1, rtol=1e-12, atol=1e-12)
        for a, b in zip(k + v, k1 + v1):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("W,N,G", [(3, 3, 3), (4, 4, 2), (2, 5, 4)])
def test_batched_generate_equals_each_request_alone_and_ar(W, N, G):
    """Batching changes no request's trajectory: per request, every call's rows,
    hit and emitted tokens equal its solo run's, and its output is its AR
    output; requests that finish early leave the batch."""
    left_early = 0
    for seed in range(6):
        m = model_for(MICRO, seed)
        prompts = [list(synth.uniform_prompt(MICRO.vocab, n, 300 + 10 * seed + n)) for n in (4, 7, 5)]
        tr = []
        outs = ob.lookahead_generate_batch(m, prompts, 20, W, N, G, trace=tr)
        for b, p in enumerate(prompts):
            assert outs[b] == la.ar_generate(m, p, 20), (seed, b)
            solo = []
            la.lookahead_generate(m, p, 20, W, N, G, trace=solo)
            mine = [s.infos[s.requests.index(b)] for s in tr if b in s.requests]
            assert [(i.Q, i.a, i.emitted) for i in mine] == [(i.Q, i.a, i.emitted) for i in solo]
        left_early += any(len(s.requests) < len(prompts) for s in tr)
    assert left_early > 0


def test_shared_cache_mistake_is_detected():
    """Planted mistake on the CPU: every request of the batch reads the first
    request's committed K/V.  The per-request AR pin then fails."""
    class SharedCache(ob.BatchedLookahead):
        def step(self, max_new):
            live = self.active(max_new)
            if live:
                self.caches = [self.caches[live[0]]] * len(self.caches)
            return super().step(max_new)

    wrong = 0
    for seed in range(6):
        m = model_for(MICRO, seed)
        prompts = [list(synth.uniform_prompt(MICRO.vocab, n, 500 + 10 * seed + n)) for n in (4, 7)]
        bl = SharedCache(m, prompts, 3, 3, 3)
        while bl.step(12) is not None:
            pass
        wrong += any(bl.out[b][:12] != la.ar_generate(m, p, 12) for b, p in enumerate(prompts))
    assert wrong > 0
