"""Pins of the Lookahead Parallelism oracle (oracle/lp.py): with P replicas
sharing the columns and candidates, re-feeding the emitted tokens instead of
copying candidate K/V, every call's verdict, the emitted stream and the
number of calls equal the single-worker loop's, which equals autoregressive
greedy decoding."""
import numpy as np
import pytest

import synth
from oracle import lookahead as la
from oracle import lp
from oracle.model import OracleModel


def tiny(vocab, seed):
    cfg = synth.ModelConfig(n_layers=1, d_model=16, n_heads=2, head_dim=8, d_ffn=32, vocab=vocab, dtype="f32",
                            init_std=0.5)
    return OracleModel(cfg, synth.llama_weights(cfg, seed))


def test_shard_plan_covers_everything_once():
    for W in (1, 5, 7, 15):
        for P in (1, 2, 3, 4):
            cols = [c for k in range(P) for c in lp.shard_columns(W, P, k)]
            assert cols == list(range(W))
            for C in (0, 1, 5, 15):
                cands = sorted(c for k in range(P) for c in lp.shard_candidates(C, P, k))
                assert cands == list(range(C))


@pytest.mark.parametrize("P", [2, 3, 4])
@pytest.mark.parametrize("W,N,G", [(5, 3, 5), (4, 4, 4), (7, 5, 6)])
def test_lp_equals_single_worker_and_ar(P, W, N, G):
    hits = 0
    for seed in range(4):
        m = tiny(6, seed)
        prompt = [int(t) for t in np.random.default_rng(seed).integers(0, 6, 10)]
        ref_trace, lp_trace = [], []
        ref = la.lookahead_generate(m, prompt, 40, W, N, G, trace=ref_trace)
        got = lp.lp_generate(m, prompt, 40, W, N, G, P, trace=lp_trace)
        assert got == ref == la.ar_generate(m, prompt, 40)
        assert len(lp_trace) == len(ref_trace)
        for a, b in zip(lp_trace, ref_trace):
            assert (a.Q, a.C_t, a.a, a.winner, a.emitted) == (b.Q, b.C_t, b.a, b.winner, b.emitted)
        hits += sum(t.a > 0 for t in lp_trace)
    assert hits > 0          # candidates were accepted, so the re-feed path ran


def test_lp_without_refeed_fails():
    """A planted mistake: after a hit, committing only the ordinary row and not
    re-feeding the accepted tokens loses them from every replica's K/V."""
    m = tiny(6, 1)
    prompt = [int(t) for t in np.random.default_rng(1).integers(0, 6, 10)]
    ar = la.ar_generate(m, prompt, 40)
    orig = lp.Worker.forward

    def forward_without_refeed(self, rows):
        self.refeed = self.refeed[-1:]
        return orig(self, rows)

    lp.Worker.forward = forward_without_refeed
    try:
        with pytest.raises(AssertionError):
            assert lp.lp_generate(m, prompt, 40, 5, 3, 5, 2) == ar
    finally:
        lp.Worker.forward = orig
