"""Pins of the oracle's sampling verifier, warping, Philox and acceptance model."""
import json
import math
import os
from fractions import Fraction
from itertools import product

import numpy as np
import pytest

from oracle import lookahead as la
from oracle import philox
from oracle import sampling as smp

GOLD = os.path.join(os.path.dirname(__file__), "golden")
G = json.load(open(os.path.join(GOLD, "sampling_examples.json")))


def _p(d, names):
    return [Fraction(d[n]) for n in names]


# ---- Philox known-answer vectors (Random123 distribution, philox4x32_10) ----

@pytest.mark.parametrize("ctr,key,out", [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
])
def test_philox_kat(ctr, key, out):
    assert philox.philox4x32_10(ctr, key) == out
    v = philox.philox4x32_10_np(*[[c] for c in ctr], *key)
    assert tuple(int(x[0]) for x in v) == out


# ---- T9: frozen audit coordinate A/B/C/D -------------------------------------

def test_abcd_worked_example_exact():
    g = G["abcd"]
    names = ["A", "B", "C", "D"]
    p = _p(g["target"], names)
    cands = [names.index(n) for n in g["candidate_rows"]]
    law = smp.enumerate_law(lambda ch: smp.verify_position(p, cands, ch, 0)[0])
    assert {names[k]: v for k, v in law.items()} == {k: Fraction(v) for k, v in g["output"].items()}
    # the residual after rejecting A and B (each tested once, in order)
    r, _ = smp._zero_and_renorm(p, 0)
    r, _ = smp._zero_and_renorm(r, 1)
    assert {names[i]: r[i] for i in (2, 3)} == {k: Fraction(v) for k, v in g["residual_after_A_B"].items()}


def test_worked_example_detects_a_missing_renormalisation():
    """Planted mistake (on the CPU, in a copy of the rule): testing against the
    un-renormalised residual changes the law, so the exact pin has power."""
    g = G["abcd"]
    names = ["A", "B", "C", "D"]
    p = _p(g["target"], names)

    def wrong(ch):
        residual = list(p)
        for t, tok in enumerate([0, 1]):
            if ch.bernoulli(residual[tok], 0, t):
                return tok
            residual[tok] = Fraction(0)          # mass removed but never renormalised
        return ch.categorical(residual, 0, 1)

    law = smp.enumerate_law(wrong)
    assert [law.get(i, 0) for i in range(4)] != p


# ---- T10: p = (0.5, 0.3, 0.2), every one-hot candidate list -----------------------

def test_abc_every_candidate_list_exact():
    p = _p(G["abc"]["target"], ["A", "B", "C"])
    for n in range(0, 4):
        for cands in product(range(3), repeat=n):
            law = smp.enumerate_law(lambda ch: smp.verify_position(p, list(cands), ch, 0)[0])
            assert [law.get(i, 0) for i in range(3)] == p, cands


def test_abc_chi_square_1e6():
    """1e6 verifier runs on Philox uniforms; chi-square with df=2 at alpha=0.001."""
    p = np.array([0.5, 0.3, 0.2])
    n = 1_000_000
    seed = 1234
    # uniforms of the same generator the verifier's PhiloxChooser uses, drawn in bulk
    i = np.arange(n, dtype=np.uint64)
    acc = [philox.philox4x32_10_np(i, np.uint64(0), np.uint64(t), np.uint64(philox.ACCEPT),
                                   seed, 0)[0] >> np.uint64(8) for t in range(2)]
    res = philox.philox4x32_10_np(i, 0, 0, np.uint64(philox.RESIDUAL), seed, 0)[0] >> np.uint64(8)
    acc = [a.astype(np.float64) / 16777216.0 for a in acc]
    res = res.astype(np.float64) / 16777216.0

    class Bulk:
        k = 0

        def bernoulli(self, prob, offset, test):
            return acc[test][self.k] < prob

        def categorical(self, probs, offset, purpose):
            return smp.categorical_index(probs, res[self.k])

    ch = Bulk()
    counts = np.zeros(3)
    cands = [1, 1, 2]            # B, B, C: duplicates and a residual draw
    for k in range(n):
        ch.k = k
        counts[smp.verify_position(p, cands, ch, 0)[0]] += 1
    # spot-check the bulk uniforms against the scalar chooser
    for k in (0, 1, 99999):
        assert acc[0][k] == philox.uniform(seed, k, 0, 0, philox.ACCEPT)
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 13.816, (counts, chi2)     # chi-square(2) upper 0.001 quantile


# ---- multi-step exactness on a toy conditional table --------------------------------

def test_multistep_joint_law_equals_ar():
    """Joint law of the first 3 tokens from the sequential verifier equals AR sampling."""
    V = 3
    rnd = np.random.default_rng(3)
    table = {}

    def cond(prefix):
        if prefix not in table:
            w = rnd.integers(1, 6, size=V)
            table[prefix] = [Fraction(int(x), int(w.sum())) for x in w]
        return table[prefix]

    cands = [(0, 1), (0, 2), (1, 1), (2, 0)]     # S = 2, shared first tokens

    def run(ch):
        em, a, w = smp.sample_verify(cands, cond(()), lambda c, s: cond(tuple(cands[c][: s + 1])), ch)
        seq = list(em)
        while len(seq) < 3:                      # continue autoregressively
            seq.append(ch.categorical(cond(tuple(seq)), 9, 2))
        return tuple(seq[:3])

    law = smp.enumerate_law(run)
    for seq in product(range(V), repeat=3):
        ar = cond(())[seq[0]] * cond(seq[:1])[seq[1]] * cond(seq[:2])[seq[2]]
        assert law.get(seq, 0) == ar, seq


def test_winner_is_the_lowest_survivor_of_the_accepted_prefix():
    """Over every outcome of the verifier (exact enumeration): with a > 0 the
    winner is the lowest-index candidate whose first a tokens are the emitted
    ones (its rows v_{w,0..a-1} carry the K/V the call commits), also when
    the next offset is rejected; with a = 0 there is none (-1)."""
    V = 3
    rnd = np.random.default_rng(11)
    table = {}

    def cond(prefix):
        if prefix not in table:
            w = rnd.integers(1, 6, size=V)
            table[prefix] = [Fraction(int(x), int(w.sum())) for x in w]
        return table[prefix]

    cands = [(1, 2, 0), (0, 1, 1), (0, 1, 2), (1, 2, 2), (0, 2, 0)]     # S = 3, shared prefixes
    seen = []

    def run(ch):
        em, a, w = smp.sample_verify(cands, cond(()), lambda c, s: cond(tuple(cands[c][: s + 1])), ch)
        want = min((c for c in range(len(cands)) if list(cands[c][:a]) == list(em[:a])), default=-1) if a else -1
        seen.append((a, w, want))
        return (a, w)

    smp.enumerate_law(run)
    assert all(w == want for _, w, want in seen)
    assert any(0 < a < 3 for a, _, _ in seen) and any(a == 3 for a, _, _ in seen)


def test_sampled_lookahead_commits_the_verified_rows():
    """A sampled lookahead decode of a tiny model (vocabulary 5, peaked
    logits, so candidates are accepted and rejected at every offset): after
    each call the committed K/V equals that of one causal forward over the
    prompt and the emitted tokens (every committed row is the row of an
    emitted token at its position), so the next call reads the same prefix
    AR sampling would."""
    from oracle import lookahead as la
    from oracle.model import KVCache, OracleModel
    import synth
    cfg = synth.ModelConfig(n_layers=1, d_model=16, n_heads=2, head_dim=8, d_ffn=32, vocab=5, dtype="f32",
                            init_std=0.8)
    m = OracleModel(cfg, synth.llama_weights(cfg, 7))
    prompt = [1, 2, 3, 1, 2, 3, 1, 2]
    samp = la.Sampling(1.0, 1.0, 55)
    cache, lg = m.prefill(prompt)
    out = [la._first_token(lg[-1], samp)]
    st = la.LookaheadState(prompt, out[0], 3, 4, 3)
    run = la.make_runner(m, cache, "meta")
    partial = 0
    while len(out) < 60:
        rows, guesses = st.plan()
        logits = run.run(rows)
        verdict = la.sample_step(logits, rows, guesses, st, samp)
        info = st.publish(rows, guesses, [int(np.argmax(x)) for x in logits], verdict)
        run.commit(rows, info.commit_rows)
        partial += 0 < info.a < st.S and len(guesses) > 0
        out.extend(info.emitted)
        _, rk, rv = m.forward(prompt + out[:-1], list(range(len(prompt) + len(out) - 1)), KVCache(1),
                              np.tril(np.ones((len(prompt) + len(out) - 1,) * 2, dtype=bool)))
        assert np.allclose(run.cache.k[0], rk[0], rtol=0, atol=1e-9)
        assert np.allclose(run.cache.v[0], rv[0], rtol=0, atol=1e-9)
    assert partial > 0          # some call accepted part of a suffix and rejected the rest


# ---- warping ---------------------------------------------------------------------

def test_warp_temperature_and_top_p():
    logits = np.log(np.array([0.1, 0.4, 0.2, 0.3]))
    q = smp.warp(logits, 1.0, 1.0)
    assert np.allclose(q, [0.1, 0.4, 0.2, 0.3])
    q = smp.warp(logits, 1.0, 0.65)       # sorted 0.4, 0.3 (0.7 >= 0.65) -> keep B, D
    assert np.allclose(q, [0, 0.4 / 0.7, 0, 0.3 / 0.7])
    q = smp.warp(logits, 1.0, 0.4)        # the crossing token alone
    assert np.allclose(q, [0, 1, 0, 0])
    q = smp.warp(np.log(np.array([0.25, 0.25, 0.25, 0.25])), 1.0, 0.5)   # ties by lower id
    assert np.allclose(q, [0.5, 0.5, 0, 0])
    q = smp.warp(logits, 0.5, 1.0)        # p^(1/T) renormalised
    r = np.array([0.1, 0.4, 0.2, 0.3]) ** 2
    assert np.allclose(q, r / r.sum())


# ---- T11: expected accepted tokens ---------------------------------------------------

def expected_tokens(alpha, gamma, b):
    return (gamma + 1) - sum((1 - alpha ** i) ** b for i in range(1, gamma + 1))


def test_expected_tokens_closed_form():
    g = G["expected_tokens"]
    v = expected_tokens(g["alpha"], g["gamma"], g["b"])
    assert abs(v - g["value"]) < 5e-5
    assert abs(v - (1 - g["alpha"] ** (g["gamma"] + 1)) / (1 - g["alpha"])) < 1e-12


@pytest.mark.parametrize("alpha,S,b", [(0.7, 4, 1), (0.5, 3, 4), (0.3, 4, 15)])
def test_greedy_acceptance_matches_model(alpha, S, b):
    rnd = np.random.default_rng(7)
    n = 20000
    tot = np.zeros(n)
    truth = list(range(1, S + 2))            # the target continuation 1, 2, ..., S+1
    for k in range(n):
        guesses = []
        for c in range(b):
            ok = rnd.random(S) < alpha
            guesses.append(tuple(truth[i] if ok[i] else 100 + i for i in range(S)))
        a, w, em = la.greedy_verify(truth[0], guesses, lambda c, s: truth[s + 1])
        tot[k] = len(em)
    m, sd = tot.mean(), tot.std() / math.sqrt(n)
    assert abs(m - expected_tokens(alpha, S, b)) < 4 * sd + 1e-9
