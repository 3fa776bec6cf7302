"""Sampling target and exact multi-draft verification (oracle; test infrastructure).

* ``warp`` — the target sampling distribution: softmax(logits / T), then the
  top-p nucleus (break the sequential dependency paper §2 names greedy, top-K
  and top-P selectors; temperature and top-p shape p before verification,
  speculative-decoding lesson Ch.1 "temperature and top-p ... live inside
  p(x)").  Order of the nucleus: probability descending, ties by lower id;
  keep the shortest prefix whose mass reaches top_p (the crossing token
  included) and renormalise.
* ``verify_position`` — M7.3 §0x05B: test each *distinct* offered token once,
  in candidate order; accept token c with probability residual(c); on
  rejection set its mass to zero and renormalise once; if every offered
  token is rejected, draw from the final residual.
* ``sample_verify`` — M7.3 §0x05B suffix filtering: after a token is
  accepted keep only the candidates that carry it at this offset and read the
  next target distribution from the lowest-index survivor's row; a full
  acceptance of all S offsets ends with a plain draw from the last survivor
  row (the bonus token).

Random decisions go through a *chooser* with two primitives, so the same
control flow runs on Philox uniforms (``PhiloxChooser``) or under an exact
enumeration of every branch with rational weights (``enumerate_law``).
"""
from __future__ import annotations

from fractions import Fraction
from typing import Callable, List, Sequence, Tuple

import numpy as np

from . import philox


def softmax(z: np.ndarray) -> np.ndarray:
    m = np.max(z)
    e = np.exp(z - m)
    return e / np.sum(e)


def warp(logits: np.ndarray, temperature: float, top_p: float) -> np.ndarray:
    """softmax(logits / T) restricted to the top-p nucleus, renormalised."""
    p = softmax(np.asarray(logits, dtype=np.float64) / temperature)
    if top_p >= 1.0:
        return p
    ids = np.arange(len(p))
    order = np.lexsort((ids, -p))            # primary: -p ascending, then id
    cum = np.cumsum(p[order])
    k = int(np.searchsorted(cum, top_p, side="left"))   # first cum >= top_p
    k = min(k, len(p) - 1)
    keep = order[: k + 1]
    q = np.zeros_like(p)
    q[keep] = p[keep]
    return q / q.sum()


def categorical_index(probs, u) -> int:
    """Inverse CDF in id order: the first id whose cumulative mass exceeds u * total."""
    if isinstance(probs, np.ndarray):
        cum = np.cumsum(probs)
        i = int(np.searchsorted(cum, u * cum[-1], side="right"))
        return min(i, len(probs) - 1)
    total = sum(probs)
    acc = 0
    x = u * total
    last = 0
    for i, pr in enumerate(probs):
        if pr > 0:
            last = i
        acc += pr
        if acc > x:
            return i
    return last


class PhiloxChooser:
    """Draws with Philox4x32-10 uniforms keyed by (seed; step, offset, test, purpose)."""

    def __init__(self, seed: int, step: int):
        self.seed, self.step = seed, step

    def bernoulli(self, prob, offset: int, test: int) -> bool:
        return philox.uniform(self.seed, self.step, offset, test, philox.ACCEPT) < prob

    def categorical(self, probs, offset: int, purpose: int) -> int:
        return categorical_index(probs, philox.uniform(self.seed, self.step, offset, 0, purpose))


def _zero_and_renorm(residual, tok):
    if isinstance(residual, np.ndarray):
        r = residual.copy()
        r[tok] = 0.0
        s = r.sum()
        return r if s <= 0 else r / s, s
    r = list(residual)
    r[tok] = 0 * r[tok]
    s = sum(r)
    return (r if s <= 0 else [x / s for x in r]), s


def verify_position(probs, offered: Sequence[int], chooser, offset: int) -> Tuple[int, bool]:
    """One output position: returns (token, accepted_from_candidates)."""
    residual = probs
    tested: List[int] = []
    for tok in offered:
        if tok in tested:            # mass of a rejected token is consumed once
            continue
        t = len(tested)
        tested.append(tok)
        if chooser.bernoulli(residual[tok], offset, t):
            return tok, True
        residual, s = _zero_and_renorm(residual, tok)
        if s <= 0:                   # all remaining mass was this token's
            return tok, True
    return chooser.categorical(residual, offset, philox.RESIDUAL), False


def sample_verify(cands: Sequence[Sequence[int]], out_probs, row_probs: Callable[[int, int], object],
                  chooser) -> Tuple[List[int], int, int]:
    """Sequential verifier over disjoint one-hot proposals.

    cands[c] is candidate c's suffix (S tokens).  row_probs(c, s) is the
    target distribution of the row whose input is cands[c][s] (it predicts
    the token after it).  Returns (emitted, a, winner) where a is the number
    of accepted candidate tokens and winner the lowest-index survivor of the
    accepted prefix (-1 when a = 0): its rows v_{w,0..a-1} are the ones whose
    K/V the call commits, whether the next offset was rejected or all S
    offsets were accepted.
    """
    S = len(cands[0]) if cands else 0
    survivors = list(range(len(cands)))
    p = out_probs
    emitted: List[int] = []
    for off in range(S):
        offered = [cands[c][off] for c in survivors]
        tok, acc = verify_position(p, offered, chooser, off)
        emitted.append(tok)
        if not acc:
            return emitted, off, (survivors[0] if off > 0 else -1)
        survivors = [c for c in survivors if cands[c][off] == tok]
        p = row_probs(survivors[0], off)
    emitted.append(chooser.categorical(p, S, philox.PLAIN))
    return emitted, S, (survivors[0] if S > 0 and survivors else -1)


# ----------------------------------------------------------------------------
# exact enumeration of a chooser-driven procedure
# ----------------------------------------------------------------------------

class _Scripted:
    def __init__(self, script):
        self.script = list(script)
        self.pos = 0
        self.weight = Fraction(1)
        self.branches = []      # (position, n_alternatives) of fresh decisions

    def _take(self, n_alt):
        if self.pos < len(self.script):
            k = self.script[self.pos]
        else:
            k = 0
            self.script.append(0)
            self.branches.append((self.pos, n_alt))
        self.pos += 1
        return k

    def bernoulli(self, prob, offset, test):
        prob = Fraction(prob)
        k = self._take(2)
        self.weight *= prob if k == 0 else (1 - prob)
        return k == 0

    def categorical(self, probs, offset, purpose):
        probs = [Fraction(x) for x in probs]
        k = self._take(len(probs))
        self.weight *= probs[k] / sum(probs)
        return k


def enumerate_law(fn) -> dict:
    """Exact law of fn(chooser) -> hashable outcome, summing rational branch weights.

    Branches of zero weight are explored too but contribute nothing.
    """
    law: dict = {}
    stack = [[]]
    while stack:
        script = stack.pop()
        ch = _Scripted(script)
        out = fn(ch)
        if ch.weight != 0:
            law[out] = law.get(out, Fraction(0)) + ch.weight
        for pos, n_alt in ch.branches:
            for alt in range(1, n_alt):
                stack.append(ch.script[:pos] + [alt])
    return law
