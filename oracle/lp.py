"""Lookahead Parallelism (oracle; test infrastructure): P workers, each a full
model replica, share one packed call (M7.3 §0x07A, "Lookahead Parallelism:
replicated-model token parallelism" and the pinned distributed path; break
the sequential dependency §3.4).

What the pages fix: every worker keeps the whole model and the shared
prefix; the lookahead branches and the verification candidates are split
into disjoint shares, one per worker; nothing is exchanged during the
forward; after it the workers all-gather the verification decision (each
share's longest hit) and the generated window slices; the K/V of accepted
candidate rows is not copied between workers: every worker truncates its
cache to its ordinary rows and re-feeds the emitted tokens through the next
call.

Readings taken where the pages leave the details open:
  - columns: worker k owns the contiguous window columns
    [k W / P, (k + 1) W / P) of every trajectory level, and computes the base
    stripe b_1 .. b_j its columns' rows see (the shared prefix is computed
    redundantly); candidates: worker k owns pool slots c with c mod P = k;
  - warm-up fills (no verification branch, level sizes still growing) run
    whole on every worker: each computes the same call;
  - merge: the longest hit over all shares, ties to the lowest global
    candidate index (the single-worker rule), its emitted tokens; with no
    hit, the ordinary row's output (every worker computes it);
  - re-feed: a call's ordinary rows are the tokens emitted by the call before
    (one after a call without a hit, a + 1 after one with a hit), at their
    consecutive positions, causal among themselves; every later row of the
    call sees them as committed context; only they are committed.
So a worker's call computes, for the rows it shares with the single-worker
call, the same values from the same visible tokens, and the merged outputs,
window, pool and emitted stream equal the single-worker loop's.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

from .lookahead import (LOOKAHEAD, ORDINARY, VERIFY, LookaheadState, Row, check_args, greedy_verify,
                        meta_mask)
from .model import KVCache, OracleModel, argmax_lowest


def shard_columns(W: int, P: int, k: int) -> List[int]:
    """Window columns worker k owns (contiguous blocks)."""
    return list(range(k * W // P, (k + 1) * W // P))


def shard_candidates(C: int, P: int, k: int) -> List[int]:
    """Pool slots worker k verifies (every P-th, from k)."""
    return [c for c in range(C) if c % P == k]


def shard_rows(rows: Sequence[Row], cols: Sequence[int], cands: Sequence[int]) -> List[Row]:
    """The rows of one packed call a worker computes: the ordinary row, the
    base stripe up to its last column, its columns at every deeper level and
    its candidates' verification rows (packed order kept)."""
    last = max(cols) if cols else 0
    keep = []
    for r in rows:
        if r.role == ORDINARY:
            keep.append(r)
        elif r.role == LOOKAHEAD and r.level == 0:
            if r.column <= last:
                keep.append(r)
        elif r.role == LOOKAHEAD:
            if r.column in cols:
                keep.append(r)
        elif r.candidate in cands:
            keep.append(r)
    return keep


@dataclasses.dataclass
class ShardResult:
    """What a worker contributes after its forward."""
    z: dict                   # column -> its deepest level's output token
    a: int                    # its longest hit
    winner: int               # the global candidate index of that hit (-1 without one)
    emitted: List[int]        # the hit's emitted tokens (a + 1)


class Worker:
    """One replica: its own committed K/V and the tokens to re-feed."""

    def __init__(self, model: OracleModel, prompt: Sequence[int]):
        self.model = model
        self.cache, logits = model.prefill(list(prompt))
        self.first = argmax_lowest(logits[-1])
        self.refeed = [self.first]          # ordinary rows of the next call

    def forward(self, rows: Sequence[Row]) -> np.ndarray:
        """Re-fed rows (causal) then `rows` (their own visibility, seeing every
        re-fed row); commits the re-fed rows; returns the logits of `rows`."""
        I = len(self.refeed)
        base = len(self.cache)
        # the call's last ordinary row is rows' ORDINARY row (the last emitted
        # token); the re-fed tokens before it sit at the positions before
        refed = self.refeed[:-1]
        assert rows[0].role == ORDINARY and rows[0].token == self.refeed[-1]
        assert rows[0].position == base + len(refed)
        toks = refed + [r.token for r in rows]
        pos = list(range(base, base + len(refed))) + [r.position for r in rows]
        n_r, Q = len(refed), len(rows)
        vis = np.zeros((n_r + Q, n_r + Q), dtype=bool)
        vis[:n_r, :n_r] = np.tril(np.ones((n_r, n_r), dtype=bool))
        vis[n_r:, :n_r] = True
        vis[n_r:, n_r:] = meta_mask(rows)
        logits, k, v = self.model.forward(toks, pos, self.cache, vis)
        # commit the re-fed rows and the ordinary row (packed index 0 of rows)
        ordinary = n_r + [i for i, r in enumerate(rows) if r.role == ORDINARY][0]
        idx = list(range(n_r)) + [ordinary]
        self.cache.append([kk[idx] for kk in k], [vv[idx] for vv in v])
        assert I == len(idx)
        return logits[n_r:]


def local_result(state: LookaheadState, rows: Sequence[Row], guesses, mine: Sequence[Row], logits,
                 cols: Sequence[int], cands: Sequence[int]) -> ShardResult:
    """A worker's share of the verdict from the logits of its rows."""
    am = {r.packed_index: argmax_lowest(logits[i]) for i, r in enumerate(mine)}
    d = max(r.level for r in rows if r.role == LOOKAHEAD)
    z = {r.column: am[r.packed_index] for r in mine if r.role == LOOKAHEAD and r.level == d and r.column in cols}
    S = state.S
    vstart = len(rows) - len(guesses) * S
    sub = [guesses[c] for c in cands]
    a, w, emitted = greedy_verify(am[0], sub, lambda c, s: am[vstart + cands[c] * S + s])
    return ShardResult(z, a, cands[w] if w >= 0 else -1, emitted)


def merge(results: Sequence[ShardResult], W: int) -> Tuple[List[int], int, int, List[int]]:
    """The call's outputs from every worker's share: all W deep-level tokens,
    the longest hit (lowest global candidate index among equals), its emitted
    tokens."""
    z = {}
    for r in results:
        z.update(r.z)
    assert sorted(z) == list(range(W))
    best = min(results, key=lambda r: (-r.a, r.winner if r.a > 0 else 0))
    return [z[j] for j in range(W)], best.a, best.winner, list(best.emitted)


def lp_generate(model: OracleModel, prompt: Sequence[int], max_new: int, W: int, N: int, G: int, P: int,
                trace: Optional[list] = None) -> List[int]:
    """Greedy lookahead decoding with P replicas (workers simulated in turn)."""
    check_args(W, N, G)
    workers = [Worker(model, prompt) for _ in range(P)]
    first = workers[0].first
    assert all(w.first == first for w in workers)
    st = LookaheadState(prompt, first, W, N, G)
    out = [first]
    while len(out) < max_new:
        rows, guesses = st.plan()
        if not st.steady:
            # warm-up fill: every worker computes the whole call
            lgs = [w.forward(rows) for w in workers]
            argmax = [argmax_lowest(x) for x in lgs[0]]
            assert all([argmax_lowest(x) for x in lg] == argmax for lg in lgs)
            info = st.publish(rows, guesses, argmax)
        else:
            results = []
            for k, w in enumerate(workers):
                cols, cands = shard_columns(W, P, k), shard_candidates(len(guesses), P, k)
                mine = shard_rows(rows, cols, cands)
                results.append(local_result(st, rows, guesses, mine, w.forward(mine), cols, cands))
            z, a, win, emitted = merge(results, W)
            argmax = [0] * len(rows)
            for j, i in zip(range(W), st.deepest_rows(rows)):
                argmax[i] = z[j]
            info = st.publish(rows, guesses, argmax, (emitted, a, win))
        for w in workers:
            w.refeed = list(info.emitted)
        if trace is not None:
            trace.append(info)
        out.extend(info.emitted)
    return out[:max_new]
