"""Lookahead decoding state machine and generate loops (oracle; test infrastructure).

Notation follows "M7.3 – Lookahead Decoding" (§0x01A, §0x03–§0x07):

* R = S = N - 1; the window holds trajectory levels u^(0..R-1).  Steady level
  sizes are [W-1, W, ..., W]; the live ordinary token x_t is the missing
  first cell of level 0 (§0x01A).
* Warm-up (§0x03A): level 0 starts with W+N-3 cells; each fill stage runs
  without a verification branch and emits one token; every existing level
  drops its first cell and the deepest level's outputs become a new level
  (the first output dropped once the deepest level is below level 0).  This
  reading reproduces both printed traces, [6,-,-] -> [5,6,-] -> [4,5,5] for
  N=4, W=5 and [5,-] -> [4,5] for N=3, W=5.
* Rows (§0x04, §0x04A): base stripe b_0..b_{W-1} (b_0 = x_t), trajectory
  rows u_{r,j}, verification rows v_{c,s}; packed level-major.  Logical
  positions: b_j at p+j, u_{r,j} at p+j+r, v_{c,s} at p+1+s (the positions
  that make every visible set one key per position and the extracted n-gram
  a run of consecutive positions, §0x03B).
* Visibility (§0x04A): Vis(b_j) = {b_k : k <= j};
  Vis(u_{r,j}) = {b_k : k <= j} u {u_{q,j} : 1 <= q <= r};
  Vis(v_{c,s}) = {b_0} u {v_{c,q} : q <= s}; the committed prefix is visible
  to every row.
* Extraction (§0x03B): k_0 = x_t, s_0 = (u^(1)_0..u^(R-1)_0, z_0);
  k_j = u^(0)_{j-1}, s_j = (u^(1)_j..u^(R-1)_j, z_j) for j = 1..W-1.
* Pool (§0x03B): per-key list of at most G suffixes, oldest first; a
  reinserted suffix moves to the back, a full bucket evicts its oldest;
  retrieval reads only the bucket of x_t, first G entries (§0x03C).
* Greedy verification (§0x05A): z^(c) = (argmax out, argmax v_{c,0}, ...,
  argmax v_{c,S-2}); hit a_c = longest prefix with g^(c)_{1:a} = z^(c)_{1:a};
  emitted = accepted tokens plus the target token after them.
* Publication (§0x06B, §0x06C): K/V of the ordinary row stays at K_in; the
  winner's first a verification rows are copied to K_in+1..K_in+a; the next
  ordinary input is the last emitted token.
* Window advance, ALWAYS_FWD_ONE (§0x03C): [u^(1)[1:], u^(2), ..., u^(R-1), z].
* Optional ALWAYS_FWD_ONE=False (§0x03C alternative; §0x06 sequence axis):
  after a steady call that accepted a > 0 tokens, every level of the advanced
  window also drops its first a cells, the rest move left and the vacated
  tail cells are refilled, level 0 first, each level in column order, from
  the seed source: the prompt cycle that seeded level 0, continued (the
  refill cell numbered c takes prompt[(W+N-3+c) mod P]).
* Optional pool seeding (§0x03A POOL_FROM_PROMPT; §0x06A "optional
  generated-prefix insertion"; Break the Sequential Dependency §5, prompt
  lookup): the n-grams of the token sequence (prompt, then every output
  token) are upserted into the same keyed LRU pool, the n-gram ending at
  sequence position k keyed by token k-S with suffix tokens k-S+1..k, in
  increasing k.  From the prompt: every n-gram that lies inside the prompt,
  once, when the request starts.  From the output: every n-gram that ends at
  an output token, when that token is appended (the first token at request
  start, after any prompt n-grams; a call's tokens after that call's
  trajectory n-grams).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

from .model import KVCache, OracleModel, argmax_lowest
from . import sampling as smp

ORDINARY, LOOKAHEAD, VERIFY = 0, 1, 2


# ----------------------------------------------------------------------------
# admission
# ----------------------------------------------------------------------------

def pinned_suffix_length(N) -> int:
    """R = S = N - 1; the pinned multilevel schedule admits integer N >= 3 (§0x01A)."""
    if type(N) is not int or N < 3:
        raise ValueError("lookahead needs an integer N >= 3 (two trajectory levels)")
    return N - 1


def check_args(W, N, G) -> int:
    S = pinned_suffix_length(N)
    if type(W) is not int or W < 1:
        raise ValueError("window width W must be a positive integer")
    if type(G) is not int or G < 0:
        raise ValueError("G must be a non-negative integer")
    return S


# ----------------------------------------------------------------------------
# rows, positions, visibility
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Row:
    packed_index: int
    role: int            # ORDINARY | LOOKAHEAD | VERIFY
    level: int           # trajectory level (0 = base stripe); -1 for VERIFY
    column: int          # window column j; -1 for VERIFY
    candidate: int       # c for VERIFY, else -1
    offset: int          # s for VERIFY, else -1
    position: int        # logical position
    token: int
    request_logit: bool


def deepest_level(levels: Sequence[Optional[Sequence[int]]]) -> int:
    d = -1
    for r, lv in enumerate(levels):
        if lv is None:
            break
        d = r
    return d


def compile_rows(x_t: int, p: int, levels, guesses: Sequence[Sequence[int]]) -> List[Row]:
    """Level-major packed rows with roles, positions and logit requests (§0x04A)."""
    d = deepest_level(levels)
    rows = [Row(0, ORDINARY, 0, 0, -1, -1, p, int(x_t), True)]
    for i, tok in enumerate(levels[0]):
        j = i + 1
        rows.append(Row(len(rows), LOOKAHEAD, 0, j, -1, -1, p + j, int(tok), d == 0))
    for r in range(1, d + 1):
        for j, tok in enumerate(levels[r]):
            rows.append(Row(len(rows), LOOKAHEAD, r, j, -1, -1, p + j + r, int(tok), r == d))
    for c, g in enumerate(guesses):
        for s, tok in enumerate(g):
            rows.append(Row(len(rows), VERIFY, -1, -1, c, s, p + 1 + s, int(tok), True))
    return rows


def vis_sets(rows: Sequence[Row]) -> List[set]:
    """The allowed in-call keys of every row, built from the three Vis equations."""
    base: Dict[int, int] = {}
    traj: Dict[Tuple[int, int], int] = {}
    cand: Dict[Tuple[int, int], int] = {}
    for rw in rows:
        if rw.role == VERIFY:
            cand[(rw.candidate, rw.offset)] = rw.packed_index
        elif rw.level == 0:
            base[rw.column] = rw.packed_index
        else:
            traj[(rw.level, rw.column)] = rw.packed_index
    out = []
    for rw in rows:
        if rw.role == VERIFY:
            s = {base[0]} | {cand[(rw.candidate, q)] for q in range(rw.offset + 1)}
        elif rw.level == 0:
            s = {base[k] for k in range(rw.column + 1)}
        else:
            s = {base[k] for k in range(rw.column + 1)} | {traj[(q, rw.column)] for q in range(1, rw.level + 1)}
        out.append(s)
    return out


def visible(a: Row, b: Row) -> bool:
    """Metadata predicate: may query row a see key row b (both in the call)?"""
    if a.role == VERIFY:
        return b.role == ORDINARY or (b.role == VERIFY and b.candidate == a.candidate and b.offset <= a.offset)
    if b.role == VERIFY:
        return False
    if b.level == 0:
        return b.column <= a.column
    return a.level >= 1 and b.column == a.column and b.level <= a.level


def dense_mask(rows: Sequence[Row]) -> np.ndarray:
    """Materialised [Q, Q] boolean mask from the Vis sets (dense packed path)."""
    Q = len(rows)
    m = np.zeros((Q, Q), dtype=bool)
    for i, s in enumerate(vis_sets(rows)):
        m[i, sorted(s)] = True
    return m


def meta_mask(rows: Sequence[Row]) -> np.ndarray:
    Q = len(rows)
    return np.array([[visible(rows[i], rows[j]) for j in range(Q)] for i in range(Q)], dtype=bool)


# ----------------------------------------------------------------------------
# pool
# ----------------------------------------------------------------------------

def extract_keyed_ngrams(x_t: int, levels, z: Sequence[int], N: int, W: int):
    """W keyed suffixes from the pre-shift steady levels and the new outputs z (§0x03B)."""
    R = N - 1
    out = []
    for j in range(W):
        key = int(x_t) if j == 0 else int(levels[0][j - 1])
        suffix = tuple(int(levels[r][j]) for r in range(1, R)) + (int(z[j]),)
        out.append((key, suffix))
    return out


def upsert_suffix_lru(pool: Dict[int, List[tuple]], key: int, suffix: tuple, G: int) -> None:
    """Per-key LRU: reinsertion moves to the back; a full bucket evicts its oldest."""
    if G <= 0:
        return
    bucket = pool.setdefault(key, [])
    if suffix in bucket:
        bucket.remove(suffix)
    elif len(bucket) >= G:
        del bucket[0]
    bucket.append(suffix)


def upsert_sequence_ngrams(pool: Dict[int, List[tuple]], seq: Sequence[int], k_lo: int, k_hi: int,
                           S: int, G: int) -> None:
    """The n-grams of ``seq`` ending at positions k_lo <= k < k_hi (those with
    k >= S): key seq[k-S], suffix seq[k-S+1..k], upserted in increasing k."""
    for k in range(max(k_lo, S), k_hi):
        upsert_suffix_lru(pool, int(seq[k - S]), tuple(int(t) for t in seq[k - S + 1:k + 1]), G)


def lookup(pool: Dict[int, List[tuple]], key: int, G: int) -> List[tuple]:
    return list(pool.get(int(key), [])[:G])


# ----------------------------------------------------------------------------
# verification and publication
# ----------------------------------------------------------------------------

def greedy_verify(out_tok: int, guesses: Sequence[Sequence[int]],
                  row_argmax: Callable[[int, int], int]) -> Tuple[int, int, List[int]]:
    """Longest accepted prefix over the candidates (§0x05A).

    Returns (a, winner, emitted); winner is the lowest candidate index among
    the longest hits (-1 when a == 0); emitted has a + 1 tokens.
    """
    best_a, best_w = 0, -1
    for c, g in enumerate(guesses):
        S = len(g)
        a_c = 0
        target = out_tok
        while a_c < S and g[a_c] == target:
            target = row_argmax(c, a_c)     # row v_{c,a_c} predicts the next token
            a_c += 1
        if a_c > best_a:
            best_a, best_w = a_c, c
    if best_a == 0:
        return 0, -1, [int(out_tok)]
    g = guesses[best_w]
    emitted = [int(t) for t in g[:best_a]] + [int(row_argmax(best_w, best_a - 1))]
    return best_a, best_w, emitted


def greedy_verify_survivors(out_tok: int, guesses, row_argmax) -> List[int]:
    """The survivor view of the same rule (§0x05A), used as a cross-check."""
    target = out_tok
    survivors = list(range(len(guesses)))
    emitted = [int(target)]
    S = len(guesses[0]) if guesses else 0
    for off in range(S):
        survivors = [c for c in survivors if guesses[c][off] == target]
        if not survivors:
            break
        conds = {row_argmax(c, off) for c in survivors}
        assert len(conds) == 1, "survivors with one accepted prefix must agree"
        target = conds.pop()
        emitted.append(int(target))
    return emitted


def pinned_commit_plan(K_in: int, step_len: int, guess_token_count: int, S: int,
                       winner: int, max_hit: int):
    """Physical K/V copies of the pinned single-worker path (§0x06C).

    Rows of the call sit at K_in .. step_len-1 in packed order.  Returns
    (copies [(src, dst)], trim_exclusive).
    """
    kvcache_len = K_in + 1
    src0 = step_len - guess_token_count + winner * S
    copies = [(src0 + j, kvcache_len + j) for j in range(max_hit)]
    return copies, kvcache_len + max_hit


def advance_window(levels, z: Sequence[int], steady: bool):
    """Steady: [u1[1:], u2, ..., u_{R-1}, z]; warm-up: every level drops its first cell, z appended."""
    R = len(levels)
    if steady:
        return [list(levels[1][1:])] + [list(l) for l in levels[2:]] + [list(z)]
    d = deepest_level(levels)
    new = [list(l[1:]) for l in levels[: d + 1]] + [list(z)]
    return new + [None] * (R - len(new))


def slice_and_refill(levels, slide: int, seed_token):
    """The ALWAYS_FWD_ONE=False alternative of §0x03C (sequence axis of §0x06):
    applied after the one-column steady shift, it drops the first ``slide`` cells
    of every level (the positions the ``slide`` accepted tokens consumed), moves
    the rest left and refills the vacated tail, level 0 first and each level in
    column order, with successive tokens of the seed source ``seed_token()``.
    Level sizes [W-1, W, ..., W] are kept."""
    out = []
    for lv in levels:
        keep = [int(t) for t in lv[slide:]]
        out.append(keep + [int(seed_token()) for _ in range(len(lv) - len(keep))])
    return out


def init_levels(prompt: Sequence[int], W: int, N: int):
    """Level 0 of W+N-3 cells seeded by cycling the prompt; deeper levels empty."""
    R = N - 1
    P = len(prompt)
    lv0 = [int(prompt[i % P]) for i in range(W + N - 3)]
    return [lv0] + [None] * (R - 1)


# ----------------------------------------------------------------------------
# state of one request
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class StepInfo:
    Q: int
    C_t: int
    steady: bool
    a: int
    winner: int
    emitted: List[int]
    commit_rows: List[int]


class LookaheadState:
    """Window, pool and frontier of one request between packed calls."""

    def __init__(self, prompt: Sequence[int], first_token: int, W: int, N: int, G: int,
                 pool_from_prompt: bool = False, pool_from_output: bool = False,
                 slice_window: bool = False):
        self.S = check_args(W, N, G)
        self.W, self.N, self.G = W, N, G
        self.levels = init_levels(prompt, W, N)
        self.prompt = [int(t) for t in prompt]
        self.slice_window = slice_window
        self.seed_next = W + N - 3     # the prompt cycle continues after level 0's seed cells
        self.pool: Dict[int, List[tuple]] = {}
        self.x_t = int(first_token)
        self.p = len(prompt)           # committed K/V length = position of x_t
        self.step = 0
        self.pool_from_output = pool_from_output
        self.seq = [int(t) for t in prompt] + [int(first_token)]   # prompt, then the output tokens
        P = len(prompt)
        if pool_from_prompt:
            upsert_sequence_ngrams(self.pool, self.seq, 0, P, self.S, G)
        if pool_from_output:
            upsert_sequence_ngrams(self.pool, self.seq, P, P + 1, self.S, G)

    def _seed_token(self) -> int:
        """Next token of the seed source: the prompt, cycled (§0x03A)."""
        t = self.prompt[self.seed_next % len(self.prompt)]
        self.seed_next += 1
        return t

    @property
    def steady(self) -> bool:
        return deepest_level(self.levels) == self.N - 2

    def plan(self):
        guesses = lookup(self.pool, self.x_t, self.G) if self.steady else []
        rows = compile_rows(self.x_t, self.p, self.levels, guesses)
        return rows, guesses

    def deepest_rows(self, rows: Sequence[Row]) -> List[int]:
        d = deepest_level(self.levels)
        idx = [r.packed_index for r in rows if r.role == LOOKAHEAD and r.level == d]
        if not self.steady and d >= 1:
            idx = idx[1:]
        return idx

    def publish(self, rows, guesses, argmax: Sequence[int],
                verdict: Optional[Tuple[List[int], int, int]] = None) -> StepInfo:
        """Apply one call's outputs.  ``argmax`` is indexed by packed row.

        ``verdict`` = (emitted, a, winner) overrides greedy verification (sampling).
        """
        steady = self.steady
        S = self.S
        vstart = len(rows) - len(guesses) * S

        def vrow(c, s):
            return vstart + c * S + s

        if verdict is None:
            if steady:
                a, w, emitted = greedy_verify(argmax[0], guesses, lambda c, s: argmax[vrow(c, s)])
            else:
                a, w, emitted = 0, -1, [int(argmax[0])]
        else:
            emitted, a, w = verdict
        z = [int(argmax[i]) for i in self.deepest_rows(rows)]
        commit = [0] + [vrow(w, j) for j in range(a)]
        if steady:
            for key, suffix in extract_keyed_ngrams(self.x_t, self.levels, z, self.N, self.W):
                upsert_suffix_lru(self.pool, key, suffix, self.G)
        n0 = len(self.seq)
        self.seq.extend(int(t) for t in emitted)
        if self.pool_from_output:
            upsert_sequence_ngrams(self.pool, self.seq, n0, len(self.seq), S, self.G)
        self.levels = advance_window(self.levels, z, steady)
        if steady and self.slice_window and a > 0:
            self.levels = slice_and_refill(self.levels, a, self._seed_token)
        info = StepInfo(len(rows), len(guesses), steady, a, w, list(emitted), commit)
        self.x_t = int(emitted[-1])
        self.p += 1 + a
        self.step += 1
        return info


# ----------------------------------------------------------------------------
# schedules of the target call
# ----------------------------------------------------------------------------

class PackedRunner:
    """One forward over all packed rows with a dense or metadata mask (§0x07A)."""

    def __init__(self, model: OracleModel, cache: KVCache, mask: str = "meta"):
        self.model, self.cache, self.mask = model, cache, mask
        self._k = self._v = None

    def run(self, rows: Sequence[Row]) -> np.ndarray:
        m = dense_mask(rows) if self.mask == "dense" else meta_mask(rows)
        logits, self._k, self._v = self.model.forward([r.token for r in rows], [r.position for r in rows],
                                                      self.cache, m)
        return logits

    def commit(self, rows: Sequence[Row], idx: Sequence[int]) -> None:
        idx = list(idx)
        self.cache.append([k[idx] for k in self._k], [v[idx] for v in self._v])


class SeparateRunner:
    """Every row as an isolated causal forward over its own path (§0x07A oracle)."""

    def __init__(self, model: OracleModel, cache: KVCache):
        self.model, self.cache = model, cache

    def run(self, rows: Sequence[Row]) -> np.ndarray:
        sets = vis_sets(rows)
        out = []
        for rw, s in zip(rows, sets):
            path = sorted(s, key=lambda i: rows[i].position)
            assert [rows[i].position for i in path] == list(range(rows[path[0]].position, rw.position + 1))
            logits, _, _ = self.model.causal([rows[i].token for i in path], rows[path[0]].position, self.cache)
            out.append(logits[-1])
        return np.stack(out)

    def commit(self, rows: Sequence[Row], idx: Sequence[int]) -> None:
        toks = [rows[i].token for i in idx]
        _, k, v = self.model.causal(toks, len(self.cache), self.cache)
        self.cache.append(k, v)


def make_runner(model, cache, schedule: str):
    if schedule == "separate":
        return SeparateRunner(model, cache)
    return PackedRunner(model, cache, "dense" if schedule == "dense" else "meta")


# ----------------------------------------------------------------------------
# generate loops
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Sampling:
    temperature: float
    top_p: float
    seed: int


FIRST_TOKEN_STEP = 0xFFFFFFFF   # Philox step index of the prefill's token


def _first_token(logits_last, sampling: Optional[Sampling]) -> int:
    if sampling is None:
        return argmax_lowest(logits_last)
    p = smp.warp(logits_last, sampling.temperature, sampling.top_p)
    return smp.PhiloxChooser(sampling.seed, FIRST_TOKEN_STEP).categorical(p, 0, 2)


def ar_generate(model: OracleModel, prompt: Sequence[int], max_new: int,
                sampling: Optional[Sampling] = None) -> List[int]:
    """Plain autoregressive decoding: one new row per call."""
    cache, logits = model.prefill(prompt)
    out = [_first_token(logits[-1], sampling)]
    t = 0
    while len(out) < max_new:
        lg, k, v = model.causal([out[-1]], len(cache), cache)
        cache.append(k, v)
        if sampling is None:
            out.append(argmax_lowest(lg[0]))
        else:
            p = smp.warp(lg[0], sampling.temperature, sampling.top_p)
            out.append(smp.PhiloxChooser(sampling.seed, t).categorical(p, 0, 2))
        t += 1
    return out[:max_new]


def lookahead_generate(model: OracleModel, prompt: Sequence[int], max_new: int, W: int, N: int, G: int,
                       schedule: str = "meta", sampling: Optional[Sampling] = None,
                       trace: Optional[list] = None, pool_from_prompt: bool = False,
                       pool_from_output: bool = False, slice_window: bool = False) -> List[int]:
    """Lookahead decoding (§0x06 loop) on one schedule of the packed call."""
    check_args(W, N, G)
    cache, logits = model.prefill(prompt)
    out = [_first_token(logits[-1], sampling)]
    st = LookaheadState(prompt, out[0], W, N, G, pool_from_prompt, pool_from_output, slice_window)
    runner = make_runner(model, cache, schedule)
    while len(out) < max_new:
        rows, guesses = st.plan()
        lg = runner.run(rows)
        argmax = [argmax_lowest(lg[i]) for i in range(len(rows))]
        verdict = None
        if sampling is not None:
            verdict = sample_step(lg, rows, guesses, st, sampling)
        info = st.publish(rows, guesses, argmax, verdict)
        runner.commit(rows, info.commit_rows)
        if trace is not None:
            trace.append(info)
        out.extend(info.emitted)
    return out[:max_new]


def sample_step(logits, rows, guesses, st: LookaheadState, sampling: Sampling):
    """Exact sampling verdict for one call (emitted, a, winner)."""
    S = st.S
    vstart = len(rows) - len(guesses) * S
    warp = lambda i: smp.warp(logits[i], sampling.temperature, sampling.top_p)
    chooser = smp.PhiloxChooser(sampling.seed, st.step)
    if not guesses:
        return [chooser.categorical(warp(0), 0, 2)], 0, -1
    return smp.sample_verify([list(g) for g in guesses], warp(0),
                             lambda c, s: warp(vstart + c * S + s), chooser)
