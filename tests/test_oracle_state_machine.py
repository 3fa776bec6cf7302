"""Pins of the oracle's integer state machine against the pages' worked examples.

Every expected value comes from tests/golden/*.json (transcribed from the
pages, each with its citation) or from a rule the pages state.
"""
import json
import os

import pytest

from oracle import jacobi
from oracle import lookahead as la

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---- T1: Jacobi toy --------------------------------------------------------

def toy_operator():
    fs = [lambda y: 2, lambda y: (y[0] + 1) % 10, lambda y: (y[0] + y[1]) % 10, lambda y: (y[2] + 1) % 10]
    return lambda i, y: fs[i](y)


def test_jacobi_toy_matches_page():
    g = gold("jacobi_toy.json")
    T = toy_operator()
    fp, n = jacobi.solve(T, g["start"], jacobi.jacobi_sweep)
    assert fp == g["fixed_point"] and n == g["jacobi_sweeps"]
    fp, n = jacobi.solve(T, g["start"], jacobi.gauss_seidel_sweep)
    assert fp == g["fixed_point"] and n == g["gauss_seidel_sweeps"]


def test_jacobi_bound_m_sweeps_random_triangular():
    """§0x02A: any triangular system reaches its fixed point within m Jacobi sweeps."""
    import random
    rnd = random.Random(5)
    for trial in range(200):
        m = rnd.randint(1, 7)
        tabs = [{} for _ in range(m)]

        def T(i, y, tabs=tabs):
            key = tuple(y)
            if key not in tabs[i]:
                tabs[i][key] = rnd.randint(0, 4)
            return tabs[i][key]

        y0 = [rnd.randint(0, 4) for _ in range(m)]
        fp, n = jacobi.solve(T, y0)
        assert n <= m
        # the fixed point is the sequential (autoregressive) solution
        seq = []
        for i in range(m):
            seq.append(T(i, seq))
        assert fp == seq


# ---- T3: extraction ---------------------------------------------------------

def test_extraction_worked_example():
    g = gold("extraction_n4_w5.json")
    got = la.extract_keyed_ngrams(g["x_t"], g["levels"], g["z"], g["N"], g["W"])
    assert [[k, list(s)] for k, s in got] == g["extracted"]


# ---- T4: LRU rules ----------------------------------------------------------

def test_lru_rules():
    pool = {}
    G = 3
    la.upsert_suffix_lru(pool, 7, (1, 2), G)
    la.upsert_suffix_lru(pool, 7, (3, 4), G)
    assert pool[7] == [(1, 2), (3, 4)]                 # append as most recent
    la.upsert_suffix_lru(pool, 7, (1, 2), G)
    assert pool[7] == [(3, 4), (1, 2)]                 # reinsertion moves to back
    la.upsert_suffix_lru(pool, 7, (5, 6), G)
    la.upsert_suffix_lru(pool, 7, (8, 9), G)
    assert pool[7] == [(1, 2), (5, 6), (8, 9)]         # full bucket evicts bucket[0]
    la.upsert_suffix_lru(pool, 8, (0, 0), G)
    assert la.lookup(pool, 7, G) == [(1, 2), (5, 6), (8, 9)]   # retrieval by key only
    assert la.lookup(pool, 7, 2) == [(1, 2), (5, 6)]           # first G (oldest first)
    assert la.lookup(pool, 9, G) == []
    # a frequent key cannot consume another key's budget
    assert pool[8] == [(0, 0)]


# ---- T5: warm-up shapes -----------------------------------------------------

def sizes(levels):
    return [None if l is None else len(l) for l in levels]


@pytest.mark.parametrize("case", gold("warmup_traces.json")["traces"])
def test_warmup_traces(case):
    N, W = case["N"], case["W"]
    prompt = list(range(100, 110))
    st = la.LookaheadState(prompt, 1, W, N, G=2)
    trace = [sizes(st.levels)]
    while not st.steady:
        rows, guesses = st.plan()
        assert guesses == []                       # no verification branch during warm-up
        st.publish(rows, guesses, [0] * len(rows))
        trace.append(sizes(st.levels))
    assert trace == case["level_sizes"]
    rows, guesses = st.plan()
    st.publish(rows, guesses, [0] * len(rows))
    assert sizes(st.levels) == case["steady"]      # steady updates keep the ragged shape


@pytest.mark.parametrize("N", gold("warmup_traces.json")["rejected_N"] + [1, 0, 3.0])
def test_rejects_unsupported_depth(N):
    with pytest.raises(ValueError):
        la.check_args(5, N, 2)


def test_warmup_emits_one_token_and_no_pool():
    st = la.LookaheadState([1, 2, 3], 4, 5, 5, 3)
    for _ in range(3):          # N-2 fill stages
        assert not st.steady
        rows, guesses = st.plan()
        info = st.publish(rows, guesses, list(range(len(rows))))
        assert len(info.emitted) == 1 and st.pool == {}
    assert st.steady
    assert sizes(st.levels) == [4, 5, 5, 5]


# ---- T6: row ledger ----------------------------------------------------------

def make_steady(W, N, C):
    levels = [list(range(10, 10 + W - 1))] + [list(range(100 * r, 100 * r + W)) for r in range(1, N - 1)]
    guesses = [tuple(range(1000 * (c + 1), 1000 * (c + 1) + N - 1)) for c in range(C)]
    return la.compile_rows(7, 128, levels, guesses), levels, guesses


def test_row_ledger_w5_n4_g2():
    case = gold("row_ledger.json")["cases"][0]
    rows, levels, guesses = make_steady(case["W"], case["N"], case["C"])
    assert [len(l) for l in levels] == case["level_sizes"]
    assert len(rows) == case["Q"]
    req = [r.packed_index for r in rows if r.request_logit]
    lo, hi = case["inp_rows"]
    glo, ghi = case["guess_rows"]
    assert req == [case["out_row"]] + list(range(lo, hi)) + list(range(glo, ghi))
    assert all(rows[i].role == la.LOOKAHEAD and rows[i].level == case["N"] - 2 for i in range(lo, hi))
    assert all(rows[i].role == la.VERIFY for i in range(glo, ghi))


def test_row_ledger_teaching_setting():
    case = gold("row_ledger.json")["cases"][1]
    rows, _, _ = make_steady(case["W"], case["N"], case["C"])
    n_la = sum(r.role == la.LOOKAHEAD for r in rows)
    n_v = sum(r.role == la.VERIFY for r in rows)
    assert (n_la, n_v, len(rows)) == (case["Q_LA"], case["Q_V"], case["Q"])
    assert len(rows) == (case["W"] + case["C"]) * (case["N"] - 1)


# ---- T7: visibility -----------------------------------------------------------

@pytest.mark.parametrize("W,N,C", [(5, 4, 2), (1, 3, 0), (3, 3, 3), (7, 5, 7), (4, 6, 1)])
def test_visibility_sets_and_predicate(W, N, C):
    rows, _, _ = make_steady(W, N, C)
    sets = la.vis_sets(rows)
    assert (la.dense_mask(rows) == la.meta_mask(rows)).all()
    for rw, s in zip(rows, sets):
        # exactly one visible key per logical position p .. pos (a causal path)
        pos = sorted(rows[i].position for i in s)
        assert pos == list(range(128, rw.position + 1))
        assert rw.packed_index in s
        roles = {rows[i].role for i in s}
        if rw.role == la.VERIFY:
            # sees b_0 and its own candidate only
            assert all(rows[i].role == la.ORDINARY or rows[i].candidate == rw.candidate for i in s)
            assert la.LOOKAHEAD not in roles
        else:
            assert la.VERIFY not in roles


def test_visibility_in_warmup_layout():
    st = la.LookaheadState(list(range(20)), 5, 5, 4, 2)
    rows, _ = st.plan()
    assert (la.dense_mask(rows) == la.meta_mask(rows)).all()
    rows_, g_ = st.plan()
    st.publish(rows_, g_, [3] * len(rows_))
    rows, _ = st.plan()
    for rw, s in zip(rows, la.vis_sets(rows)):
        assert sorted(rows[i].position for i in s) == list(range(st.p, rw.position + 1))


# ---- T8: commit trace -----------------------------------------------------------

def test_commit_trace():
    g = gold("commit_trace.json")
    copies, trim = la.pinned_commit_plan(g["K_in"], g["step_len"], g["guess_token_count"], g["S"],
                                         g["winner"], g["max_hit"])
    assert copies[0][0] == g["src0"]
    assert [list(c) for c in copies] == g["copies"]
    assert trim == g["trim_exclusive"]
    assert g["max_hit"] + 1 == g["emitted_count"]


def test_commit_rows_match_pinned_plan():
    """The oracle's row-index commit equals the pinned physical plan (rows at K_in + index)."""
    W, N, C = 5, 4, 2
    levels = [list(range(10, 14)), list(range(20, 25)), list(range(30, 35))]
    guesses = [(50, 51, 52), (60, 61, 62)]
    st = la.LookaheadState([1, 2, 3], 40, W, N, 2)
    st.levels, st.p = levels, 128
    st.pool = {40: guesses}
    rows, g = st.plan()
    assert len(rows) == 21
    argmax = [0] * 21
    # make candidate 1 hit twice: out -> 60, v_{1,0} -> 61, v_{1,1} -> 99 (mismatch with 62)
    argmax[0] = 60
    argmax[15 + 3 + 0] = 61
    argmax[15 + 3 + 1] = 99
    info = st.publish(rows, g, argmax)
    assert (info.a, info.winner, info.emitted) == (2, 1, [60, 61, 99])
    copies, trim = la.pinned_commit_plan(128, 128 + 21, 6, 3, info.winner, info.a)
    assert [128 + i for i in info.commit_rows[1:]] == [c[0] for c in copies]
    assert 128 + len(info.commit_rows) == trim
    assert st.p == trim and st.x_t == 99


# ---- greedy verification ---------------------------------------------------------

def test_greedy_verify_equals_survivor_view():
    import random
    rnd = random.Random(11)
    for _ in range(3000):
        S = rnd.randint(1, 5)
        C = rnd.randint(0, 6)
        V = rnd.randint(2, 4)
        guesses = [tuple(rnd.randrange(V) for _ in range(S)) for _ in range(C)]
        # row outputs depend only on the row's own accepted prefix so survivors agree
        table = {}

        def out_after(prefix):
            if prefix not in table:
                table[prefix] = rnd.randrange(V)
            return table[prefix]

        out_tok = out_after(())
        row_argmax = lambda c, s: out_after(tuple(guesses[c][: s + 1]))
        a, w, em = la.greedy_verify(out_tok, guesses, row_argmax)
        assert em == la.greedy_verify_survivors(out_tok, guesses, row_argmax)
        assert len(em) == a + 1 and a <= S
        if a:
            assert list(guesses[w][:a]) == em[:a]
            assert all(list(guesses[c][:a]) != em[:a] for c in range(w))   # lowest index among longest


def test_pool_updates_only_after_outputs():
    """§0x03C: a suffix inserted by a call is not offered to that same call."""
    st = la.LookaheadState([1, 2, 3, 4], 9, 3, 3, 4)
    rows, g = st.plan()
    st.publish(rows, g, [9] * len(rows))          # warm-up (N=3: one stage)
    assert st.steady
    rows, g = st.plan()
    assert g == []                                 # nothing in the pool yet
    st.publish(rows, g, [9] * len(rows))
    assert 9 in st.pool


# ---- pool seeding (POOL_FROM_PROMPT, generated-prefix insertion) ------------

def test_pool_from_prompt_hand_example():
    """The prompt's n-grams, keyed by their first token, upserted in position
    order under the per-key LRU rule (worked by hand, N=3, G=2)."""
    p = [5, 6, 7, 5, 6, 8, 5, 6, 7]
    st = la.LookaheadState(p, 9, 2, 3, 2, pool_from_prompt=True)
    assert st.pool == {5: [(6, 8), (6, 7)], 6: [(7, 5), (8, 5)], 7: [(5, 6)], 8: [(5, 6)]}


def test_pool_from_output_first_token():
    """The n-gram ending at the first output token (sequence position P) goes
    in after the prompt's: key 6 (position 7), suffix (7, 9) evicts (7, 5)."""
    p = [5, 6, 7, 5, 6, 8, 5, 6, 7]
    both = la.LookaheadState(p, 9, 2, 3, 2, pool_from_prompt=True, pool_from_output=True)
    assert both.pool[6] == [(8, 5), (7, 9)]
    only = la.LookaheadState(p, 9, 2, 3, 2, pool_from_output=True)
    assert only.pool == {6: [(7, 9)]}


def test_pool_from_output_after_a_call():
    """A call's emitted tokens add the n-grams ending at them, after the
    call's own trajectory n-grams (none in a warm-up call)."""
    p = [5, 6, 7, 5, 6, 8, 5, 6, 7]
    st = la.LookaheadState(p, 9, 2, 3, 2, pool_from_output=True)
    rows, g = st.plan()
    assert not st.steady
    info = st.publish(rows, g, [4] * len(rows))
    assert info.emitted == [4]
    assert st.pool == {6: [(7, 9)], 7: [(9, 4)]}
    assert st.seq == p + [9, 4]


def test_unseeded_pool_starts_empty():
    st = la.LookaheadState([5, 6, 7, 5, 6, 8], 9, 2, 3, 2)
    assert st.pool == {}


# ---- ALWAYS_FWD_ONE=False: slice by the accepted count, refill -------------

def _steady_hit_state(slice_window):
    """W=3, N=4 (S=3), prompt [1..5]: level 0 was seeded with prompt[0..3], so
    the refill continues the cycle at prompt[4].  The pool holds one suffix
    for x_t=9 and the outputs accept two of its tokens."""
    st = la.LookaheadState([1, 2, 3, 4, 5], 9, 3, 4, 2, slice_window=slice_window)
    st.levels = [[10, 11], [20, 21, 22], [30, 31, 32]]
    st.pool = {9: [(40, 41, 42)]}
    rows, g = st.plan()
    assert g == [(40, 41, 42)]
    z = [50, 51, 52]
    out = []
    for r in rows:
        if r.role == la.ORDINARY:
            out.append(40)
        elif r.role == la.VERIFY:
            out.append({0: 41, 1: 99}.get(r.offset, 0))
        elif r.level == 2:
            out.append(z[r.column])
        else:
            out.append(0)
    return st, st.publish(rows, g, out)


def test_slice_window_hand_example():
    """a = 2: the pinned shift gives [[21,22],[30,31,32],[50,51,52]]; each level
    then drops two cells and takes 5,1 | 2,3 | 4,5 from the prompt cycle."""
    st, info = _steady_hit_state(True)
    assert (info.a, info.emitted) == (2, [40, 41, 99])
    assert st.levels == [[5, 1], [32, 2, 3], [52, 4, 5]]
    assert st.seed_next == 10
    assert sizes(st.levels) == [2, 3, 3]


def test_slice_window_off_is_the_pinned_shift():
    st, info = _steady_hit_state(False)
    assert info.a == 2
    assert st.levels == [[21, 22], [30, 31, 32], [50, 51, 52]]


def test_slice_window_without_a_hit_is_the_pinned_shift():
    """a = 0 leaves nothing to slice: both schedules advance one column."""
    runs = []
    for flag in (False, True):
        st = la.LookaheadState([1, 2, 3, 4, 5], 9, 3, 4, 2, slice_window=flag)
        st.levels = [[10, 11], [20, 21, 22], [30, 31, 32]]
        rows, g = st.plan()
        st.publish(rows, g, [7] * len(rows))
        runs.append((st.levels, st.seed_next))
    assert runs[0] == runs[1] == ([[21, 22], [30, 31, 32], [7, 7, 7]], 4)


def test_slice_window_wider_than_a_level():
    """W=1, N=5 (S=4), a=3: level 0 is empty; levels of one cell are refilled
    whole, in level order, from the prompt cycle (level 0's seed took
    prompt[0..2], so the cycle goes on with 5, 6, 7)."""
    st = la.LookaheadState([5, 6, 7], 9, 1, 5, 1, slice_window=True)
    st.levels = [[], [20], [30], [40]]
    st.pool = {9: [(1, 2, 3, 4)]}
    rows, g = st.plan()
    out = []
    for r in rows:
        if r.role == la.ORDINARY:
            out.append(1)
        elif r.role == la.VERIFY:
            out.append({0: 2, 1: 3, 2: 8}.get(r.offset, 0))
        else:
            out.append(60 + r.level)
    info = st.publish(rows, g, out)
    assert (info.a, info.emitted) == (3, [1, 2, 3, 8])
    assert st.levels == [[], [5], [6], [7]]
