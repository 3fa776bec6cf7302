"""GPU parity on the fp32 tiny Llama (2 layers, d 128, 4 heads, FFN 512, vocab 512):
the CUDA path through the C ABI against the CPU oracle, element by element."""
import numpy as np
import pytest
import torch

import synth
from oracle import lookahead as la
from oracle.model import OracleModel, argmax_lowest
from tests.gpu_util import context, top2_gap

pytestmark = pytest.mark.gpu

CFG = synth.TINY
LOGIT_TOL = 1e-3          # fp32 model: max-abs logit difference


@pytest.fixture(scope="module")
def setup():
    from lookahead_decoding_gb300 import lib
    w_cpu = synth.llama_weights(CFG, 0)
    w = {k: v.to("cuda:0") for k, v in w_cpu.items()}
    ctx = context(CFG, w, max_ctx=512, W=8, N=5, G=8)
    oracle = OracleModel(CFG, w_cpu)
    yield lib(), ctx, oracle, w_cpu
    ctx.close()


def prompt(n=32, seed=1):
    return synth.uniform_prompt(CFG.vocab, n, seed).tolist()


def test_prefill_logits(setup):
    L, ctx, oracle, _ = setup
    L.la_set_debug(ctx.ctx, 1)
    for n in (1, 5, 32, 100):
        p = prompt(n, 7 + n)
        tok = L.la_prefill(ctx.ctx, p)
        lg, rows = L.la_debug_logits(ctx.ctx, 4, CFG.vocab)
        _, ref = oracle.prefill(p)
        assert len(rows) == 1 and rows[0] == (n - 1) % 256
        assert np.max(np.abs(lg[0] - ref[-1])) < LOGIT_TOL
        assert tok == argmax_lowest(ref[-1]) or top2_gap(ref[-1]) < 1e-2
    L.la_set_debug(ctx.ctx, 0)


def meta_fields(m):
    return m & 3, (m >> 2) & 63, (m >> 8) & 255, (m >> 16) & 255, (m >> 24) & 127


def check_rows(rows, tok, pos, meta):
    assert tok == [r.token for r in rows]
    assert pos == [r.position for r in rows]
    for r, m in zip(rows, meta):
        role, level, col, cand, off = meta_fields(m)
        assert role == r.role
        if r.role == la.VERIFY:
            assert (cand, off) == (r.candidate, r.offset)
        else:
            assert (level, col) == (r.level, r.column)


def check_state(L, ctx, st, keys):
    h, lv, _, _, _ = L.la_debug_state(ctx.ctx)
    assert h["K"] == st.p and h["x_t"] == st.x_t
    R = len(st.levels)
    assert lv[:R] == [None if l is None else list(l) for l in st.levels]
    assert all(l is None for l in lv[R:])
    for k in keys:
        assert L.la_debug_pool(ctx.ctx, k) == list(st.pool.get(k, []))


@pytest.mark.parametrize("W,N,G", [(5, 3, 5), (4, 4, 3), (1, 3, 1), (8, 5, 8)])
def test_step_by_step_against_oracle(setup, W, N, G):
    """Every call: rows, positions, metadata, needed-row logits, emitted tokens,
    window and pool equal the oracle running the same state machine."""
    L, ctx, oracle, _ = setup
    p = prompt(32, 1)
    L.la_set_debug(ctx.ctx, 1)
    first = L.la_prefill(ctx.ctx, p)
    cache, lg0 = oracle.prefill(p)
    assert first == argmax_lowest(lg0[-1])
    st = la.LookaheadState(p, first, W, N, G)
    run = la.make_runner(oracle, cache, "meta")
    hits = 0
    for step in range(24):
        rows, guesses = st.plan()
        ref = run.run(rows)
        em = L.la_step(ctx.ctx, W, N, G)
        h, _, tok, pos, meta = L.la_debug_state(ctx.ctx)
        assert h["Q"] == len(rows) and h["C_t"] == len(guesses)
        check_rows(rows, tok, pos, meta)
        lg, need = L.la_debug_logits(ctx.ctx, 512, CFG.vocab)
        assert need.tolist() == [r.packed_index for r in rows if r.request_logit]
        assert np.max(np.abs(lg - ref[need])) < LOGIT_TOL
        argmax = [argmax_lowest(x) for x in ref]
        for i in need:
            assert top2_gap(ref[i]) > 1e-4, "near-tie: oracle and GPU may legitimately differ"
        info = st.publish(rows, guesses, argmax)
        run.commit(rows, info.commit_rows)
        assert em == info.emitted
        hits += info.a
        check_state(L, ctx, st, {rows[0].token} | set(st.pool.keys()))
    L.la_set_debug(ctx.ctx, 0)


def fake_outputs(rows, V=8):
    """A deterministic stand-in for the model: the output of a row is a function
    of the last two tokens on its own visible path."""
    sets = la.vis_sets(rows)
    out = []
    for rw, s in zip(rows, sets):
        path = [rows[i].token for i in sorted(s, key=lambda i: rows[i].position)]
        a = path[-1]
        b = path[-2] if len(path) > 1 else 0
        out.append((5 * a + 3 * b + 1) % V)
    return out


@pytest.mark.parametrize("W,N,G", [(5, 3, 5), (3, 4, 2), (1, 3, 1), (8, 5, 8), (6, 4, 0), (2, 5, 8)])
def test_state_machine_with_injected_outputs(setup, W, N, G):
    """Pack, verification, pool, window and out ring are bit-exact with the oracle
    over many calls with frequent pool hits (outputs injected, model skipped)."""
    L, ctx, oracle, _ = setup
    p = [1, 2, 3, 4, 5, 6, 7, 0]
    first = L.la_prefill(ctx.ctx, p)
    st = la.LookaheadState(p, first, W, N, G)
    total_a = 0
    for step in range(60):
        rows, guesses = st.plan()
        outs = fake_outputs(rows)
        em = L.la_step_inject(ctx.ctx, W, N, G, outs)
        h, _, tok, pos, meta = L.la_debug_state(ctx.ctx)
        check_rows(rows, tok, pos, meta)
        info = st.publish(rows, guesses, outs)
        assert em == info.emitted, step
        assert (h["a"], h["winner"] if info.a else -1) == (info.a, info.winner if info.a else -1)
        total_a += info.a
        check_state(L, ctx, st, set(range(8)) | {first})
    if G > 0:
        assert total_a > 0


@pytest.mark.parametrize("opts", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("W,N,G", [(5, 3, 5), (3, 4, 2), (2, 5, 8), (1, 4, 3)])
def test_pool_seeding_with_injected_outputs(setup, W, N, G, opts):
    """Pool seeding (from the prompt, from the output, both) and the sliced
    window schedule: pack, verdicts, pool, window and out ring bit-exact with
    the oracle's state machine."""
    L, ctx, oracle, _ = setup
    p = [1, 2, 3, 4, 5, 6, 7, 0, 1, 2, 3, 5, 6, 1, 2]
    L.la_set_options(ctx.ctx, opts)
    try:
        first = L.la_prefill(ctx.ctx, p)
        st = la.LookaheadState(p, first, W, N, G, bool(opts & 1), bool(opts & 2), bool(opts & 4))
        total_a = 0
        for step in range(40):
            rows, guesses = st.plan()
            outs = fake_outputs(rows)
            em = L.la_step_inject(ctx.ctx, W, N, G, outs)
            h, _, tok, pos, meta = L.la_debug_state(ctx.ctx)
            check_rows(rows, tok, pos, meta)
            info = st.publish(rows, guesses, outs)
            assert em == info.emitted, step
            total_a += info.a
            check_state(L, ctx, st, set(range(8)) | {first})
        assert total_a > 0
    finally:
        L.la_set_options(ctx.ctx, 0)


def test_generate_with_pool_seeding_equals_ar_and_oracle(setup):
    """With both seeding options the output is still the AR output, and the
    number of packed calls equals the oracle's (same candidates, same hits)."""
    L, ctx, oracle, _ = setup
    base = prompt(12, 5)
    p = base + base + base
    ar = L.la_generate_ar(ctx.ctx, p, 48)
    assert ar == la.ar_generate(oracle, p, 48)
    L.la_set_options(ctx.ctx, L.LA_OPT_POOL_FROM_PROMPT | L.LA_OPT_POOL_FROM_OUTPUT)
    try:
        for W, N, G in [(5, 3, 5), (4, 4, 3), (2, 5, 8)]:
            st = L.la_stats()
            got = L.la_generate(ctx.ctx, p, 48, W, N, G, stats=st)
            assert got == ar, (W, N, G)
            tr = []
            la.lookahead_generate(oracle, p, 48, W, N, G, trace=tr, pool_from_prompt=True, pool_from_output=True)
            assert st.steps == len(tr), (W, N, G)
    finally:
        L.la_set_options(ctx.ctx, 0)


def test_generate_with_sliced_window_equals_ar_and_oracle(setup):
    """ALWAYS_FWD_ONE=False: still the AR output, and the same number of
    packed calls as the oracle running that schedule."""
    L, ctx, oracle, _ = setup
    p = prompt(32, 1)
    ar = L.la_generate_ar(ctx.ctx, p, 64)
    L.la_set_options(ctx.ctx, L.LA_OPT_SLICE_WINDOW)
    try:
        for W, N, G in [(5, 3, 5), (4, 4, 3), (1, 3, 1), (8, 5, 8)]:
            st = L.la_stats()
            got = L.la_generate(ctx.ctx, p, 64, W, N, G, stats=st)
            assert got == ar, (W, N, G)
            tr = []
            la.lookahead_generate(oracle, p, 64, W, N, G, trace=tr, slice_window=True)
            assert st.steps == len(tr), (W, N, G)
    finally:
        L.la_set_options(ctx.ctx, 0)


def test_generate_equals_ar_and_oracle(setup):
    L, ctx, oracle, _ = setup
    p = prompt(32, 1)
    ref = la.ar_generate(oracle, p, 64)
    ar = L.la_generate_ar(ctx.ctx, p, 64)
    assert ar == ref
    for W, N, G in [(5, 3, 5), (4, 4, 3), (1, 3, 1), (8, 5, 8), (3, 3, 0)]:
        st = L.la_stats()
        got = L.la_generate(ctx.ctx, p, 64, W, N, G, stats=st)
        assert got == ar, (W, N, G)
        assert st.tokens == 64 and 0 < st.steps <= 63


def test_row_invariance_probe(setup):
    """The ordinary row of a packed call is bit-identical to the same token decoded alone."""
    L, ctx, oracle, _ = setup
    p = prompt(40, 3)
    L.la_set_debug(ctx.ctx, 1)
    L.la_generate_ar(ctx.ctx, p, 2)
    alone, _ = L.la_debug_logits(ctx.ctx, 4, CFG.vocab)
    L.la_prefill(ctx.ctx, p)
    L.la_step(ctx.ctx, 8, 5, 8)
    packed, need = L.la_debug_logits(ctx.ctx, 512, CFG.vocab)
    assert need[0] == 0
    assert np.array_equal(alone[0].view(np.uint32), packed[0].view(np.uint32))
    L.la_set_debug(ctx.ctx, 0)


def test_error_contract(setup):
    L, ctx, oracle, _ = setup
    E = L.LaError
    # steps before any prefill of a fresh context
    from lookahead_decoding_gb300 import lib
    w = {k: v for k, v in ctx._keep.items()}
    c2 = lib().Context(CFG, w, max_ctx=64, max_W=4, max_N=4, max_G=2)
    try:
        with pytest.raises(E) as e:
            L.la_step(c2.ctx, 3, 3, 2)
        assert e.value.code == L.LA_ESTATE
        with pytest.raises(E) as e:
            L.la_prefill(c2.ctx, list(range(64)))            # no room for a new token
        assert e.value.code == L.LA_ECAPACITY
        with pytest.raises(E) as e:
            L.la_prefill(c2.ctx, [1, 2, CFG.vocab])           # id out of range
        assert e.value.code == L.LA_EINVAL
        L.la_prefill(c2.ctx, [1, 2, 3])
        with pytest.raises(E) as e:
            L.la_step(c2.ctx, 3, 2, 2)                        # N < 3
        assert e.value.code == L.LA_EINVAL
        with pytest.raises(E) as e:
            L.la_step(c2.ctx, 5, 3, 2)                        # W > max_W
        assert e.value.code == L.LA_ECAPACITY
        L.la_step(c2.ctx, 3, 3, 2)
        h0 = L.la_debug_state(c2.ctx)
        with pytest.raises(E) as e:
            L.la_step(c2.ctx, 4, 3, 2)                        # W changed without re-prefill
        assert e.value.code == L.LA_ESTATE
        assert L.la_debug_state(c2.ctx)[:2] == h0[:2]         # state untouched
        # run the context full: the step that would overflow fails closed
        code = None
        for _ in range(200):
            try:
                L.la_step(c2.ctx, 3, 3, 2)
            except E as ex:
                code = ex.code
                break
        assert code == L.LA_ECAPACITY
        h1, lv1, _, _, _ = L.la_debug_state(c2.ctx)
        with pytest.raises(E):
            L.la_step(c2.ctx, 3, 3, 2)
        h2, lv2, _, _, _ = L.la_debug_state(c2.ctx)
        assert (h1["K"], h1["n_out"], lv1) == (h2["K"], h2["n_out"], lv2)
    finally:
        c2.close()


def test_kernel_timeline_records_every_launch(setup):
    """The timeline holds one record per CTA of every kernel the library
    launched: each launch contributes its grid's CTA count of records (so the
    records weighted by 1/CTAs add up to the library's own launch count),
    every record ends after it starts, with a known kernel id and a CTA index
    inside its grid; a second start while open and a stop without one fail;
    the outputs are those of an untimed run."""
    L, ctx, _, _ = setup
    p = prompt(24, 5)
    ref = L.la_generate(ctx.ctx, p, 20, 8, 5, 8)
    st = L.la_stats()
    L.la_timeline_start(1 << 20)
    try:
        with pytest.raises(RuntimeError):
            L.la_timeline_start(16)
        out = L.la_generate(ctx.ctx, p, 20, 8, 5, 8, stats=st)
    finally:
        rec = L.la_timeline_stop(1 << 20)
    with pytest.raises(RuntimeError):
        L.la_timeline_stop(16)
    assert list(out) == list(ref)
    assert st.kernel_launches > 0
    assert abs(float(np.sum(1.0 / rec[:, 4])) - st.kernel_launches) < 1e-6 * st.kernel_launches
    assert np.all(rec[:, 1] >= rec[:, 0]) and np.all(rec[:, 0] > 0)
    assert np.all((rec[:, 2] >= 0) & (rec[:, 2] < len(L.TIMELINE_IDS)))
    assert np.all((rec[:, 3] >= 0) & (rec[:, 3] < rec[:, 4]))
    split = L.timeline_split(rec)
    assert sum(split["ns"].values()) + split["idle_ns"] == split["span_ns"]
    assert split["ns"]["gemm"] > 0 and split["ns"]["attention"] > 0 and split["ns"]["state"] > 0
