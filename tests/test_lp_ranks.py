"""Lookahead Parallelism across processes: 2 and 4 gloo ranks on CPU (one
rank per GPU over NCCL runs the same host code).  Each rank keeps a full
replica (here the oracle transformer stands in for the rank's forward) and
the request state; it computes the share lookahead_decoding_gb300.lp assigns
it, contributes its int32 record through lp.exchange, and publishes what
lp.merge returns.  Every rank's stream must equal the single-worker oracle
loop's (and AR), call by call, with accepted candidates re-fed."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W, N, G, MAX_NEW = 5, 4, 5, 40


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _model(seed):
    import synth
    from oracle.model import OracleModel
    cfg = synth.ModelConfig(n_layers=1, d_model=16, n_heads=2, head_dim=8, d_ffn=32, vocab=6, dtype="f32",
                            init_std=0.5)
    return OracleModel(cfg, synth.llama_weights(cfg, seed))


def _prompt(seed):
    return [int(t) for t in np.random.default_rng(seed).integers(0, 6, 10)]


def _rank(rank, world, port, seed, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from lookahead_decoding_gb300 import lp
    from oracle import lookahead as la
    from oracle import lp as olp
    from oracle.model import argmax_lowest
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        m = _model(seed)
        prompt = _prompt(seed)
        worker = olp.Worker(m, prompt)              # this rank's replica and its committed K/V
        st = la.LookaheadState(prompt, worker.first, W, N, G)
        out, trace, bytes_sent = [worker.first], [], 0
        while len(out) < MAX_NEW:
            rows, guesses = st.plan()
            if not st.steady:
                lg = worker.forward(rows)
                info = st.publish(rows, guesses, [argmax_lowest(x) for x in lg])
            else:
                cols = lp.shard_columns(W, world, rank)
                cands = lp.shard_candidates(len(guesses), world, rank)
                mine = olp.shard_rows(rows, cols, cands)
                lg = worker.forward(mine)
                am = {r.packed_index: argmax_lowest(lg[i]) for i, r in enumerate(mine)}
                d = max(r.level for r in rows if r.role == la.LOOKAHEAD)
                z = {r.column: am[r.packed_index] for r in mine
                     if r.role == la.LOOKAHEAD and r.level == d and r.column in cols}
                vstart = len(rows) - len(guesses) * st.S
                a, wl, em = la.greedy_verify(am[0], [guesses[c] for c in cands],
                                             lambda c, s: am[vstart + cands[c] * st.S + s])
                rec = lp.encode(W, N, z, a, cands[wl] if wl >= 0 else -1, em)
                bytes_sent += rec.nbytes
                recs = lp.exchange(rec)
                zz, a, win, emitted = lp.merge(recs, W, N)
                argmax = [0] * len(rows)
                for j, i in zip(range(W), st.deepest_rows(rows)):
                    argmax[i] = zz[j]
                info = st.publish(rows, guesses, argmax, (emitted, a, win))
            worker.refeed = list(info.emitted)
            trace.append((info.a, info.winner, info.emitted))
            out.extend(info.emitted)
        q.put((rank, out[:MAX_NEW], trace, bytes_sent))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ranks_equal_single_worker(world):
    import sys
    sys.path.insert(0, ROOT)
    from oracle import lookahead as la
    hits = 0
    for seed in (0, 1):
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, world, port, seed, q)) for r in range(world)]
        for p in procs:
            p.start()
        res = {}
        for _ in range(world):
            r, out, trace, nbytes = q.get(timeout=240)
            res[r] = (out, trace, nbytes)
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
        m, prompt = _model(seed), _prompt(seed)
        ref_trace = []
        ref = la.lookahead_generate(m, prompt, MAX_NEW, W, N, G, trace=ref_trace)
        assert ref == la.ar_generate(m, prompt, MAX_NEW)
        for r in range(world):
            out, trace, nbytes = res[r]
            assert out == ref
            assert trace == [(t.a, t.winner, t.emitted) for t in ref_trace]
            assert nbytes <= 4 * (W + 2 + N) * len(trace)      # one small int32 record per call
        hits += sum(t[0] > 0 for t in res[0][1])
    assert hits > 0              # accepted candidates, so the re-feed path ran


def test_merge_rule():
    from lookahead_decoding_gb300 import lp
    recs = np.stack([lp.encode(5, 4, {0: 7, 1: 8}, 2, 3, [1, 2, 9]),
                     lp.encode(5, 4, {2: 6, 3: 5, 4: 4}, 2, 1, [1, 2, 3])])
    z, a, win, em = lp.merge(recs, 5, 4)
    assert z == [7, 8, 6, 5, 4] and (a, win, em) == (2, 1, [1, 2, 3])     # equal hits: lowest candidate
    none = np.stack([lp.encode(3, 3, {0: 1}, 0, -1, [4]), lp.encode(3, 3, {1: 2, 2: 3}, 0, -1, [4])])
    assert lp.merge(none, 3, 3) == ([1, 2, 3], 0, -1, [4])
    with pytest.raises(ValueError):
        lp.merge(np.stack([lp.encode(2, 2, {0: 1}, 0, -1, [0]), lp.encode(2, 2, {0: 1}, 0, -1, [0])]), 2, 2)
