"""Several lookahead requests in one packed target call (oracle; test infrastructure).

The pages run one request per call: the pinned wrapper asserts a batch of
one (M7.3 §0x04C), and they say this is a property of that code, not of the
method; request admission and serving belong to M7.8 (§0x09).  The state a
call reads and writes is per request: the n-gram pool belongs to one
request (§0x03B), and so do the committed K/V, the window and the frontier
(§0x06A, §0x07).

Reading taken here for a batched call: the packed rows of B requests are
stacked in request order, each request's rows in its own packed order
(§0x04); every request keeps its own committed K/V, window, pool, frontier
and step counter; a row sees its own request's committed prefix and the rows
of its own request that its visibility set names, never another request's
rows or cache.  All requests share one knob set (W, N, G).  Each request then
verifies, publishes and advances exactly as alone, and a request that has
produced ``max_new`` tokens leaves the batch.  The batched call therefore
computes what each request's own call computes: the definition this oracle
writes out is "each request, alone", evaluated in one forward.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

from .lookahead import LookaheadState, StepInfo, check_args, meta_mask
from .model import OracleModel, argmax_lowest


@dataclasses.dataclass
class BatchStep:
    """One batched call: the requests in it (batch order) and their outcomes."""
    requests: List[int]
    rows: List[int]            # packed rows per request
    infos: List[StepInfo]
    logits: List[object]       # per request, the logits of its packed rows [rows, V]
    needed: List[List[int]]    # per request, the packed rows whose logits the step reads
    tokens: List[List[int]]    # per request, the input token of every packed row
    positions: List[List[int]] # per request, the logical position of every packed row


class BatchedLookahead:
    """B greedy lookahead requests advanced together, one packed forward per call."""

    def __init__(self, model: OracleModel, prompts: Sequence[Sequence[int]], W: int, N: int, G: int,
                 pool_from_prompt: bool = False, pool_from_output: bool = False,
                 slice_window: bool = False):
        check_args(W, N, G)
        self.model = model
        self.caches, self.states, self.out = [], [], []
        for p in prompts:
            cache, logits = model.prefill(list(p))
            first = argmax_lowest(logits[-1])
            self.caches.append(cache)
            self.states.append(LookaheadState(list(p), first, W, N, G, pool_from_prompt, pool_from_output,
                                              slice_window))
            self.out.append([first])

    def active(self, max_new: int) -> List[int]:
        return [b for b, o in enumerate(self.out) if len(o) < max_new]

    def step(self, max_new: int, choose=None) -> Optional[BatchStep]:
        """One batched call over the requests that still need tokens.

        ``choose(b, logits, needed)``, if given, returns request b's argmax per
        packed row in place of the greedy selector (a test feeds another
        implementation's decisions to keep the two state machines in step)."""
        live = self.active(max_new)
        if not live:
            return None
        plans = [self.states[b].plan() for b in live]
        calls = [([r.token for r in rows], [r.position for r in rows], self.caches[b], meta_mask(rows))
                 for b, (rows, _) in zip(live, plans)]
        results = self.model.forward_many(calls)
        infos, all_logits, needed = [], [], []
        for b, (rows, guesses), (logits, new_k, new_v) in zip(live, plans, results):
            all_logits.append(logits)
            needed.append([r.packed_index for r in rows if r.request_logit])
            need = [r.packed_index for r in rows if r.request_logit]
            argmax = (choose(b, logits, need) if choose is not None
                      else [argmax_lowest(logits[i]) for i in range(len(rows))])
            info = self.states[b].publish(rows, guesses, argmax)
            idx = list(info.commit_rows)
            self.caches[b].append([k[idx] for k in new_k], [v[idx] for v in new_v])
            self.out[b].extend(info.emitted)
            infos.append(info)
        return BatchStep(live, [len(rows) for rows, _ in plans], infos, all_logits, needed,
                         [[r.token for r in rows] for rows, _ in plans], [[r.position for r in rows] for rows, _ in plans])


def lookahead_generate_batch(model: OracleModel, prompts: Sequence[Sequence[int]], max_new: int,
                             W: int, N: int, G: int, trace: Optional[list] = None,
                             **options) -> List[List[int]]:
    """Greedy lookahead decoding of several prompts in batched packed calls."""
    bl = BatchedLookahead(model, prompts, W, N, G, **options)
    while True:
        st = bl.step(max_new)
        if st is None:
            break
        if trace is not None:
            trace.append(st)
    return [o[:max_new] for o in bl.out]
