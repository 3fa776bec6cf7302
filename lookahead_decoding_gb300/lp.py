"""Lookahead Parallelism, host side: which share of a packed call each rank
computes, and the one exchange per call (M7.3 §0x07A, replicated-model
token parallelism and the pinned distributed path; break the sequential
dependency §3.4).

Every rank holds a full replica of the model and the same request state
(window, pool, emitted tokens).  In a steady call rank k of P computes the
ordinary row, the window columns [k W / P, (k + 1) W / P) at every
trajectory level (with the base-stripe rows those columns see) and the pool
candidates c with c mod P = k; nothing is exchanged during the forward.
Afterwards each rank contributes one int32 record,

    [0, W)            the deepest-level output token of each column it owns,
                      -1 for the others
    W                 its longest accepted prefix a over its candidates
    W + 1             that candidate's global index (-1 when a = 0)
    W + 2 .. W + 2+N  the tokens that hit emits (a + 1 of them, -1 padded)

an all-gather over the process group gives every rank every record, and
merge() applies the single-worker rule: all W column tokens, the longest
hit, ties to the lowest candidate index.  Every rank then publishes the same
outputs (pool, window, emitted tokens).  The K/V of an accepted candidate's
rows exists only on the rank that verified it, so no rank commits it: each
commits its ordinary rows and feeds the emitted tokens back as the next
call's ordinary rows (a + 1 of them after a hit of a).

Warm-up fills (no candidates, level sizes still growing) are computed whole
by every rank and need no exchange.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


def shard_columns(W: int, P: int, k: int) -> List[int]:
    """Window columns rank k of P owns: a contiguous block."""
    lo, hi = (k * W) // P, ((k + 1) * W) // P
    return list(range(lo, hi))


def shard_candidates(n_candidates: int, P: int, k: int) -> List[int]:
    """Candidate slots rank k of P verifies: every P-th from k."""
    return list(range(k, n_candidates, P))


def record_len(W: int, N: int) -> int:
    return W + 2 + N


def encode(W: int, N: int, z: Dict[int, int], a: int, winner: int, emitted: Sequence[int]) -> np.ndarray:
    """One rank's int32 record (layout in the module docstring)."""
    if len(emitted) != a + 1 or a + 1 > N:
        raise ValueError("a hit of a tokens emits a + 1 <= N tokens")
    rec = np.full(record_len(W, N), -1, dtype=np.int32)
    for j, t in z.items():
        if not 0 <= j < W:
            raise ValueError("column out of range")
        rec[j] = t
    rec[W] = a
    rec[W + 1] = winner if a > 0 else -1
    rec[W + 2: W + 2 + a + 1] = list(emitted)
    return rec


def merge(records: np.ndarray, W: int, N: int) -> Tuple[List[int], int, int, List[int]]:
    """The call's outputs from every rank's record [P][record_len]: the W
    deepest-level tokens (each column owned by exactly one rank), the longest
    hit (the lowest candidate index among equal hits), its emitted tokens."""
    records = np.asarray(records, dtype=np.int32)
    owned = records[:, :W] >= 0
    if not np.all(owned.sum(axis=0) == 1):
        raise ValueError("every column needs exactly one owner")
    z = [int(records[owned[:, j], j][0]) for j in range(W)]
    a = records[:, W]
    best_a = int(a.max())
    if best_a == 0:
        return z, 0, -1, [int(records[0, W + 2])]
    tied = np.nonzero(a == best_a)[0]
    k = int(tied[np.argmin(records[tied, W + 1])])
    return z, best_a, int(records[k, W + 1]), [int(t) for t in records[k, W + 2: W + 2 + best_a + 1]]


def exchange(record: np.ndarray, group=None) -> np.ndarray:
    """All-gather of one int32 record per rank (torch.distributed; the record
    goes through the group's device, the CUDA device for NCCL)."""
    import torch
    import torch.distributed as dist
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.from_numpy(np.ascontiguousarray(record, dtype=np.int32)).to(dev)
    out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(out, t, group=group)
    return np.stack([o.cpu().numpy() for o in out])
