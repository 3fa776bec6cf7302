"""Jacobi and Gauss–Seidel sweeps over a triangular system (oracle; test infrastructure).

M7.3 §0x02: greedy decoding of m tokens is the triangular system
y_i = T_i(y_<i); one Jacobi sweep updates every coordinate from the previous
vector, y_i^(r+1) = T_i(y_<i^(r)); Gauss–Seidel consumes same-sweep updates,
y_i^(r+1) = T_i(y_<i^(r+1)).  §0x02A: Jacobi reaches the autoregressive fixed
point within m sweeps.
"""
from __future__ import annotations

from typing import Callable, List, Sequence

Operator = Callable[[int, Sequence[int]], int]   # T(i, y_<i) -> y_i  (0-based i)


def jacobi_sweep(T: Operator, y: Sequence[int]) -> List[int]:
    old = list(y)
    return [T(i, old[:i]) for i in range(len(old))]


def gauss_seidel_sweep(T: Operator, y: Sequence[int]) -> List[int]:
    new = list(y)
    for i in range(len(new)):
        new[i] = T(i, new[:i])
    return new


def solve(T: Operator, y0: Sequence[int], sweep=jacobi_sweep, max_sweeps: int = 1000):
    """Sweep until a fixed point; returns (fixed point, number of sweeps that changed y... )

    The count returned is the number of sweeps applied until the vector stops
    changing, i.e. the sweep that first produced the fixed point.
    """
    y = list(y0)
    for r in range(1, max_sweeps + 1):
        nxt = sweep(T, y)
        if nxt == y:
            return y, r - 1
        y = nxt
    raise RuntimeError("no fixed point")
