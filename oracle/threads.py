"""The oracle's forward and backward over contiguous row ranges on several
host threads.

Test infrastructure only, like the rest of ``oracle/``: the CPU-baseline leg
of ``bench.py`` and ``tests/`` use it; nothing on the CUDA path may.

Rows are independent in every op here (RMSNorm, LayerNorm, softmax; a
GroupNorm sample is a row), so the rows split into T contiguous ranges, one
per thread, and each thread runs the unchanged float64 oracle on its range.
numpy releases the interpreter lock inside its array operations, so the
threads run in parallel.  The only cross-row results are the parameter
gradients (dW and, where the op has a bias, dB): each range's float64 sum
is added to the total in range order, so the result depends only on the
number of ranges.  Adds no arithmetic of the method.
"""
from __future__ import annotations

import concurrent.futures
from typing import Callable, List, Sequence

import numpy as np


def row_ranges(rows: int, parts: int) -> List[range]:
    """``parts`` contiguous ranges covering ``rows`` rows (the last ones may
    be empty when rows < parts)."""
    parts = max(1, parts)
    return [range(rows * k // parts, rows * (k + 1) // parts) for k in range(parts)]


def map_rows(fn: Callable[[slice], Sequence], rows: int, threads: int):
    """Run ``fn(rows_slice)`` on each of ``threads`` contiguous row ranges in
    parallel and return the per-range results in range order."""
    spans = [r for r in row_ranges(rows, threads) if len(r)]
    if len(spans) <= 1:
        return [fn(slice(0, rows))]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(spans)) as ex:
        futs = [ex.submit(fn, slice(r.start, r.stop)) for r in spans]
        return [f.result() for f in futs]


def sum_in_order(parts: Sequence[np.ndarray]) -> np.ndarray:
    """Sum of per-range gradient vectors, added in range order."""
    total = np.array(parts[0], dtype=np.float64, copy=True)
    for p in parts[1:]:
        total = total + p
    return total
