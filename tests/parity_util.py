"""Helpers for the GPU parity tests: running the CPU oracle (optionally over a
spawn-started process pool, created before any GPU work is queued from a
worker) and comparing GPU output with it under the stated tolerance."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

import oracle

_POOL = None


def pool():
    """A spawn-context pool (safe with CUDA in the parent)."""
    global _POOL
    if _POOL is None:
        n = max(1, min(16, (os.cpu_count() or 2)))
        _POOL = mp.get_context("spawn").Pool(n)
    return _POOL


def _gemm_rows(args):
    wtype, w, K, qs, d, bs, rows = args
    return oracle.get().gemm(wtype, w, K, qs, d, bs, rows=rows)


def oracle_gemm(wtype, w, K, qs, d, bs, rows=None, parallel_threshold=2e8):
    """Oracle Y (fp64) and sum_b |c_b| for the given token rows (all if None)."""
    M = qs.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    work = len(rows) * w.shape[0] * K
    if work < parallel_threshold or len(rows) < 2:
        return oracle.get().gemm(wtype, w, K, qs, d, bs, rows=rows)
    p = pool()
    nchunk = min(len(rows), 4 * p._processes)
    chunks = [c for c in np.array_split(rows, nchunk) if len(c)]
    # only ship the token rows each chunk needs
    jobs = []
    for c in chunks:
        jobs.append((wtype, w, K, qs[c], d[c], bs[c], np.arange(len(c), dtype=np.int64)))
    res = p.map(_gemm_rows, jobs)
    y = np.concatenate([r[0] for r in res])
    a = np.concatenate([r[1] for r in res])
    return y, a


def tolerance(absc):
    return 2e-5 * absc + 1e-6


def assert_gemm_close(y_gpu, y_ref, absc, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    tol = tolerance(absc)
    bad = ~(err <= tol)       # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        ratio = np.nanmax(err / tol)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, "
                             f"worst err/tol {ratio:.3g}; first at {idx.tolist()}: "
                             f"gpu {y_gpu[tuple(idx[0])]} ref {y_ref[tuple(idx[0])]}")
    return float(np.max(err / tol)) if err.size else 0.0


def sample_rows(M, n, seed, tail=8):
    """n seeded random rows plus the first row and the last `tail` rows."""
    r = np.random.default_rng(seed)
    rows = set(r.choice(M, size=min(n, M), replace=False).tolist())
    rows |= {0} | set(range(max(0, M - tail), M))
    return np.array(sorted(rows), dtype=np.int64)


def tile_rows(M, n, seed, bm=128, tail=16):
    """Rows for a sampled parity check at large M: n seeded random rows, one
    seeded row inside every bm-token tile, the first row, and the last
    `tail` rows plus every row of a ragged last tile (M % bm != 0)."""
    r = np.random.default_rng(seed)
    rows = set(r.choice(M, size=min(n, M), replace=False).tolist())
    for t0 in range(0, M, bm):
        rows.add(int(r.integers(t0, min(M, t0 + bm))))
    last = M - (M % bm) if M % bm else M - min(M, tail)
    rows |= {0} | set(range(max(0, min(last, M - tail)), M))
    return np.array(sorted(rows), dtype=np.int64)
