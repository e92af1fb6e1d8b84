"""Run oracle calls in parallel worker processes (spawned, never forked, so a
CUDA context in the parent is never duplicated)."""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

_pool = None


def pool() -> ProcessPoolExecutor:
    global _pool
    if _pool is None:
        workers = max(1, min(16, os.cpu_count() or 1))
        _pool = ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))
    return _pool


def _steps_chunk(args):
    import oracle

    logits, dtype, temperature, seed, base, steps, want_gap = args
    return oracle.gumbel_argmax_steps(logits, temperature, seed, base, steps, dtype=dtype,
                                      want_gap=want_gap)


def gumbel_argmax_steps(logits, temperature, seed, base: int, steps: int, dtype: int,
                        want_gap: bool = False, chunks: int | None = None):
    """oracle.gumbel_argmax_steps spread over worker processes by step range."""
    n = chunks or max(1, min(steps, 4 * (os.cpu_count() or 1)))
    edges = np.linspace(0, steps, n + 1).astype(np.int64)
    jobs = [(logits, dtype, temperature, seed, base + int(a), int(b - a), want_gap)
            for a, b in zip(edges[:-1], edges[1:]) if b > a]
    parts = list(pool().map(_steps_chunk, jobs))
    if want_gap:
        return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))
    return np.concatenate(parts)


def _row_job(args):
    import oracle

    kind, row, dtype, T, seed, row_id, offset, extra = args
    if kind == "gumbel":
        return oracle.sample_row(row, T, seed, row_id, offset, dtype=dtype)
    if kind == "hlg":
        return oracle.hlg_sample_row(row, T, seed, row_id, offset, dtype=dtype, **extra)
    raise ValueError(kind)


def rows(kind: str, logits, dtype, T, S, O, extra=None, row_ids=None):
    """Oracle sample of the selected rows (default: all) in worker processes.
    Each row keeps its index in the full batch as the Philox row word.
    Returns (idx int64[n], gap float64[n]) in the order of row_ids."""
    B = logits.shape[0]
    row_ids = np.arange(B) if row_ids is None else np.asarray(row_ids)
    jobs = [(kind, np.ascontiguousarray(logits[r]), dtype, float(T[r]), int(S[r]), int(r),
             int(O[r]), extra or {}) for r in row_ids]
    res = list(pool().map(_row_job, jobs, chunksize=max(1, len(jobs) // 64)))
    return (np.array([r[0] for r in res], dtype=np.int64),
            np.array([r[1] for r in res], dtype=np.float64))


def _hlg_steps_job(args):
    import oracle

    row, dtype, T, seed, row_id, base, steps, extra = args
    return np.array([oracle.hlg_sample_row(row, T, seed, row_id, base + k, dtype=dtype, **extra)[0]
                     for k in range(steps)], dtype=np.int64)


def hlg_row_steps(row, dtype, T, seed, row_id, base: int, steps: int, extra: dict):
    """HLG draws of one row at offsets base .. base+steps-1, in worker processes."""
    n = max(1, min(steps, 4 * (os.cpu_count() or 1)))
    edges = np.linspace(0, steps, n + 1).astype(np.int64)
    jobs = [(np.ascontiguousarray(row), dtype, T, seed, row_id, base + int(a), int(b - a), extra)
            for a, b in zip(edges[:-1], edges[1:]) if b > a]
    return np.concatenate(list(pool().map(_hlg_steps_job, jobs)))


def rows_at_steps(kind: str, logits, dtype, T, S, steps, extra=None, row_ids=None):
    """Oracle draws of the selected rows at every decode step in `steps`
    (offset = step for every row), one (step, row) pair per task so the workers
    stay balanced. Returns (idx int64[len(steps), n], gap float64[len(steps), n])."""
    B = logits.shape[0]
    row_ids = np.arange(B) if row_ids is None else np.asarray(row_ids)
    rows_c = {int(r): np.ascontiguousarray(logits[r]) for r in row_ids}
    jobs = [(kind, rows_c[int(r)], dtype, float(T[r]), int(S[r]), int(r), int(s), extra or {})
            for s in steps for r in row_ids]
    res = list(pool().map(_row_job, jobs, chunksize=max(1, len(jobs) // 256)))
    n = len(row_ids)
    idx = np.array([r[0] for r in res], dtype=np.int64).reshape(len(steps), n)
    gap = np.array([r[1] for r in res], dtype=np.float64).reshape(len(steps), n)
    return idx, gap


def _filtered_chunk(args):
    import oracle

    logits, dtype, temperature, seed, base, steps, top_k, top_p = args
    return oracle.filtered_steps(logits, temperature, seed, base, steps, top_k=top_k,
                                 top_p=top_p, dtype=dtype)


def filtered_steps(logits, temperature, seed, base: int, steps: int, dtype: int, top_k=0,
                   top_p=1.0):
    """oracle.filtered_steps spread over worker processes by step range."""
    n = max(1, min(steps, 4 * (os.cpu_count() or 1)))
    edges = np.linspace(0, steps, n + 1).astype(np.int64)
    jobs = [(logits, dtype, temperature, seed, base + int(a), int(b - a), top_k, top_p)
            for a, b in zip(edges[:-1], edges[1:]) if b > a]
    return np.concatenate(list(pool().map(_filtered_chunk, jobs)))


def _filtered_row_job(args):
    import oracle

    row, dtype, T, seed, row_id, offset, k, p = args
    return oracle.filtered_sample_row(row, T, seed, row_id, offset, top_k=k, top_p=p, dtype=dtype)


def filtered_rows_at_steps(logits, dtype, T, S, steps, top_k, top_p, row_ids=None):
    """Filtered oracle draws of the selected rows at every step in `steps`, one
    (step, row) per task. -> (idx, gap, edge), each [len(steps), n]."""
    B = logits.shape[0]
    row_ids = np.arange(B) if row_ids is None else np.asarray(row_ids)
    rows_c = {int(r): np.ascontiguousarray(logits[r]) for r in row_ids}
    jobs = [(rows_c[int(r)], dtype, float(T[r]), int(S[r]), int(r), int(s), int(top_k[r]),
             float(top_p[r])) for s in steps for r in row_ids]
    res = list(pool().map(_filtered_row_job, jobs, chunksize=max(1, len(jobs) // 256)))
    shape = (len(steps), len(row_ids))
    return (np.array([r[0] for r in res], dtype=np.int64).reshape(shape),
            np.array([r[1] for r in res], dtype=np.float64).reshape(shape),
            np.array([r[2] for r in res], dtype=np.float64).reshape(shape))
