"""Spread ``replay_attention`` rows over worker processes.

Test infrastructure only, like the rest of this package.  Nothing here
computes: each worker calls ``core.replay_attention`` unchanged on its share
of the wanted rows, and the results are put back in row order.  The request's
arrays reach the workers as ``.npy`` files in a temporary directory that each
worker maps read-only, so a 1 GB query tensor is written once instead of
being pickled to every worker.  Workers are started with ``spawn`` (never
``fork``: the parent may already hold a CUDA context) and run numpy with one
thread each, so the worker count is the number of cores used.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os
import shutil
import tempfile
import time

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def host_cores() -> int:
    """Cores this process may run on."""
    if hasattr(os, "sched_getaffinity"):
        return len(os.sched_getaffinity(0))
    return os.cpu_count() or 1


def _load(d):
    return tuple(np.load(os.path.join(d, n + ".npy"), mmap_mode="r") for n in ("q", "k", "v"))


def _rows_job(d, ops, dtype, base, rows):
    from .core import replay_attention
    q, k, v = _load(d)
    out, _ = replay_attention(*ops, q, k, v, dtype, base, rows=rows)
    return out


def _timed_job(d, ops, dtype, base, seconds, batch, seed, T):
    """Random batches of rows until ``seconds`` have passed; returns the rows done."""
    from .core import replay_attention
    q, k, v = _load(d)
    rng = np.random.default_rng(seed)
    done, t0 = [], time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        rows = np.sort(rng.choice(T, size=batch, replace=False))
        replay_attention(*ops, q, k, v, dtype, base, rows=rows)
        done.extend(int(x) for x in rows)
    return done


class RowPool:
    """A request's arrays on disk plus a spawn-started pool of ``workers``
    processes; use as a context manager."""

    def __init__(self, q, k, v, workers=None):
        self.workers = max(1, workers or host_cores())
        self.dir = tempfile.mkdtemp(prefix="akv_oracle_")
        for name, a in (("q", q), ("k", k), ("v", v)):
            np.save(os.path.join(self.dir, name + ".npy"), np.ascontiguousarray(a))
        saved = {n: os.environ.get(n) for n in _THREAD_VARS}
        for n in _THREAD_VARS:
            os.environ[n] = "1"
        try:
            self.ex = cf.ProcessPoolExecutor(self.workers, mp_context=mp.get_context("spawn"))
            # start every worker now, while the one-thread settings are in the
            # environment they inherit
            list(self.ex.map(int, range(self.workers)))
        finally:
            for n, val in saved.items():
                if val is None:
                    os.environ.pop(n, None)
                else:
                    os.environ[n] = val

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def close(self):
        self.ex.shutdown()
        shutil.rmtree(self.dir, ignore_errors=True)

    def rows(self, ops, dtype, base, rows):
        """``core.replay_attention(..., rows=rows)[0]`` over the workers."""
        rows = np.asarray(rows, dtype=np.int64)
        ops = tuple(np.asarray(a) for a in ops)
        w = max(1, min(self.workers, len(rows)))
        # interleaved shares: early and late rows (short and long active
        # caches) are spread evenly over the workers
        order = np.argsort(rows, kind="stable")
        shares = [np.sort(rows[order[i::w]]) for i in range(w)]
        futs = [self.ex.submit(_rows_job, self.dir, ops, dtype, base, sh) for sh in shares]
        parts = [f.result() for f in futs]
        out = np.empty((len(rows),) + parts[0].shape[1:], dtype=np.float64)
        where = {int(t): i for i, t in enumerate(rows)}
        for sh, part in zip(shares, parts):
            for j, t in enumerate(sh):
                out[where[int(t)]] = part[j]
        return out

    def timed(self, ops, dtype, base, seconds, batch=4, seed=0):
        """Every worker computes random batches of ``batch`` rows for about
        ``seconds``.  Returns (rows done, wall seconds, workers)."""
        T = int(np.asarray(ops[0])[-1])
        ops = tuple(np.asarray(a) for a in ops)
        t0 = time.perf_counter()
        futs = [self.ex.submit(_timed_job, self.dir, ops, dtype, base, seconds, batch,
                               seed * 1000 + i, T) for i in range(self.workers)]
        done = [t for f in futs for t in f.result()]
        wall = time.perf_counter() - t0
        return np.array(done, dtype=np.int64), wall, self.workers


def replay_attention_rows(ops, q, k, v, dtype, base, rows, workers=None):
    """``core.replay_attention(*ops, q, k, v, dtype, base, rows=rows)[0]``
    computed by up to ``workers`` processes (default: one per host core)."""
    rows = np.asarray(rows, dtype=np.int64)
    workers = max(1, min(workers or host_cores(), len(rows)))
    if workers == 1:
        from .core import replay_attention
        return replay_attention(*ops, q, k, v, dtype, base, rows=rows)[0]
    with RowPool(q, k, v, workers) as pool:
        return pool.rows(ops, dtype, base, rows)


def timed_rows(ops, q, k, v, dtype, base, seconds, workers=None, batch=4, seed=0):
    """``RowPool.timed`` on a pool made for this call."""
    with RowPool(q, k, v, workers) as pool:
        return pool.timed(ops, dtype, base, seconds, batch=batch, seed=seed)


def _call_job(d, names, fn_path, kwargs):
    import importlib
    mod, fn = fn_path.split(":")
    f = getattr(importlib.import_module(mod), fn)
    arrays = {n: np.load(os.path.join(d, n + ".npy"), mmap_mode="r") for n in names}
    t0 = time.perf_counter()
    out = f(**arrays, **kwargs)
    return out, time.perf_counter() - t0


def timed_call(fn_path, arrays, **kwargs):
    """Run ``fn(**arrays, **kwargs)`` (``fn_path`` = "module:function" of this
    package) in one spawned worker with one numpy thread, the arrays passed as
    mapped ``.npy`` files.  Returns (result, seconds the call took in the
    worker)."""
    d = tempfile.mkdtemp(prefix="akv_oracle_")
    try:
        for name, a in arrays.items():
            np.save(os.path.join(d, name + ".npy"), np.ascontiguousarray(a))
        saved = {n: os.environ.get(n) for n in _THREAD_VARS}
        for n in _THREAD_VARS:
            os.environ[n] = "1"
        try:
            ex = cf.ProcessPoolExecutor(1, mp_context=mp.get_context("spawn"))
            fut = ex.submit(_call_job, d, list(arrays), fn_path, kwargs)
        finally:
            for n, val in saved.items():
                if val is None:
                    os.environ.pop(n, None)
                else:
                    os.environ[n] = val
        try:
            return fut.result()
        finally:
            ex.shutdown()
    finally:
        shutil.rmtree(d, ignore_errors=True)
