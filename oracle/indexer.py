"""Exact indexer scores and exact top-K by full sort (test infrastructure only).

Definition followed ("Fusing Indexer Scoring and Exact Top-k for
DeepSeek-V3.2", section 1.1 equation; section 2.3 problem definition):

    I[t, s] = sum_j w[t, j] * ReLU(q[t, j] . k[s]),   j = 1..64,

with q = q_code * q_scale[t] (one FP32 scale per query token, shared by its 64
heads) and k = k_code * k_scale[s] (one FP32 scale per key token).  Because both
scales are positive, ReLU(q_scale * k_scale * x) = q_scale * k_scale * ReLU(x),
so the scales are applied after the per-head dot, exactly as dequantisation.

Output per row: the K valid key indices with the largest scores, unordered
(section 2.3); ties may go to any valid index.  This oracle breaks ties by the
lowest index.  Rows with fewer than K valid keys return all of them followed by
-1 padding (the pages leave padding open; this is the reading taken).

Paged rows (contest write-up, "DSA TopK Indexer"): keys live in a cache of
64-token pages; logical token s of sequence b sits in physical slot
block_table[b][s // 64] * 64 + s % 64, and the returned index is that physical
slot.  Query row i of a sequence with next_n query tokens sees logical keys
[0, seq_len - next_n + i + 1).
"""
from __future__ import annotations

import numpy as np

from . import e4m3

DOT_UNIT = 2.0 ** -18   # one e4m3 unit (2^-9) squared
PAGE = 64


def exact_dots(q_units: np.ndarray, k_units: np.ndarray) -> np.ndarray:
    """Exact integer dots q_units[h] . k_units[s] -> int64 [H, L] in 2^-18 units.

    The operands are float64 arrays holding integers (|x| <= 229376 < 2^18).
    Every product is an integer below 2^36 and every partial sum of 128 of them
    an integer below 2^43 < 2^53, so a float64 matrix product is exact in any
    summation order; the cast back to int64 is exact too.
    """
    d = q_units @ k_units.T
    return d.astype(np.int64)


def combine_heads(dots: np.ndarray, w_row: np.ndarray, q_scale: float, k_scale: np.ndarray):
    """Scores I and tolerance scale E of one row from its exact dots.

    I[s] = q_scale * k_scale[s] * 2^-18 * sum_j w[j] * max(dot[j, s], 0)
    E[s] = q_scale * k_scale[s] * 2^-18 * sum_j |w[j]| * |dot[j, s]|
    (float64; E is the per-index magnitude the parity tolerance is relative to).
    """
    w64 = w_row.astype(np.float64)
    relu = np.maximum(dots, 0).astype(np.float64)
    scale = float(q_scale) * k_scale.astype(np.float64) * DOT_UNIT
    I = (w64 @ relu) * scale
    E = (np.abs(w64) @ np.abs(dots).astype(np.float64)) * scale
    return I, E


def topk_by_sort(ids: np.ndarray, I: np.ndarray, K: int, order_key: np.ndarray | None = None):
    """Full sort by (score descending, order_key ascending); first min(L, K)
    ids, then -1 padding up to K.  Returns (out[K], kth_score or None)."""
    L = len(ids)
    sec = ids if order_key is None else order_key
    order = np.lexsort((sec, -I))
    out = np.full(K, -1, np.int64)
    n = min(L, K)
    out[:n] = ids[order[:n]]
    kth = float(I[order[K - 1]]) if L >= K else None
    return out, kth


class DenseOracle:
    """Oracle for a dense (prefill) problem given as plain arrays."""

    def __init__(self, q, q_scale, k, k_scale, w, row_begin, row_end, K):
        self.qu = e4m3.decode_array_units(q).astype(np.float64)   # [Q, H, D]
        self.ku = e4m3.decode_array_units(k).astype(np.float64)   # [N, D]
        self.q_scale = np.asarray(q_scale, np.float32)
        self.k_scale = np.asarray(k_scale, np.float32)
        self.w = np.asarray(w, np.float32)
        self.row_begin = np.asarray(row_begin, np.int64)
        self.row_end = np.asarray(row_end, np.int64)
        self.K = int(K)

    @classmethod
    def from_inputs(cls, inp):
        return cls(inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin,
                   inp.row_end, inp.K)

    @property
    def Q(self):
        return self.qu.shape[0]

    def row_scores(self, t: int):
        """(ids int64[L], I float64[L], E float64[L]) over the valid keys of row t."""
        b, e = int(self.row_begin[t]), int(self.row_end[t])
        ids = np.arange(b, e, dtype=np.int64)
        if e <= b:
            return ids, np.zeros(0), np.zeros(0)
        dots = exact_dots(self.qu[t], self.ku[b:e])
        I, E = combine_heads(dots, self.w[t], self.q_scale[t], self.k_scale[b:e])
        return ids, I, E

    def topk(self, t: int):
        ids, I, E = self.row_scores(t)
        out, kth = topk_by_sort(ids, I, self.K)
        return out, ids, I, E, kth


class PagedOracle:
    """Oracle for a paged (decode) problem given as plain arrays."""

    def __init__(self, q, q_scale, k_cache, k_cache_scale, w, block_table, seq_lens, K):
        q = np.asarray(q)
        self.B, self.next_n = q.shape[0], q.shape[1]
        self.qu = e4m3.decode_array_units(q).astype(np.float64)            # [B, nn, H, D]
        kc = np.asarray(k_cache)
        self.ku = e4m3.decode_array_units(kc.reshape(-1, kc.shape[-1])).astype(np.float64)
        self.ks = np.asarray(k_cache_scale, np.float32).reshape(-1)
        self.q_scale = np.asarray(q_scale, np.float32)
        self.w = np.asarray(w, np.float32)
        self.bt = np.asarray(block_table, np.int64)
        self.seq_lens = np.asarray(seq_lens, np.int64)
        self.K = int(K)

    @classmethod
    def from_inputs(cls, inp):
        return cls(inp.q, inp.q_scale, inp.k_cache, inp.k_cache_scale, inp.w,
                   inp.block_table, inp.seq_lens, inp.K)

    def row_length(self, b: int, i: int) -> int:
        return max(0, int(self.seq_lens[b]) - self.next_n + i + 1)

    def row_slots(self, b: int, i: int) -> np.ndarray:
        """Physical slots of logical keys 0..L-1 of row (b, i), in logical order."""
        s = np.arange(self.row_length(b, i), dtype=np.int64)
        return self.bt[b, s // PAGE] * PAGE + s % PAGE

    def row_scores(self, b: int, i: int):
        slots = self.row_slots(b, i)
        if len(slots) == 0:
            return slots, np.zeros(0), np.zeros(0)
        dots = exact_dots(self.qu[b, i], self.ku[slots])
        I, E = combine_heads(dots, self.w[b, i], self.q_scale[b, i], self.ks[slots])
        return slots, I, E

    def topk(self, b: int, i: int):
        slots, I, E = self.row_scores(b, i)
        logical = np.arange(len(slots), dtype=np.int64)
        out, kth = topk_by_sort(slots, I, self.K, order_key=logical)
        return out, slots, I, E, kth


# ---------------------------------------------------------------------------
# Row-parallel driver (spawned worker processes, one BLAS thread each), used
# by the tests for larger cases and by the bench's CPU-baseline leg.
# ---------------------------------------------------------------------------
_WORKER = {}


def _init_worker(kind, arrays):
    _WORKER["o"] = DenseOracle(*arrays) if kind == "dense" else PagedOracle(*arrays)


def _dense_task(t):
    out, ids, I, E, kth = _WORKER["o"].topk(t)
    return t, out


def _paged_task(bi):
    out, *_ = _WORKER["o"].topk(*bi)
    return bi, out


class OraclePool:
    """A pool of `procs` spawned worker processes, each holding one oracle of
    the same problem (decoded once) and running single-threaded BLAS, so the
    pool uses exactly `procs` cores.  Use as a context manager."""

    def __init__(self, inp, procs: int, kind: str = "dense"):
        import multiprocessing as mp
        import os
        self.kind = kind
        if kind == "dense":
            arrays = (inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin, inp.row_end, inp.K)
        else:
            arrays = (inp.q, inp.q_scale, inp.k_cache, inp.k_cache_scale, inp.w, inp.block_table,
                      inp.seq_lens, inp.K)
        saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                                 "MKL_NUM_THREADS")}
        for v in saved:
            os.environ[v] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(procs, initializer=_init_worker,
                                                     initargs=(kind, arrays))
            # make every worker finish its initialiser before timing starts
            self.pool.map(_noop, range(procs), chunksize=1)
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
        self.procs = procs

    def topk(self, rows):
        task = _dense_task if self.kind == "dense" else _paged_task
        return dict(self.pool.map(task, list(rows), chunksize=1))

    def close(self):
        self.pool.terminate()
        self.pool.join()

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def _noop(i):
    import time
    time.sleep(0.2)
    return i


def parallel_topk(inp, rows, procs: int, kind: str = "dense"):
    """Oracle top-K of `rows` using `procs` spawned processes.

    Returns {row: out[K]}.  Each worker runs single-threaded BLAS, so `procs`
    is the number of cores used.
    """
    import multiprocessing as mp
    import os
    if kind == "dense":
        arrays = (inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin, inp.row_end, inp.K)
        task = _dense_task
    else:
        arrays = (inp.q, inp.q_scale, inp.k_cache, inp.k_cache_scale, inp.w, inp.block_table,
                  inp.seq_lens, inp.K)
        task = _paged_task
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                             "MKL_NUM_THREADS")}
    for v in saved:
        os.environ[v] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(procs, initializer=_init_worker, initargs=(kind, arrays)) as pool:
            res = dict(pool.map(task, list(rows), chunksize=1))
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    return res
