"""Shared test helpers: device upload and oracle comparison of whole outputs."""
import os

import numpy as np

from oracle import checks, indexer


def to_dev(*arrays):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def dense_args(inp):
    return to_dev(inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin, inp.row_end)


def paged_args(inp):
    return to_dev(inp.q, inp.q_scale, inp.k_cache, inp.k_cache_scale, inp.w, inp.block_table, inp.seq_lens)


def procs():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def check_dense_rows(inp, out, rows, elementwise=True, oracle=None):
    """Problems per failing row (dict row -> list); empty dict = pass."""
    o = oracle or indexer.DenseOracle.from_inputs(inp)
    out = np.asarray(out)
    bad = {}
    for t in rows:
        ids, I, E = o.row_scores(t)
        pr = checks.check_row(out[t], ids, I, E, inp.K, elementwise=elementwise)
        if pr:
            bad[t] = pr
    return bad


# worker-side checker for big cases: each spawned worker holds one oracle
_W = {}


def _init(arrays, kind):
    _W["o"] = indexer.DenseOracle(*arrays) if kind == "dense" else indexer.PagedOracle(*arrays)
    _W["kind"] = kind


def _check_task(args):
    key, out_row, K, elementwise = args
    o = _W["o"]
    if _W["kind"] == "dense":
        ids, I, E = o.row_scores(key)
        return key, checks.check_row(out_row, ids, I, E, K, elementwise=elementwise)
    slots, I, E = o.row_scores(*key)
    return key, checks.check_row(out_row, slots, I, E, K, elementwise=elementwise,
                                 order_key=np.arange(len(slots)))


def check_rows_parallel(inp, out, keys, kind="dense", elementwise=True):
    """Oracle check of many rows of a large case in spawned processes."""
    import multiprocessing as mp
    if kind == "dense":
        # only the checked rows' q/w/ranges go to the workers (all keys kept)
        keys = list(keys)
        r = np.asarray(keys, dtype=np.int64)
        arrays = (inp.q[r], inp.q_scale[r], inp.k, inp.k_scale, inp.w[r], inp.row_begin[r], inp.row_end[r],
                  inp.K)
        rows = [(i, np.asarray(out[t]), inp.K, elementwise) for i, t in enumerate(keys)]
    else:
        arrays = (inp.q, inp.q_scale, inp.k_cache, inp.k_cache_scale, inp.w, inp.block_table,
                  inp.seq_lens, inp.K)
        rows = [(k, np.asarray(out[k[0], k[1]]), inp.K, elementwise) for k in keys]
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in saved:
        os.environ[v] = "1"
    try:
        with mp.get_context("spawn").Pool(procs(), initializer=_init, initargs=(arrays, kind)) as pool:
            res = pool.map(_check_task, rows, chunksize=1)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    if kind == "dense":
        return {keys[i]: p for i, p in res if p}
    return {k: p for k, p in res if p}
