"""Parity criteria between a selection under test and the oracle (test
infrastructure only).

Exactness as defined in "Fusing Indexer Scoring and Exact Top-k for
DeepSeek-V3.2", section 2.3: indices lie in the valid range and are unique; the
K selected scores, sorted, equal the true top-K scores element by element;
ties may go to any valid index.  A float32 implementation is held to that
within a tolerance relative to E[s] = sum_j |w_j| |q_j . k_s| (dequantised):

  (i)   bit-exact: min(L, K) entries, all valid and distinct, then -1 padding;
  (ii)  every selected s has I[s] >= theta - TOL * E[s] (theta = K-th score);
  (iii) optionally, the selected scores sorted descending equal the oracle's
        sorted top-K element-wise within TOL * max(E_a, E_b).
"""
from __future__ import annotations

import numpy as np

TOL = 1e-5


def check_row(out_row, ids, I, E, K: int, elementwise: bool = True, tol: float = TOL,
              order_key=None) -> list[str]:
    """Problems found in one row's output (empty list = pass).

    out_row: the K int32 outputs under test.  ids/I/E: the row's valid ids and
    their oracle scores and tolerance scales (from DenseOracle/PagedOracle).
    """
    out = np.asarray(out_row, np.int64).reshape(-1)
    ids = np.asarray(ids, np.int64)
    L = len(ids)
    n = min(L, K)
    probs = []
    if out.shape[0] != K:
        return [f"output has {out.shape[0]} entries, expected {K}"]
    head, tail = out[:n], out[n:]
    if (tail != -1).any():
        probs.append(f"{int((tail != -1).sum())} non-padding entries after the first {n}")
    if n == 0:
        return probs
    sorter = np.argsort(ids, kind="stable")
    sids = ids[sorter]
    loc = np.clip(np.searchsorted(sids, head), 0, L - 1)
    found = sids[loc] == head
    if not found.all():
        bad = head[~found][:5]
        probs.append(f"{int((~found).sum())} indices outside the valid set, e.g. {bad.tolist()}")
        return probs
    if len(np.unique(head)) != n:
        probs.append(f"{n - len(np.unique(head))} duplicate indices")
        return probs
    if L <= K:
        return probs  # all valid ids, distinct, count L: the set is exact
    pos = sorter[loc]
    sec = ids if order_key is None else order_key
    order = np.lexsort((sec, -I))
    theta = I[order[K - 1]]
    sel_I, sel_E = I[pos], E[pos]
    low = sel_I < theta - tol * sel_E
    if low.any():
        j = np.argmax(theta - sel_I - tol * sel_E)
        probs.append(f"{int(low.sum())} selected below theta-tol*E; worst id {int(head[j])} "
                     f"I={sel_I[j]!r} theta={theta!r} E={sel_E[j]!r}")
    if elementwise:
        ao = np.argsort(-sel_I, kind="stable")
        a, ea = sel_I[ao], sel_E[ao]
        b, eb = I[order[:K]], E[order[:K]]
        diff = np.abs(a - b) > tol * np.maximum(ea, eb)
        if diff.any():
            j = int(np.argmax(diff))
            probs.append(f"{int(diff.sum())} sorted scores differ; first at rank {j}: "
                         f"{a[j]!r} vs {b[j]!r}")
    return probs
