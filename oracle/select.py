"""Plain restatement of the method's exact selection steps (test infrastructure).

"Fusing Indexer Scoring and Exact Top-k for DeepSeek-V3.2", section 3.2:

  1. estimate a threshold tau from a ~0.5% sample spread across the row,
     aiming at about 2K candidates;
  2. compare-and-append: keep every (score, index) with score >= tau;
  3. four 8-bit radix passes, most significant byte first, over
     order-preserving 32-bit keys find the exact K-th largest value theta and
     the number r of theta-equal elements still to take; emit every element
     above theta and r elements equal to it;
  certificate: if the candidate set is complete and K <= |C| <= capacity,
  TopK(row) = TopK(C); otherwise (underflow or overflow) the row is repaired
  exactly.

These functions are slow, obvious Python/numpy used to pin that logic against
a full sort in the tests.  The sample grid and constants are the readings
stated in the design notes: one sample every 200 keys (0.5%), target 2K.
"""
from __future__ import annotations

import math

import numpy as np

SAMPLE_STRIDE = 200
SAMPLE_OFFSET = SAMPLE_STRIDE // 2


def ordered_key(x) -> np.ndarray:
    """Order-preserving map float32 -> uint32 (-0 canonicalised to +0 first).

    Non-negative floats get the sign bit set; negative floats are bit-inverted,
    so unsigned comparison of keys matches float comparison.
    """
    f = np.array(x, dtype=np.float32, copy=True).reshape(-1)
    f[f == 0] = np.float32(0.0)
    b = f.view(np.uint32)
    neg = (b >> np.uint32(31)) != 0
    return np.where(neg, ~b, b | np.uint32(0x80000000)).astype(np.uint32)


def radix_select(keys: np.ndarray, K: int):
    """Four 8-bit passes, MSB first: returns (theta, r) where theta is the
    K-th largest key and r is how many theta-equal keys belong to the top K."""
    keys = np.asarray(keys, np.uint32)
    if not 1 <= K <= len(keys):
        raise ValueError("need 1 <= K <= len(keys)")
    prefix, mask, rem = 0, 0, K
    for shift in (24, 16, 8, 0):
        live = keys[(keys & np.uint32(mask)) == np.uint32(prefix)]
        hist = np.bincount(((live >> np.uint32(shift)) & np.uint32(0xFF)).astype(np.int64),
                           minlength=256)
        above = 0
        digit = 255
        while above + hist[digit] < rem:
            above += hist[digit]
            digit -= 1
        rem -= above
        prefix |= digit << shift
        mask |= 0xFF << shift
    return np.uint32(prefix), int(rem)


def emit(keys: np.ndarray, ids: np.ndarray, theta, r: int) -> np.ndarray:
    """All ids with key > theta, then the first r ids with key == theta."""
    keys = np.asarray(keys, np.uint32)
    above = ids[keys > theta]
    equal = ids[keys == theta][:r]
    return np.concatenate([above, equal])


def sample_positions(b: int, e: int) -> np.ndarray:
    """Sample grid inside [b, e): every key whose index is 100 mod 200."""
    first = b + ((SAMPLE_OFFSET - b) % SAMPLE_STRIDE)
    return np.arange(first, e, SAMPLE_STRIDE, dtype=np.int64)


def sample_rank(m: int, L: int, K: int) -> int:
    """Descending rank of tau among m samples so that about 2K of L keys pass."""
    return int(math.ceil(m * 2 * K / L)) if L > 0 else 0


def sampled_threshold_key(scores_row: np.ndarray, b: int, e: int, K: int) -> int:
    """Key of tau for the row whose valid scores (float32, index b..e-1) are
    given.  0 (every key passes) when the sample cannot reach the target."""
    pos = sample_positions(b, e)
    m, L = len(pos), e - b
    r = sample_rank(m, L, K)
    if m == 0 or r > m or r < 1:
        return 0
    sk = np.sort(ordered_key(scores_row[pos - b]))[::-1]
    return int(sk[r - 1])


def compare_and_append(keys: np.ndarray, ids: np.ndarray, tau_key: int):
    sel = keys >= np.uint32(tau_key)
    return keys[sel], ids[sel]


def certified_topk(scores_row, ids, K: int, tau_key: int, capacity: int):
    """Fast path with certificate.  Returns (status, selected ids or None);
    status is 'ok', 'underflow' or 'overflow'."""
    keys = ordered_key(scores_row)
    ck, ci = compare_and_append(keys, np.asarray(ids), tau_key)
    if len(ck) < K:
        return "underflow", None
    if len(ck) > capacity:
        return "overflow", None
    theta, r = radix_select(ck, K)
    return "ok", emit(ck, ci, theta, r)
