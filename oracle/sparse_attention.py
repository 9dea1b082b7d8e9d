"""Sparse-attention decode over the indexer's top-K indices (test
infrastructure only: the oracle of the CUDA sparse-attention kernel).

Definition followed (contest write-up, "DSA Sparse Attention" paragraph): for
each query token t and head h,

  1. gather the KV entries named by the token's sparse index list (the top-K
     physical cache slots the indexer returned; -1 entries are padding and
     take no part);
  2. logits  z_j = q_nope[t, h] . ckv[i_j] + q_pe[t, h] . kpe[i_j], scaled by
     sm_scale;
  3. a base-2 softmax: u_j = z_j * sm_scale * log2(e),
     p_j = 2^(u_j - max u) / sum_k 2^(u_k - max u)
     (the same weights as a natural-base softmax of z_j * sm_scale);
  4. out[t, h] = sum_j p_j ckv[i_j]  (the 512-dim compressed KV), and
     lse[t, h] = log2(sum_j 2^(u_j)), the log-sum-exp in the base-2 domain
     of step 3.

A token with no valid index gets out = 0 and lse = -inf.  Inputs are bf16
values (passed as float arrays holding them), everything here is float64.

Readings where the write-up is silent: the dimensions (512-dim ckv, 64-dim
rope part, heads per token) are DeepSeek-V3.2's; the LSE is returned in
base 2, in the domain of the base-2 softmax; the index list is used as given
(an index listed twice would count twice; the indexer never lists one twice).
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


def attend_one(q_nope, q_pe, ckv, kpe, idx, sm_scale):
    """(out [Dc], lse, P [L], V [L, Dc]) of one (token, head): q_nope [Dc],
    q_pe [Dp], ckv [S, Dc], kpe [S, Dp], idx [K] int (negative = padding).
    P are the softmax weights of the valid indices in list order."""
    sel = np.asarray(idx, np.int64)
    sel = sel[sel >= 0]
    dc = ckv.shape[1]
    if len(sel) == 0:
        return np.zeros(dc), -math.inf, np.zeros(0), np.zeros((0, dc))
    V = ckv[sel].astype(np.float64)
    Kp = kpe[sel].astype(np.float64)
    z = V @ np.asarray(q_nope, np.float64) + Kp @ np.asarray(q_pe, np.float64)
    u = z * float(sm_scale) * LOG2E
    m = u.max()
    e = np.exp2(u - m)
    s = e.sum()
    P = e / s
    return P @ V, m + math.log2(s), P, V


def sparse_attention(q_nope, q_pe, ckv, kpe, indices, sm_scale):
    """out [T, H, Dc], lse [T, H] for q_nope [T, H, Dc], q_pe [T, H, Dp],
    ckv [S, Dc], kpe [S, Dp] (S cache slots), indices [T, K]."""
    T, H, dc = q_nope.shape
    out = np.zeros((T, H, dc))
    lse = np.zeros((T, H))
    for t in range(T):
        for h in range(H):
            o, l, _, _ = attend_one(q_nope[t, h], q_pe[t, h], ckv, kpe, indices[t], sm_scale)
            out[t, h] = o
            lse[t, h] = l
    return out, lse


def magnitude(q_nope, q_pe, ckv, kpe, idx, sm_scale):
    """M [Dc] = sum_j p_j |ckv[i_j]| of one (token, head): the scale the output
    tolerance is relative to (a kernel that rounds the weights p_j and the
    output to bf16 errs by a few bf16 units of M)."""
    _, _, P, V = attend_one(q_nope, q_pe, ckv, kpe, idx, sm_scale)
    return P @ np.abs(V) if len(P) else np.zeros(ckv.shape[1])
