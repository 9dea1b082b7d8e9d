"""The entry point that allocates nothing (dsa_indexer_topk_from_scores_noalloc)
must return the exact top-K of each score row, and what the allocating entry
point (dsa_indexer_topk_from_scores) returns, call after call.

It exists for callers that cannot call cudaMalloc (runtimes that own all
device memory, such as a serving engine that reserves the free memory for its
KV cache at start-up, or plugin hosts with a fixed budget); its scratch is a fixed
array in device memory shared by every call, so two calls in a row also check
that each call resets what it reads.  Selection from given fp32 scores is
exact: up to ties, the sorted selected scores must equal a full sort of the
row bit for bit.

Besides random rows, each case holds rows built to take every branch of the
kernel behind this entry point: a threshold that leaves fewer than K
candidates and whose relaxed retry falls outside the sample (every key then
passes), rows where every threshold admits more candidates than fit (massive
ties: the full-row radix select), rows of exactly K and fewer than K keys, an
empty row, and -0 / +0 ties.
"""
import numpy as np
import pytest

from helpers import to_dev

pytestmark = pytest.mark.gpu

SAMPLE_STRIDE, SAMPLE_OFFSET = 200, 100   # the sampled-threshold grid (one key in 200)


def _grid(b, e):
    """Positions of the sample grid inside [b, e) (keys 100 mod 200)."""
    first = b + (SAMPLE_OFFSET - b) % SAMPLE_STRIDE
    return np.arange(first, e, SAMPLE_STRIDE)


def _case(seed, Q, N, K):
    rng = np.random.default_rng(seed)
    sc = rng.standard_normal((Q, N)).astype(np.float32)
    sc[1] = np.round(sc[1] * 3) / 3          # heavy ties
    sc[2] = 0.0
    sc[2, ::3] = -0.0                         # -0 and +0 tie
    rb = rng.integers(0, 500, Q).astype(np.int32)
    re = np.minimum(rb + rng.integers(0, N, Q), N).astype(np.int32)
    re[3] = rb[3] + K                         # exactly K valid keys
    re[4] = rb[4] + 7                         # fewer than K
    re[5] = rb[5]                             # empty
    # underflow, then a relaxed rank past the sample: the grid keys outscore
    # every other key, so the first threshold (a grid key of rank about
    # m * 2K / L) admits only that many keys; four times that rank exceeds
    # the m grid keys, so the retry threshold is "every key" (L = 4K: m = 40
    # grid keys, rank 21 then 84 > 40)
    rb[6], re[6] = 123, 123 + 4 * K
    sc[6, _grid(rb[6], re[6])] = 100.0 + np.arange(len(_grid(rb[6], re[6])), dtype=np.float32)
    # every key equal: each threshold admits the whole row, which is longer
    # than the selector keeps (overflow at every retry, then the full-row
    # radix select); and a two-valued row
    rb[7], re[7] = 0, N
    sc[7] = 1.5
    rb[8], re[8] = 11, N - 3
    sc[8] = rng.choice(np.float32([-1.0, 2.0]), N)
    return sc, rb, re


def _check_exact(sc, rb, re, K, out):
    """Valid, distinct, min(L, K) indices then -1 padding; the sorted selected
    scores equal the full sort of the row's valid scores, bit for bit."""
    for t in range(sc.shape[0]):
        L = max(int(re[t] - rb[t]), 0)
        n = min(L, K)
        assert (out[t, n:] == -1).all(), t
        sel = out[t, :n]
        assert len(np.unique(sel)) == n and np.all((sel >= rb[t]) & (sel < re[t])), t
        want = np.sort(sc[t, rb[t]:re[t]])[::-1][:n]
        got = np.sort(sc[t, sel])[::-1]
        assert np.array_equal(got, want), t


def test_noalloc_is_exact_and_matches_allocating_entry_on_two_calls_in_a_row():
    import torch

    from fp8_scoring_exact_gb300 import binding as B
    B.lib()
    for call, (seed, Q, N, K) in enumerate([(31, 24, 30000, 2048), (32, 40, 9000, 512)]):
        sc, rb, re = _case(seed, Q, N, K)
        d_sc, d_rb, d_re = to_dev(sc, rb, re)
        ref = B.topk_from_scores(d_sc, d_rb, d_re, K=K).cpu().numpy()
        out = torch.full((Q, K), -7, dtype=torch.int32, device="cuda")
        B.topk_from_scores_noalloc(d_sc, d_rb, d_re, K=K, out=out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        _check_exact(sc, rb, re, K, got)
        _check_exact(sc, rb, re, K, ref)


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    import torch

    from fp8_scoring_exact_gb300 import binding as B
    Q = 4097
    sc = torch.zeros((Q, 64), dtype=torch.float32, device="cuda")
    rb = torch.zeros(Q, dtype=torch.int32, device="cuda")
    re = torch.full((Q,), 64, dtype=torch.int32, device="cuda")
    with pytest.raises(B.IndexerError) as e:
        B.topk_from_scores_noalloc(sc, rb, re, K=16)
    assert e.value.code == B.DSA_ERR_UNSUPPORTED
