"""The entry point that allocates nothing (dsa_indexer_topk_from_scores_noalloc)
must return what the allocating entry point (dsa_indexer_topk_from_scores)
returns, call after call.

It exists for callers that cannot call cudaMalloc (runtimes that own all
device memory, such as a serving engine that reserves the free memory for its
KV cache at start-up, or plugin hosts with a fixed budget); its scratch is a fixed
array in device memory shared by every call, so two calls in a row also check
that each call resets what it reads.  Selection from given fp32 scores is
exact: up to ties, the sorted selected scores must be identical.
"""
import numpy as np
import pytest

from helpers import to_dev

pytestmark = pytest.mark.gpu


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
    return sc, rb, re


def _same_selection(sc, rb, re, K, a, b):
    for t in range(sc.shape[0]):
        n = min(max(int(re[t] - rb[t]), 0), K)
        assert (a[t, n:] == -1).all() and (b[t, n:] == -1).all(), t
        for out in (a, b):
            sel = out[t, :n]
            assert len(np.unique(sel)) == n and np.all((sel >= rb[t]) & (sel < re[t])), t
        assert np.array_equal(np.sort(sc[t, a[t, :n]]), np.sort(sc[t, b[t, :n]])), t


def test_noalloc_matches_allocating_entry_on_two_calls_in_a_row():
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
        _same_selection(sc, rb, re, K, out.cpu().numpy(), ref)


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
