"""GPU parity of the sparse-attention decode (dsa_sparse_attention) against
the float64 oracle (contest write-up, "DSA Sparse Attention").

Tolerance, from the kernel's arithmetic: bf16 inputs are multiplied exactly
and accumulated in fp32; the softmax weights are rounded to bf16 (relative
2^-9) for the weighted sum and the output to bf16 (2^-9); the fp32 logits
err by at most ~2^-10 in the weights.  Every output element must lie within
2^-7 * M of the oracle's, with M = sum_j p_j |ckv[i_j]| at that element, and
the base-2 LSE within 2^-7 (its sum of weights uses the rounded weights)."""
import numpy as np
import pytest

from fp8_scoring_exact_gb300 import synthetic as S
from oracle import sparse_attention as sa

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -7


@pytest.fixture(scope="module")
def B():
    from fp8_scoring_exact_gb300 import binding
    binding.lib()
    return binding


def _run(B, inp):
    import torch
    dev = [x.cuda() for x in (inp.q_nope, inp.q_pe, inp.ckv, inp.kpe)]
    idx = torch.from_numpy(inp.indices).cuda()
    out, lse = B.sparse_attention(*dev, idx, inp.sm_scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(inp, out, lse, tokens=None):
    qn = inp.q_nope.double().numpy()
    qp = inp.q_pe.double().numpy()
    ckv = inp.ckv.double().numpy()
    kpe = inp.kpe.double().numpy()
    for t in (range(inp.T) if tokens is None else tokens):
        for h in range(inp.H):
            o, l, P, V = sa.attend_one(qn[t, h], qp[t, h], ckv, kpe, inp.indices[t], inp.sm_scale)
            if len(P) == 0:
                assert np.all(out[t, h] == 0) and lse[t, h] == -np.inf, (t, h)
                continue
            M = P @ np.abs(V)
            err = np.abs(out[t, h] - o)
            assert np.all(err <= TOL * M + 1e-6), (t, h, float(np.max(err / (M + 1e-30))))
            assert abs(lse[t, h] - l) <= TOL, (t, h, float(lse[t, h]), l)


@pytest.mark.parametrize("T,H,K,S_", [(12, 16, 512, 5000), (12, 32, 2048, 9000), (1, 16, 2048, 4000),
                                      (300, 16, 128, 3000)])
def test_sparse_attention_matches_oracle(B, T, H, K, S_):
    """Several split counts (one token: many splits; 300 tokens: one split),
    ragged and empty index lists, 16 and 32 heads."""
    rng = np.random.default_rng(T + H + K)
    n_valid = rng.integers(1, min(K, S_) + 1, T)
    n_valid[0] = 0 if T > 1 else n_valid[0]     # a token with no valid slot
    if T > 2:
        n_valid[1] = 1                           # a single slot
        n_valid[2] = min(K, S_)                  # a full list
    inp = S.make_sparse_attention(T, H, S_, K, seed=T * 7 + K, n_valid=n_valid)
    out, lse = _run(B, inp)
    assert B.sparse_attention_last_status() == 0
    _check(inp, out, lse, tokens=range(min(T, 40)))


def test_sparse_attention_over_the_paged_indexer_result(B):
    """The indexer's paged result (physical slots of a 64-token-page cache) fed
    straight to the sparse attention over a cache with the same page layout."""
    import torch
    ip = S.make_paged(5, 2, K=512, seed=91, len_lo=200, len_hi=6000, n_short=1, short_hi=400)
    from helpers import paged_args
    idx = B.indexer_topk_paged(*paged_args(ip), K=ip.K)
    rc, _ = B.last_device_status()
    assert rc == 0
    indices = idx.reshape(-1, ip.K).cpu().numpy()
    slots = ip.k_cache.shape[0] * 64
    inp = S.make_sparse_attention(indices.shape[0], 16, slots, ip.K, seed=92, indices=indices)
    out, lse = _run(B, inp)
    assert B.sparse_attention_last_status() == 0
    _check(inp, out, lse)


def test_sparse_attention_reports_slots_outside_the_cache(B):
    inp = S.make_sparse_attention(3, 16, 1000, 64, seed=93)
    inp.indices[1, 5] = 1000 + 17                # past the cache: read as padding, reported
    out, lse = _run(B, inp)
    assert B.sparse_attention_last_status() == B.DSA_ERR_RANGE
    inp.indices[1, 5] = -1
    _check(inp, out, lse)


def test_sparse_attention_replays_from_a_cuda_graph(B):
    """The call enqueues a status reset and kernels only (its scratch sized by
    a first call), so it can be captured once and replayed on new inputs
    copied into the captured buffers."""
    import torch
    a = S.make_sparse_attention(6, 16, 3000, 512, seed=94)
    b = S.make_sparse_attention(6, 16, 3000, 512, seed=95)
    dev = [x.cuda() for x in (a.q_nope, a.q_pe, a.ckv, a.kpe)]
    idx = torch.from_numpy(a.indices).cuda()
    out = torch.empty((a.T, a.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((a.T, a.H), dtype=torch.float32, device="cuda")
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        B.sparse_attention(*dev, idx, a.sm_scale, out=out, lse=lse)  # sizes this stream's scratch
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        B.sparse_attention(*dev, idx, a.sm_scale, out=out, lse=lse)
    for d, h in zip(dev, (b.q_nope, b.q_pe, b.ckv, b.kpe)):
        d.copy_(h.cuda())
    idx.copy_(torch.from_numpy(b.indices).cuda())
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert B.sparse_attention_last_status(gs) == 0
    _check(b, out.float().cpu().numpy(), lse.cpu().numpy())
