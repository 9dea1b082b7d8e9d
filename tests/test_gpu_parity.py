"""GPU parity: the CUDA library (through its C ABI binding) against the oracle.

Criteria ("Fusing Indexer Scoring and Exact Top-k for DeepSeek-V3.2",
section 2.3, with the float32 tolerance TOL * E of oracle.checks): indices
valid, unique, min(L, K) of them then -1 padding (bit-exact); every selected
score within TOL * E of the oracle's K-th score; on the small cases the sorted
selected scores equal the oracle's element-wise.  Large cases are checked on
seeded row samples plus every row the device sent to repair.
"""
import copy

import numpy as np
import pytest

from fp8_scoring_exact_gb300 import synthetic as S
from oracle import checks, indexer

from helpers import check_dense_rows, check_rows_parallel, dense_args, paged_args, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from fp8_scoring_exact_gb300 import binding
    binding.lib()
    binding.set_option("tau_bias", 0)
    return binding


def _status_ok(B):
    rc, counters = B.last_device_status()
    assert rc == 0, f"device status {B.STATUS_NAMES.get(rc, rc)}"
    return counters


# ------------------------------------------------------------ raw scores ----
@pytest.mark.parametrize("N,causal", [(8192, False), (8192 + 77, True), (300, False)])
def test_scores_match_oracle_elementwise(B, N, causal):
    inp = S.make_dense(8 if N > 300 else 3, N, seed=N, causal=causal)
    sc = B.indexer_scores(*dense_args(inp)).cpu().numpy()
    _status_ok(B)
    o = indexer.DenseOracle.from_inputs(inp)
    for t in range(inp.Q):
        ids, I, E = o.row_scores(t)
        g = sc[t, ids].astype(np.float64)
        assert np.all(np.abs(g - I) <= checks.TOL * E), f"row {t}: max rel {np.max(np.abs(g - I) / E)}"


# ------------------------------------------------------ small full checks ----
@pytest.mark.parametrize("fn", ["fused", "unfused"])
def test_tiny_noncausal_all_rows(B, fn):
    inp = S.make_config(0)
    call = B.indexer_topk if fn == "fused" else B.indexer_topk_unfused
    out = call(*dense_args(inp), K=inp.K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


@pytest.mark.parametrize("fn", ["fused", "unfused"])
@pytest.mark.parametrize("Q,N,K,seed", [(37, 5077, 256, 1), (9, 2049, 2048, 2), (64, 12345, 1024, 3),
                                        (5, 640, 1, 4)])
def test_ragged_causal_all_rows(B, fn, Q, N, K, seed):
    inp = S.make_dense(Q, N, K=K, seed=seed, causal=True)
    call = B.indexer_topk if fn == "fused" else B.indexer_topk_unfused
    out = call(*dense_args(inp), K=K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(Q)) == {}


def test_causal_q2048_n16k_all_rows(B):
    """The 16K causal prefill chunk (shared-direction keys), every row."""
    inp = S.make_config(1)
    out = B.indexer_topk(*dense_args(inp), K=inp.K).cpu().numpy()
    _status_ok(B)
    bad = check_rows_parallel(inp, out, range(inp.Q))
    assert bad == {}, list(bad.items())[:3]


def test_causal_q2048_n16k_units_last_first(B):
    """The persistent scorer hands its work units out from a counter; each
    unit writes only its own candidate regions and count, so handing them out
    in reverse order must give an exact result too (every row)."""
    inp = S.make_config(1)
    B.set_option("unit_order", 1)
    try:
        out = B.indexer_topk(*dense_args(inp), K=inp.K).cpu().numpy()
        counters = _status_ok(B)
    finally:
        B.set_option("unit_order", 0)
    assert counters["underflow"] + counters["overflow"] <= 8
    bad = check_rows_parallel(inp, out, range(inp.Q))
    assert bad == {}, list(bad.items())[:3]


@pytest.mark.parametrize("next_n", [2, 5])
def test_paged_units_last_first(B, next_n):
    """The same for paged rows: groups of at most two rows (two epilogue teams,
    virtual units 2c and 2c + 1) and of four and one rows."""
    inp = S.make_paged(9, next_n, K=512, seed=40 + next_n, len_lo=600, len_hi=30000, n_short=2, short_hi=700)
    B.set_option("unit_order", 1)
    try:
        out = B.indexer_topk_paged(*paged_args(inp), K=inp.K).cpu().numpy()
        _status_ok(B)
    finally:
        B.set_option("unit_order", 0)
    po = indexer.PagedOracle.from_inputs(inp)
    for b in range(inp.B):
        for i in range(inp.next_n):
            slots, I, E = po.row_scores(b, i)
            pr = checks.check_row(out[b, i], slots, I, E, inp.K, order_key=np.arange(len(slots)))
            assert not pr, (b, i, pr)


# ------------------------------------------- small Q, long history; Q8192 ----
@pytest.mark.parametrize("Q", [8, 64, 152])
def test_small_q_long_history_all_rows(B, Q):
    """Fewer query rows than SMs (or about as many) over a 128K-key causal
    history: the key dimension is split into work units that all SMs share,
    and every row is exact."""
    inp = S.make_dense(Q, 131072, K=2048, seed=80 + Q)
    out = B.indexer_topk(*dense_args(inp), K=inp.K).cpu().numpy()
    _status_ok(B)
    bad = check_rows_parallel(inp, out, range(Q))
    assert bad == {}, list(bad.items())[:3]


def test_q8192_chunk_sampled_and_repaired_rows(B):
    """An 8192-row prefill chunk over 128K keys (twice the headline rows):
    64 seeded rows, the first, middle and last rows, and every repaired row."""
    inp = S.make_dense(8192, 131072, K=2048, seed=88)
    out = B.indexer_topk(*dense_args(inp), K=inp.K).cpu().numpy()
    counters = _status_ok(B)
    repaired = B.last_repaired_rows()
    assert len(repaired) == counters["underflow"] + counters["overflow"]
    rows = sorted(set(_sampled_rows(inp.Q, 64, 188)) | set(repaired))
    bad = check_rows_parallel(inp, out, rows)
    assert bad == {}, list(bad.items())[:3]


# ------------------------------------------------- full-size sampled rows ----
def _sampled_rows(Q, n, seed):
    rng = np.random.default_rng(seed)
    return sorted(set(rng.choice(Q, size=n, replace=False).tolist()) | {0, Q // 2, Q - 1})


@pytest.mark.parametrize("cid", [2, 3])
def test_full_size_sampled_rows_and_repaired_rows(B, cid):
    inp = S.make_config(cid)
    args = dense_args(inp)
    out = B.indexer_topk(*args, K=inp.K).cpu().numpy()
    counters = _status_ok(B)
    repaired = B.last_repaired_rows()
    assert len(repaired) == counters["underflow"] + counters["overflow"]
    if cid == 3:
        assert len(repaired) > 0, "the tie-stress workload is built to exercise repair"
    rows = sorted(set(_sampled_rows(inp.Q, 64, 100 + cid)) | set(repaired))
    bad = check_rows_parallel(inp, out, rows)
    assert bad == {}, list(bad.items())[:3]
    # the unfused pipeline must select the same scores on the sampled rows
    out_u = B.indexer_topk_unfused(*args, K=inp.K).cpu().numpy()
    _status_ok(B)
    bad = check_rows_parallel(inp, out_u, _sampled_rows(inp.Q, 16, 200 + cid))
    assert bad == {}, list(bad.items())[:3]


def test_paged_decode_batch_all_rows(B):
    inp = S.make_config(4)
    out = B.indexer_topk_paged(*paged_args(inp), K=inp.K).cpu().numpy()
    counters = _status_ok(B)
    L = inp.row_lengths()
    assert counters["trivial"] == int((L <= inp.K).sum())
    keys = [(b, i) for b in range(inp.B) for i in range(inp.next_n)]
    bad = check_rows_parallel(inp, out, keys, kind="paged")
    assert bad == {}, list(bad.items())[:3]


# ------------------------------------------------------------------ paged ----
@pytest.mark.parametrize("next_n", [1, 2, 3, 5])
def test_paged_small_all_rows(B, next_n):
    inp = S.make_paged(7, next_n, K=300, seed=10 + next_n, len_lo=1, len_hi=5000, n_short=3, short_hi=310)
    # a sequence shorter than next_n and one ending exactly on a page boundary
    inp.seq_lens[0] = max(0, next_n - 1)
    inp.seq_lens[1] = min(64 * int((inp.block_table[1] >= 0).sum()), 4096)
    out = B.indexer_topk_paged(*paged_args(inp), K=inp.K).cpu().numpy()
    _status_ok(B)
    po = indexer.PagedOracle.from_inputs(inp)
    for b in range(inp.B):
        for i in range(inp.next_n):
            slots, I, E = po.row_scores(b, i)
            pr = checks.check_row(out[b, i], slots, I, E, inp.K, order_key=np.arange(len(slots)))
            assert not pr, (b, i, pr)


def test_paged_bad_block_table_entries_report_range(B):
    """A used block-table entry outside [0, num_pages) is reported through the
    device status (DSA_ERR_RANGE) and never followed: one negative entry in
    a sequence whose rows are scored, one past the cache in a sequence whose
    rows take the remapping path (L <= K).  The other sequences stay exact."""
    inp = S.make_paged(6, 2, K=512, seed=71, len_lo=3000, len_hi=9000, n_short=0)
    P = inp.k_cache.shape[0]
    inp.seq_lens[1] = 300                        # remapping path (L <= K)
    inp.block_table[0, 3] = -5                   # inside sequence 0's 3000+ keys
    inp.block_table[1, 2] = P + 7                # inside sequence 1's 300 keys
    out = B.indexer_topk_paged(*paged_args(inp), K=inp.K).cpu().numpy()
    rc, _ = B.last_device_status()
    assert rc == B.DSA_ERR_RANGE
    po = indexer.PagedOracle.from_inputs(inp)
    for b in range(2, inp.B):
        for i in range(inp.next_n):
            slots, I, E = po.row_scores(b, i)
            pr = checks.check_row(out[b, i], slots, I, E, inp.K, order_key=np.arange(len(slots)))
            assert not pr, (b, i, pr)
    # the same batch with a valid table is clean
    good = S.make_paged(6, 2, K=512, seed=71, len_lo=3000, len_hi=9000, n_short=0)
    good.seq_lens[1] = 300
    B.indexer_topk_paged(*paged_args(good), K=good.K)
    _status_ok(B)


# ------------------------------------------------------- bounded waits ----
def test_bounded_wait_runs_out_and_the_next_call_is_exact(B):
    """Every pipeline wait inside the kernels is bounded.  With a test option
    the main scorer never signals its first accumulator, so its epilogue's
    wait (limit 50 ms here) runs out: the kernel lets the copies and MMAs it
    issued land, returns early, and the call reports DSA_ERR_TIMEOUT.  The
    context stays usable: the next call is exact."""
    inp = S.make_dense(16, 20000, K=512, seed=61, causal=True)
    args = dense_args(inp)
    B.set_option("wait_limit_us", 50000)
    B.set_option("test_withhold", 1)
    try:
        B.indexer_topk(*args, K=inp.K)
        rc, _ = B.last_device_status()
    finally:
        B.set_option("test_withhold", 0)
        B.set_option("wait_limit_us", 2000000)
    assert rc == B.DSA_ERR_TIMEOUT
    out = B.indexer_topk(*args, K=inp.K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


def test_math_control_runs_the_main_plan(B):
    """The math-only control (a measurement entry point) runs the fused call's
    main scorer without its score reduction and filter: it completes with a
    clean status and a finite checksum, and leaves the fused call exact."""
    import torch
    inp = S.make_dense(16, 20000, K=512, seed=62, causal=True)
    args = dense_args(inp)
    cs = B.math_control(*args, K=inp.K)
    torch.cuda.synchronize()
    _status_ok(B)
    assert np.isfinite(cs.item())
    out = B.indexer_topk(*args, K=inp.K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


# ----------------------------------------------------------------- repair ----
@pytest.mark.parametrize("bias,kind", [(1 << 31, "underflow"), (-(1 << 33), "overflow")])
def test_forced_repair_is_exact(B, bias, kind):
    """Threshold pushed to the top (every row underflows) or to zero (every
    row's candidate set overflows): all rows go through exact repair."""
    inp = S.make_dense(12, 20000, K=2048, seed=21, causal=True)
    B.set_option("tau_bias", bias)
    try:
        out = B.indexer_topk(*dense_args(inp), K=inp.K).cpu().numpy()
        counters = _status_ok(B)
    finally:
        B.set_option("tau_bias", 0)
    assert counters[kind] == inp.Q
    assert sorted(B.last_repaired_rows()) == list(range(inp.Q))
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


@pytest.mark.parametrize("bias,kind", [(1 << 31, "underflow"), (-(1 << 33), "overflow")])
def test_forced_repair_paged_is_exact(B, bias, kind):
    """The same for paged decode rows: groups of one and two rows (whose
    epilogue runs as two teams on alternate tiles) and of four rows, all
    through exact repair over the physical slots.  Every row is longer than
    the 16384 candidate slots of a row, so a zero threshold overflows it."""
    inp = S.make_paged(6, 5, K=256, seed=33, len_lo=17000, len_hi=30000, n_short=0)
    B.set_option("tau_bias", bias)
    try:
        out = B.indexer_topk_paged(*paged_args(inp), K=inp.K).cpu().numpy()
        counters = _status_ok(B)
    finally:
        B.set_option("tau_bias", 0)
    assert counters[kind] == inp.B * inp.next_n
    po = indexer.PagedOracle.from_inputs(inp)
    for b in range(inp.B):
        for i in range(inp.next_n):
            slots, I, E = po.row_scores(b, i)
            pr = checks.check_row(out[b, i], slots, I, E, inp.K, order_key=np.arange(len(slots)))
            assert not pr, (b, i, pr)


# ---------------------------------------------------- host-buffer entry ----
@pytest.mark.parametrize("chunk_rows,pinned", [(0, True), (16, True), (12, False)])
def test_host_buffer_entry_matches_device_entry(B, chunk_rows, pinned):
    """dsa_indexer_topk_host (host arrays in and out, row chunks pipelined over
    the library's copy stream) returns what the device entry returns: the
    chunks (16 or 12 rows of 45, a ragged last chunk; one chunk by default)
    are independent rows, and the selection is exact."""
    import torch
    inp = S.make_dense(45, 9000, K=512, seed=21, causal=True)
    host = [torch.from_numpy(np.ascontiguousarray(a)) for a in
            (inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin, inp.row_end)]
    if pinned:
        host = [t.pin_memory() for t in host]
    B.set_option("host_chunk_rows", chunk_rows)
    try:
        for _ in range(2):  # the staging is reused on the second call
            out = B.indexer_topk_host(*host, K=inp.K).numpy()
            assert check_dense_rows(inp, out, range(inp.Q)) == {}
    finally:
        B.set_option("host_chunk_rows", 0)
    ref = B.indexer_topk(*dense_args(inp), K=inp.K).cpu().numpy()
    o = indexer.DenseOracle.from_inputs(inp)
    for t in range(inp.Q):
        ids, I, _ = o.row_scores(t)
        pos = {int(s): i for i, s in enumerate(ids)}
        a = np.sort([I[pos[int(s)]] for s in out[t] if s >= 0])
        b = np.sort([I[pos[int(s)]] for s in ref[t] if s >= 0])
        assert np.array_equal(a, b), t


def test_host_buffer_entry_reports_bad_ranges(B):
    import torch
    inp = S.make_dense(20, 700, K=16, seed=22, causal=False)
    inp.row_begin[13], inp.row_end[13] = 10, 701     # end past N, in the second chunk
    host = [torch.from_numpy(np.ascontiguousarray(a)) for a in
            (inp.q, inp.q_scale, inp.k, inp.k_scale, inp.w, inp.row_begin, inp.row_end)]
    B.set_option("host_chunk_rows", 8)
    try:
        with pytest.raises(B.IndexerError) as e:
            B.indexer_topk_host(*host, K=16)
    finally:
        B.set_option("host_chunk_rows", 0)
    assert e.value.code == B.DSA_ERR_RANGE


# ------------------------------------------------------------- edge cases ----
def test_edge_ranges(B):
    """Empty rows, L = K, L = K + 1, offset ranges, a single key."""
    K = 64
    inp = S.make_dense(8, 1000, K=K, seed=5, causal=False)
    inp.row_begin[:] = [0, 10, 100, 0, 999, 500, 3, 0]
    inp.row_end[:] = [0, 10 + K, 101 + K, 1000, 1000, 500, 900, 1]
    for fn in (B.indexer_topk, B.indexer_topk_unfused):
        out = fn(*dense_args(inp), K=K).cpu().numpy()
        _status_ok(B)
        assert check_dense_rows(inp, out, range(inp.Q)) == {}


def test_grid_sampling_with_offset_ranges(B):
    """Rows long enough that the thresholds come from the shared sample grid
    scored by the main scorer (more than one 128-key tile of grid keys):
    ranges starting on, just before and just after grid keys, L = K, L = K + 1,
    empty, short and long rows, all exact."""
    K, N = 2048, 40000
    inp = S.make_dense(16, N, K=K, seed=9, causal=False)
    inp.row_begin[:] = [0, 1, 99, 100, 101, 12345, 39000, 5000, 5000, 20000, 300, 7, 25000, 0, 150, 33333]
    inp.row_end[:] = [N, N, N, 30000, 30000, 39999, N, 5000 + K + 1, 5000 + K, 20000, 2900, 28001, N, 12001, N - 1, N]
    out = B.indexer_topk(*dense_args(inp), K=K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


@pytest.mark.parametrize("K", [256, 1024])
def test_grid_sampling_other_k(B, K):
    """The grid-sampling path with K below 2048 (thresholds aim at 2K)."""
    inp = S.make_dense(24, 50000, K=K, seed=10 + K)
    out = B.indexer_topk(*dense_args(inp), K=K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


def test_grid_sampling_widened_stride(B):
    """Rows longer than 1024 grid keys at stride 200 (N > 204800): the grid
    stride widens so every row keeps at most 1024 samples."""
    K, N = 2048, 262144 + 999
    inp = S.make_dense(8, N, K=K, seed=11, causal=False)
    inp.row_begin[:] = [0, 0, 1, 150000, 262000, 3, 100000, 200]
    inp.row_end[:] = [N, 204800, N, N, N, 100000, 100000 + K, N - 5]
    out = B.indexer_topk(*dense_args(inp), K=K).cpu().numpy()
    _status_ok(B)
    assert check_dense_rows(inp, out, range(inp.Q)) == {}


def test_invalid_range_reports_status_and_pads(B):
    inp = S.make_dense(4, 500, K=16, seed=6, causal=False)
    inp.row_begin[1], inp.row_end[1] = 10, 501      # end past N
    inp.row_begin[2], inp.row_end[2] = 30, 20       # begin after end
    out = B.indexer_topk(*dense_args(inp), K=16).cpu().numpy()
    rc, _ = B.last_device_status()
    assert rc == B.DSA_ERR_RANGE
    assert (out[1] == -1).all() and (out[2] == -1).all()
    assert check_dense_rows(inp, out, [0, 3]) == {}


def test_ties_everywhere(B):
    """All keys identical: every valid index is a correct answer; the output
    must still be K distinct valid indices."""
    inp = S.make_dense(4, 5000, K=512, seed=7, causal=True)
    inp.k[:] = inp.k[0]
    inp.k_scale[:] = inp.k_scale[0]
    for fn in (B.indexer_topk, B.indexer_topk_unfused):
        out = fn(*dense_args(inp), K=inp.K).cpu().numpy()
        _status_ok(B)
        assert check_dense_rows(inp, out, range(inp.Q)) == {}


def test_argument_errors_are_synchronous(B):
    import torch
    inp = S.make_dense(2, 256, K=16, seed=8, causal=False)
    args = dense_args(inp)
    with pytest.raises(B.IndexerError) as e:
        B.indexer_topk(*args, K=0)
    assert e.value.code == B.DSA_ERR_ARG
    with pytest.raises(B.IndexerError):
        B.indexer_topk(*args, K=B.MAX_K + 1)
    bad = torch.empty(256 * 128 + 1, dtype=torch.uint8, device="cuda")[1:].view(256, 128)
    with pytest.raises(B.IndexerError):
        B.indexer_topk(args[0], args[1], bad, *args[3:], K=16)


# ----------------------------------------------------- standalone select ----
@pytest.fixture(params=["split", "rows"])
def matrix_path(B, request):
    """The standalone top-K both ways: rows split over the SMs (threshold
    kernel, filter, candidate selector) and one CTA per row at a time."""
    B.set_option("matrix_row_min", 1 << 40 if request.param == "split" else 0)
    yield request.param
    B.set_option("matrix_row_min", -1)


def test_topk_from_scores_exact(B, matrix_path):
    """Selection only: given fp32 scores the result is exactly determined up
    to ties, so the sorted selected values must equal a full sort bit for bit."""
    import torch
    rng = np.random.default_rng(9)
    Q, N, K = 16, 40000, 2048
    sc = rng.standard_normal((Q, N)).astype(np.float32)
    sc[3] = np.round(sc[3] * 4) / 4          # heavy ties
    sc[4] = 0.0
    sc[4, ::2] = -0.0                         # -0 and +0 tie
    sc[5] = rng.choice(np.float32([1.0, 2.0]), N)
    rb = rng.integers(0, 1000, Q).astype(np.int32)
    re = (rb + rng.integers(0, N - 1000, Q)).astype(np.int32)
    re[6] = rb[6] + K                         # exactly K
    re[7] = rb[7] + 5                         # fewer than K
    out = B.topk_from_scores(*to_dev(sc, rb, re), K=K).cpu().numpy()
    _status_ok(B)
    for t in range(Q):
        L = re[t] - rb[t]
        n = min(L, K)
        sel = out[t, :n]
        assert (out[t, n:] == -1).all()
        assert len(np.unique(sel)) == n and np.all((sel >= rb[t]) & (sel < re[t]))
        want = np.sort(sc[t, rb[t]:re[t]])[::-1][:n]
        got = np.sort(sc[t, sel])[::-1]
        assert np.array_equal(got, want), t


def test_topk_from_scores_long_rows_exact(B, matrix_path):
    """Rows of 128K keys, where the filter keeps a few percent of the scores
    (per-lane masks and one warp scan per step) or, with ties at the
    threshold, many (a ballot per score): the sorted selected values equal a
    full sort bit for bit."""
    rng = np.random.default_rng(31)
    Q, N, K = 8, 131072, 2048
    sc = rng.standard_normal((Q, N)).astype(np.float32)
    sc[1] = np.round(sc[1] * 2) / 2                      # heavy ties
    sc[2] = rng.choice(np.float32([0.5, 1.0, 1.5, 2.0]), N)  # a few values
    sc[3] = 3.0                                          # all equal
    sc[5] = (sc[5] - 3.0).astype(np.float32)             # mostly negative, the top crossing zero
    sc[6, ::3] = 7.0                                     # a third tied at the top
    rb = np.zeros(Q, np.int32)
    re = np.full(Q, N, np.int32)
    rb[4], re[4] = 3, N - 1                              # off a 4-key boundary
    rb[7], re[7] = 1, 40001
    out = B.topk_from_scores(*to_dev(sc, rb, re), K=K).cpu().numpy()
    _status_ok(B)
    for t in range(Q):
        sel = out[t]
        assert len(np.unique(sel)) == K and np.all((sel >= rb[t]) & (sel < re[t])), t
        want = np.sort(sc[t, rb[t]:re[t]])[::-1][:K]
        got = np.sort(sc[t, sel])[::-1]
        assert np.array_equal(got, want), t


@pytest.mark.parametrize("K", [1, 5, 64])
def test_topk_from_scores_small_k_and_tiny_rows(B, matrix_path, K):
    """Small K and rows a few keys long: rows inside one 4-key group (only the
    keys before and after a row's whole float4s are read one by one), rows
    of K, K + 1 and up to 12 keys, rows off a 4-key boundary, ties and -0;
    every row exact against a full sort."""
    rng = np.random.default_rng(91 + K)
    Q, N, ld = 48, 9001, 9004
    sc = np.full((Q, ld), np.nan, np.float32)           # the padding is never read
    sc[:, :N] = rng.standard_normal((Q, N)).astype(np.float32)
    sc[::7, :N] = np.round(sc[::7, :N] * 2) / 2          # ties
    sc[5, 0:N:3] = -0.0
    sc[5, 1:N:3] = 0.0
    rb = rng.integers(0, N - 20, Q).astype(np.int32)
    re = np.minimum(rb + rng.integers(0, 13, Q), N).astype(np.int32)
    re[0::4] = np.minimum(rb[0::4] + rng.integers(K + 1, 4000, len(re[0::4])), N)
    rb[1], re[1] = 5, 7                                  # inside one 4-key group
    rb[2], re[2] = 9, 9 + K                              # exactly K
    rb[3], re[3] = 10, 11 + K                            # K + 1
    rb[6], re[6] = 0, N                                  # the whole row, N odd
    d = to_dev(sc, rb, re)
    out = B.topk_from_scores(d[0], d[1], d[2], K=K, N=N).cpu().numpy()
    _status_ok(B)
    for t in range(Q):
        L = int(re[t] - rb[t])
        n = min(L, K)
        sel = out[t, :n]
        assert (out[t, n:] == -1).all(), t
        assert len(np.unique(sel)) == n and np.all((sel >= rb[t]) & (sel < re[t])), t
        want = np.sort(sc[t, rb[t]:re[t]])[::-1][:n]
        got = np.sort(sc[t, sel])[::-1]
        assert np.array_equal(got, want), t


@pytest.mark.parametrize("bias,kind", [(0, None), (1 << 31, "underflow"), (-(1 << 33), "overflow")])
def test_topk_from_scores_padded_stride_and_forced_repair(B, bias, kind, matrix_path):
    """A padded row stride (ld > N, N not a multiple of 4), ranges that end at
    N or start off a 4-key boundary, rows with ties; with the threshold pushed
    to the top every row longer than K fails the certificate, and with it at
    zero every row longer than a row's 16384 candidate slots does; those are
    selected again from their own matrix rows, and every row is exact."""
    import torch
    rng = np.random.default_rng(77)
    Q, N, K, ld = 14, 20001, 1024, 20008
    sc = np.full((Q, ld), np.nan, np.float32)   # the padding is never read
    sc[:, :N] = rng.standard_normal((Q, N)).astype(np.float32)
    sc[2, :N] = np.round(sc[2, :N] * 2) / 2     # heavy ties
    rb = rng.integers(0, 3000, Q).astype(np.int32)
    re = np.full(Q, N, np.int32)
    re[1::2] = (rb[1::2] + rng.integers(K + 1, N - 3000, Q // 2)).astype(np.int32)
    rb[3] = 4097                                # off a 4-key boundary
    re[5] = rb[5] + K                           # exactly K: trivial path
    re[6] = rb[6] + 3                           # fewer than K
    d = to_dev(sc, rb, re)
    B.set_option("tau_bias", bias)
    try:
        out = B.topk_from_scores(d[0], d[1], d[2], K=K, N=N).cpu().numpy()
        counters = _status_ok(B)
    finally:
        B.set_option("tau_bias", 0)
    long_rows = np.nonzero((re - rb) > K)[0].tolist()
    if kind == "underflow":
        assert counters[kind] == len(long_rows)
        assert sorted(B.last_repaired_rows()) == sorted(long_rows)
    elif kind == "overflow":
        past_slots = np.nonzero((re - rb) > 16384)[0].tolist()
        repaired = sorted(B.last_repaired_rows())
        assert counters[kind] == len(repaired) and set(past_slots) <= set(repaired) <= set(long_rows)
    for t in range(Q):
        L = int(re[t] - rb[t])
        n = min(L, K)
        sel = out[t, :n]
        assert (out[t, n:] == -1).all()
        assert len(np.unique(sel)) == n and np.all((sel >= rb[t]) & (sel < re[t]))
        want = np.sort(sc[t, rb[t]:re[t]])[::-1][:n]
        got = np.sort(sc[t, sel])[::-1]
        assert np.array_equal(got, want), t


@pytest.mark.parametrize("Q", [200, 60, 10])
@pytest.mark.parametrize("bias,kind", [(0, None), (1 << 31, "underflow"), (-(1 << 33), "overflow")])
def test_topk_from_scores_whole_and_half_rows_exact(B, bias, kind, Q):
    """The per-row path's items, with the grid narrowed to 8 SMs: 200 rows of
    up to 70001 keys (many long rows) and 10 rows (fewer than SMs) go by half
    rows (two items per row, the second to finish selects the row from both
    halves' lists), 60 rows by whole rows.  Ranges off a 4-key boundary,
    short and trivial rows, ties (an all-equal row keeps at most K keys at
    its threshold); with the threshold pushed to the top every row longer
    than K fails the certificate, with it at zero every row whose lists
    overflow does; every row is exact."""
    rng = np.random.default_rng(53 + Q)
    N, K, ld = 70001, 2048, 70004
    sc = np.full((Q, ld), np.nan, np.float32)   # the padding is never read
    sc[:, :N] = rng.standard_normal((Q, N)).astype(np.float32)
    sc[7, :N] = np.round(sc[7, :N] * 2) / 2     # heavy ties
    sc[8, :N] = 1.0                             # all equal
    rb = rng.integers(0, 2000, Q).astype(np.int32)
    re = np.full(Q, N, np.int32)
    re[1::3] = (rb[1::3] + rng.integers(K + 1, N - 2000, len(re[1::3]))).astype(np.int32)
    rb[3], re[3] = 4097, N - 3                  # off a 4-key boundary at both ends
    re[5] = rb[5] + K                           # exactly K: trivial path
    re[6] = rb[6] + 3                           # fewer than K
    re[9] = rb[9] + K + 1                       # one key more than K
    d = to_dev(sc, rb, re)
    B.set_option("grid_ctas", 8)
    B.set_option("tau_bias", bias)
    try:
        out = B.topk_from_scores(d[0], d[1], d[2], K=K, N=N).cpu().numpy()
        counters = _status_ok(B)
    finally:
        B.set_option("tau_bias", 0)
        B.set_option("grid_ctas", 0)
    long_rows = np.nonzero((re - rb) > K)[0].tolist()
    if kind == "underflow":
        # (a row shorter than the aim, 36 K / 16 keys, has its threshold's
        # rank outside its sample: every key passes, the bias does not
        # apply, and the row is selected without repair)
        repaired = sorted(B.last_repaired_rows())
        sampled = np.nonzero((re - rb) >= 2 * (36 * K // 16))[0].tolist()
        assert counters[kind] == len(repaired) and set(sampled) <= set(repaired) <= set(long_rows)
    elif kind == "overflow":
        repaired = sorted(B.last_repaired_rows())
        past_halves = np.nonzero((re - rb) > 2 * 8192 + 8)[0].tolist()
        assert counters[kind] == len(repaired) and set(past_halves) <= set(repaired) <= set(long_rows)
    for t in range(Q):
        L = int(re[t] - rb[t])
        n = min(L, K)
        sel = out[t, :n]
        assert (out[t, n:] == -1).all()
        assert len(np.unique(sel)) == n and np.all((sel >= rb[t]) & (sel < re[t])), t
        want = np.sort(sc[t, rb[t]:re[t]])[::-1][:n]
        got = np.sort(sc[t, sel])[::-1]
        assert np.array_equal(got, want), t


# ------------------------------------------------------------- CUDA graph ----
def test_fused_call_replays_from_a_cuda_graph(B):
    """The fused call enqueues kernels only (no host synchronisation, no
    allocation once its scratch is sized), so it can be captured into a CUDA
    graph; a replay reads the buffers' current contents: new inputs copied
    into the captured buffers give those inputs' exact top-K.  Dense rows with
    the shared sample grid, and paged rows with split sampling."""
    import torch
    a = S.make_dense(24, 60000, K=1024, seed=51, causal=True)
    b = S.make_dense(24, 60000, K=1024, seed=52, causal=True)
    pa = S.make_paged(5, 2, K=512, seed=53, len_lo=300, len_hi=40000, n_short=1, short_hi=500)
    # same shapes and page layout, new contents: the cache pages reversed,
    # the queries and weights moved one sequence on
    pb = copy.deepcopy(pa)
    pb.k_cache = np.ascontiguousarray(pa.k_cache[::-1])
    pb.k_cache_scale = np.ascontiguousarray(pa.k_cache_scale[::-1])
    pb.q = np.roll(pa.q, 1, axis=0)
    pb.q_scale = np.roll(pa.q_scale, 1, axis=0)
    pb.w = np.roll(pa.w, 1, axis=0)
    dev_d, dev_p = dense_args(a), paged_args(pa)
    out_d = torch.empty((a.Q, a.K), dtype=torch.int32, device="cuda")
    out_p = torch.empty((pa.B, pa.next_n, pa.K), dtype=torch.int32, device="cuda")
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())

    def calls():
        B.indexer_topk(*dev_d, K=a.K, out=out_d)
        B.indexer_topk_paged(*dev_p, K=pa.K, out=out_p)

    with torch.cuda.stream(gs):
        calls()  # sizes this stream's scratch
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        calls()
    for dst, src in zip(dev_d, dense_args(b)):
        dst.copy_(src)
    for dst, src in zip(dev_p, paged_args(pb)):
        dst.copy_(src)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    rc, _ = B.last_device_status(gs)
    assert rc == 0
    assert check_dense_rows(b, out_d.cpu().numpy(), range(b.Q)) == {}
    outp = out_p.cpu().numpy()
    po = indexer.PagedOracle.from_inputs(pb)
    for bb in range(pb.B):
        for i in range(pb.next_n):
            slots, I, E = po.row_scores(bb, i)
            pr = checks.check_row(outp[bb, i], slots, I, E, pb.K, order_key=np.arange(len(slots)))
            assert not pr, (bb, i, pr)
