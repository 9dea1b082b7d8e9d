"""Pins of the sparse-attention oracle (contest write-up, "DSA Sparse
Attention": gather the top-K KV entries, logits q_nope . K_c + q_pe . K_p,
base-2 softmax, 512-dim output and LSE) against things other than itself:
a worked example computed by hand, special cases with closed forms, an
independent natural-base formula written out with Python floats, invariants,
and planted mistakes that those pins must catch."""
import math

import numpy as np
import pytest

from oracle import sparse_attention as sa


def _hand_case():
    # Dc = 2, Dp = 1.  q_nope = (1, 0), q_pe = (2).  Rows: ckv0 = (1, 2),
    # kpe0 = 0.5; ckv1 = (0, 4), kpe1 = -1.
    #   z0 = 1*1 + 0*2 + 2*0.5 = 2 ;  z1 = 0 + 0 + 2*(-1) = -2
    # sm_scale = ln 2 makes u = z * sm_scale * log2(e) = z: weights 2^2 : 2^-2
    # = 4 : 1/4, so p = (16/17, 1/17);
    #   out = 16/17 (1, 2) + 1/17 (0, 4) = (16/17, 36/17)
    #   lse = log2(4 + 1/4) = log2(17) - 2
    q_nope = np.array([1.0, 0.0])
    q_pe = np.array([2.0])
    ckv = np.array([[1.0, 2.0], [0.0, 4.0]])
    kpe = np.array([[0.5], [-1.0]])
    return q_nope, q_pe, ckv, kpe, math.log(2.0)


def test_worked_example_by_hand():
    q_nope, q_pe, ckv, kpe, sc = _hand_case()
    out, lse, P, _ = sa.attend_one(q_nope, q_pe, ckv, kpe, [0, 1], sc)
    assert np.allclose(out, [16 / 17, 36 / 17], rtol=0, atol=1e-15)
    assert abs(lse - (math.log2(17) - 2)) < 1e-14
    assert np.allclose(P, [16 / 17, 1 / 17], rtol=0, atol=1e-15)


def test_padding_and_order_do_not_matter():
    q_nope, q_pe, ckv, kpe, sc = _hand_case()
    a = sa.attend_one(q_nope, q_pe, ckv, kpe, [0, 1], sc)
    b = sa.attend_one(q_nope, q_pe, ckv, kpe, [-1, 1, -1, 0, -1], sc)
    assert np.allclose(a[0], b[0], rtol=0, atol=1e-15) and abs(a[1] - b[1]) < 1e-14


def test_single_index_and_empty_list():
    q_nope, q_pe, ckv, kpe, sc = _hand_case()
    out, lse, _, _ = sa.attend_one(q_nope, q_pe, ckv, kpe, [-1, 1, -1], sc)
    assert np.array_equal(out, ckv[1]) and lse == -2.0       # u1 = z1 = -2
    out, lse, _, _ = sa.attend_one(q_nope, q_pe, ckv, kpe, [-1, -1], sc)
    assert np.array_equal(out, np.zeros(2)) and lse == -math.inf


def test_equal_logits_give_the_mean_and_log2_of_the_count():
    rng = np.random.default_rng(1)
    n, dc = 6, 8
    ckv = rng.standard_normal((n, dc))
    kpe = np.zeros((n, 3))
    q_nope = np.zeros(dc)                      # every logit is 0
    out, lse, _, _ = sa.attend_one(q_nope, np.zeros(3), ckv, kpe, np.arange(n), 0.7)
    assert np.allclose(out, ckv.mean(0), rtol=0, atol=1e-14)
    assert abs(lse - math.log2(n)) < 1e-14


def test_matches_a_natural_base_softmax_written_out():
    # independent formula: p_j = exp(z_j s) / sum_k exp(z_k s), with Python
    # floats and math.exp; lse_2 = ln(sum exp(z s)) / ln 2
    rng = np.random.default_rng(2)
    S, dc, dp = 40, 16, 4
    ckv = rng.standard_normal((S, dc))
    kpe = rng.standard_normal((S, dp))
    q_nope = rng.standard_normal(dc)
    q_pe = rng.standard_normal(dp)
    idx = [3, 17, -1, 0, 39, 22, 8]
    s = 0.3
    out, lse, _, _ = sa.attend_one(q_nope, q_pe, ckv, kpe, idx, s)
    valid = [i for i in idx if i >= 0]
    zs = [sum(q_nope[d] * ckv[i, d] for d in range(dc)) + sum(q_pe[d] * kpe[i, d] for d in range(dp))
          for i in valid]
    ws = [math.exp(z * s) for z in zs]
    tot = sum(ws)
    want = [sum(w * ckv[i, d] for w, i in zip(ws, valid)) / tot for d in range(dc)]
    assert np.allclose(out, want, rtol=1e-13, atol=1e-13)
    assert abs(lse - math.log(tot) / math.log(2)) < 1e-12


def test_shifting_every_logit_shifts_only_the_lse():
    # an extra rope dimension that is 1 on every key and c on the query adds
    # c to every logit: the weights (and so the output) are unchanged, the
    # base-2 LSE moves by c * sm_scale * log2(e)
    rng = np.random.default_rng(3)
    S, dc = 30, 8
    ckv = rng.standard_normal((S, dc))
    kpe = np.concatenate([rng.standard_normal((S, 2)), np.ones((S, 1))], 1)
    q_nope = rng.standard_normal(dc)
    idx = np.arange(0, S, 2)
    s, c = 0.5, 7.0
    o0, l0, _, _ = sa.attend_one(q_nope, np.array([0.3, -1.2, 0.0]), ckv, kpe, idx, s)
    o1, l1, _, _ = sa.attend_one(q_nope, np.array([0.3, -1.2, c]), ckv, kpe, idx, s)
    assert np.allclose(o0, o1, rtol=0, atol=1e-13)
    assert abs((l1 - l0) - c * s / math.log(2)) < 1e-12


def test_huge_logits_stay_finite():
    ckv = np.array([[1.0, 0.0], [0.0, 1.0]])
    kpe = np.array([[1.0], [1.0 - 1e-3]])
    out, lse, _, _ = sa.attend_one(np.zeros(2), np.array([1e5]), ckv, kpe, [0, 1], 1.0)
    assert np.all(np.isfinite(out)) and np.isfinite(lse)
    # u0 - u1 = 100 * log2(e): the second weight is 2^-144 of the first
    assert np.allclose(out, [1.0, 0.0], rtol=0, atol=1e-40)


def test_batched_driver_matches_per_head_calls():
    rng = np.random.default_rng(4)
    T, H, S, dc, dp, K = 3, 2, 50, 8, 2, 10
    q_nope = rng.standard_normal((T, H, dc))
    q_pe = rng.standard_normal((T, H, dp))
    ckv = rng.standard_normal((S, dc))
    kpe = rng.standard_normal((S, dp))
    idx = rng.integers(-1, S, (T, K))
    out, lse = sa.sparse_attention(q_nope, q_pe, ckv, kpe, idx, 0.25)
    for t in range(T):
        for h in range(H):
            o, l, _, _ = sa.attend_one(q_nope[t, h], q_pe[t, h], ckv, kpe, idx[t], 0.25)
            assert np.array_equal(out[t, h], o) and lse[t, h] == l
    # the head index really selects the head: heads differ
    assert not np.allclose(out[:, 0], out[:, 1])


# ------------------------------------------------------------- mutation ----
def _no_scale(q_nope, q_pe, ckv, kpe, idx, sm_scale):
    return _REAL(q_nope, q_pe, ckv, kpe, idx, 1.0)


def _natural_lse(q_nope, q_pe, ckv, kpe, idx, sm_scale):
    o, l, P, V = _REAL(q_nope, q_pe, ckv, kpe, idx, sm_scale)
    return o, l * math.log(2.0), P, V


def _padding_as_last_row(q_nope, q_pe, ckv, kpe, idx, sm_scale):
    idx = np.where(np.asarray(idx) < 0, ckv.shape[0] - 1, idx)
    return _REAL(q_nope, q_pe, ckv, kpe, idx, sm_scale)


def _no_rope_part(q_nope, q_pe, ckv, kpe, idx, sm_scale):
    return _REAL(q_nope, np.zeros_like(np.asarray(q_pe, float)), ckv, kpe, idx, sm_scale)


_REAL = sa.attend_one


@pytest.mark.parametrize("mutant", [_no_scale, _natural_lse, _padding_as_last_row, _no_rope_part])
def test_pins_catch_planted_mistakes(mutant, monkeypatch):
    monkeypatch.setattr(sa, "attend_one", mutant)
    pins = [test_worked_example_by_hand, test_padding_and_order_do_not_matter, test_single_index_and_empty_list,
            test_equal_logits_give_the_mean_and_log2_of_the_count, test_matches_a_natural_base_softmax_written_out,
            test_shifting_every_logit_shifts_only_the_lse]
    caught = 0
    for p in pins:
        try:
            p()
        except AssertionError:
            caught += 1
    assert caught >= 1, f"{mutant.__name__} escaped every pin"
