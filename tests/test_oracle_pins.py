"""Pins of the CPU oracle against things other than itself.

* e4m3 decode: hand-derived codes (tests/golden/e4m3_codes.txt) and all 256
  codes against torch's independent float8_e4m3fn decoder.
* exact dot: Python-integer brute force, bit for bit.
* score formula: hand-computed worked examples of
  I[t,s] = sum_j w[t,j] ReLU(q[t,j].k[s]) ("Fusing Indexer Scoring and Exact
  Top-k for DeepSeek-V3.2", section 1.1).
* selection: enumeration of every K-subset on tiny rows; trivial rows; ties.
* invariants: permutation equivariance, TopK(A u B) = TopK(TopK(A) u B)
  (section 3.1), paged = dense on the gathered keys.
* mutation: plausible slips planted in the oracle are caught by these pins.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import checks, e4m3, indexer

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- e4m3 ----
def _golden_codes():
    rows = []
    with open(os.path.join(GOLD, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            rows.append((int(c, 16), float(v)))
    return rows


def test_e4m3_golden_codes():
    tab = e4m3.table_f64()
    for code, val in _golden_codes():
        got = tab[code]
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val) or (val == 0 and got == 0), hex(code)


def test_e4m3_all_codes_match_torch_decoder():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.table_f64()
    nan_ref, nan_ours = np.isnan(ref), np.isnan(ours)
    assert (nan_ref == nan_ours).all()
    assert nan_ours.sum() == 2
    assert (ref[~nan_ref] == ours[~nan_ours]).all()


def test_e4m3_units_range_and_monotone():
    units, nan = e4m3.table_units()
    assert units.max() == e4m3.MAX_UNITS and units.min() == -e4m3.MAX_UNITS
    pos = units[:0x7F]              # codes 0x00..0x7E are increasing
    assert (np.diff(pos) > 0).all()
    assert (units[0x80:0xFF] == -units[0x00:0x7F]).all()
    with pytest.raises(ValueError):
        e4m3.decode_array_units(np.array([0x7F], np.uint8))


# ------------------------------------------------------------ exact dot ----
def test_exact_dots_match_python_integers():
    rng = np.random.default_rng(11)
    H, D, L = 3, 128, 7
    q = rng.integers(0, 256, size=(H, D), dtype=np.uint8)
    k = rng.integers(0, 256, size=(L, D), dtype=np.uint8)
    q[q == 0x7F] = 0x7E
    q[q == 0xFF] = 0xFE
    k[k == 0x7F] = 0x7E
    k[k == 0xFF] = 0xFE
    # extremes: largest magnitudes everywhere in one row / head
    q[0, :] = 0x7E
    k[0, :] = 0x7E
    k[1, :] = 0xFE
    qu = e4m3.decode_array_units(q).astype(np.float64)
    ku = e4m3.decode_array_units(k).astype(np.float64)
    got = indexer.exact_dots(qu, ku)
    for h in range(H):
        for s in range(L):
            want = sum(e4m3.decode_units(int(q[h, d])) * e4m3.decode_units(int(k[s, d]))
                       for d in range(D))
            assert int(got[h, s]) == want
    assert int(got[0, 0]) == 128 * e4m3.MAX_UNITS ** 2


# ------------------------------------------------------- worked examples ----
def _codes(vals):
    """Encode exactly representable values via the golden table (inverse)."""
    tab = e4m3.table_f64()
    lut = {}
    for c in range(256):
        v = tab[c]
        if not np.isnan(v) and v not in lut and not (v == 0 and c == 0x80):
            lut[v] = c
    return np.array([[lut[float(x)] for x in row] for row in vals], np.uint8)


def test_worked_example_two_heads_by_hand():
    # H=2, D=4.  q0 = (1, 2, 0, -1), q1 = (0.5, -1, 3, 0); k = (2, 0.5, -1, 1)
    # q0.k = 2 + 1 + 0 - 1 = 2 ;  q1.k = 1 - 0.5 - 3 + 0 = -2.5
    # w = (0.25, 4): I = 0.25 * ReLU(2) + 4 * ReLU(-2.5) = 0.5
    # with q_scale 2 and k_scale 0.5 the dequantised dots are scaled by 1: I = 0.5
    # E = 0.25 * 2 + 4 * 2.5 = 10.5
    q = _codes([[1, 2, 0, -1], [0.5, -1, 3, 0]])
    k = _codes([[2, 0.5, -1, 1]])
    o = indexer.DenseOracle(q[None], np.array([2.0], np.float32), k,
                            np.array([0.5], np.float32), np.array([[0.25, 4.0]], np.float32),
                            np.array([0]), np.array([1]), 1)
    ids, I, E = o.row_scores(0)
    assert ids.tolist() == [0]
    assert I[0] == 0.5 and E[0] == 10.5
    # the scales enter linearly: doubling k_scale doubles both
    o.k_scale = np.array([1.0], np.float32)
    _, I2, E2 = o.row_scores(0)
    assert I2[0] == 1.0 and E2[0] == 21.0


def test_worked_example_one_hot_key_and_single_head():
    # k_s = c * e_d (one-hot): q_j . k_s = c * q[j, d].  With a single head of
    # weight 1 the score is ReLU(c * q[0, d]) * scales.
    rng = np.random.default_rng(3)
    H, D = 64, 128
    qv = rng.choice([-2.0, -0.5, 0.25, 1.0, 3.0], size=(H, D))
    q = _codes(qv)
    keys = np.zeros((D, D))
    c = 1.5
    for d in range(D):
        keys[d, d] = c
    k = _codes(keys)
    w = np.zeros((1, H), np.float32)
    w[0, 5] = 1.0
    o = indexer.DenseOracle(q[None], np.array([1.0], np.float32), k, np.ones(D, np.float32), w,
                            np.array([0]), np.array([D]), 8)
    _, I, E = o.row_scores(0)
    want = np.maximum(c * qv[5], 0.0)
    assert np.array_equal(I, want)
    assert np.array_equal(E, np.abs(c * qv[5]))
    # negative weights flip the sign of the contribution, negative dots give 0
    o.w = -w
    _, In, _ = o.row_scores(0)
    assert np.array_equal(In, -want)


def test_relu_per_head_not_after_sum():
    # Two heads with opposite dots: per-head ReLU gives w0*d, a ReLU of the
    # weighted sum would give 0.  q0 = (1,0,..), q1 = (-1,0,..), k = (1,0,..)
    q = np.zeros((2, 4))
    q[0, 0], q[1, 0] = 1.0, -1.0
    k = np.zeros((1, 4))
    k[0, 0] = 1.0
    o = indexer.DenseOracle(_codes(q)[None], np.ones(1, np.float32), _codes(k),
                            np.ones(1, np.float32), np.array([[1.0, 1.0]], np.float32),
                            np.array([0]), np.array([1]), 1)
    _, I, E = o.row_scores(0)
    assert I[0] == 1.0 and E[0] == 2.0


def test_worked_example_offset_range_by_hand():
    # A row whose valid range starts past key 0 (section 2.3: each row has its
    # own [k_start, k_end)).  Keys are one-hot on dim 0 with distinct values
    # c_s, q has a single non-zero element q[0, 0] = 1 and the only weight is
    # w[0] = 2, so I[s] = 2 * ReLU(c_s) * q_scale * k_scale[s].
    #   s     :  0    1    2    3     4     5    6    7
    #   c_s   :  1   -1    2    3   -0.5   0.25  4   1.5
    #   k_sc  :  1    1    1    1     1    0.5   2    1
    # Row 0 sees [3, 7): I = 2*3*1, 0, 2*0.25*0.5, 2*4*2 = 6, 0, 0.25, 16
    # (q_scale 1); its top 2 are keys 6 and 3, labelled by their absolute
    # positions.
    c = [1, -1, 2, 3, -0.5, 0.25, 4, 1.5]
    keys = np.zeros((8, 4))
    keys[:, 0] = c
    q = np.zeros((2, 4))
    q[0, 0] = 1.0
    ks = np.array([1, 1, 1, 1, 1, 0.5, 2, 1], np.float32)
    o = indexer.DenseOracle(_codes(q)[None], np.ones(1, np.float32), _codes(keys), ks,
                            np.array([[2.0, 0.0]], np.float32), np.array([3]), np.array([7]), 2)
    ids, I, E = o.row_scores(0)
    assert ids.tolist() == [3, 4, 5, 6]
    assert I.tolist() == [6.0, 0.0, 0.25, 16.0]
    assert E.tolist() == [6.0, 1.0, 0.25, 16.0]
    out, *_ = o.topk(0)
    assert sorted(out.tolist()) == [3, 6]


def test_offset_range_is_the_full_row_restricted():
    # the same keys scored over [b, e) and over [0, N): the scores of the
    # offset row are the full row's entries b..e-1, under the same labels
    # (the float64 head combination may sum in another order for another
    # length, so equal to within 1e-12 E rather than bit for bit)
    q, qs, k, ks, w, _, _, K = _tiny_dense(12, Q=1)
    N = k.shape[0]
    full = indexer.DenseOracle(q, qs, k, ks, w, np.array([0]), np.array([N]), K)
    ids_f, I_f, E_f = full.row_scores(0)
    for b, e in [(37, 211), (1, N), (N - 17, N), (150, 151)]:
        part = indexer.DenseOracle(q, qs, k, ks, w, np.array([b]), np.array([e]), K)
        ids, I, E = part.row_scores(0)
        assert ids.tolist() == list(range(b, e))
        assert np.all(np.abs(I - I_f[b:e]) <= 1e-12 * E_f[b:e])
        assert np.all(np.abs(E - E_f[b:e]) <= 1e-12 * E_f[b:e])


# ------------------------------------------------------------- selection ----
def test_topk_is_maximal_by_subset_enumeration():
    rng = np.random.default_rng(5)
    for trial in range(60):
        L = int(rng.integers(1, 10))
        K = int(rng.integers(1, 5))
        I = rng.choice([-1.0, 0.0, 0.5, 1.0, 2.0, 3.0], size=L)  # many ties
        ids = np.arange(10, 10 + L)
        out, kth = indexer.topk_by_sort(ids, I, K)
        n = min(L, K)
        assert (out[n:] == -1).all()
        sel = out[:n]
        assert len(set(sel.tolist())) == n and set(sel.tolist()) <= set(ids.tolist())
        mine = np.sort(I[sel - 10])[::-1]
        for sub in itertools.combinations(range(L), n):
            other = np.sort(I[list(sub)])[::-1]
            assert (mine >= other).all()
        if L >= K:
            assert kth == np.sort(I)[::-1][K - 1]


def test_trivial_rows_return_all_then_padding():
    ids = np.array([7, 3, 9])
    out, kth = indexer.topk_by_sort(ids, np.array([0.1, 0.2, 0.3]), 5)
    assert sorted(out[:3].tolist()) == [3, 7, 9] and out[3:].tolist() == [-1, -1]
    assert kth is None


def test_ties_break_to_lowest_index():
    out, _ = indexer.topk_by_sort(np.arange(6), np.array([1.0, 2, 2, 2, 0, 2]), 2)
    assert out.tolist() == [1, 2]


# ------------------------------------------------------------ invariants ----
def _tiny_dense(seed, Q=3, N=300, K=16):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 0x7E, size=(Q, 64, 128), dtype=np.uint8)
    q |= (rng.integers(0, 2, size=q.shape, dtype=np.uint8) << 7)
    k = rng.integers(0, 0x7E, size=(N, 128), dtype=np.uint8)
    k |= (rng.integers(0, 2, size=k.shape, dtype=np.uint8) << 7)
    qs = rng.uniform(0.001, 0.01, Q).astype(np.float32)
    ks = rng.uniform(0.001, 0.01, N).astype(np.float32)
    w = rng.standard_normal((Q, 64)).astype(np.float32)
    rb = np.array([0, 10, 50])[:Q]
    re = np.array([N, N - 5, 70])[:Q]
    return q, qs, k, ks, w, rb, re, K


def test_permuting_keys_permutes_selection():
    q, qs, k, ks, w, rb, re, K = _tiny_dense(1, Q=1)
    rb, re = np.array([0]), np.array([k.shape[0]])
    o = indexer.DenseOracle(q, qs, k, ks, w, rb, re, K)
    perm = np.random.default_rng(2).permutation(k.shape[0])
    op = indexer.DenseOracle(q, qs, k[perm], ks[perm], w, rb, re, K)
    _, _, I, _, _ = o.topk(0)
    _, _, Ip, _, _ = op.topk(0)
    assert np.array_equal(Ip, I[perm])
    out, *_ = o.topk(0)
    outp, *_ = op.topk(0)
    assert np.array_equal(np.sort(I[out]), np.sort(Ip[outp]))


def test_topk_of_union_equals_topk_of_topk_union():
    rng = np.random.default_rng(9)
    K = 8
    for _ in range(20):
        I = rng.standard_normal(200).round(1)  # ties
        ids = np.arange(200)
        A, B = ids[:120], ids[120:]
        full, _ = indexer.topk_by_sort(ids, I, K)
        ta, _ = indexer.topk_by_sort(A, I[A], K)
        merged = np.concatenate([ta, B])
        tm, _ = indexer.topk_by_sort(merged, I[merged], K)
        assert np.array_equal(np.sort(I[full]), np.sort(I[tm]))


def test_paged_oracle_equals_dense_on_gathered_keys():
    rng = np.random.default_rng(4)
    B, nn, P = 2, 2, 7
    kc = rng.integers(0, 0x7E, size=(P, 64, 128), dtype=np.uint8)
    kcs = rng.uniform(0.5, 2, (P, 64)).astype(np.float32)
    q = rng.integers(0, 0x7E, size=(B, nn, 64, 128), dtype=np.uint8)
    qs = np.ones((B, nn), np.float32)
    w = rng.standard_normal((B, nn, 64)).astype(np.float32)
    bt = np.array([[3, 0, 6, -1], [5, 1, 2, 4]], np.int32)
    seq = np.array([150, 256], np.int32)
    po = indexer.PagedOracle(q, qs, kc, kcs, w, bt, seq, 32)
    # row (0, 0) sees logical keys [0, 149): pages 3, 0, 6(first 21 tokens)
    slots = po.row_slots(0, 0)
    assert len(slots) == 149
    assert slots[0] == 3 * 64 and slots[64] == 0 and slots[128] == 6 * 64 and slots[-1] == 6 * 64 + 20
    assert po.row_length(1, 1) == 256
    for b in range(B):
        for i in range(nn):
            slots, I, E = po.row_scores(b, i)
            dk = kc.reshape(-1, 128)[slots]
            do = indexer.DenseOracle(q[b, i][None], qs[b, i:i + 1], dk, kcs.reshape(-1)[slots],
                                     w[b, i][None], np.array([0]), np.array([len(slots)]), 32)
            _, Id, Ed = do.row_scores(0)
            assert np.array_equal(I, Id) and np.array_equal(E, Ed)


# -------------------------------------------------------------- checker ----
def test_checker_accepts_oracle_and_catches_planted_mistakes():
    q, qs, k, ks, w, rb, re, K = _tiny_dense(7, Q=1)
    o = indexer.DenseOracle(q, qs, k, ks, w, rb, re, K)
    out, ids, I, E, kth = o.topk(0)
    assert checks.check_row(out, ids, I, E, K) == []
    bad = out.copy()
    bad[0] = bad[1]
    assert checks.check_row(bad, ids, I, E, K)                    # duplicate
    bad = out.copy()
    bad[0] = 10 ** 6
    assert checks.check_row(bad, ids, I, E, K)                    # out of range
    worst = np.argsort(I)[0]
    bad = out.copy()
    bad[0] = ids[worst]
    assert checks.check_row(bad, ids, I, E, K)                    # low score
    bad = out.copy()
    bad[-1] = -1
    assert checks.check_row(bad, ids, I, E, K)                    # missing entry


def test_checker_elementwise_criterion_catches_a_swapped_tie():
    # Scores with a three-way tie at the K-th value (theta = 3, K = 4): the
    # exact top-4 is {5, 4, 3, 3}.  Swapping the key scoring 5 for the
    # unselected theta-tied key keeps every index valid and unique (i) and
    # every selected score at or above theta (ii), so only the element-wise
    # comparison of the sorted scores (iii) can see that 5 is missing.
    ids = np.arange(10, 20)
    I = np.array([5.0, 4.0, 3.0, 3.0, 3.0, 2.0, 1.0, 0.0, 0.0, 0.0])
    E = np.abs(I) + 1.0
    K = 4
    good = np.array([10, 11, 12, 13])
    assert checks.check_row(good, ids, I, E, K) == []
    swapped = np.array([14, 11, 12, 13])                          # 5 -> a theta tie
    assert checks.check_row(swapped, ids, I, E, K, elementwise=False) == []
    probs = checks.check_row(swapped, ids, I, E, K)
    assert len(probs) == 1 and "sorted scores differ" in probs[0]
    # a different theta-tied key in place of a tied one is a correct answer
    assert checks.check_row(np.array([10, 11, 12, 14]), ids, I, E, K) == []


# ------------------------------------------------------------- mutation ----
MUTANTS = {
    "no_relu": lambda d, w, qs, ks: (w.astype(np.float64) @ d.astype(np.float64)) * float(qs) * ks * indexer.DOT_UNIT,
    "relu_after_sum": lambda d, w, qs, ks: np.maximum(w.astype(np.float64) @ d.astype(np.float64), 0) * float(qs) * ks * indexer.DOT_UNIT,
    "no_weight": lambda d, w, qs, ks: np.maximum(d, 0).sum(0) * float(qs) * ks * indexer.DOT_UNIT,
    "no_k_scale": lambda d, w, qs, ks: (w.astype(np.float64) @ np.maximum(d, 0)) * float(qs) * indexer.DOT_UNIT,
    "abs_weight": lambda d, w, qs, ks: (np.abs(w.astype(np.float64)) @ np.maximum(d, 0)) * float(qs) * ks * indexer.DOT_UNIT,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_oracle_mistakes(name, monkeypatch):
    real = indexer.combine_heads

    def mutant(dots, w_row, q_scale, k_scale):
        I, E = real(dots, w_row, q_scale, k_scale)
        return MUTANTS[name](dots, w_row, q_scale, k_scale.astype(np.float64)), E

    monkeypatch.setattr(indexer, "combine_heads", mutant)
    pins = [test_worked_example_two_heads_by_hand, test_worked_example_one_hot_key_and_single_head,
            test_relu_per_head_not_after_sum]
    caught = 0
    for p in pins:
        try:
            p()
        except AssertionError:
            caught += 1
    assert caught >= 1, f"mutation {name} escaped every pin"


def _row_scores_keys_from_zero(self, t):
    # planted slip: the row's keys taken from position 0 instead of row_begin
    b, e = int(self.row_begin[t]), int(self.row_end[t])
    ids = np.arange(b, e, dtype=np.int64)
    dots = indexer.exact_dots(self.qu[t], self.ku[:e - b])
    I, E = indexer.combine_heads(dots, self.w[t], self.q_scale[t], self.k_scale[:e - b])
    return ids, I, E


def _row_scores_labels_from_zero(self, t):
    # planted slip: the right keys, labelled 0..L-1 instead of b..e-1
    b, e = int(self.row_begin[t]), int(self.row_end[t])
    dots = indexer.exact_dots(self.qu[t], self.ku[b:e])
    I, E = indexer.combine_heads(dots, self.w[t], self.q_scale[t], self.k_scale[b:e])
    return np.arange(e - b, dtype=np.int64), I, E


@pytest.mark.parametrize("mutant", [_row_scores_keys_from_zero, _row_scores_labels_from_zero])
def test_pins_catch_planted_offset_range_mistakes(mutant, monkeypatch):
    monkeypatch.setattr(indexer.DenseOracle, "row_scores", mutant)
    for pin in (test_worked_example_offset_range_by_hand, test_offset_range_is_the_full_row_restricted):
        with pytest.raises(AssertionError):
            pin()


def test_pins_catch_a_vacuous_elementwise_criterion(monkeypatch):
    # the checker with criterion (iii) switched off must fail its pin
    real = checks.check_row
    monkeypatch.setattr(checks, "check_row", lambda *a, **kw: real(*a, **{**kw, "elementwise": False}))
    with pytest.raises(AssertionError):
        test_checker_elementwise_criterion_catches_a_swapped_tie()


def test_pins_catch_transposed_dot(monkeypatch):
    # a transposed operand (dots over heads instead of dims) changes the
    # one-hot example
    real = indexer.exact_dots
    monkeypatch.setattr(indexer, "exact_dots", lambda qu, ku: real(qu[:, ::-1], ku))
    with pytest.raises(AssertionError):
        test_worked_example_one_hot_key_and_single_head()
