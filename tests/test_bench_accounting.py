"""The bench's roofline accounting against the sizes printed in "Fusing
Indexer Scoring and Exact Top-k for DeepSeek-V3.2" (tests/golden/paper_sizes.txt),
and the oracle's CPU-baseline sampling helpers."""
import os

import bench

GOLD = os.path.join(os.path.dirname(__file__), "golden", "paper_sizes.txt")


def golden():
    vals = {}
    for line in open(GOLD):
        line = line.strip()
        if line and not line.startswith("#"):
            name, value = line.split()[:2]
            vals[name] = int(value)
    return vals


def test_per_row_key_constants_match_the_paper():
    g = golden()
    assert bench.FLOP_PER_ROW_KEY == g["flop_per_row_key"]
    assert bench.BYTES_PER_KEY == g["bytes_per_key"]
    assert round(bench.FLOP_PER_ROW_KEY / bench.BYTES_PER_KEY) == g["intensity_floor_flop_per_b"]


def test_matrix_and_output_sizes_match_the_paper():
    g = golden()
    Q, N, K = 4096, 131072, 2048
    assert bench.score_matrix_bytes(Q, N) == g["score_matrix_bytes_q4096_n131072"]
    assert 2 * bench.score_matrix_bytes(Q, N) == g["score_roundtrip_bytes_q4096_n131072"]
    assert Q * K * 4 == g["output_bytes_q4096_k2048"]
    # algorithmic bytes: q, q scale, weights, every key once, output
    assert bench.algorithmic_bytes(Q, N, K) == Q * 8192 + Q * 4 + Q * 256 + N * 132 + Q * K * 4


def test_row_keys_of_the_causal_workloads():
    from fp8_scoring_exact_gb300 import synthetic as S
    for Q, N, want in ((2048, 16384, 31458304), (4096, 131072, 528484352), (4096, 163840, 662702080)):
        rb, re = S.causal_ranges(Q, N)
        assert int((re.astype('int64') - rb).sum()) == want
