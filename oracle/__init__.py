"""CPU oracle for the DSA indexer with exact top-K selection.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
bench's CPU-baseline leg may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or calls anything here,
and nothing here imports the product.

What it computes (from "Fusing Indexer Scoring and Exact Top-k for
DeepSeek-V3.2", section 1.1 equation and section 2.3 problem definition):

    I[t, s] = sum_{j=1..64} w[t, j] * ReLU(q[t, j] . k[s])

over every valid key s of row t, with q and k FP8 e4m3 codes dequantised by
their per-token FP32 scales, and returns the K highest-scoring key indices of
every row (unordered; ties may resolve to any valid index).

How (plain, slow, exact):
  * e4m3 codes are decoded bit by bit from the format definition into
    integers in units of 2^-9 (`e4m3.py`);
  * each 128-long dot product is formed exactly as an integer in units of
    2^-18 (`indexer.py`);
  * heads, weights and scales are combined in float64;
  * selection is a full sort by (score descending, index ascending).

`select.py` restates the method's own selection steps (sampled threshold,
compare-and-append, four-pass radix select, certificate; section 3.2) in plain
Python for unit tests of that logic.  `checks.py` holds the parity criteria.

`sparse_attention.py` is the oracle of the step downstream of the indexer
(contest write-up, "DSA Sparse Attention"): attention of each query token
over the KV entries its top-K indices name, base-2 softmax, 512-dim output
and log-sum-exp, in float64.

Pins: tests/test_oracle_*.py check every function here against the format
definition, torch's independent float8 decoder, Python-integer brute force,
hand-computed worked examples, closed-form special cases, subset enumeration
and invariants.
"""

from . import e4m3, indexer, select, checks, sparse_attention  # noqa: F401
