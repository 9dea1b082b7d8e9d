"""GB300 (sm_103a) DeepSeek-V3.2 DSA indexer with exact top-K selection.

The operator lives in the CUDA library libdsa_indexer.so (C ABI in
include/dsa_indexer.h); `binding` is its thin Python front end and
`synthetic` draws seeded inputs shaped like the indexer workloads.
"""
from .binding import (IndexerError, indexer_scores, indexer_topk, indexer_topk_paged,  # noqa: F401
                      indexer_topk_unfused, last_device_status, last_repaired_rows, launch_count, profiled_main_ms,
                      release, set_option, get_option, topk_from_scores, version)
