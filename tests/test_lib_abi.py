"""The C-ABI library loads on a host without a GPU, exports every function
declared in include/*.h, and rejects bad arguments synchronously (these calls
return before any CUDA work, so they run on CPU)."""
import ctypes
import glob
import os
import re

import pytest

from fp8_scoring_exact_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names += re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", open(h).read())
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("dsa_indexer_topk", "dsa_indexer_topk_paged", "dsa_indexer_topk_unfused",
                 "dsa_indexer_last_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol():
    L = binding.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in binding.SIGNATURES, f"binding lacks {name}"


def test_null_and_size_arguments_rejected_without_gpu():
    L = binding.lib()
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: validation fails first
    assert L.dsa_indexer_topk(None, None, None, None, None, None, None, 1, 1, 1, None, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk(fake, fake, fake, fake, fake, fake, fake, 0, 8, 16, fake, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk(fake, fake, fake, fake, fake, fake, fake, 4, 8, 0, fake, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk(fake, fake, fake, fake, fake, fake, fake, 4, 8, 4096, fake, None) == binding.DSA_ERR_ARG
    mis = P(0x1001)  # misaligned FP8 pointer
    assert L.dsa_indexer_topk(mis, fake, fake, fake, fake, fake, fake, 4, 8, 16, fake, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk_unfused(None, None, None, None, None, None, None, 1, 1, 1, None, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk_paged(fake, fake, fake, fake, fake, fake, fake, 0, 2, 4, 4, 16, fake,
                                    None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_scores(fake, fake, fake, fake, fake, fake, fake, 4, 8, fake, 6, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk_from_scores(fake, 7, fake, fake, 4, 7, 16, fake, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk_host(None, None, None, None, None, None, None, 1, 1, 1, None, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk_host(fake, fake, fake, fake, fake, fake, fake, 4, 8, 0, fake, None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_topk_host(fake, fake, fake, fake, fake, fake, fake, 1 << 25, 8, 16, fake,
                                   None) == binding.DSA_ERR_UNSUPPORTED
    # sparse attention: heads must be a multiple of 16, a positive scale, aligned bf16 arrays
    assert L.dsa_sparse_attention(fake, fake, fake, fake, fake, 4, 8, 64, 100, 0.1, fake, fake,
                                  None) == binding.DSA_ERR_ARG
    assert L.dsa_sparse_attention(fake, fake, fake, fake, fake, 4, 16, 64, 100, 0.0, fake, fake,
                                  None) == binding.DSA_ERR_ARG
    assert L.dsa_sparse_attention(mis, fake, fake, fake, fake, 4, 16, 64, 100, 0.1, fake, fake,
                                  None) == binding.DSA_ERR_ARG
    assert L.dsa_sparse_attention(None, fake, fake, fake, fake, 4, 16, 64, 100, 0.1, fake, fake,
                                  None) == binding.DSA_ERR_ARG
    assert L.dsa_indexer_math_control(None, None, None, None, None, None, None, 1, 1, 1, None,
                                      None) == binding.DSA_ERR_ARG


def test_options_roundtrip_and_validate():
    old = binding.get_option("chunk_tiles")
    binding.set_option("chunk_tiles", 32)
    assert binding.get_option("chunk_tiles") == 32
    binding.set_option("chunk_tiles", old)
    binding.set_option("host_chunk_rows", 256)
    assert binding.get_option("host_chunk_rows") == 256
    binding.set_option("host_chunk_rows", 0)
    with pytest.raises(binding.IndexerError):
        binding.set_option("host_chunk_rows", -1)
    with pytest.raises(binding.IndexerError):
        binding.set_option("chunk_tiles", 0)
    assert binding.lib().dsa_indexer_set_option(999, 1) == binding.DSA_ERR_ARG
    assert "sm_103a" in binding.version()
    # the pipeline wait limit and the test options
    assert binding.get_option("wait_limit_us") == 2000000
    binding.set_option("wait_limit_us", 50000)
    assert binding.get_option("wait_limit_us") == 50000
    binding.set_option("wait_limit_us", 2000000)
    for name, bad in (("wait_limit_us", 0), ("wait_limit_us", 60000001), ("unit_order", 2), ("test_withhold", 3)):
        with pytest.raises(binding.IndexerError):
            binding.set_option(name, bad)
    for name in ("unit_order", "test_withhold"):
        binding.set_option(name, 1)
        assert binding.get_option(name) == 1
        binding.set_option(name, 0)
    # the standalone top-K's path: -1 chosen per call (the default), 0 and up a row count
    assert binding.get_option("matrix_row_min") == -1
    binding.set_option("matrix_row_min", 0)
    assert binding.get_option("matrix_row_min") == 0
    binding.set_option("matrix_row_min", 1 << 40)
    assert binding.get_option("matrix_row_min") == 1 << 40
    with pytest.raises(binding.IndexerError):
        binding.set_option("matrix_row_min", -2)
    binding.set_option("matrix_row_min", -1)


def test_product_path_has_no_cpu_fallback():
    """The binding must not import the oracle or compute anything itself."""
    src = open(os.path.join(ROOT, "fp8_scoring_exact_gb300", "binding.py")).read()
    assert "oracle" not in src.split('"""', 2)[2]
    import torch
    with pytest.raises(TypeError):
        binding.indexer_topk(torch.zeros(1, 64, 128, dtype=torch.uint8), torch.ones(1), torch.zeros(8, 128, dtype=torch.uint8),
                             torch.ones(8), torch.ones(1, 64), torch.zeros(1, dtype=torch.int32),
                             torch.ones(1, dtype=torch.int32), K=4)
