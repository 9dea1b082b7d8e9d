"""Thin Python binding of libdsa_indexer.so (include/dsa_indexer.h).

Argument marshalling only: every step of the operator runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (FP8 data as uint8 or
torch.float8_e4m3fn); they are passed to the C ABI as raw device pointers
together with the current (or given) CUDA stream.  indexer_topk_host takes
CPU tensors instead (the library does the copies).  There is no CPU fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

DSA_OK, DSA_ERR_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_RANGE = 0, -1, -2, -3, -4, -5
STATUS_NAMES = {0: "DSA_OK", -1: "DSA_ERR_ARG", -2: "DSA_ERR_UNSUPPORTED", -3: "DSA_ERR_CUDA",
                -4: "DSA_ERR_TIMEOUT", -5: "DSA_ERR_RANGE"}
OPTIONS = {"chunk_tiles": 1, "tau_bias": 2, "profile": 3, "grid_ctas": 4, "sample_target": 5,
           "host_chunk_rows": 6, "unit_order": 7, "wait_limit_us": 8, "test_withhold": 9,
           "matrix_row_min": 10}
HEADS, HEAD_DIM, MAX_K = 64, 128, 2048

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64

# C ABI signatures, name -> (restype, argtypes)
SIGNATURES = {
    "dsa_indexer_topk": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "dsa_indexer_topk_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "dsa_indexer_topk_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "dsa_indexer_topk_unfused": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "dsa_indexer_scores": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _I64, _P]),
    "dsa_indexer_topk_from_scores": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P]),
    "dsa_indexer_topk_from_scores_noalloc": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P]),
    "dsa_indexer_math_control": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "dsa_sparse_attention": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P]),
    "dsa_sparse_attention_last_status": (_I, [_P]),
    "dsa_indexer_last_device_status": (_I, [_P, _P]),
    "dsa_indexer_last_repaired_rows": (_I, [_P, _P, _I]),
    "dsa_indexer_set_option": (_I, [_I, _I64]),
    "dsa_indexer_get_option": (_I64, [_I]),
    "dsa_indexer_profiled_main_ms": (ctypes.c_float, [_P]),
    "dsa_indexer_launch_count": (_I64, []),
    "dsa_indexer_version": (ctypes.c_char_p, []),
    "dsa_indexer_release": (_I, []),
}


class IndexerError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the library (building it first if the sources are newer)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path) or not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; build it with "
                               "python -m fp8_scoring_exact_gb300.build")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(fn, code):
    if code != DSA_OK:
        raise IndexerError(fn, code)


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _u8(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must hold e4m3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    return _dev(t, name)


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def indexer_topk(q, q_scale, k, k_scale, w, row_begin, row_end, K=2048, out=None, stream=None,
                 unfused=False):
    """Exact top-K indices per row; q [Q,64,128], k [N,128] e4m3; returns int32 [Q,K]."""
    q, k = _u8(q, "q"), _u8(k, "k")
    q_scale = _dev(q_scale, "q_scale", torch.float32)
    k_scale = _dev(k_scale, "k_scale", torch.float32)
    w = _dev(w, "w", torch.float32)
    row_begin = _dev(row_begin, "row_begin", torch.int32)
    row_end = _dev(row_end, "row_end", torch.int32)
    Q, N = q.shape[0], k.shape[0]
    if tuple(q.shape[1:]) != (HEADS, HEAD_DIM) or tuple(k.shape[1:]) != (HEAD_DIM,):
        raise ValueError("q must be [Q,64,128] and k [N,128]")
    if out is None:
        out = torch.empty((Q, K), dtype=torch.int32, device=q.device)
    _dev(out, "out", torch.int32)
    fn = "dsa_indexer_topk_unfused" if unfused else "dsa_indexer_topk"
    rc = getattr(lib(), fn)(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(row_begin),
                            _ptr(row_end), Q, N, K, _ptr(out), _stream_ptr(stream))
    _check(fn, rc)
    return out


def _host(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a CPU tensor")
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def indexer_topk_host(q, q_scale, k, k_scale, w, row_begin, row_end, K=2048, out=None, stream=None):
    """dsa_indexer_topk_host: the fused operator on CPU tensors (pinned memory lets the
    library overlap its copies with the scoring); returns int32 [Q,K] on the CPU.
    Synchronous."""
    q, k = _host(q, "q", torch.uint8), _host(k, "k", torch.uint8)
    q_scale = _host(q_scale, "q_scale", torch.float32)
    k_scale = _host(k_scale, "k_scale", torch.float32)
    w = _host(w, "w", torch.float32)
    row_begin = _host(row_begin, "row_begin", torch.int32)
    row_end = _host(row_end, "row_end", torch.int32)
    Q, N = q.shape[0], k.shape[0]
    if tuple(q.shape[1:]) != (HEADS, HEAD_DIM) or tuple(k.shape[1:]) != (HEAD_DIM,):
        raise ValueError("q must be [Q,64,128] and k [N,128]")
    if out is None:
        out = torch.empty((Q, K), dtype=torch.int32, pin_memory=q.is_pinned())
    _host(out, "out", torch.int32)
    rc = lib().dsa_indexer_topk_host(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(row_begin),
                                     _ptr(row_end), Q, N, K, _ptr(out), _stream_ptr(stream))
    _check("dsa_indexer_topk_host", rc)
    return out


def indexer_topk_unfused(*args, **kw):
    return indexer_topk(*args, unfused=True, **kw)


def indexer_topk_paged(q, q_scale, k_cache, k_cache_scale, w, block_table, seq_lens, K=2048, out=None,
                       stream=None):
    """Paged variant; q [B,next_n,64,128], k_cache [P,64,128]; returns int32 [B,next_n,K] of
    physical slots (block_table[b][s//64]*64 + s%64)."""
    q, k_cache = _u8(q, "q"), _u8(k_cache, "k_cache")
    q_scale = _dev(q_scale, "q_scale", torch.float32)
    k_cache_scale = _dev(k_cache_scale, "k_cache_scale", torch.float32)
    w = _dev(w, "w", torch.float32)
    block_table = _dev(block_table, "block_table", torch.int32)
    seq_lens = _dev(seq_lens, "seq_lens", torch.int32)
    B, nn = q.shape[0], q.shape[1]
    P = k_cache.shape[0]
    maxp = block_table.shape[1]
    if out is None:
        out = torch.empty((B, nn, K), dtype=torch.int32, device=q.device)
    _dev(out, "out", torch.int32)
    rc = lib().dsa_indexer_topk_paged(_ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(k_cache_scale), _ptr(w),
                                      _ptr(block_table), _ptr(seq_lens), B, nn, maxp, P, K, _ptr(out),
                                      _stream_ptr(stream))
    _check("dsa_indexer_topk_paged", rc)
    return out


def indexer_scores(q, q_scale, k, k_scale, w, row_begin, row_end, scores=None, stream=None):
    """FP32 scores [Q, ld] (valid entries of every row; -inf elsewhere in touched tiles)."""
    q, k = _u8(q, "q"), _u8(k, "k")
    Q, N = q.shape[0], k.shape[0]
    if scores is None:
        ld = (N + 3) // 4 * 4
        scores = torch.full((Q, ld), float("nan"), dtype=torch.float32, device=q.device)
    _dev(scores, "scores", torch.float32)
    rc = lib().dsa_indexer_scores(_ptr(q), _ptr(_dev(q_scale, "q_scale", torch.float32)), _ptr(k),
                                  _ptr(_dev(k_scale, "k_scale", torch.float32)),
                                  _ptr(_dev(w, "w", torch.float32)),
                                  _ptr(_dev(row_begin, "row_begin", torch.int32)),
                                  _ptr(_dev(row_end, "row_end", torch.int32)), Q, N, _ptr(scores),
                                  scores.shape[1], _stream_ptr(stream))
    _check("dsa_indexer_scores", rc)
    return scores


def topk_from_scores(scores, row_begin, row_end, K=2048, N=None, out=None, stream=None):
    """Exact top-K of each row of an fp32 score matrix over [row_begin, row_end)."""
    scores = _dev(scores, "scores", torch.float32)
    Q, ld = scores.shape
    N = ld if N is None else N
    if out is None:
        out = torch.empty((Q, K), dtype=torch.int32, device=scores.device)
    rc = lib().dsa_indexer_topk_from_scores(_ptr(scores), ld, _ptr(_dev(row_begin, "row_begin", torch.int32)),
                                            _ptr(_dev(row_end, "row_end", torch.int32)), Q, N, K,
                                            _ptr(_dev(out, "out", torch.int32)), _stream_ptr(stream))
    _check("dsa_indexer_topk_from_scores", rc)
    return out


def topk_from_scores_noalloc(scores, row_begin, row_end, K=2048, N=None, out=None, stream=None):
    """Same as topk_from_scores, through the entry point that allocates nothing
    (its scratch is a fixed array in device memory; at most 4096 rows).  The
    output tensor is the caller's: pass `out` to avoid even that allocation."""
    scores = _dev(scores, "scores", torch.float32)
    Q, ld = scores.shape
    N = ld if N is None else N
    if out is None:
        out = torch.empty((Q, K), dtype=torch.int32, device=scores.device)
    rc = lib().dsa_indexer_topk_from_scores_noalloc(_ptr(scores), ld,
                                                    _ptr(_dev(row_begin, "row_begin", torch.int32)),
                                                    _ptr(_dev(row_end, "row_end", torch.int32)), Q, N, K,
                                                    _ptr(_dev(out, "out", torch.int32)), _stream_ptr(stream))
    _check("dsa_indexer_topk_from_scores_noalloc", rc)
    return out


def math_control(q, q_scale, k, k_scale, w, row_begin, row_end, K=2048, checksum=None, stream=None):
    """The math-only control (a measurement): the fused call's main scorer with its
    score reduction and candidate filter removed.  Returns the checksum tensor
    (one device float, added to)."""
    q, k = _u8(q, "q"), _u8(k, "k")
    if checksum is None:
        checksum = torch.zeros(1, dtype=torch.float32, device=q.device)
    rc = lib().dsa_indexer_math_control(_ptr(q), _ptr(_dev(q_scale, "q_scale", torch.float32)), _ptr(k),
                                        _ptr(_dev(k_scale, "k_scale", torch.float32)),
                                        _ptr(_dev(w, "w", torch.float32)),
                                        _ptr(_dev(row_begin, "row_begin", torch.int32)),
                                        _ptr(_dev(row_end, "row_end", torch.int32)), q.shape[0], k.shape[0], K,
                                        _ptr(_dev(checksum, "checksum", torch.float32)), _stream_ptr(stream))
    _check("dsa_indexer_math_control", rc)
    return checksum


def sparse_attention(q_nope, q_pe, ckv, kpe, indices, sm_scale, out=None, lse=None, stream=None):
    """Sparse-attention decode over top-K slots: q_nope [T,H,512], q_pe [T,H,64] bf16,
    ckv [S,512], kpe [S,64] bf16 (slot-major cache), indices [T,K] int32 (-1: padding).
    Returns (out [T,H,512] bf16, lse [T,H] fp32, base 2)."""
    q_nope = _dev(q_nope, "q_nope", torch.bfloat16)
    q_pe = _dev(q_pe, "q_pe", torch.bfloat16)
    ckv = _dev(ckv, "ckv", torch.bfloat16)
    kpe = _dev(kpe, "kpe", torch.bfloat16)
    indices = _dev(indices, "indices", torch.int32)
    T, H = q_nope.shape[0], q_nope.shape[1]
    if tuple(q_nope.shape[2:]) != (512,) or tuple(q_pe.shape) != (T, H, 64):
        raise ValueError("q_nope must be [T,H,512] and q_pe [T,H,64]")
    ckv2, kpe2 = ckv.reshape(-1, 512), kpe.reshape(-1, 64)
    if ckv2.shape[0] != kpe2.shape[0]:
        raise ValueError("ckv and kpe must hold the same slots")
    K = indices.shape[-1]
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_nope.device)
    rc = lib().dsa_sparse_attention(_ptr(q_nope), _ptr(q_pe), _ptr(ckv2), _ptr(kpe2), _ptr(indices), T, H, K,
                                    ckv2.shape[0], float(sm_scale), _ptr(_dev(out, "out", torch.bfloat16)),
                                    _ptr(_dev(lse, "lse", torch.float32)), _stream_ptr(stream))
    _check("dsa_sparse_attention", rc)
    return out, lse


def sparse_attention_last_status(stream=None) -> int:
    return int(lib().dsa_sparse_attention_last_status(_stream_ptr(stream)))


def last_device_status(stream=None):
    """(status code, {underflow, overflow, trivial, candidates}) of the last call on the stream."""
    buf = (ctypes.c_int32 * 4)()
    rc = lib().dsa_indexer_last_device_status(_stream_ptr(stream), buf)
    return rc, {"underflow": buf[0], "overflow": buf[1], "trivial": buf[2], "candidates": buf[3]}


def last_repaired_rows(stream=None, cap=1 << 20):
    """Row ids the last selecting call on the stream sent to exact repair."""
    buf = (ctypes.c_int32 * cap)()
    n = lib().dsa_indexer_last_repaired_rows(_stream_ptr(stream), buf, cap)
    if n < 0:
        raise IndexerError("dsa_indexer_last_repaired_rows", n)
    return [buf[i] for i in range(min(n, cap))]


def set_option(name: str, value: int):
    _check("dsa_indexer_set_option", lib().dsa_indexer_set_option(OPTIONS[name], int(value)))


def get_option(name: str) -> int:
    return int(lib().dsa_indexer_get_option(OPTIONS[name]))


def profiled_main_ms(stream=None) -> float:
    return float(lib().dsa_indexer_profiled_main_ms(_stream_ptr(stream)))


def launch_count() -> int:
    return int(lib().dsa_indexer_launch_count())


def version() -> str:
    return lib().dsa_indexer_version().decode()


def release():
    _check("dsa_indexer_release", lib().dsa_indexer_release())
