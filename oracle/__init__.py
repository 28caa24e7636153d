"""fp64 CPU oracle for paged MLA decode — test infrastructure only.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy/torch CPU buffers through ctypes.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
it.  It shares nothing with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_libs = {}

D_QK = 576
D_V = 512


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE semantics are part of the definition)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src,
                               "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


_active = [None]  # path of the library the module functions use (None = the default build)


class use_library:
    """Context manager: route the module functions to another build (mutation tests)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.prev = _active[0]
        _active[0] = self.path

    def __exit__(self, *exc):
        _active[0] = self.prev


def _load():
    path = _active[0] or build()
    with _lock:
        lib = _libs.get(path)
        if lib is None:
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            D = ctypes.c_double
            common = [P, P, I, I, I, P, I, P, I, I, I, P, I, D, I, P, P, P, I64]
            lib.oracle_mla_decode.argtypes = common + [P, P, I]
            lib.oracle_mla_decode.restype = I
            lib.oracle_mla_partial.argtypes = common + [I64, I64, P, P, I]
            lib.oracle_mla_partial.restype = I
            lib.oracle_lse_merge.argtypes = [I, P, P, P, P]
            lib.oracle_lse_merge.restype = None
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = D
            lib.oracle_dequant_row.argtypes = [P, P]
            lib.oracle_dequant_row.restype = None
            lib.oracle_dequant_row_token_scale.argtypes = [P, ctypes.c_float, P]
            lib.oracle_dequant_row_token_scale.restype = None
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_fp8_quantize_row.argtypes = [P, P]
            lib.oracle_fp8_quantize_row.restype = None
            lib.oracle_fp8_cache_store.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, P]
            lib.oracle_fp8_cache_store.restype = ctypes.c_int64
            lib.oracle_sparse_prefill.argtypes = [P, P, I64, P, I, I, D, P, I64, P, P, I]
            lib.oracle_sparse_prefill.restype = None
            idx_common = [P, P, P, I, P, I, P, P, I, I, P, I, P, I]
            lib.oracle_index_scores.argtypes = idx_common + [I64, P]
            lib.oracle_index_scores.restype = I
            lib.oracle_index_topk.argtypes = idx_common + [I, P]
            lib.oracle_index_topk.restype = I
            _libs[path] = lib
    return lib


def _np(x, dtype):
    """Contiguous numpy view of a CPU tensor/array reinterpreted as ``dtype``."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().contiguous().cpu()
        import torch
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        if x.dtype == torch.float8_e4m3fn:
            x = x.view(torch.uint8)
        x = x.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != dtype:
        x = x.view(dtype) if x.dtype.itemsize == np.dtype(dtype).itemsize else x.astype(dtype)
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _args(q, kvcache, block_table, cache_seqlens, sm_scale, is_causal, indices, topk_lengths=None,
          kv_scales=None):
    qn = _np(q, np.uint16)
    batch, s_q, h_q, d = qn.shape
    assert d == D_QK
    kv = kvcache
    scales = None if kv_scales is None else np.ascontiguousarray(_np(kv_scales, np.float32))
    lens = None if topk_lengths is None else np.ascontiguousarray(_np(topk_lengths, np.int32))
    if hasattr(kv, "dtype") and str(kv.dtype) in ("torch.uint8", "uint8") and scales is not None:
        kvn = _np(kv, np.uint8)
        is_fp8 = 2
        assert kvn.shape[-1] == 640
    elif hasattr(kv, "dtype") and str(kv.dtype) in ("torch.uint8", "uint8"):
        kvn = _np(kv, np.uint8)
        is_fp8 = 1
        assert kvn.shape[-1] == 656
    else:
        kvn = _np(kv, np.uint16)
        is_fp8 = 0
        assert kvn.shape[-1] == D_QK
    num_pages, page_size = kvn.shape[0], kvn.shape[1]
    bt = _np(block_table, np.int32)
    sl = _np(cache_seqlens, np.int32)
    idx = _np(indices, np.int32)
    topk = 0 if idx is None else idx.shape[-1]
    keep = (qn, kvn, bt, sl, idx, scales, lens)
    a = [_ptr(qn), _ptr(kvn), is_fp8, num_pages, page_size, _ptr(bt), bt.shape[1], _ptr(sl), batch,
         s_q, h_q, _ptr(idx), topk, float(sm_scale), int(bool(is_causal)), _ptr(lens), _ptr(scales)]
    return a, keep, (batch, s_q, h_q)


def mla_decode(q, kvcache, block_table, cache_seqlens, sm_scale, is_causal=False, indices=None,
               rows=None, n_threads=None, topk_lengths=None, kv_scales=None):
    """Oracle decode.  Returns (out float64 [n_rows, 512], lse float64 [n_rows]).

    ``rows`` selects flat output rows ((b*s_q + i)*h_q + h); None = all rows
    (then out is reshaped to [b, s_q, h_q, 512] and lse to [b, s_q, h_q]).
    """
    lib = _load()
    a, keep, (batch, s_q, h_q) = _args(q, kvcache, block_table, cache_seqlens, sm_scale, is_causal,
                                       indices, topk_lengths, kv_scales)
    all_rows = rows is None
    r = None if all_rows else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = batch * s_q * h_q if all_rows else r.shape[0]
    out = np.zeros((n, D_V), np.float64)
    lse = np.zeros((n,), np.float64)
    nt = n_threads or os.cpu_count() or 1
    rc = lib.oracle_mla_decode(*a, _ptr(r), n, _ptr(out), _ptr(lse), int(nt))
    if rc != 0:
        raise ValueError("oracle: block_table holds an entry outside [0, num_pages)")
    del keep
    if all_rows:
        return out.reshape(batch, s_q, h_q, D_V), lse.reshape(batch, s_q, h_q)
    return out, lse


def mla_partial(q, kvcache, block_table, cache_seqlens, sm_scale, k0, k1, is_causal=False,
                indices=None, rows=None, n_threads=None, topk_lengths=None, kv_scales=None):
    """Oracle restricted to key-set positions [k0, k1) of every row (flat rows)."""
    lib = _load()
    a, keep, (batch, s_q, h_q) = _args(q, kvcache, block_table, cache_seqlens, sm_scale, is_causal,
                                       indices, topk_lengths, kv_scales)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = batch * s_q * h_q if r is None else r.shape[0]
    out = np.zeros((n, D_V), np.float64)
    lse = np.zeros((n,), np.float64)
    nt = n_threads or os.cpu_count() or 1
    rc = lib.oracle_mla_partial(*a, _ptr(r), n, int(k0), int(k1), _ptr(out), _ptr(lse), int(nt))
    if rc != 0:
        raise ValueError("oracle: block_table holds an entry outside [0, num_pages)")
    del keep
    return out, lse


def lse_merge(outs, lses):
    """Merge partials of one row: outs [n, 512], lses [n] -> (out [512], lse)."""
    lib = _load()
    o = np.ascontiguousarray(np.asarray(outs, np.float64))
    l = np.ascontiguousarray(np.asarray(lses, np.float64))
    out = np.zeros((D_V,), np.float64)
    lse = np.zeros((1,), np.float64)
    lib.oracle_lse_merge(int(l.shape[0]), _ptr(o), _ptr(l), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def e4m3_to_double(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(ctypes.c_uint8(code)))


def dequant_row(row656) -> np.ndarray:
    """Dequantise one 656-byte FP8 token row into 576 float64 (bf16-valued) numbers."""
    r = np.ascontiguousarray(np.asarray(row656, np.uint8))
    assert r.shape == (656,)
    k = np.zeros((D_QK,), np.float64)
    _load().oracle_dequant_row(_ptr(r), _ptr(k))
    return k


def e4m3_from_float(q: float) -> int:
    """float32 value -> E4M3 code: nearest value, ties to the even code, saturating at 448."""
    return int(_load().oracle_e4m3_from_float(ctypes.c_float(q)))


def fp8_quantize_row(x576) -> np.ndarray:
    """One token (576 bf16 values, torch bf16 tensor) -> its 656-byte FP8 cache row."""
    xb = np.ascontiguousarray(_np(x576, np.uint16).reshape(-1))
    assert xb.size == 576
    row = np.zeros(656, dtype=np.uint8)
    _load().oracle_fp8_quantize_row(_ptr(xb), _ptr(row))
    return row


def fp8_cache_store(x, input_row_offsets, cache_lengths, block_table, kvcache):
    """Ragged FP8 cache write into a copy of `kvcache` (uint8 [pages, page_size, 1, 656]).
    Returns (new cache as a numpy array, number of skipped tokens)."""
    xb = np.ascontiguousarray(_np(x, np.uint16))
    offs = np.ascontiguousarray(_np(input_row_offsets, np.int32))
    lens = np.ascontiguousarray(_np(cache_lengths, np.int32))
    bt = np.ascontiguousarray(_np(block_table, np.int32))
    cache = np.array(_np(kvcache, np.uint8), copy=True)
    batch = int(lens.shape[0])
    skipped = _load().oracle_fp8_cache_store(_ptr(xb), _ptr(offs), _ptr(lens), _ptr(bt), int(bt.shape[1]), batch,
                                              int(cache.shape[0]), int(cache.shape[1]), _ptr(cache))
    return cache, int(skipped)


def sparse_prefill(q, kv, indices, sm_scale, rows=None, n_threads=None):
    """Oracle sparse prefill: q [s_q, h_q, 576] bf16, kv [s_kv, 576] (or [s_kv, 1, 576]) bf16,
    indices [s_q, topk] (or [s_q, 1, topk]) int32.  Returns (out float64, lse float64):
    [s_q, h_q, 512] and [s_q, h_q] for all rows, else [n, 512] and [n] for the listed
    flat rows (i * h_q + h)."""
    lib = _load()
    qn = _np(q, np.uint16)
    s_q, h_q, d = qn.shape
    assert d == D_QK
    kvn = _np(kv, np.uint16).reshape(-1, D_QK)
    idx = _np(indices, np.int32).reshape(s_q, -1)
    topk = idx.shape[1]
    all_rows = rows is None
    r = None if all_rows else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = s_q * h_q if all_rows else r.shape[0]
    out = np.zeros((n, D_V), np.float64)
    lse = np.zeros((n,), np.float64)
    nt = n_threads or os.cpu_count() or 1
    lib.oracle_sparse_prefill(_ptr(qn), _ptr(kvn), int(kvn.shape[0]), _ptr(idx), int(topk), int(h_q),
                              float(sm_scale), _ptr(r), int(n), _ptr(out), _ptr(lse), int(nt))
    if all_rows:
        return out.reshape(s_q, h_q, D_V), lse.reshape(s_q, h_q)
    return out, lse


def _index_args(inp):
    qc = _np(inp.q_codes, np.uint8)
    qs = _np(inp.q_scales, np.float32)
    w = _np(inp.weights, np.float32)
    offs = _np(inp.row_offsets, np.int32)
    kc = _np(inp.k_codes, np.uint8)
    ks = _np(inp.k_scales, np.float32)
    bt = _np(inp.block_table, np.int32)
    sl = _np(inp.cache_seqlens, np.int32)
    h_idx = qc.shape[1]
    assert qc.shape[-1] == 128 and kc.shape[-1] == 128
    keep = (qc, qs, w, offs, kc, ks, bt, sl)
    a = [_ptr(qc), _ptr(qs), _ptr(w), h_idx, _ptr(offs), int(sl.shape[0]), _ptr(kc), _ptr(ks),
         int(kc.shape[0]), int(kc.shape[1]), _ptr(bt), int(bt.shape[1]), _ptr(sl), int(bool(inp.relu))]
    return a, keep, int(offs[-1])


def index_scores(inp, width=None):
    """Indexer scores [num_tokens, width] float64 (-inf where a key is not visible)."""
    lib = _load()
    a, keep, n = _index_args(inp)
    if width is None:
        width = max(1, int(_np(inp.cache_seqlens, np.int32).max()))
    out = np.zeros((n, width), np.float64)
    if lib.oracle_index_scores(*a, int(width), _ptr(out)) != 0:
        raise ValueError("oracle: block_table holds an entry outside [0, num_pages)")
    del keep
    return out


def index_topk(inp, topk=None):
    """Indexer top-k key ids [num_tokens, topk] int32 (descending score, ties to the smaller id, -1 fill)."""
    lib = _load()
    a, keep, n = _index_args(inp)
    k = int(inp.topk if topk is None else topk)
    out = np.zeros((n, k), np.int32)
    if lib.oracle_index_topk(*a, k, _ptr(out)) != 0:
        raise ValueError("oracle: block_table holds an entry outside [0, num_pages)")
    del keep
    return out


def dequant_row_token_scale(row640, scale) -> np.ndarray:
    """Dequantise one 640-byte per-token-scale FP8 row into 576 float64 (bf16-valued) numbers."""
    r = np.ascontiguousarray(np.asarray(row640, np.uint8))
    assert r.shape == (640,)
    k = np.zeros((D_QK,), np.float64)
    _load().oracle_dequant_row_token_scale(_ptr(r), ctypes.c_float(float(scale)), _ptr(k))
    return k
