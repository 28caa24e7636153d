"""Paged MLA decode for GB300 — thin Python binding over the libmla C ABI.

The binding only marshals arguments: it checks tensor dtypes/devices/shapes
(raising ValueError that names the argument, the MAX kernel-wrapper
convention), allocates outputs and scratch with torch when the caller does
not pass them, and calls the C entry points on the current CUDA stream.
Every step of decode runs in the library's CUDA kernels; there is no other
code path.  If ``libmla.so`` has not been built, every call raises.

    sched, num_splits = get_metadata(cache_seqlens, h_q=..., s_q=..., topk=..., is_fp8=...)
    out, lse = decode(q, kvcache, block_table, cache_seqlens, sm_scale,
                      sched, num_splits, is_causal=..., indices=...)
    out, lse = sparse_prefill(q, kv, indices, sm_scale)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import builder as _build

D_QK = 576
D_V = 512
PAGE_SIZE = 64
FP8_ROW_BYTES = 656

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
                4: "MLA_ERR_CUDA", 5: "MLA_ERR_DEVICE_BOUNDS", 6: "MLA_ERR_DEVICE_TIMEOUT"}
DEVICE_BAD_PAGE = 0x1
DEVICE_TIMEOUT = 0x2
DEVICE_BAD_SCHEDULE = 0x4

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class DecodeArgs(ctypes.Structure):
    """Mirror of ``mla_decode_args`` in include/mla.h."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("batch", ctypes.c_int), ("s_q", ctypes.c_int), ("h_q", ctypes.c_int),
        ("kvcache", ctypes.c_void_p), ("num_pages", ctypes.c_int), ("page_size", ctypes.c_int),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int),
        ("cache_seqlens", ctypes.c_void_p), ("sm_scale", ctypes.c_float), ("is_causal", ctypes.c_int),
        ("is_fp8", ctypes.c_int), ("indices", ctypes.c_void_p), ("topk", ctypes.c_int),
        ("sched", ctypes.c_void_p), ("num_splits", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("kv_scales", ctypes.c_void_p), ("topk_lengths", ctypes.c_void_p),
    ]


class SparsePrefillArgs(ctypes.Structure):
    """Mirror of ``mla_sparse_prefill_args`` in include/mla.h."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("s_q", ctypes.c_int), ("h_q", ctypes.c_int),
        ("kv", ctypes.c_void_p), ("s_kv", ctypes.c_int),
        ("indices", ctypes.c_void_p), ("topk", ctypes.c_int), ("sm_scale", ctypes.c_float),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
    ]


class IndexTopkArgs(ctypes.Structure):
    """Mirror of ``mla_index_topk_args`` in include/mla.h."""
    _fields_ = [
        ("q_codes", ctypes.c_void_p), ("q_scales", ctypes.c_void_p), ("weights", ctypes.c_void_p),
        ("num_tokens", ctypes.c_int), ("h_idx", ctypes.c_int), ("row_offsets", ctypes.c_void_p),
        ("batch", ctypes.c_int), ("max_new_tokens", ctypes.c_int), ("k_codes", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p), ("num_pages", ctypes.c_int), ("page_size", ctypes.c_int),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int),
        ("cache_seqlens", ctypes.c_void_p), ("relu", ctypes.c_int), ("topk", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t), ("indices", ctypes.c_void_p),
    ]


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libmla.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libmla.so not found at {path}: run paged_mla_decode_07_gb300.build.build()")
            L = ctypes.CDLL(path)
            I, P, S = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            L.mla_abi_version.restype = I
            L.mla_last_error.restype = ctypes.c_char_p
            L.mla_metadata_size.argtypes = [I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]
            L.mla_metadata_size.restype = I
            L.mla_workspace_size.argtypes = [I, I, I, I, I, ctypes.POINTER(S)]
            L.mla_workspace_size.restype = I
            L.mla_get_metadata.argtypes = [P, I, I, I, I, I, P, P, P]
            L.mla_get_metadata.restype = I
            L.mla_test_hooks.argtypes = [I, I]
            L.mla_test_hooks.restype = I
            L.mla_decode.argtypes = [ctypes.POINTER(DecodeArgs), P]
            L.mla_decode.restype = I
            L.mla_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            L.mla_fp8_cache_store.argtypes = [P, I, P, P, I, P, I, P, I, I, P]
            L.mla_fp8_cache_store.restype = I
            L.mla_get_device_status.restype = I
            L.mla_sparse_prefill_workspace_size.argtypes = [I, I, I, ctypes.POINTER(S)]
            L.mla_sparse_prefill_workspace_size.restype = I
            L.mla_sparse_prefill.argtypes = [ctypes.POINTER(SparsePrefillArgs), P]
            L.mla_sparse_prefill.restype = I
            L.mla_index_topk_workspace_size.argtypes = [I, I, ctypes.POINTER(S)]
            L.mla_index_topk_workspace_size.restype = I
            L.mla_index_topk.argtypes = [ctypes.POINTER(IndexTopkArgs), P]
            L.mla_index_topk.restype = I
            _lib = L
    return _lib


def last_error() -> str:
    return lib().mla_last_error().decode()


def _check(status: int):
    if status != MLA_OK:
        msg = last_error()
        if status in (1, 2, 3):
            raise ValueError(f"{STATUS_NAMES[status]}: {msg}")
        raise MLAError(status, msg)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype} (got {t.dtype})")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device} (got {t.device})")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions (got {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def metadata_size(batch: int, *, h_q: int, s_q: int, topk: int, is_fp8: bool) -> Tuple[int, int]:
    """(sched int32 elements, num_splits int32 elements) for one decode configuration."""
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(lib().mla_metadata_size(batch, h_q, s_q, topk, int(bool(is_fp8)), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def workspace_size(batch: int, *, h_q: int, s_q: int, topk: int, is_fp8: bool) -> int:
    """Scratch bytes mla_decode needs for one decode configuration."""
    n = ctypes.c_size_t()
    _check(lib().mla_workspace_size(batch, h_q, s_q, topk, int(bool(is_fp8)), ctypes.byref(n)))
    return n.value


def get_metadata(cache_seqlens: torch.Tensor, *, h_q: int, s_q: int, topk: int, is_fp8: bool, stream=None,
                 sched: Optional[torch.Tensor] = None, num_splits: Optional[torch.Tensor] = None):
    """Tile schedule for one decode step; reuse it for every layer of the step.  The keywords name
    the decode configuration (topk = 0: dense; is_fp8: the cache format) that decode() will run."""
    _need(cache_seqlens, "cache_seqlens", torch.int32, ndim=1)
    if not cache_seqlens.is_cuda:
        raise ValueError("cache_seqlens must be a CUDA tensor")
    dev = cache_seqlens.device
    batch = cache_seqlens.shape[0]
    ns, nn = metadata_size(batch, h_q=h_q, s_q=s_q, topk=topk, is_fp8=is_fp8)
    if sched is None:
        sched = torch.empty(ns, dtype=torch.int32, device=dev)
    if num_splits is None:
        num_splits = torch.empty(nn, dtype=torch.int32, device=dev)
    if sched.numel() < ns or num_splits.numel() < nn:
        raise ValueError("sched / num_splits buffers are too small")
    _check(lib().mla_get_metadata(ctypes.c_void_p(cache_seqlens.data_ptr()), batch, h_q, s_q, topk,
                                  int(bool(is_fp8)), ctypes.c_void_p(sched.data_ptr()),
                                  ctypes.c_void_p(num_splits.data_ptr()), _stream(stream)))
    return sched, num_splits


def set_test_hooks(num_parts: int = 0, debug_stall: bool = False) -> None:
    """Library test hooks (mla_test_hooks): force the schedule's part count (0 = default) and make
    the decode kernel's softmax role stall so that its bounded wait runs out."""
    _check(lib().mla_test_hooks(int(num_parts), int(bool(debug_stall))))


def decode(q: torch.Tensor, kvcache: torch.Tensor, block_table: torch.Tensor, cache_seqlens: torch.Tensor,
           sm_scale: float, sched: torch.Tensor, num_splits: torch.Tensor, is_causal: bool = False,
           indices: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None,
           kv_scales: Optional[torch.Tensor] = None, topk_lengths: Optional[torch.Tensor] = None):
    """Paged MLA decode.  Returns (out bf16 [b, s_q, h_q, 512], lse fp32 [b, s_q, h_q], base 2).
    kv_scales (fp32 [num_pages, 64]) selects the FP8 cache with one scale per token (640-byte rows);
    topk_lengths (int32 [b, s_q]) limits each sparse row to its first index slots."""
    _need(q, "q", torch.bfloat16, ndim=4)
    if not q.is_cuda:
        raise ValueError("q must be a CUDA tensor")
    dev = q.device
    batch, s_q, h_q, d = q.shape
    if d != D_QK:
        raise ValueError(f"q must have last dimension {D_QK} (got {d})")
    is_fp8 = kvcache.dtype == torch.uint8
    if is_fp8:
        _need(kvcache, "kvcache", torch.uint8, dev, 4)
        row = 640 if kv_scales is not None else FP8_ROW_BYTES
        if kvcache.shape[-1] != row or kvcache.shape[2] != 1:
            raise ValueError(f"FP8 kvcache must be [pages, page_size, 1, {row}]")
        if kv_scales is not None:
            _need(kv_scales, "kv_scales", torch.float32, dev)
            if kv_scales.numel() != kvcache.shape[0] * kvcache.shape[1]:
                raise ValueError("kv_scales must hold one scale per cached token")
    else:
        _need(kvcache, "kvcache", torch.bfloat16, dev, 4)
        if kvcache.shape[-1] != D_QK or kvcache.shape[2] != 1:
            raise ValueError(f"bf16 kvcache must be [pages, page_size, 1, {D_QK}]")
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, dev, 1)
    if block_table.shape[0] != batch or cache_seqlens.shape[0] != batch:
        raise ValueError("block_table and cache_seqlens must have batch rows")
    topk = 0
    if indices is not None:
        _need(indices, "indices", torch.int32, dev, 3)
        if tuple(indices.shape[:2]) != (batch, s_q):
            raise ValueError(f"indices must be [batch, s_q, topk] (got {tuple(indices.shape)})")
        topk = indices.shape[2]
    if topk_lengths is not None:
        _need(topk_lengths, "topk_lengths", torch.int32, dev)
        if topk_lengths.numel() != batch * s_q:
            raise ValueError("topk_lengths must be [batch, s_q]")
    _need(sched, "sched", torch.int32, dev)
    _need(num_splits, "num_splits", torch.int32, dev)
    if out is None:
        out = torch.empty((batch, s_q, h_q, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((batch, s_q, h_q), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    if out.numel() != batch * s_q * h_q * D_V or lse.numel() != batch * s_q * h_q:
        raise ValueError("out / lse have the wrong size")
    if workspace is None:
        workspace = torch.empty(max(workspace_size(batch, h_q=h_q, s_q=s_q, topk=topk, is_fp8=is_fp8), 256),
                                dtype=torch.uint8, device=dev)
    a = DecodeArgs()
    a.q = q.data_ptr()
    a.batch, a.s_q, a.h_q = batch, s_q, h_q
    a.kvcache = kvcache.data_ptr()
    a.num_pages, a.page_size = kvcache.shape[0], kvcache.shape[1]
    a.block_table = block_table.data_ptr()
    a.block_table_stride = block_table.shape[1]
    a.cache_seqlens = cache_seqlens.data_ptr()
    a.sm_scale = float(sm_scale)
    a.is_causal = int(bool(is_causal))
    a.is_fp8 = int(is_fp8)
    a.indices = indices.data_ptr() if indices is not None else None
    a.topk = topk
    a.sched = sched.data_ptr()
    a.num_splits = num_splits.data_ptr()
    a.workspace = workspace.data_ptr()
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    a.out = out.data_ptr()
    a.lse = lse.data_ptr()
    a.kv_scales = kv_scales.data_ptr() if kv_scales is not None else None
    a.topk_lengths = topk_lengths.data_ptr() if topk_lengths is not None else None
    _check(lib().mla_decode(ctypes.byref(a), _stream(stream)))
    return out.view(batch, s_q, h_q, D_V), lse.view(batch, s_q, h_q)


def fp8_cache_store(x: torch.Tensor, input_row_offsets: torch.Tensor, cache_lengths: torch.Tensor,
                    block_table: torch.Tensor, kvcache: torch.Tensor, stream=None) -> None:
    """Quantise new tokens into the FP8 cache rows (mla_fp8_cache_store).

    x bf16 [num_tokens, 576]; input_row_offsets int32 [batch + 1]; cache_lengths int32 [batch];
    block_table int32 [batch, stride]; kvcache uint8 [num_pages, 64, 1, 656] (written in place).
    """
    if not torch.is_tensor(x) or x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    dev = x.device
    _need(x, "x", torch.bfloat16, dev, 2)
    if x.shape[1] != 576:
        raise ValueError(f"x must be [num_tokens, 576] (got {tuple(x.shape)})")
    _need(input_row_offsets, "input_row_offsets", torch.int32, dev, 1)
    _need(cache_lengths, "cache_lengths", torch.int32, dev, 1)
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(kvcache, "kvcache", torch.uint8, dev, 4)
    batch = cache_lengths.shape[0]
    if input_row_offsets.shape[0] != batch + 1 or block_table.shape[0] != batch:
        raise ValueError("input_row_offsets must have batch + 1 entries and block_table batch rows")
    if kvcache.shape[2] != 1 or kvcache.shape[3] != 656:
        raise ValueError(f"kvcache must be [num_pages, page_size, 1, 656] (got {tuple(kvcache.shape)})")
    _check(lib().mla_fp8_cache_store(x.data_ptr(), x.shape[0], input_row_offsets.data_ptr(),
                                     cache_lengths.data_ptr(), batch, block_table.data_ptr(),
                                     block_table.shape[1], kvcache.data_ptr(), kvcache.shape[0], kvcache.shape[1],
                                     _stream(stream)))


def sparse_prefill_workspace_size(s_q: int, h_q: int, topk: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().mla_sparse_prefill_workspace_size(s_q, h_q, topk, ctypes.byref(n)))
    return n.value


def sparse_prefill(q: torch.Tensor, kv: torch.Tensor, indices: torch.Tensor, sm_scale: float,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None):
    """Sparse prefill (mla_sparse_prefill).  q bf16 [s_q, h_q, 576]; kv bf16 [s_kv, 576] or
    [s_kv, 1, 576]; indices int32 [s_q, topk] or [s_q, 1, topk].  Returns (out bf16
    [s_q, h_q, 512], lse fp32 [s_q, h_q], base 2)."""
    if not torch.is_tensor(q) or q.device.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    s_q, h_q, d = q.shape
    if d != D_QK:
        raise ValueError(f"q must have last dimension {D_QK} (got {d})")
    _need(kv, "kv", torch.bfloat16, dev)
    if kv.dim() == 3:
        if kv.shape[1] != 1:
            raise ValueError(f"kv must have one KV head (got {tuple(kv.shape)})")
        kv = kv.view(kv.shape[0], kv.shape[2])
    if kv.dim() != 2 or kv.shape[1] != D_QK:
        raise ValueError(f"kv must be [s_kv, {D_QK}] (got {tuple(kv.shape)})")
    _need(indices, "indices", torch.int32, dev)
    if indices.dim() == 3:
        if indices.shape[1] != 1:
            raise ValueError(f"indices must have one KV head (got {tuple(indices.shape)})")
        indices = indices.view(indices.shape[0], indices.shape[2])
    if indices.dim() != 2 or indices.shape[0] != s_q:
        raise ValueError(f"indices must be [s_q, topk] (got {tuple(indices.shape)})")
    topk = indices.shape[1]
    if out is None:
        out = torch.empty((s_q, h_q, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    if out.numel() != s_q * h_q * D_V or lse.numel() != s_q * h_q:
        raise ValueError("out / lse have the wrong size")
    if workspace is None:
        workspace = torch.empty(sparse_prefill_workspace_size(s_q, h_q, topk), dtype=torch.uint8, device=dev)
    a = SparsePrefillArgs()
    a.q = q.data_ptr()
    a.s_q, a.h_q = s_q, h_q
    a.kv = kv.data_ptr()
    a.s_kv = kv.shape[0]
    a.indices = indices.data_ptr()
    a.topk = topk
    a.sm_scale = float(sm_scale)
    a.workspace = workspace.data_ptr()
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    a.out = out.data_ptr()
    a.lse = lse.data_ptr()
    _check(lib().mla_sparse_prefill(ctypes.byref(a), _stream(stream)))
    return out.view(s_q, h_q, D_V), lse.view(s_q, h_q)


def index_topk_workspace_size(num_tokens: int, block_table_stride: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().mla_index_topk_workspace_size(num_tokens, block_table_stride, ctypes.byref(n)))
    return n.value


def index_topk(q_codes: torch.Tensor, q_scales: torch.Tensor, weights: torch.Tensor, row_offsets: torch.Tensor,
               k_codes: torch.Tensor, k_scales: torch.Tensor, block_table: torch.Tensor, cache_seqlens: torch.Tensor,
               topk: int, relu: bool = False, max_new_tokens: Optional[int] = None,
               indices: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """FP8 top-k indexer (mla_index_topk).  q_codes uint8 [T, h_idx, 128] (E4M3 codes), q_scales and
    weights fp32 [T, h_idx], row_offsets int32 [batch + 1], k_codes uint8 [num_pages, 64, 128],
    k_scales fp32 [num_pages, 64], block_table int32 [batch, stride], cache_seqlens int32 [batch].
    Returns int32 [T, topk] key ids (descending score, -1 fill).  Without max_new_tokens the
    largest row count is read from row_offsets (one device-to-host copy)."""
    if not torch.is_tensor(q_codes) or q_codes.device.type != "cuda":
        raise ValueError("q_codes must be a CUDA tensor")
    dev = q_codes.device
    _need(q_codes, "q_codes", torch.uint8, dev, 3)
    T, h_idx, d = q_codes.shape
    if d != 128:
        raise ValueError(f"q_codes must be [num_tokens, h_idx, 128] (got {tuple(q_codes.shape)})")
    _need(q_scales, "q_scales", torch.float32, dev, 2)
    _need(weights, "weights", torch.float32, dev, 2)
    if tuple(q_scales.shape) != (T, h_idx) or tuple(weights.shape) != (T, h_idx):
        raise ValueError("q_scales and weights must be [num_tokens, h_idx]")
    _need(row_offsets, "row_offsets", torch.int32, dev, 1)
    _need(k_codes, "k_codes", torch.uint8, dev, 3)
    if k_codes.shape[2] != 128:
        raise ValueError(f"k_codes must be [num_pages, page_size, 128] (got {tuple(k_codes.shape)})")
    _need(k_scales, "k_scales", torch.float32, dev, 2)
    if tuple(k_scales.shape) != tuple(k_codes.shape[:2]):
        raise ValueError("k_scales must be [num_pages, page_size]")
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, dev, 1)
    batch = cache_seqlens.shape[0]
    if row_offsets.shape[0] != batch + 1 or block_table.shape[0] != batch:
        raise ValueError("row_offsets must have batch + 1 entries and block_table batch rows")
    if max_new_tokens is None:
        max_new_tokens = max(1, int(torch.diff(row_offsets).max().item())) if batch > 0 else 1
    if indices is None:
        indices = torch.empty((T, topk), dtype=torch.int32, device=dev)
    _need(indices, "indices", torch.int32, dev)
    if indices.numel() != T * topk:
        raise ValueError("indices has the wrong size")
    if workspace is None:
        workspace = torch.empty(max(16, index_topk_workspace_size(T, block_table.shape[1])), dtype=torch.uint8,
                                device=dev)
    a = IndexTopkArgs()
    a.q_codes, a.q_scales, a.weights = q_codes.data_ptr(), q_scales.data_ptr(), weights.data_ptr()
    a.num_tokens, a.h_idx = T, h_idx
    a.row_offsets, a.batch, a.max_new_tokens = row_offsets.data_ptr(), batch, int(max_new_tokens)
    a.k_codes, a.k_scales = k_codes.data_ptr(), k_scales.data_ptr()
    a.num_pages, a.page_size = k_codes.shape[0], k_codes.shape[1]
    a.block_table, a.block_table_stride = block_table.data_ptr(), block_table.shape[1]
    a.cache_seqlens = cache_seqlens.data_ptr()
    a.relu, a.topk = int(bool(relu)), int(topk)
    a.workspace = workspace.data_ptr()
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    a.indices = indices.data_ptr()
    _check(lib().mla_index_topk(ctypes.byref(a), _stream(stream)))
    return indices.view(T, topk)


def device_status(stream=None, raise_on_error: bool = False) -> int:
    """Synchronise the stream, return and clear the device status bits."""
    flags = ctypes.c_uint32()
    st = lib().mla_get_device_status(_stream(stream), ctypes.byref(flags))
    if raise_on_error:
        _check(st)
    elif st not in (MLA_OK, 5, 6, 1):
        _check(st)
    return flags.value


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libmla.so for sm_103a (nvcc) into the package's _build folder."""
    global _lib
    path = _build.build(force=force, verbose=verbose)
    return path
