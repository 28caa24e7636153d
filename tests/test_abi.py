"""The C-ABI library builds, loads and exports every declared entry point;
host-side argument validation answers without a GPU."""
import ctypes
import os
import re

import pytest

import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import builder as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mla_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["mla_metadata_size", "mla_workspace_size", "mla_get_metadata", "mla_decode",
              "mla_get_device_status", "mla_last_error", "mla_abi_version", "mla_fp8_cache_store",
              "mla_sparse_prefill_workspace_size", "mla_sparse_prefill", "mla_index_topk_workspace_size",
              "mla_index_topk", "mla_test_hooks", "mla_decode_noalloc"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libmla.so does not export {name}"
    assert lib.mla_abi_version() == 3


@pytest.mark.parametrize("struct,cls", [("mla_decode_args", mla.DecodeArgs),
                                        ("mla_sparse_prefill_args", mla.SparsePrefillArgs),
                                        ("mla_index_topk_args", mla.IndexTopkArgs)])
def test_args_structs_match_header(struct, cls):
    # field order and count of the argument structs
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{((?:(?!typedef struct).)*?)\} " + struct + ";", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        names = [n.strip().lstrip("*") for n in re.sub(r"^(const\s+)?[\w]+\s*\*?", "", decl).split(",")]
        fields += [n for n in names if n]
    assert fields == [f for f, _ in cls._fields_]


def test_null_args_rejected(lib):
    assert lib.mla_decode(None, None) == 1
    assert "args is NULL" in mla.last_error()


def _args(**kw):
    a = mla.DecodeArgs()
    for f, v in dict(q=16, batch=1, s_q=1, h_q=16, kvcache=16, num_pages=1, page_size=64, block_table=16,
                     block_table_stride=1, cache_seqlens=16, sm_scale=0.1, sched=16, num_splits=16,
                     workspace=256, workspace_bytes=1 << 20, out=16, lse=16).items():
        setattr(a, f, v)
    for f, v in kw.items():
        setattr(a, f, v)
    return a


@pytest.mark.parametrize("field,value,status,needle", [
    ("q", None, 1, "q is NULL"),
    ("kvcache", None, 1, "kvcache is NULL"),
    ("out", None, 1, "out is NULL"),
    ("lse", None, 1, "lse is NULL"),
    ("page_size", 32, 2, "page_size must be 64"),
    ("num_pages", 0, 1, "num_pages"),
    ("block_table_stride", 0, 1, "block_table_stride"),
    ("q", 18, 1, "q is not 16-byte aligned"),
    ("sm_scale", float("nan"), 1, "sm_scale"),
])
def test_host_validation(lib, field, value, status, needle):
    a = _args(**{field: value})
    assert lib.mla_decode(ctypes.byref(a), None) == status
    assert needle in mla.last_error()


def test_decode_rejects_a_bad_is_fp8(lib):
    a = _args(is_fp8=3)
    assert lib.mla_decode(ctypes.byref(a), None) == 1 and "is_fp8" in mla.last_error()


def test_sparse_mode_rules(lib):
    a = _args(topk=64, indices=None, is_fp8=1)
    assert lib.mla_decode(ctypes.byref(a), None) == 1 and "indices is NULL" in mla.last_error()
    a = _args(topk=64, indices=16, is_fp8=0)  # sparse over the bf16 cache is a supported mode
    assert lib.mla_decode(ctypes.byref(a), None) not in (1, 2)
    a = _args(topk=64, indices=16, is_fp8=1, is_causal=1)
    assert lib.mla_decode(ctypes.byref(a), None) == 2 and "dense mode only" in mla.last_error()
    a = _args(topk=0, indices=16)
    assert lib.mla_decode(ctypes.byref(a), None) == 1


def test_size_queries_validate_before_touching_a_device(lib):
    # argument order (batch, h_q, s_q, topk, is_fp8)
    a, b = ctypes.c_int(), ctypes.c_int()
    assert lib.mla_metadata_size(0, 16, 1, 0, 0, ctypes.byref(a), ctypes.byref(b)) == 1
    assert "batch" in mla.last_error()
    n = ctypes.c_size_t()
    assert lib.mla_workspace_size(1, 16, 0, 0, 0, ctypes.byref(n)) == 1
    assert "s_q" in mla.last_error()
    assert lib.mla_workspace_size(1, 0, 1, 0, 0, ctypes.byref(n)) == 1
    assert "h_q" in mla.last_error()
    assert lib.mla_workspace_size(1, 2048, 1, 0, 0, ctypes.byref(n)) in (2, 4)
    assert lib.mla_workspace_size(1, 16, 1, 0, 2, ctypes.byref(n)) == 1
    assert "is_fp8" in mla.last_error()
    assert lib.mla_get_metadata(None, 1, 16, 1, 0, 0, None, None, None) == 1


def test_test_hooks_validate(lib):
    assert lib.mla_test_hooks(-1, 0) == 1 and "num_parts" in mla.last_error()
    assert lib.mla_test_hooks(0, 0) == 0


def test_binding_takes_the_configuration_by_keyword():
    # h_q and s_q are both ints: positional use could swap them silently, so it is refused
    with pytest.raises(TypeError):
        mla.workspace_size(1, 1, 16, 0, False)
    with pytest.raises(TypeError):
        mla.get_metadata(None, 1, 16, 0)


def test_python_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 1, 16, 576, dtype=torch.float32)
    with pytest.raises(ValueError, match="q must have dtype"):
        mla.decode(q, q, q, q, 0.1, q, q)
    q = torch.zeros(1, 1, 16, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        mla.decode(q, q, q, q, 0.1, q, q)


def _prefill_args(**kw):
    a = mla.SparsePrefillArgs()
    for f, v in dict(q=16, s_q=4, h_q=16, kv=16, s_kv=100, indices=16, topk=64, sm_scale=0.1,
                     workspace=256, workspace_bytes=1 << 30, out=16, lse=16).items():
        setattr(a, f, v)
    for f, v in kw.items():
        setattr(a, f, v)
    return a


@pytest.mark.parametrize("field,value,status,needle", [
    ("q", None, 1, "q is NULL"),
    ("kv", None, 1, "kv is NULL"),
    ("indices", None, 1, "indices is NULL"),
    ("out", None, 1, "out is NULL"),
    ("lse", None, 1, "lse is NULL"),
    ("s_q", 0, 1, "s_q"),
    ("s_kv", 0, 1, "s_kv"),
    ("topk", 0, 1, "topk"),
    ("kv", 24, 1, "kv is not 16-byte aligned"),
    ("sm_scale", float("inf"), 1, "sm_scale"),
])
def test_sparse_prefill_host_validation(lib, field, value, status, needle):
    a = _prefill_args(**{field: value})
    assert lib.mla_sparse_prefill(ctypes.byref(a), None) == status
    assert needle in mla.last_error()
    assert lib.mla_sparse_prefill(None, None) == 1


def test_sparse_prefill_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(4, 16, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        mla.sparse_prefill(q, q, q, 0.1)


def _index_args(**kw):
    a = mla.IndexTopkArgs()
    for f, v in dict(q_codes=16, q_scales=16, weights=16, num_tokens=4, h_idx=64, row_offsets=16, batch=2,
                     max_new_tokens=2, k_codes=16, k_scales=16, num_pages=4, page_size=64, block_table=16,
                     block_table_stride=4, cache_seqlens=16, relu=0, topk=64, workspace=16,
                     workspace_bytes=1 << 20, indices=16).items():
        setattr(a, f, v)
    for f, v in kw.items():
        setattr(a, f, v)
    return a


@pytest.mark.parametrize("field,value,status,needle", [
    ("q_codes", None, 1, "q_codes is NULL"),
    ("k_scales", None, 1, "k_scales is NULL"),
    ("indices", None, 1, "indices is NULL"),
    ("h_idx", 12, 2, "multiple of 8"),
    ("max_new_tokens", 5, 2, "exceeds 256"),
    ("topk", 0, 2, "topk"),
    ("topk", 20000, 2, "topk"),
    ("page_size", 32, 2, "page_size"),
    ("k_codes", 8, 1, "k_codes is not 16-byte aligned"),
    ("workspace_bytes", 100, 3, "workspace_bytes"),
])
def test_index_topk_host_validation(lib, field, value, status, needle):
    a = _index_args(**{field: value})
    assert lib.mla_index_topk(ctypes.byref(a), None) == status
    assert needle in mla.last_error()
    assert lib.mla_index_topk(None, None) == 1
