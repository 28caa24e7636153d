"""The benchmark's algorithmic FLOP and byte counts (the numerators of its
roofline fractions) against closed forms of the workloads:

* nominal FLOPs 2 * h_q * s_q * s_k * (576 + 512) per batch element, with
  s_k the cache length (dense) or top-k (sparse) — the FlashMLA article's
  FLOP count;
* valid-only FLOPs: causal dense query token i sees L - s_q + i + 1 keys;
  sparse rows count only their valid ids;
* KV bytes: each cached token once (dense, 1152 B bf16 or 656 B FP8 rows),
  each valid gathered row once (sparse; 644 B for 640-byte rows with a
  4-byte per-token scale).

Only the fields the counts read are built (no multi-GB caches on the CPU).
"""
import types

import numpy as np
import torch

import bench
from paged_mla_decode_07_gb300 import workloads as W


def fake_inputs(w, lens, indices=None):
    lens = torch.tensor(lens, dtype=torch.int32)
    pages = int(((lens.long() + 63) // 64).max())
    table = torch.zeros((w.batch, pages), dtype=torch.int32)
    return types.SimpleNamespace(workload=w, cache_seqlens=lens, indices=indices, block_table=table)


def sparse_indices(w, seqlen, invalid):
    rng = np.random.default_rng(0)
    idx = np.empty((w.batch, w.s_q, w.topk), np.int32)
    for b in range(w.batch):
        for i in range(w.s_q):
            idx[b, i] = rng.choice(seqlen, size=w.topk, replace=False)
    if invalid:
        idx[:, :, w.topk - invalid:] = -1
    return torch.from_numpy(idx)


def test_dense_compute_bound_counts():
    w = W.WORKLOADS["dense_computebound"]
    a = bench.algorithmic(fake_inputs(w, [4096] * w.batch))
    assert a["flops"] == 2 * 128 * 2 * 4096 * 1088 * 64            # 1.460e11
    assert a["valid_flops"] == 2 * 128 * (4095 + 4096) * 1088 * 64  # causal: 4095 and 4096 keys
    assert a["kv_bytes"] == 64 * 4096 * 1152                         # 302 MB


def test_dense_memory_bound_counts():
    w = W.WORKLOADS["dense_membound"]
    lens = np.random.default_rng(1).integers(1024, 8193, w.batch)
    a = bench.algorithmic(fake_inputs(w, lens.tolist()))
    assert a["kv_bytes"] == int(lens.sum()) * 1152
    assert a["flops"] == a["valid_flops"] == 2 * 16 * 1 * float(lens.sum()) * 1088
    rows = w.batch * w.s_q * w.h_q
    pages = int(((lens + 63) // 64).sum())
    assert a["bytes"] == a["kv_bytes"] + rows * 1152 + rows * (1024 + 4) + pages * 4 + w.batch * 4


def test_dense_fp8_rows_count_656_bytes():
    w = W.WORKLOADS["dense_membound_fp8"]
    a = bench.algorithmic(fake_inputs(w, [1000, 3000] + [64] * (w.batch - 2)))
    assert a["kv_bytes"] == (1000 + 3000 + 64 * (w.batch - 2)) * 656


def test_sparse_counts_valid_rows_only():
    w = W.with_fields(W.WORKLOADS["sparse_fp8"], batch=4)
    invalid = int(0.05 * w.topk)                                      # 102 of 2048
    a = bench.algorithmic(fake_inputs(w, [32768] * 4, sparse_indices(w, 32768, invalid)))
    assert a["flops"] == 2 * 128 * 2 * 2048 * 4 * 1088
    valid = 4 * 2 * (2048 - invalid)                                  # 1946 per query token
    assert a["valid_flops"] == 2 * 128 * valid * 1088
    assert a["kv_bytes"] == valid * 656


def test_sparse_token_scale_and_bf16_rows():
    for name, row in (("sparse_fp8_token", 644), ("sparse_bf16", 1152)):
        w = W.with_fields(W.WORKLOADS[name], batch=2)
        a = bench.algorithmic(fake_inputs(w, [32768] * 2, sparse_indices(w, 32768, 0)))
        assert a["kv_bytes"] == 2 * 2 * 2048 * row, name
