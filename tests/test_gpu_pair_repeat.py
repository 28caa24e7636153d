"""Repeatability of the CTA-pair decode kernel (problems of more than 64 rows).

The pair's two CTAs hand data to each other through barriers of the even
CTA: score-operand items, S read, P ready (the odd CTA's P is handed over by
an async signal copy after its threads' proxy fences), value slots.  The
result is deterministic by construction (a fixed schedule and a fixed
combine order), so a hand-over that let an MMA read stale P or overwrite S
before it was read would show as a difference between repeated runs.  Each
case runs the same decode many times and requires bitwise-identical outputs
and log-sum-exps; the first run is also checked against the oracle."""
import numpy as np
import pytest
import torch

import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import workloads as W

from gpu_helpers import compare, run_oracle

pytestmark = pytest.mark.gpu

REPEATS = 25


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def _repeat(inp):
    w = inp.workload
    d = inp.to("cuda")
    topk = 0 if d.indices is None else d.indices.shape[-1]
    sched, ns = mla.get_metadata(d.cache_seqlens, h_q=w.h_q, s_q=w.s_q, topk=topk,
                                 is_fp8=d.kvcache.dtype == torch.uint8)
    outs = []
    for _ in range(REPEATS):
        out, lse = mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns,
                              is_causal=w.causal, indices=d.indices, kv_scales=d.kv_scales,
                              topk_lengths=d.topk_lengths)
        outs.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert mla.device_status() == 0
    o0, l0 = outs[0]
    for i, (o, l) in enumerate(outs[1:], 1):
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), f"{w.name}: run {i} output differs"
        assert torch.equal(l.view(torch.int32), l0.view(torch.int32)), f"{w.name}: run {i} lse differs"
    ref_out, ref_lse = run_oracle(inp)
    compare(o0.double().cpu().numpy(), l0.double().cpu().numpy(), ref_out, ref_lse, w.name)


def test_pair_dense_repeatable():
    """Ragged lengths with tail tiles, a causal two-token query, several pairs per problem."""
    w = W.custom(name="prep_dense", batch=3, h_q=128, s_q=2, mode="dense", seqlens=(2100, 700, 1290), causal=True)
    _repeat(W.make_inputs(w, seed=2601))


def test_pair_sparse_fp8_repeatable():
    """Sparse FP8 on CTA pairs: dequantised score blocks and RoPE handed over by the odd CTA."""
    w = W.custom(name="prep_sparse", batch=3, h_q=128, s_q=2, mode="sparse", seqlens=(4000, 900, 2500), topk=512)
    _repeat(W.make_inputs(w, seed=2602))
