"""Failure detection without a GPU fault: a wait that nothing completes runs out
its (short) watchdog limit, the kernel unwinds and reports MLA_DEVICE_TIMEOUT
through the device status word, and the context stays usable.  The stall is
switched on through the library's test-hook entry point (mla_test_hooks), not
an environment variable, so production decodes cannot be stalled by accident."""
import pytest
import torch

import paged_mla_decode_07_gb300 as mla
from paged_mla_decode_07_gb300 import workloads as W

from gpu_helpers import compare, env, metadata, overrides, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["dense", "sparse", "pair", "pair_sparse"])
def test_watchdog_timeout_is_reported_and_context_survives(mode):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    if mode == "dense":
        inp = W.make_inputs("tiny")
    elif mode == "pair_sparse":
        inp = W.make_inputs(W.custom(name="wd_psparse", batch=2, h_q=128, s_q=1, mode="sparse", seqlens=(900, 300),
                                     topk=256), seed=7)
    elif mode == "pair":
        inp = W.make_inputs(W.custom(name="wd_pair", batch=2, h_q=128, s_q=1, mode="dense", seqlens=(400, 90)),
                            seed=6)
    else:
        inp = W.make_inputs(W.custom(name="wd_sparse", batch=2, h_q=64, s_q=2, mode="sparse",
                                     seqlens=(900, 300), topk=256), seed=5)
    mla.device_status()  # clear
    with env(MLA_WATCHDOG_NS=200_000_000), overrides(debug_stall=True):
        _, _, flags = run_cuda(inp)
    assert flags & mla.DEVICE_TIMEOUT
    # the status call itself reports MLA_ERR_DEVICE_TIMEOUT
    w = inp.workload
    d = inp.to("cuda")
    topk = 0 if d.indices is None else d.indices.shape[-1]
    with env(MLA_WATCHDOG_NS=200_000_000), overrides(debug_stall=True):
        sched, ns = metadata(d, w)
        mla.decode(d.q, d.kvcache, d.block_table, d.cache_seqlens, d.sm_scale, sched, ns,
                   is_causal=w.causal, indices=d.indices)
    with pytest.raises(mla.MLAError) as ei:
        mla.device_status(raise_on_error=True)
    assert ei.value.status == 6
    # the same context still computes correct results afterwards
    out, lse, flags = run_cuda(inp)
    assert flags == 0
    ref_out, ref_lse = run_oracle(inp)
    compare(out, lse, ref_out, ref_lse, "after-timeout")
