"""Failure detection without faulting a GPU: the bounded mbarrier wait used by
the attention kernel gives up on a barrier nothing arrives on, reports
GQA_FLAG_TIMEOUT through the device status word, and the context remains
usable for a normal call afterwards."""
import time

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_gqa_flash_gb300 as g
    from gpu_helpers import assert_attention_close, dev, new_status

    st = new_status()
    t0 = time.perf_counter()
    g.gqa_selftest_bounded_wait(st, 200)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) & g.GQA_FLAG_TIMEOUT
    assert 0.15 < elapsed < 5.0
    with pytest.raises(g.GQAError):
        g.gqa_selftest_bounded_wait(st, 0)
    # the context is still healthy: a regular call succeeds and is correct
    c = workloads.tiny_prefill()
    st2 = new_status()
    out = g.gqa_attn_prefill(dev(c.q), dev(c.k), dev(c.v), dev(c.mask), c.scale, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = oracle.attention(c.q, c.k, c.v, kv_dtype="f16", scale=c.scale, mask=c.mask)
    assert_attention_close(out.cpu().numpy(), ref, "prefill after timeout self-test")
