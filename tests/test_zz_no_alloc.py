"""The no-allocation paged decode entry point.

gqa_attn_paged_decode_noalloc serves callers that cannot give the library a
device buffer when they call it: engines whose device memory is divided up
once at start-up by their own allocator, and latency-sensitive callers that
stay away from cudaMalloc / cudaFree because those calls can block the host
and synchronise the device.  Instead of a caller workspace it keeps its
split-KV partial results in a fixed 16 MiB array in the library's device
image.

Checked here, through the C ABI: two calls in a row (on different inputs, so
stale contents of the shared array would show) agree with the regular entry
point and with the float64 oracle within the attention tolerance, and a problem
too large for the fixed array is refused with a clear message.  This file is
collected last.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_gqa_flash_gb300 as g
    g.library()
    return g


def _inputs(c):
    from gpu_helpers import dev
    return (dev(c.q), dev(c.k_pool), dev(c.v_pool), dev(c.page_table), dev(c.context_lens))


def test_two_calls_match_the_workspace_entry_point(lib):
    import torch
    from gpu_helpers import assert_attention_close, new_status
    cases = [
        workloads.paged_decode(num_seqs=8, ctx_lo=1, ctx_hi=2000, num_pages=1200, n_heads=16,
                               n_kv_heads=4, head_dim=128, seed=31),
        workloads.paged_decode(num_seqs=5, ctx_lo=300, ctx_hi=3000, num_pages=1100, n_heads=16,
                               n_kv_heads=4, head_dim=128, seed=32),
    ]
    for c in cases:
        args = _inputs(c)
        need = lib.gqa_attn_paged_decode_workspace_size(c.num_seqs, c.n_heads, c.head_dim,
                                                        c.max_pages_per_seq, c.page_size)
        assert need <= lib.GQA_NOALLOC_SCRATCH_BYTES
        ref = lib.gqa_attn_paged_decode(*args, c.scale)
        out = torch.full_like(ref, float("nan"))
        st = new_status()
        lib.gqa_attn_paged_decode_noalloc(*args, c.scale, out=out, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        got = out.cpu().numpy()
        assert_attention_close(got, ref.cpu().numpy().astype(np.float64),
                               "no-alloc decode vs workspace decode")
        expect = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16",
                                     page_table=c.page_table, context_lens=c.context_lens,
                                     scale=c.scale)
        assert_attention_close(got, expect, "no-alloc decode vs the oracle")


def test_oversized_problem_is_refused(lib):
    import torch
    from gpu_helpers import dev
    c = workloads.paged_decode(num_seqs=32, ctx_lo=16, ctx_hi=64, num_pages=256, n_heads=32,
                               n_kv_heads=8, head_dim=128, seed=33)
    # a page table wide enough for 65536-token contexts: 32 sequences x 64 chunks of 1024
    # tokens x 32 heads x (128 + 1) x 4 B of partials is about 34 MB, over the fixed 16 MiB
    table = np.full((32, 4096), -1, np.int32)
    table[:, :c.page_table.shape[1]] = c.page_table
    args = (dev(c.q), dev(c.k_pool), dev(c.v_pool), dev(table), dev(c.context_lens))
    need = lib.gqa_attn_paged_decode_workspace_size(32, 32, 128, 4096, 16)
    assert need > lib.GQA_NOALLOC_SCRATCH_BYTES
    out = torch.empty((32, 32, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.GQAError, match="fixed"):
        lib.gqa_attn_paged_decode_noalloc(*args, c.scale, out=out)
