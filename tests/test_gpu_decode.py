"""GPU parity of the paged decode (split-KV) against the oracle, through the C ABI.

Page gathering is checked bit for bit through an invariance (relabelling the
physical pages gives identical output bits) and numerically against the
oracle within max |err| <= 1e-2, mean |err| <= 1e-3."""
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


def _run(g, c, table=None, kpool=None, vpool=None, ctx=None):
    import torch
    from gpu_helpers import dev, new_status
    kind = "bf16" if c.kv_dtype == "bf16" else None
    st = new_status()
    out = g.gqa_attn_paged_decode(
        dev(c.q), dev(c.k_pool if kpool is None else kpool, kind),
        dev(c.v_pool if vpool is None else vpool, kind),
        dev(c.page_table if table is None else table),
        dev(c.context_lens if ctx is None else ctx), c.scale, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("head_dim,n_heads,n_kv,dtype", [
    (128, 32, 8, "f16"), (128, 8, 8, "f16"), (64, 16, 2, "f16"), (256, 16, 4, "bf16"),
    (128, 40, 2, "bf16")])
def test_small_ragged_contexts(lib, head_dim, n_heads, n_kv, dtype):
    from gpu_helpers import assert_attention_close
    # ragged edges: 1 token, exactly one page, one past a page, one chunk, one past, ...
    c = workloads.paged_decode(num_seqs=9, ctx_lo=1, ctx_hi=700, num_pages=600, n_heads=n_heads,
                               n_kv_heads=n_kv, head_dim=head_dim, kv_dtype=dtype,
                               seed=head_dim + n_heads, fixed_lens=[1, 16, 17, 256, 257, 511])
    got, st = _run(lib, c)
    assert st == 0
    ref = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype=dtype, page_table=c.page_table,
                              context_lens=c.context_lens, scale=c.scale)
    assert_attention_close(got, ref, f"decode d{head_dim} h{n_heads}/{n_kv} {dtype}")


def test_zero_context_gives_zeros(lib):
    c = workloads.paged_decode(num_seqs=3, ctx_lo=5, ctx_hi=40, num_pages=16, seed=2,
                               fixed_lens=[7, 0])
    got, st = _run(lib, c)
    assert st == 0
    assert np.all(got[1] == 0)
    assert np.all(np.isfinite(got))


def test_page_relabelling_is_bit_identical(lib):
    c = workloads.paged_decode(num_seqs=6, ctx_lo=100, ctx_hi=2000, num_pages=900, seed=8)
    base, _ = _run(lib, c)
    perm = np.random.default_rng(4).permutation(c.num_pages)
    k2 = np.empty_like(c.k_pool)
    v2 = np.empty_like(c.v_pool)
    k2[perm] = c.k_pool
    v2[perm] = c.v_pool
    t2 = np.where(c.page_table >= 0, perm[np.maximum(c.page_table, 0)], -1).astype(np.int32)
    moved, _ = _run(lib, c, table=t2, kpool=k2, vpool=v2)
    np.testing.assert_array_equal(base, moved)


def test_bad_page_ids_are_clamped_and_flagged(lib):
    from attention_gqa_flash_gb300 import GQA_FLAG_PAGE_CLAMPED, GQA_FLAG_CONTEXT_CLAMPED
    c = workloads.paged_decode(num_seqs=2, ctx_lo=20, ctx_hi=40, num_pages=8, seed=3)
    table = c.page_table.copy()
    table[0, 0] = 10 ** 6
    ctx = c.context_lens.copy()
    ctx[1] = 10 ** 6
    got, st = _run(lib, c, table=table, ctx=ctx)
    assert st & GQA_FLAG_PAGE_CLAMPED
    assert st & GQA_FLAG_CONTEXT_CLAMPED


def test_full_size_decode(lib):
    """64 sequences, contexts U{512..16384}, 65536-page pool, h32/hk8, d128: every
    (sequence, head) output."""
    from gpu_helpers import assert_attention_close
    c = workloads.paged_decode(seed=0)
    got, st = _run(lib, c)
    assert st == 0
    ref = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16", page_table=c.page_table,
                              context_lens=c.context_lens, scale=c.scale)
    assert_attention_close(got, ref, "full-size decode")
