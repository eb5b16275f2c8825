"""Pins for the oracle's paged decode.

ferrum-kernels causal_attention.rs (paged_state_regions) cuts a sequence's
logical KV stream into fixed pages in logical order; the single decode query
attends to every context token.  Pinned here by:
  * an independent gather with NumPy fancy indexing followed by unmasked
    attention over the gathered contiguous K/V;
  * invariance under a relabelling of the physical pages;
  * NaN-filled unused pages and page tails leaving every output finite.
"""
import numpy as np

import oracle
import workloads


def _small(seed=3, **kw):
    args = dict(num_seqs=5, ctx_lo=1, ctx_hi=70, num_pages=64, page_size=16, n_heads=8,
                n_kv_heads=2, head_dim=16, seed=seed)
    args.update(kw)
    return workloads.paged_decode(**args)


def test_decode_equals_attention_over_numpy_gathered_context():
    c = _small()
    out = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16", page_table=c.page_table,
                              context_lens=c.context_lens, scale=c.scale)
    for s in range(c.num_seqs):
        t = np.arange(c.context_lens[s])
        pages = c.page_table[s, t // c.page_size]
        k = np.ascontiguousarray(c.k_pool[pages, t % c.page_size])   # [ctx, hk, d]
        v = np.ascontiguousarray(c.v_pool[pages, t % c.page_size])
        ref = oracle.attention(c.q[s:s + 1], k, v, kv_dtype="f16", scale=c.scale)
        np.testing.assert_array_equal(out[s], ref[0])


def test_page_relabelling_is_invisible():
    c = _small(seed=5)
    out = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16", page_table=c.page_table,
                              context_lens=c.context_lens, scale=c.scale)
    perm = np.random.default_rng(9).permutation(c.num_pages)      # new id of old page p
    k2 = np.empty_like(c.k_pool)
    v2 = np.empty_like(c.v_pool)
    k2[perm] = c.k_pool
    v2[perm] = c.v_pool
    table2 = np.where(c.page_table >= 0, perm[np.maximum(c.page_table, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode(c.q, k2, v2, kv_dtype="f16", page_table=table2,
                               context_lens=c.context_lens, scale=c.scale)
    np.testing.assert_array_equal(out, out2)


def test_nan_outside_the_context_never_reaches_the_output():
    c = _small(seed=7)
    assert np.isnan(c.k_pool.astype(np.float32)).any()
    out = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16", page_table=c.page_table,
                              context_lens=c.context_lens, scale=c.scale)
    assert np.all(np.isfinite(out))


def test_subset_of_sequences_matches_full_run():
    c = _small(seed=11)
    full = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16",
                               page_table=c.page_table, context_lens=c.context_lens,
                               scale=c.scale)
    some = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="f16",
                               page_table=c.page_table, context_lens=c.context_lens,
                               scale=c.scale, seqs=np.array([4, 1]))
    np.testing.assert_array_equal(some[0], full[4])
    np.testing.assert_array_equal(some[1], full[1])


def test_bf16_pool():
    c = _small(seed=13, kv_dtype="bf16")
    out = oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype="bf16",
                              page_table=c.page_table, context_lens=c.context_lens,
                              scale=c.scale)
    s = 2
    t = np.arange(c.context_lens[s])
    pages = c.page_table[s, t // c.page_size]
    k = np.ascontiguousarray(c.k_pool[pages, t % c.page_size])
    v = np.ascontiguousarray(c.v_pool[pages, t % c.page_size])
    ref = oracle.attention(c.q[s:s + 1], k, v, kv_dtype="bf16", scale=c.scale)
    np.testing.assert_array_equal(out[s], ref[0])
    assert np.all(np.isfinite(out))
