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
import pytest

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


# ---------------------------------------------------------------------------
# page append and paged chunked prefill
# ---------------------------------------------------------------------------
def _strides(c):
    hk, d = c.n_kv_heads, c.head_dim
    return dict(page_stride=c.page_size * hk * d, token_stride=hk * d, head_stride=d,
                page_size=c.page_size)


def test_f16_rounding_matches_numpy():
    """The oracle's own f32 -> f16 rounding (nearest, ties to even) against NumPy's,
    over normals, subnormals, exact ties, overflow and the special values."""
    rng = np.random.default_rng(0)
    xs = [rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000)]
    ulp_ties = [(1.0 + (2 * k + 1) * 2.0 ** -11) * 2.0 ** e for k in range(8) for e in (-14, -3, 0, 7, 15)]
    sub_ties = [(2 * k + 1) * 2.0 ** -25 for k in range(16)]
    special = [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 2.0 ** -24, 2.0 ** -25,
               1.5 * 2.0 ** -25, 6.1e-5, np.inf, -np.inf]
    allx = np.concatenate(xs + [np.array(ulp_ties), -np.array(ulp_ties), np.array(sub_ties),
                                np.array(special)]).astype(np.float32)
    got = np.array([oracle.f32_to_f16(x) for x in allx], np.uint16)
    with np.errstate(over="ignore"):
        want = allx.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """f32 -> bf16 nearest-even on the bit pattern (finite inputs)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("kv", ["f16", "bf16"])
def test_append_writes_rounded_rows_into_their_slots_only(kv):
    c = workloads.paged_chunk(num_seqs=5, tokens_hi=40, prefix_hi=70, head_dim=32, seed=2,
                              kv_dtype=kv)
    kp, vp, skipped = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                          c.page_table, c.k_pool, c.v_pool, kv_dtype=kv,
                                          **_strides(c))
    rnd = (lambda x: x.astype(np.float16)) if kv == "f16" else _bf16_bits
    assert skipped == 0
    touched = np.zeros(c.k_pool.shape[:2], bool)
    for s in range(c.num_seqs):
        i = np.arange(c.token_offsets[s], c.token_offsets[s + 1])
        p = c.position_start[s] + (i - c.token_offsets[s])
        pages, slots = c.page_table[s, p // c.page_size], p % c.page_size
        np.testing.assert_array_equal(kp[pages, slots], rnd(c.k_new[i]))
        np.testing.assert_array_equal(vp[pages, slots], rnd(c.v_new[i]))
        touched[pages, slots] = True
    np.testing.assert_array_equal(kp[~touched].view(np.uint16), c.k_pool[~touched].view(np.uint16))
    np.testing.assert_array_equal(vp[~touched].view(np.uint16), c.v_pool[~touched].view(np.uint16))
    # a token beyond the page table is skipped and counted
    table = c.page_table.copy()
    s0 = 0
    last = c.position_start[s0] + c.token_offsets[1] - 1
    table[s0, last // c.page_size] = -1
    _, _, skipped = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start, table,
                                        c.k_pool, c.v_pool, kv_dtype=kv, **_strides(c))
    assert skipped >= 1


def _appended(c):
    kp, vp, _ = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                    c.page_table, c.k_pool, c.v_pool, kv_dtype=c.kv_dtype,
                                    **_strides(c))
    return kp, vp


def test_chunked_prefill_equals_masked_attention_over_gathered_context():
    """Rows at positions ps..ps+T-1 over the gathered contiguous K/V with an explicit
    causal mask (the prefill definition) give the same result as the position-range
    definition over pages."""
    c = workloads.paged_chunk(num_seqs=3, tokens_hi=20, prefix_hi=50, head_dim=32, seed=4)
    kp, vp = _appended(c)
    out = oracle.paged_prefill(c.q, kp, vp, c.page_table, c.token_offsets, c.position_start,
                               kv_dtype="f16", n_kv_heads=c.n_kv_heads, scale=c.scale,
                               **_strides(c))
    for s in range(c.num_seqs):
        T = int(c.token_offsets[s + 1] - c.token_offsets[s])
        ctx = int(c.position_start[s]) + T
        t = np.arange(ctx)
        k = np.ascontiguousarray(kp[c.page_table[s, t // c.page_size], t % c.page_size])
        v = np.ascontiguousarray(vp[c.page_table[s, t // c.page_size], t % c.page_size])
        pos_q = c.position_start[s] + np.arange(T)
        mask = np.where(t[None, :] <= pos_q[:, None], 0.0, -np.inf).astype(np.float16)
        ref = oracle.attention(c.q[c.token_offsets[s]:c.token_offsets[s + 1]], k, v, kv_dtype="f16",
                               scale=c.scale, mask=mask)
        np.testing.assert_array_equal(out[c.token_offsets[s]:c.token_offsets[s + 1]], ref)


def test_chunked_prefill_of_one_token_is_decode():
    c = workloads.paged_chunk(num_seqs=4, tokens_lo=1, tokens_hi=1, prefix_hi=90, head_dim=32,
                              seed=6)
    kp, vp = _appended(c)
    out = oracle.paged_prefill(c.q, kp, vp, c.page_table, c.token_offsets, c.position_start,
                               kv_dtype="f16", n_kv_heads=c.n_kv_heads, scale=c.scale,
                               **_strides(c))
    dec = oracle.paged_decode(c.q, kp, vp, kv_dtype="f16", page_table=c.page_table,
                              context_lens=(c.position_start + 1).astype(np.int32), scale=c.scale)
    np.testing.assert_array_equal(out, dec)


def test_chunked_prefill_is_invariant_to_page_relabelling():
    c = workloads.paged_chunk(num_seqs=3, tokens_hi=30, prefix_hi=60, head_dim=16, seed=8)
    kp, vp = _appended(c)
    kw = dict(kv_dtype="f16", n_kv_heads=c.n_kv_heads, scale=c.scale, **_strides(c))
    out = oracle.paged_prefill(c.q, kp, vp, c.page_table, c.token_offsets, c.position_start, **kw)
    perm = np.random.default_rng(1).permutation(c.num_pages).astype(np.int32)
    inv = np.argsort(perm).astype(np.int32)   # page p moves to slot inv[p]
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[inv], vp2[inv] = kp, vp
    table2 = np.where(c.page_table >= 0, inv[np.maximum(c.page_table, 0)], -1).astype(np.int32)
    out2 = oracle.paged_prefill(c.q, kp2, vp2, table2, c.token_offsets, c.position_start, **kw)
    np.testing.assert_array_equal(out, out2)
