"""GPU parity of page append (bit-exact against the oracle's rounding into the
pages) and of chunked prefill over pages (max |err| <= 1e-2, mean <= 1e-3 against
the float64 oracle), through the C ABI."""
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


def _pool_dev(pool, kv, head_major=False):
    """The pool on the device as [num_pages, page_size, hk, d]; head_major stores it
    as [num_pages, hk, page_size, d] and hands the library a permuted view."""
    import torch
    from gpu_helpers import dev
    t = dev(pool, "bf16") if kv == "bf16" else dev(pool)
    if head_major:
        t = t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    return t


def _strides(c):
    hk, d = c.n_kv_heads, c.head_dim
    return dict(page_stride=c.page_size * hk * d, token_stride=hk * d, head_stride=d,
                page_size=c.page_size)


def _append_gpu(g, c, head_major=False, table=None):
    import torch
    from gpu_helpers import dev, new_status
    kp, vp = _pool_dev(c.k_pool, c.kv_dtype, head_major), _pool_dev(c.v_pool, c.kv_dtype, head_major)
    st = new_status()
    g.gqa_paged_append(dev(c.k_new), dev(c.v_new), dev(c.token_offsets), dev(c.position_start),
                       dev(c.page_table if table is None else table), kp, vp, status=st)
    torch.cuda.synchronize()
    return kp, vp, int(st.item())


def _bits(t):
    from gpu_helpers import host_bits
    return host_bits(t.contiguous())


@pytest.mark.parametrize("kv", ["f16", "bf16"])
@pytest.mark.parametrize("head_major", [False, True])
@pytest.mark.parametrize("hk,d", [(2, 128), (8, 256), (1, 2048)])
def test_append_is_bit_exact(lib, kv, head_major, hk, d):
    """Rows of 256 elements (one round of loads per token) and of 2048 elements, over
    eight heads or one (four rounds per token), bit for bit against the oracle."""
    c = workloads.paged_chunk(num_seqs=6, tokens_hi=70, prefix_hi=200, n_heads=hk, n_kv_heads=hk,
                              head_dim=d, kv_dtype=kv, seed=11)
    kp, vp, st = _append_gpu(lib, c, head_major)
    assert st == 0
    rk, rv, skipped = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                          c.page_table, c.k_pool, c.v_pool, kv_dtype=kv,
                                          **_strides(c))
    assert skipped == 0
    np.testing.assert_array_equal(_bits(kp), rk.view(np.uint16))
    np.testing.assert_array_equal(_bits(vp), rv.view(np.uint16))


def test_append_skips_tokens_without_a_page(lib):
    c = workloads.paged_chunk(num_seqs=3, tokens_lo=20, tokens_hi=40, prefix_hi=60, head_dim=64,
                              seed=12)
    table = c.page_table.copy()
    s, last = 1, int(c.position_start[1] + c.token_offsets[2] - c.token_offsets[1] - 1)
    table[s, last // c.page_size] = -1             # no page for the last token(s) of sequence 1
    table[2, 0] = c.num_pages + 5                  # a page id outside the pool
    kp, vp, st = _append_gpu(lib, c, table=table)
    rk, rv, skipped = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                          table, c.k_pool, c.v_pool, kv_dtype="f16", **_strides(c))
    assert skipped > 0 and st == 1   # GQA_FLAG_PAGE_CLAMPED
    np.testing.assert_array_equal(_bits(kp), rk.view(np.uint16))
    np.testing.assert_array_equal(_bits(vp), rv.view(np.uint16))


CASES = [
    # num_seqs, tokens, prefix, h, hk, d, page_size, kv, head_major
    (3, (1, 40), (0, 70), 8, 2, 128, 16, "f16", False),       # short chunks: heads packed per tile
    (2, (100, 300), (0, 500), 4, 2, 256, 16, "bf16", False),  # 128-token tiles, ragged tails
    (4, (1, 8), (200, 3000), 8, 8, 128, 16, "f16", False),    # decode-like: split along the keys
    (3, (50, 200), (0, 400), 4, 1, 128, 24, "f16", True),     # 24-slot pages, head-major pool
    (2, (129, 260), (0, 300), 2, 2, 256, 256, "bf16", False), # pages longer than a key tile
    (2, (128, 128), (0, 0), 4, 2, 128, 32, "f16", False),     # no prefix, one whole tile
    # enough 128-token tiles at head_dim 256 for CTA pairs (no key splits): page boxes
    # split between the two CTAs, value rows past each context end zeroed row by row
    (4, (257, 384), (0, 1000), 16, 4, 256, 16, "f16", False),
    (8, (257, 300), (0, 500), 8, 2, 256, 32, "bf16", True),
    # CTA pairs (192 query tiles: no key splits) with page boxes of 8, 16 (48-slot pages)
    # and 64 slots: eight, four and one box per CTA half of a K tile; value stages of 8,
    # 16 and 64 rows a page
    (4, (257, 330), (0, 600), 16, 2, 256, 8, "f16", False),
    (4, (257, 330), (0, 600), 16, 2, 256, 48, "bf16", False),
    (4, (257, 330), (0, 700), 16, 2, 256, 64, "f16", True),
]


@pytest.mark.parametrize("n,tok,pre,h,hk,d,ps,kv,head_major", CASES)
def test_chunked_prefill_matches_oracle(lib, n, tok, pre, h, hk, d, ps, kv, head_major):
    import torch
    from gpu_helpers import assert_attention_close, dev, new_status
    need = n * (-(-(pre[1] + tok[1]) // ps))
    c = workloads.paged_chunk(num_seqs=n, tokens_lo=tok[0], tokens_hi=tok[1], prefix_lo=pre[0],
                              prefix_hi=pre[1], num_pages=need + 7, page_size=ps, n_heads=h,
                              n_kv_heads=hk, head_dim=d, kv_dtype=kv, seed=n * 7 + d + ps)
    kp, vp, st = _append_gpu(lib, c, head_major)
    assert st == 0
    max_tokens = int(np.diff(c.token_offsets).max())
    status = new_status()
    out = lib.gqa_attn_paged_prefill(dev(c.q), kp, vp, dev(c.page_table), dev(c.token_offsets),
                                     dev(c.position_start), max_tokens, c.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rk, rv, _ = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                    c.page_table, c.k_pool, c.v_pool, kv_dtype=kv, **_strides(c))
    ref = oracle.paged_prefill(c.q, rk, rv, c.page_table, c.token_offsets, c.position_start,
                               kv_dtype=kv, n_kv_heads=hk, scale=c.scale, **_strides(c))
    assert_attention_close(out.cpu().numpy(), ref, f"chunked prefill {c.name}")


def test_chunked_prefill_leaves_rows_of_no_sequence_alone(lib):
    """Rows past token_offsets[num_seqs] belong to no sequence and are not written."""
    import torch
    from gpu_helpers import dev, new_status
    c = workloads.paged_chunk(num_seqs=2, tokens_lo=30, tokens_hi=60, prefix_hi=100, head_dim=128,
                              seed=21)
    kp, vp, _ = _append_gpu(lib, c)
    T = c.tokens
    q = np.concatenate([c.q, np.ones((5,) + c.q.shape[1:], np.float32)])
    out = torch.full((T + 5,) + c.q.shape[1:], 7.0, dtype=torch.float32, device="cuda")
    st = new_status()
    lib.gqa_attn_paged_prefill(dev(q), kp, vp, dev(c.page_table), dev(c.token_offsets),
                               dev(c.position_start), 64, c.scale, out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.all(out[T:] == 7.0)


def test_chunked_prefill_full_size(lib):
    """8 sequences x 512 new tokens over cached prefixes of up to 7680 tokens, 16/4
    heads, head_dim 256, 16-slot f16 pages: the appended pages bit for bit, every
    output finite, and every token of three whole sequences -- the one with the
    longest cached prefix, the one with the shortest, and one more -- against the
    oracle's chunked prefill over the oracle's own appended pages."""
    import torch
    from gpu_helpers import assert_attention_close, dev, new_status
    c = workloads.paged_chunk_full(seed=0)
    kp, vp, st = _append_gpu(lib, c)
    assert st == 0
    status = new_status()
    out = lib.gqa_attn_paged_prefill(dev(c.q), kp, vp, dev(c.page_table), dev(c.token_offsets),
                                     dev(c.position_start), 512, c.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    rk, rv, _ = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                    c.page_table, c.k_pool, c.v_pool, kv_dtype="f16", **_strides(c))
    np.testing.assert_array_equal(_bits(kp), rk.view(np.uint16))
    np.testing.assert_array_equal(_bits(vp), rv.view(np.uint16))
    seqs = sorted({int(np.argmax(c.position_start)), int(np.argmin(c.position_start)), 3})
    for s in seqs:
        o0, o1 = int(c.token_offsets[s]), int(c.token_offsets[s + 1])
        ref = oracle.paged_prefill(c.q[o0:o1], rk, rv, c.page_table[s:s + 1],
                                   np.array([0, o1 - o0], np.int32), c.position_start[s:s + 1],
                                   kv_dtype="f16", n_kv_heads=c.n_kv_heads, scale=c.scale,
                                   **_strides(c))
        assert_attention_close(got[o0:o1], ref, f"chunked prefill full size, sequence {s} "
                                                f"({o1 - o0} tokens after {int(c.position_start[s])})")


def test_chunked_prefill_edge_cases(lib):
    """Sequences with no new token, a single token at position 0, 8-slot pages and
    128-slot pages (the value rows past the context come from the pool row by row)."""
    import torch
    from gpu_helpers import assert_attention_close, dev, new_status
    for ps_, tok, pre, seed in ((8, (2, 40), (0, 30), 31), (128, (2, 200), (0, 300), 32)):
        c = workloads.paged_chunk(num_seqs=4, tokens_lo=tok[0], tokens_hi=tok[1], prefix_lo=pre[0],
                                  prefix_hi=pre[1], num_pages=4 * (-(-(tok[1] + pre[1]) // ps_)) + 3,
                                  page_size=ps_, n_heads=4, n_kv_heads=2, head_dim=128, seed=seed)
        # force one empty sequence and one single token at position 0
        toks = np.diff(c.token_offsets).astype(np.int64)
        toks[1], toks[2] = 0, 1
        offs = np.concatenate([[0], np.cumsum(toks)]).astype(np.int32)
        ps = c.position_start.copy()
        ps[2] = 0
        T = int(offs[-1])
        q, kn, vn = c.q[:T], c.k_new[:T], c.v_new[:T]
        kp, vp = _pool_dev(c.k_pool, "f16"), _pool_dev(c.v_pool, "f16")
        st = new_status()
        lib.gqa_paged_append(dev(kn), dev(vn), dev(offs), dev(ps), dev(c.page_table), kp, vp, status=st)
        out = lib.gqa_attn_paged_prefill(dev(q), kp, vp, dev(c.page_table), dev(offs), dev(ps),
                                         max(1, int(toks.max())), c.scale, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        rk, rv, skipped = oracle.paged_append(kn, vn, offs, ps, c.page_table, c.k_pool, c.v_pool,
                                              kv_dtype="f16", **_strides(c))
        assert skipped == 0
        np.testing.assert_array_equal(_bits(kp), rk.view(np.uint16))
        ref = oracle.paged_prefill(q, rk, rv, c.page_table, offs, ps, kv_dtype="f16",
                                   n_kv_heads=c.n_kv_heads, scale=c.scale, **_strides(c))
        assert_attention_close(out.cpu().numpy(), ref, f"chunked prefill edges, page {ps_}")


def test_chunked_prefill_clamps_and_flags_long_sequences(lib):
    """A sequence with more tokens than max_tokens: its rows past max_tokens are not
    computed (their output keeps what was there) and GQA_FLAG_CONTEXT_CLAMPED is raised;
    the rows that are computed still match the oracle."""
    import torch
    from gpu_helpers import assert_attention_close, dev, new_status
    c = workloads.paged_chunk(num_seqs=2, tokens_lo=40, tokens_hi=60, prefix_hi=50, head_dim=128,
                              seed=33)
    kp, vp, _ = _append_gpu(lib, c)
    limit = 32
    out = torch.full(c.q.shape, 7.0, dtype=torch.float32, device="cuda")
    st = new_status()
    lib.gqa_attn_paged_prefill(dev(c.q), kp, vp, dev(c.page_table), dev(c.token_offsets),
                               dev(c.position_start), limit, c.scale, out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 2   # GQA_FLAG_CONTEXT_CLAMPED
    got = out.cpu().numpy()
    rk, rv, _ = oracle.paged_append(c.k_new, c.v_new, c.token_offsets, c.position_start,
                                    c.page_table, c.k_pool, c.v_pool, kv_dtype="f16", **_strides(c))
    ref = oracle.paged_prefill(c.q, rk, rv, c.page_table, c.token_offsets, c.position_start,
                               kv_dtype="f16", n_kv_heads=c.n_kv_heads, scale=c.scale, **_strides(c))
    for s in range(c.num_seqs):
        o0, o1 = int(c.token_offsets[s]), int(c.token_offsets[s + 1])
        assert_attention_close(got[o0:o0 + limit], ref[o0:o0 + limit], f"seq {s} computed rows")
        assert np.all(got[o0 + limit:o1] == 7.0)


def test_page_append_and_prefill_with_no_tokens(lib):
    """total_tokens = 0: both calls are accepted and do nothing."""
    import torch
    from gpu_helpers import dev, new_status
    c = workloads.paged_chunk(num_seqs=2, tokens_hi=10, prefix_hi=20, head_dim=64, seed=34)
    kp, vp = _pool_dev(c.k_pool, "f16"), _pool_dev(c.v_pool, "f16")
    before = _bits(kp).copy()
    z = np.zeros(3, np.int32)
    st = new_status()
    empty_kv = torch.empty((0, c.n_kv_heads, 64), dtype=torch.float32, device="cuda")
    lib.gqa_paged_append(empty_kv, empty_kv, dev(z), dev(c.position_start), dev(c.page_table), kp, vp,
                         status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(_bits(kp), before)


def test_chunked_prefill_page_relabelling_is_bit_identical(lib):
    """Moving every page to another physical slot (and the page table with it) gives the
    same bits: the page gather depends only on the table."""
    import torch
    from gpu_helpers import dev, new_status
    c = workloads.paged_chunk(num_seqs=3, tokens_lo=60, tokens_hi=200, prefix_hi=300, head_dim=256,
                              seed=41)
    kp, vp, _ = _append_gpu(lib, c)
    perm = np.random.default_rng(5).permutation(c.num_pages)
    inv = np.argsort(perm)
    kp2, vp2 = torch.empty_like(kp), torch.empty_like(vp)
    kp2[torch.from_numpy(inv).cuda()] = kp
    vp2[torch.from_numpy(inv).cuda()] = vp
    table2 = np.where(c.page_table >= 0, inv[np.maximum(c.page_table, 0)], -1).astype(np.int32)
    max_tokens = int(np.diff(c.token_offsets).max())
    st = new_status()
    o1 = lib.gqa_attn_paged_prefill(dev(c.q), kp, vp, dev(c.page_table), dev(c.token_offsets),
                                    dev(c.position_start), max_tokens, c.scale, status=st)
    o2 = lib.gqa_attn_paged_prefill(dev(c.q), kp2, vp2, dev(table2), dev(c.token_offsets),
                                    dev(c.position_start), max_tokens, c.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o1, o2)


def test_chunked_prefill_pair_edge_cases(lib):
    """CTA pairs (head_dim 256, 16 query heads over 2 KV heads, up to 300 rows: 192 query
    tiles): a sequence with no new token and one with a single token at position 0 beside
    two long ones whose contexts end inside a page, against the oracle."""
    import torch
    from gpu_helpers import assert_attention_close, dev, new_status
    c = workloads.paged_chunk(num_seqs=4, tokens_lo=260, tokens_hi=300, prefix_lo=0, prefix_hi=400,
                              num_pages=4 * 27 + 5, page_size=16, n_heads=16, n_kv_heads=2,
                              head_dim=256, seed=51)
    toks = np.diff(c.token_offsets).astype(np.int64)
    toks[1], toks[2] = 0, 1
    offs = np.concatenate([[0], np.cumsum(toks)]).astype(np.int32)
    ps = c.position_start.copy()
    ps[2] = 0
    assert (ps[0] + toks[0]) % 16 and (ps[3] + toks[3]) % 16  # contexts end inside a page
    T = int(offs[-1])
    q, kn, vn = c.q[:T], c.k_new[:T], c.v_new[:T]
    kp, vp = _pool_dev(c.k_pool, "f16"), _pool_dev(c.v_pool, "f16")
    st = new_status()
    lib.gqa_paged_append(dev(kn), dev(vn), dev(offs), dev(ps), dev(c.page_table), kp, vp, status=st)
    out = lib.gqa_attn_paged_prefill(dev(q), kp, vp, dev(c.page_table), dev(offs), dev(ps),
                                     int(toks.max()), c.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, skipped = oracle.paged_append(kn, vn, offs, ps, c.page_table, c.k_pool, c.v_pool,
                                          kv_dtype="f16", **_strides(c))
    assert skipped == 0
    ref = oracle.paged_prefill(q, rk, rv, c.page_table, offs, ps, kv_dtype="f16",
                               n_kv_heads=c.n_kv_heads, scale=c.scale, **_strides(c))
    assert_attention_close(out.cpu().numpy(), ref, "chunked prefill pair edges")
