"""Pins for the oracle's masked GQA attention.

What the definition O = softmax(scale * Q K^T + mask) V (one KV head per
n_heads / n_kv_heads query heads, mask added after scaling; mlx-native
flash_attn_prefill_tensor.rs module doc) fixes without an implementation:

  * one visible key returns that key's V row exactly;
  * a V that is constant over keys is returned unchanged;
  * two visible keys give a logistic blend whose weights are computed here by
    hand from a Q/K pair with a known dot product and finite mask values
    (catches a scaled mask, a sign error, a missing term);
  * GQA equals MHA over explicitly repeated KV heads (catches a wrong
    head grouping);
  * -inf keys contribute nothing, so trimming them is a no-op;
  * Q = 0 gives the mean of the visible V rows;
  * a constant added to a row of a finite mask changes nothing;
  * permuting keys (with their mask columns) changes nothing;
  * huge logits do not overflow;
  * a row with no visible key is zero (the reading the library adopts);
  * strided views evaluate like their contiguous copies.
"""
import math

import numpy as np

import oracle
from workloads import bf16_bits

RNG = np.random.default_rng(1234)


def _rand_case(rows=7, keys=11, h=6, hk=3, d=16, dtype="f16"):
    q = RNG.standard_normal((rows, h, d)).astype(np.float32)
    if dtype == "f16":
        k = RNG.standard_normal((keys, hk, d)).astype(np.float16)
        v = RNG.standard_normal((keys, hk, d)).astype(np.float16)
    else:
        k = bf16_bits(RNG.standard_normal((keys, hk, d)).astype(np.float32))
        v = bf16_bits(RNG.standard_normal((keys, hk, d)).astype(np.float32))
    return q, k, v


def _wide(x, dtype):
    if dtype == "f16":
        return x.astype(np.float64)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_single_visible_key_returns_that_value_row():
    for dtype in ("f16", "bf16"):
        q, k, v = _rand_case(dtype=dtype)
        rows, h, _ = q.shape
        keys, hk, _ = k.shape
        cols = RNG.integers(0, keys, size=rows)
        mask = np.full((rows, keys), -np.inf, dtype=np.float16)
        mask[np.arange(rows), cols] = 0
        out = oracle.attention(q, k, v, kv_dtype=dtype, scale=0.3, mask=mask)
        vw = _wide(v, dtype)
        g = h // hk
        for i in range(rows):
            for qh in range(h):
                np.testing.assert_array_equal(out[i, qh], vw[cols[i], qh // g])


def test_constant_values_are_returned():
    q, k, _ = _rand_case()
    keys, hk, d = k.shape
    row = RNG.standard_normal((1, hk, d)).astype(np.float16)
    v = np.repeat(row, keys, axis=0)
    mask = np.where(RNG.random((q.shape[0], keys)) < 0.7, 0, -np.inf).astype(np.float16)
    mask[:, 0] = 0
    out = oracle.attention(q, k, v, kv_dtype="f16", scale=1.0, mask=mask)
    g = q.shape[1] // hk
    for qh in range(q.shape[1]):
        np.testing.assert_allclose(out[:, qh], np.broadcast_to(row[0, qh // g].astype(np.float64),
                                                               out[:, qh].shape), rtol=1e-14)


def test_two_keys_closed_form():
    d = 8
    a, b0 = 1.5, 2.0            # q = a e0, k0 = b0 e0, k1 = e1 -> <q,k0> = a b0, <q,k1> = 0
    m0, m1 = -0.5, 0.25         # finite additive mask values, exact in f16
    scale = 0.75
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = a
    k = np.zeros((2, 1, d), np.float16)
    k[0, 0, 0] = b0
    k[1, 0, 1] = 1.0
    v = np.zeros((2, 1, d), np.float16)
    v[0, 0, :] = np.arange(d)
    v[1, 0, :] = -2.0 * np.arange(d) + 1
    mask = np.array([[m0, m1]], np.float16)
    s0 = scale * a * b0 + m0
    s1 = m1
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * v[0, 0].astype(np.float64) + (1 - w0) * v[1, 0].astype(np.float64)
    out = oracle.attention(q, k, v, kv_dtype="f16", scale=scale, mask=mask)
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-13)
    # the same with bf16 queries and keys
    qb = bf16_bits(q)
    kb = bf16_bits(k.astype(np.float32))
    vb = bf16_bits(v.astype(np.float32))
    out = oracle.attention(qb, kb, vb, kv_dtype="bf16", q_dtype="bf16", scale=scale,
                           mask=bf16_bits(mask.astype(np.float32)), mask_dtype="bf16")
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads():
    q, k, v = _rand_case(h=8, hk=2)
    g = 4
    k_rep = np.stack([k[:, h // g] for h in range(8)], axis=1)
    v_rep = np.stack([v[:, h // g] for h in range(8)], axis=1)
    mask = np.where(RNG.random((q.shape[0], k.shape[0])) < 0.8, 0, -np.inf).astype(np.float16)
    mask[:, 3] = 0
    a = oracle.attention(q, k, v, kv_dtype="f16", scale=0.2, mask=mask)
    b = oracle.attention(q, k_rep, v_rep, kv_dtype="f16", scale=0.2, mask=mask)
    np.testing.assert_array_equal(a, b)
    # a different grouping (h % n_kv_heads) must give a different answer
    k_alt = np.stack([k[:, h % 2] for h in range(8)], axis=1)
    v_alt = np.stack([v[:, h % 2] for h in range(8)], axis=1)
    c = oracle.attention(q, k_alt, v_alt, kv_dtype="f16", scale=0.2, mask=mask)
    assert np.abs(a - c).max() > 1e-3


def test_masked_padding_keys_contribute_nothing():
    q, k, v = _rand_case(keys=20)
    n = 13
    k[n:] = 7.0        # finite garbage in the padded rows
    v[n:] = -9.0
    mask = np.zeros((q.shape[0], 20), np.float16)
    mask[:, n:] = -np.inf
    full = oracle.attention(q, k, v, kv_dtype="f16", scale=0.4, mask=mask)
    trimmed = oracle.attention(q, k[:n], v[:n], kv_dtype="f16", scale=0.4,
                               mask=np.ascontiguousarray(mask[:, :n]))
    np.testing.assert_array_equal(full, trimmed)
    nomask = oracle.attention(q, k[:n], v[:n], kv_dtype="f16", scale=0.4)
    np.testing.assert_array_equal(full, nomask)


def test_zero_query_gives_mean_of_visible_values():
    q, k, v = _rand_case(rows=5, keys=9)
    q[:] = 0
    vis = RNG.random((5, 9)) < 0.5
    vis[:, 2] = True
    mask = np.where(vis, 0, -np.inf).astype(np.float16)
    out = oracle.attention(q, k, v, kv_dtype="f16", scale=1.0, mask=mask)
    g = q.shape[1] // k.shape[1]
    for i in range(5):
        for qh in range(q.shape[1]):
            expect = v[vis[i], qh // g].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(out[i, qh], expect, rtol=1e-13, atol=1e-15)


def test_row_shift_of_the_mask_changes_nothing():
    q, k, v = _rand_case()
    # multiples of 1/64 in [-2, 2]: adding 3 stays exact in f16
    base = (RNG.integers(-128, 129, size=(q.shape[0], k.shape[0])) / 64).astype(np.float16)
    shifted = (base.astype(np.float32) + np.float32(3.0)).astype(np.float16)
    exact = np.all(shifted.astype(np.float64) - base.astype(np.float64) == 3.0, axis=1)
    a = oracle.attention(q, k, v, kv_dtype="f16", scale=0.5, mask=base)
    b = oracle.attention(q, k, v, kv_dtype="f16", scale=0.5, mask=shifted)
    assert exact.all()
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_key_permutation_changes_nothing():
    q, k, v = _rand_case(keys=15)
    mask = np.where(RNG.random((q.shape[0], 15)) < 0.6, 0, -np.inf).astype(np.float16)
    mask[:, 0] = 0
    perm = RNG.permutation(15)
    a = oracle.attention(q, k, v, kv_dtype="f16", scale=0.3, mask=mask)
    b = oracle.attention(q, np.ascontiguousarray(k[perm]), np.ascontiguousarray(v[perm]),
                         kv_dtype="f16", scale=0.3, mask=np.ascontiguousarray(mask[:, perm]))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_huge_logits_are_stable():
    d = 4
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 1000.0
    k = np.zeros((3, 1, d), np.float16)
    k[:, 0, 0] = [50.0, 60.0, 40.0]    # logits 5e4, 6e4, 4e4: exp would overflow unshifted
    v = np.zeros((3, 1, d), np.float16)
    v[:, 0, 1] = [1.0, 2.0, 3.0]
    out = oracle.attention(q, k, v, kv_dtype="f16", scale=1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_array_equal(out[0, 0], v[1, 0].astype(np.float64))


def test_fully_masked_row_is_zero():
    q, k, v = _rand_case(rows=3)
    mask = np.zeros((3, k.shape[0]), np.float16)
    mask[1] = -np.inf
    out = oracle.attention(q, k, v, kv_dtype="f16", scale=1.0, mask=mask)
    assert np.all(out[1] == 0)
    assert np.all(np.abs(out[0]).sum(axis=-1) > 0)


def test_strided_views_match_contiguous_copies():
    q, k, v = _rand_case(rows=6, keys=10, h=4, hk=2, d=8)
    # embed each tensor in a larger buffer with padded row and head strides
    qb = np.zeros((6, 5, 12), np.float32)
    qb[:, :4, :8] = q
    kb = np.zeros((10, 3, 16), np.float16)
    kb[:, :2, :8] = k
    vb = np.zeros((10, 2, 24), np.float16)
    vb[:, :, 4:12] = v
    mask = np.where(RNG.random((6, 10)) < 0.7, 0, -np.inf).astype(np.float16)
    mask[:, 1] = 0
    mb = np.zeros((6, 16), np.float16)
    mb[:, :10] = mask
    a = oracle.attention(q, k, v, kv_dtype="f16", scale=0.7, mask=mask)
    b = oracle.attention(qb[:, :4, :8], kb[:, :2, :8], vb[:, :, 4:12], kv_dtype="f16",
                         scale=0.7, mask=mb[:, :10])
    np.testing.assert_array_equal(a, b)


def test_pairs_select_single_outputs():
    q, k, v = _rand_case()
    mask = np.zeros((q.shape[0], k.shape[0]), np.float16)
    full = oracle.attention(q, k, v, kv_dtype="f16", scale=0.3, mask=mask)
    pairs = np.array([[0, 0], [6, 5], [3, 2]], np.int32)
    some = oracle.attention(q, k, v, kv_dtype="f16", scale=0.3, mask=mask, pairs=pairs)
    for n, (i, h) in enumerate(pairs):
        np.testing.assert_array_equal(some[n], full[i, h])


def test_brute_force_textbook_on_tiny_inputs():
    """A second, independent route on tiny inputs: NumPy softmax over a dense
    score matrix (secondary to the closed forms above)."""
    q, k, v = _rand_case(rows=4, keys=6, h=4, hk=2, d=8)
    mask = np.where(RNG.random((4, 6)) < 0.7, 0, -np.inf).astype(np.float16)
    mask[:, 0] = 0
    scale = 0.35
    out = oracle.attention(q, k, v, kv_dtype="f16", scale=scale, mask=mask)
    kw, vw = k.astype(np.float64), v.astype(np.float64)
    for qh in range(4):
        kk, vv = kw[:, qh // 2], vw[:, qh // 2]
        s = scale * (q[:, qh].astype(np.float64) @ kk.T) + mask.astype(np.float64)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ref = (p / p.sum(axis=1, keepdims=True)) @ vv
        np.testing.assert_allclose(out[:, qh], ref, rtol=1e-12, atol=1e-14)
