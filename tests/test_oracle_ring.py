"""Pins for the oracle's DFlash2 ring-KV pack / mask / commit.

mlx-native 0.21.1 src/ops/dflash2_attention_pack.rs gives one worked example
(test gpu_pack_mask_and_commit_match_ring_semantics), the geometry rule
(validate / validates_fixed_packed_length) and the draft mask-row example
(gpu_mask_rows_preserve_anchors); they are stored under tests/golden/ and
checked bit for bit.  Beyond them:
  * a simulation of sequential ring writes fixes the history order (the
    j-th packed history entry is the j-th most recent token written);
  * commit followed by pack returns the committed rows newest first;
  * pack -> mask -> attention equals attention over the chronological
    sequence under a sliding window of `window` positions, built here from
    token positions without the pack's slot arithmetic.
"""
import itertools
import json
import pathlib

import numpy as np

import oracle
import workloads

GOLDEN = pathlib.Path(__file__).parent / "golden"


def _bf16(x) -> int:
    return int(workloads.bf16_bits(np.array([x], np.float32))[0])


def test_worked_example_bit_exact():
    ex = json.loads((GOLDEN / "dflash2_worked_example.json").read_text())
    gd = ex["geometry"]
    g = [gd[k] for k in ("lanes", "q_heads", "kv_heads", "head_dim", "rows", "window",
                         "packed_len", "max_commit")]
    B, H, HK, D, R, W, K, MC = g
    ring_k = np.zeros((B, HK, W, D), np.uint16)
    ring_v = np.zeros((B, HK, W, D), np.uint16)
    for s in range(W):
        ring_k[0, 0, s, 0] = _bf16(ex["ring_k_slot_element0"][s])
        ring_v[0, 0, s, 0] = _bf16(ex["ring_v_slot_element0"][s])
    cq = np.zeros((B, R, H, D), np.float32)
    ck = np.zeros((B, R, HK, D), np.float32)
    cv = np.zeros((B, R, HK, D), np.float32)
    for r in range(R):
        cq[0, r, 0, 0] = ex["current_q_row_element0"][r]
        ck[0, r, 0, 0] = ex["current_k_row_element0"][r]
        cv[0, r, 0, 0] = ex["current_v_row_element0"][r]
    lens = np.array([ex["cache_length"]], np.uint32)
    pos = np.array([ex["write_position"]], np.uint32)
    pq, pk, pv = oracle.pack_attention(ring_k, ring_v, cq, ck, cv, lens, pos, g)
    assert pq[0, 0, 0, 0] == _bf16(ex["expected_packed_q_element0"])
    assert [int(pk[0, 0, c, 0]) for c in range(K)] == \
        [_bf16(x) for x in ex["expected_packed_k_column_element0"]]
    mask = oracle.fill_mask(lens, g).reshape(-1)
    expect = [0x0000 if m == "0" else 0xff80 for m in ex["expected_mask_flat"]]
    assert [int(x) for x in mask] == expect
    counts = np.array([ex["commit_count"]], np.uint32)
    rk, rv = oracle.commit_kv(ck, cv, counts, pos, ring_k, ring_v, g)
    for slot, val in ex["expected_ring_k_after_commit_slot_element0"].items():
        assert rk[0, 0, int(slot), 0] == _bf16(val)
    # untouched slots keep their bits
    for s in range(W):
        if str(s) not in ex["expected_ring_k_after_commit_slot_element0"]:
            assert rk[0, 0, s, 0] == ring_k[0, 0, s, 0]


def test_geometry_cases():
    cases = json.loads((GOLDEN / "dflash2_geometry_cases.json").read_text())["cases"]
    for c in cases:
        assert oracle.ring_geometry_valid(c["geometry"]) == c["valid"], c["why"]
    base = [4, 32, 8, 128, 8, 2048, 2055, 8]
    bad = [
        [0, 32, 8, 128, 8, 2048, 2055, 8], [5, 32, 8, 128, 8, 2048, 2055, 8],
        [4, 30, 8, 128, 8, 2048, 2055, 8], [4, 32, 8, 64, 8, 2048, 2055, 8],
        [4, 32, 8, 128, 1, 2048, 2048, 1], [4, 32, 8, 128, 17, 2048, 2064, 8],
        [4, 32, 8, 128, 8, 8, 15, 8], [4, 32, 8, 128, 8, 2048, 2055, 0],
        [4, 32, 8, 128, 8, 2048, 2055, 9],
    ]
    assert oracle.ring_geometry_valid(base)
    assert oracle.ring_geometry_valid([4, 32, 8, 256, 16, 4096, 4111, 16])
    for g in bad:
        assert not oracle.ring_geometry_valid(g), g


def test_mask_rows_example():
    ex = json.loads((GOLDEN / "dflash2_mask_rows_example.json").read_text())
    emb = np.array([_bf16(x) for x in ex["mask_embedding"]], np.uint16)
    hid = np.array(ex["hidden_before"], np.float32).reshape(ex["lanes"] * ex["rows"], -1)
    out = oracle.set_mask_rows(emb, hid, ex["lanes"], ex["rows"])
    assert out.reshape(-1).tolist() == ex["hidden_after"]


def _ring_from_writes(W, D, wp0, n_writes):
    """Write tokens 1..n_writes one after another into a ring starting at slot
    wp0; element 0 of a slot holds the id of the token written there."""
    ring = np.zeros((1, 1, W, D), np.uint16)
    for t in range(1, n_writes + 1):
        ring[0, 0, (wp0 + t - 1) % W, 0] = _bf16(float(t))
    return ring, (wp0 + n_writes) % W, min(n_writes, W)


def test_history_order_follows_sequential_writes():
    D = 128
    for W, R in itertools.product((3, 4, 5, 8), (2, 3)):
        if W <= R:
            continue
        g = [1, 1, 1, D, R, W, W - 1 + R, R]
        for wp0, n in itertools.product(range(W), range(0, 2 * W + 1)):
            ring, wp, length = _ring_from_writes(W, D, wp0, n)
            zeros = np.zeros((1, R, 1, D), np.float32)
            _, pk, _ = oracle.pack_attention(ring, ring, zeros, zeros, zeros,
                                             np.array([length], np.uint32),
                                             np.array([wp], np.uint32), g)
            for j in range(W - 1):
                got = int(pk[0, 0, R + j, 0])
                want = _bf16(float(n - j)) if j < length else 0
                assert got == want, (W, R, wp0, n, j)
            m = oracle.fill_mask(np.array([length], np.uint32), g)[0, 0]
            for r in range(R):
                for j in range(W - 1):
                    # token n - j sits at position n - 1 - j; query r at n + r
                    visible = j < length and (n + r) - (n - 1 - j) < W
                    assert (m[r, R + j] == 0) == visible
                assert np.all(m[r, :R] == 0)


def test_commit_then_pack_returns_committed_rows_newest_first():
    c = workloads.ring(lanes=2, rows=4, window=9, q_heads=4, kv_heads=2, head_dim=128, seed=21)
    g = c.geom
    B, H, HK, D, R, W, K, MC = g
    rk, rv = oracle.commit_kv(c.new_k, c.new_v, c.commit_counts, c.write_positions,
                              c.ring_k, c.ring_v, g)
    n = np.minimum(c.commit_counts, MC)
    wp2 = ((c.write_positions + n) % W).astype(np.uint32)
    len2 = np.minimum(c.cache_lengths + n, W).astype(np.uint32)
    _, pk_old, pv_old = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                              c.cache_lengths, c.write_positions, g)
    _, pk, pv = oracle.pack_attention(rk, rv, c.cur_q, c.cur_k, c.cur_v, len2, wp2, g)
    nk = workloads.bf16_bits(c.new_k)
    nv = workloads.bf16_bits(c.new_v)
    for b in range(B):
        for j in range(W - 1):
            if j < n[b]:
                np.testing.assert_array_equal(pk[b, :, R + j], nk[b, n[b] - 1 - j])
                np.testing.assert_array_equal(pv[b, :, R + j], nv[b, n[b] - 1 - j])
            elif j < len2[b]:
                np.testing.assert_array_equal(pk[b, :, R + j], pk_old[b, :, R + j - n[b]])
                np.testing.assert_array_equal(pv[b, :, R + j], pv_old[b, :, R + j - n[b]])


def test_chain_equals_chronological_window_attention():
    c = workloads.ring(lanes=3, rows=5, window=12, q_heads=8, kv_heads=2, head_dim=128, seed=4)
    g = c.geom
    B, H, HK, D, R, W, K, MC = g
    pq, pk, pv = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                       c.cache_lengths, c.write_positions, g)
    mask = oracle.fill_mask(c.cache_lengths, g)
    out = oracle.verify_attention(pq, pk, pv, mask, g, c.scale)          # [B, R, H, D]
    ck = workloads.bf16_bits(c.cur_k)
    cv = workloads.bf16_bits(c.cur_v)
    cq = workloads.bf16_bits(c.cur_q)
    for b in range(B):
        L = int(min(c.cache_lengths[b], W))
        wp = int(c.write_positions[b]) % W
        # chronological keys: history positions 0..L-1 (oldest first), then the R current rows
        slots = [(wp - L + p) % W for p in range(L)]
        keys = np.concatenate([c.ring_k[b][:, slots].transpose(1, 0, 2),
                               ck[b]], axis=0)                              # [L+R, HK, D]
        vals = np.concatenate([c.ring_v[b][:, slots].transpose(1, 0, 2), cv[b]], axis=0)
        pos_k = np.arange(L + R)
        pos_q = L + np.arange(R)
        vis = (pos_k[None, :] >= L) | ((pos_q[:, None] - pos_k[None, :]) < W)
        m = workloads.bf16_bits(np.where(vis, 0.0, -np.inf).astype(np.float32))
        ref = oracle.attention(cq[b], np.ascontiguousarray(keys), np.ascontiguousarray(vals),
                               kv_dtype="bf16", q_dtype="bf16", scale=c.scale, mask=m,
                               mask_dtype="bf16")
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def test_counters_are_clamped():
    c = workloads.ring(lanes=2, rows=3, window=6, q_heads=2, kv_heads=1, head_dim=128, seed=8)
    g = c.geom
    big_len = np.array([100, 6], np.uint32)
    big_pos = np.array([6 * 7 + 2, 2], np.uint32)
    a = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v, big_len, big_pos, g)
    b = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                              np.array([6, 6], np.uint32), np.array([2, 2], np.uint32), g)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    rk1, _ = oracle.commit_kv(c.new_k, c.new_v, np.array([99, 3], np.uint32), big_pos,
                              c.ring_k, c.ring_v, g)
    rk2, _ = oracle.commit_kv(c.new_k, c.new_v, np.array([3, 3], np.uint32),
                              np.array([2, 2], np.uint32), c.ring_k, c.ring_v, g)
    np.testing.assert_array_equal(rk1, rk2)


# ---------------------------------------------------------------------------
# Ring-direct verify attention (the keys visited in ring-slot order)
# ---------------------------------------------------------------------------
def _chain(c, lens=None, pos=None):
    g = c.geom
    lens = c.cache_lengths if lens is None else lens
    pos = c.write_positions if pos is None else pos
    pq, pk, pv = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v, lens, pos, g)
    mask = oracle.fill_mask(lens, g)
    return oracle.verify_attention(pq, pk, pv, mask, g, c.scale)


def test_ring_direct_equals_pack_mask_verify_chain():
    """Same keys, values and visibility as the packed layout, visited in slot order;
    covers write positions that wrap, empty and full histories and clamped counters."""
    for seed, (R, W) in enumerate([(3, 11), (5, 12), (2, 40), (16, 37)]):
        c = workloads.ring(lanes=4, rows=R, window=W, q_heads=4, kv_heads=2, head_dim=128,
                           seed=20 + seed)
        lens = np.array([0, W - 1, W, 5 * W + 3][: 4], np.uint32)
        pos = np.array([W - 1, 0, W * 3 + 1, 2], np.uint32)
        for ln, ps in [(c.cache_lengths, c.write_positions), (lens, pos)]:
            got = oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                               ln, ps, c.geom, c.scale)
            np.testing.assert_allclose(got, _chain(c, ln, ps), rtol=1e-12, atol=1e-13)


def test_ring_direct_is_invariant_under_slot_rotation():
    """Rotating the ring contents by t slots together with the write position leaves
    every history index, hence the result, unchanged."""
    c = workloads.ring(lanes=2, rows=4, window=23, q_heads=4, kv_heads=1, head_dim=128, seed=31)
    base = oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                        c.cache_lengths, c.write_positions, c.geom, c.scale)
    for t in (1, 7, 22):
        rk = np.roll(c.ring_k, t, axis=2)
        rv = np.roll(c.ring_v, t, axis=2)
        pos = ((c.write_positions.astype(np.int64) + t) % 23).astype(np.uint32)
        got = oracle.verify_ring_attention(rk, rv, c.cur_q, c.cur_k, c.cur_v, c.cache_lengths,
                                           pos, c.geom, c.scale)
        np.testing.assert_allclose(got, base, rtol=1e-12, atol=1e-13)


def test_ring_direct_with_empty_history_is_attention_over_current_rows():
    c = workloads.ring(lanes=1, rows=6, window=10, q_heads=4, kv_heads=2, head_dim=128, seed=33)
    got = oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                       np.array([0], np.uint32), np.array([3], np.uint32),
                                       c.geom, c.scale)
    ref = oracle.attention(workloads.bf16_bits(c.cur_q[0]), workloads.bf16_bits(c.cur_k[0]),
                           workloads.bf16_bits(c.cur_v[0]), kv_dtype="bf16", q_dtype="bf16",
                           scale=c.scale)
    np.testing.assert_allclose(got[0], ref, rtol=1e-12, atol=1e-13)
