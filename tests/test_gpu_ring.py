"""GPU parity of the DFlash2 ring-KV kernels (pack, mask, commit, draft mask
rows) against the oracle: bit-exact, through the C ABI."""
import json
import pathlib

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

GOLDEN = pathlib.Path(__file__).parent / "golden"


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_gqa_flash_gb300 as g
    g.library()
    return g


def _run_chain(g, c, lengths=None, positions=None, counts=None):
    import torch
    from gpu_helpers import dev, host_bits, new_status
    B, H, HK, D, R, W, K, MC = c.geom
    lengths = c.cache_lengths if lengths is None else lengths
    positions = c.write_positions if positions is None else positions
    counts = c.commit_counts if counts is None else counts
    rk, rv = dev(c.ring_k, "bf16"), dev(c.ring_v, "bf16")
    pq = torch.empty((B, H, R, D), dtype=torch.bfloat16, device="cuda")
    pk = torch.empty((B, HK, K, D), dtype=torch.bfloat16, device="cuda")
    pv = torch.empty_like(pk)
    mask = torch.empty((B, H, R, K), dtype=torch.bfloat16, device="cuda")
    st = new_status()
    g.gqa_pack_attention(rk, rv, dev(c.cur_q), dev(c.cur_k), dev(c.cur_v), dev(lengths, "u32"),
                         dev(positions, "u32"), pq, pk, pv, c.geom, status=st)
    g.gqa_fill_mask(dev(lengths, "u32"), mask, c.geom, status=st)
    g.gqa_commit_kv(dev(c.new_k), dev(c.new_v), dev(counts, "u32"), dev(positions, "u32"),
                    rk, rv, c.geom, status=st)
    torch.cuda.synchronize()
    return (host_bits(pq), host_bits(pk), host_bits(pv), host_bits(mask), host_bits(rk),
            host_bits(rv), int(st.item()))


def _oracle_chain(c, lengths=None, positions=None, counts=None):
    lengths = c.cache_lengths if lengths is None else lengths
    positions = c.write_positions if positions is None else positions
    counts = c.commit_counts if counts is None else counts
    pq, pk, pv = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v, lengths,
                                       positions, c.geom)
    m = oracle.fill_mask(lengths, c.geom)
    rk, rv = oracle.commit_kv(c.new_k, c.new_v, counts, positions, c.ring_k, c.ring_v, c.geom)
    return pq, pk, pv, m, rk, rv


def _assert_same(got, ref):
    names = ("packed_q", "packed_k", "packed_v", "mask", "ring_k", "ring_v")
    for name, a, b in zip(names, got, ref):
        np.testing.assert_array_equal(a, b, err_msg=name)


def test_worked_example_through_the_abi(lib):
    import torch
    from gpu_helpers import dev, host_bits
    ex = json.loads((GOLDEN / "dflash2_worked_example.json").read_text())
    gd = ex["geometry"]
    geom = [gd[k] for k in ("lanes", "q_heads", "kv_heads", "head_dim", "rows", "window",
                            "packed_len", "max_commit")]
    B, H, HK, D, R, W, K, MC = geom
    bf = lambda x: int(workloads.bf16_bits(np.array([x], np.float32))[0])
    ring_k = np.zeros((B, HK, W, D), np.uint16)
    ring_v = np.zeros((B, HK, W, D), np.uint16)
    for s in range(W):
        ring_k[0, 0, s, 0] = bf(ex["ring_k_slot_element0"][s])
        ring_v[0, 0, s, 0] = bf(ex["ring_v_slot_element0"][s])
    cq = np.zeros((B, R, H, D), np.float32)
    ck = np.zeros((B, R, HK, D), np.float32)
    cv = np.zeros((B, R, HK, D), np.float32)
    for r in range(R):
        cq[0, r, 0, 0] = ex["current_q_row_element0"][r]
        ck[0, r, 0, 0] = ex["current_k_row_element0"][r]
        cv[0, r, 0, 0] = ex["current_v_row_element0"][r]
    rk, rv = dev(ring_k, "bf16"), dev(ring_v, "bf16")
    lens = dev(np.array([ex["cache_length"]], np.uint32), "u32")
    pos = dev(np.array([ex["write_position"]], np.uint32), "u32")
    pq = torch.empty((B, H, R, D), dtype=torch.bfloat16, device="cuda")
    pk = torch.empty((B, HK, K, D), dtype=torch.bfloat16, device="cuda")
    pv = torch.empty_like(pk)
    mask = torch.empty((B, H, R, K), dtype=torch.bfloat16, device="cuda")
    lib.gqa_pack_attention(rk, rv, dev(cq), dev(ck), dev(cv), lens, pos, pq, pk, pv, geom)
    lib.gqa_fill_mask(lens, mask, geom)
    torch.cuda.synchronize()
    assert host_bits(pq)[0, 0, 0, 0] == bf(ex["expected_packed_q_element0"])
    assert host_bits(pk)[0, 0, :, 0].tolist() == [bf(x) for x in
                                                  ex["expected_packed_k_column_element0"]]
    assert host_bits(mask).reshape(-1).tolist() == [0 if m == "0" else 0xff80
                                                    for m in ex["expected_mask_flat"]]
    counts = dev(np.array([ex["commit_count"]], np.uint32), "u32")
    lib.gqa_commit_kv(dev(ck), dev(cv), counts, pos, rk, rv, geom)
    torch.cuda.synchronize()
    got = host_bits(rk)
    for slot, val in ex["expected_ring_k_after_commit_slot_element0"].items():
        assert got[0, 0, int(slot), 0] == bf(val)


@pytest.mark.parametrize("lanes,rows,window,h,hk,d", [
    (1, 2, 5, 2, 1, 128), (3, 5, 37, 8, 2, 128), (4, 16, 300, 8, 4, 256), (2, 7, 64, 12, 3, 256)])
def test_chain_matches_oracle_bit_exact(lib, lanes, rows, window, h, hk, d):
    c = workloads.ring(lanes=lanes, rows=rows, window=window, q_heads=h, kv_heads=hk,
                       head_dim=d, seed=lanes * 100 + rows)
    got = _run_chain(lib, c)
    assert got[-1] == 0
    _assert_same(got[:-1], _oracle_chain(c))


def test_edge_counters(lib):
    c = workloads.ring(lanes=4, rows=4, window=9, q_heads=4, kv_heads=2, head_dim=128, seed=77)
    lengths = np.array([0, 9, 8, 1], np.uint32)          # empty, full window, window-1, one
    positions = np.array([0, 8, 3, 5], np.uint32)        # wrap-around at the end
    counts = np.array([0, 4, 1, 3], np.uint32)           # nothing, all, one, some
    got = _run_chain(lib, c, lengths, positions, counts)
    assert got[-1] == 0
    _assert_same(got[:-1], _oracle_chain(c, lengths, positions, counts))


def test_out_of_range_counters_are_clamped_and_flagged(lib):
    from attention_gqa_flash_gb300 import GQA_FLAG_RING_CLAMPED
    c = workloads.ring(lanes=2, rows=3, window=6, q_heads=2, kv_heads=1, head_dim=128, seed=5)
    lengths = np.array([100, 2], np.uint32)
    positions = np.array([6 * 3 + 4, 1], np.uint32)
    counts = np.array([50, 2], np.uint32)
    got = _run_chain(lib, c, lengths, positions, counts)
    assert got[-1] & GQA_FLAG_RING_CLAMPED
    _assert_same(got[:-1], _oracle_chain(c, lengths, positions, counts))


def test_full_size_verify_ring(lib):
    c = workloads.verify_full(seed=0)
    got = _run_chain(lib, c)
    assert got[-1] == 0
    _assert_same(got[:-1], _oracle_chain(c))


def test_set_mask_rows_example_and_random(lib):
    import torch
    from gpu_helpers import dev
    ex = json.loads((GOLDEN / "dflash2_mask_rows_example.json").read_text())
    emb = workloads.bf16_bits(np.array(ex["mask_embedding"], np.float32))
    hid = dev(np.array(ex["hidden_before"], np.float32).reshape(ex["lanes"] * ex["rows"], -1))
    lib.gqa_set_mask_rows(dev(emb, "bf16"), hid, ex["lanes"], ex["rows"])
    torch.cuda.synchronize()
    assert hid.cpu().numpy().reshape(-1).tolist() == ex["hidden_after"]
    rng = np.random.default_rng(3)
    emb = workloads.bf16_bits(rng.standard_normal(1000).astype(np.float32))
    hidden = rng.standard_normal((4 * 16, 1000)).astype(np.float32)
    h = dev(hidden)
    lib.gqa_set_mask_rows(dev(emb, "bf16"), h, 4, 16)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(h.cpu().numpy(), oracle.set_mask_rows(emb, hidden, 4, 16))
