"""GPU parity of the fused ring-direct verify attention, through the C ABI: against
the oracle's ring-direct definition and against the unfused GPU chain
pack -> mask -> verify (max |err| <= 1e-2, mean |err| <= 1e-3 for both)."""
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


def _expect_status(lens, pos, window):
    """Out-of-range counters are clamped and flagged (GQA_FLAG_RING_CLAMPED) by the fused
    kernel exactly as by the pack and mask kernels."""
    return 4 if (np.any(lens > window) or np.any(pos >= window)) else 0


def _fused(g, c, lens, pos):
    import torch
    from gpu_helpers import dev, new_status
    st = new_status()
    out = g.gqa_attn_verify_ring(dev(c.ring_k, "bf16"), dev(c.ring_v, "bf16"), dev(c.cur_q),
                                 dev(c.cur_k), dev(c.cur_v), dev(lens, "u32"), dev(pos, "u32"),
                                 c.geom, c.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == _expect_status(lens, pos, c.geom[5])
    return out.cpu().numpy()


def _chain(g, c, lens, pos):
    import torch
    from gpu_helpers import dev, new_status
    B, H, HK, D, R, W, K, MC = c.geom
    pq = torch.empty((B, H, R, D), dtype=torch.bfloat16, device="cuda")
    pk = torch.empty((B, HK, K, D), dtype=torch.bfloat16, device="cuda")
    pv = torch.empty_like(pk)
    mask = torch.empty((B, H, R, K), dtype=torch.bfloat16, device="cuda")
    st = new_status()
    g.gqa_pack_attention(dev(c.ring_k, "bf16"), dev(c.ring_v, "bf16"), dev(c.cur_q), dev(c.cur_k),
                         dev(c.cur_v), dev(lens, "u32"), dev(pos, "u32"), pq, pk, pv, c.geom,
                         status=st)
    g.gqa_fill_mask(dev(lens, "u32"), mask, c.geom, status=st)
    out = g.gqa_attn_verify(pq, pk, pv, mask, c.geom, c.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == _expect_status(lens, pos, c.geom[5])
    return out.cpu().numpy()


@pytest.mark.parametrize("lanes,rows,window,h,hk,d", [
    (4, 16, 512, 8, 2, 256),      # whole tiles
    (3, 5, 300, 4, 1, 256),       # window not a multiple of the 128-key tile
    (2, 16, 1000, 8, 8, 128),     # head_dim 128, one query head per KV head
    (4, 2, 129, 4, 2, 128),       # one full ring tile plus one slot
])
def test_fused_matches_oracle_and_chain(lib, lanes, rows, window, h, hk, d):
    from gpu_helpers import assert_attention_close
    c = workloads.ring(lanes=lanes, rows=rows, window=window, q_heads=h, kv_heads=hk,
                       head_dim=d, seed=window + rows)
    cases = [(c.cache_lengths, c.write_positions)]
    # empty, full and over-long histories; write positions at both ends and past the window
    edge_len = np.array([0, window - 1, window, 7 * window + 5][:lanes], np.uint32)
    edge_pos = np.array([0, window - 1, 3 * window + 2, 1][:lanes], np.uint32)
    cases.append((edge_len, edge_pos))
    for lens, pos in cases:
        got = _fused(lib, c, lens, pos)
        ref = oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v, lens,
                                           pos, c.geom, c.scale)
        assert_attention_close(got, ref, f"fused verify w{window} r{rows} d{d}")
        assert_attention_close(got, _chain(lib, c, lens, pos).astype(np.float64),
                               f"fused vs chain w{window} r{rows} d{d}")


def test_fused_full_size(lib):
    """lanes 4, rows 16, window 4096, 32 / 8 heads, head_dim 256."""
    from gpu_helpers import assert_attention_close
    c = workloads.verify_full(seed=0)
    got = _fused(lib, c, c.cache_lengths, c.write_positions)
    assert np.all(np.isfinite(got))
    ref = oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                       c.cache_lengths, c.write_positions, c.geom, c.scale)
    assert_attention_close(got, ref, "fused verify full size")
    assert_attention_close(got, _chain(lib, c, c.cache_lengths, c.write_positions).astype(np.float64),
                           "fused vs chain full size")


def test_fused_long_window_uses_fixed_key_ranges(lib):
    """A window of 20000 slots (158 key tiles, more than a unit's tile list holds): the
    splits fall back to fixed key ranges; results still match the oracle."""
    from gpu_helpers import assert_attention_close
    c = workloads.ring(lanes=2, rows=8, window=20000, q_heads=4, kv_heads=1, head_dim=128, seed=77)
    lens = np.array([19990, 7000], np.uint32)
    pos = np.array([123, 19999], np.uint32)
    got = _fused(lib, c, lens, pos)
    ref = oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v, lens, pos,
                                       c.geom, c.scale)
    assert_attention_close(got, ref, "fused verify, window 20000")
