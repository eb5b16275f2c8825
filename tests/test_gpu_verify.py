"""GPU parity of the speculative-verify chain: pack -> mask -> attention ->
commit, through the C ABI, against the oracle (bit-exact for the ring ops,
max |err| <= 1e-2 / mean |err| <= 1e-3 for the attention)."""
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


def _verify(g, c, lengths=None):
    import torch
    from gpu_helpers import dev, host_bits, new_status
    B, H, HK, D, R, W, K, MC = c.geom
    lengths = c.cache_lengths if lengths is None else lengths
    pq = torch.empty((B, H, R, D), dtype=torch.bfloat16, device="cuda")
    pk = torch.empty((B, HK, K, D), dtype=torch.bfloat16, device="cuda")
    pv = torch.empty_like(pk)
    mask = torch.empty((B, H, R, K), dtype=torch.bfloat16, device="cuda")
    st = new_status()
    g.gqa_pack_attention(dev(c.ring_k, "bf16"), dev(c.ring_v, "bf16"), dev(c.cur_q),
                         dev(c.cur_k), dev(c.cur_v), dev(lengths, "u32"),
                         dev(c.write_positions, "u32"), pq, pk, pv, c.geom, status=st)
    g.gqa_fill_mask(dev(lengths, "u32"), mask, c.geom, status=st)
    out = g.gqa_attn_verify(pq, pk, pv, mask, c.geom, c.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.cpu().numpy(), host_bits(pq), host_bits(pk), host_bits(pv), host_bits(mask)


@pytest.mark.parametrize("lanes,rows,window,h,hk,d", [
    (1, 2, 5, 2, 1, 128), (2, 16, 200, 8, 2, 128), (3, 8, 150, 8, 8, 256), (4, 16, 700, 32, 8, 256)])
def test_verify_attention_small(lib, lanes, rows, window, h, hk, d):
    from gpu_helpers import assert_attention_close
    c = workloads.ring(lanes=lanes, rows=rows, window=window, q_heads=h, kv_heads=hk,
                       head_dim=d, seed=window)
    got, pq, pk, pv, mask = _verify(lib, c)
    ref = oracle.verify_attention(pq, pk, pv, mask, c.geom, c.scale)
    assert_attention_close(got, ref, f"verify lanes{lanes} r{rows} w{window} d{d}")


def test_verify_empty_history(lib):
    from gpu_helpers import assert_attention_close
    c = workloads.ring(lanes=2, rows=4, window=70, q_heads=4, kv_heads=2, head_dim=128, seed=9)
    lengths = np.array([0, 69], np.uint32)
    got, pq, pk, pv, mask = _verify(lib, c, lengths)
    ref = oracle.verify_attention(pq, pk, pv, mask, c.geom, c.scale)
    assert_attention_close(got, ref, "verify empty history")


def test_full_size_verify_sampled(lib):
    """lanes 4, rows 16, window 4096, h32/hk8, d256: every pack/mask bit, sampled outputs."""
    from gpu_helpers import assert_attention_close
    c = workloads.verify_full(seed=0)
    got, pq, pk, pv, mask = _verify(lib, c)
    opq, opk, opv = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                          c.cache_lengths, c.write_positions, c.geom)
    np.testing.assert_array_equal(pq, opq)
    np.testing.assert_array_equal(pk, opk)
    np.testing.assert_array_equal(pv, opv)
    np.testing.assert_array_equal(mask, oracle.fill_mask(c.cache_lengths, c.geom))
    rng = np.random.default_rng(0)
    B, H, HK, D, R = c.geom[:5]
    pairs = [np.stack([rng.integers(0, R, 24), rng.integers(0, H, 24)], 1).astype(np.int32)
             for _ in range(B)]
    for p in pairs:
        p[:2] = [[0, 0], [R - 1, H - 1]]
    refs = oracle.verify_attention(pq, pk, pv, mask, c.geom, c.scale, pairs_per_lane=pairs)
    for b in range(B):
        assert_attention_close(got[b, pairs[b][:, 0], pairs[b][:, 1]], refs[b], f"lane {b}")
