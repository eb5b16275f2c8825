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


def _oracle_chain(c, lengths=None):
    """The oracle's own pack and mask from the host inputs, and its attention over them
    (nothing here comes from the GPU)."""
    lengths = c.cache_lengths if lengths is None else lengths
    opq, opk, opv = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                          lengths, c.write_positions, c.geom)
    omask = oracle.fill_mask(lengths, c.geom)
    return opq, opk, opv, omask


def _check_chain(got, pq, pk, pv, mask, ref_ops, what, scale, geom):
    """The GPU's pack and mask bit for bit, then its attention against the oracle's
    attention over the oracle's own packed operands."""
    from gpu_helpers import assert_attention_close
    opq, opk, opv, omask = ref_ops
    np.testing.assert_array_equal(pq, opq)
    np.testing.assert_array_equal(pk, opk)
    np.testing.assert_array_equal(pv, opv)
    np.testing.assert_array_equal(mask, omask)
    ref = oracle.verify_attention(opq, opk, opv, omask, geom, scale)
    assert_attention_close(got, ref, what)


@pytest.mark.parametrize("lanes,rows,window,h,hk,d", [
    (1, 2, 5, 2, 1, 128), (2, 16, 200, 8, 2, 128), (3, 8, 150, 8, 8, 256), (4, 16, 700, 32, 8, 256)])
def test_verify_attention_small(lib, lanes, rows, window, h, hk, d):
    c = workloads.ring(lanes=lanes, rows=rows, window=window, q_heads=h, kv_heads=hk,
                       head_dim=d, seed=window)
    got, pq, pk, pv, mask = _verify(lib, c)
    _check_chain(got, pq, pk, pv, mask, _oracle_chain(c), f"verify lanes{lanes} r{rows} w{window} d{d}",
                 c.scale, c.geom)


def test_verify_empty_history(lib):
    c = workloads.ring(lanes=2, rows=4, window=70, q_heads=4, kv_heads=2, head_dim=128, seed=9)
    lengths = np.array([0, 69], np.uint32)
    got, pq, pk, pv, mask = _verify(lib, c, lengths)
    _check_chain(got, pq, pk, pv, mask, _oracle_chain(c, lengths), "verify empty history",
                 c.scale, c.geom)


def test_full_size_verify(lib):
    """lanes 4, rows 16, window 4096, h32/hk8, d256: every pack and mask bit, and every
    (lane, row, head) output against the oracle's attention over its own packed operands."""
    c = workloads.verify_full(seed=0)
    got, pq, pk, pv, mask = _verify(lib, c)
    _check_chain(got, pq, pk, pv, mask, _oracle_chain(c), "full-size verify", c.scale, c.geom)
