"""GPU parity of the tcgen05 prefill attention against the oracle, through the
C ABI: max |err| <= 1e-2 and mean |err| <= 1e-3."""
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


@pytest.fixture(params=[2, 0], ids=["cta_pairs", "single_ctas"])
def pairs_mode(request, lib):
    """Run a test with two-CTA clusters on for every eligible shape (mode 2) and
    off (mode 0); shapes that cannot pair take the single-CTA kernel either way."""
    lib.gqa_attn_set_cta_pairs(request.param)
    yield request.param
    lib.gqa_attn_set_cta_pairs(1)


def _run(g, c, q=None, k=None, v=None, mask=None):
    import torch
    from gpu_helpers import dev, new_status
    kind = "bf16" if c.kv_dtype == "bf16" else None
    st = new_status()
    out = g.gqa_attn_prefill(dev(c.q) if q is None else q, dev(c.k, kind) if k is None else k,
                             dev(c.v, kind) if v is None else v,
                             dev(c.mask) if mask is None else mask, c.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.cpu().numpy()


def _oracle(c, pairs=None):
    return oracle.attention(c.q, c.k, c.v, kv_dtype=c.kv_dtype, scale=c.scale, mask=c.mask,
                            pairs=pairs)


def test_tiny_prefill_full(lib):
    from gpu_helpers import assert_attention_close
    c = workloads.tiny_prefill()
    assert_attention_close(_run(lib, c), _oracle(c), "tiny prefill")


@pytest.mark.parametrize("rows,kv_len,h,hk,d,pos0,dtype", [
    (256, 256, 4, 2, 256, 0, "f16"),       # several row tiles, causal
    (200, 330, 4, 4, 128, 130, "f16"),     # ragged rows and keys, prefix offset
    (130, 130, 2, 1, 512, 0, "f16"),       # d512 in two output halves, ragged tail
    (96, 500, 8, 2, 256, 404, "bf16"),     # bf16 K/V, few rows, prefix
    (64, 64, 4, 2, 128, 0, "bf16"),
    (256, 384, 8, 2, 256, 128, "bf16"),    # two pairs per KV head, bf16, prefix
    (128, 4000, 2, 1, 256, 3872, "f16"),   # one pair, keys split across many clusters
    (300, 700, 4, 2, 512, 400, "f16"),     # d512 pairs, ragged rows and keys
    (48, 300, 16, 2, 128, 252, "f16"),     # 8 query heads per KV head, several heads per tile
    (33, 97, 8, 1, 256, 64, "bf16"),       # one KV head for 8 query heads, odd sizes
])
def test_prefill_shapes(lib, pairs_mode, rows, kv_len, h, hk, d, pos0, dtype):
    from gpu_helpers import assert_attention_close
    c = workloads.prefill(rows=rows, kv_len=kv_len, n_heads=h, n_kv_heads=hk, head_dim=d,
                          position0=pos0, q_std=d ** -0.5, scale=1.0, kv_dtype=dtype,
                          seed=rows + d)
    assert_attention_close(_run(lib, c), _oracle(c), f"prefill {rows}x{kv_len} d{d} {dtype}")


def test_windowed_and_fully_masked_rows(lib):
    from gpu_helpers import assert_attention_close, dev
    c = workloads.prefill(rows=192, kv_len=384, n_heads=4, n_kv_heads=2, head_dim=128,
                          position0=192, window=100, seed=11)
    c.mask[5] = np.float16(-np.inf)            # a row with no visible key -> zeros
    c.mask[77, ::3] = np.float16(-0.5)         # finite non-zero mask values
    got = _run(lib, c)
    assert np.all(got[5] == 0)
    assert_attention_close(got, _oracle(c), "windowed prefill")


def test_strided_qkv(lib):
    """Q, K and V views with padded row and head strides."""
    import torch
    from gpu_helpers import assert_attention_close, dev
    c = workloads.prefill(rows=160, kv_len=192, n_heads=4, n_kv_heads=2, head_dim=128, seed=21)
    qb = torch.zeros((160, 5, 136), dtype=torch.float32, device="cuda")
    qb[:, :4, :128] = dev(c.q)
    kb = torch.zeros((192, 3, 128), dtype=torch.float16, device="cuda")
    kb[:, :2] = dev(c.k)
    vb = torch.zeros((2, 192, 136), dtype=torch.float16, device="cuda")   # head-major V
    vb[:, :, 8:] = dev(c.v).permute(1, 0, 2)
    got = _run(lib, c, q=qb[:, :4, :128], k=kb[:, :2], v=vb[:, :, 8:].permute(1, 0, 2))
    assert_attention_close(got, _oracle(c), "strided prefill")


_FULL_REF = {}


def _full_ref(name, c, pairs=None):
    """The oracle's result for a full-size workload, computed once per module (both
    tiling modes compare against it)."""
    if name not in _FULL_REF:
        _FULL_REF[name] = _oracle(c, pairs)
    return _FULL_REF[name]


def test_full_size_d256(lib, pairs_mode):
    """2048 causal queries over 2048 keys, 16/8 heads, d256: every (row, head) output."""
    from gpu_helpers import assert_attention_close
    c = workloads.prefill_d256()
    got = _run(lib, c)
    assert_attention_close(got, _full_ref("d256", c), "prefill d256 full size")


def _d512_pairs(c):
    """Every row of four heads: two heads of KV group 0 (one CTA pair), and one head of
    each half of KV group 1."""
    heads = np.array([0, 1, 9, c.n_heads - 1])
    rows = np.arange(c.rows)
    return np.stack([np.repeat(rows, heads.size), np.tile(heads, c.rows)], axis=1).astype(np.int32)


def test_full_size_d512_prefix(lib, pairs_mode):
    """1024 queries at positions 7168..8191 over 8192 keys, 16/2 heads, d512: every
    output is finite, and every row of four heads (both output halves) matches."""
    from gpu_helpers import assert_attention_close
    c = workloads.prefill_d512_prefix()
    got = _run(lib, c)
    assert np.all(np.isfinite(got))
    pairs = _d512_pairs(c)
    ref = _full_ref("d512", c, pairs)
    assert_attention_close(got[pairs[:, 0], pairs[:, 1]], ref, "prefill d512 full size")


def test_invalid_arguments_are_rejected(lib):
    import torch
    from attention_gqa_flash_gb300 import GQAError
    from gpu_helpers import dev
    c = workloads.tiny_prefill()
    q, k, v, m = dev(c.q), dev(c.k), dev(c.v), dev(c.mask)
    with pytest.raises(GQAError, match="n_heads"):
        lib.gqa_attn_prefill(q[:, :3], k, v, m, 1.0)
    with pytest.raises(GQAError, match="kv_pad"):
        lib.gqa_attn_prefill(q, k[:60], v[:60], m[:, :60].contiguous(), 1.0)
    with pytest.raises(GQAError, match="head_dim"):
        lib.gqa_attn_prefill(q[..., :64], k[..., :64], v[..., :64], m, 1.0)
    small = torch.empty((64, 4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(GQAError, match="o holds"):
        lib.gqa_attn_prefill(q, k, v, m, 1.0, out=small)
