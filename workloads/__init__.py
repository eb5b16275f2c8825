"""Seeded synthetic inputs for the GQA attention library.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic.  Both the oracle-side tests and the CUDA-side
tests/benchmark take their inputs from here, so the two sides see the same
bits.  All draws use ``numpy.random.default_rng(seed)`` in a fixed order,
as float32, then cast to the stored precision (f16 through NumPy, bf16
through PyTorch's CPU cast; both round to nearest even).

Workload shapes follow the pages' geometries:
  * prefill with an additive causal mask (mlx-native flash_attn_prefill_tensor.rs:
    f32 Q, f16 K/V with row/head strides, f16 mask [rows, kv_pad], kv_pad a
    multiple of 64);
  * paged decode over 16-token pages placed by a random permutation of the
    page pool (ferrum-kernels causal_attention.rs: 64 KiB pages of 16 tokens);
  * the DFlash2 ring KV for speculative verify (mlx-native dflash2_attention_pack.rs).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

F16_NEG_INF = np.float16(-np.inf)
CHUNK = 1 << 24


def _normal_f32(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    flat = out.reshape(-1)
    for s in range(0, flat.size, CHUNK):
        n = min(CHUNK, flat.size - s)
        flat[s:s + n] = rng.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        flat *= np.float32(std)
    return out


def _normal_f16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    flat = out.reshape(-1)
    for s in range(0, flat.size, CHUNK):
        n = min(CHUNK, flat.size - s)
        x = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        flat[s:s + n] = x.astype(np.float16)
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16) through PyTorch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).reshape(np.shape(x))


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    for s in range(0, flat.size, CHUNK):
        n = min(CHUNK, flat.size - s)
        x = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        flat[s:s + n] = bf16_bits(x)
    return out


def kv_pad_of(kv_len: int, step: int = 64) -> int:
    """kv_len rounded up to the 64-row cache step (a layout helper)."""
    return -(-kv_len // step) * step


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillCase:
    name: str
    rows: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    kv_len: int
    kv_pad: int
    position0: int
    scale: float
    kv_dtype: str
    q: np.ndarray      # f32 [rows, n_heads, head_dim]
    k: np.ndarray      # f16 or bf16-bits [kv_pad, n_kv_heads, head_dim]; rows >= kv_len zero
    v: np.ndarray
    mask: np.ndarray   # f16 [rows, kv_pad]: 0 where visible, -inf elsewhere

    @property
    def visible_pairs(self) -> int:
        """Number of (query row, key) pairs with a zero mask entry."""
        return int(np.count_nonzero(self.mask == 0))

    def flops(self) -> float:
        """Algorithmic FLOPs: 2*d for Q.K and 2*d for P.V per visible pair and head."""
        return 4.0 * self.n_heads * self.head_dim * self.visible_pairs


def causal_mask(rows: int, kv_len: int, kv_pad: int, position0: int,
                window: int | None = None) -> np.ndarray:
    """Additive f16 mask: query r sits at position position0 + r and sees key
    c when c <= position0 + r and c < kv_len (and, with a window, when the
    key is within `window` positions of the query)."""
    r = np.arange(rows)[:, None] + position0
    c = np.arange(kv_pad)[None, :]
    vis = (c <= r) & (c < kv_len)
    if window is not None:
        vis &= (r - c) < window
    return np.where(vis, np.float16(0), F16_NEG_INF).astype(np.float16)


def prefill(*, rows: int, kv_len: int, n_heads: int, n_kv_heads: int, head_dim: int,
            position0: int = 0, q_std: float = 1.0, scale: float | None = None,
            kv_dtype: str = "f16", seed: int = 0, name: str = "prefill",
            window: int | None = None) -> PrefillCase:
    rng = np.random.default_rng(seed)
    kv_pad = kv_pad_of(kv_len)
    q = _normal_f32(rng, (rows, n_heads, head_dim), q_std)
    draw = _normal_f16 if kv_dtype == "f16" else _normal_bf16
    k = draw(rng, (kv_pad, n_kv_heads, head_dim))
    v = draw(rng, (kv_pad, n_kv_heads, head_dim))
    k[kv_len:] = 0
    v[kv_len:] = 0
    mask = causal_mask(rows, kv_len, kv_pad, position0, window)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PrefillCase(name, rows, n_heads, n_kv_heads, head_dim, kv_len, kv_pad, position0,
                       float(scale), kv_dtype, q, k, v, mask)


def tiny_prefill(seed: int = 0) -> PrefillCase:
    """64 queries over 64 keys, 4 query heads / 2 KV heads, head_dim 128, causal,
    Q ~ N(0,1) f32, K/V ~ N(0,1) f16, scale 1/sqrt(128)."""
    return prefill(rows=64, kv_len=64, n_heads=4, n_kv_heads=2, head_dim=128,
                   scale=1.0 / math.sqrt(128), seed=seed, name="tiny_prefill_64x64_h4_hk2_d128")


def prefill_d256(seed: int = 0, rows: int = 2048) -> PrefillCase:
    """2048 causal queries over 2048 keys, 16 / 8 heads, head_dim 256,
    Q ~ N(0, 1/16) f32 (standard deviation 1/16), K/V ~ N(0,1) f16, scale 1."""
    return prefill(rows=rows, kv_len=rows, n_heads=16, n_kv_heads=8, head_dim=256,
                   q_std=1.0 / 16, scale=1.0, seed=seed,
                   name=f"prefill_causal_{rows}x{rows}_h16_hk8_d256")


def prefill_d512_prefix(seed: int = 0, rows: int = 1024, kv_len: int = 8192) -> PrefillCase:
    """1024 new queries at positions 7168..8191 over 8192 keys (a cached prefix of
    7168), 16 / 2 heads, head_dim 512, Q ~ N(0, 1/sqrt(512)), K/V ~ N(0,1) f16, scale 1."""
    return prefill(rows=rows, kv_len=kv_len, n_heads=16, n_kv_heads=2, head_dim=512,
                   position0=kv_len - rows, q_std=1.0 / math.sqrt(512), scale=1.0, seed=seed,
                   name=f"prefill_prefix_{rows}x{kv_len}_h16_hk2_d512")


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeCase:
    name: str
    num_seqs: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_pages_per_seq: int
    scale: float
    kv_dtype: str
    q: np.ndarray             # f32 [num_seqs, n_heads, head_dim]
    k_pool: np.ndarray        # [num_pages, page_size, n_kv_heads, head_dim]
    v_pool: np.ndarray
    page_table: np.ndarray    # int32 [num_seqs, max_pages_per_seq], -1 where unused
    context_lens: np.ndarray  # int32 [num_seqs]

    def kv_bytes(self) -> int:
        """K and V bytes the decode must read: every context token's K and V rows."""
        return int(self.context_lens.astype(np.int64).sum()) * self.n_kv_heads * \
            self.head_dim * 2 * 2


def paged_decode(*, num_seqs: int = 64, ctx_lo: int = 512, ctx_hi: int = 16384,
                 num_pages: int = 65536, page_size: int = 16, n_heads: int = 32,
                 n_kv_heads: int = 8, head_dim: int = 128, kv_dtype: str = "f16",
                 scale: float | None = None, seed: int = 0, name: str | None = None,
                 fixed_lens=None) -> DecodeCase:
    """context_lens ~ U{ctx_lo..ctx_hi}; pages are taken in order from a random
    permutation of the pool; unused pages and the unused tail of each
    sequence's last page are NaN, so a stray read poisons the result.
    fixed_lens (optional) replaces the first len(fixed_lens) drawn lengths
    before pages are assigned."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi, size=num_seqs, endpoint=True).astype(np.int32)
    if fixed_lens is not None:
        ctx[:len(fixed_lens)] = fixed_lens
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = -(-ctx_hi // page_size)
    need = -(-ctx.astype(np.int64) // page_size)
    if need.sum() > num_pages:
        raise ValueError("pool too small for the drawn context lengths")
    table = np.full((num_seqs, max_pages), -1, dtype=np.int32)
    used = np.zeros(num_pages, dtype=bool)
    pos = 0
    for s in range(num_seqs):
        ids = perm[pos:pos + need[s]]
        table[s, :need[s]] = ids
        used[ids] = True
        pos += int(need[s])
    q = _normal_f32(rng, (num_seqs, n_heads, head_dim))
    draw = _normal_f16 if kv_dtype == "f16" else _normal_bf16
    shape = (num_pages, page_size, n_kv_heads, head_dim)
    k_pool = draw(rng, shape)
    v_pool = draw(rng, shape)
    nan = np.float16(np.nan) if kv_dtype == "f16" else np.uint16(0x7fc0)
    k_pool[~used] = nan
    v_pool[~used] = nan
    for s in range(num_seqs):
        tail = int(ctx[s]) % page_size
        if tail:
            last = table[s, need[s] - 1]
            k_pool[last, tail:] = nan
            v_pool[last, tail:] = nan
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    if name is None:
        name = (f"paged_decode_{num_seqs}seq_ctx{ctx_lo}-{ctx_hi}_pool{num_pages}x{page_size}"
                f"_h{n_heads}_hk{n_kv_heads}_d{head_dim}")
    return DecodeCase(name, num_seqs, n_heads, n_kv_heads, head_dim, page_size, num_pages,
                      max_pages, float(scale), kv_dtype, q, k_pool, v_pool, table, ctx)


# ---------------------------------------------------------------------------
# paged chunked prefill and page append
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class PagedChunkCase:
    name: str
    num_seqs: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    max_pages_per_seq: int
    scale: float
    kv_dtype: str
    q: np.ndarray               # f32 [tokens, n_heads, head_dim]
    k_new: np.ndarray           # f32 [tokens, n_kv_heads, head_dim]: the new tokens' K / V
    v_new: np.ndarray
    k_pool: np.ndarray          # [num_pages, page_size, n_kv_heads, head_dim]: the prefix
    v_pool: np.ndarray          #   written, the new tokens' slots and unused pages NaN
    page_table: np.ndarray      # int32 [num_seqs, max_pages_per_seq], -1 where unused
    token_offsets: np.ndarray   # int32 [num_seqs + 1]
    position_start: np.ndarray  # int32 [num_seqs]

    @property
    def tokens(self) -> int:
        return int(self.token_offsets[-1])

    def flops(self) -> float:
        """4 h d per (query, visible key): query j of sequence s sees position_start + j + 1 keys."""
        n = 0
        for s in range(self.num_seqs):
            t = int(self.token_offsets[s + 1] - self.token_offsets[s])
            n += t * int(self.position_start[s]) + t * (t + 1) // 2
        return 4.0 * self.n_heads * self.head_dim * n


def paged_chunk(*, num_seqs: int = 4, tokens_lo: int = 1, tokens_hi: int = 64,
                prefix_lo: int = 0, prefix_hi: int = 300, num_pages: int = 256,
                page_size: int = 16, n_heads: int = 8, n_kv_heads: int = 2, head_dim: int = 128,
                kv_dtype: str = "f16", scale: float | None = None, seed: int = 0,
                name: str | None = None) -> PagedChunkCase:
    """tokens ~ U{tokens_lo..tokens_hi}, position_start ~ U{prefix_lo..prefix_hi} per
    sequence; pages taken in order from a random permutation of the pool; the prefix's K/V
    ~ N(0,1) in the pool, the new tokens' K/V ~ N(0,1) f32 (to be appended) and their slots,
    the unused pages and page tails NaN; Q ~ N(0,1) f32."""
    rng = np.random.default_rng(seed)
    toks = rng.integers(tokens_lo, tokens_hi, size=num_seqs, endpoint=True).astype(np.int32)
    ps = rng.integers(prefix_lo, prefix_hi, size=num_seqs, endpoint=True).astype(np.int32)
    ctx = (ps + toks).astype(np.int64)
    need = -(-ctx // page_size)
    max_pages = int(need.max())
    if need.sum() > num_pages:
        raise ValueError("pool too small")
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((num_seqs, max_pages), -1, np.int32)
    pos = 0
    for s in range(num_seqs):
        table[s, :need[s]] = perm[pos:pos + need[s]]
        pos += int(need[s])
    draw = _normal_f16 if kv_dtype == "f16" else _normal_bf16
    shape = (num_pages, page_size, n_kv_heads, head_dim)
    k_pool, v_pool = draw(rng, shape), draw(rng, shape)
    nan = np.float16(np.nan) if kv_dtype == "f16" else np.uint16(0x7fc0)
    written = np.zeros((num_pages, page_size), bool)
    for s in range(num_seqs):
        t = np.arange(int(ps[s]))
        written[table[s, t // page_size], t % page_size] = True
    k_pool[~written] = nan
    v_pool[~written] = nan
    offs = np.concatenate([[0], np.cumsum(toks)]).astype(np.int32)
    T = int(offs[-1])
    q = _normal_f32(rng, (T, n_heads, head_dim))
    k_new = _normal_f32(rng, (T, n_kv_heads, head_dim))
    v_new = _normal_f32(rng, (T, n_kv_heads, head_dim))
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    if name is None:
        name = (f"paged_chunk_{num_seqs}seq_tok{tokens_lo}-{tokens_hi}_pre{prefix_lo}-{prefix_hi}"
                f"_h{n_heads}_hk{n_kv_heads}_d{head_dim}")
    return PagedChunkCase(name, num_seqs, n_heads, n_kv_heads, head_dim, page_size, num_pages,
                          max_pages, float(scale), kv_dtype, q, k_new, v_new, k_pool, v_pool,
                          table, offs, ps)


def paged_chunk_full(seed: int = 0) -> PagedChunkCase:
    """Chunked prefill shaped like the paged causal-attention pages' model geometry:
    16 query heads over 4 KV heads of head_dim 256, so one token's K and V take
    4096 bytes of f16 and a 64 KiB page holds 16 tokens; 8 sequences of 512 new
    tokens each after a cached prefix of U{0..7680} tokens."""
    return paged_chunk(num_seqs=8, tokens_lo=512, tokens_hi=512, prefix_lo=0, prefix_hi=7680,
                       num_pages=4608, page_size=16, n_heads=16, n_kv_heads=4, head_dim=256,
                       kv_dtype="f16", seed=seed, name="paged_chunk_8seq_512tok_pre0-7680_h16_hk4_d256")


# ---------------------------------------------------------------------------
# DFlash2 ring KV (speculative verify)
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class RingCase:
    name: str
    geom: tuple  # (lanes, q_heads, kv_heads, head_dim, rows, window, packed_len, max_commit)
    scale: float
    ring_k: np.ndarray        # bf16 bits [lanes, kv_heads, window, head_dim]
    ring_v: np.ndarray
    cur_q: np.ndarray         # f32 [lanes, rows, q_heads, head_dim]
    cur_k: np.ndarray         # f32 [lanes, rows, kv_heads, head_dim]
    cur_v: np.ndarray
    cache_lengths: np.ndarray     # u32 [lanes]
    write_positions: np.ndarray   # u32 [lanes]
    commit_counts: np.ndarray     # u32 [lanes]
    new_k: np.ndarray         # f32 [lanes, max_commit, kv_heads, head_dim]
    new_v: np.ndarray


def ring(*, lanes: int = 4, rows: int = 16, window: int = 4096, q_heads: int = 32,
         kv_heads: int = 8, head_dim: int = 256, max_commit: int | None = None,
         scale: float | None = None, seed: int = 0, name: str | None = None) -> RingCase:
    """Ring K/V ~ N(0,1) bf16; current Q/K/V ~ N(0,1) f32;
    cache_lengths ~ U{rows..window-1}; write_positions ~ U{0..window-1};
    commit_counts ~ U{1..rows}.  The rows offered for commit are the current
    K/V rows (max_commit == rows), as in the pages' worked example."""
    if max_commit is None:
        max_commit = rows
    rng = np.random.default_rng(seed)
    ring_k = _normal_bf16(rng, (lanes, kv_heads, window, head_dim))
    ring_v = _normal_bf16(rng, (lanes, kv_heads, window, head_dim))
    cur_q = _normal_f32(rng, (lanes, rows, q_heads, head_dim))
    cur_k = _normal_f32(rng, (lanes, rows, kv_heads, head_dim))
    cur_v = _normal_f32(rng, (lanes, rows, kv_heads, head_dim))
    cache_lengths = rng.integers(rows, window - 1, size=lanes, endpoint=True).astype(np.uint32)
    write_positions = rng.integers(0, window - 1, size=lanes, endpoint=True).astype(np.uint32)
    commit_counts = rng.integers(1, rows, size=lanes, endpoint=True).astype(np.uint32)
    new_k = np.ascontiguousarray(cur_k[:, :max_commit])
    new_v = np.ascontiguousarray(cur_v[:, :max_commit])
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    geom = (lanes, q_heads, kv_heads, head_dim, rows, window, window - 1 + rows, max_commit)
    if name is None:
        name = (f"verify_ring_lanes{lanes}_rows{rows}_w{window}_h{q_heads}_hk{kv_heads}"
                f"_d{head_dim}")
    return RingCase(name, geom, float(scale), ring_k, ring_v, cur_q, cur_k, cur_v,
                    cache_lengths, write_positions, commit_counts, new_k, new_v)


def verify_full(seed: int = 0) -> RingCase:
    """lanes 4, rows 16, window 4096, 32 / 8 heads, head_dim 256, scale 1/16."""
    return ring(seed=seed)
