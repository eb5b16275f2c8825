"""TEST INFRASTRUCTURE ONLY: the float64 CPU oracle for the GQA attention library.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path never does, and nothing here is
shared with the CUDA sources.

The arithmetic lives in ``gqa_oracle.c`` (plain C, float64, OpenMP over
independent output rows).  This module only compiles it with gcc, loads it
with ctypes and marshals NumPy arrays.  Strides are taken from the arrays
themselves, so strided views are evaluated exactly as laid out.

Pinned by ``tests/test_oracle_attention.py``, ``test_oracle_conversions.py``,
``test_oracle_paged.py`` and ``test_oracle_ring.py`` against the pages' worked
examples, closed forms, invariants and library routines (see each file's header).
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess
import threading

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "gqa_oracle.c"
_BUILD = _HERE / "_build"
_SO = _BUILD / "libgqa_oracle.so"

F32, F16, BF16 = 0, 1, 2
_DTYPES = {"f32": F32, "f16": F16, "bf16": BF16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> pathlib.Path:
    """Compile gqa_oracle.c into a shared library next to it (gcc, OpenMP)."""
    _BUILD.mkdir(exist_ok=True)
    if force or not _SO.exists() or _SO.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _BUILD / f"libgqa_oracle.{os.getpid()}.so"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
             "-Wno-unknown-pragmas", str(_SRC), "-o", str(tmp), "-lm"],
            check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build()))
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.orc_attention.restype = i32
            lib.orc_attention.argtypes = [vp, i32, i64, i64, vp, i64, i64, vp, i64, i64, i32,
                                          vp, i32, i64, i64, i32, i32, i32, i32, i32, dbl,
                                          vp, i64, vp]
            lib.orc_paged_decode.restype = i32
            lib.orc_paged_decode.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, i64, vp, i32,
                                             i32, i32, i32, i32, i64, dbl, vp, i32, vp]
            for name in ("orc_pack_attention", "orc_fill_mask", "orc_commit_kv"):
                getattr(lib, name).restype = i32
            lib.orc_pack_attention.argtypes = [vp] * 11
            lib.orc_fill_mask.argtypes = [vp, vp, vp]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_paged_append.restype = i32
            lib.orc_paged_append.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, i32, i64, i64, i64,
                                             i32, i32, i32, i32, i64, vp]
            lib.orc_paged_prefill.restype = i32
            lib.orc_paged_prefill.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, i64, vp, vp,
                                              i32, i32, i32, i32, i32, i64, dbl, vp]
            lib.orc_verify_ring_attention.restype = i32
            lib.orc_verify_ring_attention.argtypes = [vp] * 8 + [dbl, vp]
            lib.orc_commit_kv.argtypes = [vp] * 7
            lib.orc_ring_geometry_valid.restype = i32
            lib.orc_ring_geometry_valid.argtypes = [vp]
            lib.orc_set_mask_rows.restype = i32
            lib.orc_set_mask_rows.argtypes = [vp, vp, ctypes.c_uint32, ctypes.c_uint32,
                                              ctypes.c_uint32]
            lib.orc_widen16.restype = dbl
            lib.orc_widen16.argtypes = [ctypes.c_uint16, i32]
            lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.orc_num_threads.restype = i32
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().orc_num_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _estrides(a: np.ndarray) -> tuple[int, ...]:
    for s in a.strides:
        if s % a.itemsize:
            raise ValueError("strides must be whole elements")
    return tuple(s // a.itemsize for s in a.strides)


def _bits16(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 or uint16 (bf16 bits), got {a.dtype}")


# --------------------------------------------------------------------------
# scalar conversions (exposed so the pins can check them against libraries)
# --------------------------------------------------------------------------
def widen16(bits: int, dtype: str) -> float:
    return float(_load().orc_widen16(int(bits), _DTYPES[dtype]))


def f32_to_bf16(x: float) -> int:
    return int(_load().orc_f32_to_bf16(float(np.float32(x))))


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    f = _load().orc_f32_to_bf16
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.fromiter((f(float(v)) for v in flat), dtype=np.uint16,
                       count=flat.size).reshape(np.shape(x))


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, kv_dtype: str,
              scale: float, mask: np.ndarray | None = None, mask_dtype: str | None = None,
              q_dtype: str = "f32", pairs: np.ndarray | None = None) -> np.ndarray:
    """Masked GQA attention in float64.

    q: [rows, n_heads, head_dim] float32 (q_dtype 'f32') or uint16 bits of
       f16/bf16 (q_dtype 'f16'/'bf16'); any strides.
    k, v: [n_keys, n_kv_heads, head_dim] float16 or uint16 bf16 bits.
    mask: None, [rows, n_keys] (shared by all heads) or [n_heads, rows, n_keys],
          float16 or uint16 bf16 bits (mask_dtype says which).
    pairs: optional int array [n, 2] of (row, head); the result is then
           [n, head_dim], else [rows, n_heads, head_dim].
    """
    rows, n_heads, d = q.shape
    n_keys, n_kv, d2 = k.shape
    if v.shape != k.shape or d2 != d:
        raise ValueError("shape mismatch")
    if q_dtype == "f32":
        if q.dtype != np.float32:
            raise TypeError("f32 queries must be float32")
        qa = q
    else:
        qa = _bits16(q)
    kb, vb = _bits16(k), _bits16(v)
    qs, ks, vs = _estrides(qa), _estrides(kb), _estrides(vb)
    if mask is not None:
        mb = _bits16(mask)
        if mask_dtype is None:
            mask_dtype = "f16" if mask.dtype == np.float16 else None
        if mask_dtype is None:
            raise ValueError("mask_dtype required for bf16 masks")
        if mb.ndim == 2:
            if mb.shape != (rows, n_keys):
                raise ValueError("mask shape")
            m_row, m_head = _estrides(mb)[0], 0
            if _estrides(mb)[1] != 1:
                raise ValueError("mask rows must be contiguous")
        else:
            if mb.shape != (n_heads, rows, n_keys):
                raise ValueError("mask shape")
            st = _estrides(mb)
            if st[2] != 1:
                raise ValueError("mask rows must be contiguous")
            m_head, m_row = st[0], st[1]
        mdt = _DTYPES[mask_dtype]
    else:
        mb, m_row, m_head, mdt = None, 0, 0, F16
    for name, st in (("q", qs), ("k", ks), ("v", vs)):
        if st[2] != 1:
            raise ValueError(f"{name} innermost dimension must be contiguous")
    if pairs is not None:
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((pairs.shape[0], d), dtype=np.float64)
        npairs = pairs.shape[0]
    else:
        out = np.zeros((rows, n_heads, d), dtype=np.float64)
        npairs = 0
    rc = _load().orc_attention(
        _ptr(qa), _DTYPES[q_dtype], qs[0], qs[1],
        _ptr(kb), ks[0], ks[1], _ptr(vb), vs[0], vs[1], _DTYPES[kv_dtype],
        _ptr(mb), mdt, m_row, m_head,
        rows, n_heads, n_kv, d, n_keys, float(scale),
        _ptr(pairs), npairs, _ptr(out))
    if rc != 0:
        raise ValueError("oracle attention rejected its arguments")
    return out


def paged_decode(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, *, kv_dtype: str,
                 page_table: np.ndarray, context_lens: np.ndarray, scale: float,
                 seqs: np.ndarray | None = None) -> np.ndarray:
    """Decode attention over a paged KV pool, float64.

    q: [num_seqs, n_heads, head_dim] float32 contiguous.
    k_pool, v_pool: [num_pages, page_size, n_kv_heads, head_dim] f16 / bf16 bits
                    (any page/token/head strides, identical for K and V).
    page_table: int32 [num_seqs, max_pages_per_seq]; context_lens: int32 [num_seqs].
    seqs: optional subset of sequence ids; result [len(seqs) or num_seqs, n_heads, head_dim].
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    num_seqs, n_heads, d = q.shape
    kb, vb = _bits16(k_pool), _bits16(v_pool)
    num_pages, page_size, n_kv, d2 = kb.shape
    if d2 != d or vb.shape != kb.shape:
        raise ValueError("pool shape")
    ks, vs = _estrides(kb), _estrides(vb)
    if ks != vs or ks[3] != 1:
        raise ValueError("K and V pools must share strides with a contiguous head_dim")
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    if seqs is not None:
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        count = seqs.size
    else:
        count = num_seqs
    out = np.zeros((count, n_heads, d), dtype=np.float64)
    rc = _load().orc_paged_decode(
        _ptr(q), _ptr(kb), _ptr(vb), _DTYPES[kv_dtype], ks[0], ks[1], ks[2],
        _ptr(pt), pt.shape[1], _ptr(cl), num_seqs, n_heads, n_kv, d, page_size, num_pages,
        float(scale), _ptr(seqs), count if seqs is not None else 0, _ptr(out))
    if rc != 0:
        raise ValueError("oracle paged decode rejected its arguments")
    return out


# --------------------------------------------------------------------------
# DFlash2 ring KV
# --------------------------------------------------------------------------
def _geom(g) -> np.ndarray:
    a = np.asarray(g, dtype=np.uint32)
    if a.shape != (8,):
        raise ValueError("geometry is 8 words")
    return np.ascontiguousarray(a)


def ring_geometry_valid(g) -> bool:
    return bool(_load().orc_ring_geometry_valid(_ptr(_geom(g))))


def _c(a, dt):
    a = np.asarray(a)
    if a.dtype != dt:
        raise TypeError(f"expected {dt}, got {a.dtype}")
    return np.ascontiguousarray(a)


def pack_attention(ring_k, ring_v, cur_q, cur_k, cur_v, cache_lengths, write_positions, g):
    """Returns (packed_q, packed_k, packed_v) as uint16 bf16 bits."""
    g = _geom(g)
    B, H, HK, D, R, W, K, _ = (int(x) for x in g)
    pq = np.zeros((B, H, R, D), np.uint16)
    pk = np.zeros((B, HK, K, D), np.uint16)
    pv = np.zeros((B, HK, K, D), np.uint16)
    args = [_c(ring_k, np.uint16), _c(ring_v, np.uint16), _c(cur_q, np.float32),
            _c(cur_k, np.float32), _c(cur_v, np.float32), _c(cache_lengths, np.uint32),
            _c(write_positions, np.uint32)]
    if args[0].shape != (B, HK, W, D) or args[2].shape != (B, R, H, D) or \
            args[3].shape != (B, R, HK, D):
        raise ValueError("ring shapes")
    rc = _load().orc_pack_attention(*[_ptr(a) for a in args], _ptr(pq), _ptr(pk), _ptr(pv),
                                    _ptr(g))
    if rc != 0:
        raise ValueError("invalid ring geometry")
    return pq, pk, pv


def verify_ring_attention(ring_k, ring_v, cur_q, cur_k, cur_v, cache_lengths, write_positions,
                          g, scale: float) -> np.ndarray:
    """Verify attention read straight from the ring (keys: the current rows, then every
    visible ring slot in slot order): float64 [lanes, rows, q_heads, d]."""
    g = _geom(g)
    B, H, HK, D, R, W, K, _ = (int(x) for x in g)
    args = [_c(ring_k, np.uint16), _c(ring_v, np.uint16), _c(cur_q, np.float32),
            _c(cur_k, np.float32), _c(cur_v, np.float32), _c(cache_lengths, np.uint32),
            _c(write_positions, np.uint32)]
    if args[0].shape != (B, HK, W, D) or args[2].shape != (B, R, H, D) or \
            args[3].shape != (B, R, HK, D):
        raise ValueError("ring shapes")
    out = np.zeros((B, R, H, D), np.float64)
    rc = _load().orc_verify_ring_attention(*[_ptr(a) for a in args], _ptr(g), float(scale),
                                           _ptr(out))
    if rc != 0:
        raise ValueError("invalid ring geometry" if rc == 1 else "out of memory")
    return out


def f32_to_f16(x) -> int:
    """IEEE binary16 bits of float32 x, round to nearest even (the oracle's own rounding)."""
    return int(_load().orc_f32_to_f16(float(np.float32(x))))


def paged_append(k_new, v_new, token_offsets, position_start, page_table, k_pool, v_pool, *,
                 kv_dtype: str, page_stride: int, token_stride: int, head_stride: int,
                 page_size: int):
    """Returns (k_pool', v_pool', skipped): copies of the pools (float16, or uint16 bf16
    bits; the result has the input's dtype) with every new token's K / V row rounded
    into its page slot."""
    kn, vn = _c(k_new, np.float32), _c(v_new, np.float32)
    offs, ps, pt = _c(token_offsets, np.int32), _c(position_start, np.int32), _c(page_table, np.int32)
    in_dtype = np.asarray(k_pool).dtype
    kp = np.array(np.ascontiguousarray(_bits16(np.asarray(k_pool))), copy=True)
    vp_ = np.array(np.ascontiguousarray(_bits16(np.asarray(v_pool))), copy=True)
    S = offs.size - 1
    T, HK, D = kn.shape
    num_pages = kp.size // page_stride
    skipped = np.zeros(1, np.int64)
    rc = _load().orc_paged_append(_ptr(kn), _ptr(vn), _ptr(offs), _ptr(ps), _ptr(pt),
                                  pt.shape[1], _ptr(kp), _ptr(vp_), _DTYPES[kv_dtype],
                                  page_stride, token_stride, head_stride, S, HK, D, page_size,
                                  num_pages, _ptr(skipped))
    if rc != 0:
        raise ValueError("invalid paged append arguments")
    return kp.view(in_dtype), vp_.view(in_dtype), int(skipped[0])


def paged_prefill(q, k_pool, v_pool, page_table, token_offsets, position_start, *,
                  kv_dtype: str, page_stride: int, token_stride: int, head_stride: int,
                  n_kv_heads: int, page_size: int, scale: float) -> np.ndarray:
    """Chunked prefill over pages: float64 [tokens, n_heads, head_dim]."""
    qq = _c(q, np.float32)
    T, H, D = qq.shape
    kp = np.ascontiguousarray(_bits16(np.asarray(k_pool)))
    vp_ = np.ascontiguousarray(_bits16(np.asarray(v_pool)))
    pt, offs, ps = _c(page_table, np.int32), _c(token_offsets, np.int32), _c(position_start, np.int32)
    out = np.zeros((T, H, D), np.float64)
    rc = _load().orc_paged_prefill(_ptr(qq), _ptr(kp), _ptr(vp_), _DTYPES[kv_dtype], page_stride,
                                   token_stride, head_stride, _ptr(pt), pt.shape[1], _ptr(offs),
                                   _ptr(ps), offs.size - 1, H, n_kv_heads, D, page_size,
                                   kp.size // page_stride, float(scale), _ptr(out))
    if rc != 0:
        raise ValueError("invalid paged prefill arguments")
    return out


def fill_mask(cache_lengths, g) -> np.ndarray:
    """bf16 bits [lanes, q_heads, rows, packed_len]."""
    g = _geom(g)
    B, H, _, _, R, _, K, _ = (int(x) for x in g)
    m = np.zeros((B, H, R, K), np.uint16)
    rc = _load().orc_fill_mask(_ptr(_c(cache_lengths, np.uint32)), _ptr(m), _ptr(g))
    if rc != 0:
        raise ValueError("invalid ring geometry")
    return m


def commit_kv(new_k, new_v, commit_counts, write_positions, ring_k, ring_v, g):
    """Returns updated copies (ring_k, ring_v); the inputs are not modified."""
    g = _geom(g)
    rk = np.array(_c(ring_k, np.uint16), copy=True)
    rv = np.array(_c(ring_v, np.uint16), copy=True)
    args = [_c(new_k, np.float32), _c(new_v, np.float32), _c(commit_counts, np.uint32),
            _c(write_positions, np.uint32)]
    rc = _load().orc_commit_kv(*[_ptr(a) for a in args], _ptr(rk), _ptr(rv), _ptr(g))
    if rc != 0:
        raise ValueError("invalid ring geometry")
    return rk, rv


def verify_attention(packed_q, packed_k, packed_v, mask, g, scale: float,
                     pairs_per_lane=None) -> np.ndarray:
    """Attention over the packed tensors of every lane: O f32-layout [lanes, rows, q_heads, d]
    as float64.  Each lane is an independent masked GQA attention with its own
    per-head bf16 mask.  pairs_per_lane: optional list (one per lane) of (row, head)
    arrays; the result is then a list of [n, d] arrays."""
    g = _geom(g)
    B, H, HK, D, R, W, K, _ = (int(x) for x in g)
    outs = []
    for b in range(B):
        q = np.asarray(packed_q[b]).transpose(1, 0, 2)          # [R, H, D] view
        k = np.asarray(packed_k[b]).transpose(1, 0, 2)          # [K, HK, D] view
        v = np.asarray(packed_v[b]).transpose(1, 0, 2)
        pairs = None if pairs_per_lane is None else pairs_per_lane[b]
        outs.append(attention(q, k, v, kv_dtype="bf16", q_dtype="bf16", scale=scale,
                              mask=np.asarray(mask[b]), mask_dtype="bf16", pairs=pairs))
    if pairs_per_lane is not None:
        return outs
    return np.stack(outs)


def set_mask_rows(embedding, hidden, lanes: int, rows: int) -> np.ndarray:
    """Returns an updated copy of hidden [lanes*rows, width] f32."""
    emb = _c(embedding, np.uint16)
    hid = np.array(_c(hidden, np.float32), copy=True)
    rc = _load().orc_set_mask_rows(_ptr(emb), _ptr(hid), lanes, rows, emb.size)
    if rc != 0:
        raise ValueError("invalid mask-row geometry")
    return hid
