"""Python binding of the GB300 GQA attention library (``include/gqa_attn.h``).

Argument marshalling only: every function takes torch CUDA tensors, passes
their device pointers, byte sizes and strides, plus the current CUDA stream,
to the C entry point of the same name, and raises ``GQAError`` with the
library's message when the call is rejected.  All work runs in the library's
CUDA kernels; there is no fallback: if the shared library is missing, import
succeeds but every call raises.

u32 device counters (cache lengths, write positions, commit counts) are
passed as torch.int32 tensors holding the same bits.
"""
from __future__ import annotations

import ctypes
import pathlib

import torch

_PKG = pathlib.Path(__file__).resolve().parent
LIB_PATH = _PKG / "lib" / "libgqa_attn.so"

GQA_DTYPE_F16 = 1
GQA_DTYPE_BF16 = 2
GQA_FLAG_PAGE_CLAMPED = 1
GQA_FLAG_CONTEXT_CLAMPED = 2
GQA_FLAG_RING_CLAMPED = 4
GQA_FLAG_TIMEOUT = 8

_KV_DTYPES = {torch.float16: GQA_DTYPE_F16, torch.bfloat16: GQA_DTYPE_BF16}


class GQAError(RuntimeError):
    """A library call returned a non-zero gqa_status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"gqa status {status}: {message}")
        self.status = status


class GqaRingParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in
                ("lanes", "q_heads", "kv_heads", "head_dim", "rows", "window", "packed_len",
                 "max_commit")]


_lib = None


def library() -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: run attention_gqa_flash_gb300.build.build()")
        lib = ctypes.CDLL(str(LIB_PATH))
        vp, sz, i32, i64, f32 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64,
                                 ctypes.c_float)
        rp = ctypes.POINTER(GqaRingParams)
        sig = {
            "gqa_last_error": (ctypes.c_char_p, []),
            "gqa_version": (ctypes.c_char_p, []),
            "gqa_device_sm_count": (i32, []),
            "gqa_timing_enable": (i32, [i32]),
            "gqa_timing_last_ms": (f32, []),
            "gqa_attn_set_cta_pairs": (i32, [i32]),
            "gqa_selftest_bounded_wait": (i32, [vp, i32, vp]),
            "gqa_kv_pad": (ctypes.c_uint32, [ctypes.c_uint32]),
            "gqa_attn_prefill_workspace_size": (sz, [i32] * 5),
            "gqa_attn_prefill": (i32, [vp, sz, i32, i32, vp, sz, i32, i32, vp, sz, i32, i32, i32,
                                       vp, sz, vp, sz, i32, i32, i32, i32, i32, f32, vp, sz, vp,
                                       vp]),
            "gqa_attn_paged_decode_workspace_size": (sz, [i32] * 5),
            "gqa_attn_paged_decode": (i32, [vp, sz, vp, vp, sz, i32, i64, i64, i64, vp, sz, i32,
                                            vp, sz, vp, sz, i32, i32, i32, i32, i32, i32, f32, vp,
                                            sz, vp, vp]),
            "gqa_attn_paged_decode_noalloc": (i32, [vp, sz, vp, vp, sz, i32, i64, i64, i64, vp, sz,
                                                    i32, vp, sz, vp, sz, i32, i32, i32, i32, i32,
                                                    i32, f32, vp, vp]),
            "gqa_paged_append": (i32, [vp, vp, sz, vp, sz, vp, sz, vp, sz, i32, vp, vp, sz, i32,
                                       i64, i64, i64, i32, i32, i32, i32, i32, i32, vp, vp]),
            "gqa_attn_paged_prefill_workspace_size": (sz, [i32] * 7),
            "gqa_attn_paged_prefill": (i32, [vp, sz, vp, vp, sz, i32, i64, i64, i64, vp, sz, i32,
                                             vp, sz, vp, sz, vp, sz, i32, i32, i32, i32, i32, i32,
                                             i32, i32, f32, vp, sz, vp, vp]),
            "gqa_ring_params_valid": (i32, [rp]),
            "gqa_pack_attention": (i32, [vp, sz] * 10 + [rp, vp, vp]),
            "gqa_fill_mask": (i32, [vp, sz, vp, sz, rp, vp, vp]),
            "gqa_attn_verify_workspace_size": (sz, [rp]),
            "gqa_attn_verify": (i32, [vp, sz] * 5 + [rp, f32, vp, sz, vp, vp]),
            "gqa_attn_verify_ring_workspace_size": (sz, [rp]),
            "gqa_attn_verify_ring": (i32, [vp, sz] * 8 + [rp, f32, vp, sz, vp, vp]),
            "gqa_commit_kv": (i32, [vp, sz] * 6 + [rp, vp, vp]),
            "gqa_set_mask_rows": (i32, [vp, sz, vp, sz, ctypes.c_uint32, ctypes.c_uint32,
                                        ctypes.c_uint32, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols() -> list[str]:
    """Names of the C entry points this binding wraps."""
    return ["gqa_last_error", "gqa_version", "gqa_device_sm_count", "gqa_timing_enable",
            "gqa_timing_last_ms", "gqa_attn_set_cta_pairs", "gqa_selftest_bounded_wait",
            "gqa_kv_pad",
            "gqa_attn_prefill_workspace_size", "gqa_attn_prefill",
            "gqa_attn_paged_decode_workspace_size", "gqa_attn_paged_decode",
            "gqa_attn_paged_decode_noalloc",
            "gqa_paged_append", "gqa_attn_paged_prefill_workspace_size", "gqa_attn_paged_prefill",
            "gqa_ring_params_valid", "gqa_pack_attention", "gqa_fill_mask",
            "gqa_attn_verify_workspace_size", "gqa_attn_verify",
            "gqa_attn_verify_ring_workspace_size", "gqa_attn_verify_ring", "gqa_commit_kv",
            "gqa_set_mask_rows"]


def _check(rc: int) -> None:
    if rc != 0:
        raise GQAError(rc, library().gqa_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _nbytes(t: torch.Tensor | None) -> int:
    """Bytes from the tensor's first element to the end of its storage."""
    if t is None:
        return 0
    st = t.untyped_storage()
    return st.nbytes() - t.storage_offset() * t.element_size()


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(name: str, t: torch.Tensor, dtypes) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")


def _contig(name: str, t: torch.Tensor) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ring(p) -> GqaRingParams:
    if isinstance(p, GqaRingParams):
        return p
    return GqaRingParams(*[int(x) for x in p])


def gqa_timing_enable(enable: bool) -> None:
    """Record CUDA events around each call's dominant kernel (measurement only)."""
    _check(library().gqa_timing_enable(1 if enable else 0))


def gqa_attn_set_cta_pairs(mode: int) -> None:
    """Prefill tiling: 0 never pair query tiles into two-CTA clusters, 1 pair
    where measured faster (head_dim 256 and 512, the default), 2 pair every eligible shape."""
    _check(library().gqa_attn_set_cta_pairs(int(mode)))


def gqa_timing_last_ms() -> float:
    """Elapsed ms of the dominant kernel of the most recent call (-1 if none)."""
    return float(library().gqa_timing_last_ms())


def gqa_selftest_bounded_wait(status: torch.Tensor, timeout_ms: int, stream=None) -> None:
    """Run the bounded-wait self-test; GQA_FLAG_TIMEOUT lands in `status`."""
    _cuda("status", status, (torch.int32,))
    _check(library().gqa_selftest_bounded_wait(_ptr(status), int(timeout_ms), _stream(stream)))


def version() -> str:
    return library().gqa_version().decode()


def gqa_kv_pad(kv_len: int) -> int:
    return int(library().gqa_kv_pad(kv_len))


def gqa_ring_params_valid(p) -> bool:
    return bool(library().gqa_ring_params_valid(ctypes.byref(_ring(p))))


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
def gqa_attn_prefill_workspace_size(rows, n_heads, n_kv_heads, head_dim, kv_pad) -> int:
    return int(library().gqa_attn_prefill_workspace_size(rows, n_heads, n_kv_heads, head_dim,
                                                         kv_pad))


def gqa_attn_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor,
                     scale: float, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """q f32 [rows, n_heads, head_dim]; k, v f16/bf16 [kv_pad, n_kv_heads, head_dim]
    (row/head strides taken from the tensors, innermost dim contiguous);
    mask f16 [rows, kv_pad] contiguous; returns o f32 [rows, n_heads, head_dim]."""
    _cuda("q", q, (torch.float32,))
    _cuda("k", k, tuple(_KV_DTYPES))
    _cuda("v", v, (k.dtype,))
    _cuda("mask", mask, (torch.float16,))
    _contig("mask", mask)
    rows, n_heads, d = q.shape
    kv_pad, n_kv, d2 = k.shape
    if v.shape != k.shape or d2 != d or mask.shape != (rows, kv_pad):
        raise ValueError("prefill shapes disagree")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.stride(2) != 1:
            raise ValueError(f"{name} innermost dimension must be contiguous")
    if out is None:
        out = torch.empty((rows, n_heads, d), dtype=torch.float32, device=q.device)
    _cuda("out", out, (torch.float32,))
    _contig("out", out)
    if workspace is None:
        n = gqa_attn_prefill_workspace_size(rows, n_heads, n_kv, d, kv_pad)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _check(library().gqa_attn_prefill(
        _ptr(q), _nbytes(q), q.stride(0), q.stride(1),
        _ptr(k), _nbytes(k), k.stride(0), k.stride(1),
        _ptr(v), _nbytes(v), v.stride(0), v.stride(1), _KV_DTYPES[k.dtype],
        _ptr(mask), _nbytes(mask), _ptr(out), _nbytes(out),
        rows, n_heads, n_kv, d, kv_pad, float(scale),
        _ptr(workspace), _nbytes(workspace), _ptr(status), _stream(stream)))
    return out


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------
def gqa_attn_paged_decode_workspace_size(num_seqs, n_heads, head_dim, max_pages_per_seq,
                                         page_size) -> int:
    return int(library().gqa_attn_paged_decode_workspace_size(num_seqs, n_heads, head_dim,
                                                               max_pages_per_seq, page_size))


def gqa_attn_paged_decode(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                          page_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                          out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                          status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q f32 [num_seqs, n_heads, head_dim]; k_pages / v_pages f16/bf16
    [num_pages, page_size, n_kv_heads, head_dim] (same strides, innermost contiguous);
    page_table int32 [num_seqs, max_pages_per_seq]; context_lens int32 [num_seqs]."""
    _cuda("q", q, (torch.float32,))
    _contig("q", q)
    _cuda("k_pages", k_pages, tuple(_KV_DTYPES))
    _cuda("v_pages", v_pages, (k_pages.dtype,))
    _cuda("page_table", page_table, (torch.int32,))
    _cuda("context_lens", context_lens, (torch.int32,))
    _contig("page_table", page_table)
    _contig("context_lens", context_lens)
    num_seqs, n_heads, d = q.shape
    num_pages, page_size, n_kv, d2 = k_pages.shape
    if v_pages.shape != k_pages.shape or v_pages.stride() != k_pages.stride() or d2 != d:
        raise ValueError("K and V pools must share shape and strides")
    if k_pages.stride(3) != 1:
        raise ValueError("pool head_dim must be contiguous")
    max_pages = page_table.shape[1]
    if out is None:
        out = torch.empty((num_seqs, n_heads, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = gqa_attn_paged_decode_workspace_size(num_seqs, n_heads, d, max_pages, page_size)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _check(library().gqa_attn_paged_decode(
        _ptr(q), _nbytes(q), _ptr(k_pages), _ptr(v_pages),
        min(_nbytes(k_pages), _nbytes(v_pages)), _KV_DTYPES[k_pages.dtype],
        k_pages.stride(0), k_pages.stride(1), k_pages.stride(2),
        _ptr(page_table), _nbytes(page_table), max_pages,
        _ptr(context_lens), _nbytes(context_lens), _ptr(out), _nbytes(out),
        num_seqs, n_heads, n_kv, d, page_size, num_pages, float(scale),
        _ptr(workspace), _nbytes(workspace), _ptr(status), _stream(stream)))
    return out


def _pool(k_pages: torch.Tensor, v_pages: torch.Tensor, head_dim: int):
    _cuda("k_pages", k_pages, tuple(_KV_DTYPES))
    _cuda("v_pages", v_pages, (k_pages.dtype,))
    num_pages, page_size, n_kv, d2 = k_pages.shape
    if v_pages.shape != k_pages.shape or v_pages.stride() != k_pages.stride() or d2 != head_dim:
        raise ValueError("K and V pools must share shape and strides")
    if k_pages.stride(3) != 1:
        raise ValueError("pool head_dim must be contiguous")
    return num_pages, page_size, n_kv


def _seq_arrays(token_offsets, position_start, page_table):
    for name, t in (("token_offsets", token_offsets), ("position_start", position_start),
                    ("page_table", page_table)):
        _cuda(name, t, (torch.int32,))
        _contig(name, t)
    num_seqs = position_start.shape[0]
    if token_offsets.shape != (num_seqs + 1,) or page_table.shape[0] != num_seqs:
        raise ValueError("token_offsets [num_seqs + 1], position_start [num_seqs], "
                         "page_table [num_seqs, max_pages]")
    return num_seqs


def gqa_paged_append(k_new: torch.Tensor, v_new: torch.Tensor, token_offsets: torch.Tensor,
                     position_start: torch.Tensor, page_table: torch.Tensor,
                     k_pages: torch.Tensor, v_pages: torch.Tensor,
                     status: torch.Tensor | None = None, stream=None) -> None:
    """k_new / v_new f32 [total_tokens, n_kv_heads, head_dim] rounded into their page
    slots of k_pages / v_pages (f16/bf16 [num_pages, page_size, n_kv_heads, head_dim]);
    token_offsets int32 [num_seqs + 1], position_start int32 [num_seqs], page_table
    int32 [num_seqs, max_pages_per_seq]."""
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _cuda(name, t, (torch.float32,))
        _contig(name, t)
    if v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must have the same shape")
    total, n_kv, d = k_new.shape
    num_pages, page_size, n_kv2 = _pool(k_pages, v_pages, d)
    if n_kv2 != n_kv:
        raise ValueError("k_new and the pools disagree on n_kv_heads")
    num_seqs = _seq_arrays(token_offsets, position_start, page_table)
    _check(library().gqa_paged_append(
        _ptr(k_new), _ptr(v_new), min(_nbytes(k_new), _nbytes(v_new)),
        _ptr(token_offsets), _nbytes(token_offsets), _ptr(position_start), _nbytes(position_start),
        _ptr(page_table), _nbytes(page_table), page_table.shape[1],
        _ptr(k_pages), _ptr(v_pages), min(_nbytes(k_pages), _nbytes(v_pages)),
        _KV_DTYPES[k_pages.dtype], k_pages.stride(0), k_pages.stride(1), k_pages.stride(2),
        num_seqs, total, n_kv, d, page_size, num_pages, _ptr(status), _stream(stream)))


def gqa_attn_paged_prefill_workspace_size(num_seqs: int, max_tokens: int, n_heads: int,
                                          n_kv_heads: int, head_dim: int, max_pages_per_seq: int,
                                          page_size: int) -> int:
    return int(library().gqa_attn_paged_prefill_workspace_size(
        num_seqs, max_tokens, n_heads, n_kv_heads, head_dim, max_pages_per_seq, page_size))


def gqa_attn_paged_prefill(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                           page_table: torch.Tensor, token_offsets: torch.Tensor,
                           position_start: torch.Tensor, max_tokens: int, scale: float,
                           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Chunked prefill over pages: q f32 [total_tokens, n_heads, head_dim]; the pools,
    page_table, token_offsets and position_start as for gqa_paged_append; max_tokens
    bounds every sequence's token count.  Returns o f32 like q."""
    _cuda("q", q, (torch.float32,))
    _contig("q", q)
    total, n_heads, d = q.shape
    num_pages, page_size, n_kv = _pool(k_pages, v_pages, d)
    num_seqs = _seq_arrays(token_offsets, position_start, page_table)
    max_pages = page_table.shape[1]
    if out is None:
        out = torch.empty((total, n_heads, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = gqa_attn_paged_prefill_workspace_size(num_seqs, max_tokens, n_heads, n_kv, d,
                                                  max_pages, page_size)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _check(library().gqa_attn_paged_prefill(
        _ptr(q), _nbytes(q), _ptr(k_pages), _ptr(v_pages),
        min(_nbytes(k_pages), _nbytes(v_pages)), _KV_DTYPES[k_pages.dtype],
        k_pages.stride(0), k_pages.stride(1), k_pages.stride(2),
        _ptr(page_table), _nbytes(page_table), max_pages,
        _ptr(token_offsets), _nbytes(token_offsets), _ptr(position_start), _nbytes(position_start),
        _ptr(out), _nbytes(out), num_seqs, total, max_tokens, n_heads, n_kv, d, page_size,
        num_pages, float(scale), _ptr(workspace), _nbytes(workspace), _ptr(status),
        _stream(stream)))
    return out


GQA_NOALLOC_SCRATCH_BYTES = 16 << 20


def gqa_attn_paged_decode_noalloc(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                                  page_table: torch.Tensor, context_lens: torch.Tensor,
                                  scale: float, out: torch.Tensor, status: torch.Tensor | None = None,
                                  stream=None) -> torch.Tensor:
    """Paged decode for callers that cannot provide device scratch: same
    arguments as gqa_attn_paged_decode, no workspace, and the output buffer
    must be passed in.  The library keeps its partial results in a fixed
    16 MiB device array; larger problems are rejected (GQAError)."""
    _cuda("q", q, (torch.float32,))
    _contig("q", q)
    _cuda("k_pages", k_pages, tuple(_KV_DTYPES))
    _cuda("v_pages", v_pages, (k_pages.dtype,))
    _cuda("page_table", page_table, (torch.int32,))
    _cuda("context_lens", context_lens, (torch.int32,))
    _cuda("out", out, (torch.float32,))
    for name, t in (("page_table", page_table), ("context_lens", context_lens), ("out", out)):
        _contig(name, t)
    num_seqs, n_heads, d = q.shape
    num_pages, page_size, n_kv, d2 = k_pages.shape
    if v_pages.shape != k_pages.shape or v_pages.stride() != k_pages.stride() or d2 != d:
        raise ValueError("K and V pools must share shape and strides")
    _check(library().gqa_attn_paged_decode_noalloc(
        _ptr(q), _nbytes(q), _ptr(k_pages), _ptr(v_pages),
        min(_nbytes(k_pages), _nbytes(v_pages)), _KV_DTYPES[k_pages.dtype],
        k_pages.stride(0), k_pages.stride(1), k_pages.stride(2),
        _ptr(page_table), _nbytes(page_table), page_table.shape[1],
        _ptr(context_lens), _nbytes(context_lens), _ptr(out), _nbytes(out),
        num_seqs, n_heads, n_kv, d, page_size, num_pages, float(scale),
        _ptr(status), _stream(stream)))
    return out


# ---------------------------------------------------------------------------
# DFlash2 ring KV
# ---------------------------------------------------------------------------
def _exact(name, t, dtype):
    _cuda(name, t, (dtype,))
    _contig(name, t)
    return _ptr(t), t.numel() * t.element_size()


def gqa_pack_attention(ring_k, ring_v, cur_q, cur_k, cur_v, cache_lengths, write_positions,
                       packed_q, packed_k, packed_v, params, status=None, stream=None) -> None:
    """Pack current f32 rows and bf16 ring history into bf16 verify operands
    (outputs written in place)."""
    args = []
    for name, t, dt in (("ring_k", ring_k, torch.bfloat16), ("ring_v", ring_v, torch.bfloat16),
                        ("cur_q", cur_q, torch.float32), ("cur_k", cur_k, torch.float32),
                        ("cur_v", cur_v, torch.float32), ("cache_lengths", cache_lengths, torch.int32),
                        ("write_positions", write_positions, torch.int32),
                        ("packed_q", packed_q, torch.bfloat16), ("packed_k", packed_k, torch.bfloat16),
                        ("packed_v", packed_v, torch.bfloat16)):
        args += list(_exact(name, t, dt))
    _check(library().gqa_pack_attention(*args, ctypes.byref(_ring(params)), _ptr(status),
                                        _stream(stream)))


def gqa_fill_mask(cache_lengths, mask, params, status=None, stream=None) -> None:
    a = _exact("cache_lengths", cache_lengths, torch.int32)
    m = _exact("mask", mask, torch.bfloat16)
    _check(library().gqa_fill_mask(*a, *m, ctypes.byref(_ring(params)), _ptr(status),
                                   _stream(stream)))


def gqa_attn_verify_workspace_size(params) -> int:
    return int(library().gqa_attn_verify_workspace_size(ctypes.byref(_ring(params))))


def gqa_attn_verify(packed_q, packed_k, packed_v, mask, params, scale: float, out=None,
                    workspace=None, status=None, stream=None) -> torch.Tensor:
    p = _ring(params)
    if out is None:
        out = torch.empty((p.lanes, p.rows, p.q_heads, p.head_dim), dtype=torch.float32,
                          device=packed_q.device)
    if workspace is None:
        n = gqa_attn_verify_workspace_size(p)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=packed_q.device)
    args = []
    for name, t, dt in (("packed_q", packed_q, torch.bfloat16), ("packed_k", packed_k, torch.bfloat16),
                        ("packed_v", packed_v, torch.bfloat16), ("mask", mask, torch.bfloat16),
                        ("out", out, torch.float32)):
        args += list(_exact(name, t, dt))
    _check(library().gqa_attn_verify(*args, ctypes.byref(p), float(scale), _ptr(workspace),
                                     _nbytes(workspace), _ptr(status), _stream(stream)))
    return out


def gqa_attn_verify_ring_workspace_size(params) -> int:
    return int(library().gqa_attn_verify_ring_workspace_size(ctypes.byref(_ring(params))))


def gqa_attn_verify_ring(ring_k, ring_v, cur_q, cur_k, cur_v, cache_lengths, write_positions,
                         params, scale: float, out=None, workspace=None, status=None,
                         stream=None) -> torch.Tensor:
    """Fused verify attention read straight from the ring (no packed copy, no mask
    tensor): O f32 [lanes, rows, q_heads, head_dim]."""
    p = _ring(params)
    if out is None:
        out = torch.empty((p.lanes, p.rows, p.q_heads, p.head_dim), dtype=torch.float32,
                          device=cur_q.device)
    if workspace is None:
        n = gqa_attn_verify_ring_workspace_size(p)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=cur_q.device)
    args = []
    for name, t, dt in (("ring_k", ring_k, torch.bfloat16), ("ring_v", ring_v, torch.bfloat16),
                        ("cur_q", cur_q, torch.float32), ("cur_k", cur_k, torch.float32),
                        ("cur_v", cur_v, torch.float32), ("cache_lengths", cache_lengths, torch.int32),
                        ("write_positions", write_positions, torch.int32), ("out", out, torch.float32)):
        args += list(_exact(name, t, dt))
    _check(library().gqa_attn_verify_ring(*args, ctypes.byref(p), float(scale), _ptr(workspace),
                                          _nbytes(workspace), _ptr(status), _stream(stream)))
    return out


def gqa_commit_kv(new_k, new_v, commit_counts, write_positions, ring_k, ring_v, params,
                  status=None, stream=None) -> None:
    args = []
    for name, t, dt in (("new_k", new_k, torch.float32), ("new_v", new_v, torch.float32),
                        ("commit_counts", commit_counts, torch.int32),
                        ("write_positions", write_positions, torch.int32),
                        ("ring_k", ring_k, torch.bfloat16), ("ring_v", ring_v, torch.bfloat16)):
        args += list(_exact(name, t, dt))
    _check(library().gqa_commit_kv(*args, ctypes.byref(_ring(params)), _ptr(status),
                                   _stream(stream)))


def gqa_set_mask_rows(mask_embedding, hidden, lanes: int, rows: int, stream=None) -> None:
    e = _exact("mask_embedding", mask_embedding, torch.bfloat16)
    h = _exact("hidden", hidden, torch.float32)
    _check(library().gqa_set_mask_rows(*e, *h, lanes, rows, mask_embedding.numel(),
                                       _stream(stream)))
