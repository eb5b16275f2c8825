"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every entry point declared in include/gqa_attn.h, the host helpers
reproduce the pages' constants, and invalid geometry is rejected before any
launch."""
import ctypes
import json
import pathlib
import re

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "gqa_attn.h"
GOLDEN = pathlib.Path(__file__).parent / "golden"


@pytest.fixture(scope="module")
def g():
    from attention_gqa_flash_gb300 import build
    build.build()
    import attention_gqa_flash_gb300 as pkg
    pkg.library()
    return pkg


def _declared() -> set[str]:
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text))


def test_every_declared_symbol_is_exported(g):
    lib = ctypes.CDLL(str(g.LIB_PATH))
    declared = _declared()
    assert len(declared) >= 15
    for name in sorted(declared):
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert declared == set(g.exported_symbols())


def test_version_and_kv_pad(g):
    assert "sm_103a" in g.version()
    ex = json.loads((GOLDEN / "prefill_kv_pad.json").read_text())
    for kv_len, pad in ex["cases"]:
        assert g.gqa_kv_pad(kv_len) == pad


def test_ring_geometry_validation(g):
    cases = json.loads((GOLDEN / "dflash2_geometry_cases.json").read_text())["cases"]
    for c in cases:
        assert g.gqa_ring_params_valid(c["geometry"]) == c["valid"]
    assert not g.gqa_ring_params_valid([4, 32, 8, 64, 8, 2048, 2055, 8])
    assert "invalid DFlash2 attention geometry" in g.library().gqa_last_error().decode()
    assert g.gqa_ring_params_valid([4, 32, 8, 256, 16, 4096, 4111, 16])


def test_prefill_rejects_bad_shapes_before_launch(g):
    lib = g.library()
    args = [None, 0, 0, 0, None, 0, 0, 0, None, 0, 0, 0, 1, None, 0, None, 0]
    rc = lib.gqa_attn_prefill(*args, 64, 5, 2, 128, 64, 1.0, None, 0, None, None)
    assert rc == 1 and "multiple of n_kv_heads" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_prefill(*args, 64, 4, 2, 128, 65, 1.0, None, 0, None, None)
    assert rc == 1 and "kv_pad" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_prefill(*args, 64, 4, 2, 96, 64, 1.0, None, 0, None, None)
    assert rc == 1 and "head_dim" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_prefill(*args, 0, 4, 2, 128, 64, 1.0, None, 0, None, None)
    assert rc == 1 and "empty shape" in lib.gqa_last_error().decode()


def test_decode_rejects_bad_shapes_before_launch(g):
    lib = g.library()
    base = [None, 0, None, None, 0, 1, 0, 0, 0, None, 0, 4, None, 0, None, 0]
    rc = lib.gqa_attn_paged_decode(*base, 2, 6, 4, 128, 16, 8, 1.0, None, 0, None, None)
    assert rc == 1 and "multiple of n_kv_heads" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_paged_decode(*base, 2, 8, 4, 96, 16, 8, 1.0, None, 0, None, None)
    assert rc == 1 and "head_dim" in lib.gqa_last_error().decode()


def test_ring_ops_reject_wrong_sizes_before_launch(g):
    lib = g.library()
    p = g.GqaRingParams(1, 1, 1, 128, 2, 4, 5, 2)
    fake = ctypes.c_void_p(256)   # never dereferenced: sizes are checked first
    rc = lib.gqa_fill_mask(fake, 4, fake, 2 * 5 * 2 - 2, ctypes.byref(p), None, None)
    assert rc == 1 and "mask must be 20 bytes" in lib.gqa_last_error().decode()
    bad = g.GqaRingParams(1, 1, 1, 128, 2, 4, 4, 2)
    rc = lib.gqa_fill_mask(fake, 4, fake, 16, ctypes.byref(bad), None, None)
    assert rc == 1


def test_page_math_matches_the_fixed_page_capability():
    """ferrum-kernels causal_attention.rs page math, restated for the library's
    page layout: 4096 B/token (kv_heads 4, head_dim 256, f16, K and V),
    64 KiB pages of 16 tokens, 17 tokens -> 2 pages, 262144 tokens -> 16384 pages."""
    ex = json.loads((GOLDEN / "paged_page_math.json").read_text())
    per_token = ex["kv_heads"] * ex["head_dim"] * ex["element_bytes"] * 2
    assert per_token == ex["state_bytes_per_token"]
    page_bytes = ex["derived_page_bytes"]
    assert page_bytes // per_token == ex["derived_tokens_per_page"]
    pages = lambda tokens: -(-tokens * per_token // page_bytes)
    assert pages(17) == ex["tokens_17_physical_pages"]
    assert pages(ex["maximum_context_tokens"]) == ex["maximum_pages"]


def test_cta_pair_mode_is_validated_and_keeps_workspace_size(g):
    lib = g.library()
    assert lib.gqa_attn_set_cta_pairs(3) == 1
    assert "mode 3" in lib.gqa_last_error().decode()
    sizes = []
    for mode in (0, 1, 2):
        assert lib.gqa_attn_set_cta_pairs(mode) == 0
        # a shape that pairs in mode 2 and splits its keys: the workspace must not depend on the mode
        sizes.append(g.gqa_attn_prefill_workspace_size(128, 2, 1, 256, 4032))
    lib.gqa_attn_set_cta_pairs(1)
    assert len(set(sizes)) == 1 and sizes[0] > 0


def test_paged_append_rejects_bad_arguments_before_launch(g):
    lib = g.library()
    fake = ctypes.c_void_p(256)
    tail = [2, 8, 2, 64, 16, 8, None, None]   # num_seqs, tokens, hk, d, page, pages, status, stream

    # a well-formed call shape, with one field broken at a time
    # k_new, v_new, new_bytes, offsets (+bytes), position starts (+bytes), page table
    # (+bytes), max pages, pools, pool bytes, dtype, page / token / head strides
    base = [fake, fake, 8 * 2 * 64 * 4, fake, 3 * 4, fake, 2 * 4, fake, 2 * 4 * 4, 4,
            fake, fake, 1 << 20, 1, 2048, 128, 64]
    rc = lib.gqa_paged_append(*base[:14], 2048, 128, 60, *tail)  # head stride not a multiple of 8
    assert rc == 1 and "multiples of 8" in lib.gqa_last_error().decode()
    rc = lib.gqa_paged_append(*base, 2, 8, 2, 60, 16, 8, None, None)  # head_dim not a multiple of 8
    assert rc == 1 and "head_dim" in lib.gqa_last_error().decode()
    rc = lib.gqa_paged_append(*base[:12], 100, *base[13:], *tail)  # pool too small for the geometry
    assert rc == 1 and "k_pages" in lib.gqa_last_error().decode()
    rc = lib.gqa_paged_append(*base[:4], 2 * 4, *base[5:], *tail)  # token_offsets needs num_seqs + 1
    assert rc == 1 and "token_offsets" in lib.gqa_last_error().decode()
    rc = lib.gqa_paged_append(*base[:13], 7, *base[14:], *tail)  # unknown dtype
    assert rc == 1 and "kv_dtype" in lib.gqa_last_error().decode()
    rc = lib.gqa_paged_append(*base[:2], 100, *base[3:], *tail)  # new rows too small
    assert rc == 1 and "k_new" in lib.gqa_last_error().decode()


def test_paged_prefill_rejects_bad_arguments_before_launch(g):
    lib = g.library()
    fake = ctypes.c_void_p(256)
    # q, q_bytes, pools, pool_bytes, dtype, strides, table, table_bytes, max_pages, offsets,
    # offs_bytes, pos, pos_bytes, o, o_bytes
    base = [fake, 1 << 20, fake, fake, 1 << 22, 1, 4096, 256, 128, fake, 2 * 4 * 4, 4,
            fake, 3 * 4, fake, 2 * 4, fake, 1 << 20]
    ok_tail = [2, 8, 8, 4, 2, 128, 16, 8, 1.0, None, 0, None, None]
    # num_seqs, total, max_tokens, h, hk, d, page, pages, scale, ws, ws_bytes, status, stream
    rc = lib.gqa_attn_paged_prefill(*base, 2, 8, 8, 5, 2, 128, 16, 8, 1.0, None, 0, None, None)
    assert rc == 1 and "n_kv_heads" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_paged_prefill(*base, 2, 8, 8, 4, 2, 64, 16, 8, 1.0, None, 0, None, None)
    assert rc == 1 and "head_dim" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_paged_prefill(*base, 2, 8, 8, 4, 2, 128, 12, 8, 1.0, None, 0, None, None)
    assert rc == 1 and "page_size" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_paged_prefill(*base, 2, 8, 0, 4, 2, 128, 16, 8, 1.0, None, 0, None, None)
    assert rc == 1 and "max_tokens" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_paged_prefill(*base[:1], 100, *base[2:], *ok_tail)   # q too small
    assert rc == 1 and "q holds" in lib.gqa_last_error().decode()
    rc = lib.gqa_attn_paged_prefill(*base, *ok_tail[:8], float("nan"), None, 0, None, None)
    assert rc == 1 and "scale" in lib.gqa_last_error().decode()
    # with the shapes right, the missing workspace is what is reported
    rc = lib.gqa_attn_paged_prefill(*base, *ok_tail)
    ws = lib.gqa_attn_paged_prefill_workspace_size(2, 8, 4, 2, 128, 4, 16)
    assert (rc == 1 and "workspace" in lib.gqa_last_error().decode()) or ws == 0
    assert lib.gqa_attn_paged_prefill_workspace_size(2, 8, 4, 2, 96, 4, 16) == 0


def test_no_cpu_fallback(g, monkeypatch):
    """The product path fails loudly: host tensors are refused, and a missing library
    raises instead of falling back to anything else."""
    import torch
    q = torch.zeros((64, 4, 128), dtype=torch.float32)
    kv = torch.zeros((64, 2, 128), dtype=torch.float16)
    mask = torch.zeros((64, 64), dtype=torch.float16)
    with pytest.raises(TypeError, match="CUDA tensor"):
        g.gqa_attn_prefill(q, kv, kv, mask, 1.0)
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", ROOT / "attention_gqa_flash_gb300" / "lib" / "absent.so")
    with pytest.raises(RuntimeError, match="missing"):
        g.library()


def _declared_arity() -> dict[str, int]:
    """Parameter count of every function declared in the header."""
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(gqa_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(g):
    """Every function the Python binding types has the header's parameter count."""
    lib = g.library()
    arity = _declared_arity()
    typed = 0
    for name, n in arity.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        typed += 1
        assert len(fn.argtypes) == n, f"{name}: binding has {len(fn.argtypes)} arguments, header {n}"
    assert typed == len(arity), "every declared function is typed by the binding"
