// api.cpp -- the C ABI declared in include/gqa_attn.h: host-side validation,
// error reporting and dispatch to the kernel launchers.
//
// Validation mirrors the pages' host checks:
//   mlx-native 0.21.1 dflash2_attention_pack.rs: DFlash2AttentionPackParams::validate,
//     count (overflow-checked element counts), require (exact dtype/shape/bytes);
//   mlx-native 0.18.0 flash_attn_prefill_tensor.rs: dispatch_flash_attn_prefill_tensor_f16
//     (non-empty shape, head divisibility, kv_pad step, int32 range, 16-byte Q
//     rows) and need_elems (stride-aware extent of every buffer);
//   ferrum-kernels 0.8.3 causal_attention.rs: CausalAttentionShape::from_attributes
//     (head divisibility, head_dim <= 256).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "gqa_attn.h"
#include "launch.h"

namespace {

thread_local std::string g_last_error;

int fail(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return GQA_INVALID_ARGUMENT;
}

int cuda_fail(const char *what, cudaError_t e) {
    g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return GQA_CUDA_ERROR;
}

int ok() {
    g_last_error.clear();
    return GQA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bytes a strided [n0][n1][width] view needs: the last element's offset + 1.
// Returns false on overflow.
bool extent_bytes(int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t width, int64_t esize,
                  uint64_t *out) {
    if (n0 <= 0 || n1 <= 0 || width <= 0) return false;
    __int128 last = (__int128)(n0 - 1) * s0 + (__int128)(n1 - 1) * s1 + width;
    __int128 bytes = last * esize;
    if (bytes < 0 || bytes > (__int128)UINT64_MAX) return false;
    *out = (uint64_t)bytes;
    return true;
}

int need(const char *name, const void *p, size_t have, uint64_t need_bytes) {
    if (!p) return fail("%s is NULL", name);
    if (have < need_bytes)
        return fail("%s holds %zu bytes, the layout needs %llu", name, have,
                    (unsigned long long)need_bytes);
    return GQA_OK;
}

// Exact-size rule of the ring ops: product of dims x element size == bytes.
int require_exact(const char *name, const void *p, size_t have, const uint64_t *dims, int nd,
                  uint64_t esize) {
    if (!p) return fail("%s is NULL", name);
    __int128 n = esize;
    for (int i = 0; i < nd; ++i) {
        n *= dims[i];
        if (n > (__int128)UINT64_MAX) return fail("%s: shape overflow", name);
    }
    if ((__int128)have != n)
        return fail("%s must be %llu bytes, got %zu", name, (unsigned long long)n, have);
    if (!aligned(p, 16)) return fail("%s must be 16-byte aligned", name);
    return GQA_OK;
}

cudaStream_t cs(gqa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

namespace gqa {

unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {
bool g_timing = false;
bool g_timing_recorded = false;
cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;
}  // namespace

void timing_mark(bool before, cudaStream_t stream) {
    if (!g_timing) return;
    cudaEvent_t ev = before ? g_ev_start : g_ev_stop;
    // under stream capture the record becomes an event node of the graph, so that
    // every replay records the kernel's time
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (stream && cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, stream);
    if (!before) g_timing_recorded = true;
}

}  // namespace gqa

extern "C" {

const char *gqa_last_error(void) { return g_last_error.c_str(); }

const char *gqa_version(void) { return "gqa-attn-gb300 0.1.0 (sm_103a)"; }

int gqa_device_sm_count(void) { return gqa::sm_count(); }

int gqa_attn_set_cta_pairs(int mode) {
    if (mode < 0 || mode > 2) return fail("gqa_attn_set_cta_pairs: mode %d is not 0, 1 or 2", mode);
    gqa::set_attention_pairs(mode);
    return ok();
}

int gqa_timing_enable(int enable) {
    if (enable && !gqa::g_ev_start) {
        cudaError_t e = cudaEventCreate(&gqa::g_ev_start);
        if (e == cudaSuccess) e = cudaEventCreate(&gqa::g_ev_stop);
        if (e != cudaSuccess) return cuda_fail("timing events", e);
    }
    gqa::g_timing = enable != 0;
    gqa::g_timing_recorded = false;
    return ok();
}

int gqa_selftest_bounded_wait(int32_t *status, int timeout_ms, gqa_stream_t stream) {
    if (!status) return fail("selftest: status must not be NULL");
    if (timeout_ms < 1 || timeout_ms > 10000) return fail("selftest: timeout_ms must be 1..10000");
    cudaError_t e = gqa::launch_bounded_wait_selftest(status, timeout_ms, cs(stream));
    if (e != cudaSuccess) return cuda_fail("selftest launch", e);
    return ok();
}

float gqa_timing_last_ms(void) {
    if (!gqa::g_timing_recorded) return -1.f;
    float ms = -1.f;
    if (cudaEventSynchronize(gqa::g_ev_stop) != cudaSuccess) return -1.f;
    if (cudaEventElapsedTime(&ms, gqa::g_ev_start, gqa::g_ev_stop) != cudaSuccess) return -1.f;
    return ms;
}

uint32_t gqa_kv_pad(uint32_t kv_len) { return (uint32_t)(((uint64_t)kv_len + 63) / 64 * 64); }

// ---------------------------------------------------------------------------
// prefill
// ---------------------------------------------------------------------------
size_t gqa_attn_prefill_workspace_size(int rows, int n_heads, int n_kv_heads, int head_dim,
                                       int kv_pad) {
    if (rows <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || kv_pad <= 0) return 0;
    return gqa::prefill_workspace_bytes(rows, n_heads, n_kv_heads, head_dim, kv_pad);
}

int gqa_attn_prefill(const float *q, size_t q_bytes, int q_row_stride, int q_head_stride,
                     const void *k, size_t k_bytes, int k_row_stride, int k_head_stride,
                     const void *v, size_t v_bytes, int v_row_stride, int v_head_stride,
                     int kv_dtype, const uint16_t *mask, size_t mask_bytes, float *o,
                     size_t o_bytes, int rows, int n_heads, int n_kv_heads, int head_dim,
                     int kv_pad, float scale, void *workspace, size_t workspace_bytes,
                     int32_t *status, gqa_stream_t stream) {
    if (rows <= 0 || n_heads <= 0 || n_kv_heads <= 0 || kv_pad <= 0)
        return fail("prefill: empty shape rows=%d n_heads=%d n_kv_heads=%d kv_pad=%d", rows,
                    n_heads, n_kv_heads, kv_pad);
    if (n_heads % n_kv_heads != 0)
        return fail("prefill: n_heads %d is not a multiple of n_kv_heads %d", n_heads, n_kv_heads);
    if (kv_pad % 64 != 0) return fail("prefill: kv_pad %d is not a multiple of 64", kv_pad);
    if (head_dim != 128 && head_dim != 256 && head_dim != 512)
        return fail("prefill: unsupported head_dim %d (128, 256 or 512)", head_dim);
    if (kv_dtype != GQA_DTYPE_F16 && kv_dtype != GQA_DTYPE_BF16)
        return fail("prefill: kv_dtype must be GQA_DTYPE_F16 or GQA_DTYPE_BF16");
    if (q_row_stride < 0 || q_head_stride < 0 || k_row_stride < 0 || k_head_stride < 0 ||
        v_row_stride < 0 || v_head_stride < 0)
        return fail("prefill: strides must be non-negative");
    if (q_row_stride % 4 || q_head_stride % 4)
        return fail("prefill: Q strides must be multiples of 4 (16-byte rows)");
    if (k_row_stride % 8 || k_head_stride % 8 || v_row_stride % 8 || v_head_stride % 8)
        return fail("prefill: K/V strides must be multiples of 8 (16-byte rows)");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(mask, 16) ||
        !aligned(o, 16))
        return fail("prefill: q, k, v, mask and o must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail("prefill: scale must be finite");
    uint64_t nb;
    int rc;
    if (!extent_bytes(rows, q_row_stride, n_heads, q_head_stride, head_dim, 4, &nb))
        return fail("prefill: q extent overflows");
    if ((rc = need("q", q, q_bytes, nb))) return rc;
    if (!extent_bytes(kv_pad, k_row_stride, n_kv_heads, k_head_stride, head_dim, 2, &nb))
        return fail("prefill: k extent overflows");
    if ((rc = need("k", k, k_bytes, nb))) return rc;
    if (!extent_bytes(kv_pad, v_row_stride, n_kv_heads, v_head_stride, head_dim, 2, &nb))
        return fail("prefill: v extent overflows");
    if ((rc = need("v", v, v_bytes, nb))) return rc;
    if ((rc = need("mask", mask, mask_bytes, (uint64_t)rows * kv_pad * 2))) return rc;
    if ((rc = need("o", o, o_bytes, (uint64_t)rows * n_heads * head_dim * 4))) return rc;
    const size_t ws_need = gqa::prefill_workspace_bytes(rows, n_heads, n_kv_heads, head_dim, kv_pad);
    if (ws_need && (rc = need("workspace", workspace, workspace_bytes, ws_need))) return rc;
    if (ws_need && !aligned(workspace, 256)) return fail("prefill: workspace must be 256-byte aligned");

    gqa::AttnProblem p{};
    p.q = q;
    p.q_is_f32 = true;
    p.q_row_stride = q_row_stride;
    p.q_head_stride = q_head_stride;
    p.q_lane_stride = 0;
    p.k = k;
    p.v = v;
    p.kv_dtype = kv_dtype;
    p.k_row_stride = k_row_stride;
    p.k_head_stride = k_head_stride;
    p.v_row_stride = v_row_stride;
    p.v_head_stride = v_head_stride;
    p.kv_lane_stride = 0;
    p.kv_rows = kv_pad;
    p.mask = mask;
    p.mask_row_stride = kv_pad;
    p.mask_head_stride = 0;
    p.mask_lane_stride = 0;
    p.o = o;
    p.o_row_stride = (int64_t)n_heads * head_dim;
    p.o_head_stride = head_dim;
    p.o_lane_stride = 0;
    p.lanes = 1;
    p.rows = rows;
    p.n_heads = n_heads;
    p.n_kv_heads = n_kv_heads;
    p.head_dim = head_dim;
    p.n_keys = kv_pad;
    p.scale = scale;
    p.status = status;
    cudaError_t e = gqa::launch_attention(p, workspace, cs(stream));
    if (e != cudaSuccess) return cuda_fail("prefill launch", e);
    return ok();
}

// ---------------------------------------------------------------------------
// paged decode
// ---------------------------------------------------------------------------
size_t gqa_attn_paged_decode_workspace_size(int num_seqs, int n_heads, int head_dim,
                                            int max_pages_per_seq, int page_size) {
    if (num_seqs <= 0 || n_heads <= 0 || head_dim <= 0 || max_pages_per_seq <= 0 || page_size <= 0)
        return 0;
    return gqa::decode_workspace_bytes(num_seqs, n_heads, head_dim, max_pages_per_seq, page_size);
}

int gqa_attn_paged_decode(const float *q, size_t q_bytes, const void *k_pages,
                          const void *v_pages, size_t pool_bytes, int kv_dtype,
                          int64_t page_stride, int64_t token_stride, int64_t head_stride,
                          const int32_t *page_table, size_t page_table_bytes,
                          int max_pages_per_seq, const int32_t *context_lens,
                          size_t context_lens_bytes, float *o, size_t o_bytes, int num_seqs,
                          int n_heads, int n_kv_heads, int head_dim, int page_size,
                          int num_pages, float scale, void *workspace, size_t workspace_bytes,
                          int32_t *status, gqa_stream_t stream) {
    if (num_seqs <= 0 || n_heads <= 0 || n_kv_heads <= 0 || num_pages <= 0 ||
        max_pages_per_seq <= 0 || page_size <= 0)
        return fail("paged decode: empty shape");
    if (n_heads % n_kv_heads != 0)
        return fail("paged decode: n_heads %d is not a multiple of n_kv_heads %d", n_heads,
                    n_kv_heads);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail("paged decode: unsupported head_dim %d (64, 128 or 256)", head_dim);
    if (kv_dtype != GQA_DTYPE_F16 && kv_dtype != GQA_DTYPE_BF16)
        return fail("paged decode: kv_dtype must be GQA_DTYPE_F16 or GQA_DTYPE_BF16");
    if (page_stride < 0 || token_stride < 0 || head_stride < 0 || page_stride % 8 ||
        token_stride % 8 || head_stride % 8)
        return fail("paged decode: pool strides must be non-negative multiples of 8");
    if ((int64_t)max_pages_per_seq * page_size > INT32_MAX)
        return fail("paged decode: max_pages_per_seq * page_size exceeds int32");
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(o, 16))
        return fail("paged decode: q, pools and o must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail("paged decode: scale must be finite");
    int rc;
    const uint64_t qo = (uint64_t)num_seqs * n_heads * head_dim * 4;
    if ((rc = need("q", q, q_bytes, qo))) return rc;
    if ((rc = need("o", o, o_bytes, qo))) return rc;
    __int128 last = (__int128)(num_pages - 1) * page_stride + (__int128)(page_size - 1) * token_stride +
                    (__int128)(n_kv_heads - 1) * head_stride + head_dim;
    if (last * 2 > (__int128)UINT64_MAX) return fail("paged decode: pool extent overflows");
    if ((rc = need("k_pages", k_pages, pool_bytes, (uint64_t)(last * 2)))) return rc;
    if ((rc = need("v_pages", v_pages, pool_bytes, (uint64_t)(last * 2)))) return rc;
    if ((rc = need("page_table", page_table, page_table_bytes,
                   (uint64_t)num_seqs * max_pages_per_seq * 4)))
        return rc;
    if ((rc = need("context_lens", context_lens, context_lens_bytes, (uint64_t)num_seqs * 4)))
        return rc;
    const size_t ws_need =
        gqa::decode_workspace_bytes(num_seqs, n_heads, head_dim, max_pages_per_seq, page_size);
    if ((rc = need("workspace", workspace, workspace_bytes, ws_need))) return rc;
    if (!aligned(workspace, 256)) return fail("paged decode: workspace must be 256-byte aligned");
    gqa::DecodeProblem p{q,          k_pages,    v_pages,   kv_dtype,  page_stride,
                         token_stride, head_stride, page_table, max_pages_per_seq, context_lens,
                         o,          num_seqs,   n_heads,   n_kv_heads, head_dim,
                         page_size,  num_pages,  scale,     status};
    cudaError_t e = gqa::launch_paged_decode(p, workspace, cs(stream));
    if (e != cudaSuccess) return cuda_fail("paged decode launch", e);
    return ok();
}

// Paged decode for callers that cannot supply a workspace: the split-KV
// partials go to the library's fixed device array (no allocation anywhere on
// this path), after which the regular entry point does all validation and the
// launch.
int gqa_attn_paged_decode_noalloc(const float *q, size_t q_bytes, const void *k_pages,
                                  const void *v_pages, size_t pool_bytes, int kv_dtype,
                                  int64_t page_stride, int64_t token_stride, int64_t head_stride,
                                  const int32_t *page_table, size_t page_table_bytes,
                                  int max_pages_per_seq, const int32_t *context_lens,
                                  size_t context_lens_bytes, float *o, size_t o_bytes,
                                  int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                                  int page_size, int num_pages, float scale, int32_t *status,
                                  gqa_stream_t stream) {
    if (num_seqs <= 0 || n_heads <= 0 || head_dim <= 0 || max_pages_per_seq <= 0 || page_size <= 0)
        return fail("paged decode (no-alloc): empty shape");
    const size_t need =
        gqa::decode_workspace_bytes(num_seqs, n_heads, head_dim, max_pages_per_seq, page_size);
    if (need > (size_t)GQA_NOALLOC_SCRATCH_BYTES)
        return fail("paged decode (no-alloc): this problem needs %zu bytes of scratch "
                    "(num_seqs x ceil(max_pages_per_seq*page_size/1024) x n_heads x (head_dim+1) x 4), "
                    "more than the fixed %u-byte array; use gqa_attn_paged_decode with a workspace",
                    need, (unsigned)GQA_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    const cudaError_t e = gqa::decode_fixed_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail("paged decode (no-alloc): scratch address lookup", e);
    return gqa_attn_paged_decode(q, q_bytes, k_pages, v_pages, pool_bytes, kv_dtype, page_stride,
                                 token_stride, head_stride, page_table, page_table_bytes,
                                 max_pages_per_seq, context_lens, context_lens_bytes, o, o_bytes,
                                 num_seqs, n_heads, n_kv_heads, head_dim, page_size, num_pages,
                                 scale, scratch, (size_t)GQA_NOALLOC_SCRATCH_BYTES, status, stream);
}

// ---------------------------------------------------------------------------
// Page append and chunked prefill over pages
// ---------------------------------------------------------------------------
namespace {

// Checks shared by the two entry points that address the pool through
// token_offsets / position_start / page_table (`what` names the caller).
int check_pool(const char *what, const void *k_pages, const void *v_pages, size_t pool_bytes,
               int kv_dtype, int64_t page_stride, int64_t token_stride, int64_t head_stride,
               const int32_t *page_table, size_t page_table_bytes, int max_pages_per_seq,
               const int32_t *token_offsets, size_t token_offsets_bytes,
               const int32_t *position_start, size_t position_start_bytes, int num_seqs,
               int n_kv_heads, int head_dim, int page_size, int num_pages) {
    if (num_seqs <= 0 || n_kv_heads <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 ||
        page_size <= 0)
        return fail("%s: empty shape", what);
    if (kv_dtype != GQA_DTYPE_F16 && kv_dtype != GQA_DTYPE_BF16)
        return fail("%s: kv_dtype must be GQA_DTYPE_F16 or GQA_DTYPE_BF16", what);
    if (page_stride <= 0 || token_stride <= 0 || head_stride <= 0 || page_stride % 8 ||
        token_stride % 8 || head_stride % 8)
        return fail("%s: pool strides must be positive multiples of 8", what);
    if ((int64_t)max_pages_per_seq * page_size > INT32_MAX)
        return fail("%s: max_pages_per_seq * page_size exceeds int32", what);
    if (!aligned(k_pages, 16) || !aligned(v_pages, 16))
        return fail("%s: pools must be 16-byte aligned", what);
    __int128 last = (__int128)(num_pages - 1) * page_stride + (__int128)(page_size - 1) * token_stride +
                    (__int128)(n_kv_heads - 1) * head_stride + head_dim;
    if (last * 2 > (__int128)UINT64_MAX) return fail("%s: pool extent overflows", what);
    int rc;
    if ((rc = need("k_pages", k_pages, pool_bytes, (uint64_t)(last * 2)))) return rc;
    if ((rc = need("v_pages", v_pages, pool_bytes, (uint64_t)(last * 2)))) return rc;
    if ((rc = need("page_table", page_table, page_table_bytes,
                   (uint64_t)num_seqs * max_pages_per_seq * 4)))
        return rc;
    if ((rc = need("token_offsets", token_offsets, token_offsets_bytes, ((uint64_t)num_seqs + 1) * 4)))
        return rc;
    if ((rc = need("position_start", position_start, position_start_bytes, (uint64_t)num_seqs * 4)))
        return rc;
    return GQA_OK;
}

}  // namespace

int gqa_paged_append(const float *k_new, const float *v_new, size_t new_bytes,
                     const int32_t *token_offsets, size_t token_offsets_bytes,
                     const int32_t *position_start, size_t position_start_bytes,
                     const int32_t *page_table, size_t page_table_bytes, int max_pages_per_seq,
                     void *k_pages, void *v_pages, size_t pool_bytes, int kv_dtype,
                     int64_t page_stride, int64_t token_stride, int64_t head_stride, int num_seqs,
                     int total_tokens, int n_kv_heads, int head_dim, int page_size, int num_pages,
                     int32_t *status, gqa_stream_t stream) {
    int rc;
    if (head_dim <= 0 || head_dim % 8 || head_dim > 4096)
        return fail("paged append: head_dim %d must be a positive multiple of 8 (at most 4096)",
                    head_dim);
    if (total_tokens < 0) return fail("paged append: total_tokens is negative");
    if ((rc = check_pool("paged append", k_pages, v_pages, pool_bytes, kv_dtype, page_stride,
                         token_stride, head_stride, page_table, page_table_bytes, max_pages_per_seq,
                         token_offsets, token_offsets_bytes, position_start, position_start_bytes,
                         num_seqs, n_kv_heads, head_dim, page_size, num_pages)))
        return rc;
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return fail("paged append: k_new and v_new must be 16-byte aligned");
    const uint64_t rows = (uint64_t)total_tokens * n_kv_heads * head_dim * 4;
    if (total_tokens > 0) {
        if ((rc = need("k_new", k_new, new_bytes, rows))) return rc;
        if ((rc = need("v_new", v_new, new_bytes, rows))) return rc;
    }
    gqa::PagedAppendProblem p{k_new,       v_new,        token_offsets, position_start,
                              page_table,  max_pages_per_seq, k_pages, v_pages,
                              kv_dtype,    page_stride,  token_stride,  head_stride,
                              num_seqs,    total_tokens, n_kv_heads,    head_dim,
                              page_size,   num_pages,    status};
    const cudaError_t e = gqa::launch_paged_append(p, cs(stream));
    if (e != cudaSuccess) return cuda_fail("paged append launch", e);
    return ok();
}

size_t gqa_attn_paged_prefill_workspace_size(int num_seqs, int max_tokens, int n_heads,
                                             int n_kv_heads, int head_dim, int max_pages_per_seq,
                                             int page_size) {
    if (num_seqs <= 0 || max_tokens <= 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads || !(head_dim == 128 || head_dim == 256) || max_pages_per_seq <= 0 ||
        page_size <= 0 || (int64_t)max_pages_per_seq * page_size > INT32_MAX)
        return 0;
    return gqa::paged_prefill_workspace_bytes(num_seqs, max_tokens, n_heads, n_kv_heads, head_dim,
                                              max_pages_per_seq, page_size);
}

int gqa_attn_paged_prefill(const float *q, size_t q_bytes, const void *k_pages,
                           const void *v_pages, size_t pool_bytes, int kv_dtype,
                           int64_t page_stride, int64_t token_stride, int64_t head_stride,
                           const int32_t *page_table, size_t page_table_bytes,
                           int max_pages_per_seq, const int32_t *token_offsets,
                           size_t token_offsets_bytes, const int32_t *position_start,
                           size_t position_start_bytes, float *o, size_t o_bytes, int num_seqs,
                           int total_tokens, int max_tokens, int n_heads, int n_kv_heads,
                           int head_dim, int page_size, int num_pages, float scale,
                           void *workspace, size_t workspace_bytes, int32_t *status,
                           gqa_stream_t stream) {
    int rc;
    if (n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0)
        return fail("paged prefill: n_heads %d is not a positive multiple of n_kv_heads %d", n_heads,
                    n_kv_heads);
    if (head_dim != 128 && head_dim != 256)
        return fail("paged prefill: unsupported head_dim %d (128 or 256)", head_dim);
    if (page_size % 8)
        return fail("paged prefill: page_size %d must be a multiple of 8", page_size);
    if (total_tokens < 0 || max_tokens <= 0)
        return fail("paged prefill: total_tokens must be >= 0 and max_tokens > 0");
    if ((int64_t)total_tokens * n_heads > INT32_MAX)
        return fail("paged prefill: total_tokens * n_heads exceeds int32");
    if ((rc = check_pool("paged prefill", k_pages, v_pages, pool_bytes, kv_dtype, page_stride,
                         token_stride, head_stride, page_table, page_table_bytes, max_pages_per_seq,
                         token_offsets, token_offsets_bytes, position_start, position_start_bytes,
                         num_seqs, n_kv_heads, head_dim, page_size, num_pages)))
        return rc;
    if (!aligned(q, 16) || !aligned(o, 16)) return fail("paged prefill: q and o must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail("paged prefill: scale must be finite");
    const uint64_t qo = (uint64_t)total_tokens * n_heads * head_dim * 4;
    if (total_tokens > 0) {
        if ((rc = need("q", q, q_bytes, qo))) return rc;
        if ((rc = need("o", o, o_bytes, qo))) return rc;
    }
    const size_t ws_need = gqa::paged_prefill_workspace_bytes(num_seqs, max_tokens, n_heads, n_kv_heads,
                                                              head_dim, max_pages_per_seq, page_size);
    if (ws_need > 0) {
        if ((rc = need("workspace", workspace, workspace_bytes, ws_need))) return rc;
        if (!aligned(workspace, 256)) return fail("paged prefill: workspace must be 256-byte aligned");
    }
    gqa::PagedPrefillProblem p{q,           o,           k_pages,          v_pages,
                               kv_dtype,    page_stride, token_stride,     head_stride,
                               page_table,  max_pages_per_seq, token_offsets, position_start,
                               num_seqs,    total_tokens, max_tokens,      n_heads,
                               n_kv_heads,  head_dim,    page_size,        num_pages,
                               scale,       status};
    const cudaError_t e = gqa::launch_paged_prefill(p, workspace, cs(stream));
    if (e != cudaSuccess) return cuda_fail("paged prefill launch", e);
    return ok();
}

// ---------------------------------------------------------------------------
// DFlash2 ring KV
// ---------------------------------------------------------------------------
int gqa_ring_params_valid(const gqa_ring_params *p) {
    if (!p) {
        fail("ring params are NULL");
        return 0;
    }
    const gqa_ring_params g = *p;
    if (g.lanes == 0 || g.lanes > 4 || g.q_heads == 0 || g.kv_heads == 0 ||
        g.q_heads % g.kv_heads != 0 || !(g.head_dim == 128 || g.head_dim == 256) || g.rows < 2 ||
        g.rows > 16 || g.window <= g.rows || g.packed_len != g.window - 1 + g.rows ||
        g.max_commit == 0 || g.max_commit > g.rows || g.window > (1u << 24) || g.q_heads > 4096) {
        fail("invalid DFlash2 attention geometry: lanes=%u q_heads=%u kv_heads=%u head_dim=%u "
             "rows=%u window=%u packed_len=%u max_commit=%u",
             g.lanes, g.q_heads, g.kv_heads, g.head_dim, g.rows, g.window, g.packed_len,
             g.max_commit);
        return 0;
    }
    ok();
    return 1;
}

#define RING_CHECK(p)                                       \
    do {                                                    \
        if (!gqa_ring_params_valid(p)) return GQA_INVALID_ARGUMENT; \
    } while (0)

int gqa_pack_attention(const uint16_t *ring_k, size_t ring_k_bytes, const uint16_t *ring_v,
                       size_t ring_v_bytes, const float *cur_q, size_t cur_q_bytes,
                       const float *cur_k, size_t cur_k_bytes, const float *cur_v,
                       size_t cur_v_bytes, const uint32_t *cache_lengths,
                       size_t cache_lengths_bytes, const uint32_t *write_positions,
                       size_t write_positions_bytes, uint16_t *packed_q, size_t packed_q_bytes,
                       uint16_t *packed_k, size_t packed_k_bytes, uint16_t *packed_v,
                       size_t packed_v_bytes, const gqa_ring_params *p, int32_t *status,
                       gqa_stream_t stream) {
    RING_CHECK(p);
    const uint64_t b = p->lanes, h = p->q_heads, hk = p->kv_heads, d = p->head_dim, r = p->rows,
                   w = p->window, k = p->packed_len;
    const uint64_t ring[] = {b, hk, w, d}, cq[] = {b, r, h, d}, ck[] = {b, r, hk, d}, lanes[] = {b},
                   pq[] = {b, h, r, d}, pk[] = {b, hk, k, d};
    int rc;
    if ((rc = require_exact("ring keys", ring_k, ring_k_bytes, ring, 4, 2))) return rc;
    if ((rc = require_exact("ring values", ring_v, ring_v_bytes, ring, 4, 2))) return rc;
    if ((rc = require_exact("current queries", cur_q, cur_q_bytes, cq, 4, 4))) return rc;
    if ((rc = require_exact("current keys", cur_k, cur_k_bytes, ck, 4, 4))) return rc;
    if ((rc = require_exact("current values", cur_v, cur_v_bytes, ck, 4, 4))) return rc;
    if ((rc = require_exact("cache lengths", cache_lengths, cache_lengths_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("write positions", write_positions, write_positions_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("packed queries", packed_q, packed_q_bytes, pq, 4, 2))) return rc;
    if ((rc = require_exact("packed keys", packed_k, packed_k_bytes, pk, 4, 2))) return rc;
    if ((rc = require_exact("packed values", packed_v, packed_v_bytes, pk, 4, 2))) return rc;
    cudaError_t e = gqa::launch_pack_attention(ring_k, ring_v, cur_q, cur_k, cur_v, cache_lengths,
                                               write_positions, packed_q, packed_k, packed_v, *p,
                                               status, cs(stream));
    if (e != cudaSuccess) return cuda_fail("pack_attention launch", e);
    return ok();
}

int gqa_fill_mask(const uint32_t *cache_lengths, size_t cache_lengths_bytes, uint16_t *mask,
                  size_t mask_bytes, const gqa_ring_params *p, int32_t *status,
                  gqa_stream_t stream) {
    RING_CHECK(p);
    const uint64_t lanes[] = {p->lanes}, m[] = {p->lanes, p->q_heads, p->rows, p->packed_len};
    int rc;
    if ((rc = require_exact("cache lengths", cache_lengths, cache_lengths_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("mask", mask, mask_bytes, m, 4, 2))) return rc;
    cudaError_t e = gqa::launch_fill_mask(cache_lengths, mask, *p, status, cs(stream));
    if (e != cudaSuccess) return cuda_fail("fill_mask launch", e);
    return ok();
}

size_t gqa_attn_verify_workspace_size(const gqa_ring_params *p) {
    if (!gqa_ring_params_valid(p)) return 0;
    return gqa::verify_workspace_bytes(*p);
}

int gqa_attn_verify(const uint16_t *packed_q, size_t packed_q_bytes, const uint16_t *packed_k,
                    size_t packed_k_bytes, const uint16_t *packed_v, size_t packed_v_bytes,
                    const uint16_t *mask, size_t mask_bytes, float *o, size_t o_bytes,
                    const gqa_ring_params *p, float scale, void *workspace,
                    size_t workspace_bytes, int32_t *status, gqa_stream_t stream) {
    RING_CHECK(p);
    if (!std::isfinite(scale)) return fail("verify: scale must be finite");
    const uint64_t b = p->lanes, h = p->q_heads, hk = p->kv_heads, d = p->head_dim, r = p->rows,
                   k = p->packed_len;
    const uint64_t pq[] = {b, h, r, d}, pk[] = {b, hk, k, d}, m[] = {b, h, r, k},
                   od[] = {b, r, h, d};
    int rc;
    if ((rc = require_exact("packed queries", packed_q, packed_q_bytes, pq, 4, 2))) return rc;
    if ((rc = require_exact("packed keys", packed_k, packed_k_bytes, pk, 4, 2))) return rc;
    if ((rc = require_exact("packed values", packed_v, packed_v_bytes, pk, 4, 2))) return rc;
    if ((rc = require_exact("mask", mask, mask_bytes, m, 4, 2))) return rc;
    if ((rc = require_exact("output", o, o_bytes, od, 4, 4))) return rc;
    const size_t ws_need = gqa::verify_workspace_bytes(*p);
    if (ws_need && (rc = need("workspace", workspace, workspace_bytes, ws_need))) return rc;
    if (ws_need && !aligned(workspace, 256)) return fail("verify: workspace must be 256-byte aligned");

    gqa::AttnProblem a{};
    a.q = packed_q;
    a.q_is_f32 = false;
    a.q_row_stride = d;            // row r of head h: (h*R + r)*D
    a.q_head_stride = r * d;
    a.q_lane_stride = h * r * d;
    a.k = packed_k;
    a.v = packed_v;
    a.kv_dtype = GQA_DTYPE_BF16;
    a.k_row_stride = d;
    a.k_head_stride = k * d;
    a.v_row_stride = d;
    a.v_head_stride = k * d;
    a.kv_lane_stride = hk * k * d;
    a.kv_rows = k;
    a.mask = mask;
    a.mask_is_bf16 = true;
    a.mask_row_stride = k;
    a.mask_head_stride = r * k;
    a.mask_lane_stride = h * r * k;
    a.o = o;
    a.o_row_stride = h * d;
    a.o_head_stride = d;
    a.o_lane_stride = r * h * d;
    a.lanes = (int)b;
    a.rows = (int)r;
    a.n_heads = (int)h;
    a.n_kv_heads = (int)hk;
    a.head_dim = (int)d;
    a.n_keys = (int)k;
    a.scale = scale;
    a.status = status;
    cudaError_t e = gqa::launch_attention(a, workspace, cs(stream));
    if (e != cudaSuccess) return cuda_fail("verify launch", e);
    return ok();
}

size_t gqa_attn_verify_ring_workspace_size(const gqa_ring_params *p) {
    if (!gqa_ring_params_valid(p)) return 0;
    return gqa::verify_ring_workspace_bytes(*p);
}

int gqa_attn_verify_ring(const uint16_t *ring_k, size_t ring_k_bytes, const uint16_t *ring_v,
                         size_t ring_v_bytes, const float *cur_q, size_t cur_q_bytes,
                         const float *cur_k, size_t cur_k_bytes, const float *cur_v,
                         size_t cur_v_bytes, const uint32_t *cache_lengths,
                         size_t cache_lengths_bytes, const uint32_t *write_positions,
                         size_t write_positions_bytes, float *o, size_t o_bytes,
                         const gqa_ring_params *p, float scale, void *workspace,
                         size_t workspace_bytes, int32_t *status, gqa_stream_t stream) {
    RING_CHECK(p);
    if (!std::isfinite(scale)) return fail("verify_ring: scale must be finite");
    const uint64_t b = p->lanes, h = p->q_heads, hk = p->kv_heads, d = p->head_dim, r = p->rows,
                   w = p->window;
    const uint64_t ring[] = {b, hk, w, d}, cq[] = {b, r, h, d}, ck[] = {b, r, hk, d}, lanes[] = {b},
                   od[] = {b, r, h, d};
    int rc;
    if ((rc = require_exact("ring keys", ring_k, ring_k_bytes, ring, 4, 2))) return rc;
    if ((rc = require_exact("ring values", ring_v, ring_v_bytes, ring, 4, 2))) return rc;
    if ((rc = require_exact("current queries", cur_q, cur_q_bytes, cq, 4, 4))) return rc;
    if ((rc = require_exact("current keys", cur_k, cur_k_bytes, ck, 4, 4))) return rc;
    if ((rc = require_exact("current values", cur_v, cur_v_bytes, ck, 4, 4))) return rc;
    if ((rc = require_exact("cache lengths", cache_lengths, cache_lengths_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("write positions", write_positions, write_positions_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("output", o, o_bytes, od, 4, 4))) return rc;
    if (!aligned(ring_k, 16) || !aligned(ring_v, 16) || !aligned(cur_q, 16) || !aligned(cur_k, 16) ||
        !aligned(cur_v, 16))
        return fail("verify_ring: rings and current rows must be 16-byte aligned");
    const size_t ws_need = gqa::verify_ring_workspace_bytes(*p);
    if (ws_need && (rc = need("workspace", workspace, workspace_bytes, ws_need))) return rc;
    if (ws_need && !aligned(workspace, 256)) return fail("verify_ring: workspace must be 256-byte aligned");

    gqa::AttnProblem a{};
    a.q = cur_q;  // [b][r][h][d] f32, rounded to bf16 in the kernel
    a.q_is_f32 = true;
    a.q_row_stride = h * d;
    a.q_head_stride = d;
    a.q_lane_stride = r * h * d;
    a.k = ring_k;
    a.v = ring_v;
    a.kv_dtype = GQA_DTYPE_BF16;
    a.k_row_stride = d;
    a.k_head_stride = w * d;
    a.v_row_stride = d;
    a.v_head_stride = w * d;
    a.kv_lane_stride = hk * w * d;
    a.kv_rows = (int)w;
    a.mask = nullptr;
    a.mask_is_bf16 = true;
    a.o = o;
    a.o_row_stride = h * d;
    a.o_head_stride = d;
    a.o_lane_stride = r * h * d;
    a.lanes = (int)b;
    a.rows = (int)r;
    a.n_heads = (int)h;
    a.n_kv_heads = (int)hk;
    a.head_dim = (int)d;
    a.n_keys = 0;
    a.scale = scale;
    a.status = status;
    a.ring = true;
    a.ring_w = (int)w;
    a.cur_k = cur_k;
    a.cur_v = cur_v;
    a.ring_len = cache_lengths;
    a.ring_wp = write_positions;
    cudaError_t e = gqa::launch_attention(a, workspace, cs(stream));
    if (e != cudaSuccess) return cuda_fail("verify_ring launch", e);
    return ok();
}

int gqa_commit_kv(const float *new_k, size_t new_k_bytes, const float *new_v,
                  size_t new_v_bytes, const uint32_t *commit_counts, size_t commit_counts_bytes,
                  const uint32_t *write_positions, size_t write_positions_bytes,
                  uint16_t *ring_k, size_t ring_k_bytes, uint16_t *ring_v, size_t ring_v_bytes,
                  const gqa_ring_params *p, int32_t *status, gqa_stream_t stream) {
    RING_CHECK(p);
    const uint64_t b = p->lanes, hk = p->kv_heads, d = p->head_dim, w = p->window,
                   c = p->max_commit;
    const uint64_t nk[] = {b, c, hk, d}, lanes[] = {b}, ring[] = {b, hk, w, d};
    int rc;
    if ((rc = require_exact("new keys", new_k, new_k_bytes, nk, 4, 4))) return rc;
    if ((rc = require_exact("new values", new_v, new_v_bytes, nk, 4, 4))) return rc;
    if ((rc = require_exact("commit counts", commit_counts, commit_counts_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("write positions", write_positions, write_positions_bytes, lanes, 1, 4)))
        return rc;
    if ((rc = require_exact("ring keys", ring_k, ring_k_bytes, ring, 4, 2))) return rc;
    if ((rc = require_exact("ring values", ring_v, ring_v_bytes, ring, 4, 2))) return rc;
    cudaError_t e = gqa::launch_commit_kv(new_k, new_v, commit_counts, write_positions, ring_k,
                                          ring_v, *p, status, cs(stream));
    if (e != cudaSuccess) return cuda_fail("commit_kv launch", e);
    return ok();
}

int gqa_set_mask_rows(const uint16_t *mask_embedding, size_t mask_embedding_bytes,
                      float *hidden, size_t hidden_bytes, uint32_t lanes, uint32_t rows,
                      uint32_t width, gqa_stream_t stream) {
    if (lanes == 0 || lanes > 4 || rows < 2 || rows > 16 || width == 0 || width > (1u << 28))
        return fail("invalid DFlash2 mask-row geometry: lanes=%u rows=%u hidden=%u", lanes, rows,
                    width);
    const uint64_t e[] = {width}, hdims[] = {(uint64_t)lanes * rows, width};
    int rc;
    if ((rc = require_exact("mask embedding", mask_embedding, mask_embedding_bytes, e, 1, 2)))
        return rc;
    if ((rc = require_exact("draft input", hidden, hidden_bytes, hdims, 2, 4))) return rc;
    cudaError_t err =
        gqa::launch_set_mask_rows(mask_embedding, hidden, (int)lanes, (int)rows, (int)width, cs(stream));
    if (err != cudaSuccess) return cuda_fail("set_mask_rows launch", err);
    return ok();
}

}  // extern "C"
