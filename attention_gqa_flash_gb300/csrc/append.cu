// append.cu -- page append: every new token's K and V rows (f32) rounded to
// the pool's 16-bit type and written into the token's page slot.
//
// Semantics follow ferrum-kernels 0.8.3 src/backend/metal/vnext_ops/causal_attention.rs:
// the prepare step of a causal-attention launch writes the new tokens' K and V
// into the paged state (dispatch_prepare, vnext_causal_prepare_f16) before the
// attention step reads them; token i of a launch sits at position
// position_start + i, and position p lives in slot p % page_size of the
// sequence's page p / page_size (paged_state_regions).  Normalisation and
// rotary embedding, which that step also applies, are model-specific and not
// part of this library: the rows arrive ready.
//
// Design (HBM-bound; each element is read once as f32 and written once as
// 16 bits, for K and for V): one thread moves one 8-element chunk of one
// (token, KV head) row of both K and V -- two 32-byte reads and two 16-byte
// stores.  Consecutive threads take consecutive chunks of a row, then the
// next KV head, then the next token, so the reads are fully coalesced and each
// row's stores fill whole sectors.  A token's sequence is the last s with
// token_offsets[s] <= i (binary search; the offsets stay in L1).
#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

struct AppendArgs {
    const float *k_new, *v_new;  // [total_tokens][n_kv_heads][head_dim]
    const int32_t *tok_off, *pos_start, *page_table;
    uint16_t *k_pool, *v_pool;
    int64_t page_stride, token_stride, head_stride;
    int num_seqs, total_tokens, n_kv_heads, chunks, page_size, num_pages, max_pages;
    int32_t *status;
};

template <class KV>
__global__ void __launch_bounds__(256) page_append_kernel(const AppendArgs a) {
    const int64_t row_chunks = (int64_t)a.n_kv_heads * a.chunks;
    const int64_t work = (int64_t)a.total_tokens * row_chunks;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int o0 = a.tok_off[0], on = a.tok_off[a.num_seqs];
        if (o0 < 0 || on > a.total_tokens || o0 > on) raise_flag(a.status, GQA_FLAG_CONTEXT_CLAMPED);
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < work; t += stride) {
        const int i = (int)(t / row_chunks);
        const int rem = (int)(t - (int64_t)i * row_chunks);
        const int g = rem / a.chunks, ch = rem - g * a.chunks;
        // the row's data first: its loads are in flight while the slot is looked up
        const int64_t src = ((int64_t)i * a.n_kv_heads + g) * (a.chunks * 8) + ch * 8;
        const float4 k0 = ld_nc_f4(a.k_new + src), k1 = ld_nc_f4(a.k_new + src + 4);
        const float4 v0 = ld_nc_f4(a.v_new + src), v1 = ld_nc_f4(a.v_new + src + 4);
        int lo = 0, hi = a.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.tok_off[mid] <= i)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int o0 = a.tok_off[lo];
        if (i < o0 || i >= a.tok_off[lo + 1]) continue;  // the token belongs to no sequence
        const int64_t p = (int64_t)a.pos_start[lo] + (i - o0);
        const int64_t pi = p >= 0 ? p / a.page_size : -1;
        const int page = (pi >= 0 && pi < a.max_pages) ? a.page_table[(int64_t)lo * a.max_pages + pi] : -1;
        if (page < 0 || page >= a.num_pages) {
            // outside the page table or the pool: not written
            if (g == 0 && ch == 0) raise_flag(a.status, GQA_FLAG_PAGE_CLAMPED);
            continue;
        }
        const int64_t dst = (int64_t)page * a.page_stride + (p - pi * a.page_size) * a.token_stride +
                            (int64_t)g * a.head_stride + ch * 8;
        st_v4(a.k_pool + dst, make_uint4(pack2(KV{}, k0.x, k0.y), pack2(KV{}, k0.z, k0.w),
                                         pack2(KV{}, k1.x, k1.y), pack2(KV{}, k1.z, k1.w)));
        st_v4(a.v_pool + dst, make_uint4(pack2(KV{}, v0.x, v0.y), pack2(KV{}, v0.z, v0.w),
                                         pack2(KV{}, v1.x, v1.y), pack2(KV{}, v1.z, v1.w)));
    }
}

}  // namespace

cudaError_t launch_paged_append(const PagedAppendProblem &p, cudaStream_t stream) {
    if (p.total_tokens == 0) return cudaSuccess;
    AppendArgs a;
    a.k_new = p.k_new;
    a.v_new = p.v_new;
    a.tok_off = p.token_offsets;
    a.pos_start = p.position_start;
    a.page_table = p.page_table;
    a.k_pool = static_cast<uint16_t *>(p.k_pool);
    a.v_pool = static_cast<uint16_t *>(p.v_pool);
    a.page_stride = p.page_stride;
    a.token_stride = p.token_stride;
    a.head_stride = p.head_stride;
    a.num_seqs = p.num_seqs;
    a.total_tokens = p.total_tokens;
    a.n_kv_heads = p.n_kv_heads;
    a.chunks = p.head_dim / 8;
    a.page_size = p.page_size;
    a.num_pages = p.num_pages;
    a.max_pages = p.max_pages_per_seq;
    a.status = p.status;
    const int64_t work = (int64_t)p.total_tokens * p.n_kv_heads * a.chunks;
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    timing_mark(true, stream);
    if (p.kv_dtype == GQA_DTYPE_BF16)
        page_append_kernel<BF16><<<(int)blocks, 256, 0, stream>>>(a);
    else
        page_append_kernel<F16><<<(int)blocks, 256, 0, stream>>>(a);
    timing_mark(false, stream);
    return cudaGetLastError();
}

}  // namespace gqa
