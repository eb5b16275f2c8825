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
// 16 bits, for K and for V): one warp per new token, a batch's tokens in one
// wave where they fit (two 8-element chunks a lane per round keep a lane at 58
// registers, so that four blocks of 8 warps fit an SM: 4864 tokens at once on
// 152 SMs).  The lanes take consecutive chunks of the token's row (all KV
// heads), every load of a round issued before the token's slot is looked up,
// so that the lookup's chain of dependent reads (the token's sequence by binary
// search over token_offsets, its start position, its page) is paid once per
// token while its data are in flight.  Reads are coalesced 32-byte pieces;
// each chunk's K and V go out as one 16-byte store each.
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

constexpr int kChunksPerLane = 2;  // chunks a lane moves per round, loads all in flight

template <class KV>
__global__ void __launch_bounds__(256, 4) page_append_kernel(const AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const int warps_per_block = blockDim.x >> 5;
    const int row_chunks = a.n_kv_heads * a.chunks;  // 8-element chunks of a token's row
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int o0 = a.tok_off[0], on = a.tok_off[a.num_seqs];
        if (o0 < 0 || on > a.total_tokens || o0 > on) raise_flag(a.status, GQA_FLAG_CONTEXT_CLAMPED);
    }
    for (int i = blockIdx.x * warps_per_block + (threadIdx.x >> 5); i < a.total_tokens;
         i += gridDim.x * warps_per_block) {
        const float *ksrc = a.k_new + (int64_t)i * row_chunks * 8;
        const float *vsrc = a.v_new + (int64_t)i * row_chunks * 8;
        bool looked_up = false, skip = false;
        int64_t slot_base = 0;  // the token's slot in its page, head 0, column 0
        for (int c0 = 0; c0 < row_chunks; c0 += 32 * kChunksPerLane) {
            float4 k0[kChunksPerLane], k1[kChunksPerLane], v0[kChunksPerLane], v1[kChunksPerLane];
#pragma unroll
            for (int u = 0; u < kChunksPerLane; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < row_chunks) {
                    k0[u] = ld_nc_f4(ksrc + c * 8);
                    k1[u] = ld_nc_f4(ksrc + c * 8 + 4);
                    v0[u] = ld_nc_f4(vsrc + c * 8);
                    v1[u] = ld_nc_f4(vsrc + c * 8 + 4);
                }
            }
            if (!looked_up) {
                looked_up = true;
                // the last sequence s with token_offsets[s] <= i (every lane reads the same
                // offsets)
                int lo = 0, hi = a.num_seqs - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (a.tok_off[mid] <= i)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                const int o0 = a.tok_off[lo];
                if (i < o0 || i >= a.tok_off[lo + 1]) {
                    skip = true;  // the token belongs to no sequence
                } else {
                    const int64_t p = (int64_t)a.pos_start[lo] + (i - o0);
                    const int64_t pi = p >= 0 ? p / a.page_size : -1;
                    const int page =
                        (pi >= 0 && pi < a.max_pages) ? a.page_table[(int64_t)lo * a.max_pages + pi] : -1;
                    if (page < 0 || page >= a.num_pages) {
                        // outside the page table or the pool: not written
                        if (lane == 0) raise_flag(a.status, GQA_FLAG_PAGE_CLAMPED);
                        skip = true;
                    } else {
                        slot_base = (int64_t)page * a.page_stride + (p - pi * a.page_size) * a.token_stride;
                    }
                }
            }
            if (skip) break;
#pragma unroll
            for (int u = 0; u < kChunksPerLane; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < row_chunks) {
                    const int g = c / a.chunks, ch = c - g * a.chunks;
                    const int64_t dst = slot_base + (int64_t)g * a.head_stride + ch * 8;
                    st_v4(a.k_pool + dst, make_uint4(pack2(KV{}, k0[u].x, k0[u].y), pack2(KV{}, k0[u].z, k0[u].w),
                                                     pack2(KV{}, k1[u].x, k1[u].y), pack2(KV{}, k1[u].z, k1[u].w)));
                    st_v4(a.v_pool + dst, make_uint4(pack2(KV{}, v0[u].x, v0[u].y), pack2(KV{}, v0[u].z, v0[u].w),
                                                     pack2(KV{}, v1[u].x, v1[u].y), pack2(KV{}, v1[u].z, v1[u].w)));
                }
            }
        }
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
    // one warp per token, one wave: 4 resident blocks of 8 warps per SM
    int64_t blocks = ((int64_t)p.total_tokens + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 4;
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
