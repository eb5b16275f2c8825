// launch.h -- internal launcher declarations (host side); not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "gqa_attn.h"

namespace gqa {

// SM count of the current device (cached per device).
int sm_count();

// Unique id (over the process lifetime) of the calling thread's current context,
// or 0 when there is none or it cannot be had.
unsigned long long current_context_id();

// Runs a set-up step (kernel function attributes, occupancy queries) once per
// device and context, thread-safely: function attributes belong to a device's
// context, so a second device, or the same device after a reset, runs it again.
// While the context id is unavailable the step runs on every call.
struct DeviceSetup {
    static constexpr int kMaxDevices = 64;
    std::mutex mu;
    unsigned long long ctx[kMaxDevices] = {};
    template <class F>
    cudaError_t run(F &&step) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long id = current_context_id();
        if (id != 0 && ctx[dev] == id) return cudaSuccess;
        e = step();
        if (e != cudaSuccess) return e;
        // the step made the device's primary context current if it was not yet
        ctx[dev] = current_context_id();
        return cudaSuccess;
    }
};

// Timing hook: record the start (before=true) or stop event around a
// dominant kernel launch when gqa_timing_enable(1) is in effect.
void timing_mark(bool before, cudaStream_t stream);

// ring.cu
cudaError_t launch_pack_attention(const uint16_t *ring_k, const uint16_t *ring_v,
                                  const float *cur_q, const float *cur_k, const float *cur_v,
                                  const uint32_t *cache_lengths, const uint32_t *write_positions,
                                  uint16_t *packed_q, uint16_t *packed_k, uint16_t *packed_v,
                                  const gqa_ring_params &p, int32_t *status, cudaStream_t stream);
cudaError_t launch_fill_mask(const uint32_t *cache_lengths, uint16_t *mask,
                             const gqa_ring_params &p, int32_t *status, cudaStream_t stream);
cudaError_t launch_commit_kv(const float *new_k, const float *new_v, const uint32_t *commit_counts,
                             const uint32_t *write_positions, uint16_t *ring_k, uint16_t *ring_v,
                             const gqa_ring_params &p, int32_t *status, cudaStream_t stream);
cudaError_t launch_set_mask_rows(const uint16_t *emb, float *hidden, int lanes, int rows,
                                 int width, cudaStream_t stream);

// attn_tc.cu -- masked GQA attention (prefill and verify)
struct AttnProblem {
    const void *q;  // f32 (q_is_f32) or 16-bit of kv_dtype
    bool q_is_f32;
    int64_t q_row_stride, q_head_stride, q_lane_stride;
    const void *k;
    const void *v;
    int kv_dtype;
    int64_t k_row_stride, k_head_stride, v_row_stride, v_head_stride, kv_lane_stride;
    int kv_rows;  // rows addressable in K/V (TMA bounds)
    const uint16_t *mask;
    bool mask_is_bf16;
    int64_t mask_row_stride, mask_head_stride, mask_lane_stride;
    float *o;
    int64_t o_row_stride, o_head_stride, o_lane_stride;
    int lanes, rows, n_heads, n_kv_heads, head_dim, n_keys;
    float scale;
    int32_t *status;
    // ring-direct verify (k, v are the rings; no mask): key tile 0 = the current rows
    bool ring;
    int ring_w;
    const float *cur_k, *cur_v;
    const uint32_t *ring_len, *ring_wp;
};
size_t prefill_workspace_bytes(int rows, int n_heads, int n_kv_heads, int head_dim, int kv_pad);
size_t verify_workspace_bytes(const gqa_ring_params &p);
size_t verify_ring_workspace_bytes(const gqa_ring_params &p);
cudaError_t launch_attention(const AttnProblem &p, void *workspace, cudaStream_t stream);

// append.cu -- page append (new tokens' K/V rows into their page slots)
struct PagedAppendProblem {
    const float *k_new, *v_new;  // [total_tokens][n_kv_heads][head_dim]
    const int32_t *token_offsets, *position_start, *page_table;
    int max_pages_per_seq;
    void *k_pool, *v_pool;
    int kv_dtype;
    int64_t page_stride, token_stride, head_stride;
    int num_seqs, total_tokens, n_kv_heads, head_dim, page_size, num_pages;
    int32_t *status;
};
cudaError_t launch_paged_append(const PagedAppendProblem &p, cudaStream_t stream);

// attn_tc.cu -- chunked prefill over pages (tcgen05 attention, keys gathered from pages)
struct PagedPrefillProblem {
    const float *q;  // [total_tokens][n_heads][head_dim]
    float *o;        // same layout
    const void *k_pool, *v_pool;
    int kv_dtype;
    int64_t page_stride, token_stride, head_stride;
    const int32_t *page_table;
    int max_pages_per_seq;
    const int32_t *token_offsets, *position_start;
    int num_seqs, total_tokens, max_tokens, n_heads, n_kv_heads, head_dim, page_size, num_pages;
    float scale;
    int32_t *status;
};
size_t paged_prefill_workspace_bytes(int num_seqs, int max_tokens, int n_heads, int n_kv_heads,
                                     int head_dim, int max_pages_per_seq, int page_size);
cudaError_t launch_paged_prefill(const PagedPrefillProblem &p, void *workspace, cudaStream_t stream);
void set_attention_pairs(int mode);
cudaError_t launch_bounded_wait_selftest(int32_t *status, int timeout_ms, cudaStream_t stream);

// decode.cu
struct DecodeProblem {
    const float *q;
    const void *k_pool;
    const void *v_pool;
    int kv_dtype;
    int64_t page_stride, token_stride, head_stride;
    const int32_t *page_table;
    int max_pages_per_seq;
    const int32_t *context_lens;
    float *o;
    int num_seqs, n_heads, n_kv_heads, head_dim, page_size, num_pages;
    float scale;
    int32_t *status;
};
size_t decode_workspace_bytes(int num_seqs, int n_heads, int head_dim, int max_pages_per_seq,
                              int page_size);
cudaError_t launch_paged_decode(const DecodeProblem &p, void *workspace, cudaStream_t stream);
// Device address (current device) of the fixed GQA_NOALLOC_SCRATCH_BYTES scratch array.
cudaError_t decode_fixed_scratch(void **ptr);

}  // namespace gqa
