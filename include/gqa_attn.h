/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) grouped-query attention library.
 *
 * What is computed.  Grouped-query attention over a KV cache,
 *     O = softmax(scale * Q K^T + mask) V,
 * evaluated flash-style with an online softmax; each KV head serves a
 * contiguous group of n_heads / n_kv_heads query heads (query head h reads
 * KV head h / (n_heads / n_kv_heads)).  The operations and their layouts
 * restate three pages:
 *   mlx-native 0.18.0, src/ops/flash_attn_prefill_tensor.rs      (prefill)
 *   ferrum-kernels 0.8.3, src/backend/metal/vnext_ops/causal_attention.rs
 *                                                                (paged decode)
 *   mlx-native 0.21.1, src/ops/dflash2_attention_pack.rs         (ring KV)
 *
 * Conventions shared by every entry point.
 *   - Return value: a gqa_status.  Validation happens on the host, before
 *     anything is enqueued; on GQA_INVALID_ARGUMENT nothing was launched and
 *     gqa_last_error() names the offending field.
 *   - Device pointers are owned by the caller; the library never allocates,
 *     frees or retains them.  Every buffer is passed with its size in bytes
 *     so that layouts can be bounds-checked on the host.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  Kernel faults surface at the caller's
 *     next synchronisation.
 *   - Strides are in elements.  Every dimension and stride must fit in int32.
 *   - Counters that live on the device (context lengths, page ids, ring
 *     lengths and positions, commit counts) cannot be checked on the host.
 *     Kernels clamp them into range and OR a GQA_FLAG_* bit into the optional
 *     device word `status` (may be NULL); they never read or write out of
 *     bounds because of them.
 *   - `workspace` is caller-owned device scratch of at least the size the
 *     matching *_workspace_size() function returns (256-byte aligned).  Two
 *     calls that run concurrently must not share a workspace.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *gqa_stream_t;

typedef enum {
    GQA_OK = 0,
    GQA_INVALID_ARGUMENT = 1, /* bad shape, dtype, stride, size or pointer */
    GQA_CUDA_ERROR = 2,       /* a CUDA runtime/driver call failed */
    GQA_DEVICE_TIMEOUT = 3    /* reported through `status` only (GQA_FLAG_TIMEOUT) */
} gqa_status;

typedef enum { GQA_DTYPE_F16 = 1, GQA_DTYPE_BF16 = 2 } gqa_dtype;

/* Bits OR-ed into the device `status` word. */
enum {
    GQA_FLAG_PAGE_CLAMPED = 1,    /* a page id outside [0, num_pages) was clamped */
    GQA_FLAG_CONTEXT_CLAMPED = 2, /* a context length outside [0, max_pages*page_size] */
    GQA_FLAG_RING_CLAMPED = 4,    /* cache_length > window, write_position >= window, or
                                     commit_count outside [0, max_commit] */
    GQA_FLAG_TIMEOUT = 8          /* a bounded pipeline wait gave up; outputs are invalid */
};

/* Thread-local description of the last error on this thread ("" if none). */
const char *gqa_last_error(void);
/* Library version string. */
const char *gqa_version(void);
/* Number of streaming multiprocessors of the current device (0 on error). */
int gqa_device_sm_count(void);

/*
 * Kernel timing for measurement tools (process-wide, not thread-safe).  While
 * enabled, every entry point records a pair of CUDA events on its stream
 * immediately before and after the launch of its dominant kernel (the
 * attention kernel of prefill/verify, the split-KV kernel of paged decode,
 * the single kernel of each ring op).  gqa_timing_last_ms() waits for the
 * most recent pair and returns its elapsed milliseconds, or -1 when nothing
 * was recorded since the last enable.  Returns GQA_CUDA_ERROR if the events
 * cannot be created.
 */
int gqa_timing_enable(int enable);
float gqa_timing_last_ms(void);

/*
 * Diagnostic: launch one thread that waits, with the same bounded mbarrier
 * wait the attention kernel uses, on a barrier nothing ever arrives on.  The
 * wait gives up after timeout_ms (1..10000) and ORs GQA_FLAG_TIMEOUT into the
 * device word `status`; the context stays usable.  Lets callers check the
 * failure path of the bounded waits without faulting or hanging a GPU.
 */
int gqa_selftest_bounded_wait(int32_t *status, int timeout_ms, gqa_stream_t stream);

/*
 * Tiling mode of gqa_attn_prefill (no counterpart on the pages: a choice of
 * this implementation).  A CTA pair runs two query tiles that see the same
 * key tiles (two heads of one KV group, 128 rows each, head_dim 256 or 512,
 * a mask shared by all heads) as one two-CTA cluster whose tensor cores share
 * each K/V tile, so each SM loads half of every K and V tile.
 *   mode 0  never pair
 *   mode 1  pair where it measured faster on GB300: head_dim 256 and 512 (default)
 *   mode 2  pair every eligible shape
 * All modes give the same result up to f32 summation order.  Process-wide,
 * not synchronised with launches in flight on other threads.  Returns
 * GQA_OK, or GQA_INVALID_ARGUMENT for a mode outside 0..2.
 */
int gqa_attn_set_cta_pairs(int mode);

/* ------------------------------------------------------------------------ */
/* Prefill (mlx-native 0.18.0 flash_attn_prefill_tensor.rs: module doc,     */
/* FlashAttnPrefillTensorParams, kv_pad, dispatch_flash_attn_prefill_tensor_f16). */
/* ------------------------------------------------------------------------ */

/* kv_len rounded up to the 64-row cache step. */
uint32_t gqa_kv_pad(uint32_t kv_len);

/* Workspace bytes gqa_attn_prefill needs for this shape (per-tile mask
 * classification and split-KV partial results). */
size_t gqa_attn_prefill_workspace_size(int rows, int n_heads, int n_kv_heads, int head_dim,
                                       int kv_pad);

/*
 * q     f32, element (row i, head h, e) at q[i*q_row_stride + h*q_head_stride + e];
 *       both strides multiples of 4 (16-byte rows).
 * k, v  kv_dtype (f16 or bf16), element (key j, kv head g, e) at
 *       k[j*k_row_stride + g*k_head_stride + e]; strides multiples of 8 and the
 *       base 16-byte aligned (TMA).  Host contract as on the page: every row
 *       below kv_pad is finite; padding rows should be zero and masked.
 * mask  f16 additive mask [rows][kv_pad] (row stride kv_pad), shared by all
 *       heads; -inf hides a key.  Added after scaling.
 * o     f32 [rows][n_heads][head_dim], contiguous.
 * head_dim in {128, 256, 512}; kv_pad a positive multiple of 64;
 * n_heads a multiple of n_kv_heads.  A query row whose mask hides every key
 * produces zeros.
 */
int gqa_attn_prefill(const float *q, size_t q_bytes, int q_row_stride, int q_head_stride,
                     const void *k, size_t k_bytes, int k_row_stride, int k_head_stride,
                     const void *v, size_t v_bytes, int v_row_stride, int v_head_stride,
                     int kv_dtype, const uint16_t *mask, size_t mask_bytes, float *o,
                     size_t o_bytes, int rows, int n_heads, int n_kv_heads, int head_dim,
                     int kv_pad, float scale, void *workspace, size_t workspace_bytes,
                     int32_t *status, gqa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Paged decode (ferrum-kernels 0.8.3 causal_attention.rs: paged_state_regions, */
/* validate_signature, MAXIMUM_HEAD_DIM, the fixed 64 KiB page).             */
/* ------------------------------------------------------------------------ */

size_t gqa_attn_paged_decode_workspace_size(int num_seqs, int n_heads, int head_dim,
                                            int max_pages_per_seq, int page_size);

/*
 * One query token per sequence attends to all context_lens[s] tokens of its
 * sequence.  Token t of sequence s is slot t % page_size of physical page
 * page_table[s*max_pages_per_seq + t/page_size]; its K (and, in the second
 * pool, V) element (kv head g, e) is at
 *     pool[page*page_stride + slot*token_stride + g*head_stride + e].
 * q  f32 [num_seqs][n_heads][head_dim] contiguous; o likewise.
 * k_pages / v_pages  kv_dtype, pool_bytes each (same layout), 16-byte aligned,
 *     strides multiples of 8.  head_dim in {64, 128, 256}.
 * page_table  int32 [num_seqs][max_pages_per_seq]; context_lens int32 [num_seqs].
 * A sequence with context length 0 produces zeros.
 */
int gqa_attn_paged_decode(const float *q, size_t q_bytes, const void *k_pages,
                          const void *v_pages, size_t pool_bytes, int kv_dtype,
                          int64_t page_stride, int64_t token_stride, int64_t head_stride,
                          const int32_t *page_table, size_t page_table_bytes,
                          int max_pages_per_seq, const int32_t *context_lens,
                          size_t context_lens_bytes, float *o, size_t o_bytes, int num_seqs,
                          int n_heads, int n_kv_heads, int head_dim, int page_size,
                          int num_pages, float scale, void *workspace, size_t workspace_bytes,
                          int32_t *status, gqa_stream_t stream);

/*
 * Paged decode without a caller-provided workspace.  (The pages have no
 * counterpart: this entry point exists for callers of this library.)
 *
 * Some callers cannot hand the library a device buffer at the moment they
 * call: a serving engine whose device memory is carved up once at start-up by
 * its own allocator has no spare allocation to give, and real-time callers
 * avoid cudaMalloc / cudaFree because those calls can block the host and
 * synchronise the device.  This variant takes the same arguments as
 * gqa_attn_paged_decode minus the workspace, allocates nothing, and keeps its
 * split-KV partial results in a fixed array of GQA_NOALLOC_SCRATCH_BYTES that
 * lives in the library's device image (every GPU that loads the library holds
 * it until the process exits).
 *   - Problems whose scratch need, gqa_attn_paged_decode_workspace_size(...),
 *     exceeds GQA_NOALLOC_SCRATCH_BYTES are rejected with GQA_INVALID_ARGUMENT.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture.  The address is cached with the identity of the context
 *     it belongs to: after a cudaDeviceReset the next call on that device
 *     looks it up again (make that call, too, outside any capture).
 *   - All calls share the one array and nothing in it needs clearing between
 *     calls, but calls whose work overlaps on the GPU (two streams, or two
 *     threads) race on it: serialise them.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (16u << 20)
int gqa_attn_paged_decode_noalloc(const float *q, size_t q_bytes, const void *k_pages,
                                  const void *v_pages, size_t pool_bytes, int kv_dtype,
                                  int64_t page_stride, int64_t token_stride, int64_t head_stride,
                                  const int32_t *page_table, size_t page_table_bytes,
                                  int max_pages_per_seq, const int32_t *context_lens,
                                  size_t context_lens_bytes, float *o, size_t o_bytes,
                                  int num_seqs, int n_heads, int n_kv_heads, int head_dim,
                                  int page_size, int num_pages, float scale, int32_t *status,
                                  gqa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Page append and chunked prefill over pages (ferrum-kernels 0.8.3          */
/* causal_attention.rs: CausalAttentionParams position_start / tokens,       */
/* dispatch_prepare writing K/V into the paged state, dispatch_attention).    */
/* ------------------------------------------------------------------------ */

/*
 * A batch of new tokens from num_seqs sequences.  Token i of the batch (rows of
 * the [total_tokens][...] arrays) belongs to the sequence s with
 *     token_offsets[s] <= i < token_offsets[s+1]
 * and sits at position p = position_start[s] + (i - token_offsets[s]) of that
 * sequence; position p is slot p % page_size of physical page
 *     page_table[s*max_pages_per_seq + p/page_size]
 * and its K (V) element (kv head g, e) lives at
 *     pool[page*page_stride + slot*token_stride + g*head_stride + e].
 * token_offsets int32 [num_seqs+1] (non-decreasing, token_offsets[0] = 0,
 * token_offsets[num_seqs] <= total_tokens), position_start int32 [num_seqs] and
 * page_table int32 [num_seqs][max_pages_per_seq] are device arrays; out-of-range
 * values are clamped or skipped and flagged (never read or written out of
 * bounds).  Pools: kv_dtype, pool_bytes each, 16-byte aligned, strides positive
 * multiples of 8 elements.
 */

/*
 * Page append: k_new / v_new f32 [total_tokens][n_kv_heads][head_dim]
 * (16-byte aligned, new_bytes each) are rounded to nearest even into kv_dtype
 * and written into every token's slot; no other slot changes.  A token whose
 * position falls outside its page table row, or whose page id is outside
 * [0, num_pages), is not written (GQA_FLAG_PAGE_CLAMPED); inconsistent
 * token_offsets raise GQA_FLAG_CONTEXT_CLAMPED.  head_dim a positive multiple
 * of 8.  Tokens of one call must not share a slot (the order of such writes
 * is undefined).
 */
int gqa_paged_append(const float *k_new, const float *v_new, size_t new_bytes,
                     const int32_t *token_offsets, size_t token_offsets_bytes,
                     const int32_t *position_start, size_t position_start_bytes,
                     const int32_t *page_table, size_t page_table_bytes, int max_pages_per_seq,
                     void *k_pages, void *v_pages, size_t pool_bytes, int kv_dtype,
                     int64_t page_stride, int64_t token_stride, int64_t head_stride, int num_seqs,
                     int total_tokens, int n_kv_heads, int head_dim, int page_size, int num_pages,
                     int32_t *status, gqa_stream_t stream);

size_t gqa_attn_paged_prefill_workspace_size(int num_seqs, int max_tokens, int n_heads,
                                             int n_kv_heads, int head_dim, int max_pages_per_seq,
                                             int page_size);

/*
 * Chunked (multi-token) prefill over pages: query token i of sequence s, at
 * position p, attends to the keys at positions 0..p of its own sequence (the
 * earlier context and the batch's tokens up to itself, which must already be
 * in the pages, e.g. by gqa_paged_append):
 *     o[i][h] = softmax_t(scale * q[i][h] . k_t) v_t,  t = 0..p,
 * KV head h / (n_heads / n_kv_heads).  q, o f32 [total_tokens][n_heads][head_dim]
 * contiguous, 16-byte aligned.  head_dim 128 or 256; page_size a multiple of 8.
 * max_tokens bounds every sequence's token count (rows beyond it are not
 * computed and raise GQA_FLAG_CONTEXT_CLAMPED), as does
 * position_start[s] + tokens <= max_pages_per_seq * page_size.  Rows of o
 * that belong to no sequence are not written.  Out-of-range page ids inside a
 * sequence's context are clamped into the pool (GQA_FLAG_PAGE_CLAMPED).
 */
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
                           gqa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* DFlash2 ring KV (mlx-native 0.21.1 dflash2_attention_pack.rs).           */
/* ------------------------------------------------------------------------ */

/* DFlash2AttentionPackParams: lanes 1..4; q_heads a multiple of kv_heads;
 * head_dim 128 or 256; rows 2..16; window > rows;
 * packed_len == window - 1 + rows; 1 <= max_commit <= rows. */
typedef struct {
    uint32_t lanes, q_heads, kv_heads, head_dim, rows, window, packed_len, max_commit;
} gqa_ring_params;

/* 1 if the geometry is valid, 0 otherwise (message in gqa_last_error()). */
int gqa_ring_params_valid(const gqa_ring_params *p);

/*
 * Pack the verify operands (b lanes, h q_heads, hk kv_heads, d head_dim,
 * r rows, w window, k packed_len; every buffer contiguous, exact size):
 *   ring_k, ring_v        bf16 [b][hk][w][d]
 *   cur_q                 f32  [b][r][h][d]
 *   cur_k, cur_v          f32  [b][r][hk][d]
 *   cache_lengths, write_positions  u32 [b] (device)
 *   packed_q              bf16 [b][h][r][d]  = bf16(cur_q), rounded to nearest even
 *   packed_k, packed_v    bf16 [b][hk][k][d]: column c < r is bf16(cur row c);
 *       column r + j is ring slot (write_position - 1 - j) mod w, copied bit for
 *       bit, when j < cache_length, else zeros.  write_position is the next slot
 *       commit writes, so the history runs newest first.
 */
int gqa_pack_attention(const uint16_t *ring_k, size_t ring_k_bytes, const uint16_t *ring_v,
                       size_t ring_v_bytes, const float *cur_q, size_t cur_q_bytes,
                       const float *cur_k, size_t cur_k_bytes, const float *cur_v,
                       size_t cur_v_bytes, const uint32_t *cache_lengths,
                       size_t cache_lengths_bytes, const uint32_t *write_positions,
                       size_t write_positions_bytes, uint16_t *packed_q, size_t packed_q_bytes,
                       uint16_t *packed_k, size_t packed_k_bytes, uint16_t *packed_v,
                       size_t packed_v_bytes, const gqa_ring_params *p, int32_t *status,
                       gqa_stream_t stream);

/*
 * Additive bf16 mask [b][h][r][k], the same for every head: column c < r is
 * visible (the draft rows see each other); column r + j is visible to row r'
 * when j < cache_length and r' + j + 1 < w (the key lies inside the window of
 * w positions that ends at the query).  Visible 0x0000 (+0), hidden 0xFF80 (-inf).
 */
int gqa_fill_mask(const uint32_t *cache_lengths, size_t cache_lengths_bytes, uint16_t *mask,
                  size_t mask_bytes, const gqa_ring_params *p, int32_t *status,
                  gqa_stream_t stream);

size_t gqa_attn_verify_workspace_size(const gqa_ring_params *p);

/*
 * Verify attention over the packed operands: for lane b and query head h,
 *   O[b][row][h][:] = softmax(scale * packed_q[b][h][row] . packed_k[b][h/g]^T
 *                             + mask[b][h][row]) packed_v[b][h/g]
 * o f32 [b][r][h][d] contiguous.  Rows with no visible key produce zeros.
 */
int gqa_attn_verify(const uint16_t *packed_q, size_t packed_q_bytes, const uint16_t *packed_k,
                    size_t packed_k_bytes, const uint16_t *packed_v, size_t packed_v_bytes,
                    const uint16_t *mask, size_t mask_bytes, float *o, size_t o_bytes,
                    const gqa_ring_params *p, float scale, void *workspace,
                    size_t workspace_bytes, int32_t *status, gqa_stream_t stream);

size_t gqa_attn_verify_ring_workspace_size(const gqa_ring_params *p);

/*
 * Fused ring-direct verify attention (mlx-native 0.21.1 dflash2_attention_pack.rs:
 * the pack and mask dispatchers and the verify attention taken together).  The
 * same result as gqa_pack_attention -> gqa_fill_mask -> gqa_attn_verify, read
 * straight from the ring: the keys of draft row r of lane b are the r current
 * rows (bf16 of cur_k / cur_v, all visible) and every ring slot s whose
 * history index j = (write_position - 1 - s) mod w satisfies
 * j < min(cache_length, w) and r + j + 1 < w; the query is bf16(cur_q).  No
 * packed copy and no mask tensor is made; the counters are read on the device.
 *   ring_k, ring_v   bf16 [b][hk][w][d]
 *   cur_q            f32  [b][r][h][d];  cur_k, cur_v f32 [b][r][hk][d]
 *   cache_lengths, write_positions  u32 [b] (device)
 *   o                f32  [b][r][h][d]
 * Every buffer contiguous with the exact size, rings and current rows 16-byte
 * aligned; workspace as gqa_attn_verify_ring_workspace_size (256-byte aligned).
 */
int gqa_attn_verify_ring(const uint16_t *ring_k, size_t ring_k_bytes, const uint16_t *ring_v,
                         size_t ring_v_bytes, const float *cur_q, size_t cur_q_bytes,
                         const float *cur_k, size_t cur_k_bytes, const float *cur_v,
                         size_t cur_v_bytes, const uint32_t *cache_lengths,
                         size_t cache_lengths_bytes, const uint32_t *write_positions,
                         size_t write_positions_bytes, float *o, size_t o_bytes,
                         const gqa_ring_params *p, float scale, void *workspace,
                         size_t workspace_bytes, int32_t *status, gqa_stream_t stream);

/*
 * Commit accepted rows: for i < min(commit_counts[b], max_commit),
 * ring slot (write_positions[b] + i) mod w of lane b receives bf16(new row i)
 * for every KV head; other slots are untouched.  new_k / new_v f32
 * [b][max_commit][hk][d].  The counters are read-only: the caller advances
 * write_positions and cache_lengths.
 */
int gqa_commit_kv(const float *new_k, size_t new_k_bytes, const float *new_v,
                  size_t new_v_bytes, const uint32_t *commit_counts, size_t commit_counts_bytes,
                  const uint32_t *write_positions, size_t write_positions_bytes,
                  uint16_t *ring_k, size_t ring_k_bytes, uint16_t *ring_v, size_t ring_v_bytes,
                  const gqa_ring_params *p, int32_t *status, gqa_stream_t stream);

/*
 * Draft-input mask rows (dispatch_dflash2_mask_rows_f32): hidden is f32
 * [lanes*rows][width]; in every lane row 0 (the anchor) is kept and rows
 * 1..rows-1 are overwritten with the widened bf16 mask_embedding [width].
 * lanes 1..4, rows 2..16, width > 0.
 */
int gqa_set_mask_rows(const uint16_t *mask_embedding, size_t mask_embedding_bytes,
                      float *hidden, size_t hidden_bytes, uint32_t lanes, uint32_t rows,
                      uint32_t width, gqa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
