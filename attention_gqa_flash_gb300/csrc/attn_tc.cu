// attn_tc.cu -- masked GQA flash attention on the 5th-generation tensor
// cores (tcgen05): prefill, the speculative-verify attention (over the packed
// copy, or read straight from the ring) and chunked prefill over pages.
//
// What it computes (mlx-native 0.18.0 src/ops/flash_attn_prefill_tensor.rs,
// module doc): O = softmax(scale * Q K^T + mask) V with one KV head per
// n_heads / n_kv_heads query heads and an additive f16 (or bf16) mask; a
// query row whose mask hides every key yields zeros.
//
// Kernel structure: a persistent grid of at most one CTA (or CTA pair) per SM,
// 384 threads each, running units of work (one 128-row query tile, one output
// half, one key split) back to back:
//   warps 0-7  softmax: two threads per query row (warp w and w+4 share the
//              TMEM lanes of rows 32(w%4)..+31, each takes half of the 128
//              columns of a key tile).  They stage Q (f32/bf16 -> f16/bf16),
//              read S from TMEM, apply scale and mask, run the online softmax
//              in the exp2 domain with lazy rescaling of O (only when the row
//              maximum grows by more than 2^8; the two halves agree on the
//              maximum through shared memory), write P over S in TMEM, and
//              finally normalise O and store it (staged, by TMA, where it can).
//   warp 8     TMA producer: builds each unit's list of visible key tiles and
//              streams Q (f32), K and V tiles (128-byte swizzle) through a ring
//              of 32 KiB stages guarded by full/empty mbarriers.
//   warp 9     MMA issuer: owns the TMEM allocation; S = Q K^T into one of two
//              TMEM buffers (the next tile's Q K^T overlaps this tile's
//              softmax), then O += P V with P read from TMEM.
//   warps 10-11 only complete the third warpgroup (register split).
// Key tiles are 128 wide so every MMA has N = 128 (narrower tcgen05 shapes
// run far below the tensor-core rate).  Tiles whose mask is entirely -inf are
// skipped (a classification pre-pass reads the mask once, 64 keys at a time);
// tiles whose mask is entirely zero do not read the mask at all.
// head_dim 512 keeps a 128x512 f32 accumulator out of reach of the 512 TMEM
// columns, so each query tile is processed as two units, one per 256-wide
// half of the output, both recomputing S.
// Few tiles (verify, short chunks) are split along the keys; partial results
// carry a log2-sum-exp and are merged by a combine kernel.
// Three ways of finding the visible keys, one kernel instance each: an
// additive mask tensor (prefill, verify), a ring read directly (fused
// verify), and pages (chunked prefill: ferrum-kernels 0.8.3
// causal_attention.rs, CausalAttentionParams position_start / tokens -- query
// token i of a sequence sits at position position_start + i and sees keys
// 0..position_start + i of its own sequence, gathered from its pages).
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises
// GQA_FLAG_TIMEOUT, unwinds, frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <numeric>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gqa {
namespace {

constexpr int BM = 128;                  // query rows per tile (TMEM lanes)
constexpr int BN = 128;                  // keys per tile
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kProducerWarp = 8, kMmaWarp = 9;  // warps 10 and 11 only complete their warpgroup
constexpr int kThreads = 384;
// Register split: the launch gives every thread the same count (at most 168 with
// three warps per SM sub-partition); the softmax warpgroups then raise theirs so
// that their 64 scores, 32 packed P words and the rest stay in registers, and
// the producer / MMA warpgroup lowers its own.  Sum: 256 x 224 + 128 x 56 = 64512,
// within 384 x 168 = 64512 (checked against the compiled count before launch).
constexpr int kSoftmaxRegs = 224, kControlRegs = 56;
constexpr int kStageBytes = 32768;       // 128 rows x 128 columns of 16-bit, or 128 x 64 f32
constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// key tiles one unit may visit (its list of visible tiles lives in shared
// memory, double-buffered so that the next unit's list is built ahead)
constexpr int kMaxListTiles = 128;
// shared memory left for the Q tile and the ring after barriers, the row-max
// exchange and the two tile lists (the dynamic shared memory base is 1024-aligned)
constexpr int kSmemBudget = 232448 - 256 - 2048 - 2 * 2 * kMaxListTiles;
// how a kernel instance finds the visible keys
constexpr int kMaskMode = 0;   // additive mask tensor, tiles classified by a pre-pass
constexpr int kRingMode = 1;   // ring-direct verify
constexpr int kPagedMode = 2;  // chunked prefill over pages, causal by position

// Per head_dim: KSUB stages per K tile, VSUB per V tile (DO output columns),
// Q in TMEM only at head_dim 128 (at 256 and 512, O and two S buffers fill
// the 512 TMEM columns).
template <int D>
struct Cfg {
    static constexpr int DO = D == 512 ? 256 : D;
    static constexpr int KSUB = D / 128, VSUB = DO / 128;
    static constexpr bool QTM = D == 128;
    static constexpr int QBYTES = QTM ? 0 : BM * D * 2;
    static constexpr int STAGES = (kSmemBudget - QBYTES) / kStageBytes;
    // TMEM columns: O [0, DO), S0/S1 [DO, DO + 256), Q [DO + 256, + D/2)
    static constexpr int kColS = DO, kColQ = DO + 2 * BN;
    static_assert(kColQ + (QTM ? D / 2 : 0) <= 512, "TMEM overflow");
    static_assert(STAGES >= 3, "ring too small");
};

// shared-memory carve-up (offsets from a 1024-byte aligned base)
template <int D>
struct Layout {
    using C = Cfg<D>;
    static constexpr int kQ = 0;                     // D/64 tiles of [128][64] (head_dim >= 256)
    static constexpr int kStages = kQ + C::QBYTES;   // STAGES x 32 KiB
    static constexpr int kBars = kStages + C::STAGES * kStageBytes;
    // barriers: full[S], empty[S], q_full, s_full[2], p_full[2], o_done[2], mma_fin,
    // list_full[2], list_free[2], o_free
    // (+ peer_full[2], peer_free[2]: the unit hand-over of a CTA pair's dynamic queue)
    static constexpr int kNumBars = 2 * C::STAGES + 17;
    static constexpr int kTmemSlot = kBars + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kNumVis = kAbort + 4;     // visible tiles of the unit in each list buffer
    static constexpr int kUid = kNumVis + 8;       // the unit in each list buffer (-1: queue ended)
    static constexpr int kQpos = kUid + 8;         // its queue position (ring-direct verify)
    static constexpr int kPeerUid = kQpos + 8;     // CTA pair, odd CTA: the units the even CTA drew
    static constexpr int kXchg = kPeerUid + 8;     // row-max exchange: [2 tiles][2 halves][128] f32
    static constexpr int kList = kXchg + 2 * 2 * BM * 4;  // two lists of visible key tiles (uint16)
    static constexpr int kEnd = kList + 2 * 2 * kMaxListTiles;
    static constexpr int kBytes = kEnd;
    static_assert(kBytes <= 232448, "shared memory overflow");
};

struct AttnArgs {
    const void *q;
    int q_f32;
    int64_t q_row, q_head, q_lane;
    int kv_bf16;
    int k_rows_dim1, v_rows_dim1;  // tensor map is {d, rows, heads} (1) or {d, heads, rows} (0)
    // prefill tiles of one head and 128 rows move Q (f32) in by TMA
    int q_tma, q_rows_dim1;
    int o_tma, o_rows_dim1;  // O out by TMA (prefill tiles of one head and 128 rows, no key split)
    const uint16_t *mask;
    int mask_bf16;
    int64_t m_row, m_head, m_lane;
    float *o;
    int64_t o_row, o_head, o_lane;
    int lanes, rows, n_heads, n_kv_heads, group, n_keys;
    int rows_per_head, heads_per_tile, row_tiles, head_tiles, tiles_total;
    int n_blk;  // key tiles of BN
    int splits, blk_per_split, d_parts;
    float scale_log2;
    const uint8_t *codes;  // [code groups][code_cols] per 64 keys: 0 skip, 1 no mask, 2 mixed
    int code_cols;
    int shared_mask;  // mask identical for all heads: code group = (lane, row tile)
    float *ws_o;      // split partials [unit][DO / 4][BM] float4 (a warp's rows are adjacent)
    float *ws_lse;    // [unit][BM]
    int32_t *status;
    // ring-direct verify: key tile 0 holds the lane's current rows (converted from
    // f32 in shared memory, padded with zero rows), key tile t >= 1 holds ring slots
    // [128 (t-1), 128 t); visibility comes from the lane's cache length and write
    // position instead of a mask
    int ring, ring_w, ring_r;
    const float *cur_k, *cur_v;           // [lanes][ring_r][n_kv_heads][head_dim]
    // the current rows rounded to bf16 by the pre-pass, [K|V][lanes * n_kv_heads][ring_r]
    // [head_dim]; key tile 0 loads them by TMA (rows ring_r..127 are out of the map's
    // bounds and arrive as zeros)
    uint16_t *cur16;
    int head_dim;
    const uint32_t *ring_len, *ring_wp;   // [lanes]
    // chunked prefill over pages: a unit's lane is a sequence s whose tokens are
    // rows tok_off[s] .. tok_off[s+1]-1 of Q and O (at most `rows` of them), query
    // token i at position pos_start[s] + i; key t of the sequence is slot
    // t % page_size of page page_table[s][t / page_size], K/V by 4-D tensor maps
    // {head_dim, kv heads, page_size, num_pages} in boxes of pg_box slots
    const int32_t *tok_off, *pos_start, *page_table;
    const uint16_t *v_pool;
    int64_t pool_page, pool_token, pool_head;  // element strides
    int total_tokens, max_pages, page_size, num_pages, pg_box;
    int pg_dim[3];  // logical coordinate (0 kv head, 1 slot, 2 page) of map dimensions 1..3
    // dynamic unit queue (unpaired): units in decreasing cost order; each CTA takes
    // the next one from the counter when it starts a unit.  Null counter: the static
    // snake assignment, over the order in sched_perm when there is one (chunked
    // prefill in CTA pairs, whose two CTAs must agree on every unit)
    const int *sched_perm;
    int *sched_counter;
    int pair;  // units are CTA-pair units (for the ordering pass)
    // key splits over the visible tiles (ring-direct verify): every split of a tile
    // scans all key tiles and takes the split-th of `splits` equal shares of the
    // visible ones, instead of a fixed range of tiles
    int vis_split;
    // ring-direct verify with splits over the visible tiles: the pre-pass gives lane l
    // lane_splits[l] of the `splits` split slots, in proportion to its visible tiles
    // (split_budget of them per query tile in all, about one unit per SM), and queues
    // the lanes' units in blocks, the lane with the most tiles per split first: lane l's
    // block starts at lane_start[l] and holds, for each of its query tiles in order,
    // its splits in order.  A unit's partial result goes to slot = its queue position.
    int *lane_splits, *lane_start, *queue_len;
    int split_budget;
};

// A sequence's tokens and start position as read from the device counters,
// clamped so that every access stays in bounds: rows [t0, t0 + ntok) of Q and O,
// positions ps .. ps + ntok - 1, keys below ps + ntok <= max_pages * page_size.
struct SeqSpan {
    int t0, ntok, ps;
};
__device__ __forceinline__ SeqSpan seq_span(const AttnArgs &a, int s, bool flag) {
    const int cap = a.max_pages * a.page_size;
    const int o0 = a.tok_off[s], o1 = a.tok_off[s + 1], ps = a.pos_start[s];
    SeqSpan q;
    q.t0 = min(max(o0, 0), a.total_tokens);
    const int t1 = min(max(o1, q.t0), a.total_tokens);
    q.ps = min(max(ps, 0), cap);
    q.ntok = min(min(t1 - q.t0, a.rows), cap - q.ps);
    if (flag && (q.t0 != o0 || t1 != o1 || q.ps != ps || q.ntok != o1 - o0))
        raise_flag(a.status, GQA_FLAG_CONTEXT_CLAMPED);
    return q;
}

// physical page of key t of sequence s (t below the sequence's context),
// clamped into the pool
__device__ __forceinline__ int page_of(const AttnArgs &a, int s, int t) {
    int page = a.page_table[(int64_t)s * a.max_pages + t / a.page_size];
    if (page < 0 || page >= a.num_pages) {
        raise_flag(a.status, GQA_FLAG_PAGE_CLAMPED);
        page = page < 0 ? 0 : a.num_pages - 1;
    }
    return page;
}

// number of slots of [a, b) inside the circular range of `len` slots that starts at
// `start` in a ring of w slots
__device__ __forceinline__ int circ_overlap(int a, int b, int start, int len, int w) {
    if (len <= 0) return 0;
    auto lin = [](int a0, int b0, int a1, int b1) { return max(0, min(b0, b1) - max(a0, a1)); };
    if (start + len <= w) return lin(a, b, start, start + len);
    return lin(a, b, start, w) + lin(a, b, 0, start + len - w);
}

// Ring-direct verify: code of key tile t (0 skip, 1 every key visible to every
// row, 2 mixed) for a lane with history length L (clamped to the window) and
// write position wp (mod the window).  History index j = (wp - 1 - slot) mod w
// is visible to draft row r when j < L and r + j + 1 < w: the slots seen by row 0
// are the L' = min(L, w - 1) newest, those seen by every row the min(L, w - rows)
// newest, each a circular range ending at slot wp - 1.
// (0 <= L <= w and 0 <= wp < w, so a range's first slot wp - len is above -w.)
__device__ __forceinline__ int ring_tile_code(const AttnArgs &a, int t, int L, int wp) {
    if (t == 0) return 2;  // current rows, then padding
    const int w = a.ring_w, s0 = (t - 1) * BN, s1 = min(s0 + BN, w);
    const int l_any = min(L, w - 1), l_all = max(0, min(L, w - a.ring_r));
    auto first = [&](int len) { return wp - len + (wp < len ? w : 0); };
    const int any = circ_overlap(s0, s1, first(l_any), l_any, w);
    if (any == 0) return 0;
    const int all = circ_overlap(s0, s1, first(l_all), l_all, w);
    return all == BN ? 1 : 2;
}

struct Tile {
    int lane, kh, ht, rt;
};

__device__ __forceinline__ Tile tile_of(const AttnArgs &a, int tile_id) {
    Tile t;
    t.ht = tile_id % a.head_tiles;
    tile_id /= a.head_tiles;
    t.kh = tile_id % a.n_kv_heads;
    tile_id /= a.n_kv_heads;
    t.lane = tile_id % a.lanes;
    t.rt = tile_id / a.lanes;
    return t;
}

// (head, row) of tile row i; false when the tile row carries no query
__device__ __forceinline__ bool row_of(const AttnArgs &a, const Tile &t, int i, int &head,
                                       int &row) {
    const int hi = i / a.rows_per_head;
    const int ri = i - hi * a.rows_per_head;
    const int hg = t.ht * a.heads_per_tile + hi;
    row = t.rt * a.rows_per_head + ri;
    head = t.kh * a.group + hg;
    return hi < a.heads_per_tile && hg < a.group && row < a.rows;
}

__device__ __forceinline__ int code_group(const AttnArgs &a, const Tile &t) {
    if (a.shared_mask) return t.lane * a.row_tiles + t.rt;
    return ((t.lane * a.n_kv_heads + t.kh) * a.head_tiles + t.ht) * a.row_tiles + t.rt;
}

// code of key tile j (BN keys = two classification blocks of 64); a tile that
// mixes skipped and mask-free blocks still has to apply the mask
__device__ __forceinline__ int tile_code(const AttnArgs &a, int cg, int j) {
    int all_skip = 1, all_free = 1;
#pragma unroll
    for (int s = 0; s < BN / 64; ++s) {
        const int c = j * (BN / 64) + s;
        const int v = c < a.code_cols ? a.codes[(int64_t)cg * a.code_cols + c] : 0;
        all_skip &= (v == 0);
        all_free &= (v == 1);
    }
    return all_skip ? 0 : (all_free ? 1 : 2);
}

__device__ __forceinline__ bool is_neg_inf(uint16_t v, int bf16) {
    return bf16 ? v == 0xff80 : v == 0xfc00;
}
__device__ __forceinline__ float mask_to_f32(uint16_t v, int bf16) {
    return bf16 ? __uint_as_float((uint32_t)v << 16) : __half2float(__ushort_as_half(v));
}

// ---------------------------------------------------------------------------
// classification pre-pass: one CTA per (code group, 64 keys), thread = tile row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(BM) classify_kernel(const AttnArgs a, uint8_t *codes) {
    tc::griddep_launch_dependents();  // the attention kernel may start its set-up now
    const int cg = blockIdx.x, cb = blockIdx.y;
    Tile t;
    if (a.shared_mask) {
        t.lane = cg / a.row_tiles;
        t.rt = cg - t.lane * a.row_tiles;
        t.kh = 0;
        t.ht = 0;
    } else {
        t.rt = cg % a.row_tiles;
        int rest = cg / a.row_tiles;
        t.ht = rest % a.head_tiles;
        rest /= a.head_tiles;
        t.kh = rest % a.n_kv_heads;
        t.lane = rest / a.n_kv_heads;
    }
    int head, row;
    const bool valid = row_of(a, t, threadIdx.x, head, row);
    int masked = 1, zero = 1;
    if (valid) {
        const uint16_t *m = a.mask + t.lane * a.m_lane + (int64_t)head * a.m_head +
                            (int64_t)row * a.m_row + (int64_t)cb * 64;
        const int ncol = min(64, a.n_keys - cb * 64);
        if (ncol < 64) zero = 0;
        if ((reinterpret_cast<uintptr_t>(m) & 15) == 0 && ncol == 64) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 x = ld_nc_v4(m + v * 8);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint16_t lo = w[e] & 0xffff, hi = w[e] >> 16;
                    masked &= is_neg_inf(lo, a.mask_bf16) & is_neg_inf(hi, a.mask_bf16);
                    zero &= ((lo & 0x7fff) == 0) & ((hi & 0x7fff) == 0);
                }
            }
        } else {
            for (int c = 0; c < ncol; ++c) {
                const uint16_t v = m[c];
                masked &= is_neg_inf(v, a.mask_bf16);
                zero &= (v & 0x7fff) == 0;
            }
        }
    }
    const int all_masked = __syncthreads_and(masked);
    const int all_zero = __syncthreads_and(zero);
    if (threadIdx.x == 0)
        codes[(int64_t)cg * a.code_cols + cb] = all_masked ? 0 : (all_zero ? 1 : 2);
}

// Bounded mbarrier wait shared by all roles of a CTA: gives up after
// kWaitLimitNs (raising GQA_FLAG_TIMEOUT and the CTA's abort flag) or as soon
// as another role of the CTA has aborted.
struct Waiter {
    volatile int *abort;
    int32_t *status;
    uint64_t limit_ns;
    bool honour_abort = true;  // false: only the time limit ends the wait
    // CLUSTER: poll without suspending, acquire at cluster scope (phases completed
    // by the other CTA of a pair)
    template <bool CLUSTER = false>
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        auto try_once = [&]() {
            return CLUSTER ? tc::mbar_test_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity);
        };
        if (try_once()) return true;
        const uint64_t t0 = tc::globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            if (try_once()) return true;
            if ((it & 127) == 0) {
                if (honour_abort && *abort) return false;
                if (tc::globaltimer_ns() - t0 > limit_ns) {
                    *abort = 1;
                    raise_flag(status, GQA_FLAG_TIMEOUT);
                    return false;
                }
            }
        }
    }
};

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on; the wait must give up after limit_ns and raise GQA_FLAG_TIMEOUT.
__global__ void bounded_wait_selftest_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    tc::mbar_init(b, 1);
    tc::fence_mbar_init();
    abort_flag = 0;
    const Waiter wt{&abort_flag, status, limit_ns};
    wt.wait(b, 0);
}

// byte offset of the 16-byte chunk `c16` of row `r` in a [128][64] 16-bit tile
// written with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int c16) {
    return (uint32_t)(r * 128 + ((c16 ^ (r & 7)) << 4));
}


// One unit of work: a query tile (one head's 128 rows for prefill, a KV group's
// heads for verify), one output half (head_dim 512) and one key split.
struct Unit {
    Tile t;
    int tile_id, dpart, split, cg, jb, je, d_off, head_idx, q_head0, q_row0;
    int t0, ntok, ps;  // chunked prefill: the sequence's span (else 0, rows, 0)
};

// Unit u of the heavy-first order (row tiles from the last, which see the most
// keys under a causal mask).  PAIR: u counts pairs of head tiles 2p, 2p + 1 of
// one (lane, KV head, row tile); `rank` picks this CTA's tile of the pair.
__device__ __forceinline__ Unit unit_of(const AttnArgs &a, int u, bool pair, uint32_t rank, int d_out) {
    Unit n;
    n.split = u % a.splits;
    u /= a.splits;
    n.dpart = u % a.d_parts;
    u /= a.d_parts;
    const int hts = pair ? a.head_tiles / 2 : a.head_tiles;
    const int per_rt = a.lanes * a.n_kv_heads * hts;
    const int pidx = (a.row_tiles - 1 - u / per_rt) * per_rt + u % per_rt;
    n.tile_id = pair ? (pidx / hts) * a.head_tiles + (pidx % hts) * 2 + (int)rank : pidx;
    n.t = tile_of(a, n.tile_id);
    n.cg = code_group(a, n.t);
    n.d_off = n.dpart * d_out;
    n.jb = a.vis_split ? 0 : n.split * a.blk_per_split;
    n.je = a.vis_split ? a.n_blk : min(a.n_blk, n.jb + a.blk_per_split);
    n.head_idx = n.t.lane * a.n_kv_heads + n.t.kh;
    n.q_head0 = n.t.kh * a.group + n.t.ht * a.heads_per_tile;
    n.q_row0 = n.t.rt * a.rows_per_head;
    n.t0 = 0;
    n.ntok = a.rows;
    n.ps = 0;
    return n;
}

__device__ __forceinline__ void set_span(const AttnArgs &a, Unit &n, bool flag) {
    const SeqSpan q = seq_span(a, n.t.lane, flag);
    n.t0 = q.t0;
    n.ntok = q.ntok;
    n.ps = q.ps;
}

// Chunked prefill: code of key tile j for a unit (0 skip, 1 visible to every
// row, 2 mixed).  The unit's rows are tokens r0 .. r0 + rows_per_head - 1 of its
// sequence (those below ntok carry a query), at positions ps + row.
__device__ __forceinline__ int paged_tile_code(const AttnArgs &a, const Unit &n, int j) {
    const int r0 = n.q_row0;
    if (r0 >= n.ntok) return 0;
    const int p0 = n.ps + r0, p1 = n.ps + min(r0 + a.rows_per_head, n.ntok) - 1;
    const int k0 = j * BN;
    if (k0 > p1) return 0;
    return k0 + BN - 1 <= p0 ? 1 : 2;
}

// Chunked prefill: visible key tiles of unit u, plus one for the unit's own overhead
// when it has any (the scheduling cost), capped at kCostBins - 1.
constexpr int kCostBins = 1024;
constexpr int kMaxQueueGroups = 10240;  // (sequence, KV head) groups the ordering pass handles (40 KiB)
__device__ __forceinline__ int paged_unit_cost(const AttnArgs &a, int u) {
    Unit un = unit_of(a, u, a.pair != 0, 0, 0);
    set_span(a, un, false);
    if (un.q_row0 >= un.ntok) return 0;
    const int p1 = un.ps + min(un.q_row0 + a.rows_per_head, un.ntok) - 1;
    const int n = max(0, min(un.je, p1 / BN + 1) - un.jb);
    return min(n + (n > 0 ? 1 : 0), kCostBins - 1);
}

// Unit j of group g = (sequence, KV head) in the queue order: row tiles from the
// last (the most keys), then head tiles (pairs of them for CTA-pair units), output
// halves and key splits.  This inverts unit_of's numbering.
__device__ __forceinline__ int unit_in_group(const AttnArgs &a, int g, int j) {
    const int split = j % a.splits;
    j /= a.splits;
    const int dpart = j % a.d_parts;
    j /= a.d_parts;
    const int hts = a.pair ? a.head_tiles / 2 : a.head_tiles;
    const int ht = j % hts;
    const int rt = a.row_tiles - 1 - j / hts;
    const int per_rt = a.lanes * a.n_kv_heads * hts;
    const int ut = (a.row_tiles - 1 - rt) * per_rt + g * hts + ht;
    return (ut * a.d_parts + dpart) * a.splits + split;
}

// Pre-pass of the dynamic unit queue (CTAs of 1024 threads), then the queue counter
// reset for the attention launch that follows.
//   CTA 0, chunked prefill: the queue order.  The units of one (sequence, KV head)
//     group read the same keys and values, so they are queued together (and run at
//     the same time, sharing those bytes through L2); groups go in decreasing order
//     of their mean unit cost (counting sort), so that the queue ends with the light
//     ones.  Dynamic shared memory: one int per group.
//   CTAs 1.., ring-direct verify: the current K and V rows rounded to bf16 for the
//     tensor map of key tile 0.
__global__ void __launch_bounds__(1024) order_units_kernel(const AttnArgs a, int units) {
    __shared__ int bins[kCostBins];
    __shared__ int wsum[32];
    extern __shared__ int gval[];  // group cost, then the group's place in the queue
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    tc::griddep_launch_dependents();  // the attention kernel may start its set-up now
    if (blockIdx.x > 0) {
        // ring-direct verify: the current K and V rows rounded to bf16 (8 per thread step)
        const int cpr = a.head_dim / 8;
        const int64_t per = (int64_t)a.lanes * a.ring_r * a.n_kv_heads * cpr;
        for (int64_t i = (int64_t)(blockIdx.x - 1) * 1024 + t; i < 2 * per; i += (int64_t)(gridDim.x - 1) * 1024) {
            const int which = (int)(i / per);
            int64_t r = i - which * per;
            const int ch = (int)(r % cpr);
            r /= cpr;
            const int g = (int)(r % a.n_kv_heads);
            r /= a.n_kv_heads;
            const int row = (int)(r % a.ring_r), ln = (int)(r / a.ring_r);
            const float *src = (which ? a.cur_v : a.cur_k) +
                               (((int64_t)ln * a.ring_r + row) * a.n_kv_heads + g) * a.head_dim + ch * 8;
            const float4 x = ld_nc_f4(src), y = ld_nc_f4(src + 4);
            uint16_t *dst = a.cur16 + (((which * (int64_t)a.lanes + ln) * a.n_kv_heads + g) * a.ring_r + row) *
                                          a.head_dim + ch * 8;
            st_v4(dst, make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y),
                                  pack_bf16x2(y.z, y.w)));
        }
        return;
    }
    if (a.lane_start) return;  // ring-direct verify: the attention kernel works out its plan
    if (!a.sched_perm) return;
    const int groups = a.lanes * a.n_kv_heads, per_group = units / groups;
    bins[t] = 0;
    for (int g = t; g < groups; g += 1024) gval[g] = 0;
    __syncthreads();
    for (int u = t; u < units; u += 1024) {
        const Unit un = unit_of(a, u, a.pair != 0, 0, 0);
        atomicAdd(&gval[un.t.lane * a.n_kv_heads + un.t.kh], paged_unit_cost(a, u));
    }
    __syncthreads();
    for (int g = t; g < groups; g += 1024) {
        gval[g] = min((gval[g] + per_group - 1) / per_group, kCostBins - 1);
        atomicAdd(&bins[gval[g]], 1);
    }
    __syncthreads();
    // thread t takes key c = kCostBins - 1 - t; start[c] = groups with a larger key
    const int c = kCostBins - 1 - t;
    const int v = bins[c];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const int start = x - v + (warp > 0 ? wsum[warp - 1] : 0);
    __syncthreads();
    bins[c] = start;
    __syncthreads();
    for (int g = t; g < groups; g += 1024) gval[g] = atomicAdd(&bins[gval[g]], 1);
    __syncthreads();
    int *perm = const_cast<int *>(a.sched_perm);
    for (int i = t; i < units; i += 1024) {
        const int g = i / per_group, j = i - g * per_group;
        perm[gval[g] * per_group + j] = unit_in_group(a, g, j);
    }
    if (t == 0 && a.sched_counter) *a.sched_counter = 0;
}

// The k-th unit of work slot `slot` of `slots` (a slot is a CTA, or a CTA pair):
// slots take the heavy-first units in snake order (0..S-1, then S-1..0, ...), so
// that each slot's total work is close to the mean; -1 when the slot is done.
__device__ __forceinline__ int slot_unit(int k, int slot, int slots, int units) {
    const int u = k * slots + ((k & 1) ? slots - 1 - slot : slot);
    return u < units ? u : -1;
}

// Persistent tcgen05 attention: each CTA (or CTA pair) owns a TMEM allocation,
// its barriers and its ring for the whole launch and runs the units of its slot
// back to back.  The producer builds the next unit's tile list and prefetches
// its Q and K/V while the current unit finishes; the softmax warps convert the
// next unit's Q before writing the current unit's O, so that the next unit's
// first Q.K^T products overlap that epilogue.  Ring positions and the phases of
// the S / P / O barriers continue across units.
//
// PAIR: the two CTAs of a cluster process two query tiles (two heads of one KV
// group, same rows, same visible key tiles) with one 256-row MMA per step
// (cta_group::2).  Each CTA loads only half of every K tile (64 of its keys) and
// half of every V tile (half of the output columns), so the K/V bytes an SM takes
// in per tile are halved; the even CTA issues all MMAs.
template <int D, class KV, bool PAIR, int MODE = kMaskMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmv1) {
    using C = Cfg<D>;
    using L = Layout<D>;
    constexpr int DO = C::DO, KSUB = C::KSUB, VSUB = C::VSUB, NS = C::STAGES;
    constexpr bool kBf16 = KV::kind == GQA_DTYPE_BF16;
    constexpr int kQStages = D / 64;  // an f32 Q tile crosses the ring 64 columns per stage
    static_assert(!PAIR || D >= 256, "CTA pairs stage Q in shared memory (head_dim >= 256)");
    constexpr bool RING = MODE == kRingMode, PAGED = MODE == kPagedMode;
    static_assert(!(PAIR && MODE == kRingMode), "ring-direct verify runs unpaired");
    static_assert(!(PAIR && MODE == kPagedMode && D != 256), "chunked prefill pairs at head_dim 256");
    // ring stages per K and per V tile (PAIR: one stage holds this CTA's 64 keys x
    // 256 columns of K, or its 128 keys x 128 output columns of V)
    constexpr int KST = PAIR ? D / 256 : KSUB;
    constexpr int VST = PAIR ? 1 : VSUB;

    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
    auto full = [&](int s) { return bar(s); };
    auto empty = [&](int s) { return bar(NS + s); };
    const uint32_t q_full = bar(2 * NS);
    auto s_full = [&](int b) { return bar(2 * NS + 1 + b); };
    auto p_full = [&](int b) { return bar(2 * NS + 3 + b); };
    auto o_done = [&](int b) { return bar(2 * NS + 5 + b); };
    const uint32_t mma_fin = bar(2 * NS + 7);
    auto list_full = [&](int b) { return bar(2 * NS + 8 + b); };
    auto list_free = [&](int b) { return bar(2 * NS + 10 + b); };
    const uint32_t o_free = bar(2 * NS + 12);
    // CTA pair with a dynamic queue: the even CTA draws each unit and hands it to the odd
    // CTA (peer_full, in the odd CTA), which gives the slot back (peer_free, in the even)
    auto peer_full = [&](int b) { return bar(2 * NS + 13 + b); };
    auto peer_free = [&](int b) { return bar(2 * NS + 15 + b); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::kTmemSlot);
    volatile int *n_vis_smem = reinterpret_cast<volatile int *>(smem + L::kNumVis);
    volatile int *uid_smem = reinterpret_cast<volatile int *>(smem + L::kUid);
    volatile int *qpos_smem = reinterpret_cast<volatile int *>(smem + L::kQpos);
    float *xchg = reinterpret_cast<float *>(smem + L::kXchg);
    uint16_t *lists = reinterpret_cast<uint16_t *>(smem + L::kList);
    const Waiter wt{abort_flag, a.status, kWaitLimitNs};
    // the swizzled layouts below assume a 1024-byte aligned shared-memory base
    if (sbase & 1023u) {
        if (threadIdx.x == 0) raise_flag(a.status, GQA_FLAG_TIMEOUT);
        return;
    }

    const uint32_t rank = PAIR ? (blockIdx.x & 1u) : 0u;
    const int slot = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int slots = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int units = a.tiles_total * a.d_parts * a.splits / (PAIR ? 2 : 1);
    // ring positions taken by one unit's loads: Q (f32, by TMA) and K, V of every visible tile
    const int q_pos = a.q_tma ? kQStages : 0;
    auto unit_positions = [&](int nv) { return q_pos + nv * (KST + VST); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        // PAIR: a stage is free again only once both CTAs are done with it (each
        // CTA's softmax releases its Q stages in both CTAs; the MMA releases K/V
        // stages with two commits), so that the odd CTA's loads, which complete on
        // the even CTA's full barrier, never land in a phase of the even CTA's own
        // Q load
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), PAIR ? 2 : 1);
        }
        // PAIR: one arrival per softmax warp of both CTAs, on the even CTA's barrier
        tc::mbar_init(q_full, PAIR ? 2 * kSoftmaxWarps : kSoftmaxThreads);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(s_full(b), 1);
            // one arrival per softmax warp; the even CTA's barrier also takes the odd
            // CTA's relayed arrival
            tc::mbar_init(p_full(b), PAIR ? kSoftmaxWarps + (rank == 0 ? 1 : 0) : kSoftmaxThreads);
            tc::mbar_init(o_done(b), 1);
            tc::mbar_init(list_full(b), 1);
            // softmax warps + the MMA issuer (even CTA) or the relay (odd CTA)
            tc::mbar_init(list_free(b), kSoftmaxWarps + 1);
        }
        tc::mbar_init(mma_fin, 1);
        tc::mbar_init(o_free, kSoftmaxWarps + ((PAIR && rank == 0) ? 1 : 0));
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(peer_full(b), 1);
            tc::mbar_init(peer_free(b), 1);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        if constexpr (PAIR) {
            tc::tmem_alloc_pair<512>(smem_u32(tslot));
            tc::tmem_relinquish_pair();
        } else {
            tc::tmem_alloc<512>(smem_u32(tslot));
            tc::tmem_relinquish();
        }
    }
    tc::tc_fence_before();
    if constexpr (PAIR)
        tc::cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
    else
        __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tm_o = tmem;             // O: DO columns
    const uint32_t tm_s = tmem + C::kColS;  // S: two buffers of BN columns (P over S)
    const uint32_t tm_q = tmem + C::kColQ;  // Q: D/2 columns (head_dim 128)

    // Register split per warpgroup (every warp of a warpgroup executes its
    // setmaxnreg): warps 8-11 (producer, MMA issuer, two idle) lower theirs, the
    // softmax warpgroups raise theirs.
    if (warp >= kSoftmaxWarps) {
        tc::setmaxnreg_dec<kControlRegs>();
        if (warp == kProducerWarp) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                tc::prefetch_tmap(&tmk);
                tc::prefetch_tmap(&tmv);
                if (a.q_tma) tc::prefetch_tmap(&tmq);
            }
            int stage = 0;
            uint32_t round = 0;
            auto next = [&]() {
                if (++stage == NS) {
                    stage = 0;
                    ++round;
                }
            };
            bool ok = true;
            // while the pre-pass runs: the first unit's f32 Q into L2 (its rows and heads do
            // not depend on the pre-pass when the units are assigned statically)
            if (!a.sched_counter && !a.sched_perm && a.q_tma && lane == 0 && !RING) {
                const int uid0 = slot_unit(0, slot, slots, units);
                if (uid0 >= 0) {
                    Unit u0 = unit_of(a, uid0, PAIR, rank, DO);
                    if constexpr (PAGED) set_span(a, u0, false);
                    for (int qs = 0; qs < kQStages; ++qs)
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx)
                            tc::tma_prefetch_3d(&tmq, qs * 64 + bx * 32,
                                                a.q_rows_dim1 ? u0.t0 + u0.q_row0 : u0.q_head0,
                                                a.q_rows_dim1 ? u0.q_head0 : u0.t0 + u0.q_row0);
                }
            }
            // ring-direct verify with a split plan: only key tile 0 (the current rows, which
            // the pre-pass rounds to bf16) depends on the pre-pass; the plan is worked out
            // here and everything else is loaded without waiting for it
            const bool ring_plan = RING && a.lane_start;
            bool prepass_done = !ring_plan;
            // the pre-pass (tile classes, or the unit queue) is complete and visible from
            // here on
            if (!ring_plan) tc::griddep_wait();
            int qlen = a.queue_len ? *a.queue_len : units;
            // ring-direct verify: every lane's history length, write position, split count
            // and queue block, lane l holding lane l's (at most 32 lanes this way)
            uint32_t my_rl = 0, my_rp = 0;
            int my_ls = a.splits, my_start = 0;
            if (RING && a.lanes <= 32 && lane < a.lanes) {
                my_rl = a.ring_len[lane];
                my_rp = a.ring_wp[lane];
            }
            if (ring_plan) {
                // Lane l gets S_l = ceil(vis_l / C) of the split slots, C the least cost (key
                // tiles per unit) for which they add up to at most split_budget (no lane
                // takes more than `splits`); its block of units (kv head major, head tile,
                // split) follows the blocks of the lanes with dearer units.
                // visible tiles of lane l (on lane l): key tile 0, and the ring tiles that
                // meet the circular range of its min(L, w - 1) newest slots (the range
                // ring_tile_code tests), counted in closed form
                int vis = 0;
                if (lane < a.lanes) {
                    const int w = a.ring_w;
                    const int la = min((int)min(my_rl, (uint32_t)w), w - 1);
                    const int wp = (int)(my_rp % (uint32_t)w);
                    vis = 1;
                    if (la > 0) {
                        int st = wp - la;
                        if (st >= 0) {
                            vis += (wp - 1) / BN - st / BN + 1;
                        } else {
                            st += w;
                            vis += (w + BN - 1) / BN - st / BN;  // slots [st, w)
                            if (wp > 0) vis += (wp - 1) / BN + 1 - ((wp - 1) / BN == st / BN ? 1 : 0);
                        }
                    }
                }
                auto warp_max = [](int v) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
                    return v;
                };
                // split slots the lanes take at cost C: the sum of ceil(vis_l / C)
                auto need = [&](int C) {
                    int t = 0;
                    for (int l = 0; l < a.lanes; ++l) {
                        const int v = __shfl_sync(0xffffffffu, vis, l);
                        t += (v + C - 1) / C;
                    }
                    return t;
                };
                // the least feasible C in [lo, hi] (need is non-increasing in C; hi when
                // none is), 32 candidates per pass
                int lo = max(warp_max((vis + a.splits - 1) / a.splits), 1), hi = max(warp_max(vis), lo);
                while (lo < hi) {
                    const int step = (hi - lo + 31) / 32;
                    const unsigned fit = __ballot_sync(0xffffffffu, need(min(lo + lane * step, hi)) <= a.split_budget);
                    if (!fit) {
                        lo = min(lo + 31 * step + 1, hi);  // none of the candidates fits
                        continue;
                    }
                    const int f = __ffs(fit) - 1;
                    const int cf = min(lo + f * step, hi);
                    if (step == 1 || f == 0) {
                        lo = hi = cf;
                        break;
                    }
                    lo = lo + (f - 1) * step + 1;  // C_{f-1} does not fit
                    hi = cf;
                }
                int S = 0, cost = -1;
                if (lane < a.lanes) {
                    S = max((vis + lo - 1) / lo, 1);
                    cost = (vis + S - 1) / S;
                }
                const int cnt = lane < a.lanes ? S * a.n_kv_heads * a.head_tiles : 0;
                int start = 0;
                for (int l = 0; l < a.lanes; ++l) {
                    const int cl = __shfl_sync(0xffffffffu, cost, l), nl = __shfl_sync(0xffffffffu, cnt, l);
                    if (cl > cost || (cl == cost && l < lane)) start += nl;
                }
                int sum = cnt;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                my_ls = S;
                my_start = start;
                qlen = sum;
                // the split combine reads the plan after this launch
                if (blockIdx.x == 0 && lane < a.lanes) {
                    a.lane_splits[lane] = S;
                    a.lane_start[lane] = start;
                }
            }
            for (int k = 0; ok; ++k) {
                int uid;
                int qpos = -1;
                if (a.sched_counter) {
                    int idx = 0;
                    if (ring_plan) {
                        // the plan gives every CTA its queue positions (about one unit each)
                        idx = (int)blockIdx.x + k * (int)gridDim.x;
                    } else if (PAIR) {
                        // the even CTA draws the unit and hands it to the odd CTA; the hand-over
                        // slot k & 1 is reused once the odd CTA has read unit k - 2 from it
                        volatile int *peer_uid = reinterpret_cast<volatile int *>(smem + L::kPeerUid);
                        const int pb = k & 1;
                        bool hw = true;
                        if (lane == 0) {
                            if (rank == 0) {
                                if (k >= 2) hw = wt.template wait<true>(peer_free(pb), ((k - 2) >> 1) & 1);
                                idx = hw ? atomicAdd(a.sched_counter, 1) : 0x7fffffff;
                                tc::st_shared_cluster_u32(tc::mapa_shared(smem_u32((const void *)(peer_uid + pb)), 1),
                                                          (uint32_t)idx);
                                tc::mbar_arrive_cluster(tc::mapa_shared(peer_full(pb), 1));
                            } else {
                                hw = wt.template wait<true>(peer_full(pb), (k >> 1) & 1);
                                idx = hw ? peer_uid[pb] : 0x7fffffff;
                                tc::mbar_arrive_cluster(tc::mapa_shared(peer_free(pb), 0));  // after the read
                            }
                        }
                        idx = __shfl_sync(0xffffffffu, idx, 0);
                    } else {
                        if (lane == 0) idx = atomicAdd(a.sched_counter, 1);
                        idx = __shfl_sync(0xffffffffu, idx, 0);
                    }
                    qpos = idx;
                    if (RING && a.lane_start) {
                        // the lane whose block holds queue position idx; then its query
                        // tile and split
                        const int per_lane = my_ls * a.n_kv_heads * a.head_tiles;
                        const unsigned own = __ballot_sync(
                            0xffffffffu, lane < a.lanes && idx >= my_start && idx < my_start + per_lane);
                        uid = -1;
                        if (own && idx < qlen) {
                            const int o = __ffs(own) - 1;
                            const int S = __shfl_sync(0xffffffffu, my_ls, o);
                            const int rem = idx - __shfl_sync(0xffffffffu, my_start, o);
                            const int tile_in_lane = rem / S;  // kv head major, head tile minor
                            uid = (o * a.n_kv_heads * a.head_tiles + tile_in_lane) * a.splits + (rem - tile_in_lane * S);
                        }
                    } else {
                        uid = idx < qlen ? a.sched_perm[idx] : -1;
                    }
                } else {
                    uid = slot_unit(k, slot, slots, units);
                    if (uid < 0) break;
                    if (a.sched_perm) uid = a.sched_perm[uid];
                }
                const int b = k & 1;
                uint16_t *list = lists + b * kMaxListTiles;
                // the list buffer of unit k - 2 must have been read by every role
                if (k >= 2) ok = __all_sync(0xffffffffu, wt.wait(list_free(b), ((k - 2) >> 1) & 1));
                if (!ok) break;
                if (uid < 0) {
                    // the queue is empty: tell the other roles, then stop
                    if (lane == 0) {
                        uid_smem[b] = -1;
                        n_vis_smem[b] = 0;
                        qpos_smem[b] = -1;
                        tc::mbar_arrive(list_full(b));
                    }
                    break;
                }
                Unit un = unit_of(a, uid, PAIR, rank, DO);
                if constexpr (PAGED) set_span(a, un, lane == 0);
                // ring-direct verify: the lane's history length and write position
                int ring_l = 0, ring_p = 0;
                int lane_splits_here = a.splits;
                if constexpr (RING) {
                    uint32_t rl, rp;
                    if (a.lanes <= 32) {
                        rl = __shfl_sync(0xffffffffu, my_rl, un.t.lane);
                        rp = __shfl_sync(0xffffffffu, my_rp, un.t.lane);
                        lane_splits_here = __shfl_sync(0xffffffffu, my_ls, un.t.lane);
                    } else {
                        rl = a.ring_len[un.t.lane];
                        rp = a.ring_wp[un.t.lane];
                        if (a.lane_splits) lane_splits_here = a.lane_splits[un.t.lane];
                    }
                    // out-of-range counters are clamped, as by the pack and mask kernels
                    if (lane == 0 && (rl > (uint32_t)a.ring_w || rp >= (uint32_t)a.ring_w))
                        raise_flag(a.status, GQA_FLAG_RING_CLAMPED);
                    ring_l = (int)min(rl, (uint32_t)a.ring_w);
                    ring_p = (int)(rp % (uint32_t)a.ring_w);
                }
                // visible key tiles in order: (j - jb) | 0x8000 when the mask applies
                auto code_of = [&](int j) {
                    return j >= un.je ? 0
                           : RING     ? ring_tile_code(a, j, ring_l, ring_p)
                           : PAGED    ? paged_tile_code(a, un, j)
                                      : tile_code(a, un.cg, j);
                };
                // splits over the visible tiles: this unit keeps visible tiles [lo, hi)
                // (a unit spans at most kMaxListTiles key tiles: each lane's codes are
                // worked out once)
                int codes[kMaxListTiles / 32];
#pragma unroll
                for (int q = 0; q < kMaxListTiles / 32; ++q)
                    codes[q] = un.jb + 32 * q < un.je ? code_of(un.jb + 32 * q + lane) : 0;
                int lo = 0, hi = 0x7fffffff;
                if (a.vis_split) {
                    int all = 0;
#pragma unroll
                    for (int q = 0; q < kMaxListTiles / 32; ++q)
                        all += __popc(__ballot_sync(0xffffffffu, codes[q] != 0));
                    const int S = (RING && a.lane_splits) ? lane_splits_here : a.splits;
                    lo = (int)((int64_t)un.split * all / S);
                    hi = (int)((int64_t)(un.split + 1) * all / S);
                }
                int n = 0, seen = 0;
#pragma unroll
                for (int q = 0; q < kMaxListTiles / 32; ++q) {
                    const int j = un.jb + 32 * q + lane;
                    const int code = codes[q];
                    const unsigned vis = __ballot_sync(0xffffffffu, code != 0);
                    const int idx = seen + __popc(vis & ((1u << lane) - 1u));
                    const bool keep = code != 0 && idx >= lo && idx < hi;
                    const unsigned kept = __ballot_sync(0xffffffffu, keep);
                    if (keep)
                        list[n + __popc(kept & ((1u << lane) - 1u))] =
                            (uint16_t)((j - un.jb) | (code == 2 ? 0x8000 : 0));
                    n += __popc(kept);
                    seen += __popc(vis);
                }
                __syncwarp();
                if (ring_plan && n > 1 && un.jb == 0 && list[0] == 0x8000) {
                    // key tile 0 (the current rows) last: its load waits for the pre-pass
                    __syncwarp();
                    uint16_t e[kMaxListTiles / 32];
#pragma unroll
                    for (int q = 0; q < kMaxListTiles / 32; ++q) {
                        const int i = lane + 32 * q;
                        e[q] = i < n ? list[(i + 1) % n] : 0;
                    }
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < kMaxListTiles / 32; ++q) {
                        const int i = lane + 32 * q;
                        if (i < n) list[i] = e[q];
                    }
                }
                if (lane == 0) {
                    n_vis_smem[b] = n;
                    uid_smem[b] = uid;
                    qpos_smem[b] = qpos;
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(list_full(b));
                auto tile_at = [&](int v) { return un.jb + (list[v] & 0x7fff); };
                // Every lane walks the ring positions; lane 0 waits for a free slot and
                // issues the TMA loads, and the whole warp fills the current-rows tile of a
                // ring-direct verify.
                auto slot_free = [&]() -> bool {
                    bool w = true;
                    if (lane == 0) w = wt.wait(empty(stage), (round & 1) ^ 1);
                    return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
                };
                // f32 Q tile first (consumed by the softmax warps): [128 rows][32 f32]
                // boxes, completing on this CTA's own barrier
                for (int qs = 0; qs < (n > 0 ? q_pos : 0) && ok; ++qs) {
                    if (!(ok = slot_free())) break;
                    if (lane == 0) {
                        const uint32_t dst = sbase + L::kStages + stage * kStageBytes;
                        tc::mbar_arrive_expect_tx(full(stage), kStageBytes);
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx)
                            if constexpr (RING)  // {d, rows, heads, lanes}: 128 / rows heads x rows
                                tc::tma_load_4d(dst + bx * 16384, &tmq, full(stage), qs * 64 + bx * 32, 0,
                                                un.q_head0, un.t.lane);
                            else
                                tc::tma_load_3d(dst + bx * 16384, &tmq, full(stage), qs * 64 + bx * 32,
                                                a.q_rows_dim1 ? un.t0 + un.q_row0 : un.q_head0,
                                                a.q_rows_dim1 ? un.q_head0 : un.t0 + un.q_row0);
                    }
                    next();
                }
                // chunked prefill: one stage of K or V of key tile j over the sequence's
                // pages, as BN / pg_box boxes of [pg_box slots][64 columns] (pg_box divides
                // the page size, so no box straddles two pages), each lane issuing one.
                // Keys at or past the context end ctx are never visible: their K rows
                // are left as they are (their scores are replaced by -inf), their V rows
                // are zeroed, so that the zero probabilities meet finite values; the V
                // box holding the context end is copied row by row.
                auto fill_paged = [&](uint32_t dst, bool is_v, int j, int d0, int page) {
                    const int ctx = un.ps + un.ntok;
                    const int kb = j * BN, key0 = kb + lane * a.pg_box;
                    const bool tma = lane * a.pg_box < BN && key0 < ctx && (!is_v || key0 + a.pg_box <= ctx);
                    if (is_v && kb + BN > ctx) {
                        uint8_t *img = smem + (dst - sbase);
                        const int m0 = max((ctx / a.pg_box) * a.pg_box - kb, 0);  // first row not by TMA
                        for (int q = m0 * 16 + lane; q < BN * 16; q += 32) {
                            const int row = q >> 4, c = (q >> 3) & 1, ch = q & 7;
                            const int key = kb + row;
                            uint4 v = make_uint4(0u, 0u, 0u, 0u);
                            if (key < ctx)
                                v = ld_nc_v4(a.v_pool + (int64_t)page_of(a, un.t.lane, key) * a.pool_page +
                                             (int64_t)(key % a.page_size) * a.pool_token +
                                             (int64_t)un.t.kh * a.pool_head + d0 + c * 64 + ch * 8);
                            *reinterpret_cast<uint4 *>(img + c * (BN * 128) + sw128(row, ch)) = v;
                        }
                        tc::fence_async_smem();
                    }
                    const int boxes = __popc(__ballot_sync(0xffffffffu, tma));
                    __syncwarp();
                    if (lane == 0) {
                        if (boxes)
                            tc::mbar_arrive_expect_tx(full(stage), (uint32_t)boxes * a.pg_box * 256u);
                        else
                            tc::mbar_arrive(full(stage));
                    }
                    __syncwarp();
                    if (tma) {
                        const int slot_in_page = key0 % a.page_size;
                        auto crd = [&](int w) { return w == 0 ? un.t.kh : (w == 1 ? slot_in_page : page); };
                        const int c1 = crd(a.pg_dim[0]), c2 = crd(a.pg_dim[1]), c3 = crd(a.pg_dim[2]);
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tc::tma_load_4d(dst + c * (BN * 128) + lane * a.pg_box * 128,
                                            is_v ? (const void *)&tmv : (const void *)&tmk, full(stage),
                                            d0 + c * 64, c1, c2, c3);
                    }
                };
                // chunked prefill: the page of this lane's box of key tile j (its load is
                // issued a tile ahead of the stages that use it, so that its latency is
                // not on the producer's path)
                auto box_page = [&](int j) -> int {
                    const int key0 = j * BN + lane * a.pg_box;
                    if (!PAGED || lane * a.pg_box >= BN || key0 >= un.ps + un.ntok) return 0;
                    return ld_s32(a.page_table + (int64_t)un.t.lane * a.max_pages + key0 / a.page_size);
                };
                auto checked = [&](int page) {
                    if (page < 0 || page >= a.num_pages) {
                        raise_flag(a.status, GQA_FLAG_PAGE_CLAMPED);
                        page = page < 0 ? 0 : a.num_pages - 1;
                    }
                    return page;
                };
                // one stage of K or V: two boxes of [BN rows][64 columns] from column d0
                auto load = [&](int j, bool is_v, int d0, int page = 0) -> bool {
                    if (!slot_free()) return false;
                    const uint32_t dst = sbase + L::kStages + stage * kStageBytes;
                    if (PAGED) {
                        fill_paged(dst, is_v, j, d0, checked(page));
                    } else if (RING && j == 0) {
                        // the current rows (bf16, padded with zero rows by the tensor map; K of
                        // all heads, then V), rounded by the pre-pass
                        if (!prepass_done) {
                            if (lane == 0) tc::griddep_wait();
                            prepass_done = true;
                        }
                        if (lane == 0) {
                            tc::mbar_arrive_expect_tx(full(stage), kStageBytes);
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                tc::tma_load_3d(dst + c * (BN * 128), &tmo, full(stage), d0 + c * 64, 0,
                                                (is_v ? a.lanes * a.n_kv_heads : 0) + un.head_idx);
                        }
                    } else if (lane == 0) {
                        tc::mbar_arrive_expect_tx(full(stage), kStageBytes);
                        const int rows_dim1 = is_v ? a.v_rows_dim1 : a.k_rows_dim1;
                        const int kr = (RING ? j - 1 : j) * BN;
                        const int c1 = rows_dim1 ? kr : un.head_idx;
                        const int c2 = rows_dim1 ? un.head_idx : kr;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tc::tma_load_3d(dst + c * (BN * 128), is_v ? (const void *)&tmv : (const void *)&tmk,
                                            full(stage), d0 + c * 64, c1, c2);
                    }
                    next();
                    return true;
                };
                // PAIR: one stage of this CTA's half of a tile, counted on the even CTA's
                // full barrier (which expects both halves): K = keys [64 rank, +64) of the
                // tile, columns [d0, d0 + 256); V = all 128 keys, output columns
                // [d_off + 128 rank, +128)
                auto load_half = [&](int j, bool is_v, int d0, int page = 0) -> bool {
                    if (!slot_free()) return false;
                    if constexpr (PAGED) {
                        // chunked prefill: lane b issues box b of the tile (pg_box keys of one
                        // page) if it falls in this CTA's half.  Every stage carries its whole
                        // bytes, as the even CTA's barrier expects: a box past the context end
                        // ctx reads the zero fill of an out-of-range page, and the V box holding
                        // ctx goes one row at a time, rows past ctx from an out-of-range slot,
                        // so that V rows past ctx are zero (they meet zero probabilities); K
                        // rows past ctx inside a box are left as they are (their scores are
                        // replaced by -inf).
                        const uint32_t dst = sbase + L::kStages + stage * kStageBytes;
                        if (lane == 0 && rank == 0) tc::mbar_arrive_expect_tx(full(stage), 2 * kStageBytes);
                        const uint32_t fb = tc::mapa_shared(full(stage), 0);
                        const int ctx = un.ps + un.ntok;
                        const int k_lo = is_v ? 0 : (int)rank * (BN / 2), k_n = is_v ? BN : BN / 2;
                        const int r0 = lane * a.pg_box - k_lo;  // the box's first row in this CTA's image
                        if (r0 >= 0 && r0 < k_n) {
                            const int key0 = j * BN + lane * a.pg_box;
                            const int slot0 = key0 % a.page_size;
                            const int pg = key0 < ctx ? checked(page) : a.num_pages;
                            auto crd = [&](int w, int slot) { return w == 0 ? un.t.kh : (w == 1 ? slot : pg); };
                            if (!is_v) {
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    tc::tma_load_4d_pair(dst + c * (BN / 2 * 128) + r0 * 128, &tmk, fb, d0 + c * 64,
                                                         crd(a.pg_dim[0], slot0), crd(a.pg_dim[1], slot0),
                                                         crd(a.pg_dim[2], slot0));
                            } else if (key0 + a.pg_box <= ctx || key0 >= ctx) {
                                // V stage page-major: both 64-column chunks of the page's rows
                                // in one copy, {64 columns, slots, chunks, kv head, page}
                                tc::tma_load_5d_pair(dst + r0 * 256, &tmv, fb, 0, slot0,
                                                     (un.d_off + (int)rank * 128) / 64, un.t.kh, pg);
                            } else {
                                for (int rr = 0; rr < a.pg_box; ++rr) {
                                    const int slot = key0 + rr < ctx ? slot0 + rr : a.page_size;
#pragma unroll
                                    for (int c = 0; c < 2; ++c)
                                        tc::tma_load_4d_pair(dst + r0 * 256 + c * a.pg_box * 128 + rr * 128, &tmv1, fb,
                                                             un.d_off + (int)rank * 128 + c * 64,
                                                             crd(a.pg_dim[0], slot), crd(a.pg_dim[1], slot),
                                                             crd(a.pg_dim[2], slot));
                                }
                            }
                        }
                        next();
                        return true;
                    }
                    if (lane == 0) {
                        const uint32_t dst = sbase + L::kStages + stage * kStageBytes;
                        if (rank == 0) tc::mbar_arrive_expect_tx(full(stage), 2 * kStageBytes);
                        const uint32_t fb = tc::mapa_shared(full(stage), 0);
                        if (is_v) {
                            const int c1 = a.v_rows_dim1 ? j * BN : un.head_idx;
                            const int c2 = a.v_rows_dim1 ? un.head_idx : j * BN;
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                tc::tma_load_3d_pair(dst + c * (BN * 128), &tmv, fb,
                                                     un.d_off + (int)rank * 128 + c * 64, c1, c2);
                        } else {
                            const int kr = j * BN + (int)rank * (BN / 2);
                            const int c1 = a.k_rows_dim1 ? kr : un.head_idx;
                            const int c2 = a.k_rows_dim1 ? un.head_idx : kr;
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                tc::tma_load_3d_pair(dst + c * (BN / 2 * 128), &tmk, fb, d0 + c * 64, c1, c2);
                        }
                    }
                    next();
                    return true;
                };
                // the MMA issuer consumes K of tile v+1 before V of tile v: K0, K1, V0, K2, V1, ...
                if constexpr (PAIR) {
                    // (chunked prefill: the pages of tiles v and v + 1)
                    int pg_v = PAGED && n > 0 ? box_page(tile_at(0)) : 0;
                    int pg_n = PAGED && n > 1 ? box_page(tile_at(1)) : 0;
                    for (int ks = 0; ks < KST && ok && n > 0; ++ks) ok = load_half(tile_at(0), false, ks * 256, pg_v);
                    for (int v = 0; ok && v < n; ++v) {
                        const int pg_nn = PAGED && v + 2 < n ? box_page(tile_at(v + 2)) : 0;
                        for (int ks = 0; ks < KST && ok && v + 1 < n; ++ks)
                            ok = load_half(tile_at(v + 1), false, ks * 256, pg_n);
                        if (ok) ok = load_half(tile_at(v), true, 0, pg_v);
                        pg_v = pg_n;
                        pg_n = pg_nn;
                    }
                } else {
                    // pages of tiles v and v + 1 (chunked prefill)
                    int pg_v = n > 0 ? box_page(tile_at(0)) : 0;
                    int pg_n = n > 1 ? box_page(tile_at(1)) : 0;
                    for (int ks = 0; ks < KSUB && ok && n > 0; ++ks) ok = load(tile_at(0), false, ks * 128, pg_v);
                    for (int v = 0; ok && v < n; ++v) {
                        const int pg_nn = v + 2 < n ? box_page(tile_at(v + 2)) : 0;
                        for (int ks = 0; ks < KSUB && ok && v + 1 < n; ++ks)
                            ok = load(tile_at(v + 1), false, ks * 128, pg_n);
                        for (int vs = 0; vs < VSUB && ok; ++vs) ok = load(tile_at(v), true, un.d_off + vs * 128, pg_v);
                        pg_v = pg_n;
                        pg_n = pg_nn;
                    }
                }
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            // (PAIR: the even CTA issues for both; the odd CTA's MMA warp relays)
            if (lane == 0 && rank == 0) {
                const uint32_t idesc_qk = tc::idesc_f16(PAIR ? 2 * BM : BM, BN, kBf16, false);
                const uint32_t idesc_pv = tc::idesc_f16(PAIR ? 2 * BM : BM, PAIR ? DO : 128, kBf16, true);
                int stage = 0;
                uint32_t round = 0;
                auto next = [&]() {
                    if (++stage == NS) {
                        stage = 0;
                        ++round;
                    }
                };
                // S(g) = Q K^T into buffer g & 1
                auto issue_s = [&](int g) -> bool {
                    const uint32_t d_tm = tm_s + (uint32_t)(g & 1) * BN;
                    for (int ks = 0; ks < KST; ++ks) {
                        if (!wt.template wait<PAIR>(full(stage), round & 1)) return false;
                        tc::tc_fence_after();
                        const uint32_t kb = sbase + L::kStages + stage * kStageBytes;
                        if constexpr (PAIR) {
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk) {
                                const int dq = ks * 256 + kk * 16;
                                const uint64_t db = tc::smem_desc_sw128(
                                    kb + (kk / 4) * (BN / 2 * 128) + (kk % 4) * 32, 16, 1024);
                                const uint64_t da = tc::smem_desc_sw128(
                                    sbase + L::kQ + (dq / 64) * (BM * 128) + ((dq % 64) / 16) * 32, 16, 1024);
                                tc::mma_f16_ss_pair(d_tm, da, db, idesc_qk, (ks | kk) != 0);
                            }
                            // two arrivals: see the empty barriers' count
                            tc::mma_commit_pair(empty(stage));
                            tc::mma_commit_pair(empty(stage));
                        } else {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const int dq = ks * 128 + kk * 16;
                                const uint64_t db =
                                    tc::smem_desc_sw128(kb + (kk / 4) * (BN * 128) + (kk % 4) * 32, 16, 1024);
                                if constexpr (C::QTM) {
                                    tc::mma_f16_ts(d_tm, tm_q + dq / 2, db, idesc_qk, (ks | kk) != 0);
                                } else {
                                    const uint64_t da = tc::smem_desc_sw128(
                                        sbase + L::kQ + (dq / 64) * (BM * 128) + ((dq % 64) / 16) * 32, 16,
                                        1024);
                                    tc::mma_f16_ss(d_tm, da, db, idesc_qk, (ks | kk) != 0);
                                }
                            }
                            tc::mma_commit(empty(stage));
                        }
                        next();
                    }
                    if constexpr (PAIR)
                        tc::mma_commit_pair(s_full(g & 1));
                    else
                        tc::mma_commit(s_full(g & 1));
                    return true;
                };
                bool ok = true;
                int g = 0;        // global index of the unit's first tile
                int with_o = 0;   // units so far that produced O (one o_free phase each)
                for (int k = 0; ok; ++k) {
                    if (!a.sched_counter && slot_unit(k, slot, slots, units) < 0) break;
                    const int b = k & 1;
                    if (!(ok = wt.wait(list_full(b), (k >> 1) & 1))) break;
                    if (uid_smem[b] < 0) break;  // the unit queue has ended
                    const int n = n_vis_smem[b];
                    tc::mbar_arrive(list_free(b));
                    if (n == 0) continue;  // no visible key: no loads, no Q, no O
                    for (int q = 0; q < q_pos; ++q) next();  // the Q stages are the softmax's
                    if (!(ok = wt.template wait<PAIR>(q_full, (with_o & 1)))) break;
                    tc::tc_fence_after();
                    ok = issue_s(g);
                    for (int i = 0; ok && i < n; ++i) {
                        const int gi = g + i;
                        if (i + 1 < n && !(ok = issue_s(gi + 1))) break;
                        if (!(ok = wt.template wait<PAIR>(p_full(gi & 1), (gi >> 1) & 1))) break;
                        // the first P.V of a unit overwrites O: the previous unit's O must
                        // have been read out of TMEM
                        if (i == 0 && with_o > 0 && !(ok = wt.template wait<PAIR>(o_free, (with_o - 1) & 1)))
                            break;
                        tc::tc_fence_after();
                        if constexpr (PAIR) {
                            // one stage: this CTA's and the peer's halves of V, N = DO
                            if (!(ok = wt.template wait<true>(full(stage), round & 1))) break;
                            tc::tc_fence_after();
                            const uint32_t vb = sbase + L::kStages + stage * kStageBytes;
                            // (chunked prefill: V stages are page-major, [page][2 column
                            // chunks][pg_box rows][128 B], so that one copy brings a page's
                            // rows of both chunks: a 16-key step starts in its page's block,
                            // the chunks are pg_box rows apart, and the two 8-key row groups
                            // 1 KiB apart within a page, or a page block apart for 8-slot pages)
                            const int lg = PAGED ? __ffs(a.pg_box) - 1 : 7;  // log2 of the page box (a power of 2)
                            const uint32_t v_lbo = 128u << lg;
                            const uint32_t v_sbo = lg < 4 ? 256u << lg : 1024u;
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk) {
                                const uint32_t va = PAGED ? vb + ((uint32_t)((kk * 16) >> lg) << (lg + 8)) +
                                                                ((uint32_t)((kk * 16) & ((1 << lg) - 1)) << 7)
                                                          : vb + kk * 16 * 128;
                                const uint64_t db = tc::smem_desc_sw128(va, v_lbo, v_sbo);
                                tc::mma_f16_ts_pair(tm_o, tm_s + (uint32_t)(gi & 1) * BN + kk * 8, db, idesc_pv,
                                                    (i | kk) != 0);
                            }
                            tc::mma_commit_pair(empty(stage));
                            tc::mma_commit_pair(empty(stage));
                            next();
                            tc::mma_commit_pair(o_done(gi & 1));
                            continue;
                        }
                        // the VSUB stages of V follow each other in the ring
                        int st[VSUB];
#pragma unroll
                        for (int vs = 0; vs < VSUB; ++vs) {
                            if (ok) ok = wt.wait(full(stage), round & 1);
                            st[vs] = stage;
                            next();
                        }
                        if (!ok) break;
                        tc::tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
#pragma unroll
                            for (int vs = 0; vs < VSUB; ++vs) {
                                const uint32_t vb = sbase + L::kStages + st[vs] * kStageBytes;
                                const uint64_t db = tc::smem_desc_sw128(vb + kk * 16 * 128, BN * 128, 1024);
                                tc::mma_f16_ts(tm_o + vs * 128, tm_s + (uint32_t)(gi & 1) * BN + kk * 8, db,
                                               idesc_pv, (i | kk) != 0);
                            }
#pragma unroll
                        for (int vs = 0; vs < VSUB; ++vs) tc::mma_commit(empty(st[vs]));
                        tc::mma_commit(o_done(gi & 1));
                    }
                    g += n;
                    ++with_o;
                }
                // every MMA of this thread has finished before TMEM can be released
                // (this wait ignores the abort flag: only the time limit ends it)
                if constexpr (PAIR)
                    tc::mma_commit_pair(mma_fin);
                else
                    tc::mma_commit(mma_fin);
                const Waiter fin{abort_flag, a.status, kWaitLimitNs, false};
                fin.wait(mma_fin, 0);
            }
            if constexpr (PAIR) {
                // odd CTA: forward each tile's "P written" and each unit's "O read out"
                // from this CTA's softmax warps to the even CTA's barriers with one
                // arrival each, so that the softmax warps only arrive locally.  Every
                // phase is seen in turn: P(g + 2) needs S(g + 2), which the even CTA
                // issues only after this arrival for P(g), and a unit's O is read out
                // only after all its P.V, which follow the previous forward of O.  The
                // tensor-memory accesses behind each signal are complete
                // (tcgen05.wait::st / ::ld) before the warps arrive locally, so the
                // forwarded arrival needs no release.
                if (lane == 0 && rank == 1) {
                    bool ok = true;
                    int g = 0, with_o = 0;
                    for (int k = 0; ok; ++k) {
                        if (!a.sched_counter && slot_unit(k, slot, slots, units) < 0) break;
                        const int b = k & 1;
                        if (!(ok = wt.wait(list_full(b), (k >> 1) & 1))) break;
                        if (uid_smem[b] < 0) break;  // the unit queue has ended
                        const int n = n_vis_smem[b];
                        tc::mbar_arrive(list_free(b));
                        for (int i = 0; ok && i < n; ++i) {
                            const int gi = g + i;
                            if (!(ok = wt.template wait<true>(p_full(gi & 1), (gi >> 1) & 1))) break;
                            tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(p_full(gi & 1), 0));
                        }
                        if (!ok || n == 0) continue;
                        if (!(ok = wt.template wait<true>(o_free, with_o & 1))) break;
                        tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(o_free, 0));
                        g += n;
                        ++with_o;
                    }
                }
            }
            __syncwarp();
        }
    } else {
        tc::setmaxnreg_inc<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax
        // warp w: rows 32 (w % 4) .. + 31 (TMEM lanes), column half h = w / 4
        const int r = (warp & 3) * 32 + lane;
        const int h = warp >> 2;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int pair_bar = 2 + (warp & 3);  // named barrier of warps w and w + 4
        // parameters read every tile, held in registers: a kernel-parameter read
        // that misses the constant cache (shared with this large kernel's
        // instructions) costs an L2 round trip on the critical path
        float scale_log2 = a.scale_log2;
        int n_keys = a.n_keys, mask_bf16 = a.mask_bf16;
        asm volatile("" : "+f"(scale_log2), "+r"(n_keys), "+r"(mask_bf16));
        bool ok = true;
        // PAIR, odd CTA: this CTA's full barriers complete a phase only for its own Q
        // loads (its K/V loads complete on the even CTA's barriers), so the parity of
        // its Q waits is the count of earlier Q uses of the slot, kept per slot here
        uint32_t q_uses = 0;

        // ---- release a ring slot this CTA's softmax is done with (PAIR: in both CTAs)
        auto release_slot = [&](int stage) {
            tc::mbar_arrive(empty(stage));
            // PAIR: the other CTA's producer reloads this slot only once both CTAs'
            // Q stages in it are consumed
            if constexpr (PAIR) tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(empty(stage), rank ^ 1));
        };
        // ---- Q of unit `un` (ring positions from qpos when it arrives by TMA): this
        // thread's 32 columns of each 64-column block, as f16/bf16.  With `hold`, the
        // f32 stages are kept (not released) to stage the previous unit's O.
        auto convert_q = [&](const Unit &un, int qpos, bool hold) {
            int head = 0, row = 0;
            const bool valid = row_of(a, un.t, r, head, row) && row < un.ntok;
            auto put_q = [&](int cb, const uint32_t(&w)[16]) {
                if constexpr (C::QTM) {
                    tc::tmem_st16(tm_q + cb * 32 + h * 16 + lane_base, w);
                } else {
                    uint8_t *qs = smem + L::kQ + cb * (BM * 128);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(qs + sw128(r, h * 4 + c)) =
                            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                }
            };
            if (a.q_tma) {
                // f32 Q arrives by TMA through kQStages ring stages; half h converts box h
                for (int qs = 0; qs < kQStages; ++qs) {
                    const int stage = (qpos + qs) % NS;
                    const uint32_t round = (uint32_t)((qpos + qs) / NS);
                    const uint32_t parity = (PAIR && rank == 1) ? (q_uses >> stage) & 1u : round & 1u;
                    q_uses ^= 1u << stage;
                    if (ok) ok = wt.wait(full(stage), parity);
                    ok = __all_sync(0xffffffffu, ok);
                    if (ok) {
                        const uint8_t *src = smem + L::kStages + stage * kStageBytes + h * 16384;
                        uint32_t w[16];
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 x =
                                *reinterpret_cast<const float4 *>(src + r * 128 + ((c4 ^ (r & 7)) << 4));
                            w[c4 * 2] = pack2(KV{}, x.x, x.y);
                            w[c4 * 2 + 1] = pack2(KV{}, x.z, x.w);
                        }
                        put_q(qs, w);
                    }
                    ok = tc::named_bar_and(1, kSoftmaxThreads, ok);  // every softmax thread is done with this stage
                    if (threadIdx.x == 0 && !hold) release_slot(stage);
                }
            } else if (!a.q_f32) {
                // 16-bit Q: each thread reads its half of its own row with all loads in
                // flight at once, then stores the blocks
                uint4 x[D / 64][4];
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb)
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        x[cb][v] = valid ? ld_nc_v4(static_cast<const uint16_t *>(a.q) + un.t.lane * a.q_lane +
                                                    (int64_t)head * a.q_head + (int64_t)(un.t0 + row) * a.q_row +
                                                    cb * 64 + h * 32 + v * 8)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb) {
                    uint32_t w[16];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        w[4 * v] = x[cb][v].x;
                        w[4 * v + 1] = x[cb][v].y;
                        w[4 * v + 2] = x[cb][v].z;
                        w[4 * v + 3] = x[cb][v].w;
                    }
                    put_q(cb, w);
                }
            } else if constexpr (!C::QTM) {
                // f32 Q without TMA, Q in shared memory: each warp converts its 32 rows'
                // half (the columns its threads own), a row per load instruction -- eight
                // lanes per 32-column segment, so a warp reads whole 128-byte lines (a
                // thread-per-row load would touch 32 rows per instruction) -- with every
                // load of the warp in flight at once
                constexpr int SEG = D / 64;           // 32-column segments of a row half
                constexpr int PER = SEG * 32 / 128;   // float4 loads per lane per row
                const int rbase = (warp & 3) * 32;
                // rows that carry no query load row 0 of the tensor (any valid address) and
                // are zeroed at conversion, so that no load result is consumed before all
                // loads are issued
                constexpr int RB = 32 / PER;          // rows per batch: 32 loads in flight
#pragma unroll
                for (int j0 = 0; j0 < 32; j0 += RB) {
                    float4 x[RB][PER];
                    uint32_t rows_ok = 0;
#pragma unroll
                    for (int j = 0; j < RB; ++j) {
                        int hd = 0, rw = 0;
                        const bool ok_row = row_of(a, un.t, rbase + j0 + j, hd, rw) && rw < un.ntok;
                        rows_ok |= (ok_row ? 1u : 0u) << j;
                        const float *src = static_cast<const float *>(a.q) +
                                           (ok_row ? un.t.lane * a.q_lane + (int64_t)hd * a.q_head +
                                                         (int64_t)(un.t0 + rw) * a.q_row
                                                   : 0) +
                                           h * 32 + (lane & 7) * 4;
#pragma unroll
                        for (int k = 0; k < PER; ++k) x[j][k] = ld_nc_f4(src + (lane / 8 + 4 * k) * 64);
                    }
#pragma unroll
                    for (int j = 0; j < RB; ++j)
#pragma unroll
                        for (int k = 0; k < PER; ++k) {
                            const int cb = lane / 8 + 4 * k, rr = rbase + j0 + j;
                            const bool ok_row = (rows_ok >> j) & 1u;
                            *reinterpret_cast<uint2 *>(smem + L::kQ + cb * (BM * 128) +
                                                       sw128(rr, h * 4 + (lane & 7) / 2) + (lane & 1) * 8) =
                                ok_row ? make_uint2(pack2(KV{}, x[j][k].x, x[j][k].y),
                                                    pack2(KV{}, x[j][k].z, x[j][k].w))
                                       : make_uint2(0u, 0u);
                        }
                }
            } else {
                // f32 Q without TMA, Q in tensor memory: each thread reads its half of its
                // own row (its TMEM lane), every load in flight at once, then converts and
                // stores the blocks
                float4 x[D / 64][8];
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb)
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        x[cb][v] = valid ? ld_nc_f4(static_cast<const float *>(a.q) + un.t.lane * a.q_lane +
                                                    (int64_t)head * a.q_head + (int64_t)(un.t0 + row) * a.q_row +
                                                    cb * 64 + h * 32 + v * 4)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb) {
                    uint32_t w[16];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        w[2 * v] = pack2(KV{}, x[cb][v].x, x[cb][v].y);
                        w[2 * v + 1] = pack2(KV{}, x[cb][v].z, x[cb][v].w);
                    }
                    put_q(cb, w);
                }
            }
            if constexpr (C::QTM)
                tc::tmem_st_wait();
            else
                tc::fence_async_smem();
            tc::tc_fence_before();
            if constexpr (PAIR) {
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(tc::mapa_shared(q_full, 0));
            } else {
                tc::mbar_arrive(q_full);
            }
        };

        int k = 0;
        int uid = -1;
        Unit cur{};
        int cur_n = 0, cur_pos = 0;  // visible tiles and first ring position of unit k
        int cur_qpos = -1;           // its queue position (ring-direct verify)
        if (a.sched_counter || slot_unit(0, slot, slots, units) >= 0) {
            ok = __all_sync(0xffffffffu, wt.wait(list_full(0), 0));
            ok = tc::named_bar_and(1, kSoftmaxThreads, ok);
            uid = ok ? uid_smem[0] : -1;
            cur_qpos = qpos_smem[0];
            if (uid >= 0) {
                cur = unit_of(a, uid, PAIR, rank, DO);
                if constexpr (PAGED) set_span(a, cur, false);
                cur_n = n_vis_smem[0];
                if (cur_n > 0) convert_q(cur, 0, false);
            }
        }
        int g = 0;  // global index of the current unit's first tile
        while (uid >= 0 && ok) {
            const uint16_t *list = lists + (k & 1) * kMaxListTiles;
            int head = 0, row = 0;
            const bool valid = row_of(a, cur.t, r, head, row) && row < cur.ntok;
            const uint16_t *mrow = valid ? a.mask + cur.t.lane * a.m_lane + (int64_t)head * a.m_head +
                                               (int64_t)row * a.m_row + h * 64
                                         : nullptr;
            const bool m_vec = valid && (reinterpret_cast<uintptr_t>(mrow) & 15) == 0;
            // ring-direct verify: ring slot s is visible to this draft row when its history
            // index (wp - 1 - s) mod w is below min(L, w - 1 - row)
            int ring_p = 0, ring_lim = 0;
            if constexpr (RING) {
                const int rl = (int)min(a.ring_len[cur.t.lane], (uint32_t)a.ring_w);
                ring_p = (int)(a.ring_wp[cur.t.lane] % (uint32_t)a.ring_w);
                ring_lim = min(rl, a.ring_w - 1 - row);
            }
            float m_ref = kNegInf, l = 0.f;
            int n_done = 0;  // tiles whose P this thread has handed to the MMA issuer
            // ---- key tiles: this thread owns columns [h*64, h*64 + 64) of every tile.
            // Both warps of a row pair run every iteration and every pair barrier, even
            // after a failed wait (they then skip the work), so neither can be left at
            // a barrier its partner never reaches.
            for (int i = 0; i < cur_n; ++i) {
                const int gi = g + i;
                const int j = cur.jb + (list[i] & 0x7fff);
                const int code = (list[i] & 0x8000) ? 2 : 1;
                if (ok) ok = __all_sync(0xffffffffu, wt.wait(s_full(gi & 1), (gi >> 1) & 1));
                float s[64];
                float mx = kNegInf;
                float sc = 1.f;  // factor still to apply to s (log2 domain)
                if (ok) {
                    tc::tc_fence_after();
                    {
                        uint32_t rr[64];
                        tc::tmem_ld32(tm_s + (uint32_t)(gi & 1) * BN + h * 64 + lane_base,
                                      *reinterpret_cast<uint32_t(*)[32]>(rr));
                        tc::tmem_ld32(tm_s + (uint32_t)(gi & 1) * BN + h * 64 + 32 + lane_base,
                                      *reinterpret_cast<uint32_t(*)[32]>(rr + 32));
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            asm volatile("" : "+r"(rr[c]));  // keep every use after the wait
                            s[c] = __uint_as_float(rr[c]);
                        }
                    }
                    if (!valid) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) s[c] = kNegInf;
                    } else if (code == 1) {
                        // no mask: s stays unscaled; the scale is applied inside the exponent
                        // argument below, and the row maximum is taken on the raw scores
                        sc = scale_log2;
                    } else if constexpr (PAGED) {
                        // keys up to this query's position are visible
                        const int lim = cur.ps + row - (j * BN + h * 64);  // last visible s[c]
#pragma unroll
                        for (int c = 0; c < 64; ++c) s[c] = c <= lim ? s[c] * scale_log2 : kNegInf;
                    } else if constexpr (RING) {
                        if (j == 0) {
                            // the current rows, then padding
#pragma unroll
                            for (int c = 0; c < 64; ++c)
                                s[c] = (h * 64 + c < a.ring_r) ? s[c] * scale_log2 : kNegInf;
                        } else {
                            const int s0 = (j - 1) * BN + h * 64;  // ring slot of s[0]
#pragma unroll
                            for (int c = 0; c < 64; ++c) {
                                int jj = ring_p - 1 - (s0 + c);
                                jj += jj < 0 ? a.ring_w : 0;
                                s[c] = (s0 + c < a.ring_w && jj < ring_lim) ? s[c] * scale_log2 : kNegInf;
                            }
                        }
                    } else {
                        const int c0 = j * BN + h * 64;  // key index of s[0]
                        const uint16_t *mt = mrow + j * BN;
                        if (m_vec && c0 + 64 <= n_keys) {
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const uint4 x = *reinterpret_cast<const uint4 *>(mt + v * 8);
                                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const uint16_t mv = (uint16_t)(w[e / 2] >> ((e & 1) * 16));
                                    s[v * 8 + e] = fmaf(s[v * 8 + e], scale_log2,
                                                        mask_to_f32(mv, mask_bf16) * kLog2e);
                                }
                            }
                        } else {
                            // the row ends inside this half (or the row is not 16-byte
                            // aligned): loads at clamped, valid indices, all independent so
                            // that their latencies overlap
                            uint16_t mv[64];
#pragma unroll
                            for (int c = 0; c < 64; ++c) mv[c] = mt[min(c0 + c, n_keys - 1) - c0];
#pragma unroll
                            for (int c = 0; c < 64; ++c)
                                s[c] = (c0 + c < n_keys)
                                           ? fmaf(s[c], scale_log2, mask_to_f32(mv[c], mask_bf16) * kLog2e)
                                           : kNegInf;
                        }
                    }
                    // row max of sc * s over this half (four chains of three-input max; with
                    // a negative scale the maximum comes from the smallest raw score)
                    float mq[4] = {s[0], s[1], s[2], s[3]};
                    if (sc >= 0.f) {
#pragma unroll
                        for (int c = 4; c < 60; c += 8)
#pragma unroll
                            for (int k = 0; k < 4; ++k) mq[k] = fmax3(mq[k], s[c + k], s[c + 4 + k]);
#pragma unroll
                        for (int k = 0; k < 4; ++k) mq[k] = fmaxf(mq[k], s[60 + k]);
                        mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
                    } else {
#pragma unroll
                        for (int c = 4; c < 60; c += 8)
#pragma unroll
                            for (int k = 0; k < 4; ++k) mq[k] = fmin3(mq[k], s[c + k], s[c + 4 + k]);
#pragma unroll
                        for (int k = 0; k < 4; ++k) mq[k] = fminf(mq[k], s[60 + k]);
                        mx = fmin3(mq[0], mq[1], fminf(mq[2], mq[3]));
                    }
                    mx *= sc;
                }
                // agree with the other half of the row on the maximum
                float *xs = xchg + (gi & 1) * 2 * BM;
                xs[h * BM + r] = mx;
                tc::named_bar(pair_bar, 64);
                mx = fmaxf(mx, xs[(1 - h) * BM + r]);
                if (!ok) continue;
                float factor = 1.f;
                bool resc = false;
                if (m_ref == kNegInf) {
                    m_ref = mx;
                } else if (mx > m_ref + kRescaleThreshold) {
                    factor = ex2(m_ref - mx);
                    m_ref = mx;
                    resc = true;
                }
                const float nmu = m_ref == kNegInf ? 0.f : -m_ref;
                uint32_t pk[32];
                float ra0 = 0.f, ra1 = 0.f, rb0 = 0.f, rb1 = 0.f;
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    // p = 2^(sc * s - mu): one packed FMA per two arguments
                    float x0, x1, x2, x3;
                    ffma2(x0, x1, s[c], s[c + 1], sc, sc, nmu, nmu);
                    ffma2(x2, x3, s[c + 2], s[c + 3], sc, sc, nmu, nmu);
                    const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
                    fadd2(ra0, ra1, ra0, ra1, p0, p1);
                    fadd2(rb0, rb1, rb0, rb1, p2, p3);
                    pk[c / 2] = pack2(KV{}, p0, p1);
                    pk[c / 2 + 1] = pack2(KV{}, p2, p3);
                }
                l = l * factor + ((ra0 + ra1) + (rb0 + rb1));
                // P.V of the previous tile must be done before O is rescaled.  P goes
                // over this tile's own S buffer, which the previous P.V does not read,
                // so without a rescale the softmax runs ahead of the tensor pipe.
                // Parity waits are unambiguous: S(i) complete implies every MMA issued
                // before it (P.V up to tile i-2) completed, and P.V(i) cannot complete
                // before P(i) is written.
                const bool any_resc = __any_sync(0xffffffffu, resc);
                if (i > 0 && any_resc) {
                    ok = __all_sync(0xffffffffu, wt.wait(o_done((gi - 1) & 1), ((gi - 1) >> 1) & 1));
                    if (!ok) continue;
                    tc::tc_fence_after();
                }
                if (any_resc) {
#pragma unroll 1
                    for (int cb = 0; cb < DO / 64; ++cb) {
                        const uint32_t col = tm_o + h * (DO / 2) + cb * 32 + lane_base;
                        uint32_t rr[32];
                        tc::tmem_ld32(col, rr);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            asm volatile("" : "+r"(rr[e]));
                            rr[e] = __float_as_uint(__uint_as_float(rr[e]) * factor);
                        }
                        tc::tmem_st32(col, rr);
                    }
                }
                // P over the first 64 columns of the S buffer it came from
                tc::tmem_st32(tm_s + (uint32_t)(gi & 1) * BN + h * 32 + lane_base, pk);
                tc::tmem_st_wait();
                tc::tc_fence_before();
                if constexpr (PAIR) {
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(p_full(gi & 1));
                } else {
                    tc::mbar_arrive(p_full(gi & 1));
                }
                n_done = i + 1;
            }
            // ---- unit k's tile list is no longer read
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(list_free(k & 1));
            // ---- the next unit's Q is converted before this unit's epilogue, so that its
            // first Q.K^T products overlap the epilogue (all of unit k's S are complete:
            // nothing reads the Q staging area any more)
            int nuid = -1, nxt_qpos = -1;
            Unit nxt{};
            int nxt_n = 0;
            const int nxt_pos = cur_pos + (cur_n > 0 ? unit_positions(cur_n) : 0);
            // O goes out by TMA, staged in shared memory.  head_dim <= 256: in the ring
            // slots of the next unit's f32 Q, held until the stores have read them
            // (512 D >= 512 DO bytes; the next Q is converted first, so its first Q.K^T
            // overlaps this epilogue), or after the last unit in the idle ring.  head_dim
            // 512 (its 8 Q stages cycle through a 3-stage ring and cannot be held): in
            // the Q tile area (128 KiB), before the next unit's Q is converted.
            constexpr bool kHoldQ = kQStages <= NS;
            // (chunked prefill: only tiles whose rows all belong to the sequence)
            const bool stage_o = a.o_tma && cur_n > 0 && (!PAGED || cur.q_row0 + BM <= cur.ntok);
            int o_slot0 = 0;       // first ring position of the staging area
            bool hold_q = false;   // staging in the next unit's Q slots
            // every softmax warp takes the same path from here (a failed wait in one of
            // them ends the loop for all)
            ok = tc::named_bar_and(1, kSoftmaxThreads, ok);
            if (ok && (a.sched_counter || slot_unit(k + 1, slot, slots, units) >= 0)) {
                ok = __all_sync(0xffffffffu, wt.wait(list_full((k + 1) & 1), ((k + 1) >> 1) & 1));
                ok = tc::named_bar_and(1, kSoftmaxThreads, ok);
                nuid = ok ? uid_smem[(k + 1) & 1] : -1;
                nxt_qpos = qpos_smem[(k + 1) & 1];
            }
            if (nuid >= 0) {
                nxt = unit_of(a, nuid, PAIR, rank, DO);
                if constexpr (PAGED) set_span(a, nxt, false);
                nxt_n = n_vis_smem[(k + 1) & 1];
                if constexpr (kHoldQ) {
                    hold_q = stage_o && nxt_n > 0;
                    if (ok && nxt_n > 0) convert_q(nxt, nxt_pos, hold_q);
                    o_slot0 = nxt_pos;
                }
            }
            const bool use_stage = stage_o && (!kHoldQ || hold_q || nuid < 0);

            // ---- epilogue of unit k: both outstanding P.V (tiles n-2 and n-1) must be complete
            if (ok && n_done > 0) {
                const int ga = g + n_done - 1;
                ok = __all_sync(0xffffffffu, wt.wait(o_done(ga & 1), (ga >> 1) & 1));
                if (ok && n_done >= 2)
                    ok = __all_sync(0xffffffffu, wt.wait(o_done((ga - 1) & 1), ((ga - 1) >> 1) & 1));
                tc::tc_fence_after();
            }
            ok = tc::named_bar_and(1, kSoftmaxThreads, ok);
            // row sum = both halves' partial sums (the second barrier keeps the next
            // unit's first row-max exchange, which reuses this buffer, behind the reads)
            {
                float *xs = xchg + ((g + n_done) & 1) * 2 * BM;
                xs[h * BM + r] = l;
                tc::named_bar(pair_bar, 64);
                l += xs[(1 - h) * BM + r];
                tc::named_bar(pair_bar, 64);
            }
            const bool have_o = ok && n_done > 0;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // all of this thread's O columns out of TMEM, then O may be overwritten
            constexpr int NCB = DO / 64;
            uint32_t rr[NCB][32];
            if (have_o) {
#pragma unroll
                for (int cb = 0; cb < NCB; ++cb) tc::tmem_ld32(tm_o + h * (DO / 2) + cb * 32 + lane_base, rr[cb]);
                tc::tmem_ld_wait();
            } else {
#pragma unroll
                for (int cb = 0; cb < NCB; ++cb)
#pragma unroll
                    for (int e = 0; e < 32; ++e) rr[cb][e] = 0u;
            }
            if (cur_n > 0) {
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(o_free);
            }
            if (ok && use_stage) {
                // [128 rows][32 f32] boxes (128-byte swizzle), two per 32 KiB slot; each half
                // of the rows' threads stages its DO/64 boxes, and a box goes out as soon as
                // its 128 writers are done
                const bool issuer = threadIdx.x == h * (kSoftmaxThreads / 2);
#pragma unroll
                for (int cb = 0; cb < NCB; ++cb) {
                    const int box = h * NCB + cb;
                    uint8_t *stg = kHoldQ ? smem + L::kStages + ((o_slot0 + box / 2) % NS) * kStageBytes +
                                                (box & 1) * 16384
                                          : smem + L::kQ + box * 16384;
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        asm volatile("" : "+r"(rr[cb][4 * c4]), "+r"(rr[cb][4 * c4 + 1]), "+r"(rr[cb][4 * c4 + 2]),
                                     "+r"(rr[cb][4 * c4 + 3]));
                        *reinterpret_cast<float4 *>(stg + r * 128 + ((c4 ^ (r & 7)) << 4)) =
                            make_float4(__uint_as_float(rr[cb][4 * c4]) * inv, __uint_as_float(rr[cb][4 * c4 + 1]) * inv,
                                        __uint_as_float(rr[cb][4 * c4 + 2]) * inv,
                                        __uint_as_float(rr[cb][4 * c4 + 3]) * inv);
                    }
                    tc::fence_async_smem();
                    tc::named_bar(6 + h, kSoftmaxThreads / 2);
                    if (issuer && !*abort_flag)
                        tc::tma_store_3d(&tmo, smem_u32(stg), cur.d_off + box * 32,
                                         a.o_rows_dim1 ? cur.t0 + cur.q_row0 : cur.q_head0,
                                         a.o_rows_dim1 ? cur.q_head0 : cur.t0 + cur.q_row0);
                }
                if (issuer) {
                    tc::bulk_commit();
                    tc::bulk_wait_read0();
                }
            } else if (ok) {
                float *dst;
                if (a.splits == 1) {
                    dst = valid ? a.o + cur.t.lane * a.o_lane + (int64_t)head * a.o_head +
                                      (int64_t)(cur.t0 + row) * a.o_row + cur.d_off + h * (DO / 2)
                                : nullptr;
                } else {
                    // partials column-chunk major: the 32 rows of a warp store 512
                    // contiguous bytes per instruction
                    int64_t unit = ((int64_t)cur.tile_id * a.d_parts + cur.dpart) * a.splits + cur.split;
                    if (a.lane_start)  // ring-direct verify: the unit's queue position
                        unit = cur_qpos;
                    dst = nullptr;
                    if (valid) {
                        if (h == 0) a.ws_lse[unit * BM + r] = l > 0.f ? m_ref + __log2f(l) : kNegInf;
                        float4 *base = reinterpret_cast<float4 *>(a.ws_o) + (unit * (DO / 4) + h * (DO / 8)) * BM + r;
#pragma unroll
                        for (int cb = 0; cb < NCB; ++cb)
#pragma unroll
                            for (int e = 0; e < 32; e += 4) {
                                asm volatile("" : "+r"(rr[cb][e]), "+r"(rr[cb][e + 1]), "+r"(rr[cb][e + 2]),
                                             "+r"(rr[cb][e + 3]));
                                base[(cb * 8 + e / 4) * BM] =
                                    make_float4(__uint_as_float(rr[cb][e]) * inv, __uint_as_float(rr[cb][e + 1]) * inv,
                                                __uint_as_float(rr[cb][e + 2]) * inv,
                                                __uint_as_float(rr[cb][e + 3]) * inv);
                            }
                    }
                }
                if (dst) {
#pragma unroll
                    for (int cb = 0; cb < NCB; ++cb)
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            asm volatile("" : "+r"(rr[cb][e]), "+r"(rr[cb][e + 1]), "+r"(rr[cb][e + 2]),
                                         "+r"(rr[cb][e + 3]));
                            *reinterpret_cast<float4 *>(dst + cb * 32 + e) =
                                make_float4(__uint_as_float(rr[cb][e]) * inv, __uint_as_float(rr[cb][e + 1]) * inv,
                                            __uint_as_float(rr[cb][e + 2]) * inv,
                                            __uint_as_float(rr[cb][e + 3]) * inv);
                        }
                }
            }
            // the held Q slots of the next unit go back to the producer once both row
            // halves' stores have read them
            if (hold_q) {
                tc::named_bar(1, kSoftmaxThreads);
                if (threadIdx.x == 0)
                    for (int qs = 0; qs < kQStages; ++qs) release_slot((nxt_pos + qs) % NS);
            }
            if constexpr (!kHoldQ) {
                // head_dim 512: the staged O has been read out of the Q area; now the next Q
                if (use_stage) tc::named_bar(1, kSoftmaxThreads);
                if (nuid >= 0 && ok && nxt_n > 0) convert_q(nxt, nxt_pos, false);
            }
            g += cur_n;
            cur = nxt;
            cur_n = nxt_n;
            cur_pos = nxt_pos;
            cur_qpos = nxt_qpos;
            uid = nuid;
            ++k;
        }
    }

    // ---- teardown: TMEM is released only after every role (of both CTAs of a
    // pair) is done with it
    tc::tc_fence_before();
    if constexpr (PAIR)
        tc::cluster_sync_all();
    else
        __syncthreads();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        if constexpr (PAIR)
            tc::tmem_dealloc_pair<512>(tmem);
        else
            tc::tmem_dealloc<512>(tmem);
    }
}

// One warp per (tile, output half, tile row): merge the key splits.
template <int DO>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnArgs a, int tiles) {
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= tiles * a.d_parts * BM) return;
    const int r = wid % BM;
    const int dpart = (wid / BM) % a.d_parts;
    const int tile_id = wid / (BM * a.d_parts);
    const Tile t = tile_of(a, tile_id);
    int head, row;
    if (!row_of(a, t, r, head, row)) return;
    if (a.tok_off) {
        // chunked prefill: tile rows past the sequence's tokens carry no query
        const SeqSpan q = seq_span(a, t.lane, false);
        if (row >= q.ntok) return;
        row += q.t0;
    }
    const int64_t u0 = ((int64_t)tile_id * a.d_parts + dpart) * a.splits;
    // the splits in use and where their partials are
    const int S = a.lane_splits ? a.lane_splits[t.lane] : a.splits;
    auto slot = [&](int s) -> int64_t {
        return a.lane_start ? a.lane_start[t.lane] + (int64_t)((t.kh * a.head_tiles + t.ht) * S + s) : u0 + s;
    };
    // the splits' log-sum-exps, lane s holding split s0 + s (32 splits per pass)
    static_assert(DO % 128 == 0, "a lane merges DO / 128 float4 columns");
    const float lse0 = lane < S ? a.ws_lse[slot(lane) * BM + r] : kNegInf;
    float M = lse0;
    for (int s = 32 + lane; s < S; s += 32) M = fmaxf(M, a.ws_lse[slot(s) * BM + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // column chunk q = lane + 32 k (four columns) of row r: the float4 at (unit * DO/4 + q) * BM + r
    float4 acc[DO / 128];
#pragma unroll
    for (int k = 0; k < DO / 128; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != kNegInf) {
        for (int s0 = 0; s0 < S; s0 += 32) {
            const float lse = s0 == 0 ? lse0 : (s0 + lane < S ? a.ws_lse[slot(s0 + lane) * BM + r] : kNegInf);
            const float wl = s0 + lane < S ? ex2(lse - M) : 0.f;
            L += wl;
            const int ns = min(32, S - s0);
            // every split's loads are independent of the weights: four splits in flight
#pragma unroll 4
            for (int i = 0; i < ns; ++i) {
                const float w = __shfl_sync(0xffffffffu, wl, i);
                const float4 *src = reinterpret_cast<const float4 *>(a.ws_o) + slot(s0 + i) * (DO / 4) * BM + r;
#pragma unroll
                for (int k = 0; k < DO / 128; ++k) {
                    const float4 x = ld_nc_f4(reinterpret_cast<const float *>(src + (int64_t)(lane + 32 * k) * BM));
                    acc[k].x += w * x.x;
                    acc[k].y += w * x.y;
                    acc[k].z += w * x.z;
                    acc[k].w += w * x.w;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    }
    float *out = a.o + t.lane * a.o_lane + (int64_t)head * a.o_head + (int64_t)row * a.o_row +
                 dpart * DO;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
#pragma unroll
    for (int k = 0; k < DO / 128; ++k) {
        const float4 v = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
        float *dst = out + 4 * (lane + 32 * k);
        if (vec) {
            *reinterpret_cast<float4 *>(dst) = v;
        } else {
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
    }
}

}  // namespace
}  // namespace gqa

// ===========================================================================
// host side
// ===========================================================================
namespace gqa {
namespace {

struct Plan {
    int bn, do_, d_parts;
    int rows_per_head, heads_per_tile, row_tiles, head_tiles, tiles;
    int n_blk, code_cols, code_groups, splits, bps;
    bool shared_mask, pair, vis_split;
    int split_budget;
    size_t codes_bytes, part_o_bytes, part_lse_bytes;
    size_t sched_bytes;  // dynamic unit queue: counter (256 bytes) + order
    size_t cur_bytes;    // ring-direct verify: the current rows in bf16
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// 0: never pair; 1: pair where it measured faster (head_dim 256 and 512, i.e. every
// shape that can pair today); 2: pair every eligible shape
int g_pair_mode = 1;

// CTA pairs need two query tiles that see the same key tiles: one head each,
// 128 rows each, the same rows, a mask shared by all heads, an even number of
// head tiles per KV group, and Q staged in shared memory (head_dim >= 256).
// (same_keys: the heads' rows see the same keys without a shared mask, as in a
// chunked prefill, where visibility follows the token positions alone)
bool pairable(int rows, int n_heads, int n_kv_heads, int head_dim, bool shared_mask, bool same_keys) {
    const int group = n_heads / n_kv_heads;
    if (g_pair_mode == 0 || (g_pair_mode == 1 && head_dim < 256)) return false;
    return (shared_mask || same_keys) && head_dim >= 256 && rows >= BM && group % 2 == 0;
}

Plan make_plan(int lanes, int rows, int n_heads, int n_kv_heads, int head_dim, int n_keys,
               bool shared_mask, bool ring = false, bool same_keys = false) {
    const bool vis_split = ring;
    Plan p{};
    p.bn = BN;
    p.do_ = head_dim == 512 ? 256 : head_dim;
    p.d_parts = head_dim / p.do_;
    const int group = n_heads / n_kv_heads;
    p.rows_per_head = rows < BM ? rows : BM;
    p.heads_per_tile = BM / p.rows_per_head;
    if (p.heads_per_tile > group) p.heads_per_tile = group;
    p.row_tiles = (rows + p.rows_per_head - 1) / p.rows_per_head;
    p.head_tiles = (group + p.heads_per_tile - 1) / p.heads_per_tile;
    p.tiles = lanes * n_kv_heads * p.head_tiles * p.row_tiles;
    p.n_blk = (n_keys + p.bn - 1) / p.bn;
    p.code_cols = (n_keys + 63) / 64;
    p.shared_mask = shared_mask;
    p.code_groups = shared_mask ? lanes * p.row_tiles : p.tiles;
    p.pair = p.heads_per_tile == 1 && p.rows_per_head == BM &&
             pairable(rows, n_heads, n_kv_heads, head_dim, shared_mask, same_keys);
    // a pair occupies two SMs
    const int units = p.tiles * p.d_parts / (p.pair ? 2 : 1);
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    if (p.pair) sms /= 2;
    p.splits = 1;
    // (the unit queue of the ordering pass is required: its group table and the lane
    // split counts in the queue header bound the lanes and groups)
    // (the lane blocks of the queue are worked out by one warp: at most 30 lanes, whose
    // split counts and block starts fit in the queue header)
    p.vis_split = vis_split && !p.pair && p.n_blk <= kMaxListTiles && lanes <= 30;
    if (p.vis_split) {
        // splits share out each tile's visible key tiles: at most sms / (query tiles per
        // lane) per lane (the pre-pass hands them out in proportion to the lanes' visible
        // tiles, about one unit per SM in all)
        int s = sms / (n_kv_heads * p.head_tiles);
        p.split_budget = s < 1 ? 1 : s;
        p.splits = p.split_budget > p.n_blk ? p.n_blk : p.split_budget;
        p.bps = p.n_blk;
    } else if (units < sms && p.n_blk > 1) {
        // one CTA per SM at most: a CTA past the SM count would run as a second wave and
        // double the time of the whole launch
        int s = sms / units;
        if (s > p.n_blk) s = p.n_blk;
        p.splits = s;
    }
    if (!p.vis_split) {
        p.bps = (p.n_blk + p.splits - 1) / p.splits;
        if (p.bps > kMaxListTiles) p.bps = kMaxListTiles;  // a unit's tile list fits in shared memory
        p.splits = (p.n_blk + p.bps - 1) / p.bps;
    }
    p.codes_bytes = align256((size_t)p.code_groups * p.code_cols);
    if (p.splits > 1) {
        size_t nunits = (size_t)p.tiles * p.d_parts * p.splits;
        // splits over the visible tiles: the lanes' split counts add up to at most
        // split_budget + lanes, each used by every query tile of its lane
        if (p.vis_split) {
            const size_t used = (size_t)(p.split_budget + lanes) * n_kv_heads * p.head_tiles * p.d_parts;
            if (used < nunits) nunits = used;
        }
        p.part_o_bytes = align256(nunits * BM * p.do_ * 4);
        p.part_lse_bytes = align256(nunits * BM * 4);
    }
    if (p.vis_split)  // counter, queue length, lane split counts and block starts
        p.sched_bytes = 256;
    if (ring) p.cur_bytes = align256((size_t)2 * lanes * n_kv_heads * rows * head_dim * 2);
    return p;
}

size_t plan_bytes(const Plan &p) {
    return p.codes_bytes + p.part_o_bytes + p.part_lse_bytes + p.sched_bytes + p.cur_bytes;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// rows x heads x D view with element strides (row, head).  The two outer
// dimensions are ordered by increasing stride; with a box of one head the
// shared-memory image is the same [bn rows][64 columns] either way.
bool rows_first(int heads, int64_t row_stride, int64_t head_stride) {
    return heads == 1 || row_stride <= head_stride;
}

// A 3-D tiled map over a [rows][heads][d] view with element strides (row,
// head): box = box_inner columns x box_rows rows x one head, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int d, int rows,
              int heads, int64_t row_stride, int64_t head_stride, int box_inner, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const bool rf = rows_first(heads, row_stride, head_stride);
    const int64_t hs = heads > 1 ? head_stride : row_stride * rows;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)(rf ? rows : heads),
                          (cuuint64_t)(rf ? heads : rows)};
    cuuint64_t strides[2] = {(cuuint64_t)(rf ? row_stride : hs) * esize,
                             (cuuint64_t)(rf ? hs : row_stride) * esize};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, rf ? (cuuint32_t)box_rows : 1u,
                         rf ? 1u : (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A 4-D tiled map over a page pool: head_dim x (kv heads, page slots, pages) with
// element strides (hs, ts, ps), the three outer dimensions ordered by increasing
// stride; box = 64 columns x box_rows slots of one head and one page, 128-byte
// swizzle, so that its shared-memory image is [box_rows][64 columns] whatever the
// order.  dim_of[i] receives the logical coordinate (0 head, 1 slot, 2 page) of
// map dimension i + 1.
bool make_paged_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int d, int hk,
                    int page_size, int num_pages, int64_t hs, int64_t ts, int64_t ps, int box_rows,
                    int dim_of[3]) {
    auto fn = encode_fn();
    if (!fn) return false;
    struct Dim {
        int64_t size, stride;
        int which;
    } v[3] = {{hk, hs, 0}, {page_size, ts, 1}, {num_pages, ps, 2}};
    // a dimension of one element is never stepped along: give it a harmless stride
    for (auto &x : v)
        if (x.size == 1) x.stride = std::max<int64_t>(x.stride, 8);
    std::stable_sort(v, v + 3, [](const Dim &x, const Dim &y) { return x.stride < y.stride; });
    cuuint64_t dims[4] = {(cuuint64_t)d, 0, 0, 0};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {64, 1, 1, 1};
    for (int i = 0; i < 3; ++i) {
        dims[i + 1] = (cuuint64_t)v[i].size;
        strides[i] = (cuuint64_t)v[i].stride * 2;
        if (v[i].which == 1) box[i + 1] = (cuuint32_t)box_rows;
        dim_of[i] = v[i].which;
    }
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, dt, 4, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A 5-D tiled map over a V page pool for page-major stages: {64 columns, page slots, the
// head_dim / 64 column chunks, kv heads, pages} with element strides (ts, 64, hs, ps); a box is
// box_rows slots x 2 chunks of one head and one page, 128-byte swizzle, so that its
// shared-memory image is [2 chunks][box_rows][64 columns].
bool make_paged_v_chunk_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int d, int hk,
                            int page_size, int num_pages, int64_t hs, int64_t ts, int64_t ps, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5] = {64, (cuuint64_t)page_size, (cuuint64_t)(d / 64), (cuuint64_t)hk, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {(cuuint64_t)ts * 2, 128, (cuuint64_t)hs * 2, (cuuint64_t)ps * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)box_rows, 2, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, dt, 5, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, class KV, bool PAIR, int MODE = kMaskMode>
cudaError_t run_attn(const AttnArgs &a, const CUtensorMap *maps, int units, int tiles,
                     cudaStream_t stream) {
    auto kern = attn_kernel<D, KV, PAIR, MODE>;
    // function attributes belong to each device's context: set once per device (and
    // again after a reset)
    static DeviceSetup setup;
    cudaError_t se = setup.run([&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Layout<D>::kBytes);
        if (e != cudaSuccess) return e;
        // the register split must fit in what the block is launched with, or the
        // softmax warpgroups' increase would wait forever
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (2 * 128 * kSoftmaxRegs + 128 * kControlRegs > kThreads * fa.numRegs ||
            kSoftmaxRegs < fa.numRegs || kControlRegs > fa.numRegs)
            return cudaErrorInvalidConfiguration;
        return cudaSuccess;
    });
    if (se != cudaSuccess) return se;
    timing_mark(true, stream);
    {
        // programmatic dependent launch: the kernel's set-up (barriers, TMEM, tensor-map
        // prefetch) overlaps the pre-pass, whose results the producer waits for
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.gridDim = dim3(units);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Layout<D>::kBytes;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = PAIR ? 2 : 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, maps[0], maps[1], maps[2], maps[3], maps[4]);
        if (e != cudaSuccess) return e;
    }
    timing_mark(false, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.splits == 1) return e;
    const int warps = tiles * a.d_parts * BM;
    attn_combine_kernel<Cfg<D>::DO><<<(warps + 3) / 4, 128, 0, stream>>>(a, tiles);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int32_t *status, int timeout_ms, cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 1, 0, stream>>>(status, (uint64_t)timeout_ms * 1000000ull);
    return cudaGetLastError();
}

size_t prefill_workspace_bytes(int rows, int n_heads, int n_kv_heads, int head_dim, int kv_pad) {
    // sized for either tiling, so that changing the pairing mode never
    // invalidates a workspace the caller already holds
    const int saved = g_pair_mode;
    g_pair_mode = 2;
    const size_t with = plan_bytes(make_plan(1, rows, n_heads, n_kv_heads, head_dim, kv_pad, true));
    g_pair_mode = 0;
    const size_t without = plan_bytes(make_plan(1, rows, n_heads, n_kv_heads, head_dim, kv_pad, true));
    g_pair_mode = saved;
    return with > without ? with : without;
}

void set_attention_pairs(int mode) { g_pair_mode = mode; }

size_t verify_workspace_bytes(const gqa_ring_params &p) {
    return plan_bytes(make_plan((int)p.lanes, (int)p.rows, (int)p.q_heads, (int)p.kv_heads,
                                (int)p.head_dim, (int)p.packed_len, false));
}

// key space of a ring-direct verify: one tile of current rows, then the ring slots
int ring_keys(int window) { return BN + window; }

size_t verify_ring_workspace_bytes(const gqa_ring_params &p) {
    return plan_bytes(make_plan((int)p.lanes, (int)p.rows, (int)p.q_heads, (int)p.kv_heads,
                                (int)p.head_dim, ring_keys((int)p.window), false, true));
}

// Chunked prefill: sequences are the lanes, max_tokens their rows, the key space
// max_pages_per_seq * page_size; no mask classification, never paired.
static Plan paged_plan(int num_seqs, int max_tokens, int n_heads, int n_kv_heads, int head_dim,
                       int max_pages_per_seq, int page_size) {
    // CTA pairs (head_dim 256) halve the page boxes each SM copies per tile; they run
    // without key splits
    // (a CTA's half of a K tile, 64 keys, must hold whole page boxes: gcd(page, 128) <= 64)
    Plan pl = make_plan(num_seqs, max_tokens, n_heads, n_kv_heads, head_dim,
                        max_pages_per_seq * page_size, false, false,
                        head_dim == 256 && std::gcd(page_size, BN) <= BN / 2);
    if (pl.pair && pl.splits > 1)
        pl = make_plan(num_seqs, max_tokens, n_heads, n_kv_heads, head_dim, max_pages_per_seq * page_size,
                       false);
    pl.codes_bytes = 0;
    // units differ in cost with each sequence's prefix: a cost-ordered dynamic queue
    pl.sched_bytes = 256 + align256((size_t)pl.tiles * pl.d_parts * pl.splits * 4);
    return pl;
}

size_t paged_prefill_workspace_bytes(int num_seqs, int max_tokens, int n_heads, int n_kv_heads,
                                     int head_dim, int max_pages_per_seq, int page_size) {
    return plan_bytes(paged_plan(num_seqs, max_tokens, n_heads, n_kv_heads, head_dim,
                                 max_pages_per_seq, page_size));
}

cudaError_t launch_paged_prefill(const PagedPrefillProblem &p, void *workspace, cudaStream_t stream) {
    if (p.total_tokens == 0) return cudaSuccess;
    const Plan pl = paged_plan(p.num_seqs, p.max_tokens, p.n_heads, p.n_kv_heads, p.head_dim,
                               p.max_pages_per_seq, p.page_size);
    AttnArgs a{};
    const int64_t row = (int64_t)p.n_heads * p.head_dim;
    a.q = p.q;
    a.q_f32 = 1;
    a.q_row = row;
    a.q_head = p.head_dim;
    a.kv_bf16 = p.kv_dtype == GQA_DTYPE_BF16;
    a.o = p.o;
    a.o_row = row;
    a.o_head = p.head_dim;
    a.lanes = p.num_seqs;
    a.rows = p.max_tokens;
    a.n_heads = p.n_heads;
    a.n_kv_heads = p.n_kv_heads;
    a.group = p.n_heads / p.n_kv_heads;
    a.n_keys = p.max_pages_per_seq * p.page_size;
    a.rows_per_head = pl.rows_per_head;
    a.heads_per_tile = pl.heads_per_tile;
    a.row_tiles = pl.row_tiles;
    a.head_tiles = pl.head_tiles;
    a.tiles_total = pl.tiles;
    a.n_blk = pl.n_blk;
    a.splits = pl.splits;
    a.blk_per_split = pl.bps;
    a.d_parts = pl.d_parts;
    a.scale_log2 = p.scale * kLog2e;
    char *ws = static_cast<char *>(workspace);
    a.ws_o = pl.splits > 1 ? reinterpret_cast<float *>(ws) : nullptr;
    a.ws_lse = pl.splits > 1 ? reinterpret_cast<float *>(ws + pl.part_o_bytes) : nullptr;
    char *sched = ws + pl.part_o_bytes + pl.part_lse_bytes;
    a.sched_counter = reinterpret_cast<int *>(sched);
    a.sched_perm = reinterpret_cast<const int *>(sched + 256);
    a.status = p.status;
    a.tok_off = p.token_offsets;
    a.pos_start = p.position_start;
    a.page_table = p.page_table;
    a.v_pool = static_cast<const uint16_t *>(p.v_pool);
    a.pool_page = p.page_stride;
    a.pool_token = p.token_stride;
    a.pool_head = p.head_stride;
    a.total_tokens = p.total_tokens;
    a.max_pages = p.max_pages_per_seq;
    a.page_size = p.page_size;
    a.num_pages = p.num_pages;
    a.pg_box = std::gcd(p.page_size, BN);  // >= 8: the page size is a multiple of 8

    CUtensorMap maps[5];
    memset(maps, 0, sizeof maps);
    const CUtensorMapDataType kvt =
        a.kv_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    int dim_k[3], dim_v[3];
    if (!make_paged_map(&maps[0], p.k_pool, kvt, p.head_dim, p.n_kv_heads, p.page_size, p.num_pages,
                        p.head_stride, p.token_stride, p.page_stride, a.pg_box, dim_k) ||
        !make_paged_map(&maps[1], p.v_pool, kvt, p.head_dim, p.n_kv_heads, p.page_size, p.num_pages,
                        p.head_stride, p.token_stride, p.page_stride, a.pg_box, dim_v))
        return cudaErrorInvalidValue;
    for (int i = 0; i < 3; ++i) a.pg_dim[i] = dim_k[i];
    // CTA pairs: V in page-major stages (one box per page for both of a CTA's column
    // chunks), and V pages one row high, for the box that holds a sequence's context end
    if (pl.pair && (!make_paged_v_chunk_map(&maps[1], p.v_pool, kvt, p.head_dim, p.n_kv_heads, p.page_size,
                                            p.num_pages, p.head_stride, p.token_stride, p.page_stride,
                                            a.pg_box) ||
                    !make_paged_map(&maps[4], p.v_pool, kvt, p.head_dim, p.n_kv_heads, p.page_size,
                                    p.num_pages, p.head_stride, p.token_stride, p.page_stride, 1, dim_v)))
        return cudaErrorInvalidValue;
    a.pair = pl.pair ? 1 : 0;
    // f32 Q in by TMA and O out by TMA for one head's 128-token tiles
    if (pl.heads_per_tile == 1 && pl.rows_per_head == BM &&
        make_map(&maps[2], p.q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.head_dim, p.total_tokens,
                 p.n_heads, row, p.head_dim, 32, BM)) {
        a.q_tma = 1;
        a.q_rows_dim1 = rows_first(p.n_heads, row, p.head_dim) ? 1 : 0;
        if (pl.splits == 1 &&
            make_map(&maps[3], p.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.head_dim, p.total_tokens,
                     p.n_heads, row, p.head_dim, 32, BM)) {
            a.o_tma = 1;
            a.o_rows_dim1 = a.q_rows_dim1;
        }
    }
    // units: query tiles (CTA pairs: pairs of them) x output halves x key splits
    const int units = pl.tiles * pl.d_parts * pl.splits / (pl.pair ? 2 : 1);
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    const int ctas = pl.pair ? 2 * std::min(units, sms / 2) : std::min(units, sms);
    const int groups = p.num_seqs * p.n_kv_heads;
    if (groups <= kMaxQueueGroups) {
        order_units_kernel<<<1, 1024, groups * sizeof(int), stream>>>(a, units);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else {
        a.sched_perm = nullptr;  // too many groups for one CTA's table: static snake order
        a.sched_counter = nullptr;
    }
    const bool bf = a.kv_bf16;
    switch (p.head_dim) {
        case 128:
            return bf ? run_attn<128, BF16, false, kPagedMode>(a, maps, ctas, pl.tiles, stream)
                      : run_attn<128, F16, false, kPagedMode>(a, maps, ctas, pl.tiles, stream);
        case 256:
            if (pl.pair)
                return bf ? run_attn<256, BF16, true, kPagedMode>(a, maps, ctas, pl.tiles, stream)
                          : run_attn<256, F16, true, kPagedMode>(a, maps, ctas, pl.tiles, stream);
            return bf ? run_attn<256, BF16, false, kPagedMode>(a, maps, ctas, pl.tiles, stream)
                      : run_attn<256, F16, false, kPagedMode>(a, maps, ctas, pl.tiles, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attention(const AttnProblem &p, void *workspace, cudaStream_t stream) {
    const bool shared = !p.ring && p.mask_head_stride == 0;
    const int n_keys = p.ring ? ring_keys(p.ring_w) : p.n_keys;
    const Plan pl = make_plan(p.lanes, p.rows, p.n_heads, p.n_kv_heads, p.head_dim, n_keys, shared, p.ring);
    AttnArgs a{};
    a.q = p.q;
    a.q_f32 = p.q_is_f32 ? 1 : 0;
    a.q_row = p.q_row_stride;
    a.q_head = p.q_head_stride;
    a.q_lane = p.q_lane_stride;
    a.kv_bf16 = p.kv_dtype == GQA_DTYPE_BF16;
    a.mask = p.mask;
    a.mask_bf16 = p.mask_is_bf16 ? 1 : 0;
    a.m_row = p.mask_row_stride;
    a.m_head = p.mask_head_stride;
    a.m_lane = p.mask_lane_stride;
    a.o = p.o;
    a.o_row = p.o_row_stride;
    a.o_head = p.o_head_stride;
    a.o_lane = p.o_lane_stride;
    a.lanes = p.lanes;
    a.rows = p.rows;
    a.n_heads = p.n_heads;
    a.n_kv_heads = p.n_kv_heads;
    a.group = p.n_heads / p.n_kv_heads;
    a.n_keys = n_keys;
    a.ring = p.ring ? 1 : 0;
    a.ring_w = p.ring_w;
    a.ring_r = p.rows;
    a.cur_k = p.cur_k;
    a.cur_v = p.cur_v;
    a.ring_len = p.ring_len;
    a.ring_wp = p.ring_wp;
    a.rows_per_head = pl.rows_per_head;
    a.heads_per_tile = pl.heads_per_tile;
    a.row_tiles = pl.row_tiles;
    a.head_tiles = pl.head_tiles;
    a.tiles_total = pl.tiles;
    a.n_blk = pl.n_blk;
    a.splits = pl.splits;
    a.blk_per_split = pl.bps;
    a.d_parts = pl.d_parts;
    a.scale_log2 = p.scale * kLog2e;
    a.code_cols = pl.code_cols;
    a.shared_mask = shared ? 1 : 0;
    char *ws = static_cast<char *>(workspace);
    a.codes = reinterpret_cast<uint8_t *>(ws);
    a.ws_o = pl.splits > 1 ? reinterpret_cast<float *>(ws + pl.codes_bytes) : nullptr;
    a.ws_lse = pl.splits > 1 ? reinterpret_cast<float *>(ws + pl.codes_bytes + pl.part_o_bytes) : nullptr;
    a.vis_split = pl.vis_split ? 1 : 0;
    if (pl.sched_bytes) {
        char *sched = ws + pl.codes_bytes + pl.part_o_bytes + pl.part_lse_bytes;
        a.sched_counter = reinterpret_cast<int *>(sched);
        if (pl.vis_split) {
            a.queue_len = reinterpret_cast<int *>(sched + 4);
            a.lane_splits = reinterpret_cast<int *>(sched + 8);
            a.lane_start = reinterpret_cast<int *>(sched + 8 + 30 * 4);
            a.split_budget = pl.split_budget;
        } else {
            a.sched_perm = reinterpret_cast<const int *>(sched + 256);
        }
    }
    a.head_dim = p.head_dim;
    if (p.ring)
        a.cur16 = reinterpret_cast<uint16_t *>(ws + pl.codes_bytes + pl.part_o_bytes + pl.part_lse_bytes +
                                               pl.sched_bytes);
    a.status = p.status;

    // K, V (and, for single-head 128-row prefill tiles, f32 Q and O) tensor maps
    CUtensorMap maps[5];
    memset(maps, 0, sizeof maps);
    const int heads = p.lanes * p.n_kv_heads;
    const CUtensorMapDataType kvt =
        a.kv_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    a.k_rows_dim1 = rows_first(heads, p.k_row_stride, p.k_head_stride) ? 1 : 0;
    a.v_rows_dim1 = rows_first(heads, p.v_row_stride, p.v_head_stride) ? 1 : 0;
    // CTA pairs load K in boxes of 64 keys (each CTA half of a tile)
    if (!make_map(&maps[0], p.k, kvt, 2, p.head_dim, p.kv_rows, heads, p.k_row_stride,
                  p.k_head_stride, 64, pl.pair ? pl.bn / 2 : pl.bn) ||
        !make_map(&maps[1], p.v, kvt, 2, p.head_dim, p.kv_rows, heads, p.v_row_stride,
                  p.v_head_stride, 64, pl.bn))
        return cudaErrorInvalidValue;
    const bool single_head_tiles = p.lanes == 1 && pl.heads_per_tile == 1 && pl.rows_per_head == BM;
    if (single_head_tiles && p.q_is_f32 &&
        make_map(&maps[2], p.q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.head_dim, p.rows, p.n_heads,
                 p.q_row_stride, p.q_head_stride, 32, BM)) {
        a.q_tma = 1;
        a.q_rows_dim1 = rows_first(p.n_heads, p.q_row_stride, p.q_head_stride) ? 1 : 0;
    }
    // O out by TMA, staged where the next unit's f32 Q arrives (so only with Q by TMA)
    if (a.q_tma && pl.splits == 1 &&
        make_map(&maps[3], p.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.head_dim, p.rows, p.n_heads,
                 p.o_row_stride, p.o_head_stride, 32, BM)) {
        a.o_tma = 1;
        a.o_rows_dim1 = rows_first(p.n_heads, p.o_row_stride, p.o_head_stride) ? 1 : 0;
    }

    // ring-direct verify classifies its tiles from the history length and write position
    if (!p.ring) {
        classify_kernel<<<dim3(pl.code_groups, pl.code_cols), BM, 0, stream>>>(a, const_cast<uint8_t *>(a.codes));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // persistent launch: one CTA (or CTA pair) per SM (or SM pair) at most; each runs
    // the units of its slot back to back
    const int units = pl.tiles * pl.d_parts * pl.splits;  // query tiles x output halves x key splits
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    const int ctas = pl.pair ? 2 * std::min(units / 2, sms / 2) : std::min(units, sms);
    const bool bf = a.kv_bf16;
    if (p.ring) {
        // ring-direct verify: bf16 rings, head_dim 128 or 256, unpaired
        if (!bf || pl.pair) return cudaErrorInvalidValue;
        // key tile 0: the current rows in bf16, [K|V][lanes * kv heads][rows][head_dim], read
        // in boxes of 128 rows (the rows past `rows` are out of bounds: zeros)
        const int kvh = p.lanes * p.n_kv_heads;
        const size_t half = (size_t)kvh * p.rows * p.head_dim;
        if (!make_map(&maps[3], a.cur16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.head_dim, p.rows, 2 * kvh,
                      p.head_dim, (int64_t)p.rows * p.head_dim, 64, BM))
            return cudaErrorInvalidValue;
        // f32 Q [lanes][rows][heads][d] by TMA: a box of 128 / rows heads x rows x 32
        // columns lands as the tile's (head, row) rows in order (rows dividing 128)
        if (BM % p.rows == 0 && pl.heads_per_tile * p.rows <= BM) {
            auto fn = encode_fn();
            cuuint64_t dims[4] = {(cuuint64_t)p.head_dim, (cuuint64_t)p.rows, (cuuint64_t)p.n_heads,
                                  (cuuint64_t)p.lanes};
            cuuint64_t strides[3] = {(cuuint64_t)p.q_row_stride * 4, (cuuint64_t)p.q_head_stride * 4,
                                     (cuuint64_t)p.q_lane_stride * 4};
            cuuint32_t box[4] = {32, (cuuint32_t)p.rows, (cuuint32_t)(BM / p.rows), 1};
            cuuint32_t es[4] = {1, 1, 1, 1};
            if (fn && fn(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(p.q), dims, strides,
                         box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
                a.q_tma = 1;
        }
        const int64_t chunks = (int64_t)2 * half / 8;
        const int conv = (int)std::min<int64_t>(64, (chunks + 1023) / 1024);
        order_units_kernel<<<1 + conv, 1024, sizeof(int), stream>>>(a, units);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (p.head_dim == 128) return run_attn<128, BF16, false, kRingMode>(a, maps, ctas, pl.tiles, stream);
        if (p.head_dim == 256) return run_attn<256, BF16, false, kRingMode>(a, maps, ctas, pl.tiles, stream);
        return cudaErrorInvalidValue;
    }
    switch (p.head_dim) {
        case 128:
            return bf ? run_attn<128, BF16, false>(a, maps, ctas, pl.tiles, stream)
                      : run_attn<128, F16, false>(a, maps, ctas, pl.tiles, stream);
        case 256:
            if (pl.pair)
                return bf ? run_attn<256, BF16, true>(a, maps, ctas, pl.tiles, stream)
                          : run_attn<256, F16, true>(a, maps, ctas, pl.tiles, stream);
            return bf ? run_attn<256, BF16, false>(a, maps, ctas, pl.tiles, stream)
                      : run_attn<256, F16, false>(a, maps, ctas, pl.tiles, stream);
        case 512:
            if (pl.pair)
                return bf ? run_attn<512, BF16, true>(a, maps, ctas, pl.tiles, stream)
                          : run_attn<512, F16, true>(a, maps, ctas, pl.tiles, stream);
            return bf ? run_attn<512, BF16, false>(a, maps, ctas, pl.tiles, stream)
                      : run_attn<512, F16, false>(a, maps, ctas, pl.tiles, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace gqa
