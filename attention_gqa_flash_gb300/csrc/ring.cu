// ring.cu -- DFlash2 ring-KV kernels: pack, mask, commit, draft mask rows.
//
// Layouts and semantics follow mlx-native 0.21.1 src/ops/dflash2_attention_pack.rs
// (dispatch_dflash2_pack_attention_bf16, dispatch_dflash2_attention_mask_bf16,
// dispatch_dflash2_commit_kv_bf16, dispatch_dflash2_mask_rows_f32 and the worked
// example in gpu_pack_mask_and_commit_match_ring_semantics).
//
// All four are pure data movement: every thread moves 16 bytes of output
// (8 bf16) with 16-byte loads/stores, so each warp touches whole 128-byte
// lines.  Grids are sized to a few waves of the SM count and stride over
// the work.
#include "common.cuh"
#include "launch.h"

namespace gqa {

struct RingGeom {
    int B, H, HK, D, R, W, K, MC;
};

// Clamp the two ring counters of lane b; report when they were out of range.
__device__ __forceinline__ void ring_counters(const uint32_t *cache_lengths,
                                              const uint32_t *write_positions, int b, int W,
                                              int32_t *status, int &len, int &wp) {
    uint32_t l = cache_lengths[b];
    uint32_t p = write_positions ? write_positions[b] : 0u;
    if (l > (uint32_t)W || p >= (uint32_t)W) raise_flag(status, GQA_FLAG_RING_CLAMPED);
    len = l > (uint32_t)W ? W : (int)l;
    wp = (int)(p % (uint32_t)W);
}

__device__ __forceinline__ uint4 f32x8_to_bf16x8(const float *src) {
    float4 a = ld_nc_f4(src);
    float4 b = ld_nc_f4(src + 4);
    return make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                      pack_bf16x2(b.z, b.w));
}

// Grid row y < B*HK packs the K/V columns of (lane, KV head) y; grid row
// B*HK + (b*H + qh) packs the query rows of head qh of lane b.  Within a grid
// row every thread moves one 8-element chunk (16 bytes of output) per step, so
// the index arithmetic is 32-bit with a compile-time chunk count.
template <int D>
__global__ void __launch_bounds__(256) pack_attention_kernel(
    const uint16_t *__restrict__ ring_k, const uint16_t *__restrict__ ring_v,
    const float *__restrict__ cur_q, const float *__restrict__ cur_k,
    const float *__restrict__ cur_v, const uint32_t *__restrict__ cache_lengths,
    const uint32_t *__restrict__ write_positions, uint16_t *__restrict__ packed_q,
    uint16_t *__restrict__ packed_k, uint16_t *__restrict__ packed_v, RingGeom g,
    int32_t *status) {
    constexpr int chunks = D / 8;
    const int y = blockIdx.y;
    const int step = gridDim.x * blockDim.x;
    if (y < g.B * g.HK) {
        const int b = y / g.HK, kh = y - (y / g.HK) * g.HK;
        int len, wp;
        ring_counters(cache_lengths, write_positions, b, g.W,
                      blockIdx.x == 0 && threadIdx.x == 0 ? status : nullptr, len, wp);
        const uint16_t *rk = ring_k + (int64_t)y * g.W * D;
        const uint16_t *rv = ring_v + (int64_t)y * g.W * D;
        uint16_t *pk = packed_k + (int64_t)y * g.K * D;
        uint16_t *pv = packed_v + (int64_t)y * g.K * D;
        const int work = g.K * chunks;
        for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < work; u += step) {
            const int c = u / chunks, ch = u % chunks;
            uint4 vk, vv;
            if (c < g.R) {
                const int64_t src = (((int64_t)b * g.R + c) * g.HK + kh) * D + ch * 8;
                vk = f32x8_to_bf16x8(cur_k + src);
                vv = f32x8_to_bf16x8(cur_v + src);
            } else if (c - g.R < len) {
                int slot = wp - 1 - (c - g.R);
                slot += (slot < 0) ? g.W : 0;
                vk = ld_nc_v4(rk + (int64_t)slot * D + ch * 8);
                vv = ld_nc_v4(rv + (int64_t)slot * D + ch * 8);
            } else {
                vk = make_uint4(0, 0, 0, 0);
                vv = vk;
            }
            st_v4(pk + (int64_t)u * 8, vk);
            st_v4(pv + (int64_t)u * 8, vv);
        }
    } else {
        const int bq = y - g.B * g.HK;  // b * H + qh
        const int b = bq / g.H, qh = bq - (bq / g.H) * g.H;
        const int work = g.R * chunks;
        for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < work; u += step) {
            const int r = u / chunks, ch = u % chunks;
            const int64_t src = (((int64_t)b * g.R + r) * g.H + qh) * D + ch * 8;
            st_v4(packed_q + ((int64_t)bq * g.R + r) * D + ch * 8, f32x8_to_bf16x8(cur_q + src));
        }
    }
}

// Mask: every row (b, h, r) of the [B][H][R][K] array is a threshold: columns
// c < R + min(len_b, W-1-r) are visible (the draft rows, then the history entries
// inside the window), the rest are hidden.
template <typename IDX>
__device__ __forceinline__ int mask_threshold(const uint32_t *cache_lengths, const RingGeom &g,
                                              IDX row) {
    const int r = (int)(row % g.R);
    const int b = (int)(row / ((IDX)g.H * g.R));
    const uint32_t l = cache_lengths[b];
    const int len = l > (uint32_t)g.W ? g.W : (int)l;
    const int hist = len < g.W - 1 - r ? len : g.W - 1 - r;
    return g.R + (hist > 0 ? hist : 0);
}

// One warp per mask row (b, h, r): the row is a threshold, so a lane writes 16-byte
// chunks of eight 0 / -inf values with no per-element index arithmetic; the few
// elements before the row's first 16-byte boundary and after its last one (a row of
// K bf16 values starts wherever row * K puts it) are written one by one.
__global__ void __launch_bounds__(256) fill_mask_kernel(const uint32_t *__restrict__ cache_lengths,
                                                        uint16_t *__restrict__ mask, RingGeom g,
                                                        int32_t *status) {
    const int64_t rows = (int64_t)g.B * g.H * g.R;
    if (blockIdx.x == 0 && threadIdx.x < g.B) {
        if (cache_lengths[threadIdx.x] > (uint32_t)g.W) raise_flag(status, GQA_FLAG_RING_CLAMPED);
    }
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); row < rows;
         row += warps) {
        const int thr = mask_threshold<int64_t>(cache_lengths, g, row);
        uint16_t *m = mask + row * g.K;
        const int head = (int)((8 - ((row * g.K) & 7)) & 7);  // elements before a 16-byte boundary
        const int n = g.K;
        const int lead = head < n ? head : n;
        if (lane < lead) m[lane] = lane < thr ? 0x0000u : 0xff80u;
        const int body = (n - lead) / 8;
        for (int c = lane; c < body; c += 32) {
            const int col0 = lead + c * 8;
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = (col0 + 2 * i < thr ? 0x0000u : 0xff80u) |
                       ((col0 + 2 * i + 1 < thr ? 0x0000u : 0xff80u) << 16);
            st_v4(m + col0, make_uint4(w[0], w[1], w[2], w[3]));
        }
        const int col = lead + body * 8 + lane;
        if (col < n) m[col] = col < thr ? 0x0000u : 0xff80u;
    }
}

// Commit: one thread per 8-element chunk of an offered (lane, row, kv head).
__global__ void __launch_bounds__(256) commit_kv_kernel(
    const float *__restrict__ new_k, const float *__restrict__ new_v,
    const uint32_t *__restrict__ commit_counts, const uint32_t *__restrict__ write_positions,
    uint16_t *__restrict__ ring_k, uint16_t *__restrict__ ring_v, RingGeom g, int32_t *status) {
    const int chunks = g.D / 8;
    const int64_t work = (int64_t)g.B * g.MC * g.HK * chunks;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < work; t += stride) {
        const int ch = (int)(t % chunks);
        const int64_t rest = t / chunks;
        const int kh = (int)(rest % g.HK);
        const int64_t bi = rest / g.HK;
        const int i = (int)(bi % g.MC);
        const int b = (int)(bi / g.MC);
        // the offered row's data first (every offered row is in bounds): its loads are in
        // flight while the counters are read
        const int64_t src = rest * g.D + ch * 8;
        const float4 k0 = ld_nc_f4(new_k + src), k1 = ld_nc_f4(new_k + src + 4);
        const float4 v0 = ld_nc_f4(new_v + src), v1 = ld_nc_f4(new_v + src + 4);
        const uint32_t cnt = commit_counts[b];
        const uint32_t pos = write_positions[b];
        if (i == 0 && kh == 0 && ch == 0 && (cnt > (uint32_t)g.MC || pos >= (uint32_t)g.W))
            raise_flag(status, GQA_FLAG_RING_CLAMPED);
        const int n = cnt > (uint32_t)g.MC ? g.MC : (int)cnt;
        if (i >= n) continue;
        const int slot = (int)((pos % (uint32_t)g.W + (uint32_t)i) % (uint32_t)g.W);
        const int64_t dst = (((int64_t)b * g.HK + kh) * g.W + slot) * g.D + ch * 8;
        st_v4(ring_k + dst, make_uint4(pack_bf16x2(k0.x, k0.y), pack_bf16x2(k0.z, k0.w),
                                       pack_bf16x2(k1.x, k1.y), pack_bf16x2(k1.z, k1.w)));
        st_v4(ring_v + dst, make_uint4(pack_bf16x2(v0.x, v0.y), pack_bf16x2(v0.z, v0.w),
                                       pack_bf16x2(v1.x, v1.y), pack_bf16x2(v1.z, v1.w)));
    }
}

// Draft mask rows: rows 1..R-1 of every lane become the widened embedding.
__global__ void __launch_bounds__(256) set_mask_rows_kernel(const uint16_t *__restrict__ emb,
                                                            float *__restrict__ hidden, int lanes,
                                                            int rows, int width) {
    const int64_t work = (int64_t)lanes * (rows - 1) * width;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < work; t += stride) {
        const int e = (int)(t % width);
        const int64_t lr = t / width;
        const int r = 1 + (int)(lr % (rows - 1));
        const int l = (int)(lr / (rows - 1));
        hidden[((int64_t)l * rows + r) * width + e] = __uint_as_float((uint32_t)emb[e] << 16);
    }
}

static int grid_for(int64_t work, int sms) {
    int64_t blocks = (work + 255) / 256;
    int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

static RingGeom geom_of(const gqa_ring_params &p) {
    return RingGeom{(int)p.lanes, (int)p.q_heads,  (int)p.kv_heads,   (int)p.head_dim,
                    (int)p.rows,  (int)p.window,   (int)p.packed_len, (int)p.max_commit};
}

cudaError_t launch_pack_attention(const uint16_t *ring_k, const uint16_t *ring_v,
                                  const float *cur_q, const float *cur_k, const float *cur_v,
                                  const uint32_t *cache_lengths, const uint32_t *write_positions,
                                  uint16_t *packed_q, uint16_t *packed_k, uint16_t *packed_v,
                                  const gqa_ring_params &p, int32_t *status, cudaStream_t stream) {
    RingGeom g = geom_of(p);
    // x blocks per slab: the K/V slabs (nearly all the bytes) alone get about 8
    // CTAs per SM, and no slab gets more than one chunk per thread
    const int slabs = g.B * g.HK + g.B * g.H;
    const int per_slab = (int)(((int64_t)g.K * (g.D / 8) + 255) / 256);
    int bx = (sm_count() * 8 + g.B * g.HK - 1) / (g.B * g.HK);
    if (bx > per_slab) bx = per_slab;
    if (bx < 1) bx = 1;
    const dim3 grid(bx, slabs);
    timing_mark(true, stream);
    if (g.D == 128)
        pack_attention_kernel<128><<<grid, 256, 0, stream>>>(ring_k, ring_v, cur_q, cur_k, cur_v,
                                                             cache_lengths, write_positions, packed_q,
                                                             packed_k, packed_v, g, status);
    else
        pack_attention_kernel<256><<<grid, 256, 0, stream>>>(ring_k, ring_v, cur_q, cur_k, cur_v,
                                                             cache_lengths, write_positions, packed_q,
                                                             packed_k, packed_v, g, status);
    timing_mark(false, stream);
    return cudaGetLastError();
}

cudaError_t launch_fill_mask(const uint32_t *cache_lengths, uint16_t *mask,
                             const gqa_ring_params &p, int32_t *status, cudaStream_t stream) {
    RingGeom g = geom_of(p);
    // one warp per row, eight warps per block, at most 8 blocks per SM
    const int64_t rows = (int64_t)g.B * g.H * g.R;
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    timing_mark(true, stream);
    fill_mask_kernel<<<(int)(blocks < 1 ? 1 : blocks), 256, 0, stream>>>(cache_lengths, mask, g, status);
    timing_mark(false, stream);
    return cudaGetLastError();
}

cudaError_t launch_commit_kv(const float *new_k, const float *new_v, const uint32_t *commit_counts,
                             const uint32_t *write_positions, uint16_t *ring_k, uint16_t *ring_v,
                             const gqa_ring_params &p, int32_t *status, cudaStream_t stream) {
    RingGeom g = geom_of(p);
    int64_t work = (int64_t)g.B * g.MC * g.HK * (g.D / 8);
    timing_mark(true, stream);
    commit_kv_kernel<<<grid_for(work, sm_count()), 256, 0, stream>>>(
        new_k, new_v, commit_counts, write_positions, ring_k, ring_v, g, status);
    timing_mark(false, stream);
    return cudaGetLastError();
}

cudaError_t launch_set_mask_rows(const uint16_t *emb, float *hidden, int lanes, int rows,
                                 int width, cudaStream_t stream) {
    int64_t work = (int64_t)lanes * (rows - 1) * width;
    timing_mark(true, stream);
    set_mask_rows_kernel<<<grid_for(work, sm_count()), 256, 0, stream>>>(emb, hidden, lanes, rows,
                                                                          width);
    timing_mark(false, stream);
    return cudaGetLastError();
}

}  // namespace gqa
