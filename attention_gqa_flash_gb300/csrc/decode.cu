// decode.cu -- paged decode attention: split-KV (flash-decoding) over
// fixed-size pages, then a combine of the per-chunk partial results.
//
// Semantics follow ferrum-kernels 0.8.3 src/backend/metal/vnext_ops/causal_attention.rs:
// a sequence's KV stream is cut into fixed pages taken in logical order
// (paged_state_regions), each token holding K and V for every KV head
// (validate_signature), and the decode query attends to every context token.
//
// Design (HBM-bound: each context token's K and V rows are read exactly once):
//   * work unit = (sequence, KV head, 16-query-head group, 1024-token chunk:
//     larger chunks measured slower at 4096, smaller ones write and merge more
//     partial results);
//     a persistent grid walks the units chunk-major, skipping chunks past a
//     sequence's end without a launch;
//   * the CTA's 4 warps take interleaved 16-token sub-tiles; each warp gathers
//     its K and V rows with 16-byte cp.async (double buffered, XOR-swizzled
//     shared memory so ldmatrix is conflict-free);
//   * the GQA group is the M dimension of m16n8k16 mma.sync (rows = query
//     heads sharing the KV head), so every K/V element loaded serves all of
//     the group's query heads from registers;
//   * online softmax in the exp2 domain; warps merge in shared memory and
//     write one normalised partial (o, log2-sum-exp) per unit;
//   * a combine kernel merges a sequence's chunks, one warp per (seq, head).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace gqa {
namespace {

constexpr int kWarps = 4;
constexpr int kSub = 16;                // tokens per warp step
constexpr int kChunk = 1024;            // tokens per work unit
constexpr float kNegInf = -INFINITY;

struct DecodeArgs {
    const float *q;
    const uint16_t *k_pool;
    const uint16_t *v_pool;
    int64_t page_stride, token_stride, head_stride;
    const int32_t *page_table;
    int max_pages;
    const int32_t *context_lens;
    int num_seqs, n_heads, n_kv_heads, group, head_groups, page_size, num_pages, max_chunks;
    int max_ctx;
    float scale_log2;
    float *ws_o;    // [S][max_chunks][H][D]
    float *ws_lse;  // [S][max_chunks][H]
    float *o;
    int32_t *status;
};

template <int D>
struct Smem {
    static constexpr int kTile = kSub * D;           // halves in one K (or V) sub-tile
    static constexpr int kWarpHalves = 2 * 2 * kTile;  // 2 stages x (K, V)
    static constexpr int kMergeStride = D + 4;       // floats per merged row
    static constexpr size_t kQ = 16 * D * 2;
    static constexpr size_t kKV = (size_t)kWarps * kWarpHalves * 2;
    static constexpr size_t kMerge = (size_t)kWarps * 16 * (kMergeStride + 2) * 4;
    static constexpr size_t kBytes = kQ + (kKV > kMerge ? kKV : kMerge);
};

// element offset of (row, 16-byte chunk) in a swizzled [rows][D] half tile
template <int D>
__device__ __forceinline__ int swz(int row, int chunk) {
    return row * D + ((chunk ^ (row & 7)) << 3);
}

__device__ __forceinline__ int clamp_ctx(const DecodeArgs &a, int s) {
    int ctx = a.context_lens[s];
    return ctx < 0 ? 0 : (ctx > a.max_ctx ? a.max_ctx : ctx);
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <class KV, int D>
__global__ void __launch_bounds__(kWarps * 32) paged_decode_kernel(const DecodeArgs a) {
    using S = Smem<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t *sq = reinterpret_cast<uint16_t *>(smem);
    uint16_t *skv = reinterpret_cast<uint16_t *>(smem + S::kQ);
    float *smerge = reinterpret_cast<float *>(smem + S::kQ);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint16_t *mine = skv + warp * S::kWarpHalves;
    const int per_chunk = a.num_seqs * a.n_kv_heads * a.head_groups;
    const int units = per_chunk * a.max_chunks;

    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int c = u / per_chunk;
        const int rest = u - c * per_chunk;
        const int s = rest / (a.n_kv_heads * a.head_groups);
        const int khg = rest - s * (a.n_kv_heads * a.head_groups);
        const int kh = khg / a.head_groups;
        const int hg = khg - kh * a.head_groups;
        const int ctx = clamp_ctx(a, s);
        const int t0 = c * kChunk;
        if (t0 >= ctx) continue;  // uniform over the CTA
        const int t1 = min(t0 + kChunk, ctx);
        const int rows = min(16, a.group - hg * 16);
        const int h0 = kh * a.group + hg * 16;

        __syncthreads();  // the previous unit's merge is done with shared memory
        // Q tile: 16 rows (query heads) x D, rows >= `rows` zero, rounded to KV's type.
        for (int i = threadIdx.x; i < 16 * (D / 8); i += kWarps * 32) {
            const int r = i / (D / 8), ch = i % (D / 8);
            uint4 val = make_uint4(0, 0, 0, 0);
            if (r < rows) {
                const float *src = a.q + ((int64_t)s * a.n_heads + h0 + r) * D + ch * 8;
                const float4 x = ld_nc_f4(src), y = ld_nc_f4(src + 4);
                val = make_uint4(pack2(KV{}, x.x, x.y), pack2(KV{}, x.z, x.w),
                                 pack2(KV{}, y.x, y.y), pack2(KV{}, y.z, y.w));
            }
            *reinterpret_cast<uint4 *>(sq + swz<D>(r, ch)) = val;
        }
        __syncthreads();

        const int nsub = (t1 - t0 + kSub - 1) / kSub;
        const int my_n = nsub > warp ? (nsub - warp + kWarps - 1) / kWarps : 0;

        // gather one 16-token sub-tile of K and V into stage `stage`
        auto issue = [&](int j, int stage) {
            const int tb = t0 + kSub * (warp + kWarps * j);
            int64_t off = 0;
            int valid = 0;
            if (lane < kSub) {
                const int t = tb + lane;
                if (t < t1) {
                    int page = a.page_table[(int64_t)s * a.max_pages + t / a.page_size];
                    if (page < 0 || page >= a.num_pages) {
                        raise_flag(a.status, GQA_FLAG_PAGE_CLAMPED);
                        page = page < 0 ? 0 : a.num_pages - 1;
                    }
                    off = (int64_t)page * a.page_stride + (int64_t)(t % a.page_size) * a.token_stride +
                          (int64_t)kh * a.head_stride;
                    valid = 1;
                }
            }
            uint16_t *kt = mine + stage * 2 * S::kTile;
            uint16_t *vt = kt + S::kTile;
#pragma unroll
            for (int q = 0; q < (kSub * D / 8) / 32; ++q) {
                const int i = lane + 32 * q;
                const int t = i / (D / 8), ch = i % (D / 8);
                const int64_t o = __shfl_sync(0xffffffffu, off, t);
                const int ok = __shfl_sync(0xffffffffu, valid, t);
                const int e = swz<D>(t, ch);
                cp_async16(smem_u32(kt + e), ok ? a.k_pool + o + ch * 8 : a.k_pool, ok ? 16 : 0);
                cp_async16(smem_u32(vt + e), ok ? a.v_pool + o + ch * 8 : a.v_pool, ok ? 16 : 0);
            }
        };

        float acc[D / 8][4];
#pragma unroll
        for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;

        if (my_n > 0) issue(0, 0);
        cp_async_commit();
        if (my_n > 1) issue(1, 1);
        cp_async_commit();
        for (int j = 0; j < my_n; ++j) {
            cp_async_wait<1>();
            __syncwarp();
            const int stage = j & 1;
            const uint16_t *kt = mine + stage * 2 * S::kTile;
            const uint16_t *vt = kt + S::kTile;
            const int tb = t0 + kSub * (warp + kWarps * j);

            // S = Q K^T for 16 tokens (two n-tiles of 8)
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kc = 0; kc < D / 16; ++kc) {
                uint32_t qa[4], kb[4];
                ldsm_x4(smem_u32(sq + swz<D>(((lane >> 3) & 1) * 8 + (lane & 7), kc * 2 + (lane >> 4))),
                        qa[0], qa[1], qa[2], qa[3]);
                ldsm_x4(smem_u32(kt + swz<D>((lane >> 4) * 8 + (lane & 7), kc * 2 + ((lane >> 3) & 1))),
                        kb[0], kb[1], kb[2], kb[3]);
                mma16816(KV{}, sc[0], qa, kb[0], kb[1]);
                mma16816(KV{}, sc[1], qa, kb[2], kb[3]);
            }
            // online softmax (log2 domain); rows g and g+8 of this lane's quad
            float x[2][4];
            float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = tb + nt * 8 + (lane & 3) * 2 + (e & 1);
                    x[nt][e] = t < t1 ? sc[nt][e] * a.scale_log2 : kNegInf;
                    if (e < 2)
                        mx0 = fmaxf(mx0, x[nt][e]);
                    else
                        mx1 = fmaxf(mx1, x[nt][e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float u0 = n0 == kNegInf ? 0.f : n0, u1 = n1 == kNegInf ? 0.f : n1;
            const float al0 = ex2(m0 - u0), al1 = ex2(m1 - u1);
            m0 = n0;
            m1 = n1;
            float p[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) p[nt][e] = ex2(x[nt][e] - (e < 2 ? u0 : u1));
            l0 = l0 * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
            l1 = l1 * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                acc[n][0] *= al0;
                acc[n][1] *= al0;
                acc[n][2] *= al1;
                acc[n][3] *= al1;
            }
            const uint32_t pa[4] = {pack2(KV{}, p[0][0], p[0][1]), pack2(KV{}, p[0][2], p[0][3]),
                                    pack2(KV{}, p[1][0], p[1][1]), pack2(KV{}, p[1][2], p[1][3])};
            // O += P V
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj) {
                uint32_t vb[4];
                ldsm_x4_t(smem_u32(vt + swz<D>(((lane >> 3) & 1) * 8 + (lane & 7), jj * 2 + (lane >> 4))),
                          vb[0], vb[1], vb[2], vb[3]);
                mma16816(KV{}, acc[2 * jj], pa, vb[0], vb[1]);
                mma16816(KV{}, acc[2 * jj + 1], pa, vb[2], vb[3]);
            }
            __syncwarp();
            if (j + 2 < my_n) issue(j + 2, stage);
            cp_async_commit();
        }
        cp_async_wait<0>();
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

        __syncthreads();  // every warp is done with its K/V stages
        {
            float *mo = smerge + warp * 16 * S::kMergeStride;
            float *ml = smerge + kWarps * 16 * S::kMergeStride + warp * 32;
            const int g = lane >> 2, cq = lane & 3;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                mo[g * S::kMergeStride + n * 8 + cq * 2] = acc[n][0];
                mo[g * S::kMergeStride + n * 8 + cq * 2 + 1] = acc[n][1];
                mo[(g + 8) * S::kMergeStride + n * 8 + cq * 2] = acc[n][2];
                mo[(g + 8) * S::kMergeStride + n * 8 + cq * 2 + 1] = acc[n][3];
            }
            if (cq == 0) {
                ml[2 * g] = m0;
                ml[2 * g + 1] = l0;
                ml[2 * (g + 8)] = m1;
                ml[2 * (g + 8) + 1] = l1;
            }
        }
        __syncthreads();
        const float *ml_all = smerge + kWarps * 16 * S::kMergeStride;
        for (int i = threadIdx.x; i < rows * D; i += kWarps * 32) {
            const int r = i / D, d = i - (i / D) * D;
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml_all[w * 32 + 2 * r]);
            float L = 0.f, O = 0.f;
            if (M != kNegInf) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float f = ex2(ml_all[w * 32 + 2 * r] - M);
                    L += f * ml_all[w * 32 + 2 * r + 1];
                    O += f * smerge[(w * 16 + r) * S::kMergeStride + d];
                }
            }
            const int64_t part = ((int64_t)s * a.max_chunks + c) * a.n_heads + h0 + r;
            a.ws_o[part * D + d] = L > 0.f ? O / L : 0.f;
            if (d == 0) a.ws_lse[part] = L > 0.f ? M + lg2(L) : kNegInf;
        }
    }
}

// One warp per (sequence, query head): merge the sequence's chunk partials.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a) {
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= a.num_seqs * a.n_heads) return;
    const int s = wid / a.n_heads, h = wid - (wid / a.n_heads) * a.n_heads;
    const int raw = a.context_lens[s];
    if (h == 0 && lane == 0 && (raw < 0 || raw > a.max_ctx))
        raise_flag(a.status, GQA_FLAG_CONTEXT_CLAMPED);
    const int ctx = clamp_ctx(a, s);
    const int nch = (ctx + kChunk - 1) / kChunk;
    const int64_t base = (int64_t)s * a.max_chunks * a.n_heads + h;
    float M = kNegInf;
    for (int i = lane; i < nch; i += 32) M = fmaxf(M, a.ws_lse[base + (int64_t)i * a.n_heads]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] = 0.f;
    float L = 0.f;
    if (M != kNegInf) {
        for (int i = 0; i < nch; ++i) {
            const int64_t part = base + (int64_t)i * a.n_heads;
            const float w = ex2(a.ws_lse[part] - M);
            L += w;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) acc[k] += w * a.ws_o[part * D + lane + 32 * k];
        }
    }
    float *out = a.o + ((int64_t)s * a.n_heads + h) * D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) out[lane + 32 * k] = L > 0.f ? acc[k] / L : 0.f;
}

template <class KV, int D>
cudaError_t run(const DecodeArgs &a, cudaStream_t stream) {
    const size_t smem = Smem<D>::kBytes;
    auto kern = paged_decode_kernel<KV, D>;
    // resident CTAs per SM for this instantiation, per device (function attributes
    // belong to each device's context)
    static DeviceSetup setup;
    static int occ_of[DeviceSetup::kMaxDevices] = {0};
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    if (dev < 0 || dev >= DeviceSetup::kMaxDevices) return cudaErrorInvalidDevice;
    de = setup.run([&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWarps * 32, smem);
        if (e != cudaSuccess) return e;
        occ_of[dev] = occ < 1 ? 1 : occ;
        return cudaSuccess;
    });
    if (de != cudaSuccess) return de;
    const int occ = occ_of[dev];
    const int64_t units = (int64_t)a.num_seqs * a.n_kv_heads * a.head_groups * a.max_chunks;
    int64_t grid = (int64_t)sm_count() * occ;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    timing_mark(true, stream);
    kern<<<(int)grid, kWarps * 32, smem, stream>>>(a);
    timing_mark(false, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int warps = a.num_seqs * a.n_heads;
    decode_combine_kernel<D><<<(warps + 3) / 4, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

static int max_chunks_of(int max_pages_per_seq, int page_size) {
    const int64_t max_ctx = (int64_t)max_pages_per_seq * page_size;
    return (int)((max_ctx + kChunk - 1) / kChunk);
}

size_t decode_workspace_bytes(int num_seqs, int n_heads, int head_dim, int max_pages_per_seq,
                              int page_size) {
    const size_t parts = (size_t)num_seqs * max_chunks_of(max_pages_per_seq, page_size) * n_heads;
    const size_t o_bytes = (parts * head_dim * 4 + 255) / 256 * 256;
    return o_bytes + (parts * 4 + 255) / 256 * 256;
}

cudaError_t launch_paged_decode(const DecodeProblem &p, void *workspace, cudaStream_t stream) {
    DecodeArgs a;
    a.q = p.q;
    a.k_pool = static_cast<const uint16_t *>(p.k_pool);
    a.v_pool = static_cast<const uint16_t *>(p.v_pool);
    a.page_stride = p.page_stride;
    a.token_stride = p.token_stride;
    a.head_stride = p.head_stride;
    a.page_table = p.page_table;
    a.max_pages = p.max_pages_per_seq;
    a.context_lens = p.context_lens;
    a.num_seqs = p.num_seqs;
    a.n_heads = p.n_heads;
    a.n_kv_heads = p.n_kv_heads;
    a.group = p.n_heads / p.n_kv_heads;
    a.head_groups = (a.group + 15) / 16;
    a.page_size = p.page_size;
    a.num_pages = p.num_pages;
    a.max_chunks = max_chunks_of(p.max_pages_per_seq, p.page_size);
    a.max_ctx = (int)((int64_t)p.max_pages_per_seq * p.page_size);
    a.scale_log2 = p.scale * kLog2e;
    const size_t parts = (size_t)p.num_seqs * a.max_chunks * p.n_heads;
    a.ws_o = static_cast<float *>(workspace);
    a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                         (parts * p.head_dim * 4 + 255) / 256 * 256);
    a.o = p.o;
    a.status = p.status;
    const bool bf = p.kv_dtype == GQA_DTYPE_BF16;
    switch (p.head_dim) {
        case 64: return bf ? run<BF16, 64>(a, stream) : run<F16, 64>(a, stream);
        case 128: return bf ? run<BF16, 128>(a, stream) : run<F16, 128>(a, stream);
        case 256: return bf ? run<BF16, 256>(a, stream) : run<F16, 256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gqa

// ---------------------------------------------------------------------------
// Fixed scratch for gqa_attn_paged_decode_noalloc: callers that cannot give the
// library a device buffer get the split-KV partials kept here instead.  The
// array is part of the library's device image; its device address is looked
// up with the device current and cached per device, together with the
// identity of the context it was looked up in: a device reset destroys that
// context (and the module holding the array), so an address cached before the
// reset is never handed out after it -- the next call looks it up again.
// ---------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace gqa {
namespace {
static __device__ __align__(256) unsigned char g_decode_fixed_scratch[GQA_NOALLOC_SCRATCH_BYTES];
std::mutex g_fixed_scratch_mu;
constexpr int kMaxDevices = 64;
void *g_fixed_scratch_addr[kMaxDevices] = {nullptr};
unsigned long long g_fixed_scratch_ctx[kMaxDevices] = {0};

}  // namespace

cudaError_t decode_fixed_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_fixed_scratch_addr[dev] || ctx == 0 || ctx != g_fixed_scratch_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_fixed_scratch);
        if (e != cudaSuccess) return e;
        g_fixed_scratch_addr[dev] = p;
        // the lookup makes the device's primary context current if it was not yet
        g_fixed_scratch_ctx[dev] = current_context_id();
    }
    *ptr = g_fixed_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace gqa
