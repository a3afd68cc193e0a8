// moe.cu -- dispatch and combine of the routed ReLU^2 expert block ("Nemotron
// Kernels From Inference To Backpropagation" -- "Kernel 4: Routed ReLU2 MoE":
// select, execute, weight and combine; the backward returns d_hidden,
// d_routing_weights, d_expert_up and d_expert_down; the dispatch is held fixed).
//
// The (token, slot) assignments of each expert are laid out back to back in
// token order, each expert's segment padded to a multiple of 256 rows, so the
// experts' GEMMs run as grouped GEMMs over one row space (gemm_tc.cuh, M- and
// K-grouped).  Every order is fixed: ranks follow (token, slot) order, the
// combine and the RMSNorm backward's dn gather (rowops.cu) add slots in slot
// order.
#include "mlpblk_internal.h"

namespace mlpblk {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kSegPad = 256;
constexpr int kZeroChunkFloats = 2048;  // one warp item of the dout kernel's gradient clearing
constexpr int kChunk = kMoeRouteChunk;  // routing entries per CTA (8 warps x 128)
constexpr int kMaxExperts = 256;

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack8(uint4 u, float (&v)[8]) {
    v[0] = bf16f(u.x & 0xFFFFu); v[1] = bf16f(u.x >> 16);
    v[2] = bf16f(u.y & 0xFFFFu); v[3] = bf16f(u.y >> 16);
    v[4] = bf16f(u.z & 0xFFFFu); v[5] = bf16f(u.z >> 16);
    v[6] = bf16f(u.w & 0xFFFFu); v[7] = bf16f(u.w >> 16);
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}

// Routing runs in two launches over chunks of kChunk (token, slot) entries:
// route_count (one CTA per chunk: the chunk's entries per expert) and route_place
// (one CTA per chunk: the counts' prefix and the padded segment offsets, then
// every entry's rank in (token, slot) order, its row, and the row -> (token,
// slot) map).

// chunk_count[b][e] = entries of chunk b with idx == e.  Entries outside
// [0, experts) belong to no expert.
__global__ void __launch_bounds__(kRouteThreads)
route_count_kernel(const int *__restrict__ idx, int64_t n, int experts, int *__restrict__ chunk_count) {
    __shared__ int cnt[kMaxExperts];
    griddep_enter();
    for (int e = threadIdx.x; e < experts; e += kRouteThreads) cnt[e] = 0;
    __syncthreads();
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int64_t i1 = min(n, i0 + kChunk);
    for (int64_t i = i0 + threadIdx.x; i < i1; i += kRouteThreads) {
        const int e = idx[i];
        if (e >= 0 && e < experts) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < experts; e += kRouteThreads)
        chunk_count[static_cast<int64_t>(blockIdx.x) * experts + e] = cnt[e];
}

// CTA b places chunk b.  It first adds up the chunk counts itself: the entries of
// each expert in the chunks before b (its first rank in this chunk) and in all
// chunks (the expert's count), then lays out the padded segments (CTA 0 publishes
// them).  Warp w walks its kChunk/8 entries in groups of 32 in order; lanes with
// the same expert (match_any) take consecutive ranks, so an entry's rank counts
// the entries of its expert before it in (token, slot) order.  pos[i] = seg[e] +
// rank (-1 for an entry that selects nothing), row_token / row_slot of that row;
// padding rows get row_token = -1.
__global__ void __launch_bounds__(kRouteThreads)
route_place_kernel(const int *__restrict__ idx, int64_t n, int k, int experts, int chunks,
                   const int *__restrict__ chunk_count, int *__restrict__ count, int *__restrict__ seg,
                   int *__restrict__ pos, int *__restrict__ row_token, int *__restrict__ row_slot) {
    constexpr int kWarps = kRouteThreads / 32;
    constexpr int kPerWarp = kChunk / kWarps;
    __shared__ int wcnt[kWarps][kMaxExperts];
    __shared__ int cbase[kMaxExperts];
    __shared__ int tot[kMaxExperts];
    __shared__ int segs[kMaxExperts + 1];
    griddep_enter();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kWarps * experts; i += kRouteThreads) wcnt[i / experts][i % experts] = 0;
    for (int e = threadIdx.x; e < experts; e += kRouteThreads) {
        int before = 0, all = 0;
        for (int b = 0; b < chunks; ++b) {
            const int c = chunk_count[static_cast<int64_t>(b) * experts + e];
            if (b < static_cast<int>(blockIdx.x)) before += c;
            all += c;
        }
        cbase[e] = before;
        tot[e] = all;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int off = 0;
        for (int e = 0; e < experts; ++e) {
            segs[e] = off;
            off += (tot[e] + kSegPad - 1) / kSegPad * kSegPad;
        }
        segs[experts] = off;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= experts; e += kRouteThreads) {
            seg[e] = segs[e];
            if (e < experts) count[e] = tot[e];
        }
    }
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kChunk + wid * kPerWarp;
    const unsigned lt = (1u << lane) - 1u;
    // pass 1: this warp's entries per expert
    for (int g = 0; g < kPerWarp; g += 32) {
        const int64_t i = w0 + g + lane;
        int e = i < n ? idx[i] : -1;
        if (e < 0 || e >= experts) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & lt) == 0) wcnt[wid][e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // the warp's first rank per expert: the chunk's, plus the warps before it
    for (int e = threadIdx.x; e < experts; e += kRouteThreads) {
        int run = cbase[e];
        for (int w = 0; w < kWarps; ++w) {
            const int c = wcnt[w][e];
            wcnt[w][e] = run;
            run += c;
        }
    }
    __syncthreads();
    // pass 2: ranks in order
    for (int g = 0; g < kPerWarp; g += 32) {
        const int64_t i = w0 + g + lane;
        int e = i < n ? idx[i] : -1;
        if (e < 0 || e >= experts) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int base = e >= 0 ? wcnt[wid][e] : 0;
        __syncwarp();
        if (e >= 0 && (peers & lt) == 0) wcnt[wid][e] = base + __popc(peers);
        __syncwarp();
        if (i < n) {
            if (e < 0) {
                pos[i] = -1;
            } else {
                const int p = segs[e] + base + __popc(peers & lt);
                pos[i] = p;
                row_token[p] = static_cast<int>(i / k);
                row_slot[p] = static_cast<int>(i % k);
            }
        }
    }
    // padding rows: expert e's rows [seg[e] + count[e], seg[e + 1])
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kRouteThreads + threadIdx.x;
         q < static_cast<int64_t>(experts) * kSegPad; q += static_cast<int64_t>(gridDim.x) * kRouteThreads) {
        const int e = static_cast<int>(q / kSegPad);
        const int r = segs[e] + tot[e] + static_cast<int>(q % kSegPad);
        if (r < segs[e + 1]) {
            row_token[r] = -1;
            row_slot[r] = 0;
        }
    }
}

// One warp per row r of the expert row space: x_perm[r] = x[token] and
// rstd_perm[r] = rstd[token], zeros for padding rows.
__global__ void gather_rows_kernel(const uint16_t *__restrict__ x, const float *__restrict__ rstd,
                                   const int *__restrict__ row_token, const int *__restrict__ seg, int experts,
                                   int64_t d, uint16_t *__restrict__ x_perm, float *__restrict__ rstd_perm) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    const int64_t rows = seg[experts];
    for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows;
         r += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const int t = row_token[r];
#pragma unroll 4
        for (int64_t c = lane * 8; c < d; c += 256) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t >= 0) v = __ldg(reinterpret_cast<const uint4 *>(x + t * d + c));
            *reinterpret_cast<uint4 *>(x_perm + r * d + c) = v;
        }
        if (lane == 0) rstd_perm[r] = t >= 0 ? rstd[t] : 0.0f;
    }
}

// One warp per token: y[t] = x[t] + sum_j p[t,j] * o_perm[pos[t,j]] (slot order).
__global__ void combine_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ o_perm,
                               const float *__restrict__ p, const int *__restrict__ pos, int64_t T, int k,
                               int64_t d, uint16_t *__restrict__ y) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    for (int64_t t = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; t < T;
         t += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        for (int64_t c = lane * 8; c < d; c += 256) {
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int j = 0; j < k; ++j) {
                const int r = pos[t * k + j];
                if (r < 0) continue;
                float o[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(o_perm + r * d + c)), o);
                const float w = p[t * k + j];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += w * o[i];
            }
            float xv[8];
            unpack8(__ldg(reinterpret_cast<const uint4 *>(x + t * d + c)), xv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += xv[i];
            *reinterpret_cast<uint4 *>(y + t * d + c) = pack8(acc);
        }
    }
}

// One warp per (token, slot) entry i = t*k + j with row r = pos[i]:
//   dp[i] = <dy[t], o_perm[r]>  (lane sums, then a fixed shuffle tree),
//   do_perm[r] = p[i] * dy[t]   (bf16);
// dp[i] = 0 for an entry that selects nothing.  Warps past the entries zero the
// padding rows of do_perm (expert e's rows [seg[e] + count[e], seg[e + 1])).
__global__ void dout_kernel(const uint16_t *__restrict__ dy, const uint16_t *__restrict__ o_perm,
                            const float *__restrict__ p, const int *__restrict__ pos,
                            const int *__restrict__ count, const int *__restrict__ seg, int64_t n, int k,
                            int experts, int64_t d, float *__restrict__ dp, uint16_t *__restrict__ do_perm,
                            float *__restrict__ dw1s, float *__restrict__ dw2s, int64_t ffn) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    const int64_t pad_end = n + static_cast<int64_t>(experts) * kSegPad;
    // overwrite: the experts without tokens get zero gradient blocks, in chunks
    // of 8 KB over the concatenation of the expert's dW1 and dW2 blocks
    const int64_t fd = ffn * d;
    const int64_t chunks = dw1s ? (2 * fd + kZeroChunkFloats - 1) / kZeroChunkFloats : 0;
    const int64_t items = pad_end + static_cast<int64_t>(experts) * chunks;
    for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; i < items;
         i += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        if (i >= pad_end) {
            const int e = static_cast<int>((i - pad_end) / chunks);
            if (count[e] != 0) continue;
            const int64_t c0 = ((i - pad_end) % chunks) * kZeroChunkFloats;
            for (int64_t f = c0 + 4 * lane; f < c0 + kZeroChunkFloats && f < 2 * fd; f += 128) {
                float *dst = f < fd ? dw1s + e * fd + f : dw2s + e * fd + (f - fd);
                *reinterpret_cast<float4 *>(dst) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            continue;
        }
        if (i >= n) {
            const int e = static_cast<int>((i - n) / kSegPad);
            const int r = seg[e] + count[e] + static_cast<int>((i - n) % kSegPad);
            if (r < seg[e + 1])
                for (int64_t c = lane * 8; c < d; c += 256)
                    *reinterpret_cast<uint4 *>(do_perm + r * d + c) = make_uint4(0, 0, 0, 0);
            continue;
        }
        const int r = pos[i];
        const int64_t t = i / k;
        float s = 0.0f;
        if (r >= 0) {
            const float w = p[i];
#pragma unroll 2
            for (int64_t c = lane * 8; c < d; c += 256) {
                float a[8], b[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(dy + t * d + c)), a);
                unpack8(__ldg(reinterpret_cast<const uint4 *>(o_perm + r * d + c)), b);
#pragma unroll
                for (int q = 0; q < 8; ++q) s += a[q] * b[q];
#pragma unroll
                for (int q = 0; q < 8; ++q) a[q] *= w;
                *reinterpret_cast<uint4 *>(do_perm + r * d + c) = pack8(a);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) dp[i] = s;
    }
}

int sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

unsigned grid_items(int64_t items, int per_block) {
    int64_t g = (items + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(sms()) * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<unsigned>(g);
}

}  // namespace

int launch_moe_route(const int *idx, int64_t n, int k, int experts, int *chunk_count, int *count, int *seg,
                     int *pos, int *row_token, int *row_slot, int step, cudaStream_t s) {
    const int chunks = static_cast<int>(moe_route_chunks(n));
    if (experts > kMaxExperts) return MLPBLK_EINVAL;
    if (step == 0)
        return launch_pdl(route_count_kernel, dim3(static_cast<unsigned>(chunks)), dim3(kRouteThreads), 0, s, idx,
                          n, experts, chunk_count);
    return launch_pdl(route_place_kernel, dim3(static_cast<unsigned>(chunks)), dim3(kRouteThreads), 0, s, idx, n,
                      k, experts, chunks, chunk_count, count, seg, pos, row_token, row_slot);
}

int launch_moe_gather(const void *x, const float *rstd, const int *row_token, const int *seg, int experts,
                      int64_t rows_max, int64_t d, void *x_perm, float *rstd_perm, cudaStream_t s) {
    return launch_pdl(gather_rows_kernel, dim3(grid_items(rows_max * 32, 256)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(x), rstd, row_token, seg, experts, d,
                      static_cast<uint16_t *>(x_perm), rstd_perm);
}

int launch_moe_combine(const void *x, const void *o_perm, const float *p, const int *pos, int64_t T, int k,
                       int64_t d, void *y, cudaStream_t s) {
    return launch_pdl(combine_kernel, dim3(grid_items(T * 32, 256)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(o_perm), p, pos, T, k, d,
                      static_cast<uint16_t *>(y));
}

int launch_moe_dout(const void *dy, const void *o_perm, const float *p, const int *pos, const int *count,
                    const int *seg, int64_t T, int k, int experts, int64_t d, float *dp, void *do_perm,
                    float *dw1s, float *dw2s, int64_t ffn, cudaStream_t s) {
    const int64_t items = T * k + static_cast<int64_t>(experts) * kSegPad;
    return launch_pdl(dout_kernel, dim3(grid_items(items * 32, 256)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(dy), static_cast<const uint16_t *>(o_perm), p, pos, count, seg,
                      T * k, k, experts, d, dp, static_cast<uint16_t *>(do_perm), dw1s, dw2s, ffn);
}

}  // namespace mlpblk
