// moe.cu -- dispatch and combine of the routed ReLU^2 expert block ("Nemotron
// Kernels From Inference To Backpropagation" -- "Kernel 4: Routed ReLU2 MoE":
// select, execute, weight and combine; the backward returns d_hidden,
// d_routing_weights, d_expert_up and d_expert_down; the dispatch is held fixed).
//
// The (token, slot) assignments of each expert are laid out back to back in
// token order, each expert's segment padded to a multiple of 256 rows, so the
// experts' GEMMs run as grouped GEMMs over one row space (gemm_tc.cuh, M- and
// K-grouped).  Every order is fixed: ranks follow (token, slot) order, the
// combine and the dn scatter add slots in slot order.
#include "mlpblk_internal.h"

namespace mlpblk {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kSegPad = 256;

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

// Block e: rank[i] = number of entries idx[i'] == e with i' < i (row-major
// (token, slot) order) for every i with idx[i] == e; count[e] = their number.
// Entries outside [0, experts) belong to no expert.
__global__ void __launch_bounds__(kRouteThreads)
route_rank_kernel(const int *__restrict__ idx, int64_t n, int experts, int *__restrict__ rank,
                  int *__restrict__ count) {
    __shared__ int warp_sums[kRouteThreads / 32];
    griddep_enter();
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int running = 0;
    for (int64_t base = 0; base < n; base += kRouteThreads) {
        const int64_t i = base + threadIdx.x;
        const bool hit = i < n && idx[i] == e;
        const unsigned ballot = __ballot_sync(0xffffffffu, hit);
        const int before = __popc(ballot & ((1u << lane) - 1u));
        if (lane == 0) warp_sums[wid] = __popc(ballot);
        __syncthreads();
        int prefix = 0, total = 0;
        for (int w = 0; w < kRouteThreads / 32; ++w) {
            if (w < wid) prefix += warp_sums[w];
            total += warp_sums[w];
        }
        if (hit) rank[i] = running + prefix + before;
        running += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) count[e] = running;
}

// seg[e] = sum over e' < e of count[e'] rounded up to 256; seg[experts] = rows used.
__global__ void route_offsets_kernel(const int *__restrict__ count, int experts, int *__restrict__ seg) {
    griddep_enter();
    if (threadIdx.x == 0) {
        int off = 0;
        for (int e = 0; e < experts; ++e) {
            seg[e] = off;
            off += (count[e] + kSegPad - 1) / kSegPad * kSegPad;
        }
        seg[experts] = off;
    }
}

// row_token[r] = -1 (a padding row until an assignment claims it).
__global__ void route_clear_kernel(int *__restrict__ row_token, int64_t rows) {
    griddep_enter();
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < rows;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x)
        row_token[r] = -1;
}

// pos[i] = seg[idx[i]] + rank[i]; row_token / row_slot of that row.
__global__ void route_place_kernel(const int *__restrict__ idx, const int *__restrict__ rank,
                                   const int *__restrict__ seg, int64_t n, int k, int experts,
                                   int *__restrict__ pos, int *__restrict__ row_token, int *__restrict__ row_slot) {
    griddep_enter();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int e = idx[i];
        if (e < 0 || e >= experts) {
            pos[i] = -1;
            continue;
        }
        const int p = seg[e] + rank[i];
        pos[i] = p;
        row_token[p] = static_cast<int>(i / k);
        row_slot[p] = static_cast<int>(i % k);
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

// One warp per (token, slot): dp[t,j] = <dy[t], o_perm[pos[t,j]]> (lane sums, then
// a fixed shuffle tree).
__global__ void routing_grad_kernel(const uint16_t *__restrict__ dy, const uint16_t *__restrict__ o_perm,
                                    const int *__restrict__ pos, int64_t n, int k, int64_t d,
                                    float *__restrict__ dp) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; i < n;
         i += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const int r = pos[i];
        const int64_t t = i / k;
        float s = 0.0f;
        if (r >= 0) {
            for (int64_t c = lane * 8; c < d; c += 256) {
                float a[8], b[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(dy + t * d + c)), a);
                unpack8(__ldg(reinterpret_cast<const uint4 *>(o_perm + r * d + c)), b);
#pragma unroll
                for (int q = 0; q < 8; ++q) s += a[q] * b[q];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) dp[i] = s;
    }
}

// One warp per row: do_perm[r] = p[t, slot] * dy[t] (bf16), zeros for padding rows.
__global__ void gather_dout_kernel(const uint16_t *__restrict__ dy, const float *__restrict__ p,
                                   const int *__restrict__ row_token, const int *__restrict__ row_slot,
                                   const int *__restrict__ seg, int experts, int k, int64_t d,
                                   uint16_t *__restrict__ do_perm) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    const int64_t rows = seg[experts];
    for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows;
         r += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const int t = row_token[r];
        const float w = t >= 0 ? p[static_cast<int64_t>(t) * k + row_slot[r]] : 0.0f;
        for (int64_t c = lane * 8; c < d; c += 256) {
            float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (t >= 0) {
                unpack8(__ldg(reinterpret_cast<const uint4 *>(dy + t * d + c)), v);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] *= w;
            }
            *reinterpret_cast<uint4 *>(do_perm + r * d + c) = pack8(v);
        }
    }
}

// One warp per token: dn_s[t] = sum_j dn_perm[pos[t,j]] (slot order, fp32).
__global__ void scatter_dn_kernel(const float *__restrict__ dn_perm, const int *__restrict__ pos, int64_t T,
                                  int k, int64_t d, float *__restrict__ dn_s) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    for (int64_t t = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; t < T;
         t += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        for (int64_t c = lane * 4; c < d; c += 128) {
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int j = 0; j < k; ++j) {
                const int r = pos[t * k + j];
                if (r < 0) continue;
                const float4 v = __ldg(reinterpret_cast<const float4 *>(dn_perm + r * d + c));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            *reinterpret_cast<float4 *>(dn_s + t * d + c) = acc;
        }
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

int launch_moe_route_clear(int *row_token, int64_t rows_max, cudaStream_t s) {
    return launch_pdl(route_clear_kernel, dim3(grid_items(rows_max, 256)), dim3(256), 0, s, row_token, rows_max);
}

int launch_moe_route_rank(const int *idx, int64_t n, int experts, int *rank, int *count, cudaStream_t s) {
    return launch_pdl(route_rank_kernel, dim3(static_cast<unsigned>(experts)), dim3(kRouteThreads), 0, s, idx, n,
                      experts, rank, count);
}

int launch_moe_route_offsets(const int *count, int experts, int *seg, cudaStream_t s) {
    return launch_pdl(route_offsets_kernel, dim3(1), dim3(32), 0, s, count, experts, seg);
}

int launch_moe_route_place(const int *idx, const int *rank, const int *seg, int64_t n, int k, int experts,
                           int *pos, int *row_token, int *row_slot, cudaStream_t s) {
    return launch_pdl(route_place_kernel, dim3(grid_items(n, 256)), dim3(256), 0, s, idx, rank, seg, n, k,
                      experts, pos, row_token, row_slot);
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

int launch_moe_routing_grad(const void *dy, const void *o_perm, const int *pos, int64_t T, int k, int64_t d,
                            float *dp, cudaStream_t s) {
    return launch_pdl(routing_grad_kernel, dim3(grid_items(T * k * 32, 256)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(dy), static_cast<const uint16_t *>(o_perm), pos, T * k, k, d,
                      dp);
}

int launch_moe_gather_dout(const void *dy, const float *p, const int *row_token, const int *row_slot,
                           const int *seg, int experts, int k, int64_t rows_max, int64_t d, void *do_perm,
                           cudaStream_t s) {
    return launch_pdl(gather_dout_kernel, dim3(grid_items(rows_max * 32, 256)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(dy), p, row_token, row_slot, seg, experts, k, d,
                      static_cast<uint16_t *>(do_perm));
}

int launch_moe_scatter_dn(const float *dn_perm, const int *pos, int64_t T, int k, int64_t d, float *dn_s,
                          cudaStream_t s) {
    return launch_pdl(scatter_dn_kernel, dim3(grid_items(T * 32, 256)), dim3(256), 0, s, dn_perm, pos, T, k, d,
                      dn_s);
}

}  // namespace mlpblk
