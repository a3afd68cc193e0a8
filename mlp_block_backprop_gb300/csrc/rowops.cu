// rowops.cu -- the HBM-bound kernels of the block: gamma folding for the W1
// GEMM, the fp32-path rstd, the RMSNorm backward row kernel (with the residual
// gradient and the dgamma partial sums), the fixed-order dgamma reduction, and
// zero_grads / scale_grads.
#include <cuda_bf16.h>

#include "mlpblk_internal.h"
#include "ptx.cuh"

namespace mlpblk {

namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float bf(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

// 8 consecutive elements <-> 8 floats, for bf16 storage (one 16-byte access)
// and for fp32 storage (two 16-byte accesses).
template <class T>
struct Io8;

template <>
struct Io8<uint16_t> {
    __device__ static void load(const uint16_t *p, float (&v)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        v[0] = bf(u.x & 0xFFFFu); v[1] = bf(u.x >> 16);
        v[2] = bf(u.y & 0xFFFFu); v[3] = bf(u.y >> 16);
        v[4] = bf(u.z & 0xFFFFu); v[5] = bf(u.z >> 16);
        v[6] = bf(u.w & 0xFFFFu); v[7] = bf(u.w >> 16);
    }
    __device__ static void store(uint16_t *p, const float (&v)[8]) {
        uint4 u;
        u.x = pack2(v[0], v[1]);
        u.y = pack2(v[2], v[3]);
        u.z = pack2(v[4], v[5]);
        u.w = pack2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};

template <>
struct Io8<float> {
    __device__ static void load(const float *p, float (&v)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    __device__ static void store(float *p, const float (&v)[8]) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
};

// W1g[f,k] = W1[f,k] * gamma[k], rounded to the storage type.  One thread per
// 8 consecutive elements (d is a multiple of 8, so a group never crosses rows).
template <class T>
__global__ void fold_gamma_kernel(const T *__restrict__ w1, const T *__restrict__ gamma,
                                  T *__restrict__ w1g, int64_t groups, int64_t d, int *zero_flags,
                                  int zero_count) {
    griddep_enter();
    // the following GEMM's stream-K flags start from zero
    if (zero_flags && blockIdx.x == 0)
        for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_flags[i] = 0;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t e = g * 8;
        const int64_t k = e % d;
        float w[8], s[8];
        Io8<T>::load(w1 + e, w);
        Io8<T>::load(gamma + k, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] *= s[i];
        Io8<T>::store(w1g + e, w);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The forward's statistics pass, one launch with two jobs.  Blocks below
// row_blocks: rstd[t] = 1/sqrt(mean_k x[t,k]^2 + eps), one warp per row (the
// per-row statistic of RMSNorm; the normalisation itself is applied by the W1
// GEMM, gamma through its B operand and rstd in its epilogue).  The other
// blocks: W1g = W1 * gamma (8 elements per thread).
template <class T>
__global__ void __launch_bounds__(256)
norm_prep_kernel(const T *__restrict__ x, float *__restrict__ rstd, int64_t T_rows, int64_t d,
                 float eps, const T *__restrict__ w1, const T *__restrict__ gamma,
                 T *__restrict__ w1g, int64_t groups, int row_blocks, int *zero_flags, int zero_count) {
    griddep_enter();
    // the following GEMM's stream-K flags start from zero
    if (zero_flags && blockIdx.x == 0)
        for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_flags[i] = 0;
    if (static_cast<int>(blockIdx.x) < row_blocks) {
        const int lane = threadIdx.x & 31;
        const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
        const int64_t nw = (static_cast<int64_t>(row_blocks) * blockDim.x) >> 5;
        const float inv_d = 1.0f / static_cast<float>(d);
        for (int64_t t = wid; t < T_rows; t += nw) {
            const T *row = x + t * d;
            float ss = 0.0f;
            for (int64_t c = lane * 8; c < d; c += 256) {
                float v[8];
                Io8<T>::load(row + c, v);
#pragma unroll
                for (int i = 0; i < 8; ++i) ss += v[i] * v[i];
            }
            ss = warp_sum(ss);
            if (lane == 0) rstd[t] = 1.0f / sqrtf(ss * inv_d + eps);
        }
        return;
    }
    const int64_t nthreads = static_cast<int64_t>(gridDim.x - row_blocks) * blockDim.x;
    for (int64_t g = (blockIdx.x - row_blocks) * static_cast<int64_t>(blockDim.x) + threadIdx.x;
         g < groups; g += nthreads) {
        const int64_t e = g * 8;
        const int64_t k = e % d;
        float w[8], s[8];
        Io8<T>::load(w1 + e, w);
        Io8<T>::load(gamma + k, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] *= s[i];
        Io8<T>::store(w1g + e, w);
    }
}

// rstd[t] = 1/sqrt(mean_k x[t,k]^2 + eps) for the fp32 path (the bf16 path
// computes it inside the W1 GEMM).  One warp per row.
__global__ void rstd_f32_kernel(const float *__restrict__ x, float *__restrict__ rstd, int64_t T,
                                int64_t d, float eps) {
    griddep_enter();
    const int lane = threadIdx.x & 31;
    const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = wid; t < T; t += nw) {
        const float *row = x + t * d;
        float ss = 0.0f;
        for (int64_t c = lane * 8; c < d; c += 256) {
            float v[8];
            Io8<float>::load(row + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) ss += v[i] * v[i];
        }
        ss = warp_sum(ss);
        if (lane == 0) rstd[t] = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    }
}

// 8 consecutive elements kept in their storage type (bf16: one 16-byte register
// quad), widened to float on use; keeps the norm kernel at two CTAs per SM.
template <class T>
struct Chunk;

template <>
struct Chunk<uint16_t> {
    uint4 u;
    __device__ void load(const uint16_t *p) { u = __ldg(reinterpret_cast<const uint4 *>(p)); }
    __device__ void zero() { u = make_uint4(0, 0, 0, 0); }
    __device__ float operator[](int i) const {
        const uint32_t w = i < 2 ? u.x : (i < 4 ? u.y : (i < 6 ? u.z : u.w));
        return (i & 1) ? bf(w >> 16) : bf(w & 0xFFFFu);
    }
};

template <>
struct Chunk<float> {
    float4 a, b;
    __device__ void load(const float *p) {
        a = __ldg(reinterpret_cast<const float4 *>(p));
        b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ void zero() { a = b = make_float4(0.0f, 0.0f, 0.0f, 0.0f); }
    __device__ void add(const Chunk &o) {
        a.x += o.a.x; a.y += o.a.y; a.z += o.a.z; a.w += o.a.w;
        b.x += o.b.x; b.y += o.b.y; b.z += o.b.z; b.w += o.b.w;
    }
    __device__ float operator[](int i) const {
        const float4 &v = i < 4 ? a : b;
        const int k = i & 3;
        return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
    }
};

// Eight consecutive elements of dn as floats: dn is float32, or bf16 where the
// dgrad-n GEMM stores it so (the bf16 block: half the bytes to write and read).
__device__ __forceinline__ void load_dn(Chunk<float> &c, const float *p) { c.load(p); }
__device__ __forceinline__ void load_dn(Chunk<float> &c, const uint16_t *p) {
    Chunk<uint16_t> u;
    u.load(p);
    c.a = make_float4(u[0], u[1], u[2], u[3]);
    c.b = make_float4(u[4], u[5], u[6], u[7]);
}

// RMSNorm backward with the residual gradient.  The gradient input carries the
// per-row scale already, dn_s = rstd * dn (the dgrad GEMM writes it that way);
// kScaleDn = true instead takes the plain dn and applies rstd here.  With
// x_hat = x*r and g = dn*gamma the backward of n = x*r*gamma is
//   dx = dy + r*(g - x_hat*mean_k(g*x_hat)) = dy + gamma*dn_s - x*c,
//   c  = r^2 * mean_k(gamma * dn_s * x),
//   dgamma[k] += sum_t dn[t,k]*x_hat[t,k] = sum_t dn_s[t,k]*x[t,k].
//
// A row is shared by a group of G threads (a power of two, 8..256); thread l of
// the group owns the 8-column chunks l, l+G, ..., l+(CPT-1)G, keeps them in
// registers between the row reduction and the dx pass (so no element is read
// twice), and keeps gamma and its dgamma share for those columns in registers
// for all rows of the CTA.  256/G rows are in flight per CTA.  The row sum is a
// shuffle butterfly plus, for G > 32, a shared-memory sum over the group's warps
// in warp order; the CTA's row groups then add their dgamma shares in group
// order and the CTA writes one partial row.  Every sum has a fixed order.
//
// kGather (routed experts): row t's dn_s is the sum over its k slots of the rows
// pos[t*k + j] of dn_s (slot order, from zero; a slot with pos < 0 adds nothing).
constexpr int kGatherRegs = 4;
template <class T, int CPT, bool kScaleDn, bool kGather, class DN>
__global__ void __launch_bounds__(kRowThreads, (CPT <= 2 ? 3 : (CPT <= 3 ? 2 : 1)))
rmsnorm_bwd_kernel(const T *__restrict__ x, const DN *__restrict__ dn_s, const T *__restrict__ dy,
                   const float *__restrict__ rstd, const T *__restrict__ gamma, T *__restrict__ dx,
                   float *__restrict__ dg_part, int64_t T_rows, int64_t d, int64_t rows_per_cta,
                   int G, const int *__restrict__ pos, int k) {
    extern __shared__ float sm[];
    griddep_enter();
    const int R = kRowThreads / G;
    const int grp = threadIdx.x / G;
    const int gl = threadIdx.x - grp * G;
    const int chunks = static_cast<int>(d / 8);
    const float inv_d = 1.0f / static_cast<float>(d);

    Chunk<T> gch[CPT];
    float acc[CPT][8];
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int q = gl + G * j;
        if (q < chunks) gch[j].load(gamma + 8 * q);
        else gch[j].zero();
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
    }

    const int64_t t0 = blockIdx.x * rows_per_cta;
    const int64_t t1 = min(T_rows, t0 + rows_per_cta);
    // kGather with k <= kGatherRegs: a row's slot rows are read one row ahead,
    // so the dn loads do not wait on the pos load
    const bool pre = kGather && k <= kGatherRegs;
    int rnext[kGatherRegs];
    if (pre) {
        const int64_t tn = t0 + grp;
#pragma unroll
        for (int sl = 0; sl < kGatherRegs; ++sl) rnext[sl] = (tn < t1 && sl < k) ? pos[tn * k + sl] : -1;
    }
    int parity = 0;
    for (int64_t base = t0; base < t1; base += R, parity ^= 1) {
        const int64_t t = base + grp;
        const bool valid = t < t1;
        const float r = valid ? rstd[t] : 0.0f;
        int rcur[kGatherRegs];
        if (pre) {
            const int64_t tn = t + R;
#pragma unroll
            for (int sl = 0; sl < kGatherRegs; ++sl) {
                rcur[sl] = rnext[sl];
                rnext[sl] = (tn < t1 && sl < k) ? pos[tn * k + sl] : -1;
            }
        }
        Chunk<T> xch[CPT], ych[CPT];
        Chunk<float> nch[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int q = gl + G * j;
            if (valid && q < chunks) {
                xch[j].load(x + t * d + 8 * q);
                if (kGather && pre) {
                    nch[j].zero();
#pragma unroll
                    for (int sl = 0; sl < kGatherRegs; ++sl) {
                        if (rcur[sl] < 0) continue;
                        Chunk<float> v;
                        load_dn(v, dn_s + static_cast<int64_t>(rcur[sl]) * d + 8 * q);
                        nch[j].add(v);
                    }
                } else if (kGather) {
                    nch[j].zero();
                    for (int sl = 0; sl < k; ++sl) {
                        const int r = pos[t * k + sl];
                        if (r < 0) continue;
                        Chunk<float> v;
                        load_dn(v, dn_s + static_cast<int64_t>(r) * d + 8 * q);
                        nch[j].add(v);
                    }
                } else {
                    load_dn(nch[j], dn_s + t * d + 8 * q);
                }
                ych[j].load(dy + t * d + 8 * q);
            } else {
                xch[j].zero();
                nch[j].zero();
                ych[j].zero();
            }
        }
        const float nscale = kScaleDn ? r : 1.0f;
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < CPT; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) s += gch[j][i] * (nch[j][i] * nscale) * xch[j][i];
        for (int o = (G < 32 ? G : 32) / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (G > 32) {
            float *rs = sm + parity * (R * 8);  // a group spans at most 8 warps
            if ((threadIdx.x & 31) == 0) rs[grp * 8 + (gl >> 5)] = s;
            __syncthreads();
            s = 0.0f;
            for (int w = 0; w < G / 32; ++w) s += rs[grp * 8 + w];
        }
        const float cr = r * r * s * inv_d;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int q = gl + G * j;
            if (valid && q < chunks) {
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float nv = nch[j][i] * nscale;
                    const float xv = xch[j][i];
                    o[i] = ych[j][i] + gch[j][i] * nv - xv * cr;
                    acc[j][i] += nv * xv;
                }
                Io8<T>::store(dx + t * d + 8 * q, o);
            }
        }
    }

    float *out = dg_part + blockIdx.x * d;
    if (R == 1) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int q = gl + G * j;
            if (q < chunks) Io8<float>::store(out + 8 * q, acc[j]);
        }
    } else {
        __syncthreads();
        float *red = sm;  // [R][d]
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int q = gl + G * j;
            if (q < chunks) Io8<float>::store(red + grp * d + 8 * q, acc[j]);
        }
        __syncthreads();
        for (int64_t i = threadIdx.x; i < d; i += kRowThreads) {
            float v = 0.0f;
            for (int g2 = 0; g2 < R; ++g2) v += red[g2 * d + i];
            out[i] = v;
        }
    }
}

// The same arithmetic when a row takes all kRowThreads threads (G = 256: d = 2048
// with one chunk per thread, d = 4096 with two): each CTA takes two consecutive
// rows per iteration and issues both rows' loads before either row's reduction.
// With one row per iteration a CTA had one row's loads in flight, and the launch
// took the same time whether dn_s was 4 or 2 bytes per element: it is bound by the
// rows in flight per SM (two CTAs of two rows here, three of one before).  Sums
// keep the single-row kernel's order (shuffle tree, then the warps in order).
template <class T, int CPT, bool kScaleDn, class DN>
__global__ void __launch_bounds__(kRowThreads, 2)
rmsnorm_bwd_rows2_kernel(const T *__restrict__ x, const DN *__restrict__ dn_s, const T *__restrict__ dy,
                         const float *__restrict__ rstd, const T *__restrict__ gamma, T *__restrict__ dx,
                         float *__restrict__ dg_part, int64_t T_rows, int64_t d, int64_t rows_per_cta) {
    constexpr int kWarps = kRowThreads / 32;
    __shared__ float rsum[2][2][kWarps];  // [parity][row][warp]
    griddep_enter();
    const int tid = threadIdx.x;
    const int wid = tid >> 5, lane = tid & 31;
    const int chunks = static_cast<int>(d / 8);
    const float inv_d = 1.0f / static_cast<float>(d);
    Chunk<T> gch[CPT];
    float acc[CPT][8];
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int q = tid + kRowThreads * j;
        if (q < chunks) gch[j].load(gamma + 8 * q);
        else gch[j].zero();
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
    }
    const int64_t t0 = blockIdx.x * rows_per_cta;
    const int64_t t1 = min(T_rows, t0 + rows_per_cta);
    int parity = 0;
    for (int64_t base = t0; base < t1; base += 2, parity ^= 1) {
        Chunk<T> xch[2][CPT], ych[2][CPT];
        Chunk<float> nch[2][CPT];
        float r[2];
        bool valid[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t t = base + rr;
            valid[rr] = t < t1;
            r[rr] = valid[rr] ? rstd[t] : 0.0f;
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const int q = tid + kRowThreads * j;
                if (valid[rr] && q < chunks) {
                    xch[rr][j].load(x + t * d + 8 * q);
                    load_dn(nch[rr][j], dn_s + t * d + 8 * q);
                    ych[rr][j].load(dy + t * d + 8 * q);
                } else {
                    xch[rr][j].zero();
                    nch[rr][j].zero();
                    ych[rr][j].zero();
                }
            }
        }
        float s[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float nscale = kScaleDn ? r[rr] : 1.0f;
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < CPT; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) v += gch[j][i] * (nch[rr][j][i] * nscale) * xch[rr][j][i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            s[rr] = v;
        }
        if (lane == 0) {
            rsum[parity][0][wid] = s[0];
            rsum[parity][1][wid] = s[1];
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            if (!valid[rr]) continue;
            float v = 0.0f;
            for (int w = 0; w < kWarps; ++w) v += rsum[parity][rr][w];
            const float cr = r[rr] * r[rr] * v * inv_d;
            const float nscale = kScaleDn ? r[rr] : 1.0f;
            const int64_t t = base + rr;
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const int q = tid + kRowThreads * j;
                if (q >= chunks) continue;
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float nv = nch[rr][j][i] * nscale;
                    const float xv = xch[rr][j][i];
                    o[i] = ych[rr][j][i] + gch[j][i] * nv - xv * cr;
                    acc[j][i] += nv * xv;
                }
                Io8<T>::store(dx + t * d + 8 * q, o);
            }
        }
    }
    float *out = dg_part + blockIdx.x * d;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int q = tid + kRowThreads * j;
        if (q < chunks) Io8<float>::store(out + 8 * q, acc[j]);
    }
}

// Staged RMSNorm backward for the routed experts' gathered dn (bf16 x and dy, d a
// multiple of 256 up to 4096, k <= 4 slot rows per token; dn_s already scaled by
// rstd): a token's k slot rows sit at scattered rows of dn_s.  The same
// arithmetic as rmsnorm_bwd_kernel, but the rows reach shared memory by bulk
// copies issued up to kStagedMaxStages iterations ahead, counted by an mbarrier
// per stage.  A producer warp beside the row threads issues them: it
// holds the row map and rstd of kMetaRows rows at a time in registers (the next
// kMetaRows already loading) and writes each stage's rstd and valid-slot mask
// into the stage before its arrival, so the loop loads nothing from global memory
// but the bulk copies, and the copies' issue (~0.7 us a stage) runs while the row
// threads compute instead of between their iterations.  Both take part in the one
// CTA barrier per iteration, after which the producer refills the stage just read.
// The row threads of a CTA, 256 (d <= 2048: three CTAs per SM) or 512 (d = 4096),
// take R = 8 * threads / d rows per iteration, d/8 threads per row, 8 columns per
// thread.  Stage layout: x [R][d] bf16, dy [R][d] bf16, dn [R][k][d] (bf16 as
// launched), rstd [R] fp32, slot mask [R] int.  The row sum is a shuffle tree per warp then
// the row's warps in order; the dgamma partial of the CTA is each thread's
// running sum, then the R row groups in order.
constexpr int kStagedMaxThreads = 512;

// AND of pred over the nthreads threads that reach named barrier id (which may
// arrive from different code: the producer warp and the row threads).
__device__ __forceinline__ bool barrier_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n"
        "  .reg .pred p, q;\n"
        "  setp.ne.u32 p, %1, 0;\n"
        "  bar.red.and.pred q, %2, %3, p;\n"
        "  selp.u32 %0, 1, 0, q;\n"
        "}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}
constexpr int kStagedMaxStages = 4;
constexpr int kMetaRows = 32;

// kMaxK: 2 (k <= 2) or 4.  kThreads: the row threads, 256 (three CTAs per SM) or
// kStagedMaxThreads (one CTA per SM); the block has kThreads + 32 threads.
template <int kMaxK, class DN, int kThreads>
__global__ void __launch_bounds__(kThreads + 32, kThreads == 256 ? 3 : 1)
rmsnorm_bwd_staged_kernel(const uint16_t *__restrict__ x, const DN *__restrict__ dn_s,
                          const uint16_t *__restrict__ dy, const float *__restrict__ rstd,
                          const uint16_t *__restrict__ gamma, uint16_t *__restrict__ dx,
                          float *__restrict__ dg_part, int64_t T_rows, int64_t d, int64_t rows_per_cta, int R,
                          int S, int stage_bytes, const int *__restrict__ pos, int k) {
    extern __shared__ __align__(128) uint8_t smem_st[];
    uint8_t *stages = smem_st;
    float *red = reinterpret_cast<float *>(smem_st + static_cast<size_t>(S) * stage_bytes);  // [2][R][16]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * R * 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + kStagedMaxStages);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const bool producer = tid >= kThreads;
    const int cpr = static_cast<int>(d / 8);  // threads per row (a multiple of 32)
    const int grp = tid / cpr;
    const int gl = tid - grp * cpr;
    const int wpr = cpr / 32;                 // warps per row
    const bool active = !producer && grp < R;
    const float inv_d = 1.0f / static_cast<float>(d);
    const int64_t t0 = blockIdx.x * rows_per_cta;
    const int64_t t1 = min(T_rows, t0 + rows_per_cta);
    const int iters = static_cast<int>((t1 - t0 + R - 1) / R);
    const size_t x_bytes = static_cast<size_t>(R) * d * 2;
    const size_t meta_off = 2 * x_bytes + static_cast<size_t>(R) * k * d * sizeof(DN);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    float g[8], acc[8];
    if (active) Io8<uint16_t>::load(gamma + 8 * gl, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    __syncthreads();
    griddep_enter();

    // The producer: lane l holds rstd and the k slot indices of row (chunk base + l) of
    // the current and the next chunk of kMetaRows rows.
    float cur_r = 0.0f, nxt_r = 0.0f;
    int cur_p[kMaxK], nxt_p[kMaxK];
    int cur_chunk = 0;
    auto load_chunk = [&](int c, float &rv, int (&pv)[kMaxK]) {
        const int64_t t = t0 + static_cast<int64_t>(c) * kMetaRows + lane;
        const bool v = t < t1;
        rv = v ? rstd[t] : 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) pv[j] = (v && j < k) ? pos[t * k + j] : -1;
    };
    // Issues iteration it into stage it % S: lane r < R writes row r's rstd and
    // slot mask; lane j < R * kMaxK copies slot j % kMaxK of row j / kMaxK; lane 0
    // arrives with the stage's byte count and copies the x and dy rows.
    auto issue = [&](int it) {
        const int c = it * R / kMetaRows;  // R divides kMetaRows
        if (c != cur_chunk) {
            cur_r = nxt_r;
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) cur_p[j] = nxt_p[j];
            cur_chunk = c;
            load_chunk(c + 1, nxt_r, nxt_p);
        }
        const int st = it % S;
        uint8_t *sx = stages + static_cast<size_t>(st) * stage_bytes;
        uint8_t *sy = sx + x_bytes;
        uint8_t *sn = sy + x_bytes;
        float *m_r = reinterpret_cast<float *>(sx + meta_off);
        int *m_mask = reinterpret_cast<int *>(m_r + R);
        const int base = it * R - c * kMetaRows;
        const int64_t tb = t0 + static_cast<int64_t>(it) * R;
        const int nr = static_cast<int>(min(static_cast<int64_t>(R), t1 - tb));
        // the lane's own row as a meta writer, and its (row, slot) as a copier
        const int mrow = min(lane, R - 1);
        const int crow = min(lane / kMaxK, R - 1);
        const int cslot = lane % kMaxK;
        const float rv = __shfl_sync(0xffffffffu, cur_r, base + mrow);
        int mask = 0, prow = -1;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            const int vm = __shfl_sync(0xffffffffu, cur_p[j], base + mrow);
            const int vc = __shfl_sync(0xffffffffu, cur_p[j], base + crow);
            if (vm >= 0) mask |= 1 << j;
            if (j == cslot) prow = vc;
        }
        const bool copies = lane < R * kMaxK && lane / kMaxK < nr && cslot < k && prow >= 0;
        uint32_t mine = copies ? static_cast<uint32_t>(d) * sizeof(DN) : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        if (lane < R) {
            m_r[lane] = lane < nr ? rv : 0.0f;
            m_mask[lane] = lane < nr ? mask : 0;
        }
        __syncwarp();  // the meta stores before lane 0's (release) arrival
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nr) * static_cast<uint32_t>(d) * 4u + mine);
            bulk_copy_g2s(sx, x + tb * d, static_cast<uint32_t>(nr * d * 2), &full[st]);
            bulk_copy_g2s(sy, dy + tb * d, static_cast<uint32_t>(nr * d * 2), &full[st]);
        }
        if (copies)
            bulk_copy_g2s(sn + (static_cast<size_t>(lane / kMaxK) * k + cslot) * d * sizeof(DN),
                          dn_s + static_cast<int64_t>(prow) * d, static_cast<uint32_t>(d * sizeof(DN)), &full[st]);
        __syncwarp();
    };
    int issued = 0;
    int it = 0;
    if (producer) {
        load_chunk(0, cur_r, cur_p);
        load_chunk(1, nxt_r, nxt_p);
        for (; issued < S && issued < iters; ++issued) issue(issued);
        // one barrier per iteration with the row threads; after it the stage they
        // just read is free
        for (; it < iters; ++it) {
            if (!barrier_and(1, kThreads + 32, true)) break;
            if (issued < iters) issue(issued++);
        }
    }
    for (; !producer && it < iters; ++it) {
        const int st = it % S;
        const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
        const int64_t t = t0 + static_cast<int64_t>(it) * R + grp;
        const bool valid = active && t < t1;
        // every thread waits on the stage's barrier; the block-wide vote below
        // (which also publishes the warp sums) leaves the loop together if any gave up
        const bool ok = mbar_wait(&full[st], ph, abort_flag);
        const uint8_t *sx = stages + static_cast<size_t>(st) * stage_bytes;
        const uint8_t *sy = sx + x_bytes;
        const uint8_t *sn = sy + x_bytes;
        const float *m_r = reinterpret_cast<const float *>(sx + meta_off);
        const int *m_mask = reinterpret_cast<const int *>(m_r + R);
        float xv[8], yv[8], nv[8];
        float part = 0.0f, r = 0.0f;
        if (valid && ok) {
            r = m_r[grp];
            const int mask = m_mask[grp];
            const uint4 ux = *reinterpret_cast<const uint4 *>(sx + (static_cast<size_t>(grp) * d + 8 * gl) * 2);
            const uint4 uy = *reinterpret_cast<const uint4 *>(sy + (static_cast<size_t>(grp) * d + 8 * gl) * 2);
            xv[0] = bf(ux.x & 0xFFFFu); xv[1] = bf(ux.x >> 16); xv[2] = bf(ux.y & 0xFFFFu); xv[3] = bf(ux.y >> 16);
            xv[4] = bf(ux.z & 0xFFFFu); xv[5] = bf(ux.z >> 16); xv[6] = bf(ux.w & 0xFFFFu); xv[7] = bf(ux.w >> 16);
            yv[0] = bf(uy.x & 0xFFFFu); yv[1] = bf(uy.x >> 16); yv[2] = bf(uy.y & 0xFFFFu); yv[3] = bf(uy.y >> 16);
            yv[4] = bf(uy.z & 0xFFFFu); yv[5] = bf(uy.z >> 16); yv[6] = bf(uy.w & 0xFFFFu); yv[7] = bf(uy.w >> 16);
#pragma unroll
            for (int i = 0; i < 8; ++i) nv[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) {
                if (!((mask >> j) & 1)) continue;
                const DN *q = reinterpret_cast<const DN *>(sn) + (static_cast<size_t>(grp) * k + j) * d + 8 * gl;
                if (sizeof(DN) == 4) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(q);
                    const float4 a1 = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(q) + 4);
                    nv[0] += a0.x; nv[1] += a0.y; nv[2] += a0.z; nv[3] += a0.w;
                    nv[4] += a1.x; nv[5] += a1.y; nv[6] += a1.z; nv[7] += a1.w;
                } else {
                    const uint4 u = *reinterpret_cast<const uint4 *>(q);
                    nv[0] += bf(u.x & 0xFFFFu); nv[1] += bf(u.x >> 16); nv[2] += bf(u.y & 0xFFFFu);
                    nv[3] += bf(u.y >> 16); nv[4] += bf(u.z & 0xFFFFu); nv[5] += bf(u.z >> 16);
                    nv[6] += bf(u.w & 0xFFFFu); nv[7] += bf(u.w >> 16);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) part += g[i] * nv[i] * xv[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        float *rr = red + (it & 1) * R * 16;
        if (active && lane == 0) rr[grp * 16 + gl / 32] = part;
        // every thread has read stage st and written its warp sum
        if (!barrier_and(1, kThreads + 32, ok)) break;
        if (valid) {
            float sum = 0.0f;
            for (int w = 0; w < wpr; ++w) sum += rr[grp * 16 + w];
            const float cr = r * r * sum * inv_d;
            float o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i] = yv[i] + g[i] * nv[i] - xv[i] * cr;
                acc[i] += nv[i] * xv[i];
            }
            const uint4 u = make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
            *reinterpret_cast<uint4 *>(dx + t * d + 8 * gl) = u;
        }
    }
    if (it < iters) {
        // gave up: let the copies already issued land before the CTA exits
        if (producer && lane == 0)
            for (int j = it; j < issued; ++j) mbar_drain(&full[j % S], static_cast<uint32_t>(j / S) & 1u);
        __syncthreads();
        return;
    }
    // the CTA's dgamma partial row: the R row groups' sums in group order
    __syncthreads();
    float *gsum = reinterpret_cast<float *>(stages);  // [R][d], the stages are free now
    if (active) {
#pragma unroll
        for (int i = 0; i < 8; ++i) gsum[static_cast<size_t>(grp) * d + 8 * gl + i] = acc[i];
    }
    __syncthreads();
    float *out = dg_part + blockIdx.x * d;
    for (int64_t i = tid; i < d; i += blockDim.x) {
        float v = 0.0f;
        for (int g2 = 0; g2 < R; ++g2) v += gsum[static_cast<size_t>(g2) * d + i];
        out[i] = v;
    }
}

// dgamma[k] += (or =, overwrite) sum of the partial rows.  A CTA covers 32 columns with 128
// slices: slice s adds partial rows s, s+128, ... in increasing order (4 columns
// per thread), then the 128 slice sums meet in a fixed pairwise tree.
__global__ void __launch_bounds__(1024)
dgamma_finalize_kernel(const float *__restrict__ part, int parts, float *__restrict__ dgamma,
                       int64_t d, int overwrite) {
    __shared__ float4 red[128][9];
    griddep_enter();
    const int lane = threadIdx.x & 7;
    const int slice = threadIdx.x >> 3;
    const int64_t col = blockIdx.x * 32 + lane * 4;
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (col < d) {
#pragma unroll 4
        for (int p = slice; p < parts; p += 128) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(part + p * d + col));
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
    }
    red[slice][lane] = s;
    __syncthreads();
    for (int w = 64; w >= 1; w >>= 1) {
        if (slice < w) {
            const float4 v = red[slice + w][lane];
            float4 t = red[slice][lane];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
            red[slice][lane] = t;
        }
        __syncthreads();
    }
    if (slice == 0 && col < d) {
        const float4 t = red[0][lane];
        float4 *g = reinterpret_cast<float4 *>(dgamma + col);
        float4 o = overwrite ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : *g;
        o.x += t.x;
        o.y += t.y;
        o.z += t.z;
        o.w += t.w;
        *g = o;
    }
}

// The three gradient buffers in one launch: p_b[i] = 0 (kZero) or p_b[i] *= s,
// over the concatenated float4 index space of the buffers.
template <bool kZero>
__global__ void grads_kernel(float4 *p0, int64_t n0, float4 *p1, int64_t n1, float4 *p2,
                             int64_t n2, float s) {
    griddep_enter();
    const int64_t n = n0 + n1 + n2;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 *p = i < n0 ? p0 + i : (i < n0 + n1 ? p1 + (i - n0) : p2 + (i - n0 - n1));
        if (kZero) {
            *p = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else {
            float4 v = *p;
            v.x *= s;
            v.y *= s;
            v.z *= s;
            v.w *= s;
            *p = v;
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

int grid_for(int64_t work_items, int threads) {
    const int64_t want = (work_items + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

// Row-group shape of the norm backward for width d: chunks per thread (1..4)
// and group size G (power of two, 8..256) with the fewest masked chunk slots.
void norm_shape(int64_t d, int *cpt_out, int *g_out) {
    const int chunks = static_cast<int>(d / 8);
    int best_c = 0, best_g = 0, best_waste = 1 << 30;
    for (int c = 1; c <= 4; ++c) {
        const int need = (chunks + c - 1) / c;
        int g = 8;
        while (g < need) g <<= 1;
        if (g > kRowThreads) continue;
        const int waste = g * c - chunks;
        if (waste < best_waste) {
            best_waste = waste;
            best_c = c;
            best_g = g;
        }
    }
    *cpt_out = best_c;
    *g_out = best_g;
}

// One CTA per resident slot (at most max_parts), rows split in whole multiples
// of the rows in flight; the number of CTAs (= dgamma partial rows) is returned.
template <class E, int CPT, bool kScaleDn, bool kGather, class DN>
int run_norm_bwd(const void *x, const DN *dn, const void *dy, const float *rstd,
                 const void *gamma, void *dx, float *part, int64_t T, int64_t d, int max_parts,
                 int *parts_out, int G, const int *pos, int k, cudaStream_t s) {
    const int R = kRowThreads / G;
    const int64_t floats = R > 1 ? (R * d > 2 * R * 8 ? R * d : 2 * R * 8) : 2 * 8;
    const size_t smem = floats * sizeof(float);
    int occ = 0;
    const int rc = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ, rmsnorm_bwd_kernel<E, CPT, kScaleDn, kGather, DN>, kRowThreads, smem));
    if (rc != MLPBLK_OK) return rc;
    int64_t parts = static_cast<int64_t>(occ > 0 ? occ : 1) * sm_count();
    if (parts > max_parts) parts = max_parts;
    const int64_t groups = (T + R - 1) / R;
    if (parts > groups) parts = groups;
    if (parts < 1) parts = 1;
    const int64_t rows_per_cta = ((T + parts - 1) / parts + R - 1) / R * R;
    parts = (T + rows_per_cta - 1) / rows_per_cta;
    *parts_out = static_cast<int>(parts);
    return launch_pdl(rmsnorm_bwd_kernel<E, CPT, kScaleDn, kGather, DN>, dim3(static_cast<unsigned>(parts)),
                      dim3(kRowThreads), smem, s, static_cast<const E *>(x), dn,
                      static_cast<const E *>(dy), rstd, static_cast<const E *>(gamma),
                      static_cast<E *>(dx), part, T, d, rows_per_cta, G, pos, k);
}

template <class E, int CPT, bool kScaleDn, class DN>
int run_norm_bwd_rows2(const void *x, const DN *dn, const void *dy, const float *rstd, const void *gamma,
                       void *dx, float *part, int64_t T, int64_t d, int max_parts, int *parts_out, cudaStream_t s) {
    int occ = 0;
    const int rc = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ, rmsnorm_bwd_rows2_kernel<E, CPT, kScaleDn, DN>, kRowThreads, 0));
    if (rc != MLPBLK_OK) return rc;
    int64_t parts = static_cast<int64_t>(occ > 0 ? occ : 1) * sm_count();
    if (parts > max_parts) parts = max_parts;
    const int64_t pairs = (T + 1) / 2;
    if (parts > pairs) parts = pairs;
    if (parts < 1) parts = 1;
    const int64_t rows_per_cta = ((T + parts - 1) / parts + 1) / 2 * 2;
    parts = (T + rows_per_cta - 1) / rows_per_cta;
    *parts_out = static_cast<int>(parts);
    return launch_pdl(rmsnorm_bwd_rows2_kernel<E, CPT, kScaleDn, DN>, dim3(static_cast<unsigned>(parts)),
                      dim3(kRowThreads), 0, s, static_cast<const E *>(x), dn, static_cast<const E *>(dy), rstd,
                      static_cast<const E *>(gamma), static_cast<E *>(dx), part, T, d, rows_per_cta);
}

// Two rows per CTA iteration where a bf16 row takes the whole CTA
// (MLPBLK_NORM_ROWS2=0: one row per iteration, the general kernel).
bool rows2_enabled() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_NORM_ROWS2");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1;
}

template <class E, bool kScaleDn, bool kGather = false, class DN = float>
int dispatch_norm_bwd(const void *x, const DN *dn, const void *dy, const float *rstd,
                      const void *gamma, void *dx, float *part, int64_t T, int64_t d, int max_parts,
                      int *parts_out, cudaStream_t s, const int *pos = nullptr, int k = 0) {
    int cpt = 0, G = 0;
    norm_shape(d, &cpt, &G);
    if (!kGather && sizeof(E) == 2 && G == kRowThreads && cpt <= 2 && T > 0 && rows2_enabled()) {
        if (cpt == 1)
            return run_norm_bwd_rows2<E, 1, kScaleDn, DN>(x, dn, dy, rstd, gamma, dx, part, T, d, max_parts,
                                                          parts_out, s);
        return run_norm_bwd_rows2<E, 2, kScaleDn, DN>(x, dn, dy, rstd, gamma, dx, part, T, d, max_parts,
                                                      parts_out, s);
    }
#define MLPBLK_NB(C) \
    return run_norm_bwd<E, C, kScaleDn, kGather, DN>(x, dn, dy, rstd, gamma, dx, part, T, d, max_parts, parts_out, G, \
                                                 pos, k, s)
    switch (cpt) {
        case 1: MLPBLK_NB(1);
        case 2: MLPBLK_NB(2);
        case 3: MLPBLK_NB(3);
        case 4: MLPBLK_NB(4);
        default: return MLPBLK_ENOTSUP;
    }
#undef MLPBLK_NB
}

}  // namespace

int launch_fold_gamma(int dtype, const void *w1, const void *gamma, void *w1g, int64_t F,
                      int64_t d, int *zero_flags, int zero_count, cudaStream_t s) {
    const int64_t groups = F * d / 8;
    const int grid = grid_for(groups, 256);
    if (dtype == MLPBLK_BF16)
        return launch_pdl(fold_gamma_kernel<uint16_t>, dim3(grid), dim3(256), 0, s,
                          static_cast<const uint16_t *>(w1), static_cast<const uint16_t *>(gamma),
                          static_cast<uint16_t *>(w1g), groups, d, zero_flags, zero_count);
    return launch_pdl(fold_gamma_kernel<float>, dim3(grid), dim3(256), 0, s,
                      static_cast<const float *>(w1), static_cast<const float *>(gamma),
                      static_cast<float *>(w1g), groups, d, zero_flags, zero_count);
}

int launch_norm_prep(int dtype, const void *x, float *rstd, int64_t T, int64_t d, float eps,
                     const void *w1, const void *gamma, void *w1g, int64_t F, int *zero_flags,
                     int zero_count, cudaStream_t s) {
    const int64_t groups = F * d / 8;
    int64_t rb = (T * 32 + 255) / 256;  // one warp per row
    const int64_t rb_cap = static_cast<int64_t>(sm_count()) * 4;
    if (rb > rb_cap) rb = rb_cap;
    if (rb < 1) rb = 1;
    const int fold_blocks = grid_for(groups, 256);
    const int grid = static_cast<int>(rb) + fold_blocks;
    if (dtype == MLPBLK_BF16)
        return launch_pdl(norm_prep_kernel<uint16_t>, dim3(grid), dim3(256), 0, s,
                          static_cast<const uint16_t *>(x), rstd, T, d, eps,
                          static_cast<const uint16_t *>(w1), static_cast<const uint16_t *>(gamma),
                          static_cast<uint16_t *>(w1g), groups, static_cast<int>(rb), zero_flags,
                          zero_count);
    return launch_pdl(norm_prep_kernel<float>, dim3(grid), dim3(256), 0, s,
                      static_cast<const float *>(x), rstd, T, d, eps, static_cast<const float *>(w1),
                      static_cast<const float *>(gamma), static_cast<float *>(w1g), groups,
                      static_cast<int>(rb), zero_flags, zero_count);
}

int launch_rstd_f32(const float *x, float *rstd, int64_t T, int64_t d, float eps, cudaStream_t s) {
    return launch_pdl(rstd_f32_kernel, dim3(grid_for(T * 32, 256)), dim3(256), 0, s, x, rstd, T, d, eps);
}

namespace {

// Shape of the staged kernel for width d and k slot rows (0 when it does not
// apply): rows per iteration R, stages S, bytes per stage.
struct StagedShape {
    int R, S, stage_bytes, threads;
    size_t smem;
};

StagedShape staged_shape(int64_t d, int k, int dn_bytes) {
    StagedShape sh = {0, 0, 0, 0, 0};
    if (d % 256 != 0 || d > 4096 || k < 1 || k > 4) return sh;
    const int threads = d <= 2048 ? 256 : 512;
    const int R = static_cast<int>(8 * threads / d);
    if (R * (k <= 2 ? 2 : 4) > 32 || kMetaRows % R != 0) return sh;  // one copy lane per (row, slot)
    // x, dy, the slot rows, then each row's rstd and slot mask
    const int64_t bytes =
        (static_cast<int64_t>(R) * d * 4 + static_cast<int64_t>(R) * k * d * dn_bytes + 8 * R + 127) / 128 * 128;
    const int64_t extra = 2 * R * 16 * 4 + kStagedMaxStages * 8 + 16;
    const int64_t budget = threads == 256 ? 66 * 1024 : 200 * 1024;  // 256 threads: three CTAs per SM
    int S = static_cast<int>((budget - extra) / bytes);
    if (S > kStagedMaxStages) S = kStagedMaxStages;
    if (S < 2) return sh;
    sh.R = R;
    sh.S = S;
    sh.threads = threads;
    sh.stage_bytes = static_cast<int>(bytes);
    sh.smem = static_cast<size_t>(S) * bytes + extra;
    return sh;
}

template <int kMaxK, class DN, int kThreads>
int run_norm_bwd_staged_t(const StagedShape &sh, const void *x, const DN *dn, const void *dy, const float *rstd,
                          const void *gamma, void *dx, float *part, int64_t T, int64_t d, int max_parts,
                          int *parts_out, const int *pos, int k, cudaStream_t s) {
    static bool attr[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLPBLK_ECUDA;
    if (!attr[dev]) {
        const int rc = cuda_status(cudaFuncSetAttribute(rmsnorm_bwd_staged_kernel<kMaxK, DN, kThreads>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024 + 4096));
        if (rc != MLPBLK_OK) return rc;
        attr[dev] = true;
    }
    int64_t parts = static_cast<int64_t>(sm_count()) * (kThreads == 256 ? 3 : 1);
    if (parts > max_parts) parts = max_parts;
    const int64_t groups = (T + sh.R - 1) / sh.R;
    if (parts > groups) parts = groups;
    if (parts < 1) parts = 1;
    const int64_t rows_per_cta = ((T + parts - 1) / parts + sh.R - 1) / sh.R * sh.R;
    parts = (T + rows_per_cta - 1) / rows_per_cta;
    *parts_out = static_cast<int>(parts);
    return launch_pdl(rmsnorm_bwd_staged_kernel<kMaxK, DN, kThreads>, dim3(static_cast<unsigned>(parts)),
                      dim3(kThreads + 32), sh.smem, s, static_cast<const uint16_t *>(x), dn,
                      static_cast<const uint16_t *>(dy), rstd, static_cast<const uint16_t *>(gamma),
                      static_cast<uint16_t *>(dx), part, T, d, rows_per_cta, sh.R, sh.S, sh.stage_bytes, pos, k);
}

template <int kMaxK>
int run_norm_bwd_staged(const StagedShape &sh, const void *x, const uint16_t *dn, const void *dy, const float *rstd,
                        const void *gamma, void *dx, float *part, int64_t T, int64_t d, int max_parts,
                        int *parts_out, const int *pos, int k, cudaStream_t s) {
    if (sh.threads == 256)
        return run_norm_bwd_staged_t<kMaxK, uint16_t, 256>(sh, x, dn, dy, rstd, gamma, dx, part, T, d, max_parts,
                                                           parts_out, pos, k, s);
    return run_norm_bwd_staged_t<kMaxK, uint16_t, kStagedMaxThreads>(sh, x, dn, dy, rstd, gamma, dx, part, T, d,
                                                                     max_parts, parts_out, pos, k, s);
}

}  // namespace

int launch_rmsnorm_bwd(int dtype, const void *x, const void *dn_s, int dn_bf16, const void *dy,
                       const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                       int64_t T, int64_t d, int max_parts, int *parts_out, cudaStream_t s) {
    if (dtype == MLPBLK_BF16 && dn_bf16)
        return dispatch_norm_bwd<uint16_t, false, false, uint16_t>(x, static_cast<const uint16_t *>(dn_s), dy, rstd,
                                                                   gamma, dx, dgamma_part, T, d, max_parts, parts_out, s);
    if (dtype == MLPBLK_BF16)
        return dispatch_norm_bwd<uint16_t, false>(x, static_cast<const float *>(dn_s), dy, rstd, gamma, dx,
                                                  dgamma_part, T, d, max_parts, parts_out, s);
    return dispatch_norm_bwd<float, false>(x, static_cast<const float *>(dn_s), dy, rstd, gamma, dx, dgamma_part,
                                           T, d, max_parts, parts_out, s);
}

int launch_rmsnorm_bwd_unscaled(int dtype, const void *x, const float *dn, const void *dy,
                                const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                                int64_t T, int64_t d, int max_parts, int *parts_out, cudaStream_t s) {
    if (dtype == MLPBLK_BF16)
        return dispatch_norm_bwd<uint16_t, true>(x, dn, dy, rstd, gamma, dx, dgamma_part, T, d,
                                                 max_parts, parts_out, s);
    return dispatch_norm_bwd<float, true>(x, dn, dy, rstd, gamma, dx, dgamma_part, T, d, max_parts,
                                          parts_out, s);
}

int launch_rmsnorm_bwd_gather(const void *x, const void *dn_rows, int dn_bf16, const int *pos, int k,
                              const void *dy, const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                              int64_t T, int64_t d, int max_parts, int *parts_out, cudaStream_t s) {
    if (T > 0 && dn_bf16) {
        const StagedShape sh = staged_shape(d, k, 2);
        const uint16_t *dn = static_cast<const uint16_t *>(dn_rows);
        if (sh.R > 0 && k <= 2)
            return run_norm_bwd_staged<2>(sh, x, dn, dy, rstd, gamma, dx, dgamma_part, T, d, max_parts, parts_out,
                                          pos, k, s);
        if (sh.R > 0)
            return run_norm_bwd_staged<4>(sh, x, dn, dy, rstd, gamma, dx, dgamma_part, T, d, max_parts, parts_out,
                                          pos, k, s);
    }
    if (dn_bf16)
        return dispatch_norm_bwd<uint16_t, false, true, uint16_t>(x, static_cast<const uint16_t *>(dn_rows), dy, rstd,
                                                                  gamma, dx, dgamma_part, T, d, max_parts, parts_out,
                                                                  s, pos, k);
    return dispatch_norm_bwd<uint16_t, false, true>(x, static_cast<const float *>(dn_rows), dy, rstd, gamma, dx,
                                                    dgamma_part, T, d, max_parts, parts_out, s, pos, k);
}

int take_device_error_rowops() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLPBLK_ECUDA;
    if (v != 0) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
    return v;
}

int launch_dgamma_finalize(const float *part, int parts, float *dgamma, int64_t d, cudaStream_t s,
                           int overwrite) {
    return launch_pdl(dgamma_finalize_kernel, dim3(static_cast<unsigned>((d + 31) / 32)), dim3(1024), 0,
                      s, part, parts, dgamma, d, overwrite);
}

namespace {

// kZeroSlices blocks per split tile of `a` (then of `b`), each clearing a slice of
// the tile's rows of C with 16-byte stores; the last block clears dgamma.
constexpr int kZeroSlices = 8;
__global__ void __launch_bounds__(256)
zero_split_tiles_kernel(SplitTiles a, SplitTiles b, float *__restrict__ dgamma, int64_t d) {
    griddep_enter();
    const int na = a.tiles - a.dp_tiles, nb = b.tiles - b.dp_tiles;
    int idx = static_cast<int>(blockIdx.x) / kZeroSlices;
    const int slice = static_cast<int>(blockIdx.x) % kZeroSlices;
    if (idx >= na + nb) {
        for (int64_t i = threadIdx.x; i < d; i += blockDim.x) dgamma[i] = 0.0f;
        return;
    }
    const SplitTiles &g = idx < na ? a : b;
    if (idx >= na) idx -= na;
    int mi = 0, ni = 0;
    raster_tile(g.dp_tiles + idx, g.m_tiles, g.n_tiles, g.group_m, mi, ni);
    const int rows = (g.tile_m + kZeroSlices - 1) / kZeroSlices;
    const int r0 = mi * g.tile_m + slice * rows;
    const int r1 = min(min(g.M, mi * g.tile_m + g.tile_m), r0 + rows);
    if (r0 >= r1) return;
    const int c0 = ni * g.tile_n, c1 = min(g.N, c0 + g.tile_n);
    const int cols4 = (c1 - c0) / 4;  // N and the tile widths are multiples of 8
    const int64_t n4 = static_cast<int64_t>(r1 - r0) * cols4;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const int r = r0 + static_cast<int>(i / cols4);
        const int c = c0 + 4 * static_cast<int>(i % cols4);
        *reinterpret_cast<float4 *>(g.c + r * g.ldc + c) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
}

}  // namespace

SplitTiles split_tiles_of(const GemmArgs &plan, float *c, int64_t ldc) {
    SplitTiles t;
    t.c = c;
    t.ldc = ldc;
    t.M = plan.M;
    t.N = plan.N;
    t.tiles = plan.tiles;
    t.dp_tiles = plan.dp_tiles < plan.tiles ? plan.dp_tiles : plan.tiles;
    t.m_tiles = plan.m_tiles;
    t.n_tiles = plan.n_tiles;
    t.group_m = plan.group_m;
    t.tile_m = plan.tile_m;
    t.tile_n = plan.tile_n;
    return t;
}

int launch_zero_split_tiles(const SplitTiles &a, const SplitTiles &b, float *dgamma, int64_t d, cudaStream_t s) {
    const int blocks = ((a.tiles - a.dp_tiles) + (b.tiles - b.dp_tiles)) * kZeroSlices + 1;
    return launch_pdl(zero_split_tiles_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a, b, dgamma,
                      d);
}

int launch_grads(bool zero, float sc, float *p0, int64_t n0, float *p1, int64_t n1, float *p2,
                 int64_t n2, cudaStream_t s) {
    const int64_t a = n0 / 4, b = n1 / 4, c = n2 / 4;
    const int grid = grid_for(a + b + c, 256);
    float4 *q0 = reinterpret_cast<float4 *>(p0), *q1 = reinterpret_cast<float4 *>(p1),
           *q2 = reinterpret_cast<float4 *>(p2);
    if (zero) return launch_pdl(grads_kernel<true>, dim3(grid), dim3(256), 0, s, q0, a, q1, b, q2, c, 0.0f);
    return launch_pdl(grads_kernel<false>, dim3(grid), dim3(256), 0, s, q0, a, q1, b, q2, c, sc);
}

}  // namespace mlpblk
