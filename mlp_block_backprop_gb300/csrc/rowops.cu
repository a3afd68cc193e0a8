// rowops.cu -- the HBM-bound kernels of the block: gamma folding for the W1
// GEMM, the fp32-path rstd, the RMSNorm backward row kernel (with the residual
// gradient and the dgamma partial sums), the fixed-order dgamma reduction, and
// zero_grads / scale_grads.
#include <cuda_bf16.h>

#include "mlpblk_internal.h"

namespace mlpblk {

namespace {

constexpr int kRowThreads = 256;  // 8 warps, one row per warp at a time

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
                                  T *__restrict__ w1g, int64_t groups, int64_t d) {
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

// rstd[t] = 1/sqrt(mean_k x[t,k]^2 + eps) for the fp32 path (the bf16 path
// computes it inside the W1 GEMM).  One warp per row.
__global__ void rstd_f32_kernel(const float *__restrict__ x, float *__restrict__ rstd, int64_t T,
                                int64_t d, float eps) {
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

// RMSNorm backward with the residual gradient, one warp per row.  Inputs carry
// the per-row scale already: dn_s = rstd * dn (from the dgrad GEMM).  With
// x_hat = x*r and g = dn*gamma the backward of n = x*r*gamma is
//   dx = dy + r*(g - x_hat*mean_k(g*x_hat)) = dy + gamma*dn_s - x*c,
//   c  = r^2 * mean_k(gamma * dn_s * x),
//   dgamma[k] += sum_t dn[t,k]*x_hat[t,k] = sum_t dn_s[t,k]*x[t,k].
// Lane l owns the 8-column chunks l, l+32, ...; its share of dgamma stays in
// registers for all of the CTA's rows, then the CTA adds its warps' shares in
// warp order and writes one partial row; dgamma_finalize adds the partials in
// CTA order, so the result does not depend on timing.
// kScaleDn = true takes the plain gradient dn of the normalised output and
// applies the row's rstd to it in the kernel (dn_s = rstd * dn).
template <class T, int NCH, bool kScaleDn = false>
__global__ void __launch_bounds__(kRowThreads)
rmsnorm_bwd_kernel(const T *__restrict__ x, const float *__restrict__ dn_s, const T *__restrict__ dy,
                   const float *__restrict__ rstd, const T *__restrict__ gamma, T *__restrict__ dx,
                   float *__restrict__ dg_part, int64_t T_rows, int64_t d, int64_t rows_per_cta) {
    extern __shared__ float sm[];
    float *g_s = sm;        // gamma as float [d]
    float *red = sm + d;    // dgamma share of the CTA [d]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int64_t i = threadIdx.x * 8; i < d; i += kRowThreads * 8) {
        float v[8];
        Io8<T>::load(gamma + i, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) g_s[i + j] = v[j];
    }
    __syncthreads();

    float acc[NCH][8];
#pragma unroll
    for (int j = 0; j < NCH; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;

    const int64_t t0 = blockIdx.x * rows_per_cta;
    const int64_t t1 = min(T_rows, t0 + rows_per_cta);
    const float inv_d = 1.0f / static_cast<float>(d);
    for (int64_t t = t0 + warp; t < t1; t += kRowThreads / 32) {
        const T *xr = x + t * d;
        const float *nr = dn_s + t * d;
        const float rr = kScaleDn ? rstd[t] : 1.0f;
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int64_t c = (lane + 32 * j) * 8;
            if (c < d) {
                float xv[8], nv[8];
                Io8<T>::load(xr + c, xv);
                Io8<float>::load(nr + c, nv);
                if (kScaleDn) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) nv[i] *= rr;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) s += g_s[c + i] * nv[i] * xv[i];
            }
        }
        s = warp_sum(s);
        const float r = rstd[t];
        const float cr = r * r * s * inv_d;
        const T *dyr = dy + t * d;
        T *dxr = dx + t * d;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int64_t c = (lane + 32 * j) * 8;
            if (c < d) {
                float xv[8], nv[8], gv[8], o[8];
                Io8<T>::load(xr + c, xv);
                Io8<float>::load(nr + c, nv);
                if (kScaleDn) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) nv[i] *= rr;
                }
                Io8<T>::load(dyr + c, gv);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[i] = gv[i] + g_s[c + i] * nv[i] - xv[i] * cr;
                    acc[j][i] += nv[i] * xv[i];
                }
                Io8<T>::store(dxr + c, o);
            }
        }
    }

    // CTA share of dgamma: warps add in order 0, 1, ..., 7.
    for (int w = 0; w < kRowThreads / 32; ++w) {
        if (warp == w) {
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const int64_t c = (lane + 32 * j) * 8;
                if (c < d) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) red[c + i] = (w == 0 ? 0.0f : red[c + i]) + acc[j][i];
                }
            }
        }
        __syncthreads();
    }
    float *out = dg_part + blockIdx.x * d;
    for (int64_t i = threadIdx.x; i < d; i += kRowThreads) out[i] = red[i];
}

// dgamma[k] += sum_p part[p][k], p in increasing order.
__global__ void dgamma_finalize_kernel(const float *__restrict__ part, int parts,
                                       float *__restrict__ dgamma, int64_t d) {
    const int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (k >= d) return;
    float s = 0.0f;
    for (int p = 0; p < parts; ++p) s += part[p * d + k];
    dgamma[k] += s;
}

__global__ void fill_zero_kernel(float4 *p, int64_t n4) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

__global__ void scale_kernel(float4 *p, int64_t n4, float s) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 v = p[i];
        v.x *= s;
        v.y *= s;
        v.z *= s;
        v.w *= s;
        p[i] = v;
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

int status() { return launch_status(); }

template <class E, int NCH, bool kScaleDn = false>
int run_norm_bwd(const void *x, const float *dn_s, const void *dy, const float *rstd,
                 const void *gamma, void *dx, float *part, int64_t T, int64_t d, int parts,
                 cudaStream_t s) {
    const int64_t rows_per_cta = (T + parts - 1) / parts;
    const size_t smem = static_cast<size_t>(2 * d) * sizeof(float);
    rmsnorm_bwd_kernel<E, NCH, kScaleDn><<<parts, kRowThreads, smem, s>>>(
        static_cast<const E *>(x), dn_s, static_cast<const E *>(dy), rstd,
        static_cast<const E *>(gamma), static_cast<E *>(dx), part, T, d, rows_per_cta);
    return status();
}

template <class E, bool kScaleDn = false>
int dispatch_norm_bwd(const void *x, const float *dn_s, const void *dy, const float *rstd,
                      const void *gamma, void *dx, float *part, int64_t T, int64_t d, int parts,
                      cudaStream_t s) {
    const int64_t nch = (d + 255) / 256;
#define MLPBLK_NB(N) \
    if (nch <= N) return run_norm_bwd<E, N, kScaleDn>(x, dn_s, dy, rstd, gamma, dx, part, T, d, parts, s)
    MLPBLK_NB(1);
    MLPBLK_NB(2);
    MLPBLK_NB(3);
    MLPBLK_NB(4);
    MLPBLK_NB(6);
    MLPBLK_NB(8);
    MLPBLK_NB(12);
    MLPBLK_NB(16);
#undef MLPBLK_NB
    return MLPBLK_ENOTSUP;
}

}  // namespace

int launch_fold_gamma(int dtype, const void *w1, const void *gamma, void *w1g, int64_t F,
                      int64_t d, cudaStream_t s) {
    const int64_t groups = F * d / 8;
    const int grid = grid_for(groups, 256);
    if (dtype == MLPBLK_BF16)
        fold_gamma_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t *>(w1),
                                                        static_cast<const uint16_t *>(gamma),
                                                        static_cast<uint16_t *>(w1g), groups, d);
    else
        fold_gamma_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(w1),
                                                     static_cast<const float *>(gamma),
                                                     static_cast<float *>(w1g), groups, d);
    return status();
}

int launch_rstd_f32(const float *x, float *rstd, int64_t T, int64_t d, float eps, cudaStream_t s) {
    rstd_f32_kernel<<<grid_for(T * 32, 256), 256, 0, s>>>(x, rstd, T, d, eps);
    return status();
}

int launch_rmsnorm_bwd(int dtype, const void *x, const float *dn_s, const void *dy,
                       const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                       int64_t T, int64_t d, int parts, cudaStream_t s) {
    if (dtype == MLPBLK_BF16)
        return dispatch_norm_bwd<uint16_t>(x, dn_s, dy, rstd, gamma, dx, dgamma_part, T, d, parts, s);
    return dispatch_norm_bwd<float>(x, dn_s, dy, rstd, gamma, dx, dgamma_part, T, d, parts, s);
}

int launch_rmsnorm_bwd_unscaled(int dtype, const void *x, const float *dn, const void *dy,
                                const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                                int64_t T, int64_t d, int parts, cudaStream_t s) {
    if (dtype == MLPBLK_BF16)
        return dispatch_norm_bwd<uint16_t, true>(x, dn, dy, rstd, gamma, dx, dgamma_part, T, d, parts, s);
    return dispatch_norm_bwd<float, true>(x, dn, dy, rstd, gamma, dx, dgamma_part, T, d, parts, s);
}

int launch_dgamma_finalize(const float *part, int parts, float *dgamma, int64_t d, cudaStream_t s) {
    dgamma_finalize_kernel<<<static_cast<int>((d + 255) / 256), 256, 0, s>>>(part, parts, dgamma, d);
    return status();
}

int launch_fill_zero(float *p, int64_t n, cudaStream_t s) {
    const int64_t n4 = n / 4;
    fill_zero_kernel<<<grid_for(n4, 256), 256, 0, s>>>(reinterpret_cast<float4 *>(p), n4);
    return status();
}

int launch_scale(float *p, int64_t n, float sc, cudaStream_t s) {
    const int64_t n4 = n / 4;
    scale_kernel<<<grid_for(n4, 256), 256, 0, s>>>(reinterpret_cast<float4 *>(p), n4, sc);
    return status();
}

}  // namespace mlpblk
