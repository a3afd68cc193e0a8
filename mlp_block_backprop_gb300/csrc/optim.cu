// optim.cu -- the optimizer-side steps next to the block ("grow_a_language_model_
// backprop": the two-stage gradient-norm reduction and the gradient scale used for
// clipping, and AdamW with its two moment buffers per weight).  All HBM-bound.
//
//   grad norm, stage 1: each CTA sums g^2 over a fixed slice of the gradients
//                       (float32 with a compensation term per thread, then float64
//                       across the CTA) and writes one float64 partial;
//   grad norm, stage 2: one CTA adds the partials in CTA order, norm = sqrt(sum),
//                       clip scale = min(1, max_norm / (norm + 1e-6));
//   clip:               g *= scale, the scale read from device memory;
//   AdamW:              decoupled weight decay, bias-corrected moments, on float32
//                       master weights, writing the working copy in the block's
//                       element type (bf16 rounded to nearest even).
// The partition and every sum order are fixed, so results do not depend on timing.
#include "mlpblk_internal.h"

namespace mlpblk {

namespace {

constexpr int kNormThreads = 256;

struct GradList {
    const float4 *p[3];
    int64_t n4[3];  // float4 elements per tensor
};

__device__ __forceinline__ float sumsq4(float4 v) { return v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w; }

// Compensated float32 accumulation (s, comp) += q.
__device__ __forceinline__ void kahan_add(float &s, float &comp, float q) {
    const float y = q - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
}

// Stage 1.  Each tensor is cut into gridDim.x equal slices; CTA b sums slice b of
// every tensor.  Four independent 16-byte loads per thread are in flight per
// iteration, then added in index order.
__global__ void __launch_bounds__(kNormThreads)
grad_norm_partial_kernel(GradList g, double *partial) {
    __shared__ double red[kNormThreads / 32];
    griddep_enter();
    float s = 0.0f, comp = 0.0f;
    for (int t = 0; t < 3; ++t) {
        const float4 *p = g.p[t];
        const int64_t n = g.n4[t];
        const int64_t per = (n + gridDim.x - 1) / gridDim.x;
        const int64_t b0 = blockIdx.x * per;
        const int64_t b1 = min(n, b0 + per);
        int64_t i = b0 + threadIdx.x;
        for (; i + 3 * kNormThreads < b1; i += 4 * kNormThreads) {
            const float4 v0 = __ldg(p + i);
            const float4 v1 = __ldg(p + i + kNormThreads);
            const float4 v2 = __ldg(p + i + 2 * kNormThreads);
            const float4 v3 = __ldg(p + i + 3 * kNormThreads);
            kahan_add(s, comp, sumsq4(v0));
            kahan_add(s, comp, sumsq4(v1));
            kahan_add(s, comp, sumsq4(v2));
            kahan_add(s, comp, sumsq4(v3));
        }
        for (; i < b1; i += kNormThreads) kahan_add(s, comp, sumsq4(__ldg(p + i)));
    }
    double d = static_cast<double>(s) - static_cast<double>(comp);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kNormThreads / 32; ++w) t += red[w];
        partial[blockIdx.x] = t;
    }
}

// Stage 2.  One CTA of 32 threads: lane l adds partials l, l+32, ... in order,
// then lane 0 adds the 32 lane sums in lane order.
__global__ void grad_norm_final_kernel(const double *partial, int parts, float max_norm, float *norm_out,
                                       float *scale_out) {
    __shared__ double lanes[32];
    griddep_enter();
    double s = 0.0;
    for (int p = threadIdx.x; p < parts; p += 32) s += partial[p];
    lanes[threadIdx.x] = s;
    __syncwarp();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int l = 0; l < 32; ++l) t += lanes[l];
        const double norm = sqrt(t);
        if (norm_out) *norm_out = static_cast<float>(norm);
        if (scale_out) {
            const double c = static_cast<double>(max_norm) / (norm + 1e-6);
            *scale_out = static_cast<float>(c < 1.0 ? c : 1.0);
        }
    }
}

struct MutGradList {
    float4 *p[3];
    int64_t n4[3];
};

// g *= scale[0] over the three tensors' concatenated float4 index space.
__global__ void clip_grads_kernel(MutGradList g, const float *__restrict__ scale) {
    griddep_enter();
    const float c = *scale;
    const int64_t total = g.n4[0] + g.n4[1] + g.n4[2];
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t j = i;
        int t = 0;
        while (t < 2 && j >= g.n4[t]) j -= g.n4[t++];
        float4 v = g.p[t][j];
        v.x *= c;
        v.y *= c;
        v.z *= c;
        v.w *= c;
        g.p[t][j] = v;
    }
}

constexpr int kMaxAdamTensors = 8;

struct AdamList {
    float *master[kMaxAdamTensors];
    void *weight[kMaxAdamTensors];
    const float *grad[kMaxAdamTensors];
    float *m[kMaxAdamTensors];
    float *v[kMaxAdamTensors];
    int64_t n4[kMaxAdamTensors];
    float decay_factor[kMaxAdamTensors];  // 1 - lr*wd, or 1 where the tensor takes no decay
    int count;
};

struct AdamScalars {
    float beta1, one_minus_beta1, beta2, one_minus_beta2;
    float step_size;     // lr / (1 - beta1^t)
    float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
    float eps;
};

__device__ __forceinline__ uint32_t bf16_rne_pair(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float adam_one(float w, float g, float &m, float &v, float decay,
                                          const AdamScalars &k, const float gs) {
    g *= gs;
    w *= decay;
    m = k.beta1 * m + k.one_minus_beta1 * g;
    v = k.beta2 * v + k.one_minus_beta2 * (g * g);
    const float denom = sqrtf(v) * k.inv_sqrt_bc2 + k.eps;
    return w - k.step_size * (m / denom);
}

template <bool kBf16>
__global__ void adamw_kernel(AdamList L, AdamScalars k, const float *__restrict__ grad_scale) {
    griddep_enter();
    const float gs = grad_scale ? *grad_scale : 1.0f;
    int64_t total = 0;
    for (int t = 0; t < L.count; ++t) total += L.n4[t];
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t j = i;
        int t = 0;
        while (t < L.count - 1 && j >= L.n4[t]) j -= L.n4[t++];
        float4 w = reinterpret_cast<const float4 *>(L.master[t])[j];
        const float4 g = __ldg(reinterpret_cast<const float4 *>(L.grad[t]) + j);
        float4 m = reinterpret_cast<const float4 *>(L.m[t])[j];
        float4 v = reinterpret_cast<const float4 *>(L.v[t])[j];
        const float dec = L.decay_factor[t];
        w.x = adam_one(w.x, g.x, m.x, v.x, dec, k, gs);
        w.y = adam_one(w.y, g.y, m.y, v.y, dec, k, gs);
        w.z = adam_one(w.z, g.z, m.z, v.z, dec, k, gs);
        w.w = adam_one(w.w, g.w, m.w, v.w, dec, k, gs);
        reinterpret_cast<float4 *>(L.master[t])[j] = w;
        reinterpret_cast<float4 *>(L.m[t])[j] = m;
        reinterpret_cast<float4 *>(L.v[t])[j] = v;
        if (L.weight[t]) {
            if (kBf16) {
                uint2 o;
                o.x = bf16_rne_pair(w.x, w.y);
                o.y = bf16_rne_pair(w.z, w.w);
                reinterpret_cast<uint2 *>(L.weight[t])[j] = o;
            } else {
                reinterpret_cast<float4 *>(L.weight[t])[j] = w;
            }
        }
    }
}

int sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

int elementwise_grid(int64_t items) {
    const int64_t want = (items + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms()) * 8;
    return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

int launch_grad_norm_partial(const float *g0, int64_t n0, const float *g1, int64_t n1, const float *g2,
                             int64_t n2, double *partial, int max_parts, int *parts_out, cudaStream_t s) {
    GradList g;
    g.p[0] = reinterpret_cast<const float4 *>(g0);
    g.p[1] = reinterpret_cast<const float4 *>(g1);
    g.p[2] = reinterpret_cast<const float4 *>(g2);
    g.n4[0] = n0 / 4;
    g.n4[1] = n1 / 4;
    g.n4[2] = n2 / 4;
    // four CTAs per SM keep ~10 MB of loads in flight; tiny inputs get fewer
    int64_t parts = static_cast<int64_t>(sms()) * 4;
    const int64_t biggest = g.n4[0] > g.n4[1] ? (g.n4[0] > g.n4[2] ? g.n4[0] : g.n4[2])
                                              : (g.n4[1] > g.n4[2] ? g.n4[1] : g.n4[2]);
    const int64_t useful = (biggest + kNormThreads - 1) / kNormThreads;
    if (parts > useful) parts = useful;
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    *parts_out = static_cast<int>(parts);
    return launch_pdl(grad_norm_partial_kernel, dim3(static_cast<unsigned>(parts)), dim3(kNormThreads), 0, s,
                      g, partial);
}

int launch_grad_norm_final(const double *partial, int parts, float max_norm, float *norm_out, float *scale_out,
                           cudaStream_t s) {
    return launch_pdl(grad_norm_final_kernel, dim3(1), dim3(32), 0, s, partial, parts, max_norm, norm_out,
                      scale_out);
}

int launch_clip_grads(float *g0, int64_t n0, float *g1, int64_t n1, float *g2, int64_t n2, const float *scale,
                      cudaStream_t s) {
    MutGradList g;
    g.p[0] = reinterpret_cast<float4 *>(g0);
    g.p[1] = reinterpret_cast<float4 *>(g1);
    g.p[2] = reinterpret_cast<float4 *>(g2);
    g.n4[0] = n0 / 4;
    g.n4[1] = n1 / 4;
    g.n4[2] = n2 / 4;
    return launch_pdl(clip_grads_kernel, dim3(elementwise_grid(g.n4[0] + g.n4[1] + g.n4[2])), dim3(256), 0, s,
                      g, scale);
}

int launch_adamw(const AdamTensor *tensors, int count, float lr, float beta1, float beta2, float eps,
                 float weight_decay, int64_t step, bool bf16, const float *grad_scale, cudaStream_t s) {
    const double bc1 = 1.0 - pow(static_cast<double>(beta1), static_cast<double>(step));
    const double bc2 = 1.0 - pow(static_cast<double>(beta2), static_cast<double>(step));
    AdamScalars k;
    k.beta1 = beta1;
    k.one_minus_beta1 = 1.0f - beta1;
    k.beta2 = beta2;
    k.one_minus_beta2 = 1.0f - beta2;
    k.step_size = static_cast<float>(static_cast<double>(lr) / bc1);
    k.inv_sqrt_bc2 = static_cast<float>(1.0 / sqrt(bc2));
    k.eps = eps;
    const float decay = static_cast<float>(1.0 - static_cast<double>(lr) * static_cast<double>(weight_decay));
    for (int base = 0; base < count; base += kMaxAdamTensors) {
        AdamList L = {};
        L.count = count - base < kMaxAdamTensors ? count - base : kMaxAdamTensors;
        int64_t total = 0;
        for (int t = 0; t < L.count; ++t) {
            const AdamTensor &a = tensors[base + t];
            L.master[t] = a.master;
            L.weight[t] = a.weight;
            L.grad[t] = a.grad;
            L.m[t] = a.m;
            L.v[t] = a.v;
            L.n4[t] = a.n / 4;
            L.decay_factor[t] = a.decay ? decay : 1.0f;
            total += L.n4[t];
        }
        const int rc = bf16 ? launch_pdl(adamw_kernel<true>, dim3(elementwise_grid(total)), dim3(256), 0, s, L, k,
                                         grad_scale)
                            : launch_pdl(adamw_kernel<false>, dim3(elementwise_grid(total)), dim3(256), 0, s, L,
                                         k, grad_scale);
        if (rc != MLPBLK_OK) return rc;
    }
    return MLPBLK_OK;
}

}  // namespace mlpblk
