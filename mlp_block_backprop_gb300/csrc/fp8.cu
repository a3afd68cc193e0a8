// fp8.cu -- E4M3 quantisation for the FP8-operand variant of the block's GEMMs
// ("Nemotron Kernels From Inference To Backpropagation" -- "Where Quantization
// Fits": a storage and arithmetic policy for particular tensor edges).
//
// Per-tensor scaling: amax = max |v| over the tensor (two launches: per-CTA
// maxima, then one CTA), codes q = E4M3(v * (448 / amax)) rounded to nearest
// even and saturated, dequantised by s = amax / 448 in the GEMM epilogue.  The
// normalised input n' = x * rstd needs no amax: |n'| <= sqrt(d) <= 64 < 448 for
// every row, so its scale is 1 and it is written by the statistics kernel that
// computes rstd.  All HBM-bound, 16-byte accesses.
#include "mlpblk_internal.h"

namespace mlpblk {

namespace {

constexpr int kQThreads = 256;
constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Two floats -> two E4M3 bytes (lo in the low byte), nearest-even, saturating.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
    return r;
}

// 8 bf16 values (one 16-byte load) as floats.
__device__ __forceinline__ void load8(const uint16_t *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    v[0] = bf16f(u.x & 0xFFFFu); v[1] = bf16f(u.x >> 16);
    v[2] = bf16f(u.y & 0xFFFFu); v[3] = bf16f(u.y >> 16);
    v[4] = bf16f(u.z & 0xFFFFu); v[5] = bf16f(u.z >> 16);
    v[6] = bf16f(u.w & 0xFFFFu); v[7] = bf16f(u.w >> 16);
}

// 8 floats * inv -> 8 E4M3 bytes (one 8-byte store).
__device__ __forceinline__ void store8(uint8_t *p, const float (&v)[8], float inv) {
    uint2 o;
    o.x = static_cast<uint32_t>(e4m3x2(v[0] * inv, v[1] * inv)) |
          (static_cast<uint32_t>(e4m3x2(v[2] * inv, v[3] * inv)) << 16);
    o.y = static_cast<uint32_t>(e4m3x2(v[4] * inv, v[5] * inv)) |
          (static_cast<uint32_t>(e4m3x2(v[6] * inv, v[7] * inv)) << 16);
    *reinterpret_cast<uint2 *>(p) = o;
}

// Stage 1 of amax: CTA b takes groups of 8 values [b*per, (b+1)*per); a value is
// v[i] (bf16), times colmul[i % cols] when colmul is given (W1 * gamma).
__global__ void __launch_bounds__(kQThreads)
amax_partial_kernel(const uint16_t *__restrict__ v, const uint16_t *__restrict__ colmul, int64_t cols,
                    int64_t groups, int64_t per, float *__restrict__ partial) {
    __shared__ float red[kQThreads / 32];
    griddep_enter();
    const int64_t g0 = blockIdx.x * per;
    const int64_t g1 = min(groups, g0 + per);
    float m = 0.0f;
    // four 16-byte loads in flight per thread
    for (int64_t g = g0 + threadIdx.x; g < g1; g += 4 * kQThreads) {
        float x[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t gu = g + u * kQThreads;
            if (gu < g1) load8(v + gu * 8, x[u]);
            else
#pragma unroll
                for (int i = 0; i < 8; ++i) x[u][i] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t gu = g + u * kQThreads;
            if (colmul && gu < g1) {
                float c[8];
                load8(colmul + (gu * 8) % cols, c);
#pragma unroll
                for (int i = 0; i < 8; ++i) x[u][i] *= c[i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[u][i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < kQThreads / 32; ++w) t = fmaxf(t, red[w]);
        partial[blockIdx.x] = t;
    }
}

// Stage 2: one warp.  scale = {amax, 448 / amax, amax / 448, 0} (1, 1 for a zero
// tensor); also zeroes the next GEMM's stream-K flags when asked.
__global__ void scale_final_kernel(const float *__restrict__ partial, int parts, float *__restrict__ scale,
                                   int *zero_flags, int zero_count) {
    griddep_enter();
    if (zero_flags)
        for (int i = threadIdx.x; i < zero_count; i += 32) zero_flags[i] = 0;
    float m = 0.0f;
    for (int p = threadIdx.x; p < parts; p += 32) m = fmaxf(m, partial[p]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) {
        scale[0] = m;
        scale[1] = m > 0.0f ? kE4M3Max / m : 1.0f;
        scale[2] = m > 0.0f ? m / kE4M3Max : 1.0f;
        scale[3] = 0.0f;
    }
}

// q = E4M3(v * colmul * scale[1]) over groups of 8 values.
__global__ void quantize_kernel(const uint16_t *__restrict__ v, const uint16_t *__restrict__ colmul,
                                int64_t cols, int64_t groups, const float *__restrict__ scale,
                                uint8_t *__restrict__ q) {
    griddep_enter();
    const float inv = scale[1];
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float x[8];
        load8(v + g * 8, x);
        if (colmul) {
            float c[8];
            load8(colmul + (g * 8) % cols, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] *= c[i];
        }
        store8(q + g * 8, x, inv);
    }
}

// rstd[t] = 1/sqrt(mean_k x^2 + eps) and n8[t,:] = E4M3(x[t,:] * rstd[t]) (scale 1).
// One warp per row; the row's second read comes from L1/L2.
__global__ void __launch_bounds__(256)
norm_quant_kernel(const uint16_t *__restrict__ x, float *__restrict__ rstd, uint8_t *__restrict__ n8,
                  int64_t T, int64_t d, float eps, int *zero_flags, int zero_count) {
    griddep_enter();
    // the next GEMM's stream-K flags start from zero
    if (zero_flags && blockIdx.x == 0)
        for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_flags[i] = 0;
    const int lane = threadIdx.x & 31;
    const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const float inv_d = 1.0f / static_cast<float>(d);
    for (int64_t t = wid; t < T; t += nw) {
        const uint16_t *row = x + t * d;
        float ss = 0.0f;
        for (int64_t c = lane * 8; c < d; c += 256) {
            float v[8];
            load8(row + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) ss += v[i] * v[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = 1.0f / sqrtf(ss * inv_d + eps);
        if (lane == 0) rstd[t] = r;
        for (int64_t c = lane * 8; c < d; c += 256) {
            float v[8];
            load8(row + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= r;
            store8(n8 + t * d + c, v, 1.0f);
        }
    }
}

int sm_total() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

int launch_amax_e4m3(const void *v, const void *colmul, int64_t cols, int64_t n, float *partial, int max_parts,
                     int *parts_out, cudaStream_t s) {
    const int64_t groups = n / 8;
    int64_t parts = static_cast<int64_t>(sm_total()) * 4;
    const int64_t useful = (groups + kQThreads - 1) / kQThreads;
    if (parts > useful) parts = useful;
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    int64_t per = (groups + parts - 1) / parts;
    if (per < 1) per = 1;
    parts = (groups + per - 1) / per;
    if (parts < 1) parts = 1;
    *parts_out = static_cast<int>(parts);
    return launch_pdl(amax_partial_kernel, dim3(static_cast<unsigned>(parts)), dim3(kQThreads), 0, s,
                      static_cast<const uint16_t *>(v), static_cast<const uint16_t *>(colmul), cols, groups, per,
                      partial);
}

int launch_scale_e4m3(const float *partial, int parts, float *scale, int *zero_flags, int zero_count,
                      cudaStream_t s) {
    return launch_pdl(scale_final_kernel, dim3(1), dim3(32), 0, s, partial, parts, scale, zero_flags, zero_count);
}

int launch_apply_e4m3(const void *v, const void *colmul, int64_t cols, int64_t n, const float *scale, uint8_t *q,
                      cudaStream_t s) {
    const int64_t groups = n / 8;
    int64_t grid = (groups + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_total()) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_pdl(quantize_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(v), static_cast<const uint16_t *>(colmul), cols, groups, scale, q);
}

int launch_norm_quant(const void *x, float *rstd, uint8_t *n8, int64_t T, int64_t d, float eps, int *zero_flags,
                      int zero_count, cudaStream_t s) {
    int64_t blocks = (T * 32 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_total()) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(norm_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(x), rstd, n8, T, d, eps, zero_flags, zero_count);
}

}  // namespace mlpblk
