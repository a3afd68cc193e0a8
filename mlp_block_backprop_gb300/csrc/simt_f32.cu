// simt_f32.cu -- fp32 CUDA-core GEMM with the block's epilogues, for the fp32
// element type.  No tensor-core kind keeps fp32 accuracy (TF32 has a 10-bit
// mantissa), so the fp32 path multiplies with FFMA.  It carries the same fused
// epilogues as the tensor-core path and follows the same data flow (gamma folded
// into W1, rstd folded into dh).
#include "mlpblk_internal.h"

namespace mlpblk {

namespace {

constexpr int kTile = 64;
constexpr int kTk = 16;

// C[m,n] = sum_k A(m,k) B(n,k); 256 threads, each a 4x4 block of C.
template <int EPI>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const float *__restrict__ A, int64_t sam, int64_t sak, const float *__restrict__ B,
                 int64_t sbn, int64_t sbk, int M, int N, int K, float *__restrict__ C0,
                 float *__restrict__ C1, SimtEpi e) {
    __shared__ float As[kTk][kTile + 4];
    __shared__ float Bs[kTk][kTile + 4];
    griddep_enter();
    const int tx = threadIdx.x % 16;
    const int ty = threadIdx.x / 16;
    const int m0 = blockIdx.y * kTile;
    const int n0 = blockIdx.x * kTile;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += kTk) {
        for (int i = threadIdx.x; i < kTk * kTile; i += 256) {
            const int kk = i / kTile, mm = i % kTile;
            const int m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < M && k < K) ? A[m * sam + k * sak] : 0.0f;
            const int n = n0 + mm;
            Bs[kk][mm] = (n < N && k < K) ? B[n * sbn + k * sbk] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kTk; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            const int64_t o = static_cast<int64_t>(m) * N + n;
            const float v = acc[i][j];
            if (EPI == kEpiFwdW1) {
                const float h = e.rstd[m] * v;
                C0[o] = h;
                C1[o] = h > 0.0f ? h * h : 0.0f;
            } else if (EPI == kEpiFwdW2) {
                C0[o] = e.aux[o] + v;
            } else if (EPI == kEpiDgradH) {
                const float h = e.aux[o];
                C0[o] = h > 0.0f ? e.rstd[m] * v * (2.0f * h) : 0.0f;
            } else if (EPI == kEpiStoreF32) {
                C0[o] = v;
            } else if (EPI == kEpiAccF32) {
                C0[o] += v;
            } else {  // kEpiAccF32ColScale
                C0[o] += e.colscale[n] * v;
            }
        }
    }
}

}  // namespace

int launch_gemm_simt(int epi, int M, int N, int K, const float *A, int64_t sam, int64_t sak,
                     const float *B, int64_t sbn, int64_t sbk, float *C0, float *C1,
                     const SimtEpi &e, cudaStream_t s) {
    dim3 grid((N + kTile - 1) / kTile, (M + kTile - 1) / kTile);
    switch (epi) {
#define MLPBLK_SIMT(E) \
    case E: return launch_pdl(gemm_simt_kernel<E>, grid, dim3(256), 0, s, A, sam, sak, B, sbn, sbk, M, N, K, C0, C1, e)
        MLPBLK_SIMT(kEpiFwdW1);
        MLPBLK_SIMT(kEpiFwdW2);
        MLPBLK_SIMT(kEpiDgradH);
        MLPBLK_SIMT(kEpiStoreF32);
        MLPBLK_SIMT(kEpiAccF32);
        MLPBLK_SIMT(kEpiAccF32ColScale);
#undef MLPBLK_SIMT
        default: return MLPBLK_EINVAL;
    }
    return launch_status();
}

}  // namespace mlpblk
