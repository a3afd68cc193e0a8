// gemm_fwd.cu -- tensor-core GEMMs of the block forward.
//   W1 GEMM: acc = x . (W1*gamma)^T; rstd from the x stages (RMSNorm prologue);
//            epilogue h = rstd*acc, a = relu(h)^2      ("Kernel 3: Dense ReLU2 ...")
//   W2 GEMM: y = x + a . W2^T                           (residual add in the epilogue)
#include "gemm_tc.cuh"

namespace mlpblk {

int launch_gemm_tc_fwd(int epi, int M, int N, int K, const void *A, const void *B, void *C0,
                       void *C1, const GemmArgs &extra, int num_sms, cudaStream_t s) {
    const int bn = choose_bn(M, N, K, false, num_sms);
    if (epi == kEpiFwdW1) {
        return bn == 256
                   ? run_gemm_tc<GemmCfg<256, kEpiFwdW1, false, false>>(M, N, K, A, B, C0, C1, extra, num_sms, s)
                   : run_gemm_tc<GemmCfg<128, kEpiFwdW1, false, false>>(M, N, K, A, B, C0, C1, extra, num_sms, s);
    }
    if (epi == kEpiFwdW2) {
        return bn == 256
                   ? run_gemm_tc<GemmCfg<256, kEpiFwdW2, false, false>>(M, N, K, A, B, C0, C1, extra, num_sms, s)
                   : run_gemm_tc<GemmCfg<128, kEpiFwdW2, false, false>>(M, N, K, A, B, C0, C1, extra, num_sms, s);
    }
    return MLPBLK_EINVAL;
}

int take_device_error_gemm_fwd() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLPBLK_ECUDA;
    if (v != 0) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
    return v;
}

}  // namespace mlpblk
