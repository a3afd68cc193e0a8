// gemm_fwd.cu -- tensor-core GEMMs of the block forward.
//   W1 GEMM: acc = x . (W1*gamma)^T, epilogue h = rstd*acc, a = relu(h)^2
//            ("Kernel 3: Dense ReLU2 ..."); rstd comes from the preceding
//            statistics pass (kEpiFwdW1Pre) or from the GEMM's own RMSNorm
//            prologue warps reading the x stages (kEpiFwdW1)
//   W2 GEMM: y = x + a . W2^T                           (residual add in the epilogue)
#include <stdlib.h>

#include "gemm_tc.cuh"

namespace mlpblk {

int launch_gemm_tc_fwd(int epi, int M, int N, int K, const void *A, const void *B, void *C0,
                       void *C1, const GemmArgs &extra, int num_sms, cudaStream_t s) {
    // Pair tiles except for the W1 GEMM with the in-kernel RMSNorm prologue: in
    // pair mode its shared-memory reads slow the partner SM's operand reads
    // (measured 2.3x slower), so that variant keeps single-CTA tiles.
    const int mode = choose_tile(M, N, K, false, num_sms, pair_tiles_enabled() && epi != kEpiFwdW1);
#define MLPBLK_RUN(E)                                                                                   \
    switch (mode) {                                                                                     \
        case kTilePair256:                                                                              \
            return run_gemm_tc<GemmCfg<256, E, false, false, true>>(M, N, K, A, B, C0, C1, extra, num_sms, s); \
        case kTile256:                                                                                  \
            return run_gemm_tc<GemmCfg<256, E, false, false>>(M, N, K, A, B, C0, C1, extra, num_sms, s); \
        default:                                                                                        \
            return run_gemm_tc<GemmCfg<128, E, false, false>>(M, N, K, A, B, C0, C1, extra, num_sms, s); \
    }
    if (epi == kEpiFwdW1) { MLPBLK_RUN(kEpiFwdW1) }
    if (epi == kEpiFwdW1Pre) { MLPBLK_RUN(kEpiFwdW1Pre) }
    if (epi == kEpiFwdW2) { MLPBLK_RUN(kEpiFwdW2) }
#undef MLPBLK_RUN
    return MLPBLK_EINVAL;
}

int take_device_error_gemm_fwd() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLPBLK_ECUDA;
    if (v != 0) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
    return v;
}

}  // namespace mlpblk
