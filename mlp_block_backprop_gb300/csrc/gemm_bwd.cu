// gemm_bwd.cu -- tensor-core GEMMs of the block backward (MatMul rule g.B^T and
// A^T.g of "Reverse-mode automatic differentiation", section 5):
//   dgrad h : dh_s = rstd * (dy . W2) * 2 relu(h)       (ReLU^2 gate in the epilogue;
//                                                         W2 read MN-major)
//   wgrad W2: dW2 += dy^T . a                             (both operands MN-major)
//   dgrad n : dn_s = dh_s . W1                            (bf16 out, or fp32 on the FP8
//                                                         path; W1 MN-major)
//   wgrad W1: dW1 += (dh_s^T . x) * gamma[col]            (both operands MN-major;
//             for d_model <= 768 its side warps also run the RMSNorm backward rows)
// dh_s = rstd*dh and dn_s = rstd*dn carry the per-row RMSNorm scale, so the
// normalised input n never has to be stored or rebuilt: dh^T.n = (dh_s^T.x)*gamma.
#include <stdlib.h>

#include "gemm_tc.cuh"

namespace mlpblk {

int launch_gemm_tc_bwd(int epi, int M, int N, int K, const void *A, const void *B, void *C0,
                       void *C1, const GemmArgs &extra, int num_sms, cudaStream_t s) {
    // B is MN-major in every backward GEMM, so only 256-wide pairs exist
    const int pairs = pair_tiles_enabled() ? kAllowPair256 : 0;
    const bool reduce = epi == kEpiAccF32 || epi == kEpiAccF32ColScale || epi == kEpiAccF32ColScaleNorm;
    const int choice = choose_tile(M, N, K, streamk_enabled(), reduce, num_sms, pairs);
    const int mode = choice & ~kUseStreamK;
    GemmArgs args = extra;
    args.whole_tiles = (choice & kUseStreamK) ? 0 : 1;
#define MLPBLK_RUN_MODE(E, AMN, BNV, PAIRV) \
    return run_gemm_tc<GemmCfg<BNV, E, AMN, true, PAIRV>>(M, N, K, A, B, C0, C1, args, num_sms, s)
#define MLPBLK_RUN_SINGLE(E, AMN)                           \
    switch (mode) {                                         \
        case kTile256: MLPBLK_RUN_MODE(E, AMN, 256, false); \
        case kTile192: MLPBLK_RUN_MODE(E, AMN, 192, false); \
        default: MLPBLK_RUN_MODE(E, AMN, 128, false);       \
    }
#define MLPBLK_RUN(E, AMN)                                                   \
    if (mode == kTilePair256) { MLPBLK_RUN_MODE(E, AMN, 256, true); }       \
    MLPBLK_RUN_SINGLE(E, AMN)
    switch (epi) {
        case kEpiDgradH: { MLPBLK_RUN(kEpiDgradH, false) }
        case kEpiStoreF32: { MLPBLK_RUN(kEpiStoreF32, false) }
        case kEpiStoreBf16: { MLPBLK_RUN(kEpiStoreBf16, false) }
        case kEpiAccF32: { MLPBLK_RUN(kEpiAccF32, true) }
        case kEpiAccF32ColScale: { MLPBLK_RUN(kEpiAccF32ColScale, true) }
        case kEpiAccF32ColScaleNorm: { MLPBLK_RUN(kEpiAccF32ColScaleNorm, true) }
        default: return MLPBLK_EINVAL;
    }
#undef MLPBLK_RUN
#undef MLPBLK_RUN_SINGLE
#undef MLPBLK_RUN_MODE
}

int take_device_error_gemm_bwd() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLPBLK_ECUDA;
    if (v != 0) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
    return v;
}

}  // namespace mlpblk
