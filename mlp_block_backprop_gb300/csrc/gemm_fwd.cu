// gemm_fwd.cu -- tensor-core GEMMs of the block forward.
//   W1 GEMM: acc = x . (W1*gamma)^T, epilogue h = rstd*acc, a = relu(h)^2
//            ("Kernel 3: Dense ReLU2 ..."); rstd comes from the preceding
//            statistics pass (kEpiFwdW1Pre) or from the GEMM's own RMSNorm
//            prologue warps reading the x stages (kEpiFwdW1)
//   W2 GEMM: y = x + a . W2^T                           (residual add in the epilogue)
//   W1 GEMM, a only (kEpiFwdW1A): the recompute variant's forward keeps no h
//   plain bf16 store (kEpiStoreBf16): the routed experts' down projections
#include <stdlib.h>

#include "gemm_tc.cuh"

namespace mlpblk {

int launch_gemm_tc_fwd(int epi, int M, int N, int K, const void *A, const void *B, void *C0,
                       void *C1, const GemmArgs &extra, int num_sms, cudaStream_t s) {
    // Both operands are K-major here, so both pair widths are possible
    const int pairs = pair_tiles_enabled() ? (kAllowPair256 | kAllowPair192) : 0;
    // the in-kernel prologue needs whole tiles (all of K) per segment
    const int choice = choose_tile(M, N, K, epi != kEpiFwdW1 && streamk_enabled(), false, num_sms, pairs);
    const int mode = choice & ~kUseStreamK;
    GemmArgs args = extra;
    args.whole_tiles = (choice & kUseStreamK) ? 0 : 1;
#define MLPBLK_RUN_MODE(E, BNV, PAIRV) \
    return run_gemm_tc<GemmCfg<BNV, E, false, false, PAIRV>>(M, N, K, A, B, C0, C1, args, num_sms, s)
#define MLPBLK_RUN(E)                                         \
    switch (mode) {                                           \
        case kTilePair256: MLPBLK_RUN_MODE(E, 256, true);     \
        case kTilePair192: MLPBLK_RUN_MODE(E, 192, true);     \
        case kTile256: MLPBLK_RUN_MODE(E, 256, false);        \
        case kTile192: MLPBLK_RUN_MODE(E, 192, false);        \
        default: MLPBLK_RUN_MODE(E, 128, false);              \
    }
    if (epi == kEpiFwdW1) { MLPBLK_RUN(kEpiFwdW1) }
    if (epi == kEpiFwdW1Pre) { MLPBLK_RUN(kEpiFwdW1Pre) }
    if (epi == kEpiFwdW1A) { MLPBLK_RUN(kEpiFwdW1A) }
    if (epi == kEpiFwdW2) { MLPBLK_RUN(kEpiFwdW2) }
    if (epi == kEpiStoreBf16) { MLPBLK_RUN(kEpiStoreBf16) }
#undef MLPBLK_RUN
#undef MLPBLK_RUN_MODE
    return MLPBLK_EINVAL;
}

int take_device_error_gemm_fwd() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLPBLK_ECUDA;
    if (v != 0) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
    return v;
}

}  // namespace mlpblk
