// gemm_f8.cu -- the block's six GEMMs with E4M3 operands (tcgen05.mma
// kind::f8f6f4, fp32 accumulator in TMEM), for the FP8-operand variant.  Same
// kernel, schedule and fused epilogues as the bf16 GEMMs (gemm_fwd.cu,
// gemm_bwd.cu); the epilogue first multiplies the accumulator by the operands'
// dequantisation scales.  Operand layouts as in the bf16 path: forward both
// K-major; dgrad B MN-major; wgrad both MN-major.
#include "gemm_tc.cuh"

namespace mlpblk {

int launch_gemm_tc_f8(int epi, int M, int N, int K, const void *A, const void *B, void *C0, void *C1,
                      const GemmArgs &extra, int num_sms, cudaStream_t s) {
    const bool reduce = epi == kEpiAccF32 || epi == kEpiAccF32ColScale;
    const int pairs = pair_tiles_enabled() ? kAllowPair256 : 0;
    const int choice = choose_tile(M, N, K, streamk_enabled(), reduce, num_sms, pairs, 1);
    int mode = choice & ~kUseStreamK;
    if (mode == kTile192) mode = kTile256;  // 256 / 128 wide and 256 x 256 pairs only
    if (mode == kTilePair192) mode = kTilePair256;
    GemmArgs args = extra;
    args.whole_tiles = (choice & kUseStreamK) ? 0 : 1;
#define MLPBLK_RUN_MODE(E, AMN, BMN, BNV, PAIRV) \
    return run_gemm_tc<GemmCfg<BNV, E, AMN, BMN, PAIRV, true>>(M, N, K, A, B, C0, C1, args, num_sms, s)
#define MLPBLK_RUN(E, AMN, BMN)                                          \
    switch (mode) {                                                      \
        case kTilePair256: MLPBLK_RUN_MODE(E, AMN, BMN, 256, true);     \
        case kTile256: MLPBLK_RUN_MODE(E, AMN, BMN, 256, false);        \
        default: MLPBLK_RUN_MODE(E, AMN, BMN, 128, false);              \
    }
    switch (epi) {
        case kEpiFwdW1Pre: { MLPBLK_RUN(kEpiFwdW1Pre, false, false) }
        case kEpiFwdW2: { MLPBLK_RUN(kEpiFwdW2, false, false) }
        case kEpiDgradH: { MLPBLK_RUN(kEpiDgradH, false, true) }
        case kEpiAccF32: { MLPBLK_RUN(kEpiAccF32, true, true) }
        case kEpiStoreF32: { MLPBLK_RUN(kEpiStoreF32, false, true) }
        case kEpiAccF32ColScale: { MLPBLK_RUN(kEpiAccF32ColScale, true, true) }
        default: return MLPBLK_EINVAL;
    }
#undef MLPBLK_RUN
#undef MLPBLK_RUN_MODE
}

int take_device_error_gemm_f8() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLPBLK_ECUDA;
    if (v != 0) cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
    return v;
}

}  // namespace mlpblk
