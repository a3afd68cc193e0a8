// mlpblk_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mlpblk.h"

namespace mlpblk {

// A bounded device-side wait gives up after this long (two seconds).  Kernels of
// this library run for milliseconds, so only a broken pipeline gets here.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Host: the most recent failing CUDA runtime status seen by the library
// (reported by mlpblk_cuda_error_string).
extern int g_last_cuda_error;

// Host: MLPBLK_OK if `e` is cudaSuccess, else records it and returns MLPBLK_ECUDA.
inline int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MLPBLK_OK;
    g_last_cuda_error = static_cast<int>(e);
    return MLPBLK_ECUDA;
}

// Host: status of the kernel launch just made.
inline int launch_status() { return cuda_status(cudaGetLastError()); }

// Programmatic dependent launch.  Kernels of this library are launched so that
// the next kernel in the stream may start while this one finishes.  Every
// kernel calls griddep_wait() before its first global-memory access: it returns
// once the preceding kernel has completed and its writes are visible
// (immediately when there is none).
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream be scheduled (it still waits in
// griddep_wait for this kernel's completion before touching memory).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Both, at the top of a kernel that has no set-up worth overlapping.
__device__ __forceinline__ void griddep_enter() {
    griddep_launch_dependents();
    griddep_wait();
}

// Host: launches `kernel` on `s` with programmatic stream serialisation, so it
// may be scheduled while the previous kernel of the stream finishes (every
// kernel of the library waits for its predecessor before touching memory).
template <class... KArgs, class... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...));
}

// Each translation unit that runs kernels with bounded waits has its own device
// error word (internal linkage); mlpblk_last_error() collects all of them.
static __device__ int g_device_error;

// Epilogues of the tensor-core GEMM D[M,N] = sum_k A[m,k] B[n,k].
enum Epilogue : int {
    kEpiFwdW1 = 0,    // h = rstd*acc, a = relu(h)^2 (bf16 x2); rstd from A in-kernel
    kEpiFwdW2 = 1,    // y = x + acc (bf16); x read from global
    kEpiDgradH = 2,   // dh_s = rstd * acc * 2 relu(h) (bf16); h, rstd read from global
    kEpiStoreF32 = 3, // out = acc (fp32)
    kEpiAccF32 = 4,   // out += acc (fp32, TMA reduce-add)
    kEpiAccF32ColScale = 5,  // out += colscale[n] * acc (fp32, TMA reduce-add)
    kEpiFwdW1Pre = 6, // h = rstd*acc, a = relu(h)^2 (bf16 x2); rstd read from global
    kEpiFwdW1A = 7,   // a = relu(rstd*acc)^2 only (bf16); rstd read from global
    kEpiStoreBf16 = 8,  // out = acc (bf16): the routed experts' outputs
    kEpiAccF32ColScaleNorm = 9,  // kEpiAccF32ColScale, and side warps run the RMSNorm
                                 // backward rows (GemmArgs::side) meanwhile
};

// The RMSNorm backward rows that the wgrad-W1 GEMM's side warps compute while
// its tensor-core pipeline runs (bf16 block, d_model <= kSideNormMaxD): the row
// kernel's arithmetic on dn_s = rstd * dn, one warp per row, one dgamma partial
// row per CTA.
constexpr int kSideNormMaxD = 768;
constexpr int kSideWarps = 6;
struct SideNorm {
    const uint16_t *x, *dy, *gamma;  // bf16 [T, d], [T, d], [d]
    const uint16_t *dn_s;            // bf16 [T, d]: rstd * dn
    const float *rstd;               // fp32 [T]
    uint16_t *dx;                    // bf16 [T, d] (written)
    float *part;                     // fp32 [gridDim.x, d]: this launch's dgamma partial rows
    float *dgamma;                   // fp32 [d]: += the sum of the partial rows
    int *arrive;                     // CTAs whose partial row is complete (zero at launch)
    int64_t T;
    int d;
};

// Tile t of a GEMM rastered in groups of group_m M-tiles that sweep all N-tiles
// together: its M-tile and N-tile indices.
__host__ __device__ inline void raster_tile(int t, int m_tiles, int n_tiles, int group_m, int &mi, int &ni) {
    const int group = group_m * n_tiles;
    const int g = t / group;
    const int first_m = g * group_m;
    const int gm = (m_tiles - first_m) < group_m ? (m_tiles - first_m) : group_m;
    const int r = t - g * group;
    ni = r / gm;
    mi = first_m + r % gm;
}

// Arguments of one GEMM launch (the tensor maps travel separately).
// Stream-K partial accumulators: one slot of 128 x 256 fp32 per CTA, and per
// slot one flag word per epilogue warp.
constexpr int kMaxSkSlots = 160;
constexpr int kSkSlotFloats = 128 * 256;
constexpr int kMaxEpiWarps = 8;                    // epilogue warps of a GEMM CTA, at most
constexpr int kSkFlagsPerSet = kMaxSkSlots * kMaxEpiWarps;  // one flag per slot and epilogue warp

enum GroupMode : int { kGroupNone = 0, kGroupM = 1, kGroupK = 2 };

// How a GEMM orders itself against its neighbours in the stream (programmatic
// dependent launch).  A kernel's completion must imply its predecessor's, so a
// deferred GEMM waits before it exits, and it follows a kWaitFirst GEMM, whose
// successor is launched only once everything before that GEMM has completed.
enum PdlOrder : int {
    kPdlDefault = 0,    // launch the successor, then wait for the predecessor
    kPdlWaitFirst = 1,  // wait for the predecessor, clear zero_flags, then launch the successor
    kPdlDeferWait = 2,  // launch the successor and start at once: reads nothing the
                        // predecessor writes; waits for it just before exiting
};

struct GemmArgs {
    int M, N, K;
    int m_tiles, n_tiles, k_blocks;
    int tiles;                 // m_tiles * n_tiles
    int group_m;               // raster: this many M tiles sweep N together
    // Schedule over `workers` persistent workers (CTAs, or CTA pairs): tiles
    // [0, dp_tiles) are dealt whole, round robin; the sk_total k-block
    // iterations of tiles [dp_tiles, tiles) are cut into contiguous ranges of
    // sk_base (+1 for the first sk_rem workers) each ("stream-K").
    int workers, dp_tiles, sk_base, sk_rem, sk_total;
    // reduce (+=) GEMMs whose operands exceed L2: the tiles after dp_tiles are
    // cut into sub_parts ranges of sub_kb k-blocks, dealt round robin part by
    // part, so that the workers of a round stream the same k-range of tiles
    // that share operand panels (0: the stream-K ranges above)
    int sub_parts, sub_kb;
    float *sk_partial;         // kMaxSkSlots slots of kSkSlotFloats: split-tile partial sums
    int *sk_flags;             // kSkFlagsPerSet words, zero at launch: partial slot ready
    int *zero_flags;           // the next GEMM's flag set, zeroed by this launch (or null)
    int overwrite;             // reduce epilogues: C = (not +=) each tile one worker sums whole
                               // (K-grouped: every tile; otherwise tiles below dp_tiles);
                               // the split tiles at or beyond dp_tiles still add into C,
                               // which the caller has cleared there (zero_split_tiles)
    int whole_tiles;           // host-side: schedule whole tiles only (no stream-K)
    const float *deq_a, *deq_b;  // E4M3 operands: dequantisation scales (device scalars)
    float *amax_out;           // W1 (a) and dgrad-h (dh) epilogues: max |bf16 output| per
                               // epilogue warp, kMaxSkSlots * kMaxEpiWarps floats (unused 0)
    // grouped GEMMs of the routed experts (kGroupNone otherwise)
    int grp_mode, grp_count;   // kGroupM / kGroupK; number of experts
    const int *grp_rows;       // device [grp_count + 1]: padded segment starts (rows)
    int grp_b_off;             // M-grouped: per-expert offset into B (rows or K)
    int grp_c_off;             // K-grouped: per-expert rows of C
    int grp_split;             // M-grouped: split schedule computed in the kernel from
                               // the device row count (host-side: set by the launcher)
    const uint16_t *aux;       // bf16 [M, ld_aux]: x (FwdW2) or h (DgradH)
    int ld_aux;
    const float *rstd_in;      // DgradH: per-row rstd
    float *rstd_out;           // FwdW1: per-row rstd written by the n-tile-0 CTAs
    const uint16_t *colscale;  // AccF32ColScale: bf16 per-column scale (gamma)
    float inv_k;               // FwdW1: 1/d
    float eps;                 // FwdW1: RMSNorm epsilon
    int a_mn3d, b_mn3d;        // launcher-set: the MN-major operand's map is 3-D (one copy
                               // of all its boxes per k-block)
    int skip_loads;            // test fault: the producer issues no loads (waits run out)
    int pdl;                   // PdlOrder
    SideNorm side;             // kEpiAccF32ColScaleNorm: the side warps' rows
    int *grid_out;             // host-side: the launcher stores the grid size (CTAs) here
    GemmArgs *plan_out;        // host-side: when set, the launcher resolves the schedule,
                               // stores these arguments here and launches nothing
    int tile_m, tile_n;        // launcher-set: rows and columns of an output tile
};

// Operand / output views handed to the GEMM launcher (row-major 2-D tensors).
struct Mat {
    const void *ptr;
    int64_t rows, cols;  // logical shape of the stored array
};

// Host: launch one tensor-core GEMM.  A is [M,K] (K-major: stored [M][K]) or
// MN-major (stored [K][M]); B likewise with N.  Returns an MLPBLK_* code.
int launch_gemm_tc(int epi, bool a_mn, bool b_mn, int M, int N, int K,
                   const void *A, const void *B, void *C0, void *C1, const GemmArgs &extra,
                   int num_sms, cudaStream_t stream);
int take_device_error_gemm();

// Host: row/element kernels (rowops.cu).  All return MLPBLK_* codes.
int launch_fold_gamma(int dtype, const void *w1, const void *gamma, void *w1g, int64_t F,
                      int64_t d, int *zero_flags, int zero_count, cudaStream_t s);
int launch_rstd_f32(const float *x, float *rstd, int64_t T, int64_t d, float eps,
                    cudaStream_t s);
// Forward statistics pass: rstd[T] of x and W1g = W1 * gamma in one launch.
int launch_norm_prep(int dtype, const void *x, float *rstd, int64_t T, int64_t d, float eps,
                     const void *w1, const void *gamma, void *w1g, int64_t F, int *zero_flags,
                     int zero_count, cudaStream_t s);
// RMSNorm statistics inside the W1 GEMM (its prologue warps) when
// MLPBLK_RMS_IN_GEMM=1; by default the statistics pass computes rstd.
bool rms_in_gemm();
// RMSNorm backward rows; writes at most max_parts dgamma partial rows of d
// floats to dgamma_part and returns their count in *parts_out.  dn_s is float32,
// or bf16 when dn_bf16 is set (the bf16 block's dgrad-n GEMM stores it so).
int launch_rmsnorm_bwd(int dtype, const void *x, const void *dn_s, int dn_bf16, const void *dy,
                       const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                       int64_t T, int64_t d, int max_parts, int *parts_out, cudaStream_t s);
int take_device_error_rowops();
// Clears the output regions of the tiles that a dense reduce GEMM planned with
// `plan` splits between workers (tiles plan.dp_tiles .. plan.tiles - 1, which add
// into C when the GEMM overwrites), for up to two GEMMs (b may have tiles == 0),
// and dgamma[0, d).  C is fp32 [M][ldc].
struct SplitTiles {
    float *c;
    int64_t ldc;
    int M, N, tiles, dp_tiles, m_tiles, n_tiles, group_m, tile_m, tile_n;
};
SplitTiles split_tiles_of(const GemmArgs &plan, float *c, int64_t ldc);
int launch_zero_split_tiles(const SplitTiles &a, const SplitTiles &b, float *dgamma, int64_t d, cudaStream_t s);

// dgamma += (or =, overwrite != 0) the sum of the partial rows, in a fixed order.
int launch_dgamma_finalize(const float *part, int parts, float *dgamma, int64_t d,
                           cudaStream_t s, int overwrite = 0);
// Same row kernel, fed the plain gradient dn of the normalised output (the rstd
// scale is applied inside the kernel).
// Routed experts, bf16: row t's dn_s is the sum of the rows pos[t*k + j] of
// dn_rows (slot order; pos < 0 adds nothing).
int launch_rmsnorm_bwd_gather(const void *x, const void *dn_rows, int dn_bf16, const int *pos, int k,
                              const void *dy, const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                              int64_t T, int64_t d, int max_parts, int *parts_out, cudaStream_t s);
int launch_rmsnorm_bwd_unscaled(int dtype, const void *x, const float *dn, const void *dy,
                                const float *rstd, const void *gamma, void *dx, float *dgamma_part,
                                int64_t T, int64_t d, int max_parts, int *parts_out,
                                cudaStream_t s);
// zero_grads (zero = true) or scale_grads of three float32 buffers of n0, n1,
// n2 elements (multiples of 4, 16-byte aligned) in one launch.
int launch_grads(bool zero, float sc, float *p0, int64_t n0, float *p1, int64_t n1, float *p2,
                 int64_t n2, cudaStream_t s);

// Host: optimizer-side kernels (optim.cu).  Tensor sizes in elements, multiples
// of 4, 16-byte aligned.
struct AdamTensor {
    float *master;       // fp32 master weights (updated)
    void *weight;        // working copy in the block's element type (written), or null
    const float *grad;   // fp32 gradient
    float *m, *v;        // moments (updated)
    int64_t n;
    int decay;           // apply the weight decay to this tensor
};
int launch_grad_norm_partial(const float *g0, int64_t n0, const float *g1, int64_t n1, const float *g2,
                             int64_t n2, double *partial, int max_parts, int *parts_out, cudaStream_t s);
int launch_grad_norm_final(const double *partial, int parts, float max_norm, float *norm_out, float *scale_out,
                           cudaStream_t s);
int launch_clip_grads(float *g0, int64_t n0, float *g1, int64_t n1, float *g2, int64_t n2, const float *scale,
                      cudaStream_t s);
int launch_adamw(const AdamTensor *tensors, int count, float lr, float beta1, float beta2, float eps,
                 float weight_decay, int64_t step, bool bf16, const float *grad_scale, cudaStream_t s);

// Host: E4M3 quantisation (fp8.cu) and the E4M3 GEMMs (gemm_f8.cu).  A scale
// record is 4 floats {amax, 448 / amax, amax / 448, 0}.  n is a multiple of 8.
int launch_amax_e4m3(const void *v, const void *colmul, int64_t cols, int64_t n, float *partial, int max_parts,
                     int *parts_out, cudaStream_t s);
int launch_scale_e4m3(const float *partial, int parts, float *scale, int *zero_flags, int zero_count,
                      cudaStream_t s);
int launch_apply_e4m3(const void *v, const void *colmul, int64_t cols, int64_t n, const float *scale, uint8_t *q,
                      cudaStream_t s);
int launch_norm_quant(const void *x, float *rstd, uint8_t *n8, int64_t T, int64_t d, float eps, int *zero_flags,
                      int zero_count, cudaStream_t s);
int launch_gemm_tc_f8(int epi, int M, int N, int K, const void *A, const void *B, void *C0, void *C1,
                      const GemmArgs &extra, int num_sms, cudaStream_t s);
int take_device_error_gemm_f8();

// Host: dispatch / combine of the routed experts (moe.cu).  Rows are the
// experts' segments of (token, slot) assignments, each padded to 256 rows.
constexpr int kMoeRouteChunk = 1024;  // routing entries per CTA
inline int64_t moe_route_chunks(int64_t n) { return (n + kMoeRouteChunk - 1) / kMoeRouteChunk; }
// Routing in two launches: step 0 counts each chunk's entries per expert, step 1
// ranks and places them (the counts' prefix and the segment offsets computed per
// CTA).  chunk_count holds moe_route_chunks(n) * experts ints.
constexpr int kMoeRouteLaunches = 2;
int launch_moe_route(const int *idx, int64_t n, int k, int experts, int *chunk_count, int *count, int *seg,
                     int *pos, int *row_token, int *row_slot, int step, cudaStream_t s);
int launch_moe_gather(const void *x, const float *rstd, const int *row_token, const int *seg, int experts,
                      int64_t rows_max, int64_t d, void *x_perm, float *rstd_perm, cudaStream_t s);
int launch_moe_combine(const void *x, const void *o_perm, const float *p, const int *pos, int64_t T, int k,
                       int64_t d, void *y, cudaStream_t s);
// d_routing_weights and the slots' output gradients p * dy in segment order;
// with dw1s / dw2s non-null, also zero the [ffn, d] / [d, ffn] gradient blocks of
// every expert without tokens
int launch_moe_dout(const void *dy, const void *o_perm, const float *p, const int *pos, const int *count,
                    const int *seg, int64_t T, int k, int experts, int64_t d, float *dp, void *do_perm,
                    float *dw1s, float *dw2s, int64_t ffn, cudaStream_t s);

// Host: fp32 CUDA-core GEMM path (simt_f32.cu).  Strides are in elements:
// A(m,k) = A[m*sam + k*sak], B(n,k) = B[n*sbn + k*sbk], outputs row-major [M][N].
struct SimtEpi {
    const float *aux;       // FwdW2: x;  DgradH: h   (row-major [M][N])
    const float *rstd;      // FwdW1, DgradH
    const float *colscale;  // AccF32ColScale
};
int launch_gemm_simt(int epi, int M, int N, int K, const float *A, int64_t sam, int64_t sak,
                     const float *B, int64_t sbn, int64_t sbk, float *C0, float *C1,
                     const SimtEpi &e, cudaStream_t s);

constexpr int64_t kMaxNormD = 4096;  // RMSNorm backward keeps a row's dgamma share in registers

}  // namespace mlpblk
