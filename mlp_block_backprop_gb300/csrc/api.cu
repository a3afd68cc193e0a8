// api.cu -- the C ABI (include/mlpblk.h): argument checks, workspace layout and
// the order of kernels for one microbatch forward and backward.
//
// Forward  (bf16): fold gamma into W1 -> W1 GEMM (rstd prologue, h/a epilogue)
//                  -> W2 GEMM (residual epilogue)
// Backward (bf16): wgrad W2 GEMM (+=) -> dgrad-h GEMM (gate, dh_s = rstd*dh)
//                  -> dgrad-n GEMM (dn_s = rstd*dn, bf16) -> wgrad W1 GEMM (+= , gamma)
//                  -> RMSNorm backward rows (dx, dgamma partials) -> dgamma (+=)
//                  (d_model <= 768: the rows and the dgamma sum run on the
//                  wgrad-W1 GEMM's side warps)
// The fp32 element type runs the same sequence on CUDA cores.
#include <math.h>
#include <stdlib.h>

#include <new>

#include "mlpblk_internal.h"

namespace mlpblk {
int launch_gemm_tc_fwd(int epi, int M, int N, int K, const void *A, const void *B, void *C0,
                       void *C1, const GemmArgs &extra, int num_sms, cudaStream_t s);
int launch_gemm_tc_bwd(int epi, int M, int N, int K, const void *A, const void *B, void *C0,
                       void *C1, const GemmArgs &extra, int num_sms, cudaStream_t s);
int take_device_error_gemm_fwd();
int take_device_error_gemm_bwd();
}  // namespace mlpblk

namespace mlpblk {
int g_last_cuda_error = 0;
}  // namespace mlpblk

using namespace mlpblk;

namespace {

constexpr int kMaxParts = 512;  // dgamma partial rows the workspace holds

int64_t align256(int64_t b) { return (b + 255) & ~static_cast<int64_t>(255); }

int check_desc(const mlpblk_desc *d) {
    if (!d) return MLPBLK_EINVAL;
    if (d->dtype != MLPBLK_BF16 && d->dtype != MLPBLK_FP32) return MLPBLK_ENOTSUP;
    if (d->tokens < 0 || d->d_model <= 0 || d->ffn <= 0) return MLPBLK_EINVAL;
    if (d->d_model % 8 != 0 || d->ffn % 8 != 0) return MLPBLK_ENOTSUP;
    if (!(d->eps >= 0.0f) || !isfinite(d->eps)) return MLPBLK_EINVAL;
    const int64_t lim = static_cast<int64_t>(1) << 31;
    const int64_t wide = d->d_model > d->ffn ? d->d_model : d->ffn;
    if (d->ffn >= lim / d->d_model) return MLPBLK_EINVAL;
    if (d->tokens >= lim / wide) return MLPBLK_EINVAL;
    if (d->d_model > kMaxNormD) return MLPBLK_ENOTSUP;
    return MLPBLK_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct WsLayout {
    int64_t w1g, dh, h, a, dn, part, sk_partial, sk_flags, total;
};

// Stream-K flag sets, one per tensor-core GEMM that can split a tile; each set
// is zeroed by the kernel launched just before that GEMM.
// kSetSide: the wgrad-W1 side warps' arrival count (its first word).
enum SkFlagSet : int { kSetFwdW1 = 0, kSetFwdW2 = 1, kSetDgradH = 2, kSetDgradN = 3, kSetSide = 4, kSkSets = 5 };

// Workspace regions.  W1*gamma (forward, and the recompute backward's first
// GEMM) shares its region with dh_s (backward).  `recompute` adds the T x F
// h and a that the recompute variant keeps in the workspace instead of saving.
WsLayout ws_layout(const mlpblk_desc *d, bool recompute) {
    const int64_t elt = d->dtype == MLPBLK_BF16 ? 2 : 4;
    const int64_t tf = align256(d->tokens * d->ffn * elt);
    const int64_t fd = align256(d->ffn * d->d_model * elt);
    WsLayout l;
    l.w1g = 0;
    l.dh = 0;
    int64_t off = recompute ? (tf > fd ? tf : fd) : tf;
    l.h = recompute ? off : -1;
    if (recompute) off += tf;
    l.a = recompute ? off : -1;
    if (recompute) off += tf;
    l.dn = off;
    l.part = l.dn + align256(d->tokens * d->d_model * elt);  // dn_s in the block dtype
    const int64_t bwd = l.part + align256(static_cast<int64_t>(kMaxParts) * d->d_model * 4);
    // the GEMMs' stream-K partial sums and flags, apart from everything above
    l.sk_partial = fd > bwd ? fd : bwd;
    l.sk_flags = l.sk_partial + align256(static_cast<int64_t>(kMaxSkSlots) * kSkSlotFloats * 4);
    l.total = l.sk_flags + align256(static_cast<int64_t>(kSkSets) * kSkFlagsPerSet * 4);
    return l;
}

// Workspace of the FP8-operand variant (forward and backward regions overlap
// where they are never live together).
struct WsLayoutF8 {
    int64_t t16;   // a (forward) or dh (backward), bf16 [T, F]
    int64_t dh8;   // dh in E4M3 [T, F]
    int64_t w1q;   // W1*gamma (forward) or W1 (backward) in E4M3 [F, d]
    int64_t w2q;   // W2 in E4M3 [d, F]
    int64_t dyq;   // dy in E4M3 [T, d]
    int64_t dn;    // dn_s fp32 [T, d]
    int64_t part;  // dgamma partials [kMaxParts, d]
    int64_t amax;  // per-CTA maxima of the amax passes
    int64_t scales;  // scale records: 0 W1, 1 W2, 2 dy, 3 dh
    int64_t sk_partial, sk_flags, total;
};

constexpr int kAmaxParts = 2048;
static_assert(kAmaxParts >= kMaxSkSlots * kMaxEpiWarps, "the GEMM epilogues' maxima fit the amax scratch");

WsLayoutF8 ws_layout_f8(const mlpblk_desc *dsc) {
    const int64_t T = dsc->tokens, d = dsc->d_model, F = dsc->ffn;
    WsLayoutF8 l;
    int64_t off = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = off;
        off += align256(bytes);
        return at;
    };
    l.t16 = take(T * F * 2);
    l.dh8 = take(T * F);
    l.w1q = take(F * d);
    l.w2q = take(d * F);
    l.dyq = take(T * d);
    l.dn = take(T * d * 4);
    l.part = take(static_cast<int64_t>(kMaxParts) * d * 4);
    l.amax = take(kAmaxParts * 4);
    l.scales = take(4 * 16);
    l.sk_partial = take(static_cast<int64_t>(kMaxSkSlots) * kSkSlotFloats * 4);
    l.sk_flags = take(static_cast<int64_t>(kSkSets) * kSkFlagsPerSet * 4);
    l.total = off;
    return l;
}

// Device properties, checked once per device: sm_103 and its SM count.
int device_sms(int *sms) {
    static int cached[64] = {0};  // 0 unknown, -1 unsupported, else SM count
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != MLPBLK_OK || dev < 0 || dev >= 64) return MLPBLK_ECUDA;
    if (cached[dev] == 0) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MLPBLK_ECUDA;
        cached[dev] = (major == 10 && minor == 3 && n > 0) ? n : -1;
    }
    if (cached[dev] < 0) return MLPBLK_ENODEV;
    // MLPBLK_MAX_SMS caps the SMs the GEMMs spread over (an even count, to leave
    // SMs to concurrent work); unset, they use every SM
    static int cap = -1;
    if (cap < 0) {
        const char *e = getenv("MLPBLK_MAX_SMS");
        const int v = e ? atoi(e) : 0;
        cap = v >= 2 ? (v & ~1) : 0;
    }
    *sms = (cap > 0 && cap < cached[dev]) ? cap : cached[dev];
    return MLPBLK_OK;
}

#define MLPBLK_TRY(expr)              \
    do {                              \
        const int rc_ = (expr);       \
        if (rc_ != MLPBLK_OK) return rc_; \
    } while (0)

// Launch trace (mlpblk_trace_begin/end): caller-owned events around each launch.
struct Trace {
    cudaEvent_t *events = nullptr;
    int *kinds = nullptr;
    int capacity = 0;
    int count = 0;
    bool on = false;
} g_trace;

}  // namespace

namespace mlpblk {
// Where the forward's RMSNorm statistic is computed (mlpblk_set_rmsnorm_mode);
// the environment variable MLPBLK_RMS_IN_GEMM=1 sets the initial mode.
int g_rms_mode = -1;

bool rms_in_gemm() {
    if (g_rms_mode < 0) {
        const char *e = getenv("MLPBLK_RMS_IN_GEMM");
        g_rms_mode = (e && e[0] == '1') ? MLPBLK_RMSNORM_IN_W1_PROLOGUE : MLPBLK_RMSNORM_STATS_PASS;
    }
    return g_rms_mode == MLPBLK_RMSNORM_IN_W1_PROLOGUE;
}
}  // namespace mlpblk

namespace {

// The bf16 backward runs the RMSNorm backward rows on the wgrad-W1 GEMM's side
// warps when d_model <= kSideNormMaxD, unless MLPBLK_SIDE_NORM=0 selects the
// separate row kernel (both paths are parity-tested).
bool side_norm(int64_t d) {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("MLPBLK_SIDE_NORM");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1 && d <= kSideNormMaxD;
}

// One-shot test fault (mlpblk_set_test_fault): consumed by the next bf16 forward.
int g_test_fault = 0;

int take_test_fault() {
    const int f = g_test_fault;
    g_test_fault = 0;
    return f == MLPBLK_TEST_FAULT_SKIP_LOADS ? 1 : 0;
}

// Runs one launcher, bracketed by the trace events when a trace is active.
template <class F>
int traced(int kind, cudaStream_t s, F &&launch) {
    if (!g_trace.on) return launch();
    const int i = g_trace.count++;
    const bool rec = i < g_trace.capacity;
    // under stream capture the records become external event nodes, which keep
    // their timestamps when the graph is replayed
    unsigned int flags = cudaEventRecordDefault;
    if (rec) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        MLPBLK_TRY(cuda_status(cudaStreamIsCapturing(s, &cs)));
        if (cs == cudaStreamCaptureStatusActive) flags = cudaEventRecordExternal;
        g_trace.kinds[i] = kind;
        MLPBLK_TRY(cuda_status(cudaEventRecordWithFlags(g_trace.events[2 * i], s, flags)));
    }
    MLPBLK_TRY(launch());
    if (rec) MLPBLK_TRY(cuda_status(cudaEventRecordWithFlags(g_trace.events[2 * i + 1], s, flags)));
    return MLPBLK_OK;
}

#define MLPBLK_LAUNCH(kind, stream, call) MLPBLK_TRY(traced(kind, stream, [&]() { return (call); }))


}  // namespace

extern "C" {

int mlpblk_version(void) { return 100; }

const char *mlpblk_strerror(int code) {
    switch (code) {
        case MLPBLK_OK: return "success";
        case MLPBLK_EINVAL: return "invalid argument (null or misaligned pointer, bad size or eps)";
        case MLPBLK_ENOTSUP: return "unsupported dtype or shape (d_model, ffn multiples of 8; d_model <= 4096)";
        case MLPBLK_EWORKSPACE: return "workspace smaller than mlpblk_workspace_size()";
        case MLPBLK_ECUDA: return "CUDA runtime error or kernel launch failure";
        case MLPBLK_ETIMEOUT: return "a device-side bounded wait gave up; outputs are invalid";
        case MLPBLK_ENODEV: return "current device is not sm_103 (GB300)";
        default: return "unknown mlpblk status code";
    }
}

size_t mlpblk_workspace_size(const mlpblk_desc *desc) {
    if (check_desc(desc) != MLPBLK_OK) return 0;
    return static_cast<size_t>(ws_layout(desc, false).total);
}

}  // extern "C"

namespace {

// The forward's launches.  h_out may be null on the bf16 path (a_only: the
// recompute variant's forward, whose W1 epilogue writes a alone).
// prefolded: w1g already holds W1 * gamma (mlpblk_fold_weights); gamma and w1
// are not read.
int forward_impl(const mlpblk_desc *desc, const void *x, const void *gamma, const void *w1,
                 const void *w2, void *y, void *h_out, void *a_out, float *rstd_saved, void *w1g,
                 float *sk_partial, int *sk_flags, int sms, cudaStream_t s, bool a_only,
                 bool prefolded = false) {
    const int64_t T = desc->tokens, d = desc->d_model, F = desc->ffn;
    const bool stats_in_gemm = desc->dtype == MLPBLK_BF16 && !a_only && rms_in_gemm();
    if (stats_in_gemm) {
        // rstd inside the W1 GEMM (whole tiles: no stream-K flags to clear)
        if (!prefolded)
            MLPBLK_LAUNCH(MLPBLK_KERNEL_FOLD_GAMMA, s,
                          launch_fold_gamma(desc->dtype, w1, gamma, w1g, F, d, nullptr, 0, s));
    } else {
        // rstd, and W1 * gamma unless it is given
        MLPBLK_LAUNCH(prefolded ? MLPBLK_KERNEL_RSTD : MLPBLK_KERNEL_FOLD_GAMMA, s,
                      launch_norm_prep(desc->dtype, x, rstd_saved, T, d, desc->eps, prefolded ? nullptr : w1,
                                       gamma, prefolded ? nullptr : w1g, prefolded ? 0 : F,
                                       sk_flags + kSetFwdW1 * kSkFlagsPerSet, kSkFlagsPerSet, s));
    }
    if (desc->dtype == MLPBLK_BF16) {
        GemmArgs g1 = {};
        if (stats_in_gemm) {
            g1.rstd_out = rstd_saved;
            g1.inv_k = 1.0f / static_cast<float>(d);
            g1.eps = desc->eps;
        } else {
            g1.rstd_in = rstd_saved;
        }
        g1.skip_loads = take_test_fault();
        g1.sk_partial = sk_partial;
        g1.sk_flags = sk_flags + kSetFwdW1 * kSkFlagsPerSet;
        g1.zero_flags = sk_flags + kSetFwdW2 * kSkFlagsPerSet;
        const int epi1 = a_only ? kEpiFwdW1A : (stats_in_gemm ? kEpiFwdW1 : kEpiFwdW1Pre);
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W1, s,
                      launch_gemm_tc_fwd(epi1, (int)T, (int)F, (int)d, x, w1g, a_only ? a_out : h_out,
                                         a_only ? nullptr : a_out, g1, sms, s));
        GemmArgs g2 = {};
        g2.aux = static_cast<const uint16_t *>(x);
        g2.ld_aux = (int)d;
        g2.sk_partial = sk_partial;
        g2.sk_flags = sk_flags + kSetFwdW2 * kSkFlagsPerSet;
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W2, s, launch_gemm_tc_fwd(kEpiFwdW2, (int)T, (int)d, (int)F, a_out, w2, y, nullptr, g2, sms, s));
    } else {
        const float *xf = static_cast<const float *>(x);
        SimtEpi e1 = {nullptr, rstd_saved, nullptr};
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W1, s, launch_gemm_simt(kEpiFwdW1, (int)T, (int)F, (int)d, xf, d, 1,
                                    static_cast<const float *>(w1g), d, 1,
                                    static_cast<float *>(h_out), static_cast<float *>(a_out), e1, s));
        SimtEpi e2 = {xf, nullptr, nullptr};
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W2, s, launch_gemm_simt(kEpiFwdW2, (int)T, (int)d, (int)F,
                                    static_cast<const float *>(a_out), F, 1,
                                    static_cast<const float *>(w2), F, 1, static_cast<float *>(y),
                                    nullptr, e2, s));
    }
    return MLPBLK_OK;
}

// The backward's launches, from saved (or recomputed) h and a.
int backward_impl(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                  const void *w1, const void *w2, const void *h_saved, const void *a_saved,
                  const float *rstd_saved, void *dx, float *dgamma, float *dw1, float *dw2,
                  void *dh_s, void *dn_s, float *part, float *sk_partial, int *sk_flags, int sms,
                  cudaStream_t s, bool overwrite) {
    const int64_t T = desc->tokens, d = desc->d_model, F = desc->ffn;
    int parts = 0;  // dgamma partial rows written by the norm kernel
    if (desc->dtype == MLPBLK_BF16) {
        // dW2 first: it needs no flags and zeroes the dgrad-h GEMM's.  The two
        // independent pairs (dW2, dh) and (dn, dW1) overlap at their boundary:
        // the second of each starts on the SMs the first frees without waiting
        // for all of it (kPdlDeferWait), which the first allows by launching it
        // only after its own predecessor has completed (kPdlWaitFirst)
        GemmArgs gw2 = {};
        gw2.zero_flags = sk_flags + kSetDgradH * kSkFlagsPerSet;
        gw2.pdl = kPdlWaitFirst;
        GemmArgs gd = {};
        gd.aux = static_cast<const uint16_t *>(h_saved);
        gd.ld_aux = (int)F;
        gd.rstd_in = rstd_saved;
        gd.sk_partial = sk_partial;
        gd.sk_flags = sk_flags + kSetDgradH * kSkFlagsPerSet;
        gd.zero_flags = sk_flags + kSetDgradN * kSkFlagsPerSet;
        gd.pdl = kPdlDeferWait;
        GemmArgs gn = {};
        gn.sk_partial = sk_partial;
        gn.sk_flags = sk_flags + kSetDgradN * kSkFlagsPerSet;
        gn.zero_flags = side_norm(d) ? sk_flags + kSetSide * kSkFlagsPerSet : nullptr;
        gn.pdl = kPdlWaitFirst;
        GemmArgs gw1 = {};
        gw1.colscale = static_cast<const uint16_t *>(gamma);
        gw1.pdl = kPdlDeferWait;
        const bool side = side_norm(d);
        if (side) {
            // the RMSNorm backward rows run on the wgrad-W1 GEMM's side warps,
            // one dgamma partial row per CTA of that launch, summed into dgamma
            // by the same warps once every CTA's row is complete
            gw1.side.x = static_cast<const uint16_t *>(x);
            gw1.side.dy = static_cast<const uint16_t *>(dy);
            gw1.side.gamma = static_cast<const uint16_t *>(gamma);
            gw1.side.dn_s = static_cast<const uint16_t *>(dn_s);
            gw1.side.rstd = rstd_saved;
            gw1.side.dx = static_cast<uint16_t *>(dx);
            gw1.side.part = part;
            gw1.side.dgamma = dgamma;
            gw1.side.arrive = sk_flags + kSetSide * kSkFlagsPerSet;
            gw1.side.T = T;
            gw1.side.d = (int)d;
            gw1.grid_out = &parts;
        }
        const int epi_w1 = side ? kEpiAccF32ColScaleNorm : kEpiAccF32ColScale;
        if (overwrite) {
            // = instead of +=: the weight-gradient GEMMs store every tile one
            // worker sums whole, and add the split tiles' parts into regions
            // that one small launch clears first (with dgamma, which the norm
            // backward then adds into).  It runs before dW2's GEMM, whose
            // completion dW1's GEMM follows through the chain of waits above.
            gw2.overwrite = 1;
            gw1.overwrite = 1;
            GemmArgs plan2 = {}, plan1 = {};
            GemmArgs q2 = gw2, q1 = gw1;
            q2.plan_out = &plan2;
            q1.plan_out = &plan1;
            MLPBLK_TRY(launch_gemm_tc_bwd(kEpiAccF32, (int)d, (int)F, (int)T, dy, a_saved, dw2, nullptr, q2, sms, s));
            MLPBLK_TRY(launch_gemm_tc_bwd(epi_w1, (int)F, (int)d, (int)T, dh_s, x, dw1, nullptr, q1, sms, s));
            MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s,
                          launch_zero_split_tiles(split_tiles_of(plan2, dw2, F), split_tiles_of(plan1, dw1, d),
                                                  dgamma, d, s));
        }
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W2, s, launch_gemm_tc_bwd(kEpiAccF32, (int)d, (int)F, (int)T, dy, a_saved, dw2, nullptr, gw2, sms, s));
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_H, s, launch_gemm_tc_bwd(kEpiDgradH, (int)T, (int)F, (int)d, dy, w2, dh_s, nullptr, gd, sms, s));
        // dn_s = rstd * dn stored in bf16 like dh_s (rstd rides in dh_s already)
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_N, s, launch_gemm_tc_bwd(kEpiStoreBf16, (int)T, (int)d, (int)F, dh_s, w1, dn_s, nullptr, gn, sms, s));
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W1, s, launch_gemm_tc_bwd(epi_w1, (int)F, (int)d, (int)T, dh_s, x, dw1, nullptr, gw1, sms, s));
        if (side) {
            if (parts <= 0 || parts > kMaxParts) return MLPBLK_ECUDA;
            return MLPBLK_OK;
        }
    } else {
        // CUDA-core path, = instead of +=: the gradients are cleared, then added into
        if (overwrite)
            MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s,
                          launch_grads(true, 0.0f, dgamma, d, dw1, F * d, dw2, d * F, s));
        const float *dyf = static_cast<const float *>(dy);
        const float *xf = static_cast<const float *>(x);
        const float *dhf = static_cast<const float *>(dh_s);
        SimtEpi ed = {static_cast<const float *>(h_saved), rstd_saved, nullptr};
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_H, s, launch_gemm_simt(kEpiDgradH, (int)T, (int)F, (int)d, dyf, d, 1,
                                    static_cast<const float *>(w2), 1, F, static_cast<float *>(dh_s),
                                    nullptr, ed, s));
        SimtEpi e0 = {nullptr, nullptr, nullptr};
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W2, s, launch_gemm_simt(kEpiAccF32, (int)d, (int)F, (int)T, dyf, 1, d,
                                    static_cast<const float *>(a_saved), 1, F, dw2, nullptr, e0, s));
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_N, s, launch_gemm_simt(kEpiStoreF32, (int)T, (int)d, (int)F, dhf, F, 1,
                                    static_cast<const float *>(w1), 1, d, static_cast<float *>(dn_s), nullptr, e0, s));
        SimtEpi ec = {nullptr, nullptr, static_cast<const float *>(gamma)};
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W1, s, launch_gemm_simt(kEpiAccF32ColScale, (int)F, (int)d, (int)T, dhf, 1, F, xf, 1, d,
                                    dw1, nullptr, ec, s));
    }
    MLPBLK_LAUNCH(MLPBLK_KERNEL_NORM_BWD, s, launch_rmsnorm_bwd(desc->dtype, x, dn_s, desc->dtype == MLPBLK_BF16, dy, rstd_saved, gamma, dx, part, T, d, kMaxParts, &parts, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_DGAMMA_REDUCE, s, launch_dgamma_finalize(part, parts, dgamma, d, s));
    return MLPBLK_OK;
}

}  // namespace

extern "C" {

int mlpblk_forward(const mlpblk_desc *desc, const void *x, const void *gamma, const void *w1,
                   const void *w2, void *y, void *h_saved, void *a_saved, float *rstd_saved,
                   void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (desc->tokens == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(w1) || !aligned16(w2) || !aligned16(y) ||
        !aligned16(h_saved) || !aligned16(a_saved) || !aligned16(rstd_saved) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (y == x) return MLPBLK_EINVAL;
    const WsLayout l = ws_layout(desc, false);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    return forward_impl(desc, x, gamma, w1, w2, y, h_saved, a_saved, rstd_saved, ws + l.w1g,
                        reinterpret_cast<float *>(ws + l.sk_partial), reinterpret_cast<int *>(ws + l.sk_flags),
                        sms, static_cast<cudaStream_t>(stream), false);
}

}  // extern "C"

namespace {

int backward_entry(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                   const void *w1, const void *w2, const void *h_saved, const void *a_saved,
                   const float *rstd_saved, void *dx, float *dgamma, float *dw1, float *dw2,
                   void *workspace, size_t workspace_bytes, void *stream, bool overwrite) {
    MLPBLK_TRY(check_desc(desc));
    if (desc->tokens == 0) {
        // no rows: += adds nothing; = leaves zero gradients
        if (!overwrite) return MLPBLK_OK;
        if (!aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2)) return MLPBLK_EINVAL;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const int64_t d = desc->d_model, F = desc->ffn;
        MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s, launch_grads(true, 0.0f, dgamma, d, dw1, F * d, dw2, d * F, s));
        return MLPBLK_OK;
    }
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(w1) || !aligned16(w2) ||
        !aligned16(h_saved) || !aligned16(a_saved) || !aligned16(rstd_saved) || !aligned16(dx) ||
        !aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (dx == dy || dx == x) return MLPBLK_EINVAL;
    const WsLayout l = ws_layout(desc, false);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    return backward_impl(desc, dy, x, gamma, w1, w2, h_saved, a_saved, rstd_saved, dx, dgamma, dw1, dw2,
                         ws + l.dh, ws + l.dn, reinterpret_cast<float *>(ws + l.part),
                         reinterpret_cast<float *>(ws + l.sk_partial), reinterpret_cast<int *>(ws + l.sk_flags),
                         sms, static_cast<cudaStream_t>(stream), overwrite);
}

}  // namespace

extern "C" {

int mlpblk_backward(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                    const void *w1, const void *w2, const void *h_saved, const void *a_saved,
                    const float *rstd_saved, void *dx, float *dgamma, float *dw1, float *dw2,
                    void *workspace, size_t workspace_bytes, void *stream) {
    return backward_entry(desc, dy, x, gamma, w1, w2, h_saved, a_saved, rstd_saved, dx, dgamma, dw1, dw2,
                          workspace, workspace_bytes, stream, false);
}

int mlpblk_backward_overwrite(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                              const void *w1, const void *w2, const void *h_saved, const void *a_saved,
                              const float *rstd_saved, void *dx, float *dgamma, float *dw1, float *dw2,
                              void *workspace, size_t workspace_bytes, void *stream) {
    return backward_entry(desc, dy, x, gamma, w1, w2, h_saved, a_saved, rstd_saved, dx, dgamma, dw1, dw2,
                          workspace, workspace_bytes, stream, true);
}

int mlpblk_fold_weights(const mlpblk_desc *desc, const void *gamma, const void *w1, void *w1g,
                        void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (!aligned16(gamma) || !aligned16(w1) || !aligned16(w1g)) return MLPBLK_EINVAL;
    if (w1g == w1) return MLPBLK_EINVAL;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MLPBLK_LAUNCH(MLPBLK_KERNEL_FOLD_GAMMA, s,
                  launch_fold_gamma(desc->dtype, w1, gamma, w1g, desc->ffn, desc->d_model, nullptr, 0, s));
    return MLPBLK_OK;
}

int mlpblk_forward_prefolded(const mlpblk_desc *desc, const void *x, const void *w1g, const void *w2,
                             void *y, void *h_saved, void *a_saved, float *rstd_saved, void *workspace,
                             size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (desc->tokens == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(w1g) || !aligned16(w2) || !aligned16(y) || !aligned16(h_saved) ||
        !aligned16(a_saved) || !aligned16(rstd_saved) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (y == x) return MLPBLK_EINVAL;
    const WsLayout l = ws_layout(desc, false);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    return forward_impl(desc, x, nullptr, nullptr, w2, y, h_saved, a_saved, rstd_saved, const_cast<void *>(w1g),
                        reinterpret_cast<float *>(ws + l.sk_partial), reinterpret_cast<int *>(ws + l.sk_flags),
                        sms, static_cast<cudaStream_t>(stream), false, true);
}

size_t mlpblk_workspace_size_recompute(const mlpblk_desc *desc) {
    if (check_desc(desc) != MLPBLK_OK) return 0;
    return static_cast<size_t>(ws_layout(desc, true).total);
}

int mlpblk_forward_recompute(const mlpblk_desc *desc, const void *x, const void *gamma,
                             const void *w1, const void *w2, void *y, float *rstd_saved,
                             void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (desc->tokens == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(w1) || !aligned16(w2) || !aligned16(y) ||
        !aligned16(rstd_saved) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (y == x) return MLPBLK_EINVAL;
    const WsLayout l = ws_layout(desc, true);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    // bf16: the W1 epilogue writes a alone; fp32: h goes to scratch
    const bool bf16 = desc->dtype == MLPBLK_BF16;
    return forward_impl(desc, x, gamma, w1, w2, y, bf16 ? nullptr : ws + l.h, ws + l.a, rstd_saved,
                        ws + l.w1g, reinterpret_cast<float *>(ws + l.sk_partial),
                        reinterpret_cast<int *>(ws + l.sk_flags), sms, static_cast<cudaStream_t>(stream), bf16);
}

int mlpblk_backward_recompute(const mlpblk_desc *desc, const void *dy, const void *x,
                              const void *gamma, const void *w1, const void *w2,
                              const float *rstd_saved, void *dx, float *dgamma, float *dw1,
                              float *dw2, void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (desc->tokens == 0) return MLPBLK_OK;
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(w1) || !aligned16(w2) ||
        !aligned16(rstd_saved) || !aligned16(dx) || !aligned16(dgamma) || !aligned16(dw1) ||
        !aligned16(dw2) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (dx == dy || dx == x) return MLPBLK_EINVAL;
    const WsLayout l = ws_layout(desc, true);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = desc->tokens, d = desc->d_model, F = desc->ffn;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *w1g = ws + l.w1g;
    void *h = ws + l.h;
    void *a = ws + l.a;
    float *sk_partial = reinterpret_cast<float *>(ws + l.sk_partial);
    int *sk_flags = reinterpret_cast<int *>(ws + l.sk_flags);
    // h and a again, from x and the saved rstd: the forward's W1 GEMM (same
    // configuration and schedule, so the same bits)
    MLPBLK_LAUNCH(MLPBLK_KERNEL_FOLD_GAMMA, s,
                  launch_fold_gamma(desc->dtype, w1, gamma, w1g, F, d, sk_flags + kSetFwdW1 * kSkFlagsPerSet,
                                    kSkFlagsPerSet, s));
    if (desc->dtype == MLPBLK_BF16) {
        GemmArgs g1 = {};
        g1.rstd_in = rstd_saved;
        g1.sk_partial = sk_partial;
        g1.sk_flags = sk_flags + kSetFwdW1 * kSkFlagsPerSet;
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W1, s,
                      launch_gemm_tc_fwd(kEpiFwdW1Pre, (int)T, (int)F, (int)d, x, w1g, h, a, g1, sms, s));
    } else {
        SimtEpi e1 = {nullptr, rstd_saved, nullptr};
        MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W1, s,
                      launch_gemm_simt(kEpiFwdW1, (int)T, (int)F, (int)d, static_cast<const float *>(x), d, 1,
                                       static_cast<const float *>(w1g), d, 1, static_cast<float *>(h),
                                       static_cast<float *>(a), e1, s));
    }
    // dh_s takes the W1*gamma region, which the GEMM above was the last to read
    return backward_impl(desc, dy, x, gamma, w1, w2, h, a, rstd_saved, dx, dgamma, dw1, dw2, ws + l.dh,
                         ws + l.dn, reinterpret_cast<float *>(ws + l.part),
                         sk_partial, sk_flags, sms, s, false);
}

int mlpblk_grad_norm(const mlpblk_desc *desc, const float *dgamma, const float *dw1, const float *dw2,
                     float max_norm, float *norm_out, float *clip_scale_out, void *workspace,
                     size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (!aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (!norm_out && !clip_scale_out) return MLPBLK_EINVAL;
    if ((norm_out && (reinterpret_cast<uintptr_t>(norm_out) & 3u)) ||
        (clip_scale_out && (reinterpret_cast<uintptr_t>(clip_scale_out) & 3u)))
        return MLPBLK_EINVAL;
    if (!(max_norm > 0.0f) || !isfinite(max_norm)) return MLPBLK_EINVAL;
    const WsLayout l = ws_layout(desc, false);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    const int64_t d = desc->d_model, F = desc->ffn;
    const int64_t part_bytes = static_cast<int64_t>(kMaxParts) * d * 4;
    const int max_parts = static_cast<int>(part_bytes / 8 < 1024 ? part_bytes / 8 : 1024);
    double *partial = reinterpret_cast<double *>(static_cast<uint8_t *>(workspace) + l.part);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int parts = 0;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GRAD_NORM, s,
                  launch_grad_norm_partial(dgamma, d, dw1, F * d, dw2, F * d, partial, max_parts, &parts, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GRAD_NORM_FINAL, s,
                  launch_grad_norm_final(partial, parts, max_norm, norm_out, clip_scale_out, s));
    return MLPBLK_OK;
}

int mlpblk_clip_grads(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2, const float *clip_scale,
                      void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (!aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2)) return MLPBLK_EINVAL;
    if (!clip_scale || (reinterpret_cast<uintptr_t>(clip_scale) & 3u)) return MLPBLK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_CLIP_GRADS, s, launch_clip_grads(dgamma, d, dw1, F * d, dw2, F * d, clip_scale, s));
    return MLPBLK_OK;
}

int mlpblk_adamw_step(const mlpblk_param *params, int count, const mlpblk_adamw *hp, int64_t step, int dtype,
                      const float *grad_scale, void *stream) {
    if (!params || count < 1 || count > 1024 || !hp || step < 1) return MLPBLK_EINVAL;
    if (dtype != MLPBLK_BF16 && dtype != MLPBLK_FP32) return MLPBLK_ENOTSUP;
    const float vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (float v : vals)
        if (!isfinite(v) || v < 0.0f) return MLPBLK_EINVAL;
    if (!(hp->beta1 < 1.0f) || !(hp->beta2 < 1.0f)) return MLPBLK_EINVAL;
    if (grad_scale && (reinterpret_cast<uintptr_t>(grad_scale) & 3u)) return MLPBLK_EINVAL;
    const uintptr_t walign = dtype == MLPBLK_BF16 ? 7u : 15u;
    AdamTensor t[1024];
    for (int i = 0; i < count; ++i) {
        const mlpblk_param &p = params[i];
        if (!aligned16(p.master) || !aligned16(p.grad) || !aligned16(p.m) || !aligned16(p.v)) return MLPBLK_EINVAL;
        if (p.weight && (reinterpret_cast<uintptr_t>(p.weight) & walign)) return MLPBLK_EINVAL;
        if (p.n <= 0 || p.n % 4 != 0) return MLPBLK_EINVAL;
        t[i] = AdamTensor{p.master, p.weight, p.grad, p.m, p.v, p.n, p.decay != 0};
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MLPBLK_LAUNCH(MLPBLK_KERNEL_ADAMW, s,
                  launch_adamw(t, count, hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, step,
                               dtype == MLPBLK_BF16, grad_scale, s));
    return MLPBLK_OK;
}

static int check_fp8_desc(const mlpblk_desc *desc) {
    MLPBLK_TRY(check_desc(desc));
    if (desc->dtype != MLPBLK_BF16) return MLPBLK_ENOTSUP;
    if (desc->d_model % 16 != 0 || desc->ffn % 16 != 0) return MLPBLK_ENOTSUP;  // 16-byte E4M3 rows
    return MLPBLK_OK;
}

size_t mlpblk_workspace_size_fp8(const mlpblk_desc *desc) {
    if (check_fp8_desc(desc) != MLPBLK_OK) return 0;
    return static_cast<size_t>(ws_layout_f8(desc).total);
}

}  // extern "C"

namespace {

// E4M3 codes of the weights, each with its scale record {amax, 448/amax, amax/448, 0}.
struct F8Weights {
    const uint8_t *w1g, *w2, *w1;  // W1*gamma [F,d], W2 [d,F], W1 [F,d]
    const float *s_w1g, *s_w2, *s_w1;
};

// A caller-owned pre-quantised weight buffer: the three code tensors, then the
// three scale records.
struct WqLayout {
    int64_t w1g, w2, w1, scales, total;
};

WqLayout wq_layout(const mlpblk_desc *d) {
    WqLayout l;
    const int64_t fd = align256(d->ffn * d->d_model);
    l.w1g = 0;
    l.w2 = fd;
    l.w1 = 2 * fd;
    l.scales = 3 * fd;
    l.total = 3 * fd + 256;
    return l;
}

// amax pass, scale record, codes of one tensor (colmul: per-column bf16 factor)
int quantize_tensor(const void *v, const void *colmul, int64_t cols, int64_t n, float *amax, float *rec,
                    uint8_t *codes, cudaStream_t s) {
    int parts = 0;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_AMAX, s, launch_amax_e4m3(v, colmul, cols, n, amax, kAmaxParts, &parts, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_SCALE, s, launch_scale_e4m3(amax, parts, rec, nullptr, 0, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_APPLY, s, launch_apply_e4m3(v, colmul, cols, n, rec, codes, s));
    return MLPBLK_OK;
}

int forward_fp8_impl(const mlpblk_desc *desc, const void *x, const F8Weights &w, void *y, void *h_saved,
                     void *a8_saved, void *n8_saved, float *rstd_saved, float *scales_saved, uint8_t *ws,
                     const WsLayoutF8 &l, int sms, cudaStream_t s) {
    const int64_t T = desc->tokens, d = desc->d_model, F = desc->ffn;
    float *amax = reinterpret_cast<float *>(ws + l.amax);
    float *sk_partial = reinterpret_cast<float *>(ws + l.sk_partial);
    int *sk_flags = reinterpret_cast<int *>(ws + l.sk_flags);
    void *a16 = ws + l.t16;
    // n' = x * rstd in E4M3 (scale 1) and rstd; clears the W1 GEMM's flags
    MLPBLK_LAUNCH(MLPBLK_KERNEL_NORM_QUANT, s,
                  launch_norm_quant(x, rstd_saved, static_cast<uint8_t *>(n8_saved), T, d, desc->eps,
                                    sk_flags + kSetFwdW1 * kSkFlagsPerSet, kSkFlagsPerSet, s));
    // h (saved, bf16) and a (bf16, scratch) = relu(h)^2, h = (n' . (W1*gamma)^T) * s_w1g
    // (the epilogue also leaves max |a| per epilogue warp in amax)
    GemmArgs g1 = {};
    g1.deq_b = w.s_w1g + 2;
    g1.sk_partial = sk_partial;
    g1.sk_flags = sk_flags + kSetFwdW1 * kSkFlagsPerSet;
    g1.amax_out = amax;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W1, s,
                  launch_gemm_tc_f8(kEpiFwdW1Pre, (int)T, (int)F, (int)d, n8_saved, w.w1g, h_saved, a16, g1, sms, s));
    // a in E4M3 (saved with its scale record; clears the W2 GEMM's flags)
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_SCALE, s,
                  launch_scale_e4m3(amax, kMaxSkSlots * kMaxEpiWarps, scales_saved, sk_flags + kSetFwdW2 * kSkFlagsPerSet,
                                    kSkFlagsPerSet, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_APPLY, s,
                  launch_apply_e4m3(a16, nullptr, F, T * F, scales_saved, static_cast<uint8_t *>(a8_saved), s));
    // y = x + (a . W2^T) * s_a * s_w2
    GemmArgs g2 = {};
    g2.aux = static_cast<const uint16_t *>(x);
    g2.ld_aux = (int)d;
    g2.deq_a = scales_saved + 2;
    g2.deq_b = w.s_w2 + 2;
    g2.sk_partial = sk_partial;
    g2.sk_flags = sk_flags + kSetFwdW2 * kSkFlagsPerSet;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W2, s,
                  launch_gemm_tc_f8(kEpiFwdW2, (int)T, (int)d, (int)F, a8_saved, w.w2, y, nullptr, g2, sms, s));
    return MLPBLK_OK;
}

int backward_fp8_impl(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma, const F8Weights &w,
                      const void *h_saved, const void *a8_saved, const void *n8_saved, const float *rstd_saved,
                      const float *scales_saved, void *dx, float *dgamma, float *dw1, float *dw2, uint8_t *ws,
                      const WsLayoutF8 &l, int sms, cudaStream_t s, bool overwrite) {
    const int64_t T = desc->tokens, d = desc->d_model, F = desc->ffn;
    float *amax = reinterpret_cast<float *>(ws + l.amax);
    float *sc = reinterpret_cast<float *>(ws + l.scales);  // records: 2 dy, 3 dh
    float *sk_partial = reinterpret_cast<float *>(ws + l.sk_partial);
    int *sk_flags = reinterpret_cast<int *>(ws + l.sk_flags);
    uint8_t *dyq = ws + l.dyq, *dh8 = ws + l.dh8;
    void *dh16 = ws + l.t16;
    float *dn_s = reinterpret_cast<float *>(ws + l.dn);
    float *part = reinterpret_cast<float *>(ws + l.part);
    int parts = 0;
    // dW2 += (dy^T . a) * s_dy * s_a; clears the dgrad-h GEMM's flags
    GemmArgs gw2 = {};
    gw2.deq_a = sc + 8 + 2;
    gw2.deq_b = scales_saved + 2;
    gw2.zero_flags = sk_flags + kSetDgradH * kSkFlagsPerSet;
    gw2.pdl = kPdlWaitFirst;  // (dW2, dh) and (dn, dW1) overlap as in the bf16 backward
    // dW1 += gamma[col] * (dh^T . n') * s_dh
    GemmArgs gw1 = {};
    gw1.colscale = static_cast<const uint16_t *>(gamma);
    gw1.deq_a = sc + 12 + 2;
    gw1.pdl = kPdlDeferWait;
    if (overwrite) {
        // = instead of +=, as in the bf16 backward: whole tiles stored, the split
        // tiles' regions (and dgamma) cleared by the call's first launch
        gw2.overwrite = 1;
        gw1.overwrite = 1;
        GemmArgs plan2 = {}, plan1 = {};
        GemmArgs q2 = gw2, q1 = gw1;
        q2.plan_out = &plan2;
        q1.plan_out = &plan1;
        MLPBLK_TRY(launch_gemm_tc_f8(kEpiAccF32, (int)d, (int)F, (int)T, dyq, a8_saved, dw2, nullptr, q2, sms, s));
        MLPBLK_TRY(launch_gemm_tc_f8(kEpiAccF32ColScale, (int)F, (int)d, (int)T, dh8, n8_saved, dw1, nullptr, q1,
                                     sms, s));
        MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s,
                      launch_zero_split_tiles(split_tiles_of(plan2, dw2, F), split_tiles_of(plan1, dw1, d), dgamma,
                                              d, s));
    }
    MLPBLK_TRY(quantize_tensor(dy, nullptr, d, T * d, amax, sc + 8, dyq, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W2, s,
                  launch_gemm_tc_f8(kEpiAccF32, (int)d, (int)F, (int)T, dyq, a8_saved, dw2, nullptr, gw2, sms, s));
    // dh = (dy . W2) * s_dy * s_w2 * 2 relu(h)   (bf16; the row scale goes to dgrad-n)
    // (the epilogue also leaves max |dh| per epilogue warp in amax)
    GemmArgs gd = {};
    gd.aux = static_cast<const uint16_t *>(h_saved);
    gd.ld_aux = (int)F;
    gd.deq_a = sc + 8 + 2;
    gd.deq_b = w.s_w2 + 2;
    gd.sk_partial = sk_partial;
    gd.sk_flags = sk_flags + kSetDgradH * kSkFlagsPerSet;
    gd.amax_out = amax;
    gd.pdl = kPdlDeferWait;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_H, s,
                  launch_gemm_tc_f8(kEpiDgradH, (int)T, (int)F, (int)d, dyq, w.w2, dh16, nullptr, gd, sms, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_SCALE, s,
                  launch_scale_e4m3(amax, kMaxSkSlots * kMaxEpiWarps, sc + 12, sk_flags + kSetDgradN * kSkFlagsPerSet,
                                    kSkFlagsPerSet, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_QUANT_APPLY, s, launch_apply_e4m3(dh16, nullptr, F, T * F, sc + 12, dh8, s));
    // dn_s = rstd * (dh . W1) * s_dh * s_w1   (fp32)
    GemmArgs gn = {};
    gn.rstd_in = rstd_saved;
    gn.deq_a = sc + 12 + 2;
    gn.deq_b = w.s_w1 + 2;
    gn.sk_partial = sk_partial;
    gn.sk_flags = sk_flags + kSetDgradN * kSkFlagsPerSet;
    gn.pdl = kPdlWaitFirst;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_N, s,
                  launch_gemm_tc_f8(kEpiStoreF32, (int)T, (int)d, (int)F, dh8, w.w1, dn_s, nullptr, gn, sms, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W1, s,
                  launch_gemm_tc_f8(kEpiAccF32ColScale, (int)F, (int)d, (int)T, dh8, n8_saved, dw1, nullptr, gw1,
                                    sms, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_NORM_BWD, s, launch_rmsnorm_bwd(desc->dtype, x, dn_s, 0, dy, rstd_saved, gamma, dx, part, T, d, kMaxParts, &parts, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_DGAMMA_REDUCE, s, launch_dgamma_finalize(part, parts, dgamma, d, s));
    return MLPBLK_OK;
}

}  // namespace

extern "C" {

int mlpblk_forward_fp8(const mlpblk_desc *desc, const void *x, const void *gamma, const void *w1, const void *w2,
                       void *y, void *h_saved, void *a8_saved, void *n8_saved, float *rstd_saved,
                       float *scales_saved, void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_fp8_desc(desc));
    if (desc->tokens == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(w1) || !aligned16(w2) || !aligned16(y) ||
        !aligned16(h_saved) || !aligned16(a8_saved) || !aligned16(n8_saved) || !aligned16(rstd_saved) ||
        !aligned16(scales_saved) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (y == x) return MLPBLK_EINVAL;
    const WsLayoutF8 l = ws_layout_f8(desc);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *amax = reinterpret_cast<float *>(ws + l.amax);
    float *sc = reinterpret_cast<float *>(ws + l.scales);  // records: 0 W1*gamma, 1 W2
    uint8_t *w1q = ws + l.w1q, *w2q = ws + l.w2q;
    // W1 * gamma and W2 in E4M3, into the workspace
    MLPBLK_TRY(quantize_tensor(w1, gamma, d, F * d, amax, sc + 0, w1q, s));
    MLPBLK_TRY(quantize_tensor(w2, nullptr, F, d * F, amax, sc + 4, w2q, s));
    const F8Weights w = {w1q, w2q, nullptr, sc + 0, sc + 4, nullptr};
    return forward_fp8_impl(desc, x, w, y, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved, ws, l, sms, s);
}

}  // extern "C"

namespace {

// T = 0: += adds nothing; = leaves zero gradients.
int empty_backward(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2, void *stream, bool overwrite) {
    if (!overwrite) return MLPBLK_OK;
    if (!aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2)) return MLPBLK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s, launch_grads(true, 0.0f, dgamma, d, dw1, F * d, dw2, d * F, s));
    return MLPBLK_OK;
}

int backward_fp8_entry(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma, const void *w1,
                       const void *w2, const void *h_saved, const void *a8_saved, const void *n8_saved,
                       const float *rstd_saved, const float *scales_saved, void *dx, float *dgamma, float *dw1,
                       float *dw2, void *workspace, size_t workspace_bytes, void *stream, bool overwrite) {
    MLPBLK_TRY(check_fp8_desc(desc));
    if (desc->tokens == 0) return empty_backward(desc, dgamma, dw1, dw2, stream, overwrite);
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(w1) || !aligned16(w2) ||
        !aligned16(h_saved) || !aligned16(a8_saved) || !aligned16(n8_saved) || !aligned16(rstd_saved) ||
        !aligned16(scales_saved) || !aligned16(dx) || !aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2) ||
        !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (dx == dy || dx == x) return MLPBLK_EINVAL;
    const WsLayoutF8 l = ws_layout_f8(desc);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *amax = reinterpret_cast<float *>(ws + l.amax);
    float *sc = reinterpret_cast<float *>(ws + l.scales);  // records: 0 W1, 1 W2
    uint8_t *w1q = ws + l.w1q, *w2q = ws + l.w2q;
    MLPBLK_TRY(quantize_tensor(w2, nullptr, F, d * F, amax, sc + 4, w2q, s));
    MLPBLK_TRY(quantize_tensor(w1, nullptr, d, F * d, amax, sc + 0, w1q, s));
    const F8Weights w = {nullptr, w2q, w1q, nullptr, sc + 4, sc + 0};
    return backward_fp8_impl(desc, dy, x, gamma, w, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved, dx,
                             dgamma, dw1, dw2, ws, l, sms, s, overwrite);
}

int backward_fp8_prequant_entry(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                                const void *wq, const void *h_saved, const void *a8_saved, const void *n8_saved,
                                const float *rstd_saved, const float *scales_saved, void *dx, float *dgamma,
                                float *dw1, float *dw2, void *workspace, size_t workspace_bytes, void *stream,
                                bool overwrite) {
    MLPBLK_TRY(check_fp8_desc(desc));
    if (desc->tokens == 0) return empty_backward(desc, dgamma, dw1, dw2, stream, overwrite);
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(wq) || !aligned16(h_saved) ||
        !aligned16(a8_saved) || !aligned16(n8_saved) || !aligned16(rstd_saved) || !aligned16(scales_saved) ||
        !aligned16(dx) || !aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (dx == dy || dx == x) return MLPBLK_EINVAL;
    const WsLayoutF8 l = ws_layout_f8(desc);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    const WqLayout q = wq_layout(desc);
    const uint8_t *b = static_cast<const uint8_t *>(wq);
    const float *rec = reinterpret_cast<const float *>(b + q.scales);
    const F8Weights w = {b + q.w1g, b + q.w2, b + q.w1, rec + 0, rec + 4, rec + 8};
    return backward_fp8_impl(desc, dy, x, gamma, w, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved, dx,
                             dgamma, dw1, dw2, static_cast<uint8_t *>(workspace), l, sms,
                             static_cast<cudaStream_t>(stream), overwrite);
}

}  // namespace

extern "C" {

int mlpblk_backward_fp8(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma, const void *w1,
                        const void *w2, const void *h_saved, const void *a8_saved, const void *n8_saved,
                        const float *rstd_saved, const float *scales_saved, void *dx, float *dgamma, float *dw1,
                        float *dw2, void *workspace, size_t workspace_bytes, void *stream) {
    return backward_fp8_entry(desc, dy, x, gamma, w1, w2, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved, dx,
                              dgamma, dw1, dw2, workspace, workspace_bytes, stream, false);
}

int mlpblk_backward_fp8_overwrite(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                                  const void *w1, const void *w2, const void *h_saved, const void *a8_saved,
                                  const void *n8_saved, const float *rstd_saved, const float *scales_saved,
                                  void *dx, float *dgamma, float *dw1, float *dw2, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    return backward_fp8_entry(desc, dy, x, gamma, w1, w2, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved, dx,
                              dgamma, dw1, dw2, workspace, workspace_bytes, stream, true);
}

size_t mlpblk_fp8_weights_size(const mlpblk_desc *desc) {
    if (check_fp8_desc(desc) != MLPBLK_OK) return 0;
    return static_cast<size_t>(wq_layout(desc).total);
}

int mlpblk_fp8_quantize_weights(const mlpblk_desc *desc, const void *gamma, const void *w1, const void *w2,
                                void *wq, size_t wq_bytes, void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_fp8_desc(desc));
    if (!aligned16(gamma) || !aligned16(w1) || !aligned16(w2) || !aligned16(wq) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    const WqLayout q = wq_layout(desc);
    const WsLayoutF8 l = ws_layout_f8(desc);
    if (wq_bytes < static_cast<size_t>(q.total) || workspace_bytes < static_cast<size_t>(l.total))
        return MLPBLK_EWORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    uint8_t *b = static_cast<uint8_t *>(wq);
    float *rec = reinterpret_cast<float *>(b + q.scales);  // [3][4]: W1*gamma, W2, W1
    float *amax = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + l.amax);
    MLPBLK_TRY(quantize_tensor(w1, gamma, d, F * d, amax, rec + 0, b + q.w1g, s));
    MLPBLK_TRY(quantize_tensor(w2, nullptr, F, d * F, amax, rec + 4, b + q.w2, s));
    MLPBLK_TRY(quantize_tensor(w1, nullptr, d, F * d, amax, rec + 8, b + q.w1, s));
    return MLPBLK_OK;
}

int mlpblk_forward_fp8_prequant(const mlpblk_desc *desc, const void *x, const void *wq, void *y, void *h_saved,
                                void *a8_saved, void *n8_saved, float *rstd_saved, float *scales_saved,
                                void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_fp8_desc(desc));
    if (desc->tokens == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(wq) || !aligned16(y) || !aligned16(h_saved) || !aligned16(a8_saved) ||
        !aligned16(n8_saved) || !aligned16(rstd_saved) || !aligned16(scales_saved) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (y == x) return MLPBLK_EINVAL;
    const WsLayoutF8 l = ws_layout_f8(desc);
    if (workspace_bytes < static_cast<size_t>(l.total)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    const WqLayout q = wq_layout(desc);
    const uint8_t *b = static_cast<const uint8_t *>(wq);
    const float *rec = reinterpret_cast<const float *>(b + q.scales);
    const F8Weights w = {b + q.w1g, b + q.w2, b + q.w1, rec + 0, rec + 4, rec + 8};
    return forward_fp8_impl(desc, x, w, y, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved,
                            static_cast<uint8_t *>(workspace), l, sms, static_cast<cudaStream_t>(stream));
}

int mlpblk_backward_fp8_prequant(const mlpblk_desc *desc, const void *dy, const void *x, const void *gamma,
                                 const void *wq, const void *h_saved, const void *a8_saved, const void *n8_saved,
                                 const float *rstd_saved, const float *scales_saved, void *dx, float *dgamma,
                                 float *dw1, float *dw2, void *workspace, size_t workspace_bytes, void *stream) {
    return backward_fp8_prequant_entry(desc, dy, x, gamma, wq, h_saved, a8_saved, n8_saved, rstd_saved,
                                       scales_saved, dx, dgamma, dw1, dw2, workspace, workspace_bytes, stream, false);
}

int mlpblk_backward_fp8_prequant_overwrite(const mlpblk_desc *desc, const void *dy, const void *x,
                                           const void *gamma, const void *wq, const void *h_saved,
                                           const void *a8_saved, const void *n8_saved, const float *rstd_saved,
                                           const float *scales_saved, void *dx, float *dgamma, float *dw1,
                                           float *dw2, void *workspace, size_t workspace_bytes, void *stream) {
    return backward_fp8_prequant_entry(desc, dy, x, gamma, wq, h_saved, a8_saved, n8_saved, rstd_saved,
                                       scales_saved, dx, dgamma, dw1, dw2, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

namespace {

// Buffers of the routed-expert block.  R = the row space of the experts'
// segments: T*k assignments plus up to 255 padding rows per expert, rounded to 256.
struct MoeLayout {
    int64_t R;
    // saved
    int64_t rstd, pos, row_token, row_slot, seg, count, chunk_count, rstd_perm, x_perm, h_perm, a_perm, o_perm, saved;
    // workspace
    int64_t w1g, do_perm, dh_perm, dn_perm, part, sk_partial, sk_flags, ws;
};

int check_moe_desc(const mlpblk_moe_desc *m) {
    if (!m) return MLPBLK_EINVAL;
    MLPBLK_TRY(check_desc(&m->base));
    if (m->base.dtype != MLPBLK_BF16) return MLPBLK_ENOTSUP;
    if (m->experts < 1 || m->experts > 256 || m->top_k < 1 || m->top_k > m->experts) return MLPBLK_EINVAL;
    const int64_t lim = static_cast<int64_t>(1) << 31;
    const int64_t T = m->base.tokens, d = m->base.d_model, F = m->base.ffn, E = m->experts;
    if (T * m->top_k + E * 256 >= lim / (d > F ? d : F)) return MLPBLK_EINVAL;
    if (E * F >= lim / d) return MLPBLK_EINVAL;
    return MLPBLK_OK;
}

MoeLayout moe_layout(const mlpblk_moe_desc *m) {
    const int64_t T = m->base.tokens, d = m->base.d_model, F = m->base.ffn, E = m->experts, k = m->top_k;
    MoeLayout l;
    l.R = (T * k + E * 255 + 255) / 256 * 256;
    int64_t off = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = off;
        off += align256(bytes);
        return at;
    };
    l.rstd = take(T * 4);
    l.pos = take(T * k * 4);
    l.row_token = take(l.R * 4);
    l.row_slot = take(l.R * 4);
    l.seg = take((E + 1) * 4);
    l.count = take(E * 4);
    l.chunk_count = take(moe_route_chunks(T * k) * E * 4);
    l.rstd_perm = take(l.R * 4);
    l.x_perm = take(l.R * d * 2);
    l.h_perm = take(l.R * F * 2);
    l.a_perm = take(l.R * F * 2);
    l.o_perm = take(l.R * d * 2);
    l.saved = off;
    // workspace: the forward's W1*gamma and the backward's buffers share it
    off = 0;
    const int64_t w1g = align256(E * F * d * 2);
    l.w1g = 0;
    l.do_perm = take(l.R * d * 2);
    l.dh_perm = take(l.R * F * 2);
    l.dn_perm = take(l.R * d * 2);
    l.part = take(static_cast<int64_t>(kMaxParts) * d * 4);
    // the M-grouped GEMMs' split schedule: partial sums and flags, apart from the
    // forward's W1*gamma (both live in the forward)
    off = off > w1g ? off : w1g;
    l.sk_partial = take(static_cast<int64_t>(kMaxSkSlots) * kSkSlotFloats * 4);
    l.sk_flags = take(static_cast<int64_t>(kSkSets) * kSkFlagsPerSet * 4);
    l.ws = off;
    return l;
}

}  // namespace

extern "C" {

size_t mlpblk_moe_saved_size(const mlpblk_moe_desc *desc) {
    if (check_moe_desc(desc) != MLPBLK_OK) return 0;
    return static_cast<size_t>(moe_layout(desc).saved);
}

size_t mlpblk_moe_workspace_size(const mlpblk_moe_desc *desc) {
    if (check_moe_desc(desc) != MLPBLK_OK) return 0;
    return static_cast<size_t>(moe_layout(desc).ws);
}

int mlpblk_moe_forward(const mlpblk_moe_desc *desc, const void *x, const void *gamma, const void *w1s,
                       const void *w2s, const int32_t *expert_idx, const float *routing_weights, void *y,
                       void *saved, size_t saved_bytes, void *workspace, size_t workspace_bytes, void *stream) {
    MLPBLK_TRY(check_moe_desc(desc));
    if (desc->base.tokens == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(w1s) || !aligned16(w2s) || !aligned16(expert_idx) ||
        !aligned16(routing_weights) || !aligned16(y) || !aligned16(saved) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (y == x) return MLPBLK_EINVAL;
    const MoeLayout l = moe_layout(desc);
    if (saved_bytes < static_cast<size_t>(l.saved) || workspace_bytes < static_cast<size_t>(l.ws))
        return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = desc->base.tokens, d = desc->base.d_model, F = desc->base.ffn;
    const int E = desc->experts, k = desc->top_k;
    uint8_t *sv = static_cast<uint8_t *>(saved);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *rstd = reinterpret_cast<float *>(sv + l.rstd);
    int *pos = reinterpret_cast<int *>(sv + l.pos);
    int *row_token = reinterpret_cast<int *>(sv + l.row_token);
    int *row_slot = reinterpret_cast<int *>(sv + l.row_slot);
    int *seg = reinterpret_cast<int *>(sv + l.seg);
    int *count = reinterpret_cast<int *>(sv + l.count);
    int *chunk_count = reinterpret_cast<int *>(sv + l.chunk_count);
    float *rstd_perm = reinterpret_cast<float *>(sv + l.rstd_perm);
    void *x_perm = sv + l.x_perm, *h_perm = sv + l.h_perm, *a_perm = sv + l.a_perm, *o_perm = sv + l.o_perm;
    void *w1g = ws + l.w1g;
    float *sk_partial = reinterpret_cast<float *>(ws + l.sk_partial);
    int *sk_flags = reinterpret_cast<int *>(ws + l.sk_flags);
    // rstd and every expert's W1 * gamma (the experts' W1 as one [E*F, d] matrix);
    // clears the W1 GEMM's flags
    MLPBLK_LAUNCH(MLPBLK_KERNEL_FOLD_GAMMA, s,
                  launch_norm_prep(MLPBLK_BF16, x, rstd, T, d, desc->base.eps, w1s, gamma, w1g, E * F,
                                   sk_flags + kSetFwdW1 * kSkFlagsPerSet, kSkFlagsPerSet, s));
    for (int step = 0; step < kMoeRouteLaunches; ++step)
        MLPBLK_LAUNCH(MLPBLK_KERNEL_MOE_ROUTE, s,
                      launch_moe_route(expert_idx, T * k, k, E, chunk_count, count, seg, pos, row_token, row_slot,
                                       step, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_MOE_GATHER, s,
                  launch_moe_gather(x, rstd, row_token, seg, E, l.R, d, x_perm, rstd_perm, s));
    GemmArgs g1 = {};
    g1.rstd_in = rstd_perm;
    g1.grp_mode = kGroupM;
    g1.grp_count = E;
    g1.grp_rows = seg;
    g1.grp_b_off = static_cast<int>(F);
    g1.sk_partial = sk_partial;
    g1.sk_flags = sk_flags + kSetFwdW1 * kSkFlagsPerSet;
    g1.zero_flags = sk_flags + kSetFwdW2 * kSkFlagsPerSet;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W1, s,
                  launch_gemm_tc_fwd(kEpiFwdW1Pre, (int)l.R, (int)F, (int)d, x_perm, w1g, h_perm, a_perm, g1, sms, s));
    GemmArgs g2 = {};
    g2.grp_mode = kGroupM;
    g2.grp_count = E;
    g2.grp_rows = seg;
    g2.grp_b_off = static_cast<int>(d);
    g2.sk_partial = sk_partial;
    g2.sk_flags = sk_flags + kSetFwdW2 * kSkFlagsPerSet;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_FWD_W2, s,
                  launch_gemm_tc_fwd(kEpiStoreBf16, (int)l.R, (int)d, (int)F, a_perm, w2s, o_perm, nullptr, g2, sms, s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_MOE_COMBINE, s, launch_moe_combine(x, o_perm, routing_weights, pos, T, k, d, y, s));
    return MLPBLK_OK;
}

}  // extern "C"

namespace {

int moe_backward_entry(const mlpblk_moe_desc *desc, const void *dy, const void *x, const void *gamma,
                       const void *w1s, const void *w2s, const float *routing_weights, const void *saved,
                       void *dx, float *d_routing_weights, float *dgamma, float *dw1s, float *dw2s,
                       void *workspace, size_t workspace_bytes, void *stream, bool overwrite) {
    MLPBLK_TRY(check_moe_desc(desc));
    if (desc->base.tokens == 0) {
        // no rows: += adds nothing; = leaves zero gradients
        if (!overwrite) return MLPBLK_OK;
        if (!aligned16(dgamma) || !aligned16(dw1s) || !aligned16(dw2s)) return MLPBLK_EINVAL;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const int64_t d = desc->base.d_model, EF = static_cast<int64_t>(desc->experts) * desc->base.ffn;
        MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s,
                      launch_grads(true, 0.0f, dgamma, d, dw1s, EF * d, dw2s, d * EF, s));
        return MLPBLK_OK;
    }
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(w1s) || !aligned16(w2s) ||
        !aligned16(routing_weights) || !aligned16(saved) || !aligned16(dx) || !aligned16(d_routing_weights) ||
        !aligned16(dgamma) || !aligned16(dw1s) || !aligned16(dw2s) || !aligned16(workspace))
        return MLPBLK_EINVAL;
    if (dx == dy || dx == x) return MLPBLK_EINVAL;
    const MoeLayout l = moe_layout(desc);
    if (workspace_bytes < static_cast<size_t>(l.ws)) return MLPBLK_EWORKSPACE;
    int sms = 0;
    MLPBLK_TRY(device_sms(&sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = desc->base.tokens, d = desc->base.d_model, F = desc->base.ffn;
    const int E = desc->experts, k = desc->top_k;
    const uint8_t *sv = static_cast<const uint8_t *>(saved);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const float *rstd = reinterpret_cast<const float *>(sv + l.rstd);
    const int *pos = reinterpret_cast<const int *>(sv + l.pos);
    const int *seg = reinterpret_cast<const int *>(sv + l.seg);
    const int *count = reinterpret_cast<const int *>(sv + l.count);
    const float *rstd_perm = reinterpret_cast<const float *>(sv + l.rstd_perm);
    const void *x_perm = sv + l.x_perm, *h_perm = sv + l.h_perm, *a_perm = sv + l.a_perm, *o_perm = sv + l.o_perm;
    void *do_perm = ws + l.do_perm, *dh_perm = ws + l.dh_perm;
    uint16_t *dn_perm = reinterpret_cast<uint16_t *>(ws + l.dn_perm);  // bf16
    float *part = reinterpret_cast<float *>(ws + l.part);
    float *sk_partial = reinterpret_cast<float *>(ws + l.sk_partial);
    int *sk_flags = reinterpret_cast<int *>(ws + l.sk_flags);
    int parts = 0;
    // d_routing_weights and each slot's output gradient p * dy in segment order
    // (overwrite: it also clears the gradient blocks of experts no token chose,
    // which the K-grouped wgrads skip)
    MLPBLK_LAUNCH(MLPBLK_KERNEL_MOE_DP, s,
                  launch_moe_dout(dy, o_perm, routing_weights, pos, count, seg, T, k, E, d, d_routing_weights, do_perm,
                                  overwrite ? dw1s : nullptr, overwrite ? dw2s : nullptr, F, s));
    GemmArgs gw2 = {};
    gw2.grp_mode = kGroupK;
    gw2.grp_count = E;
    gw2.grp_rows = seg;
    gw2.grp_c_off = static_cast<int>(d);
    gw2.overwrite = overwrite ? 1 : 0;  // whole tiles: a store instead of an add
    gw2.zero_flags = sk_flags + kSetDgradH * kSkFlagsPerSet;
    gw2.pdl = kPdlWaitFirst;  // (dW2, dh) and (dn, dW1) overlap as in the dense backward
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W2, s,
                  launch_gemm_tc_bwd(kEpiAccF32, (int)d, (int)F, (int)l.R, do_perm, a_perm, dw2s, nullptr, gw2, sms, s));
    GemmArgs gd = {};
    gd.aux = static_cast<const uint16_t *>(h_perm);
    gd.ld_aux = (int)F;
    gd.rstd_in = rstd_perm;
    gd.grp_mode = kGroupM;
    gd.grp_count = E;
    gd.grp_rows = seg;
    gd.grp_b_off = static_cast<int>(d);
    gd.sk_partial = sk_partial;
    gd.sk_flags = sk_flags + kSetDgradH * kSkFlagsPerSet;
    gd.zero_flags = sk_flags + kSetDgradN * kSkFlagsPerSet;
    gd.pdl = kPdlDeferWait;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_H, s,
                  launch_gemm_tc_bwd(kEpiDgradH, (int)l.R, (int)F, (int)d, do_perm, w2s, dh_perm, nullptr, gd, sms, s));
    GemmArgs gn = {};
    gn.grp_mode = kGroupM;
    gn.grp_count = E;
    gn.grp_rows = seg;
    gn.grp_b_off = static_cast<int>(F);
    gn.sk_partial = sk_partial;
    gn.sk_flags = sk_flags + kSetDgradN * kSkFlagsPerSet;
    gn.pdl = kPdlWaitFirst;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_DGRAD_N, s,
                  launch_gemm_tc_bwd(kEpiStoreBf16, (int)l.R, (int)d, (int)F, dh_perm, w1s, dn_perm, nullptr, gn, sms, s));
    GemmArgs gw1 = {};
    gw1.colscale = static_cast<const uint16_t *>(gamma);
    gw1.grp_mode = kGroupK;
    gw1.grp_count = E;
    gw1.grp_rows = seg;
    gw1.grp_c_off = static_cast<int>(F);
    gw1.overwrite = overwrite ? 1 : 0;
    gw1.pdl = kPdlDeferWait;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_GEMM_WGRAD_W1, s,
                  launch_gemm_tc_bwd(kEpiAccF32ColScale, (int)F, (int)d, (int)l.R, dh_perm, x_perm, dw1s, nullptr, gw1,
                                     sms, s));
    // the slots' dn meet at n (sum rule) inside the RMSNorm backward
    MLPBLK_LAUNCH(MLPBLK_KERNEL_NORM_BWD, s,
                  launch_rmsnorm_bwd_gather(x, dn_perm, 1, pos, k, dy, rstd, gamma, dx, part, T, d, kMaxParts, &parts,
                                            s));
    MLPBLK_LAUNCH(MLPBLK_KERNEL_DGAMMA_REDUCE, s,
                  launch_dgamma_finalize(part, parts, dgamma, d, s, overwrite ? 1 : 0));
    return MLPBLK_OK;
}

}  // namespace

extern "C" {

int mlpblk_moe_backward(const mlpblk_moe_desc *desc, const void *dy, const void *x, const void *gamma,
                        const void *w1s, const void *w2s, const float *routing_weights, const void *saved, void *dx,
                        float *d_routing_weights, float *dgamma, float *dw1s, float *dw2s, void *workspace,
                        size_t workspace_bytes, void *stream) {
    return moe_backward_entry(desc, dy, x, gamma, w1s, w2s, routing_weights, saved, dx, d_routing_weights, dgamma,
                              dw1s, dw2s, workspace, workspace_bytes, stream, false);
}

int mlpblk_moe_backward_overwrite(const mlpblk_moe_desc *desc, const void *dy, const void *x, const void *gamma,
                                  const void *w1s, const void *w2s, const float *routing_weights, const void *saved,
                                  void *dx, float *d_routing_weights, float *dgamma, float *dw1s, float *dw2s,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    return moe_backward_entry(desc, dy, x, gamma, w1s, w2s, routing_weights, saved, dx, d_routing_weights, dgamma,
                              dw1s, dw2s, workspace, workspace_bytes, stream, true);
}

int mlpblk_zero_grads(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2, void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (!aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2)) return MLPBLK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_ZERO_GRADS, s,
                  launch_grads(true, 0.0f, dgamma, d, dw1, F * d, dw2, F * d, s));
    return MLPBLK_OK;
}

int mlpblk_scale_grads(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2, float sc,
                       void *stream) {
    MLPBLK_TRY(check_desc(desc));
    if (!aligned16(dgamma) || !aligned16(dw1) || !aligned16(dw2)) return MLPBLK_EINVAL;
    if (!isfinite(sc)) return MLPBLK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t d = desc->d_model, F = desc->ffn;
    MLPBLK_LAUNCH(MLPBLK_KERNEL_SCALE_GRADS, s,
                  launch_grads(false, sc, dgamma, d, dw1, F * d, dw2, F * d, s));
    return MLPBLK_OK;
}

int mlpblk_set_rmsnorm_mode(int mode) {
    if (mode != MLPBLK_RMSNORM_STATS_PASS && mode != MLPBLK_RMSNORM_IN_W1_PROLOGUE) return MLPBLK_EINVAL;
    g_rms_mode = mode;
    return MLPBLK_OK;
}

int mlpblk_set_test_fault(int fault) {
    if (fault != MLPBLK_TEST_FAULT_NONE && fault != MLPBLK_TEST_FAULT_SKIP_LOADS) return MLPBLK_EINVAL;
    g_test_fault = fault;
    return MLPBLK_OK;
}

int mlpblk_trace_begin(void **events, int *kinds, int capacity) {
    if (!events || !kinds || capacity < 1) return MLPBLK_EINVAL;
    g_trace.events = reinterpret_cast<cudaEvent_t *>(events);
    g_trace.kinds = kinds;
    g_trace.capacity = capacity;
    g_trace.count = 0;
    g_trace.on = true;
    return MLPBLK_OK;
}

int mlpblk_trace_end(void) {
    g_trace.on = false;
    return g_trace.count;
}

const char *mlpblk_cuda_error_string(void) {
    if (g_last_cuda_error == 0) return "no CUDA error recorded";
    return cudaGetErrorString(static_cast<cudaError_t>(g_last_cuda_error));
}

int mlpblk_last_error(void) {
    if (cuda_status(cudaDeviceSynchronize()) != MLPBLK_OK) return MLPBLK_ECUDA;
    const int a = take_device_error_gemm_fwd();
    const int b = take_device_error_gemm_bwd();
    const int c = take_device_error_gemm_f8();
    const int r = take_device_error_rowops();
    return a != MLPBLK_OK ? a : (b != MLPBLK_OK ? b : (c != MLPBLK_OK ? c : r));
}

}  // extern "C"
