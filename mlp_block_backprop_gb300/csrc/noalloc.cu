// noalloc.cu -- mlpblk_rmsnorm_backward_noalloc: the RMSNorm backward row
// kernel (with the residual gradient and dgamma) for callers that cannot hand
// the library any device scratch.  Its only scratch, the per-block dgamma
// partial sums, lives in a fixed array owned by the library.
#include <atomic>

#include "mlpblk_internal.h"

using namespace mlpblk;

namespace {

// dgamma partial rows of mlpblk_rmsnorm_backward_noalloc: P rows of d_model
// floats, P <= kScratchFloats / d_model.  4 MiB, held by every GPU that loads
// the library until the process exits.
constexpr int64_t kScratchFloats = int64_t(1) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

// In host code g_noalloc_scratch names a host-side stand-in, not device
// memory; kernels get the device address looked up here, once per device.
// Host threads may make a device's first call at the same time: each looks the
// address up (the same value) and publishes it with a release store, so a
// reader that sees the pointer sees a finished lookup.
std::atomic<float *> g_scratch_dev[64];

int device_setup(float **scratch) {
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != MLPBLK_OK || dev < 0 || dev >= 64) return MLPBLK_ECUDA;
    float *known = g_scratch_dev[dev].load(std::memory_order_acquire);
    if (known == nullptr) {
        int major = 0, minor = 0;
        if (cuda_status(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            cuda_status(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)))
            return MLPBLK_ECUDA;
        if (major != 10 || minor != 3) return MLPBLK_ENODEV;
        void *p = nullptr;
        const int rc = cuda_status(cudaGetSymbolAddress(&p, g_noalloc_scratch));
        if (rc != MLPBLK_OK) return rc;
        known = static_cast<float *>(p);
        g_scratch_dev[dev].store(known, std::memory_order_release);
    }
    *scratch = known;
    return MLPBLK_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int mlpblk_rmsnorm_backward_noalloc(const mlpblk_desc *desc, const void *x,
                                               const float *dn, const void *dy, const void *gamma,
                                               const float *rstd, void *dx, float *dgamma,
                                               void *stream) {
    if (!desc) return MLPBLK_EINVAL;
    if (desc->dtype != MLPBLK_BF16 && desc->dtype != MLPBLK_FP32) return MLPBLK_ENOTSUP;
    const int64_t T = desc->tokens, d = desc->d_model;
    if (T < 0 || d <= 0) return MLPBLK_EINVAL;
    if (d % 8 != 0) return MLPBLK_ENOTSUP;
    if (d > kMaxNormD || d > kScratchFloats) return MLPBLK_ENOTSUP;  // beyond the array's row width
    if (T == 0) return MLPBLK_OK;
    if (!aligned16(x) || !aligned16(dn) || !aligned16(dy) || !aligned16(gamma) || !aligned16(rstd) ||
        !aligned16(dx) || !aligned16(dgamma))
        return MLPBLK_EINVAL;
    if (dx == dy || dx == x) return MLPBLK_EINVAL;
    float *scratch = nullptr;
    const int rc = device_setup(&scratch);
    if (rc != MLPBLK_OK) return rc;
    int max_parts = 512;
    if (max_parts > kScratchFloats / d) max_parts = static_cast<int>(kScratchFloats / d);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every one of the `parts` partial rows is written before it is read, so
    // nothing left in the array by an earlier call reaches the result
    int parts = 0;
    const int r1 = launch_rmsnorm_bwd_unscaled(desc->dtype, x, dn, dy, rstd, gamma, dx, scratch, T,
                                               d, max_parts, &parts, s);
    if (r1 != MLPBLK_OK) return r1;
    return launch_dgamma_finalize(scratch, parts, dgamma, d, s);
}
