/*
 * mlpblk.h -- C ABI of the GB300 (sm_103a) forward and backward of the
 * pre-normalised residual ReLU² MLP block
 *
 *     n = RMSNorm(x) = x * r * gamma,     r[t] = 1 / sqrt(mean_k x[t,k]^2 + eps)
 *     h = n . W1^T                        (saved)
 *     a = relu(h)^2                       (saved: it is also the W2 operand)
 *     y = x + a . W2^T
 *
 * Sources (page title -- section):
 *   "Nemotron Kernels From Inference To Backpropagation" -- "Setup: The Shared
 *     Transformer Shell" (pre-norm residual shell; backward starts at the residual
 *     split; RMSNorm backward needs x, gamma and the inverse RMS) and "Kernel 3:
 *     Dense ReLU2 Inference And Backpropagation" (project, relu squared, project;
 *     the pre-activation is kept for backward).
 *   "Reverse-mode automatic differentiation" -- section 5 (MatMul: g.B^T and
 *     A^T.g; Relu; LayerNorm rule, here without the mean terms).
 *   "grow_a_language_model_backprop" -- forward/backward kernel pairing, saved
 *     tensors, += accumulation across microbatches, scale_grads(1/n), zero_grads(),
 *     preallocated buffers.
 *
 * Conventions shared by every entry point
 *   - All tensors are dense and row-major.  x, y, dy, dx: [tokens, d_model];
 *     h, a: [tokens, ffn]; W1, dW1: [ffn, d_model]; W2, dW2: [d_model, ffn];
 *     gamma, dgamma: [d_model]; rstd: [tokens].
 *   - Element types.  MLPBLK_BF16: x, gamma, W1, W2, y, h, a, dy, dx are bfloat16
 *     (passed as 16-bit storage); rstd and the gradient buffers dgamma, dW1, dW2
 *     are float32.  MLPBLK_FP32: every tensor is float32.
 *   - Every pointer except `stream` is a DEVICE pointer, 16-byte aligned, owned by
 *     the caller.  The library allocates no device memory and keeps no per-call
 *     state; the scratch it needs lives in the caller's workspace.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and does not synchronise the host.  Argument errors are
 *     reported by the return value before anything is enqueued.  A device-side
 *     failure (a bounded wait that gave up) is reported later by
 *     mlpblk_last_error().
 *   - Limits: d_model and ffn positive multiples of 8 (16-byte rows); tokens >= 0
 *     and tokens * max(d_model, ffn) < 2^31; eps finite and >= 0.  tokens == 0 is a
 *     valid empty microbatch: the call checks the descriptor and returns MLPBLK_OK
 *     without touching any buffer.
 *   - No C++ exception crosses this boundary.
 */
#ifndef MLPBLK_H
#define MLPBLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MLPBLK_OK          0  /* success (work enqueued)                                 */
#define MLPBLK_EINVAL      1  /* null or misaligned pointer, bad size, bad eps          */
#define MLPBLK_ENOTSUP     2  /* unknown dtype, or d_model/ffn not a multiple of 8      */
#define MLPBLK_EWORKSPACE  3  /* workspace smaller than mlpblk_workspace_size()         */
#define MLPBLK_ECUDA       4  /* a CUDA runtime call or a kernel launch failed          */
#define MLPBLK_ETIMEOUT    5  /* a device-side bounded wait gave up (mlpblk_last_error) */
#define MLPBLK_ENODEV      6  /* the current device is not sm_103 (GB300)               */

/* Element-type selector for mlpblk_desc.dtype. */
#define MLPBLK_BF16 1
#define MLPBLK_FP32 2

/* Shape of one microbatch through one block. */
typedef struct {
    int64_t tokens;   /* T: rows of x in this microbatch                     */
    int64_t d_model;  /* d: model width                                      */
    int64_t ffn;      /* F: hidden width of the MLP                          */
    float   eps;      /* RMSNorm epsilon, added to mean(x^2) inside the root */
    int32_t dtype;    /* MLPBLK_BF16 or MLPBLK_FP32                          */
} mlpblk_desc;

/*
 * Bytes of device workspace that mlpblk_forward and mlpblk_backward need for
 * `desc` (one size serves both).  Returns 0 for an invalid descriptor.  The
 * workspace holds scratch only (gamma-folded W1, the rstd-scaled dh, dn, the
 * per-block dgamma partials, and the GEMMs' stream-K partial sums and flags,
 * which every call initialises itself); its contents need not be preserved
 * between calls, but two calls in flight at once must not share one workspace.
 */
size_t mlpblk_workspace_size(const mlpblk_desc *desc);

/*
 * Forward of one microbatch ("Setup: The Shared Transformer Shell";
 * "Kernel 3: Dense ReLU2 ...").
 *   in : x[T,d], gamma[d], w1[F,d], w2[d,F]
 *   out: y[T,d]          = x + relu(h)^2 . W2^T                      (written)
 *        h_saved[T,F]    = RMSNorm(x) . W1^T, rounded to the dtype    (written)
 *        a_saved[T,F]    = relu(h)^2, rounded to the dtype            (written)
 *        rstd_saved[T]   = 1/sqrt(mean_k x^2 + eps), float32          (written)
 * y must not alias x.  Returns an MLPBLK_* code.
 */
int mlpblk_forward(const mlpblk_desc *desc,
                   const void *x, const void *gamma, const void *w1, const void *w2,
                   void *y, void *h_saved, void *a_saved, float *rstd_saved,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * W1 * gamma, the forward's first GEMM operand (RMSNorm's gamma folded into W1
 * along d: w1g[f,k] = w1[f,k] * gamma[k], rounded once to the dtype).  It depends
 * on the weights only, so a caller that runs several microbatches with the same
 * weights (gradient accumulation, "grow_a_language_model_backprop", accumulating
 * across microbatches) makes it once per weight update and passes it to
 * mlpblk_forward_prefolded; mlpblk_forward folds on every call.
 *   in : gamma[d], w1[F,d] (desc->dtype)      out: w1g[F,d] (desc->dtype, written)
 * desc->tokens and desc->eps are not used.  w1g must not alias w1.  Pointers
 * are device pointers, 16-byte aligned.  Returns an MLPBLK_* code.
 */
int mlpblk_fold_weights(const mlpblk_desc *desc, const void *gamma, const void *w1, void *w1g,
                        void *stream);

/*
 * mlpblk_forward with the folded weight from mlpblk_fold_weights in place of
 * gamma and w1: the same outputs, bit for bit, without the per-call fold.
 * Workspace as for mlpblk_forward (mlpblk_workspace_size).
 */
int mlpblk_forward_prefolded(const mlpblk_desc *desc, const void *x, const void *w1g, const void *w2,
                             void *y, void *h_saved, void *a_saved, float *rstd_saved,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward of one microbatch (the residual branch copies forward and adds
 * backward; d relu(h)^2/dh = 2 relu(h), 0 at h = 0; RMSNorm backward from the
 * saved rstd).  Consumes the forward's saved h, a and rstd for the same x.
 *   in : dy[T,d], x[T,d], gamma[d], w1[F,d], w2[d,F], h_saved, a_saved, rstd_saved
 *   out: dx[T,d]        = dy + RMSNorm backward of dn                 (written)
 *        dgamma[d]     += sum_t dn[t,k] * x[t,k] * r[t]      float32 (accumulated)
 *        dw1[F,d]      += dh^T . n                           float32 (accumulated)
 *        dw2[d,F]      += dy^T . a                           float32 (accumulated)
 *   where dh = (dy . W2) * 2 relu(h) and dn = dh . W1.  The gradient buffers keep
 *   a running sum across calls until mlpblk_zero_grads.  dx must not alias dy or
 *   x.  Returns an MLPBLK_* code.
 */
int mlpblk_backward(const mlpblk_desc *desc,
                    const void *dy, const void *x, const void *gamma,
                    const void *w1, const void *w2,
                    const void *h_saved, const void *a_saved, const float *rstd_saved,
                    void *dx, float *dgamma, float *dw1, float *dw2,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * The first microbatch of an accumulation window: the same backward with the
 * gradients set rather than added into ("grow_a_language_model_backprop" --
 * accumulation across microbatches: zero_grads() then += is = for the first
 * microbatch):
 *        dgamma[d]  = sum_t dn[t,k] * x[t,k] * r[t]
 *        dw1[F,d]   = dh^T . n,   dw2[d,F] = dy^T . a        (float32, written)
 * The buffers' prior contents do not matter (NaN included), so the window needs
 * no mlpblk_zero_grads; with T = 0 they are set to zero.  The weight-gradient
 * GEMMs store every output tile that one worker sums whole and add the parts of
 * the tiles they split between workers into regions that the call's first
 * launch clears (with dgamma), so the values are those of mlpblk_zero_grads +
 * mlpblk_backward up to the order in which a split tile's parts are added (the
 * fp32 path clears all three buffers and adds).  dx, the other arguments, the
 * workspace and the return codes are as for mlpblk_backward.
 */
int mlpblk_backward_overwrite(const mlpblk_desc *desc,
                              const void *dy, const void *x, const void *gamma,
                              const void *w1, const void *w2,
                              const void *h_saved, const void *a_saved, const float *rstd_saved,
                              void *dx, float *dgamma, float *dw1, float *dw2,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Recompute variant: save x and rstd only, and rebuild h and a at the start of
 * the backward ("Nemotron Kernels From Inference To Backpropagation" -- Part II:
 * training must preserve or later recompute what reverse mode needs, and an
 * engine states what is saved and what is recomputed; "grow_a_language_model_
 * backprop" -- saved tensors dominate activation memory).  It trades the
 * 2*T*F*elt bytes of saved h and a per block for one more W1 GEMM
 * (2*T*d*F FLOP) in the backward; h and a live in the workspace only while a
 * call runs, so one workspace serves every block of a model.
 *
 * mlpblk_workspace_size_recompute: bytes of workspace both recompute calls
 * need (larger than mlpblk_workspace_size by the T x F h and a).  0 for an
 * invalid descriptor.
 *
 * mlpblk_forward_recompute: y and rstd_saved exactly as mlpblk_forward writes
 * them (same kernels and schedule, the W1 epilogue writing a alone into the
 * workspace; bf16 keeps no h at all).
 *
 * mlpblk_backward_recompute: recomputes h and a from x, W1, gamma and
 * rstd_saved with the forward's W1 GEMM (the same bits the forward produced),
 * then runs mlpblk_backward's kernels; dx written, dgamma/dw1/dw2 += as there.
 * Argument rules and return codes as for mlpblk_forward / mlpblk_backward.
 */
size_t mlpblk_workspace_size_recompute(const mlpblk_desc *desc);

int mlpblk_forward_recompute(const mlpblk_desc *desc,
                             const void *x, const void *gamma, const void *w1, const void *w2,
                             void *y, float *rstd_saved,
                             void *workspace, size_t workspace_bytes, void *stream);

int mlpblk_backward_recompute(const mlpblk_desc *desc,
                              const void *dy, const void *x, const void *gamma,
                              const void *w1, const void *w2, const float *rstd_saved,
                              void *dx, float *dgamma, float *dw1, float *dw2,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Optimizer-side steps after the accumulation loop ("grow_a_language_model_
 * backprop" -- the two-stage gradient-norm kernels and the gradient scale used
 * for clipping; "optimizer state": AdamW holds a first and a second moment per
 * weight; "Losing small gradient contributions in BF16": the state an update
 * accumulates into stays float32).  All asynchronous on `stream`; the norm and
 * the clip scale stay on the device, so clipping needs no host round trip.
 *
 * mlpblk_grad_norm: norm_out[0] = sqrt(sum of g^2 over dgamma[d], dw1[F,d],
 *   dw2[d,F]) and clip_scale_out[0] = min(1, max_norm / (norm + 1e-6)), both
 *   float32 device scalars (either may be NULL, not both).  Per-CTA partial sums
 *   (float32 with compensation, then float64) go to `workspace`
 *   (>= mlpblk_workspace_size(desc) bytes) and are added in a fixed order.
 *   max_norm > 0 and finite.  desc->tokens is ignored.
 *
 * mlpblk_clip_grads: dgamma, dw1, dw2 *= clip_scale[0] (a device scalar, e.g.
 *   the one mlpblk_grad_norm wrote).
 *
 * mlpblk_adamw_step: one AdamW update (decoupled weight decay; Loshchilov &
 *   Hutter, "Decoupled Weight Decay Regularization", Algorithm 2) of `count`
 *   tensors, `step` >= 1 counting updates:
 *     g <- g * grad_scale[0] (if grad_scale is not NULL), w <- w * (1 - lr*wd)
 *     (tensors with decay != 0), m <- b1*m + (1-b1)*g, v <- b2*v + (1-b2)*g^2,
 *     w <- w - lr/(1-b1^step) * m / (sqrt(v)/sqrt(1-b2^step) + eps)
 *   on the float32 master weights, then weight = w in `dtype` (MLPBLK_BF16:
 *   rounded to nearest even; weight may be NULL).  master, grad, m, v 16-byte
 *   aligned, weight 8-byte (bf16) / 16-byte (fp32) aligned, n a positive
 *   multiple of 4; grads are read only.  Returns MLPBLK_EINVAL on bad
 *   hyper-parameters (0 <= beta < 1, lr >= 0, eps >= 0, wd >= 0, finite).
 */
typedef struct {
    float       *master;  /* float32 master weights [n] (updated)                 */
    void        *weight;  /* working copy in `dtype` [n] (written) or NULL         */
    const float *grad;    /* float32 gradient [n]                                  */
    float       *m, *v;   /* AdamW first and second moments [n] (updated)         */
    int64_t      n;       /* elements                                             */
    int32_t      decay;   /* nonzero: apply the weight decay to this tensor        */
} mlpblk_param;

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} mlpblk_adamw;

int mlpblk_grad_norm(const mlpblk_desc *desc, const float *dgamma, const float *dw1,
                     const float *dw2, float max_norm, float *norm_out, float *clip_scale_out,
                     void *workspace, size_t workspace_bytes, void *stream);

int mlpblk_clip_grads(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2,
                      const float *clip_scale, void *stream);

int mlpblk_adamw_step(const mlpblk_param *params, int count, const mlpblk_adamw *hp,
                      int64_t step, int dtype, const float *grad_scale, void *stream);

/*
 * FP8-operand variant: the same block with the six GEMMs on E4M3 operands
 * (tcgen05 kind::f8f6f4, float32 accumulators; "Nemotron Kernels From
 * Inference To Backpropagation" -- "Where Quantization Fits": quantisation as a
 * policy for particular tensor edges, higher-precision accumulators kept).
 * Tensors in and out are bf16 (desc->dtype = MLPBLK_BF16), d_model and ffn
 * multiples of 16.  Per-tensor scaling: s = amax / 448, codes E4M3(v / s)
 * nearest-even and saturated, the GEMM epilogue multiplies by the operands'
 * scales.  Quantised: n' = x * rstd (scale 1, |n'| <= sqrt(d)), W1 * gamma, W2,
 * a (from its bf16 value), dy, dh (from its bf16 value), W1; everything else as
 * in mlpblk_forward / mlpblk_backward.
 *
 * Saved by the forward for the backward (caller-owned):
 *   h_saved[T,F] bf16, a8_saved[T,F] E4M3 codes (1 byte), n8_saved[T,d] E4M3
 *   codes of n', rstd_saved[T] float32, scales_saved[4] float32 (a's scale
 *   record {amax, 448/amax, amax/448, 0}).
 * mlpblk_workspace_size_fp8: scratch bytes both calls need; 0 for an invalid or
 *   unsupported descriptor.
 */
size_t mlpblk_workspace_size_fp8(const mlpblk_desc *desc);

int mlpblk_forward_fp8(const mlpblk_desc *desc,
                       const void *x, const void *gamma, const void *w1, const void *w2,
                       void *y, void *h_saved, void *a8_saved, void *n8_saved,
                       float *rstd_saved, float *scales_saved,
                       void *workspace, size_t workspace_bytes, void *stream);

int mlpblk_backward_fp8(const mlpblk_desc *desc,
                        const void *dy, const void *x, const void *gamma,
                        const void *w1, const void *w2,
                        const void *h_saved, const void *a8_saved, const void *n8_saved,
                        const float *rstd_saved, const float *scales_saved,
                        void *dx, float *dgamma, float *dw1, float *dw2,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * The same FP8 calls with the weights quantised once, e.g. once per optimizer
 * step for every microbatch of a gradient-accumulation window (the weights do not
 * change between the microbatches, so neither do their codes).
 *
 * mlpblk_fp8_weights_size: bytes of a pre-quantised weight buffer `wq`
 *   (caller-owned, 16-byte aligned): E4M3 codes of W1*gamma [F,d], W2 [d,F] and
 *   W1 [F,d], then their three scale records; 0 for an invalid descriptor.
 * mlpblk_fp8_quantize_weights: fills `wq` from gamma, w1, w2 (bf16) with the same
 *   per-tensor scaling as mlpblk_forward_fp8 / mlpblk_backward_fp8 (uses the FP8
 *   workspace for its amax scratch).  Call it again whenever gamma, W1 or W2
 *   change.
 * mlpblk_forward_fp8_prequant / mlpblk_backward_fp8_prequant: as
 *   mlpblk_forward_fp8 / mlpblk_backward_fp8, reading the weights' codes and
 *   scales from `wq`; outputs are bitwise those of the quantising calls (dW1 and
 *   dW2 up to the order of the reduce-adds of a split weight-gradient tile).
 * Returns an MLPBLK_* code.
 */
size_t mlpblk_fp8_weights_size(const mlpblk_desc *desc);

int mlpblk_fp8_quantize_weights(const mlpblk_desc *desc,
                                const void *gamma, const void *w1, const void *w2,
                                void *wq, size_t wq_bytes,
                                void *workspace, size_t workspace_bytes, void *stream);

int mlpblk_forward_fp8_prequant(const mlpblk_desc *desc,
                                const void *x, const void *wq,
                                void *y, void *h_saved, void *a8_saved, void *n8_saved,
                                float *rstd_saved, float *scales_saved,
                                void *workspace, size_t workspace_bytes, void *stream);

int mlpblk_backward_fp8_prequant(const mlpblk_desc *desc,
                                 const void *dy, const void *x, const void *gamma, const void *wq,
                                 const void *h_saved, const void *a8_saved, const void *n8_saved,
                                 const float *rstd_saved, const float *scales_saved,
                                 void *dx, float *dgamma, float *dw1, float *dw2,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* The two FP8 backwards with dgamma, dw1 and dw2 set instead of added into (the
 * first microbatch of an accumulation window), as mlpblk_backward_overwrite is
 * to mlpblk_backward: the weight-gradient GEMMs store the tiles one worker sums
 * whole and add split tiles' parts into regions the call's first launch clears.
 * Arguments, layouts, ownership and error codes are those of the adding forms;
 * the old contents of the three gradient buffers are never read (NaN is fine).
 * With tokens == 0 the call zeroes dgamma, dw1 and dw2 (MLPBLK_EINVAL if one of
 * them is not 16-byte aligned). */
int mlpblk_backward_fp8_overwrite(const mlpblk_desc *desc,
                                  const void *dy, const void *x, const void *gamma,
                                  const void *w1, const void *w2,
                                  const void *h_saved, const void *a8_saved, const void *n8_saved,
                                  const float *rstd_saved, const float *scales_saved,
                                  void *dx, float *dgamma, float *dw1, float *dw2,
                                  void *workspace, size_t workspace_bytes, void *stream);
int mlpblk_backward_fp8_prequant_overwrite(const mlpblk_desc *desc,
                                           const void *dy, const void *x, const void *gamma, const void *wq,
                                           const void *h_saved, const void *a8_saved, const void *n8_saved,
                                           const float *rstd_saved, const float *scales_saved,
                                           void *dx, float *dgamma, float *dw1, float *dw2,
                                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Routed ReLU^2 experts ("Nemotron Kernels From Inference To Backpropagation" --
 * "Kernel 4: Routed ReLU2 MoE Inference And Backpropagation"): the pre-norm
 * shell around a mixture of ReLU^2 experts with a given top-k dispatch,
 *   y[t] = x[t] + sum_j p[t,j] * W2_e relu(W1_e n[t])^2,  e = expert_idx[t,j],
 * n = RMSNorm(x) as in mlpblk_forward.  The dispatch is held fixed ("Hard
 * Top-K Has No Ordinary Derivative"); the backward returns d_hidden (dx),
 * d_routing_weights (dp), d_expert_up (dw1s +=), d_expert_down (dw2s +=) and
 * dgamma (+=).  bf16 tensors (base.dtype = MLPBLK_BF16), float32 routing
 * weights and gradients, int32 expert ids; an id outside [0, experts) selects
 * nothing.  Weights: w1s[E][F][d], w2s[E][d][F].
 *
 * Each expert's (token, slot) assignments run as one segment of a grouped GEMM
 * (segments padded to 256 rows, token order within a segment); every sum has a
 * fixed order except the weight-gradient accumulation (TMA reduce-add).
 *
 * saved: written by the forward, read by the backward (rstd, the dispatch, the
 * gathered inputs, h, a and the experts' outputs); mlpblk_moe_saved_size bytes.
 * workspace: scratch; mlpblk_moe_workspace_size bytes.  Both sizes are 0 for an
 * invalid descriptor (experts 1..256, top_k 1..experts, d_model <= 4096).
 */
typedef struct {
    mlpblk_desc base;   /* tokens, d_model, ffn (per expert), eps, dtype        */
    int32_t experts;    /* E                                                    */
    int32_t top_k;      /* k: experts per token                                 */
} mlpblk_moe_desc;

size_t mlpblk_moe_saved_size(const mlpblk_moe_desc *desc);
size_t mlpblk_moe_workspace_size(const mlpblk_moe_desc *desc);

int mlpblk_moe_forward(const mlpblk_moe_desc *desc,
                       const void *x, const void *gamma, const void *w1s, const void *w2s,
                       const int32_t *expert_idx, const float *routing_weights,
                       void *y, void *saved, size_t saved_bytes,
                       void *workspace, size_t workspace_bytes, void *stream);

int mlpblk_moe_backward(const mlpblk_moe_desc *desc,
                        const void *dy, const void *x, const void *gamma,
                        const void *w1s, const void *w2s, const float *routing_weights,
                        const void *saved, void *dx, float *d_routing_weights,
                        float *dgamma, float *dw1s, float *dw2s,
                        void *workspace, size_t workspace_bytes, void *stream);

/* As mlpblk_moe_backward, with dgamma, dw1s and dw2s set instead of added
 * into (the first microbatch of an accumulation window; see
 * mlpblk_backward_overwrite).  Here each expert's weight-gradient tile is one
 * worker's whole sum, so the GEMMs store it where they would add it (bitwise
 * the same values), and the blocks of experts that no token chose are set to
 * zero by the first launch of the backward. */
int mlpblk_moe_backward_overwrite(const mlpblk_moe_desc *desc,
                                  const void *dy, const void *x, const void *gamma,
                                  const void *w1s, const void *w2s, const float *routing_weights,
                                  const void *saved, void *dx, float *d_routing_weights,
                                  float *dgamma, float *dw1s, float *dw2s,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * zero_grads() of the accumulation loop ("grow_a_language_model_backprop" --
 * accumulation across microbatches): dgamma[d], dw1[F,d], dw2[d,F] = 0 (float32).
 * desc->tokens is ignored.  Returns an MLPBLK_* code.
 */
int mlpblk_zero_grads(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2,
                      void *stream);

/*
 * scale_grads(s) of the same loop, e.g. s = 1/n_microbatches:
 * dgamma, dw1, dw2 *= s (float32, one rounding per element).  s must be finite.
 * desc->tokens is ignored.  Returns an MLPBLK_* code.
 */
int mlpblk_scale_grads(const mlpblk_desc *desc, float *dgamma, float *dw1, float *dw2,
                       float s, void *stream);

/*
 * First device-side error recorded since the previous call (MLPBLK_OK if none),
 * then clears it.  Synchronises the current device.  MLPBLK_ETIMEOUT means a
 * kernel's bounded wait on a pipeline barrier gave up and the kernel returned
 * early: its outputs are not valid.
 */
int mlpblk_last_error(void);

/*
 * RMSNorm backward with the residual gradient, for callers that cannot give
 * the library any device scratch memory.  The paper has no counterpart to this
 * entry point: it is the row kernel of mlpblk_backward offered on its own.
 *
 * Who needs it: code that runs inside a host engine which owns all device
 * memory and plans every buffer once at start-up, and gives its extensions no
 * way to allocate (a cudaMalloc there breaks the memory plan and can fail with
 * out-of-memory in the middle of a step); and code on threads that must not
 * stall on the implicit device synchronisation cudaMalloc and cudaFree can
 * cause.  This call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  Its scratch (the per-block dgamma partial sums)
 * is a fixed 4 MiB array inside the library, held by every GPU that loads the
 * library until the process exits.
 *
 *   in : x[T,d], dy[T,d], gamma[d] (desc->dtype), dn[T,d] float32 = the gradient
 *        of the normalised output n = x * r * gamma, rstd[T] float32 = r
 *   out: dx[T,d]     = dy + r * (g - xh * mean_k(g * xh)),  xh = x*r, g = dn*gamma
 *                                                                        (written)
 *        dgamma[d]  += sum_t dn[t,k] * xh[t,k]                float32 (accumulated)
 * Limits: d_model a multiple of 8 and at most 4096 (MLPBLK_ENOTSUP beyond: one
 * partial row must fit the array); any tokens >= 0 (rows are indexed in 64
 * bits; at most min(512, 1048576 / d_model) partial rows are used, and with
 * more tokens each partial row sums more of them).
 * desc->ffn and desc->eps are not used.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, so make one call on every
 * device before capturing any stream of that device into a CUDA graph.  Host
 * threads may make a device's first call at the same time (each finds the same
 * address).  Every call also queries the current device, its SM count and the
 * row kernel's occupancy on the host; these enqueue nothing.
 * Every call in a process shares the one array of a device, and each call
 * overwrites the part it reads, so nothing needs clearing; but calls that
 * overlap on the GPU (on other streams, from other threads) race on it and
 * must be serialised by the caller.  Another process has an array of its own.  Pointers are device pointers, 16-byte
 * aligned.  Returns an MLPBLK_* code.
 */
int mlpblk_rmsnorm_backward_noalloc(const mlpblk_desc *desc, const void *x, const float *dn,
                                    const void *dy, const void *gamma, const float *rstd,
                                    void *dx, float *dgamma, void *stream);

/*
 * Kernel timing hook for profiling harnesses (CUDA events, no profiler needed).
 * Kinds reported for each kernel launch the library makes:
 */
#define MLPBLK_KERNEL_FOLD_GAMMA      1  /* statistics pass: rstd, W1g = W1 * gamma;
                                            mlpblk_fold_weights: W1g alone           */
#define MLPBLK_KERNEL_GEMM_FWD_W1     2  /* h, a = RMSNorm(x) . W1^T, relu^2         */
#define MLPBLK_KERNEL_GEMM_FWD_W2     3  /* y = x + a . W2^T                          */
#define MLPBLK_KERNEL_GEMM_DGRAD_H    4  /* dh = (dy . W2) * 2 relu(h)                */
#define MLPBLK_KERNEL_GEMM_WGRAD_W2   5  /* dW2 += dy^T . a                           */
#define MLPBLK_KERNEL_GEMM_DGRAD_N    6  /* dn = dh . W1                              */
#define MLPBLK_KERNEL_GEMM_WGRAD_W1   7  /* dW1 += dh^T . n                           */
#define MLPBLK_KERNEL_NORM_BWD        8  /* RMSNorm backward + residual, dgamma parts */
#define MLPBLK_KERNEL_DGAMMA_REDUCE   9  /* dgamma += sum of parts                    */
#define MLPBLK_KERNEL_ZERO_GRADS     10
#define MLPBLK_KERNEL_SCALE_GRADS    11
#define MLPBLK_KERNEL_RSTD           12  /* statistics pass alone: rstd (prefolded)   */
#define MLPBLK_KERNEL_GRAD_NORM      13  /* per-CTA partial sums of g^2               */
#define MLPBLK_KERNEL_CLIP_GRADS     14  /* g *= clip scale (device scalar)           */
#define MLPBLK_KERNEL_ADAMW          15  /* fused AdamW update                        */
#define MLPBLK_KERNEL_GRAD_NORM_FINAL 16 /* partials -> norm and clip scale           */
#define MLPBLK_KERNEL_QUANT_AMAX     17  /* E4M3: per-CTA maxima of |v|               */
#define MLPBLK_KERNEL_QUANT_SCALE    18  /* E4M3: amax -> scale record                */
#define MLPBLK_KERNEL_QUANT_APPLY    19  /* E4M3: v -> codes                          */
#define MLPBLK_KERNEL_NORM_QUANT     20  /* E4M3: rstd and n' = x * rstd              */
#define MLPBLK_KERNEL_MOE_ROUTE      21  /* experts: counts, segments, ranks, row map */
#define MLPBLK_KERNEL_MOE_GATHER     22  /* experts: rows in segment order            */
#define MLPBLK_KERNEL_MOE_COMBINE    23  /* experts: y = x + weighted outputs         */
#define MLPBLK_KERNEL_MOE_DP         24  /* experts: d_routing_weights and p * dy     */
#define MLPBLK_KERNEL_MOE_SCATTER    25  /* reserved (dn's slot sum is in NORM_BWD)   */

/*
 * mlpblk_trace_begin: from now on, launch i of this library records
 * events[2i] on its stream just before the kernel and events[2i+1] just after
 * it, and stores its MLPBLK_KERNEL_* kind in kinds[i], for i < capacity; later
 * launches are not recorded.  events (2*capacity cudaEvent_t handles created by
 * the caller) and kinds (capacity ints, host memory) stay owned by the caller
 * and must outlive the trace.  One trace at a time per process; not
 * thread-safe.  Returns MLPBLK_EINVAL for NULL arrays or capacity < 1.
 * mlpblk_trace_end: stops recording and returns how many launches were
 * recorded (may exceed capacity: the launches beyond it were only counted).
 */
int mlpblk_trace_begin(void **events, int *kinds, int capacity);
int mlpblk_trace_end(void);

/*
 * Failure-detection test hook.  MLPBLK_TEST_FAULT_SKIP_LOADS makes the W1 GEMM
 * of the next bf16 mlpblk_forward issue none of its operand loads: its pipeline
 * waits then run out after their bound (about 2 s), the kernel unwinds (TMEM
 * freed, no trap) and MLPBLK_ETIMEOUT is recorded for mlpblk_last_error(); that
 * forward's outputs are not valid, and the context stays usable.  One-shot; not
 * thread-safe.  Returns MLPBLK_EINVAL for an unknown fault.
 */
#define MLPBLK_RMSNORM_STATS_PASS      0
#define MLPBLK_RMSNORM_IN_W1_PROLOGUE  1
/*
 * Where the bf16 forward computes the RMSNorm statistic rstd[t] ("Setup: The
 * Shared Transformer Shell": the norm feeds the W1 projection):
 *   MLPBLK_RMSNORM_STATS_PASS (default): one HBM pass over x ahead of the W1
 *     GEMM computes rstd and, in the same launch, W1*gamma; the GEMM applies
 *     rstd in its epilogue and runs 256 x 256 pair tiles.
 *   MLPBLK_RMSNORM_IN_W1_PROLOGUE: four extra warps of the W1 GEMM sum x^2 per
 *     row from the x tiles already staged in shared memory for the MMAs (no
 *     extra pass over x; W1*gamma still takes one pass over W1).  Whole-tile
 *     schedule only (every tile needs all of K for its rows' sums).
 * Same results up to float32 summation order.  Process-wide; applies to later
 * mlpblk_forward calls (the recompute variant always uses the statistics
 * pass).  Returns MLPBLK_EINVAL for an unknown mode.
 */
int mlpblk_set_rmsnorm_mode(int mode);

#define MLPBLK_TEST_FAULT_NONE        0
#define MLPBLK_TEST_FAULT_SKIP_LOADS  1
int mlpblk_set_test_fault(int fault);

/* The CUDA runtime's message for the most recent failing CUDA call made inside
 * the library (behind an MLPBLK_ECUDA), or "no CUDA error recorded". */
const char *mlpblk_cuda_error_string(void);

/* Static, NUL-terminated description of an MLPBLK_* code. */
const char *mlpblk_strerror(int code);

/* ABI version (major * 100 + minor). */
int mlpblk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLPBLK_H */
