"""Python binding of libmlpblk.so, the GB300 forward/backward of the pre-norm
residual ReLU² MLP block (C ABI in include/mlpblk.h).

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (device memory and streams are the
only things torch provides); the functions keep the C names and raise
``MlpBlkError`` on a non-zero status.  Importing this package fails loudly when
the library has not been built: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmlpblk.so")

MLPBLK_OK = 0
MLPBLK_EINVAL = 1
MLPBLK_ENOTSUP = 2
MLPBLK_EWORKSPACE = 3
MLPBLK_ECUDA = 4
MLPBLK_ETIMEOUT = 5
MLPBLK_ENODEV = 6
MLPBLK_BF16 = 1
MLPBLK_FP32 = 2

EXPORTED = ("mlpblk_workspace_size", "mlpblk_forward", "mlpblk_backward", "mlpblk_zero_grads",
            "mlpblk_scale_grads", "mlpblk_last_error", "mlpblk_strerror", "mlpblk_version",
            "mlpblk_trace_begin", "mlpblk_trace_end", "mlpblk_cuda_error_string",
            "mlpblk_rmsnorm_backward_noalloc", "mlpblk_set_test_fault",
            "mlpblk_workspace_size_recompute", "mlpblk_forward_recompute", "mlpblk_backward_recompute",
            "mlpblk_grad_norm", "mlpblk_clip_grads", "mlpblk_adamw_step", "mlpblk_set_rmsnorm_mode",
            "mlpblk_workspace_size_fp8", "mlpblk_forward_fp8", "mlpblk_backward_fp8",
            "mlpblk_fp8_weights_size", "mlpblk_fp8_quantize_weights", "mlpblk_forward_fp8_prequant",
            "mlpblk_backward_fp8_prequant",
            "mlpblk_moe_saved_size", "mlpblk_moe_workspace_size", "mlpblk_moe_forward", "mlpblk_moe_backward",
            "mlpblk_fold_weights", "mlpblk_forward_prefolded", "mlpblk_backward_overwrite",
            "mlpblk_moe_backward_overwrite", "mlpblk_backward_fp8_overwrite",
            "mlpblk_backward_fp8_prequant_overwrite")
MLPBLK_RMSNORM_STATS_PASS = 0
MLPBLK_RMSNORM_IN_W1_PROLOGUE = 1
MLPBLK_TEST_FAULT_NONE = 0
MLPBLK_TEST_FAULT_SKIP_LOADS = 1

KERNEL_NAMES = {1: "fold_gamma", 2: "gemm_fwd_w1", 3: "gemm_fwd_w2", 4: "gemm_dgrad_h",
                5: "gemm_wgrad_w2", 6: "gemm_dgrad_n", 7: "gemm_wgrad_w1", 8: "norm_bwd",
                9: "dgamma_reduce", 10: "zero_grads", 11: "scale_grads", 12: "rstd",
                13: "grad_norm", 14: "clip_grads", 15: "adamw", 16: "grad_norm_final",
                17: "quant_amax", 18: "quant_scale", 19: "quant_apply", 20: "norm_quant",
                21: "moe_route", 22: "moe_gather", 23: "moe_combine", 24: "moe_dp", 25: "moe_scatter"}


class MlpBlkError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        extra = ""
        if code == MLPBLK_ECUDA:
            extra = "; CUDA: " + lib.mlpblk_cuda_error_string().decode()
        super().__init__(f"{where}: status {code} ({strerror(code)}{extra})")


class Desc(ctypes.Structure):
    """mlpblk_desc: shape of one microbatch through one block."""
    _fields_ = [("tokens", ctypes.c_int64), ("d_model", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int32)]


class MoeDesc(ctypes.Structure):
    """mlpblk_moe_desc: the dense descriptor plus the expert count and top-k."""
    _fields_ = [("base", Desc), ("experts", ctypes.c_int32), ("top_k", ctypes.c_int32)]


class Param(ctypes.Structure):
    """mlpblk_param: one tensor of an AdamW update."""
    _fields_ = [("master", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("m", ctypes.c_void_p), ("v", ctypes.c_void_p), ("n", ctypes.c_int64), ("decay", ctypes.c_int32)]


class AdamW(ctypes.Structure):
    """mlpblk_adamw: AdamW hyper-parameters."""
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: run mlp_block_backprop_gb300.build.build_library() "
                          "(or __graft_entry__.build()) first; there is no non-CUDA fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    pd = ctypes.POINTER(Desc)
    lib.mlpblk_workspace_size.argtypes = [pd]
    lib.mlpblk_workspace_size.restype = sz
    lib.mlpblk_forward.argtypes = [pd] + [vp] * 9 + [sz, vp]
    lib.mlpblk_forward.restype = i32
    lib.mlpblk_backward.argtypes = [pd] + [vp] * 13 + [sz, vp]
    lib.mlpblk_fold_weights.argtypes = [pd, vp, vp, vp, vp]
    lib.mlpblk_fold_weights.restype = i32
    lib.mlpblk_forward_prefolded.argtypes = [pd] + [vp] * 8 + [sz, vp]
    lib.mlpblk_forward_prefolded.restype = i32
    lib.mlpblk_backward.restype = i32
    lib.mlpblk_backward_overwrite.argtypes = lib.mlpblk_backward.argtypes
    lib.mlpblk_backward_overwrite.restype = i32
    lib.mlpblk_workspace_size_recompute.argtypes = [pd]
    lib.mlpblk_workspace_size_recompute.restype = sz
    lib.mlpblk_forward_recompute.argtypes = [pd] + [vp] * 7 + [sz, vp]
    lib.mlpblk_forward_recompute.restype = i32
    lib.mlpblk_backward_recompute.argtypes = [pd] + [vp] * 11 + [sz, vp]
    lib.mlpblk_backward_recompute.restype = i32
    lib.mlpblk_grad_norm.argtypes = [pd, vp, vp, vp, f32, vp, vp, vp, sz, vp]
    lib.mlpblk_grad_norm.restype = i32
    lib.mlpblk_clip_grads.argtypes = [pd, vp, vp, vp, vp, vp]
    lib.mlpblk_clip_grads.restype = i32
    lib.mlpblk_adamw_step.argtypes = [ctypes.POINTER(Param), i32, ctypes.POINTER(AdamW), ctypes.c_int64, i32, vp, vp]
    lib.mlpblk_adamw_step.restype = i32
    lib.mlpblk_workspace_size_fp8.argtypes = [pd]
    lib.mlpblk_workspace_size_fp8.restype = sz
    lib.mlpblk_forward_fp8.argtypes = [pd] + [vp] * 11 + [sz, vp]
    lib.mlpblk_forward_fp8.restype = i32
    lib.mlpblk_backward_fp8.argtypes = [pd] + [vp] * 15 + [sz, vp]
    lib.mlpblk_backward_fp8.restype = i32
    lib.mlpblk_fp8_weights_size.argtypes = [pd]
    lib.mlpblk_fp8_weights_size.restype = sz
    lib.mlpblk_fp8_quantize_weights.argtypes = [pd, vp, vp, vp, vp, sz, vp, sz, vp]
    lib.mlpblk_fp8_quantize_weights.restype = i32
    lib.mlpblk_forward_fp8_prequant.argtypes = [pd] + [vp] * 9 + [sz, vp]
    lib.mlpblk_forward_fp8_prequant.restype = i32
    lib.mlpblk_backward_fp8_prequant.argtypes = [pd] + [vp] * 14 + [sz, vp]
    lib.mlpblk_backward_fp8_prequant.restype = i32
    lib.mlpblk_backward_fp8_overwrite.argtypes = lib.mlpblk_backward_fp8.argtypes
    lib.mlpblk_backward_fp8_overwrite.restype = i32
    lib.mlpblk_backward_fp8_prequant_overwrite.argtypes = lib.mlpblk_backward_fp8_prequant.argtypes
    lib.mlpblk_backward_fp8_prequant_overwrite.restype = i32
    pm = ctypes.POINTER(MoeDesc)
    lib.mlpblk_moe_saved_size.argtypes = [pm]
    lib.mlpblk_moe_saved_size.restype = sz
    lib.mlpblk_moe_workspace_size.argtypes = [pm]
    lib.mlpblk_moe_workspace_size.restype = sz
    lib.mlpblk_moe_forward.argtypes = [pm] + [vp] * 8 + [sz, vp, sz, vp]
    lib.mlpblk_moe_forward.restype = i32
    lib.mlpblk_moe_backward.argtypes = [pm] + [vp] * 13 + [sz, vp]
    lib.mlpblk_moe_backward.restype = i32
    lib.mlpblk_moe_backward_overwrite.argtypes = lib.mlpblk_moe_backward.argtypes
    lib.mlpblk_moe_backward_overwrite.restype = i32
    lib.mlpblk_zero_grads.argtypes = [pd, vp, vp, vp, vp]
    lib.mlpblk_zero_grads.restype = i32
    lib.mlpblk_scale_grads.argtypes = [pd, vp, vp, vp, f32, vp]
    lib.mlpblk_scale_grads.restype = i32
    lib.mlpblk_last_error.argtypes = []
    lib.mlpblk_last_error.restype = i32
    lib.mlpblk_strerror.argtypes = [i32]
    lib.mlpblk_strerror.restype = ctypes.c_char_p
    lib.mlpblk_version.argtypes = []
    lib.mlpblk_version.restype = i32
    lib.mlpblk_trace_begin.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int), i32]
    lib.mlpblk_trace_begin.restype = i32
    lib.mlpblk_rmsnorm_backward_noalloc.argtypes = [pd] + [vp] * 8
    lib.mlpblk_rmsnorm_backward_noalloc.restype = i32
    lib.mlpblk_set_rmsnorm_mode.argtypes = [i32]
    lib.mlpblk_set_rmsnorm_mode.restype = i32
    lib.mlpblk_set_test_fault.argtypes = [i32]
    lib.mlpblk_set_test_fault.restype = i32
    lib.mlpblk_cuda_error_string.argtypes = []
    lib.mlpblk_cuda_error_string.restype = ctypes.c_char_p
    lib.mlpblk_trace_end.argtypes = []
    lib.mlpblk_trace_end.restype = i32
    return lib


lib = _load()


def strerror(code: int) -> str:
    return lib.mlpblk_strerror(int(code)).decode()


def make_desc(tokens: int, d_model: int, ffn: int, eps: float = 1e-6, dtype: int = MLPBLK_BF16) -> Desc:
    return Desc(int(tokens), int(d_model), int(ffn), float(eps), int(dtype))


def _ptr(t):
    """Device address of a tensor, an int address, or None (NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc, where):
    if rc != MLPBLK_OK:
        raise MlpBlkError(rc, where)


def mlpblk_workspace_size(desc: Desc) -> int:
    return int(lib.mlpblk_workspace_size(ctypes.byref(desc)))


def mlpblk_forward(desc, x, gamma, w1, w2, y, h_saved, a_saved, rstd_saved, workspace,
                   workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib.mlpblk_forward(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(w1), _ptr(w2), _ptr(y),
                            _ptr(h_saved), _ptr(a_saved), _ptr(rstd_saved), _ptr(workspace),
                            nbytes, _stream(stream))
    _check(rc, "mlpblk_forward")


def mlpblk_fold_weights(desc, gamma, w1, w1g, stream=None):
    _check(lib.mlpblk_fold_weights(ctypes.byref(desc), _ptr(gamma), _ptr(w1), _ptr(w1g), _stream(stream)),
           "mlpblk_fold_weights")


def mlpblk_forward_prefolded(desc, x, w1g, w2, y, h_saved, a_saved, rstd_saved, workspace,
                             workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib.mlpblk_forward_prefolded(ctypes.byref(desc), _ptr(x), _ptr(w1g), _ptr(w2), _ptr(y),
                                      _ptr(h_saved), _ptr(a_saved), _ptr(rstd_saved), _ptr(workspace),
                                      nbytes, _stream(stream))
    _check(rc, "mlpblk_forward_prefolded")


def mlpblk_backward(desc, dy, x, gamma, w1, w2, h_saved, a_saved, rstd_saved, dx, dgamma, dw1, dw2,
                    workspace, workspace_bytes=None, stream=None, overwrite=False):
    """overwrite=True calls mlpblk_backward_overwrite (gradients written, not added into)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    fn = lib.mlpblk_backward_overwrite if overwrite else lib.mlpblk_backward
    rc = fn(ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(gamma), _ptr(w1), _ptr(w2),
            _ptr(h_saved), _ptr(a_saved), _ptr(rstd_saved), _ptr(dx), _ptr(dgamma),
            _ptr(dw1), _ptr(dw2), _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "mlpblk_backward_overwrite" if overwrite else "mlpblk_backward")


def mlpblk_workspace_size_recompute(desc: Desc) -> int:
    return int(lib.mlpblk_workspace_size_recompute(ctypes.byref(desc)))


def mlpblk_forward_recompute(desc, x, gamma, w1, w2, y, rstd_saved, workspace, workspace_bytes=None,
                             stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib.mlpblk_forward_recompute(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(w1), _ptr(w2),
                                      _ptr(y), _ptr(rstd_saved), _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "mlpblk_forward_recompute")


def mlpblk_backward_recompute(desc, dy, x, gamma, w1, w2, rstd_saved, dx, dgamma, dw1, dw2, workspace,
                              workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib.mlpblk_backward_recompute(ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(gamma), _ptr(w1),
                                       _ptr(w2), _ptr(rstd_saved), _ptr(dx), _ptr(dgamma), _ptr(dw1),
                                       _ptr(dw2), _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "mlpblk_backward_recompute")


def mlpblk_grad_norm(desc, dgamma, dw1, dw2, max_norm, norm_out, clip_scale_out, workspace,
                     workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib.mlpblk_grad_norm(ctypes.byref(desc), _ptr(dgamma), _ptr(dw1), _ptr(dw2), float(max_norm),
                              _ptr(norm_out), _ptr(clip_scale_out), _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "mlpblk_grad_norm")


def mlpblk_clip_grads(desc, dgamma, dw1, dw2, clip_scale, stream=None):
    rc = lib.mlpblk_clip_grads(ctypes.byref(desc), _ptr(dgamma), _ptr(dw1), _ptr(dw2), _ptr(clip_scale),
                               _stream(stream))
    _check(rc, "mlpblk_clip_grads")


def mlpblk_adamw_step(params, hp, step, dtype, grad_scale=None, stream=None):
    """params: sequence of (master, weight, grad, m, v, decay) tensors/flags; hp: AdamW."""
    arr = (Param * len(params))()
    for i, (master, weight, grad, m, v, decay) in enumerate(params):
        arr[i] = Param(_ptr(master), _ptr(weight), _ptr(grad), _ptr(m), _ptr(v), master.numel(), int(decay))
    rc = lib.mlpblk_adamw_step(arr, len(params), ctypes.byref(hp), int(step), int(dtype), _ptr(grad_scale),
                               _stream(stream))
    _check(rc, "mlpblk_adamw_step")


def mlpblk_workspace_size_fp8(desc: Desc) -> int:
    return int(lib.mlpblk_workspace_size_fp8(ctypes.byref(desc)))


def mlpblk_forward_fp8(desc, x, gamma, w1, w2, y, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved,
                       workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    rc = lib.mlpblk_forward_fp8(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(w1), _ptr(w2), _ptr(y),
                                _ptr(h_saved), _ptr(a8_saved), _ptr(n8_saved), _ptr(rstd_saved),
                                _ptr(scales_saved), _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "mlpblk_forward_fp8")


def mlpblk_backward_fp8(desc, dy, x, gamma, w1, w2, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved,
                        dx, dgamma, dw1, dw2, workspace, workspace_bytes=None, stream=None, overwrite=False):
    """overwrite=True calls mlpblk_backward_fp8_overwrite (gradients set, not added into)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    fn = lib.mlpblk_backward_fp8_overwrite if overwrite else lib.mlpblk_backward_fp8
    rc = fn(ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(gamma), _ptr(w1), _ptr(w2),
            _ptr(h_saved), _ptr(a8_saved), _ptr(n8_saved), _ptr(rstd_saved),
            _ptr(scales_saved), _ptr(dx), _ptr(dgamma), _ptr(dw1), _ptr(dw2),
            _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "mlpblk_backward_fp8_overwrite" if overwrite else "mlpblk_backward_fp8")


def mlpblk_fp8_weights_size(desc: Desc) -> int:
    return int(lib.mlpblk_fp8_weights_size(ctypes.byref(desc)))


def mlpblk_fp8_quantize_weights(desc, gamma, w1, w2, wq, workspace, stream=None):
    rc = lib.mlpblk_fp8_quantize_weights(ctypes.byref(desc), _ptr(gamma), _ptr(w1), _ptr(w2), _ptr(wq),
                                         wq.numel() * wq.element_size(), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mlpblk_fp8_quantize_weights")


def mlpblk_forward_fp8_prequant(desc, x, wq, y, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved,
                                workspace, stream=None):
    rc = lib.mlpblk_forward_fp8_prequant(ctypes.byref(desc), _ptr(x), _ptr(wq), _ptr(y), _ptr(h_saved),
                                         _ptr(a8_saved), _ptr(n8_saved), _ptr(rstd_saved), _ptr(scales_saved),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream))
    _check(rc, "mlpblk_forward_fp8_prequant")


def mlpblk_backward_fp8_prequant(desc, dy, x, gamma, wq, h_saved, a8_saved, n8_saved, rstd_saved, scales_saved,
                                 dx, dgamma, dw1, dw2, workspace, stream=None, overwrite=False):
    """overwrite=True calls mlpblk_backward_fp8_prequant_overwrite (gradients set, not added into)."""
    fn = lib.mlpblk_backward_fp8_prequant_overwrite if overwrite else lib.mlpblk_backward_fp8_prequant
    rc = fn(ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(gamma), _ptr(wq),
            _ptr(h_saved), _ptr(a8_saved), _ptr(n8_saved), _ptr(rstd_saved),
            _ptr(scales_saved), _ptr(dx), _ptr(dgamma), _ptr(dw1), _ptr(dw2),
            _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream))
    _check(rc, "mlpblk_backward_fp8_prequant_overwrite" if overwrite else "mlpblk_backward_fp8_prequant")


def make_moe_desc(tokens, d_model, ffn, experts, top_k, eps=1e-6) -> MoeDesc:
    return MoeDesc(make_desc(tokens, d_model, ffn, eps, MLPBLK_BF16), int(experts), int(top_k))


def mlpblk_moe_saved_size(desc: MoeDesc) -> int:
    return int(lib.mlpblk_moe_saved_size(ctypes.byref(desc)))


def mlpblk_moe_workspace_size(desc: MoeDesc) -> int:
    return int(lib.mlpblk_moe_workspace_size(ctypes.byref(desc)))


def mlpblk_moe_forward(desc, x, gamma, w1s, w2s, expert_idx, routing_weights, y, saved, workspace, stream=None):
    rc = lib.mlpblk_moe_forward(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(w1s), _ptr(w2s), _ptr(expert_idx),
                                _ptr(routing_weights), _ptr(y), _ptr(saved), saved.numel(), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "mlpblk_moe_forward")


def mlpblk_moe_backward(desc, dy, x, gamma, w1s, w2s, routing_weights, saved, dx, d_routing_weights, dgamma,
                        dw1s, dw2s, workspace, stream=None, overwrite=False):
    """overwrite=True calls mlpblk_moe_backward_overwrite (gradients written, not added into)."""
    fn = lib.mlpblk_moe_backward_overwrite if overwrite else lib.mlpblk_moe_backward
    rc = fn(ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(gamma), _ptr(w1s), _ptr(w2s),
            _ptr(routing_weights), _ptr(saved), _ptr(dx), _ptr(d_routing_weights),
            _ptr(dgamma), _ptr(dw1s), _ptr(dw2s), _ptr(workspace), workspace.numel(),
            _stream(stream))
    _check(rc, "mlpblk_moe_backward_overwrite" if overwrite else "mlpblk_moe_backward")


class MoeBuffers:
    """Device buffers of one routed-expert block (bf16 tensors, fp32 routing weights
    and gradients, int32 expert ids)."""

    def __init__(self, tokens, d_model, ffn, experts, top_k, eps=1e-6, device="cuda"):
        import torch
        self.desc = make_moe_desc(tokens, d_model, ffn, experts, top_k, eps)
        T, d, F, E, k = tokens, d_model, ffn, experts, top_k
        e = dict(device=device)
        bf = torch.bfloat16
        self.gamma = torch.empty(d, dtype=bf, **e)
        self.w1s = torch.empty(E, F, d, dtype=bf, **e)
        self.w2s = torch.empty(E, d, F, dtype=bf, **e)
        self.x = torch.empty(T, d, dtype=bf, **e)
        self.dy = torch.empty(T, d, dtype=bf, **e)
        self.y = torch.empty(T, d, dtype=bf, **e)
        self.dx = torch.empty(T, d, dtype=bf, **e)
        self.idx = torch.empty(T, k, dtype=torch.int32, **e)
        self.p = torch.empty(T, k, dtype=torch.float32, **e)
        self.dp = torch.empty(T, k, dtype=torch.float32, **e)
        self.dgamma = torch.zeros(d, dtype=torch.float32, **e)
        self.dw1s = torch.zeros(E, F, d, dtype=torch.float32, **e)
        self.dw2s = torch.zeros(E, d, F, dtype=torch.float32, **e)
        sv, ws = mlpblk_moe_saved_size(self.desc), mlpblk_moe_workspace_size(self.desc)
        if sv == 0 or ws == 0:
            raise MlpBlkError(MLPBLK_EINVAL, "mlpblk_moe_saved_size")
        self.saved = torch.empty(sv, dtype=torch.uint8, **e)
        self.ws = torch.empty(ws, dtype=torch.uint8, **e)

    def forward(self, stream=None):
        mlpblk_moe_forward(self.desc, self.x, self.gamma, self.w1s, self.w2s, self.idx, self.p, self.y, self.saved,
                           self.ws, stream=stream)

    def backward(self, stream=None, overwrite=False):
        mlpblk_moe_backward(self.desc, self.dy, self.x, self.gamma, self.w1s, self.w2s, self.p, self.saved,
                            self.dx, self.dp, self.dgamma, self.dw1s, self.dw2s, self.ws, stream=stream,
                            overwrite=overwrite)

    def zero_grads(self, stream=None):
        # the experts' gradients as one block's of ffn E*F (same element counts)
        d = self.desc
        flat = make_desc(0, d.base.d_model, d.base.ffn * d.experts)
        mlpblk_zero_grads(flat, self.dgamma, self.dw1s, self.dw2s, stream=stream)


def mlpblk_zero_grads(desc, dgamma, dw1, dw2, stream=None):
    _check(lib.mlpblk_zero_grads(ctypes.byref(desc), _ptr(dgamma), _ptr(dw1), _ptr(dw2),
                                 _stream(stream)), "mlpblk_zero_grads")


def mlpblk_scale_grads(desc, dgamma, dw1, dw2, s, stream=None):
    _check(lib.mlpblk_scale_grads(ctypes.byref(desc), _ptr(dgamma), _ptr(dw1), _ptr(dw2), float(s),
                                  _stream(stream)), "mlpblk_scale_grads")


def mlpblk_rmsnorm_backward_noalloc(desc, x, dn, dy, gamma, rstd, dx, dgamma, stream=None):
    """RMSNorm backward + residual gradient with no workspace argument, for
    callers that cannot allocate device scratch (see include/mlpblk.h)."""
    _check(lib.mlpblk_rmsnorm_backward_noalloc(ctypes.byref(desc), _ptr(x), _ptr(dn), _ptr(dy),
                                               _ptr(gamma), _ptr(rstd), _ptr(dx), _ptr(dgamma),
                                               _stream(stream)), "mlpblk_rmsnorm_backward_noalloc")


def mlpblk_set_rmsnorm_mode(mode: int) -> None:
    _check(lib.mlpblk_set_rmsnorm_mode(int(mode)), "mlpblk_set_rmsnorm_mode")


def mlpblk_set_test_fault(fault: int) -> None:
    _check(lib.mlpblk_set_test_fault(int(fault)), "mlpblk_set_test_fault")


def mlpblk_last_error() -> int:
    return int(lib.mlpblk_last_error())


def mlpblk_version() -> int:
    return int(lib.mlpblk_version())


class KernelTrace:
    """Records CUDA events around every kernel the library launches while active
    (mlpblk_trace_begin/end); durations() then gives (kind name, ms) per launch."""

    def __init__(self, capacity):
        import torch
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:  # torch creates the CUDA event on its first record
            e.record()
        torch.cuda.synchronize()
        if any(not e.cuda_event for e in self.events):
            raise RuntimeError("torch did not create the CUDA events for the kernel trace")
        self._handles = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self._kinds = (ctypes.c_int * capacity)()
        self.count = 0

    def __enter__(self):
        _check(lib.mlpblk_trace_begin(self._handles, self._kinds, self.capacity), "mlpblk_trace_begin")
        return self

    def __exit__(self, *exc):
        self.count = int(lib.mlpblk_trace_end())
        return False

    def durations(self):
        """[(kind name, milliseconds)] of the recorded launches (call after a sync)."""
        n = min(self.count, self.capacity)
        return [(KERNEL_NAMES.get(self._kinds[i], str(self._kinds[i])),
                 self.events[2 * i].elapsed_time(self.events[2 * i + 1])) for i in range(n)]


class BlockBuffers:
    """Device buffers of one block for microbatches of up to `tokens` rows:
    parameters, saved tensors, outputs, fp32 gradient buffers and workspace.
    recompute=True uses the recompute variant (no h and a buffers; a larger
    workspace holds them during each call)."""

    def __init__(self, tokens, d_model, ffn, dtype="bf16", eps=1e-6, device="cuda", recompute=False,
                 fp8=False):
        import torch
        self.torch = torch
        self.dt = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.code = MLPBLK_BF16 if dtype == "bf16" else MLPBLK_FP32
        self.T, self.d, self.F, self.eps = tokens, d_model, ffn, eps
        self.desc = make_desc(tokens, d_model, ffn, eps, self.code)
        e = dict(device=device)
        T, d, F = tokens, d_model, ffn
        self.gamma = torch.empty(d, dtype=self.dt, **e)
        self.w1 = torch.empty(F, d, dtype=self.dt, **e)
        self.w2 = torch.empty(d, F, dtype=self.dt, **e)
        self.x = torch.empty(T, d, dtype=self.dt, **e)
        self.dy = torch.empty(T, d, dtype=self.dt, **e)
        self.y = torch.empty(T, d, dtype=self.dt, **e)
        self.recompute = recompute
        self.fp8 = fp8
        self.h = None if recompute else torch.empty(T, F, dtype=self.dt, **e)
        self.a = None if (recompute or fp8) else torch.empty(T, F, dtype=self.dt, **e)
        if fp8:  # E4M3 codes of a and n' and a's scale record, saved for the backward
            self.a8 = torch.empty(T, F, dtype=torch.uint8, **e)
            self.n8 = torch.empty(T, d, dtype=torch.uint8, **e)
            self.scales = torch.empty(4, dtype=torch.float32, **e)
            # the weights' E4M3 codes, for the pre-quantised calls
            self.wq = torch.empty(mlpblk_fp8_weights_size(self.desc), dtype=torch.uint8, **e)
        self.rstd = torch.empty(T, dtype=torch.float32, **e)
        self.dx = torch.empty(T, d, dtype=self.dt, **e)
        self.dgamma = torch.zeros(d, dtype=torch.float32, **e)
        self.dw1 = torch.zeros(F, d, dtype=torch.float32, **e)
        self.dw2 = torch.zeros(d, F, dtype=torch.float32, **e)
        ws = (mlpblk_workspace_size_fp8 if fp8 else
              mlpblk_workspace_size_recompute if recompute else mlpblk_workspace_size)(self.desc)
        if ws == 0:
            raise MlpBlkError(MLPBLK_EINVAL, "mlpblk_workspace_size")
        self.ws = torch.empty(ws, dtype=torch.uint8, **e)

    def forward(self, stream=None):
        if self.fp8:
            mlpblk_forward_fp8(self.desc, self.x, self.gamma, self.w1, self.w2, self.y, self.h, self.a8, self.n8,
                               self.rstd, self.scales, self.ws, stream=stream)
            return
        if self.recompute:
            mlpblk_forward_recompute(self.desc, self.x, self.gamma, self.w1, self.w2, self.y, self.rstd,
                                     self.ws, stream=stream)
            return
        mlpblk_forward(self.desc, self.x, self.gamma, self.w1, self.w2, self.y, self.h, self.a,
                       self.rstd, self.ws, stream=stream)

    def fold_weights(self, stream=None):
        """W1 * gamma into self.w1g (allocated on first use), for forward_prefolded."""
        if getattr(self, "w1g", None) is None:
            self.w1g = self.torch.empty_like(self.w1)
        mlpblk_fold_weights(self.desc, self.gamma, self.w1, self.w1g, stream=stream)

    def forward_prefolded(self, stream=None):
        mlpblk_forward_prefolded(self.desc, self.x, self.w1g, self.w2, self.y, self.h, self.a, self.rstd,
                                 self.ws, stream=stream)

    def backward(self, stream=None, overwrite=False):
        """overwrite: set the gradients instead of adding into them (the saving
        and FP8 variants; the recompute variant only adds)."""
        if overwrite and self.recompute:
            raise MlpBlkError(MLPBLK_EINVAL, "overwrite is not offered by the recompute variant")
        if self.fp8:
            mlpblk_backward_fp8(self.desc, self.dy, self.x, self.gamma, self.w1, self.w2, self.h, self.a8,
                                self.n8, self.rstd, self.scales, self.dx, self.dgamma, self.dw1, self.dw2, self.ws,
                                stream=stream, overwrite=overwrite)
            return
        if self.recompute:
            mlpblk_backward_recompute(self.desc, self.dy, self.x, self.gamma, self.w1, self.w2, self.rstd,
                                      self.dx, self.dgamma, self.dw1, self.dw2, self.ws, stream=stream)
            return
        mlpblk_backward(self.desc, self.dy, self.x, self.gamma, self.w1, self.w2, self.h, self.a,
                        self.rstd, self.dx, self.dgamma, self.dw1, self.dw2, self.ws, stream=stream,
                        overwrite=overwrite)

    def zero_grads(self, stream=None):
        mlpblk_zero_grads(self.desc, self.dgamma, self.dw1, self.dw2, stream=stream)

    def scale_grads(self, s, stream=None):
        mlpblk_scale_grads(self.desc, self.dgamma, self.dw1, self.dw2, s, stream=stream)
