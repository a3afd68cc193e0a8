"""The C-ABI library on the host (no GPU needed): it builds, loads, exports every
entry point include/mlpblk.h declares, and rejects bad arguments before it
enqueues anything."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mb():
    import __graft_entry__
    __graft_entry__.build()
    import mlp_block_backprop_gb300
    return mlp_block_backprop_gb300


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mlpblk_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(mb):
    declared = _declared()
    assert {"mlpblk_forward", "mlpblk_backward", "mlpblk_zero_grads"} <= declared
    lib = ctypes.CDLL(mb.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(mb.EXPORTED) <= declared


def _declared_parameters():
    """{function: number of parameters} of every declaration in include/*.h."""
    import glob
    out = {}
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for name, params in re.findall(r"\b(mlpblk_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
            ps = [q.strip() for q in params.split(",") if q.strip()]
            out[name] = 0 if ps == ["void"] else len(ps)
    return out


def test_binding_declares_every_parameter(mb):
    """The binding's ctypes argtypes list every parameter the header declares, so
    no argument (the stream last of all) falls to ctypes' default int conversion."""
    decl = _declared_parameters()
    assert len(decl) >= 30
    wrong = {n: (k, len(getattr(mb.lib, n).argtypes or []))
             for n, k in decl.items() if len(getattr(mb.lib, n).argtypes or []) != k}
    assert not wrong, f"header parameters vs argtypes: {wrong}"


def test_version_and_strerror(mb):
    assert mb.mlpblk_version() >= 100
    for code in range(0, 7):
        assert mb.strerror(code)
    assert "unknown" in mb.strerror(99)


def test_workspace_size(mb):
    d = mb.make_desc(8192, 768, 3072)
    ws = mb.mlpblk_workspace_size(d)
    # backward scratch: dh (bf16 T x F), dn (fp32 T x d), dgamma partials
    assert ws >= 8192 * 3072 * 2 + 8192 * 768 * 4
    assert ws % 256 == 0
    assert mb.mlpblk_workspace_size(mb.make_desc(8, 100, 64)) == 0       # d not a multiple of 8
    assert mb.mlpblk_workspace_size(mb.make_desc(-1, 64, 64)) == 0
    assert mb.mlpblk_workspace_size(mb.make_desc(8, 64, 64, dtype=7)) == 0
    assert mb.mlpblk_workspace_size(mb.make_desc(8, 64, 64, eps=float("nan"))) == 0
    assert mb.mlpblk_workspace_size(mb.make_desc(8, 8192, 64)) == 0      # beyond the norm kernel's width
    assert mb.mlpblk_workspace_size(mb.make_desc(1 << 20, 4096, 4096)) == 0  # index range


def _fwd(mb, desc, ptrs, ws_bytes=1 << 40):
    return mb.lib.mlpblk_forward(ctypes.byref(desc), *ptrs, ws_bytes, None)


def test_forward_argument_errors_need_no_device(mb):
    good = [0x10000 * (i + 1) for i in range(9)]  # aligned, never dereferenced
    d = mb.make_desc(64, 128, 256)
    bad_null = list(good)
    bad_null[0] = None
    assert _fwd(mb, d, bad_null) == mb.MLPBLK_EINVAL
    bad_align = list(good)
    bad_align[3] += 8
    assert _fwd(mb, d, bad_align) == mb.MLPBLK_EINVAL
    alias = list(good)
    alias[4] = alias[0]  # y == x
    assert _fwd(mb, d, alias) == mb.MLPBLK_EINVAL
    assert _fwd(mb, d, good, ws_bytes=16) == mb.MLPBLK_EWORKSPACE
    assert _fwd(mb, mb.make_desc(64, 100, 256), good) == mb.MLPBLK_ENOTSUP
    assert _fwd(mb, mb.make_desc(64, 128, 256, dtype=3), good) == mb.MLPBLK_ENOTSUP
    assert _fwd(mb, mb.make_desc(64, 128, 256, eps=-1.0), good) == mb.MLPBLK_EINVAL
    assert mb.lib.mlpblk_forward(None, *good, 1 << 40, None) == mb.MLPBLK_EINVAL
    # an empty microbatch is valid and does nothing, whatever the pointers
    assert _fwd(mb, mb.make_desc(0, 128, 256), [None] * 9) == mb.MLPBLK_OK


def test_backward_and_grad_argument_errors_need_no_device(mb):
    good = [0x10000 * (i + 1) for i in range(13)]
    d = mb.make_desc(64, 128, 256)
    args = list(good)
    args[9] = args[9] + 4  # dgamma misaligned
    assert mb.lib.mlpblk_backward(ctypes.byref(d), *args, 1 << 40, None) == mb.MLPBLK_EINVAL
    args = list(good)
    args[8] = args[0]  # dx == dy
    assert mb.lib.mlpblk_backward(ctypes.byref(d), *args, 1 << 40, None) == mb.MLPBLK_EINVAL
    assert mb.lib.mlpblk_backward(ctypes.byref(d), *good, 0, None) == mb.MLPBLK_EWORKSPACE
    assert mb.lib.mlpblk_backward(ctypes.byref(mb.make_desc(0, 128, 256)), *([None] * 13), 0,
                                  None) == mb.MLPBLK_OK
    assert mb.lib.mlpblk_zero_grads(ctypes.byref(d), None, 0x10000, 0x20000, None) == mb.MLPBLK_EINVAL
    assert mb.lib.mlpblk_scale_grads(ctypes.byref(d), 0x10000, 0x20000, 0x30000, float("inf"),
                                     None) == mb.MLPBLK_EINVAL


def test_recompute_argument_errors_need_no_device(mb):
    d = mb.make_desc(64, 128, 256)
    assert mb.lib.mlpblk_workspace_size_recompute(ctypes.byref(d)) >= (
        mb.lib.mlpblk_workspace_size(ctypes.byref(d)) + 2 * 64 * 256 * 2)
    assert mb.lib.mlpblk_workspace_size_recompute(ctypes.byref(mb.make_desc(8, 100, 64))) == 0
    fwd = [0x10000 * (i + 1) for i in range(7)]
    f = lambda args, ws=1 << 40: mb.lib.mlpblk_forward_recompute(ctypes.byref(d), *args, ws, None)
    bad = list(fwd)
    bad[5] = None  # rstd
    assert f(bad) == mb.MLPBLK_EINVAL
    alias = list(fwd)
    alias[4] = alias[0]  # y == x
    assert f(alias) == mb.MLPBLK_EINVAL
    # the saving path's workspace is too small for the recompute variant
    assert f(fwd, mb.lib.mlpblk_workspace_size(ctypes.byref(d))) == mb.MLPBLK_EWORKSPACE
    bwd = [0x10000 * (i + 1) for i in range(11)]
    b = lambda args, ws=1 << 40: mb.lib.mlpblk_backward_recompute(ctypes.byref(d), *args, ws, None)
    bad = list(bwd)
    bad[7] += 4  # dgamma misaligned
    assert b(bad) == mb.MLPBLK_EINVAL
    alias = list(bwd)
    alias[6] = alias[1]  # dx == x
    assert b(alias) == mb.MLPBLK_EINVAL
    assert b(bwd, 16) == mb.MLPBLK_EWORKSPACE
    empty = ctypes.byref(mb.make_desc(0, 128, 256))
    assert mb.lib.mlpblk_backward_recompute(empty, *([None] * 11), 0, None) == mb.MLPBLK_OK


def test_optimizer_argument_errors_need_no_device(mb):
    d = mb.make_desc(1, 128, 256)
    g = [0x10000, 0x20000, 0x30000]
    ws = 1 << 40
    norm = lambda *a: mb.lib.mlpblk_grad_norm(ctypes.byref(d), *a)
    assert norm(*g, 1.0, None, None, 0x40000, ws, None) == mb.MLPBLK_EINVAL        # no output
    assert norm(*g, 0.0, 0x50000, None, 0x40000, ws, None) == mb.MLPBLK_EINVAL     # max_norm 0
    assert norm(*g, float("nan"), 0x50000, None, 0x40000, ws, None) == mb.MLPBLK_EINVAL
    assert norm(g[0] + 4, g[1], g[2], 1.0, 0x50000, None, 0x40000, ws, None) == mb.MLPBLK_EINVAL
    assert norm(*g, 1.0, 0x50002, None, 0x40000, ws, None) == mb.MLPBLK_EINVAL    # misaligned scalar
    assert norm(*g, 1.0, 0x50000, None, 0x40000, 16, None) == mb.MLPBLK_EWORKSPACE
    assert mb.lib.mlpblk_clip_grads(ctypes.byref(d), *g, None, None) == mb.MLPBLK_EINVAL
    p = mb.Param(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 64, 1)
    hp = mb.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.1)
    step = lambda params, n, h, t=1, dt=mb.MLPBLK_BF16: mb.lib.mlpblk_adamw_step(params, n, h, t, dt, None, None)
    arr = (mb.Param * 1)(p)
    assert step(arr, 0, ctypes.byref(hp)) == mb.MLPBLK_EINVAL                      # no tensors
    assert step(arr, 1, ctypes.byref(hp), t=0) == mb.MLPBLK_EINVAL                 # step counts from 1
    assert step(arr, 1, ctypes.byref(hp), dt=9) == mb.MLPBLK_ENOTSUP
    assert step(arr, 1, ctypes.byref(mb.AdamW(1e-3, 1.0, 0.999, 1e-8, 0.0))) == mb.MLPBLK_EINVAL
    assert step(arr, 1, ctypes.byref(mb.AdamW(-1e-3, 0.9, 0.999, 1e-8, 0.0))) == mb.MLPBLK_EINVAL
    bad = (mb.Param * 1)(mb.Param(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 66, 1))   # n % 4
    assert step(bad, 1, ctypes.byref(hp)) == mb.MLPBLK_EINVAL
    bad = (mb.Param * 1)(mb.Param(0x10008, 0x20000, 0x30000, 0x40000, 0x50000, 64, 1))   # master align
    assert step(bad, 1, ctypes.byref(hp)) == mb.MLPBLK_EINVAL


def test_fp8_argument_errors_need_no_device(mb):
    d = mb.make_desc(64, 128, 256)
    assert mb.lib.mlpblk_workspace_size_fp8(ctypes.byref(d)) > 0
    assert mb.lib.mlpblk_workspace_size_fp8(ctypes.byref(mb.make_desc(64, 136, 256))) == 0   # d % 16
    assert mb.lib.mlpblk_workspace_size_fp8(ctypes.byref(mb.make_desc(64, 128, 256, dtype=mb.MLPBLK_FP32))) == 0
    fwd = [0x10000 * (i + 1) for i in range(11)]   # x ... scales, workspace
    f = lambda args, ws=1 << 40, dd=d: mb.lib.mlpblk_forward_fp8(ctypes.byref(dd), *args, ws, None)
    assert f(fwd, dd=mb.make_desc(64, 136, 256)) == mb.MLPBLK_ENOTSUP
    bad = list(fwd)
    bad[9] += 4   # scales misaligned
    assert f(bad) == mb.MLPBLK_EINVAL
    assert f(fwd, 16) == mb.MLPBLK_EWORKSPACE
    bwd = [0x10000 * (i + 1) for i in range(15)]   # dy ... dw2, workspace
    b = lambda args, ws=1 << 40: mb.lib.mlpblk_backward_fp8(ctypes.byref(d), *args, ws, None)
    alias = list(bwd)
    alias[10] = alias[0]   # dx == dy
    assert b(alias) == mb.MLPBLK_EINVAL
    assert b(bwd, 16) == mb.MLPBLK_EWORKSPACE


def test_fp8_prequant_argument_errors_need_no_device(mb):
    d = mb.make_desc(64, 128, 256)
    wq_size = mb.lib.mlpblk_fp8_weights_size(ctypes.byref(d))
    assert wq_size >= 3 * 128 * 256 + 48            # three code tensors and three scale records
    assert mb.lib.mlpblk_fp8_weights_size(ctypes.byref(mb.make_desc(64, 136, 256))) == 0
    q = lambda wq_bytes, ws=1 << 40, g=0x10000: mb.lib.mlpblk_fp8_quantize_weights(
        ctypes.byref(d), g, 0x20000, 0x30000, 0x40000, wq_bytes, 0x50000, ws, None)
    assert q(wq_size - 1) == mb.MLPBLK_EWORKSPACE
    assert q(wq_size, ws=16) == mb.MLPBLK_EWORKSPACE
    assert q(wq_size, g=0x10004) == mb.MLPBLK_EINVAL  # gamma misaligned
    fwd = [0x10000 * (i + 1) for i in range(9)]
    f = lambda args, ws=1 << 40: mb.lib.mlpblk_forward_fp8_prequant(ctypes.byref(d), *args, ws, None)
    alias = list(fwd)
    alias[2] = alias[0]   # y == x
    assert f(alias) == mb.MLPBLK_EINVAL
    assert f(fwd, 16) == mb.MLPBLK_EWORKSPACE
    bwd = [0x10000 * (i + 1) for i in range(14)]   # dy ... dw2, workspace
    b = lambda args, ws=1 << 40: mb.lib.mlpblk_backward_fp8_prequant(ctypes.byref(d), *args, ws, None)
    bad = list(bwd)
    bad[3] += 8   # wq misaligned
    assert b(bad) == mb.MLPBLK_EINVAL
    assert b(bwd, 16) == mb.MLPBLK_EWORKSPACE
    empty = mb.make_desc(0, 128, 256)
    assert mb.lib.mlpblk_forward_fp8_prequant(ctypes.byref(empty), *fwd, 1 << 40, None) == mb.MLPBLK_OK


def test_moe_argument_errors_need_no_device(mb):
    d = mb.make_moe_desc(64, 128, 256, 4, 2)
    assert mb.lib.mlpblk_moe_saved_size(ctypes.byref(d)) > 0
    assert mb.lib.mlpblk_moe_workspace_size(ctypes.byref(d)) > 0
    for bad in (mb.make_moe_desc(64, 128, 256, 4, 5), mb.make_moe_desc(64, 128, 256, 0, 1),
                mb.make_moe_desc(64, 100, 256, 4, 2)):
        assert mb.lib.mlpblk_moe_saved_size(ctypes.byref(bad)) == 0
    args = [0x10000 * (i + 1) for i in range(8)]
    f = lambda a, sv=1 << 40, ws=1 << 40: mb.lib.mlpblk_moe_forward(ctypes.byref(d), *a, sv, 0x900000, ws, None)
    bad = list(args)
    bad[4] += 4   # expert ids misaligned
    assert f(bad) == mb.MLPBLK_EINVAL
    alias = list(args)
    alias[6] = alias[0]   # y == x
    assert f(alias) == mb.MLPBLK_EINVAL
    assert f(args, sv=16) == mb.MLPBLK_EWORKSPACE
    bargs = [0x10000 * (i + 1) for i in range(13)]
    b = lambda a, ws=1 << 40: mb.lib.mlpblk_moe_backward(ctypes.byref(d), *a, ws, None)
    assert b(bargs, 16) == mb.MLPBLK_EWORKSPACE
    alias = list(bargs)
    alias[7] = alias[0]   # dx == dy
    assert b(alias) == mb.MLPBLK_EINVAL


def test_overwrite_argument_errors_need_no_device(mb):
    """The forms that set the gradients check their arguments as the adding forms
    do, before any device call; with no tokens they only check the gradient
    buffers (they still zero them, which needs a device)."""
    d = mb.make_desc(64, 128, 256)
    empty = mb.make_desc(0, 128, 256)
    good = [0x10000 * (i + 1) for i in range(13)]
    b = lambda a, ws=1 << 40, dd=d: mb.lib.mlpblk_backward_overwrite(ctypes.byref(dd), *a, ws, None)
    bad = list(good)
    bad[11] += 4   # dw2 misaligned
    assert b(bad) == mb.MLPBLK_EINVAL
    assert b(bad, dd=empty) == mb.MLPBLK_EINVAL
    alias = list(good)
    alias[8] = alias[1]   # dx == x
    assert b(alias) == mb.MLPBLK_EINVAL
    assert b(good, 0) == mb.MLPBLK_EWORKSPACE
    f8 = [0x10000 * (i + 1) for i in range(15)]
    b8 = lambda a, ws=1 << 40, dd=d: mb.lib.mlpblk_backward_fp8_overwrite(ctypes.byref(dd), *a, ws, None)
    bad = list(f8)
    bad[13] += 8   # dw2 misaligned
    assert b8(bad) == mb.MLPBLK_EINVAL
    assert b8(bad, dd=empty) == mb.MLPBLK_EINVAL
    assert b8(f8, 16) == mb.MLPBLK_EWORKSPACE
    assert b8(f8, dd=mb.make_desc(64, 136, 256)) == mb.MLPBLK_ENOTSUP
    q8 = [0x10000 * (i + 1) for i in range(14)]
    bq = lambda a, ws=1 << 40, dd=d: mb.lib.mlpblk_backward_fp8_prequant_overwrite(ctypes.byref(dd), *a, ws, None)
    bad = list(q8)
    bad[10] += 4   # dgamma misaligned
    assert bq(bad) == mb.MLPBLK_EINVAL
    assert bq(bad, dd=empty) == mb.MLPBLK_EINVAL
    alias = list(q8)
    alias[9] = alias[0]   # dx == dy
    assert bq(alias) == mb.MLPBLK_EINVAL
    assert bq(q8, 16) == mb.MLPBLK_EWORKSPACE
    md = mb.make_moe_desc(64, 128, 256, 4, 2)
    margs = [0x10000 * (i + 1) for i in range(13)]
    bm = lambda a, ws=1 << 40, dd=md: mb.lib.mlpblk_moe_backward_overwrite(ctypes.byref(dd), *a, ws, None)
    assert bm(margs, 16) == mb.MLPBLK_EWORKSPACE
    bad = list(margs)
    bad[10] += 4   # dw1s misaligned
    assert bm(bad) == mb.MLPBLK_EINVAL
    assert bm(bad, dd=mb.make_moe_desc(0, 128, 256, 4, 2)) == mb.MLPBLK_EINVAL


def test_grad_buffers_are_float32_by_contract():
    """The gradient accumulators are declared float32: the bf16 loss of a small
    contribution next to a large running sum is why."""
    src = open(os.path.join(ROOT, "include", "mlpblk.h")).read()
    assert re.search(r"float\s*\*dgamma,\s*float\s*\*dw1,\s*float\s*\*dw2", src)
