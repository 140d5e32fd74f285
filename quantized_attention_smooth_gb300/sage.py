"""Thin ctypes binding of libsage.so (the C ABI declared in include/sage.h).

Argument marshalling only: every step of the quantized attention runs in the
library's CUDA kernels.  torch supplies device memory and the current stream.
There is no fallback: if the library is missing or cannot load, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

F16, BF16 = 0, 1
HND, NHD = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT = range(6)
STATUS_NAMES = ["OK", "INVALID_ARG", "UNSUPPORTED", "WORKSPACE", "CUDA", "DEVICE_TIMEOUT"]

# Every entry point declared in include/sage.h.
EXPORTS = (
    "sage_workspace_bytes", "sage_workspace_bytes_varlen", "sage_quant_prologue",
    "sage_quant_prologue_varlen", "sage_attn_quantized", "sage_attn_fwd",
    "sage_attn_fwd_varlen", "sage_debug_qk_int32", "sage_debug_e4m3",
    "sage_debug_set_fault", "sage_debug_set_prologue_launches", "sage_device_status",
    "sage_last_error",
    "sage_kv_stats_noalloc", "sage_launch_count", "sage_quant_prologue_strided",
    "sage_attn_fwd_strided", "sage_quant_prologue_pv16", "sage_attn_fwd_pv16",
    "sage_workspace_bytes_host", "sage_attn_fwd_host", "sage_attn_fwd_host_pv16",
    "sage_debug_pv_accum", "sage_debug_set_fault_launches", "sage_kv_stats_noalloc_status",
    "sage_debug_tc_rate", "sage_workspace_bytes_varlen_host", "sage_attn_fwd_varlen_host",
    "sage_debug_set_host_fail_chunk",
)


class SageError(RuntimeError):
    def __init__(self, status: int, where: str, reason: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: SAGE_ERR_{name}: {reason}")
        self.status = status


class Quantized(ctypes.Structure):
    """Mirror of sage_quantized (pointers into the workspace)."""
    _fields_ = [
        ("nseg", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
        ("Lq", ctypes.c_int64), ("Lk", ctypes.c_int64), ("D", ctypes.c_int64),
        ("Dp", ctypes.c_int64), ("dtype", ctypes.c_int32), ("varlen", ctypes.c_int32),
        ("total_q", ctypes.c_int64), ("total_k", ctypes.c_int64),
        ("max_q", ctypes.c_int32), ("max_k", ctypes.c_int32),
        ("q_head_rows", ctypes.c_int64), ("k_head_rows", ctypes.c_int64),
        ("q_rows", ctypes.c_int64), ("k_rows", ctypes.c_int64),
        ("v_rows", ctypes.c_int64), ("v_cols", ctypes.c_int64),
        ("cu_q", ctypes.c_void_p), ("cu_k", ctypes.c_void_p),
        ("q16", ctypes.c_void_p), ("k16", ctypes.c_void_p), ("v8", ctypes.c_void_p),
        ("s_q", ctypes.c_void_p), ("s_k", ctypes.c_void_p), ("s_v", ctypes.c_void_p),
        ("k_mean", ctypes.c_void_p), ("stats", ctypes.c_void_p),
        ("status", ctypes.c_void_p), ("v_fp16", ctypes.c_int32),
    ]


def _load():
    path = _build.LIB
    if not _build.up_to_date():
        path = _build.build()
    lib = ctypes.CDLL(path)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    F = ctypes.c_float
    QP = ctypes.POINTER(Quantized)
    sig = {
        "sage_workspace_bytes": ([I64] * 6, SZ),
        "sage_workspace_bytes_host": ([I64] * 7, SZ),
        "sage_attn_fwd_host": ([P, P, P, P, I64, I64, I64, I64, I64, I64, I, I, F, I, I64, P, SZ,
                                P], I),
        "sage_attn_fwd_host_pv16": ([P, P, P, P, I64, I64, I64, I64, I64, I64, I, I, F, I, I64, P,
                                     SZ, P], I),
        "sage_workspace_bytes_varlen": ([I64] * 6, SZ),
        "sage_workspace_bytes_varlen_host": ([I64] * 7, SZ),
        "sage_attn_fwd_varlen_host": ([P, P, P, P, P, P, I64, I64, I64, I, I, I64, I64, I64, I,
                                       F, I, I64, P, SZ, P], I),
        "sage_quant_prologue": ([P, P, P, I, I, I64, I64, I64, I64, I64, I64, P, SZ, QP, P], I),
        "sage_quant_prologue_varlen": ([P, P, P, I, P, P, I64, I64, I64, I, I, I64, I64, I64,
                                        P, SZ, QP, P], I),
        "sage_quant_prologue_strided": ([P, P, P, I, I64, I64, I64, I64, I64, I64, P, P, P, SZ,
                                         QP, P], I),
        "sage_attn_fwd_strided": ([P, P, P, P, I64, I64, I64, I64, I64, I64, P, P, I, I, F, I,
                                   P, SZ, P], I),
        "sage_quant_prologue_pv16": ([P, P, P, I, I, I64, I64, I64, I64, I64, I64, P, SZ, QP,
                                      P], I),
        "sage_attn_fwd_pv16": ([P, P, P, P, I64, I64, I64, I64, I64, I64, I, I, F, I, P, SZ, P],
                               I),
        "sage_attn_quantized": ([QP, P, I, I, F, P], I),
        "sage_attn_fwd": ([P, P, P, P, I64, I64, I64, I64, I64, I64, I, I, F, I, P, SZ, P], I),
        "sage_attn_fwd_varlen": ([P, P, P, P, P, P, I64, I64, I64, I, I, I64, I64, I64, I, F,
                                  I, P, SZ, P], I),
        "sage_debug_qk_int32": ([QP, I64, I64, I64, I64, P, P], I),
        "sage_debug_e4m3": ([P, P, I64, P], I),
        "sage_debug_pv_accum": ([P, P, I64, I64, P, P, P], I),
        "sage_debug_set_fault": ([I, ctypes.c_uint64], None),
        "sage_debug_set_prologue_launches": ([I], None),
        "sage_debug_set_fault_launches": ([I], None),
        "sage_debug_set_host_fail_chunk": ([I], None),
        "sage_debug_tc_rate": ([I, I64, P, P], I),
        "sage_kv_stats_noalloc_status": ([P], I),
        "sage_device_status": ([P, P], I),
        "sage_last_error": ([], ctypes.c_char_p),
        "sage_kv_stats_noalloc": ([P, P, I, I, I64, I64, I64, I64, P, P, P], I),
        "sage_launch_count": ([], ctypes.c_uint64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()
lib = _lib


def last_error() -> str:
    return _lib.sage_last_error().decode()


def launch_count() -> int:
    """Kernels this library has launched in this process (host-side count)."""
    return int(_lib.sage_launch_count())


def _check(rc: int, where: str):
    if rc != OK:
        raise SageError(rc, where, last_error())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"q/k/v must be float16 or bfloat16, got {t.dtype}")


def _require_dense(where, q, k, v, out=None):
    """The dense and packed entry points read q, k, v (and write out) as
    contiguous arrays of one dtype on a CUDA device.  Anything else is
    refused here, before any call: a view must go through the *_strided
    calls, which take its strides."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{where}: {name} is not on a CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} is not contiguous; pass views to "
                             f"quant_prologue_strided / attn_fwd_strided")
        if t.dtype != q.dtype:
            raise TypeError(f"{where}: {name} is {t.dtype}, q is {q.dtype}")
    if out is not None:
        import torch
        if not out.is_cuda or not out.is_contiguous() or out.dtype != torch.float32:
            raise ValueError(f"{where}: out must be a contiguous float32 CUDA tensor")
        if tuple(out.shape) != tuple(q.shape):
            raise ValueError(f"{where}: out has shape {tuple(out.shape)}, q {tuple(q.shape)}")


def _layout_code(layout) -> int:
    if layout in (HND, "HND"):
        return HND
    if layout in (NHD, "NHD"):
        return NHD
    raise ValueError(f"layout must be 'HND' or 'NHD', got {layout!r}")


def _dims(q, k, layout):
    if layout == HND:
        B, Hq, Lq, D = q.shape
        _, Hkv, Lk, _ = k.shape
    else:
        B, Lq, Hq, D = q.shape
        _, Lk, Hkv, _ = k.shape
    return B, Hq, Hkv, Lq, Lk, D


def workspace_bytes(B, Hq, Hkv, Lq, Lk, D) -> int:
    return int(_lib.sage_workspace_bytes(B, Hq, Hkv, Lq, Lk, D))


def workspace_bytes_varlen(nseq, total_q, total_k, Hq, Hkv, D) -> int:
    return int(_lib.sage_workspace_bytes_varlen(nseq, total_q, total_k, Hq, Hkv, D))


def alloc_workspace(nbytes: int, device="cuda"):
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def quant_prologue(q, k, v, layout="HND", ws=None, stream=None) -> Quantized:
    _require_dense("quant_prologue", q, k, v)
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(B, Hq, Hkv, Lq, Lk, D), q.device)
    qt = Quantized()
    rc = _lib.sage_quant_prologue(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), lay, B, Hq,
                                  Hkv, Lq, Lk, D, _ptr(ws), ws.numel(), ctypes.byref(qt),
                                  _stream(stream))
    _check(rc, "sage_quant_prologue")
    qt._ws = ws
    return qt


def quant_prologue_pv16(q, k, v, layout="HND", ws=None, stream=None) -> Quantized:
    """Prologue of the FP16-PV variant: INT8 Q/K as usual, V kept in fp16."""
    _require_dense("quant_prologue_pv16", q, k, v)
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(B, Hq, Hkv, Lq, Lk, D), q.device)
    qt = Quantized()
    rc = _lib.sage_quant_prologue_pv16(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), lay, B, Hq,
                                       Hkv, Lq, Lk, D, _ptr(ws), ws.numel(), ctypes.byref(qt),
                                       _stream(stream))
    _check(rc, "sage_quant_prologue_pv16")
    qt._ws = ws
    return qt


def quant_prologue_varlen(q, k, v, cu_q, cu_k, max_q, max_k, ws=None, stream=None):
    _require_dense("quant_prologue_varlen", q, k, v)
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    nseq = cu_q.numel() - 1
    if ws is None:
        ws = alloc_workspace(workspace_bytes_varlen(nseq, total_q, total_k, Hq, Hkv, D),
                             q.device)
    qt = Quantized()
    rc = _lib.sage_quant_prologue_varlen(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q),
                                         _ptr(cu_q), _ptr(cu_k), nseq, total_q, total_k,
                                         int(max_q), int(max_k), Hq, Hkv, D, _ptr(ws),
                                         ws.numel(), ctypes.byref(qt), _stream(stream))
    _check(rc, "sage_quant_prologue_varlen")
    qt._ws = ws
    return qt


def attn_quantized(qt: Quantized, out, layout="HND", is_causal=False, sm_scale=None,
                   stream=None):
    rc = _lib.sage_attn_quantized(ctypes.byref(qt), _ptr(out), _layout_code(layout),
                                  int(bool(is_causal)), float(sm_scale or 0.0),
                                  _stream(stream))
    _check(rc, "sage_attn_quantized")
    return out


def attn_fwd(q, k, v, out, layout="HND", is_causal=False, sm_scale=None, ws=None,
             stream=None):
    _require_dense("attn_fwd", q, k, v, out)
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(B, Hq, Hkv, Lq, Lk, D), q.device)
    rc = _lib.sage_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, Lq, Lk, D,
                            lay, int(bool(is_causal)), float(sm_scale or 0.0),
                            _dtype_code(q), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "sage_attn_fwd")
    return out


def attn_fwd_pv16(q, k, v, out, layout="HND", is_causal=False, sm_scale=None, ws=None,
                 stream=None):
    """Prologue + FP16-PV attention (dense)."""
    _require_dense("attn_fwd_pv16", q, k, v, out)
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(B, Hq, Hkv, Lq, Lk, D), q.device)
    rc = _lib.sage_attn_fwd_pv16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, Lq, Lk, D,
                                 lay, int(bool(is_causal)), float(sm_scale or 0.0),
                                 _dtype_code(q), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "sage_attn_fwd_pv16")
    return out


def workspace_bytes_host(B, Hq, Hkv, Lq, Lk, D, chunk_kv_heads=0) -> int:
    return int(_lib.sage_workspace_bytes_host(B, Hq, Hkv, Lq, Lk, D, int(chunk_kv_heads)))


def attn_fwd_host(q, k, v, out, layout="HND", is_causal=False, sm_scale=None,
                  chunk_kv_heads=0, ws=None, stream=None, pv16=False):
    """Attention on host tensors (page-locked for overlap): the library copies
    chunks in, computes them and copies the output back, pipelined.  `out`
    is a host float32 tensor of q's shape; `stream` completes when it is
    filled."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"attn_fwd_host: {name} must be a contiguous host tensor")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("attn_fwd_host: q, k and v must share one dtype")
    if out.dtype != torch.float32 or tuple(out.shape) != tuple(q.shape):
        raise ValueError("attn_fwd_host: out must be float32 with q's shape")
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes_host(B, Hq, Hkv, Lq, Lk, D, chunk_kv_heads))
    fn = _lib.sage_attn_fwd_host_pv16 if pv16 else _lib.sage_attn_fwd_host
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, Lq, Lk, D, lay,
            int(bool(is_causal)), float(sm_scale or 0.0), _dtype_code(q), int(chunk_kv_heads),
            _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "sage_attn_fwd_host_pv16" if pv16 else "sage_attn_fwd_host")
    return out


def attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max_q, max_k, is_causal=False,
                    sm_scale=None, ws=None, stream=None):
    _require_dense("attn_fwd_varlen", q, k, v, out)
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    nseq = cu_q.numel() - 1
    if ws is None:
        ws = alloc_workspace(workspace_bytes_varlen(nseq, total_q, total_k, Hq, Hkv, D),
                             q.device)
    rc = _lib.sage_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(cu_q),
                                   _ptr(cu_k), nseq, total_q, total_k, int(max_q),
                                   int(max_k), Hq, Hkv, D, int(bool(is_causal)),
                                   float(sm_scale or 0.0), _dtype_code(q), _ptr(ws),
                                   ws.numel(), _stream(stream))
    _check(rc, "sage_attn_fwd_varlen")
    return out


def view_strides(t, layout) -> tuple:
    """(batch, head, token) strides in elements of a q/k/v view in `layout`;
    the channel stride must be 1."""
    lay = _layout_code(layout)
    st = t.stride()
    if st[3] != 1:
        raise ValueError(f"strided views need contiguous channels (channel stride {st[3]})")
    return (st[0], st[1], st[2]) if lay == HND else (st[0], st[2], st[1])


def _strides_arg(vals):
    return (ctypes.c_int64 * 3)(*[int(x) for x in vals])


def _kv_strides(k, v, layout):
    ks, vs = view_strides(k, layout), view_strides(v, layout)
    if ks != vs:
        raise ValueError(f"k and v views must share their strides (k {ks}, v {vs})")
    return ks


def quant_prologue_strided(q, k, v, layout="HND", ws=None, stream=None) -> Quantized:
    """Prologue on q/k/v views (e.g. slices of one fused projection)."""
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(B, Hq, Hkv, Lq, Lk, D), q.device)
    qt = Quantized()
    rc = _lib.sage_quant_prologue_strided(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, Hq, Hkv, Lq, Lk, D,
        _strides_arg(view_strides(q, lay)), _strides_arg(_kv_strides(k, v, lay)), _ptr(ws),
        ws.numel(), ctypes.byref(qt), _stream(stream))
    _check(rc, "sage_quant_prologue_strided")
    qt._ws = ws
    return qt


def attn_fwd_strided(q, k, v, out, layout="HND", is_causal=False, sm_scale=None, ws=None,
                     stream=None):
    """Prologue + attention on q/k/v views; out is dense fp32 in `layout`."""
    lay = _layout_code(layout)
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k, lay)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(B, Hq, Hkv, Lq, Lk, D), q.device)
    rc = _lib.sage_attn_fwd_strided(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, Lq, Lk, D,
        _strides_arg(view_strides(q, lay)), _strides_arg(_kv_strides(k, v, lay)), lay,
        int(bool(is_causal)), float(sm_scale or 0.0), _dtype_code(q), _ptr(ws), ws.numel(),
        _stream(stream))
    _check(rc, "sage_attn_fwd_strided")
    return out


def sageattn(q, k, v, tensor_layout="HND", is_causal=False, sm_scale=None):
    """Drop-in style call: fp16/bf16 q, k, v on the GPU -> fp32 output.  Views
    (for instance the slices of a fused qkv projection) go through the
    strided entry point; a view it cannot serve raises with the reason."""
    import torch
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if q.is_contiguous() and k.is_contiguous() and v.is_contiguous():
        return attn_fwd(q, k, v, out, tensor_layout, is_causal, sm_scale)
    return attn_fwd_strided(q, k, v, out, tensor_layout, is_causal, sm_scale)


def sageattn_qk_int8_pv_fp16(q, k, v, tensor_layout="HND", is_causal=False, sm_scale=None):
    """The more accurate variant: INT8 QK^T, fp16 P and V (dense inputs)."""
    import torch
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    return attn_fwd_pv16(q, k, v, out, tensor_layout, is_causal, sm_scale)


def debug_qk_int32(qt: Quantized, seg, hq, qtile, ktile, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty(128 * 128, dtype=torch.int32, device="cuda")
    rc = _lib.sage_debug_qk_int32(ctypes.byref(qt), seg, hq, qtile, ktile, _ptr(out),
                                  _stream(stream))
    _check(rc, "sage_debug_qk_int32")
    return out.view(128, 128)


def debug_e4m3(x, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    rc = _lib.sage_debug_e4m3(_ptr(x), _ptr(out), x.numel(), _stream(stream))
    _check(rc, "sage_debug_e4m3")
    return out


def debug_pv_accum(p8, v8, status, out=None, stream=None):
    """sum_t P~_t V~_t^T through the attention kernel's own FP8 PV instructions.
    p8: uint8 CUDA tensor [ntiles, 128, 128] (e4m3 codes, key fastest);
    v8: uint8 CUDA tensor [ntiles, Dp, 128] (channel-major); status: a 4-byte
    CUDA tensor the call clears (read with device_status).  Returns fp32
    [128, Dp]."""
    import torch
    for name, t in (("p8", p8), ("v8", v8)):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.uint8):
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor")
    ntiles, dp = v8.shape[0], v8.shape[1]
    if tuple(p8.shape) != (ntiles, 128, 128) or tuple(v8.shape) != (ntiles, dp, 128):
        raise ValueError("p8 must be [ntiles,128,128] and v8 [ntiles,Dp,128]")
    if out is None:
        out = torch.empty(128, dp, dtype=torch.float32, device=p8.device)
    rc = _lib.sage_debug_pv_accum(_ptr(p8), _ptr(v8), ntiles, dp, _ptr(out), _ptr(status),
                                  _stream(stream))
    _check(rc, "sage_debug_pv_accum")
    return out


def kv_stats_noalloc(k, v, layout, k_mean, s_v, stream=None):
    """K channel means and V channel scales with no device allocation at all:
    the scratch is a static array inside the library (B*Hkv*Dp <= 16384).
    k_mean and s_v are caller-owned contiguous fp32 CUDA tensors of at least
    B*Hkv*Dp elements (Dp = 64 if D <= 64 else 128).  kv_stats_noalloc_status
    reports a failure on the device."""
    import torch
    if k.dim() != 4 or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"kv_stats_noalloc: k {tuple(k.shape)} and v {tuple(v.shape)} must be "
                         "4-D tensors of one shape")
    lay = _layout_code(layout)
    if lay == HND:
        B, Hkv, Lk, D = k.shape
    else:
        B, Lk, Hkv, D = k.shape
    need = B * Hkv * (64 if D <= 64 else 128)
    for name, t in (("k_mean", k_mean), ("s_v", s_v)):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"kv_stats_noalloc: {name} must be a contiguous float32 tensor")
        if t.numel() < need:
            raise ValueError(f"kv_stats_noalloc: {name} has {t.numel()} elements, needs {need}")
    _require_dense("kv_stats_noalloc", k, k, v)
    for name, t in (("k_mean", k_mean), ("s_v", s_v)):
        if not t.is_cuda:
            raise ValueError(f"kv_stats_noalloc: {name} is not on a CUDA device")
    rc = _lib.sage_kv_stats_noalloc(_ptr(k), _ptr(v), _dtype_code(k), lay, B, Hkv, Lk, D,
                                    _ptr(k_mean), _ptr(s_v), _stream(stream))
    _check(rc, "sage_kv_stats_noalloc")
    return k_mean, s_v


def workspace_bytes_varlen_host(nseq, total_q, total_k, Hq, Hkv, D, chunk_kv_heads=0) -> int:
    return int(_lib.sage_workspace_bytes_varlen_host(nseq, total_q, total_k, Hq, Hkv, D,
                                                     int(chunk_kv_heads)))


def attn_fwd_varlen_host(q, k, v, out, cu_q, cu_k, max_q, max_k, is_causal=False,
                         sm_scale=None, chunk_kv_heads=0, ws=None, stream=None):
    """Packed-sequence attention on host tensors (q, k, v packed (T, H, D),
    page-locked for overlap; out float32 of q's shape; cu_q and cu_k int32
    host tensors of nseq + 1 offsets): the library copies chunks of kv heads
    in, computes them and copies the output back, pipelined.  `stream`
    completes when `out` is filled."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("cu_q", cu_q),
                    ("cu_k", cu_k)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"attn_fwd_varlen_host: {name} must be a contiguous host tensor")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("attn_fwd_varlen_host: q, k and v must share one dtype")
    if cu_q.dtype != torch.int32 or cu_k.dtype != torch.int32:
        raise TypeError("attn_fwd_varlen_host: cu_q and cu_k must be int32")
    if q.dim() != 3 or k.dim() != 3 or tuple(v.shape) != tuple(k.shape):
        raise ValueError("attn_fwd_varlen_host: q, k, v must be packed (T, H, D), v like k")
    if out.dtype != torch.float32 or tuple(out.shape) != tuple(q.shape):
        raise ValueError("attn_fwd_varlen_host: out must be float32 with q's shape")
    if cu_q.numel() != cu_k.numel() or cu_q.numel() < 2:
        raise ValueError("attn_fwd_varlen_host: cu_q and cu_k need the same nseq + 1 >= 2 entries")
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    nseq = cu_q.numel() - 1
    if ws is None:
        ws = alloc_workspace(workspace_bytes_varlen_host(nseq, total_q, total_k, Hq, Hkv, D,
                                                         chunk_kv_heads))
    rc = _lib.sage_attn_fwd_varlen_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(cu_q),
                                        _ptr(cu_k), nseq, total_q, total_k, int(max_q),
                                        int(max_k), Hq, Hkv, D, int(bool(is_causal)),
                                        float(sm_scale or 0.0), _dtype_code(q),
                                        int(chunk_kv_heads), _ptr(ws), ws.numel(),
                                        _stream(stream))
    _check(rc, "sage_attn_fwd_varlen_host")
    return out


def debug_tc_rate(kind: int, n_mma: int, status, stream=None):
    """Enqueues n_mma back-to-back M=128 N=128 tcgen05 MMAs per SM (kind 0:
    fp16 K=16, kind 1: e4m3 K=32); time it with events on `stream`."""
    _check(_lib.sage_debug_tc_rate(int(kind), int(n_mma), _ptr(status), _stream(stream)),
           "sage_debug_tc_rate")


def kv_stats_noalloc_status(stream=None) -> int:
    """Device status of the last kv_stats_noalloc call on this device."""
    return int(_lib.sage_kv_stats_noalloc_status(_stream(stream)))


def set_fault(skip_kv_tile: int = -1, timeout_ns: int = 0, launches: int = -1):
    """Failure injection: attention launches skip key/value tile skip_kv_tile
    (-1: off) and give up waiting after timeout_ns; launches >= 0 limits the
    fault to that many launches."""
    _lib.sage_debug_set_fault_launches(int(launches))
    _lib.sage_debug_set_fault(int(skip_kv_tile), int(timeout_ns))


def set_prologue_launches(launches: int = 0):
    """Test hook: 1 or 2 prologue launches, 0 to choose by size."""
    _lib.sage_debug_set_prologue_launches(int(launches))


def set_host_fail_chunk(chunk: int = -1):
    """Test hook: the host-buffer calls fail at chunk `chunk` (-1: off)."""
    _lib.sage_debug_set_host_fail_chunk(int(chunk))


def device_status(ws, stream=None) -> int:
    return int(_lib.sage_device_status(_ptr(ws), _stream(stream)))


def ws_view(qt: Quantized, field: str, dtype, shape):
    """A torch view of one workspace buffer (for tests and inspection)."""
    import torch
    ws = qt._ws
    off = getattr(qt, field) - ws.data_ptr()
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).view(*shape)
