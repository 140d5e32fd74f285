"""The C-ABI library builds, loads and exports every declared symbol; host-side
validation rejects bad arguments before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from quantized_attention_smooth_gb300 import sage

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "sage.h")).read()
    return set(re.findall(r"SAGE_API\s+[\w\s\*]+?\b(sage_\w+)\s*\(", src))


def test_header_declares_the_binding_exports():
    assert _declared() == set(sage.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(sage._build.LIB)
    for name in _declared():
        assert hasattr(lib, name), name


def test_workspace_sizes():
    n = sage.workspace_bytes(2, 24, 24, 4096, 4096, 128)
    # q16 + k16 (2 B) + the V region (2 B: e4m3, or fp16 in the FP16-PV
    # variant) per padded element dominate
    assert 2 * 24 * 4096 * 128 * 6 <= n <= 2 * 24 * 4096 * 128 * 6 * 1.05
    assert sage.workspace_bytes(1, 3, 2, 10, 10, 64) == 0      # Hq % Hkv
    assert sage.workspace_bytes(1, 2, 2, 10, 10, 0) == 0       # D = 0
    assert sage.workspace_bytes(1, 2, 2, 10, 10, 129) == 0     # D > 128
    assert sage.workspace_bytes(1, 2, 2, 100, 100, 40) > 0
    # padded D: 40 -> 64, 80 -> 128
    assert (sage.workspace_bytes(1, 2, 2, 128, 128, 40) ==
            sage.workspace_bytes(1, 2, 2, 128, 128, 64))
    assert (sage.workspace_bytes(1, 2, 2, 128, 128, 80) ==
            sage.workspace_bytes(1, 2, 2, 128, 128, 128))
    assert sage.workspace_bytes_varlen(8, 1000, 1000, 16, 16, 80) > 0
    assert sage.workspace_bytes_varlen(8, 1000, 1000, 16, 3, 80) == 0


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first


def _fwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=2, Hkv=2, Lq=128, Lk=128,
             D=64, layout=0, causal=0, scale=0.0, dtype=0, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return sage.lib.sage_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"],
                                  a["Hkv"], a["Lq"], a["Lk"], a["D"], a["layout"],
                                  a["causal"], a["scale"], a["dtype"], a["ws"],
                                  a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(D=129), sage.ERR_UNSUPPORTED, "head_dim"),
    (dict(D=0), sage.ERR_UNSUPPORTED, "head_dim"),
    (dict(Hq=3, Hkv=2), sage.ERR_INVALID_ARG, "multiple"),
    (dict(Hkv=0), sage.ERR_INVALID_ARG, "multiple"),
    (dict(dtype=7), sage.ERR_INVALID_ARG, "dtype"),
    (dict(layout=5), sage.ERR_INVALID_ARG, "layout"),
    (dict(q=ctypes.c_void_p(0)), sage.ERR_INVALID_ARG, "non-null"),
    (dict(k=ctypes.c_void_p(0x10001)), sage.ERR_INVALID_ARG, "aligned"),
    (dict(out=ctypes.c_void_p(0)), sage.ERR_INVALID_ARG, "out"),
    (dict(out=ctypes.c_void_p(0x10002)), sage.ERR_INVALID_ARG, "out"),
    (dict(B=-1), sage.ERR_INVALID_ARG, "negative"),
    (dict(ws=ctypes.c_void_p(0x10010)), sage.ERR_WORKSPACE, "256-byte"),
    (dict(ws_bytes=1000), sage.ERR_WORKSPACE, "needs"),
])
def test_bad_arguments_are_rejected_on_the_host(kw, status, needle):
    rc = _fwd(**kw)
    assert rc == status
    assert needle in sage.last_error()


def test_empty_problem_is_a_no_op():
    assert _fwd(B=0) == sage.OK
    assert _fwd(Lq=0) == sage.OK
    assert sage.last_error() == ""


def test_varlen_rejects_bad_arguments():
    lib = sage.lib
    rc = lib.sage_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, ctypes.c_void_p(0), FAKE, 2, 10,
                                  10, 5, 5, 2, 2, 64, 0, 0.0, 0, FAKE, 1 << 30, None)
    assert rc == sage.ERR_INVALID_ARG and "cu_seqlens" in sage.last_error()
    rc = lib.sage_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 10, 5, 5, 2,
                                  2, 300, 0, 0.0, 0, FAKE, 1 << 30, None)
    assert rc == sage.ERR_UNSUPPORTED
    assert lib.sage_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, 1, 1, 2, 2,
                                    64, 0, 0.0, 0, FAKE, 0, None) == sage.OK


def test_quantized_call_rejects_unfilled_struct():
    qt = sage.Quantized()
    rc = sage.lib.sage_attn_quantized(ctypes.byref(qt), FAKE, 0, 0, 0.0, None)
    assert rc == sage.ERR_INVALID_ARG
    rc = sage.lib.sage_debug_qk_int32(ctypes.byref(qt), 0, 0, 0, 0, FAKE, None)
    assert rc == sage.ERR_INVALID_ARG


def test_sage_error_carries_reason():
    with pytest.raises(sage.SageError, match="head_dim"):
        sage._check(_fwd(D=200), "sage_attn_fwd")


def _strided(qs, kvs, **kw):
    a = dict(B=1, Hq=2, Hkv=2, Lq=128, Lk=128, D=64, layout=0)
    a.update(kw)
    arr = lambda x: None if x is None else (ctypes.c_int64 * 3)(*x)
    return sage.lib.sage_attn_fwd_strided(FAKE, FAKE, FAKE, FAKE, a["B"], a["Hq"], a["Hkv"],
                                          a["Lq"], a["Lk"], a["D"], arr(qs), arr(kvs),
                                          a["layout"], 0, 0.0, 0, FAKE, 1 << 30, None)


@pytest.mark.parametrize("qs,kvs,status,needle", [
    (None, (1, 1, 1), sage.ERR_INVALID_ARG, "strides"),
    ((0, 64, 384), (24576, 64, 384), sage.ERR_UNSUPPORTED, "zero (broadcast)"),
    ((24576, 64, 384), (24576, -64, 384), sage.ERR_UNSUPPORTED, "positive"),
    ((1 << 39, 64, 384), (24576, 64, 384), sage.ERR_UNSUPPORTED, "2^39"),
])
def test_strided_views_refused_with_a_reason(qs, kvs, status, needle):
    """Views the strided entry cannot serve are refused before any launch,
    with the reason in the error text (the pages' fused q/k/v note: a refusal
    carries its reason)."""
    rc = _strided(qs, kvs)
    assert rc == status
    assert needle in sage.last_error()


def test_view_strides_of_fused_projection_slices():
    torch = pytest.importorskip("torch")
    B, L, H, D = 2, 5, 3, 8
    qkv = torch.empty(B, L, 3, H, D, dtype=torch.float16)
    q, k, v = qkv.unbind(2)                       # NHD views, token stride 3*H*D
    assert sage.view_strides(q, "NHD") == (L * 3 * H * D, D, 3 * H * D)
    assert sage.view_strides(k, "NHD") == sage.view_strides(v, "NHD")
    t = torch.empty(B, H, L, 2 * D, dtype=torch.float16)[..., :D]   # HND, token stride 2D
    assert sage.view_strides(t, "HND") == (H * L * 2 * D, L * 2 * D, 2 * D)
    with pytest.raises(ValueError, match="contiguous channels"):
        sage.view_strides(torch.empty(B, H, L, D, dtype=torch.float16).transpose(2, 3), "HND")


def test_binding_refuses_tensors_it_would_misread():
    """The dense wrappers refuse tensors they would read wrongly (host-side,
    before any call): not on a CUDA device, and (on a GPU) not contiguous,
    mixed dtypes or a wrong output."""
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 2, 128, 64, dtype=torch.float16)
    out = torch.zeros(1, 2, 128, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        sage.attn_fwd(q, q, q, out)
    with pytest.raises(ValueError, match="CUDA"):
        sage.quant_prologue(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        sage.quant_prologue_pv16(q, q, q)


def test_host_buffer_call_sizes_and_refusals():
    """sage_workspace_bytes_host: the chunk prologue's workspace plus two
    staging slots (q, k, v, out of one chunk); sage_attn_fwd_host refuses bad
    arguments before touching a device."""
    L = sage.lib
    whole = L.sage_workspace_bytes(1, 4, 2, 256, 256, 64)
    one = L.sage_workspace_bytes_host(3, 4, 2, 256, 256, 64, 1)
    two = L.sage_workspace_bytes_host(3, 4, 2, 256, 256, 64, 2)
    chunk1 = 2 * 256 * 64 * 2 + 2 * (1 * 256 * 64 * 2) + 2 * 256 * 64 * 4   # q, k, v, out
    assert one >= 2 * chunk1
    assert two > one >= whole // 2
    assert L.sage_workspace_bytes_host(1, 3, 2, 256, 256, 64, 0) == 0       # Hq % Hkv
    assert L.sage_workspace_bytes_host(1, 2, 2, 256, 256, 129, 0) == 0      # D > 128

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=2, Hkv=2, Lq=128, Lk=128, D=64,
                 layout=0, causal=0, scale=0.0, dtype=0, chunk=0, ws=FAKE, ws_bytes=1 << 30)
        a.update(kw)
        return L.sage_attn_fwd_host(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"],
                                    a["Hkv"], a["Lq"], a["Lk"], a["D"], a["layout"],
                                    a["causal"], a["scale"], a["dtype"], a["chunk"], a["ws"],
                                    a["ws_bytes"], None)
    assert call(B=0) == sage.OK
    assert call(Lq=0) == sage.OK
    assert call(layout=5) == sage.ERR_INVALID_ARG
    assert call(Lk=0) == sage.ERR_INVALID_ARG
    assert call(q=None) == sage.ERR_INVALID_ARG
    assert call(dtype=7) == sage.ERR_INVALID_ARG
    assert call(Hq=3) == sage.ERR_INVALID_ARG


def test_host_buffer_call_automatic_chunk():
    """The automatic chunk holds one wave of query-tile pairs (one per SM; the
    plan assumes GB300's 152 SMs when no device answers), or one kv head fewer
    when that still fills 90 % of the wave: at B=2 H=24 L=4096, 16 pairs per
    head, 10 heads would spill 8 pairs into a second wave and 9 heads (144
    pairs) fill 95 % of one."""
    import torch
    L = sage.lib
    if torch.cuda.is_available():
        pytest.skip("the device's own SM count decides on a GPU")
    auto = L.sage_workspace_bytes_host(2, 24, 24, 4096, 4096, 128, 0)
    assert auto == L.sage_workspace_bytes_host(2, 24, 24, 4096, 4096, 128, 9)
    assert auto != L.sage_workspace_bytes_host(2, 24, 24, 4096, 4096, 128, 10)
    # B=1 H=24 L=32768: attention outlasts the copies (13107 flops per copied
    # byte over D), so the chunk fills whole waves: 7 kv heads, 896 pairs in
    # 6 waves of 152 (1.8 % idle)
    long = L.sage_workspace_bytes_host(1, 24, 24, 32768, 32768, 128, 0)
    assert long == L.sage_workspace_bytes_host(1, 24, 24, 32768, 32768, 128, 7)
    # B=4 L=8192 with 4 query heads per kv head stays copy-bound (4681): two
    # kv heads, the one-wave rule
    gqa = L.sage_workspace_bytes_host(4, 32, 8, 8192, 8192, 128, 0)
    assert gqa == L.sage_workspace_bytes_host(4, 32, 8, 8192, 8192, 128, 2)
    # a chunk never exceeds the kv heads there are
    assert (L.sage_workspace_bytes_host(1, 8, 2, 128, 128, 64, 0) ==
            L.sage_workspace_bytes_host(1, 8, 2, 128, 128, 64, 2))


def test_varlen_host_call_sizes_and_refusals():
    """sage_workspace_bytes_varlen_host: the chunk's varlen prologue
    workspace, the device copy of both offset arrays and two staging slots;
    sage_attn_fwd_varlen_host checks its host offset arrays (start 0, end at
    the total, lengths within the maxima) before touching a device."""
    import ctypes
    L = sage.lib
    one = L.sage_workspace_bytes_varlen_host(3, 700, 900, 4, 2, 64, 1)
    two = L.sage_workspace_bytes_varlen_host(3, 700, 900, 4, 2, 64, 2)
    chunk1 = 2 * 700 * 64 * 2 + 2 * (900 * 64 * 2) + 2 * 700 * 64 * 4     # q, k, v, out
    assert one >= 2 * chunk1 + L.sage_workspace_bytes_varlen(3, 700, 900, 2, 1, 64)
    assert two > one
    assert L.sage_workspace_bytes_varlen_host(0, 700, 900, 4, 2, 64, 0) == 0     # nseq
    assert L.sage_workspace_bytes_varlen_host(3, 700, 900, 3, 2, 64, 0) == 0     # Hq % Hkv
    assert L.sage_workspace_bytes_varlen_host(3, 700, 900, 4, 2, 129, 0) == 0    # D > 128

    def cu(*xs):
        return (ctypes.c_int32 * len(xs))(*xs)

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, cu_q=cu(0, 300, 700), cu_k=cu(0, 400, 900),
                 nseq=2, total_q=700, total_k=900, max_q=400, max_k=500, Hq=2, Hkv=2, D=64,
                 causal=0, scale=0.0, dtype=0, chunk=0, ws=FAKE, ws_bytes=1 << 30)
        a.update(kw)
        return L.sage_attn_fwd_varlen_host(
            a["q"], a["k"], a["v"], a["out"], ctypes.cast(a["cu_q"], ctypes.c_void_p),
            ctypes.cast(a["cu_k"], ctypes.c_void_p), a["nseq"], a["total_q"], a["total_k"],
            a["max_q"], a["max_k"], a["Hq"], a["Hkv"], a["D"], a["causal"], a["scale"],
            a["dtype"], a["chunk"], a["ws"], a["ws_bytes"], None)
    assert call(nseq=0) == sage.OK
    assert call(total_q=0) == sage.OK
    assert call(total_k=0) == sage.ERR_INVALID_ARG
    assert call(q=None) == sage.ERR_INVALID_ARG
    assert call(dtype=7) == sage.ERR_INVALID_ARG
    assert call(Hq=3) == sage.ERR_INVALID_ARG
    assert call(cu_q=cu(1, 300, 700)) == sage.ERR_INVALID_ARG        # does not start at 0
    assert "cu_seqlens_q" in sage.last_error()
    assert call(cu_k=cu(0, 400, 901)) == sage.ERR_INVALID_ARG        # does not end at total_k
    assert "cu_seqlens_k" in sage.last_error()
    assert call(cu_q=cu(0, 301, 300)) == sage.ERR_INVALID_ARG        # negative length
    assert call(max_k=450) == sage.ERR_INVALID_ARG                   # a length above max_k
    assert "length 500" in sage.last_error()
    assert call(nseq=70000) == sage.ERR_UNSUPPORTED


def test_varlen_host_call_automatic_chunk():
    """Packed sequences: the automatic chunk holds four waves of query-tile
    pairs (152 SMs assumed without a device).  8 sequences, 73514 tokens:
    at most 575 + 8 query tiles per head, 292 pairs, so 3 kv heads."""
    import torch
    L = sage.lib
    if torch.cuda.is_available():
        pytest.skip("the device's own SM count decides on a GPU")
    auto = L.sage_workspace_bytes_varlen_host(8, 73514, 73514, 16, 16, 40, 0)
    assert auto == L.sage_workspace_bytes_varlen_host(8, 73514, 73514, 16, 16, 40, 3)
    assert auto != L.sage_workspace_bytes_varlen_host(8, 73514, 73514, 16, 16, 40, 2)


def test_varlen_host_binding_refuses_device_or_misshaped_tensors():
    import torch
    q = torch.zeros(10, 2, 64, dtype=torch.float16)
    out = torch.zeros(10, 2, 64, dtype=torch.float32)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(TypeError, match="int32"):
        sage.attn_fwd_varlen_host(q, q, q, out, cu.long(), cu, 10, 10)
    with pytest.raises(ValueError, match="float32"):
        sage.attn_fwd_varlen_host(q, q, q, out.half(), cu, cu, 10, 10)
    with pytest.raises(ValueError, match="same nseq"):
        sage.attn_fwd_varlen_host(q, q, q, out, cu, torch.tensor([0, 5, 10], dtype=torch.int32),
                                  10, 10)
    with pytest.raises(ValueError, match="packed"):
        sage.attn_fwd_varlen_host(q, q[None], q[None], out, cu, cu, 10, 10)


@pytest.mark.parametrize("case,needle", [
    ("v_shape", "one shape"),
    ("mean_dtype", "contiguous float32"),
    ("mean_view", "contiguous float32"),
    ("mean_small", "needs"),
    ("on_cpu", "not on a CUDA device"),
])
def test_noalloc_statistics_binding_refuses_bad_tensors(case, needle):
    """The binding's own checks of the allocation-free statistics call, which
    the C ABI cannot make (it sees plain pointers); every refusal is raised
    before any call."""
    import torch
    k = torch.zeros(1, 2, 128, 64, dtype=torch.float16)
    v = torch.zeros(1, 2, 128, 64, dtype=torch.float16)
    k_mean = torch.zeros(2 * 64)
    s_v = torch.zeros(2 * 64)
    if case == "v_shape":
        v = torch.zeros(1, 2, 100, 64, dtype=torch.float16)
    elif case == "mean_dtype":
        k_mean = torch.zeros(2 * 64, dtype=torch.float64)
    elif case == "mean_view":
        k_mean = torch.zeros(2 * 64 * 2)[::2]
    elif case == "mean_small":
        s_v = torch.zeros(2 * 64 - 1)
    with pytest.raises(ValueError, match=needle):
        sage.kv_stats_noalloc(k, v, "HND", k_mean, s_v)
