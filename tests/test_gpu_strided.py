"""Strided q/k/v views through the strided entry points (SageAttention-RDNA4
v0.3.0, "Fused q/k/v views": q, k and v arrive as views into one fused
projection, so their token stride is 3*H*D).

For every view layout the quantised tensors must be bit-exact against the
oracle run on contiguous copies, and the outputs within the usual tolerance.
The cases cover the tensor-copy path and the element-wise path (D % 8 != 0),
GQA, bf16 and causal masking."""
import numpy as np
import pytest

from quantized_attention_smooth_gb300 import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sage():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_smooth_gb300 import sage as s
    return s


CASES = [
    dict(name="fused_qkv_nhd_d128", kind="fused", B=2, Hq=4, Hkv=4, L=300, D=128,
         dtype=wl.F16, causal=False),
    dict(name="fused_qkv_nhd_d36_elementwise", kind="fused", B=1, Hq=2, Hkv=2, L=200, D=36,
         dtype=wl.F16, causal=False),
    dict(name="fused_kv_gqa_bf16_causal", kind="fused_kv", B=2, Hq=8, Hkv=2, L=260, D=64,
         dtype=wl.BF16, causal=True),
    dict(name="hnd_sliced_channels", kind="slice_hnd", B=2, Hq=3, Hkv=3, L=333, D=64,
         dtype=wl.BF16, causal=False),
]


def _normal_bits(rng, shape, dtype, k_offset=None):
    x = rng.standard_normal(shape, dtype=np.float32)
    if k_offset is not None:
        x = x + k_offset
    return wl.to_bits(x, dtype)


def _device(bits, dtype):
    return H.to_device(np.ascontiguousarray(bits), dtype)


def _views(c, seed):
    """(workload, contiguous oracle inputs, device views q, k, v)."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, L, D, dt = c["B"], c["Hq"], c["Hkv"], c["L"], c["D"], c["dtype"]
    off = rng.normal(0.0, 3.0, size=D).astype(np.float32)
    if c["kind"] == "fused":                      # [B, L, 3, H, D], NHD views
        parts = [_normal_bits(rng, (B, L, 1, Hq, D), dt, off if i == 1 else None)
                 for i in range(3)]
        fused = np.concatenate(parts, axis=2)
        t = _device(fused, dt)
        q, k, v = t.unbind(2)
        inp = {n: np.ascontiguousarray(fused[:, :, i]) for i, n in enumerate("qkv")}
        layout = wl.NHD
    elif c["kind"] == "fused_kv":                 # q sliced from [B, L, Hq, 2D]; kv fused
        qwide = _normal_bits(rng, (B, L, Hq, 2 * D), dt)
        kv = np.concatenate([_normal_bits(rng, (B, L, 1, Hkv, D), dt, off),
                             _normal_bits(rng, (B, L, 1, Hkv, D), dt)], axis=2)
        q = _device(qwide, dt)[..., :D]
        k, v = _device(kv, dt).unbind(2)
        inp = dict(q=np.ascontiguousarray(qwide[..., :D]),
                   k=np.ascontiguousarray(kv[:, :, 0]), v=np.ascontiguousarray(kv[:, :, 1]))
        layout = wl.NHD
    else:                                         # HND tensors sliced to D channels
        wide = [_normal_bits(rng, (B, h, L, 2 * D), dt, np.concatenate([off, off])
                             if i == 1 else None)
                for i, h in enumerate((Hq, Hkv, Hkv))]
        q, k, v = (_device(x, dt)[..., :D] for x in wide)
        inp = {n: np.ascontiguousarray(x[..., :D]) for n, x in zip("qkv", wide)}
        layout = wl.HND
    w = wl.Workload(c["name"], B=B, Hq=Hq, Hkv=Hkv, Lq=L, Lk=L, D=D, dtype=dt,
                    layout=layout, causal=c["causal"], seed=seed)
    return w, inp, (q, k, v)


@pytest.mark.parametrize("c", CASES, ids=[c["name"] for c in CASES])
def test_strided_views_bit_exact_and_outputs(sage, orc, c):
    w, inp, (q, k, v) = _views(c, seed=300 + CASES.index(c))
    assert not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous())
    lay = "HND" if w.layout == wl.HND else "NHD"
    qt = sage.quant_prologue_strided(q, k, v, lay)
    torch.cuda.synchronize()
    ws = H.Workspace(sage, qt, w, inp)
    pros = {}
    for s in range(w.nseg):
        qs, ks, vs = wl.segment(w, inp, s)
        pros[s] = orc.prologue(qs, ks, vs, w.dtype)
        mism = H.compare_prologue(pros[s], ws.segment(s), w.D)
        assert not any(mism.values()), f"segment {s}: {mism}"
        assert ws.padding_is_zero(s)
    assert sage.device_status(qt._ws) == sage.OK

    scale = wl.default_sm_scale(w)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    sage.attn_quantized(qt, out, lay, w.causal, scale)
    out_np = out.cpu().numpy()
    worst, cmin = 0.0, 1.0
    for s in range(w.nseg):
        qs, ks, vs = wl.segment(w, inp, s)
        ref = orc.attn(pros[s], w.causal, scale)
        ex = orc.attn_exact(qs, ks, vs, w.dtype, w.causal, scale)
        got = wl.out_segment(w, out_np, s, None)
        assert np.all(np.isfinite(got))
        worst = max(worst, float(np.max(np.abs(got.astype(np.float64) - ref))))
        cmin = min(cmin, H.cosine(got, ex))
    assert worst <= H.ATOL_ORACLE, worst
    assert cmin >= H.COS_EXACT, cmin

    # the one-call drop-in path routes the views through the strided entry
    again = sage.sageattn(q, k, v, lay, w.causal, scale)
    torch.cuda.synchronize()
    assert torch.equal(again, out)


def test_strided_views_two_launch_prologue(sage, orc):
    """Strided views through the prologue's two-launch plan (forced)."""
    sage.set_prologue_launches(2)
    try:
        test_strided_views_bit_exact_and_outputs(sage, orc, CASES[2])
    finally:
        sage.set_prologue_launches(0)


def test_dense_wrappers_refuse_views_and_mixed_dtypes(sage):
    """A view passed to a dense wrapper would be read as if contiguous: the
    binding refuses it (pointing at the strided calls), as it refuses mixed
    q/k/v dtypes and an output of the wrong type or shape."""
    fused = torch.zeros(1, 128, 3, 2, 64, dtype=torch.float16, device="cuda")
    q, k, v = fused.unbind(2)
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError, match="strided"):
        sage.attn_fwd(q, k, v, out, "NHD")
    with pytest.raises(ValueError, match="strided"):
        sage.quant_prologue(q, k, v, "NHD")
    qc, kc = q.contiguous(), k.contiguous()
    with pytest.raises(TypeError):
        sage.attn_fwd(qc, kc.to(torch.bfloat16), v.contiguous(), out, "NHD")
    with pytest.raises(ValueError, match="out"):
        sage.attn_fwd(qc, kc, v.contiguous(), out.half(), "NHD")
