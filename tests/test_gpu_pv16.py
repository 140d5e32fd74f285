"""GPU parity of the FP16-PV variant (INT8 QK^T with fp16 P and V: the
SageAttention overview's sageattn_qk_int8_pv_fp16 backend, the most accurate
one in the SageAttention 2.2.0 sm_120a wheel page's accuracy table).

* Q/K operands, their scales and the K mean: bit-exact against the oracle;
* V in fp16 (channel-major in the workspace): bit-exact against the oracle;
* outputs: max-abs <= 2e-3 against the oracle's FP16-PV attention, cosine
  >= 0.9999 against fp64 attention, and the one-call entry point equal to
  prologue + attention.
"""
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


def _w(name, **kw):
    base = dict(B=1, Hq=2, Hkv=2, Lq=256, Lk=256, D=64, dtype=wl.F16, layout=wl.HND,
                causal=False, seed=500, k_offset_sigma=2.0)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    _w("pv16_d64"),
    _w("pv16_d128_ragged", Lq=300, Lk=333, D=128, seed=501),
    _w("pv16_d40_bf16", D=40, Lq=200, Lk=260, dtype=wl.BF16, seed=502),
    _w("pv16_causal", Lq=384, Lk=384, causal=True, D=128, seed=503),
    _w("pv16_gqa_nhd_bf16", B=2, Hq=8, Hkv=2, Lq=200, Lk=300, D=128, layout=wl.NHD,
       dtype=wl.BF16, seed=504, k_outliers=(7, 42), k_outlier_value=15.0, k_offset_sigma=0.0),
    _w("pv16_lk1", Lq=64, Lk=1, seed=505),
    _w("pv16_cross", Lq=600, Lk=150, D=128, causal=True, seed=506),
]


def _v16_segment(sage, qt, w, s):
    """The fp16 V of segment s from the workspace, as [Hkv, Lk, Dp] bits."""
    v = sage.ws_view(qt, "v8", torch.int16, (qt.v_rows, qt.v_cols)).cpu().numpy()
    Lk = w.seg_lengths()[s][1]
    rows = s * qt.Hkv * qt.Dp
    return np.stack([v[rows + h * qt.Dp: rows + (h + 1) * qt.Dp, :Lk].T
                     for h in range(qt.Hkv)]).view(np.uint16)


def _check(sage, orc, w, rows_of=None):
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    lay = "HND" if w.layout == wl.HND else "NHD"
    qt = sage.quant_prologue_pv16(d["q"], d["k"], d["v"], lay)
    torch.cuda.synchronize()
    assert qt.v_fp16 == 1
    ws = H.Workspace(sage, qt, w, inp)
    scale = wl.default_sm_scale(w)
    out = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    sage.attn_quantized(qt, out, lay, w.causal, scale)
    out_np = out.cpu().numpy()
    worst, cmin = 0.0, 1.0
    for s in range(w.nseg):
        q, k, v = wl.segment(w, inp, s)
        pro = orc.prologue(q, k, v, w.dtype)
        got = ws.segment(s)
        for name in ("q8", "s_q", "k8", "s_k", "k_mean"):
            a, b = np.asarray(pro[name]), np.asarray(got[name])
            if name == "k_mean":
                a, b = a[:, :w.D], b[:, :w.D]
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name
        v16 = orc.v16(v, w.dtype)
        assert np.array_equal(_v16_segment(sage, qt, w, s), v16), "v16"
        lq = w.seg_lengths()[s][0]
        rows = rows_of(lq) if rows_of else (0, lq)
        ref = orc.attn_pv16(pro, v16, w.causal, scale, rows=rows)
        ex = orc.attn_exact(q, k, v, w.dtype, w.causal, scale, rows=rows)
        g = wl.out_segment(w, out_np, s, None)[:, rows[0]:rows[1]]
        r, e = ref[:, rows[0]:rows[1]], ex[:, rows[0]:rows[1]]
        assert np.all(np.isfinite(g))
        worst = max(worst, float(np.max(np.abs(g.astype(np.float64) - r))))
        if np.linalg.norm(e) > 0:
            cmin = min(cmin, H.cosine(g, e))
    assert sage.device_status(qt._ws) == sage.OK
    assert worst <= H.ATOL_ORACLE, worst
    assert cmin >= 0.9999, cmin
    # the one-call entry point runs the same kernels
    again = torch.empty_like(out)
    sage.attn_fwd_pv16(d["q"], d["k"], d["v"], again, lay, w.causal, scale)
    torch.cuda.synchronize()
    assert torch.equal(again, out)
    return worst


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_pv16_small_shapes(sage, orc, w):
    _check(sage, orc, w)


def test_pv16_bench_shape_sampled_rows(sage, orc):
    w = wl.WORKLOADS["b2_h24_l4096_d128"]
    _check(sage, orc, w, rows_of=lambda lq: (lq - 200, lq))


def test_pv16_two_launch_prologue(sage, orc):
    """The prologue's two-launch plan (forced) writes the same fp16 V and
    Q/K operands, bit-exactly, and the outputs keep the tolerance."""
    sage.set_prologue_launches(2)
    try:
        _check(sage, orc, _w("pv16_two_launch", Lq=300, Lk=333, D=128, seed=507,
                             dtype=wl.BF16))
    finally:
        sage.set_prologue_launches(0)
