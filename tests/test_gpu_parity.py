"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* quantized tensors (int8 codes, e4m3 codes, every scale, the K mean) and the
  INT32 QK^T tiles: bit-exact;
* fp32 outputs: max-abs <= 2e-3 against the oracle and cosine >= 0.999
  against fp64 exact attention, on every row for small shapes and on sampled
  rows (first, middle and ragged last query tiles of several heads) for the
  full-size workloads.
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


def _small(name, **kw):
    base = dict(B=1, Hq=2, Hkv=2, Lq=256, Lk=256, D=64, dtype=wl.F16, layout=wl.HND,
                causal=False, seed=77, k_offset_sigma=2.0)
    base.update(kw)
    return wl.Workload(name, **base)


def _lengths(n, lo, hi, seed, zeros=0):
    """n sequence lengths drawn uniformly from [lo, hi] (seeded), `zeros` of
    them, chosen at random, set to 0."""
    rng = np.random.default_rng(seed)
    x = rng.integers(lo, hi + 1, size=n)
    if zeros:
        x[rng.choice(n, size=zeros, replace=False)] = 0
    return tuple(int(v) for v in x)


SMALL = [
    wl.WORKLOADS["small_d64"],
    _small("d128_ragged", Lq=300, Lk=333, D=128, seed=1),
    _small("d1", D=1, Lq=130, Lk=129, seed=2),
    _small("d16", D=16, seed=3),
    _small("d40", D=40, Lq=200, Lk=200, seed=4, k_outliers=(3, 17), k_outlier_value=20.0),
    _small("d65", D=65, seed=5),
    _small("d80", D=80, Lq=129, Lk=257, seed=6, dtype=wl.BF16),
    _small("d100_odd", D=100, Lq=77, Lk=391, seed=7),
    _small("d127", D=127, seed=8),
    _small("lk1", Lq=64, Lk=1, seed=9),
    _small("lq1", Lq=1, Lk=700, seed=10, D=128),
    _small("cross_lq_gt_lk", Lq=600, Lk=150, seed=11, D=128),
    _small("causal_square", Lq=384, Lk=384, causal=True, seed=12, D=128),
    _small("causal_lq_gt_lk", Lq=500, Lk=260, causal=True, seed=13, D=128, dtype=wl.BF16),
    _small("causal_lq_lt_lk", Lq=200, Lk=450, causal=True, seed=14, D=64),
    _small("gqa_nhd", B=2, Hq=8, Hkv=2, Lq=200, Lk=300, D=128, layout=wl.NHD, seed=15,
           dtype=wl.BF16, k_outliers=(7, 42), k_outlier_value=15.0, k_offset_sigma=0.0),
    _small("gqa_causal_nhd", B=2, Hq=4, Hkv=1, Lq=256, Lk=256, D=128, layout=wl.NHD,
           causal=True, seed=16),
    _small("batch3_hnd", B=3, Hq=3, Hkv=3, Lq=140, Lk=140, D=96, seed=17),
    _small("varlen_small", B=0, Hq=4, Hkv=2, Lq=0, Lk=0, D=80, layout=wl.NHD, seed=18,
           seqlens_q=(1, 130, 257, 128), seqlens_k=(5, 128, 300, 1)),
    _small("varlen_causal", B=0, Hq=2, Hkv=2, Lq=0, Lk=0, D=40, layout=wl.NHD, seed=19,
           causal=True, seqlens_q=(200, 64, 333), seqlens_k=(200, 64, 333)),
    _small("varlen_empty_keys", B=0, Hq=4, Hkv=2, Lq=0, Lk=0, D=64, layout=wl.NHD, seed=20,
           seqlens_q=(130, 7, 256), seqlens_k=(140, 0, 129)),
    # many short packed sequences: every segment's offsets, ragged tiles and
    # (for some) an empty key set
    _small("dense_many_batches", B=32, Hq=2, Hkv=1, Lq=70, Lk=90, D=128, layout=wl.NHD,
           seed=23),
    _small("gqa8_causal_bf16", B=1, Hq=16, Hkv=2, Lq=256, Lk=384, D=64, causal=True,
           dtype=wl.BF16, seed=24),
    _small("varlen_many", B=0, Hq=4, Hkv=2, Lq=0, Lk=0, D=64, layout=wl.NHD, seed=21,
           seqlens_q=_lengths(96, 1, 300, 210), seqlens_k=_lengths(96, 0, 300, 211, zeros=8)),
    _small("varlen_many_causal_bf16", B=0, Hq=2, Hkv=2, Lq=0, Lk=0, D=128, layout=wl.NHD,
           seed=22, dtype=wl.BF16, causal=True,
           seqlens_q=_lengths(64, 1, 400, 212), seqlens_k=_lengths(64, 1, 400, 212)),
    # more sequences than the prologue holds offsets for in shared memory:
    # the work lists sized by the longest sequence (D = 64: at D = 32 a
    # sequence of 4 queries over 52 keys has cosine 0.99897 to exact
    # attention in the oracle itself, below the bar)
    _small("varlen_300_sequences", B=0, Hq=2, Hkv=1, Lq=0, Lk=0, D=64, layout=wl.NHD, seed=23,
           seqlens_q=_lengths(300, 1, 60, 213), seqlens_k=_lengths(300, 0, 60, 214, zeros=12)),
]


# Stress shapes (many short packed sequences, 14k rows each): their rows span
# millions of P~ codes, so a near-tie that the kernel's exp2 rounds the other
# way (H.near_tie_rows) lands on a heavily weighted key now and then; one such
# row measured 2.8e-3.  Everything else stays within H.ATOL_ORACLE.
STRESS = {"varlen_many", "varlen_many_causal_bf16", "varlen_300_sequences"}


def _check_prologue(sage, orc, w, inp, d):
    qt = H.run_prologue(sage, w, d)
    torch.cuda.synchronize()
    ws = H.Workspace(sage, qt, w, inp)
    bad = {}
    ws.oracle = {}
    for s in range(w.nseg):
        q, k, v = wl.segment(w, inp, s)
        ref = orc.prologue(q, k, v, w.dtype)
        ws.oracle[s] = ref
        got = ws.segment(s)
        mism = H.compare_prologue(ref, got, w.D)
        if any(mism.values()):
            bad[s] = mism
        assert ws.padding_is_zero(s), f"segment {s}: padding not zeroed"
    assert not bad, f"bit mismatches per segment: {bad}"
    assert sage.device_status(qt._ws) == sage.OK
    return qt, ws


def _check_rows(orc, w, inp, out_np, samples, pros=None, allow_ties=False):
    """samples: list of (segment, (h0, h1), (r0, r1)).  Returns the largest
    difference to the oracle and the smallest cosine to fp64 attention.  With
    allow_ties, rows beyond H.ATOL_ORACLE whose excess a P~ near-tie explains
    are checked against H.FLIP_CAP here and left out of the largest
    difference; anything else still counts."""
    worst, cos_min = 0.0, 1.0
    pros = {} if pros is None else pros
    for s, heads, rows in samples:
        q, k, v = wl.segment(w, inp, s)
        if s not in pros:
            pros[s] = orc.prologue(q, k, v, w.dtype)
        scale = wl.default_sm_scale(w)
        ref = orc.attn(pros[s], w.causal, scale, heads=heads, rows=rows)
        ex = orc.attn_exact(q, k, v, w.dtype, w.causal, scale, heads=heads, rows=rows)
        got = wl.out_segment(w, out_np, s, inp.get("cu_q"))
        sl = (slice(*heads), slice(*rows))
        g, r, e = got[sl], ref[sl], ex[sl]
        assert np.all(np.isfinite(g)), f"non-finite output in segment {s}"
        err = np.max(np.abs(g.astype(np.float64) - r), axis=-1)        # [heads, rows]
        for hh, ii in zip(*np.nonzero(err > H.ATOL_ORACLE) if allow_ties else ([], [])):
            h, i = heads[0] + int(hh), rows[0] + int(ii)
            assert err[hh, ii] <= H.FLIP_CAP, (s, h, i, float(err[hh, ii]))
            assert H.near_tie_rows(orc, pros[s], h, [i], w.causal, scale)[0], \
                f"segment {s} head {h} row {i}: {float(err[hh, ii])} with no P~ near-tie"
            err[hh, ii] = 0.0
        worst = max(worst, float(err.max()) if err.size else 0.0)
        if np.linalg.norm(e) > 0:
            cos_min = min(cos_min, H.cosine(g, e))
    return worst, cos_min


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_shapes_bit_exact_and_all_rows(sage, orc, w):
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    _, ws = _check_prologue(sage, orc, w, inp, d)
    out = H.run_attention(sage, w, d).cpu().numpy()
    samples = []
    for s, (lq, lk) in enumerate(w.seg_lengths()):
        if lq > 0:
            samples.append((s, (0, w.Hq), (0, lq)))
    worst, cmin = _check_rows(orc, w, inp, out, samples, ws.oracle,
                              allow_ties=w.name in STRESS)
    assert worst <= H.ATOL_ORACLE, worst
    assert cmin >= H.COS_EXACT, cmin


def test_bf16_key_means_exact_over_extreme_ranges(sage, orc):
    """bf16 key sums where a channel mixes magnitudes far apart: partial sums
    that fp32 cannot hold exactly, partials more than 34 binades apart,
    subnormals, all-zero channels and values near the top of the range.  The
    K mean (and every code that depends on it) must still match the oracle's
    fp64 sum bit for bit."""
    w = _small("bf16_extreme", D=64, Lq=128, Lk=300, dtype=wl.BF16, seed=21,
               k_offset_sigma=0.0)
    inp = wl.make_inputs(w)
    k = wl.bits_to_float(inp["k"], wl.BF16).copy()          # (B, H, L, D)
    # (the oracle sums exactly in 128 bits, so each channel keeps its
    # exponent span within that)
    k[:, :, ::37, 0] = 2.0 ** 30                               # fp32 partials inexact
    k[:, :, 5::53, 0] = 2.0 ** -40
    k[:, :, 3::101, 1] = 2.0 ** 40                             # partials > 34 binades apart
    k[:, :, :, 2] = 0.0                                        # subnormals only
    k[:, :, :, 3] = 0.0                                        # all zero
    k[:, :, :, 4] = 0.0                                        # near the top of the range
    k[:, :, 11::97, 4] = 2.0 ** 124
    k[:, :, 13::89, 4] = -(2.0 ** 123)
    k[:, 1, 17, 5] = -(2.0 ** 60)
    bits = wl.to_bits(k, wl.BF16)
    bits[0, 0, 7, 2] = 0x0001
    bits[0, 1, 9, 2] = 0x8003
    bits[0, 0, 200, 2] = 0x0042
    inp["k"] = bits
    d = H.device_inputs(w, inp)
    _check_prologue(sage, orc, w, inp, d)


FULL = ["small_d64", "b2_h24_l4096_d128", "gqa_causal_b4_l8192", "dit_self_l32768",
        "dit_cross_l32768x512", "varlen_d80", "varlen_d40"]


def _samples(w):
    out = []
    for s, (lq, lk) in enumerate(w.seg_lengths()):
        if s not in (0, w.nseg - 1) and w.nseg > 2 and not w.varlen:
            continue
        last = max(0, lq - 200)
        mid = max(0, (lq // 2) // 128 * 128)
        for h in sorted({0, w.Hq - 1}):
            for r0 in sorted({0, mid, last}):
                out.append((s, (h, h + 1), (r0, min(lq, r0 + 200))))
    return out


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads(sage, orc, name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    _, wsh = _check_prologue(sage, orc, w, inp, d)
    ws = H.workspace_for(sage, w)
    out = H.run_attention(sage, w, d, ws=ws)
    assert sage.device_status(ws) == sage.OK
    out_np = out.cpu().numpy()
    worst, cmin = _check_rows(orc, w, inp, out_np, _samples(w), wsh.oracle)
    assert worst <= H.ATOL_ORACLE, worst
    assert cmin >= H.COS_EXACT, cmin
    # property that holds at any size: every written output is finite
    assert bool(torch.isfinite(out).all())


@pytest.mark.parametrize("D", [64, 128])
def test_qk_int32_tiles_bit_exact(sage, orc, D):
    w = _small("tiles", B=2, Hq=4, Hkv=2, Lq=300, Lk=520, D=D, seed=40 + D)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    qt, ws = _check_prologue(sage, orc, w, inp, d)
    for s in range(2):
        q, k, v = wl.segment(w, inp, s)
        ref = orc.prologue(q, k, v, w.dtype)
        for hq in (0, 3):
            hk = hq // 2
            for qtile, ktile in ((0, 0), (2, 4), (1, 3)):
                tile = sage.debug_qk_int32(qt, s, hq, qtile, ktile).cpu().numpy()
                qa = np.zeros((128, ref["q8"].shape[-1]), np.int64)
                ka = np.zeros((128, ref["k8"].shape[-1]), np.int64)
                qrows = ref["q8"][hq, qtile * 128:(qtile + 1) * 128]
                krows = ref["k8"][hk, ktile * 128:(ktile + 1) * 128]
                qa[:len(qrows)] = qrows
                ka[:len(krows)] = krows
                np.testing.assert_array_equal(tile, (qa @ ka.T).astype(np.int32))


def test_qk_int32_extreme_codes_exact(sage):
    """All codes +-127 along D=128 with matching sign rows: |S| reaches
    128 * 127^2 = 2,064,512 and stays exact in the fp32 accumulator."""
    rng = np.random.default_rng(5)
    # +-1 keys with every channel balanced over the 128 tokens: the channel
    # mean is exactly 0, smoothing leaves +-1 and every code is +-127
    signs = np.ones((128, 128), np.float32)
    for c in range(128):
        signs[rng.permutation(128)[:64], c] = -1.0
    k = torch.from_numpy(signs).to(torch.float16).cuda().view(1, 1, 128, 128)
    q = k.clone()                               # row i of Q equals key i
    v = torch.randn(1, 1, 128, 128, dtype=torch.float16, device="cuda")
    qt = sage.quant_prologue(q, k, v, "HND")
    tile = sage.debug_qk_int32(qt, 0, 0, 0, 0).cpu().numpy().astype(np.int64)
    q8 = sage.ws_view(qt, "q16", torch.float16, (128, 128)).float().cpu().numpy()
    k8 = sage.ws_view(qt, "k16", torch.float16, (128, 128)).float().cpu().numpy()
    assert np.all(np.abs(q8) == 127) and np.all(np.abs(k8) == 127)
    ref = q8.astype(np.int64) @ k8.astype(np.int64).T
    np.testing.assert_array_equal(tile, ref)
    assert np.abs(ref).max() == 128 * 127 * 127


def test_e4m3_conversion_matches_oracle_on_all_floats(sage, orc):
    """The kernel's fp32 -> e4m3 conversion over every fp32 bit pattern."""
    chunk = 1 << 28
    for c in range((1 << 32) // chunk):
        bits = np.arange(chunk, dtype=np.uint32) + np.uint32(c * chunk)
        x = bits.view(np.float32)
        gpu = sage.debug_e4m3(torch.from_numpy(x.view(np.int32)).cuda().view(torch.float32))
        g = gpu.cpu().numpy()
        ref = orc.e4m3_encode(x)
        nan = np.isnan(x)
        assert np.all((g[nan] & 0x7F) == 0x7F), "NaN must stay NaN"
        diff = np.nonzero((g != ref) & ~nan)[0]
        assert diff.size == 0, (f"chunk {c}: {diff.size} mismatches, first input "
                                f"{x[diff[0]]!r} bits {bits[diff[0]]:#x}: gpu {g[diff[0]]:#x} "
                                f"oracle {ref[diff[0]]:#x}")


def test_large_magnitude_causal_inputs_stay_finite(sage, orc):
    """Huge causal logits (q, k x 300, |x| ~ 1e4 in base 2): no NaN or Inf (the
    wheel page's accuracy section), and the output within the usual 2e-3 of
    the oracle.  At this magnitude one fp32 rounding of a logit is worth
    ~5e-4 in the exponent, so the kernel must round x = RN(S c) and then
    RN(x - m') in the oracle's order; a fused S c - m' misses by up to 0.1."""
    w = _small("huge", Lq=512, Lk=512, D=128, causal=True, seed=50, dtype=wl.BF16)
    inp = wl.make_inputs(w)
    scale = np.float32(300.0)
    for key in ("q", "k"):
        inp[key] = wl.to_bits(wl.bits_to_float(inp[key], w.dtype) * scale, w.dtype)
    d = H.device_inputs(w, inp)
    out = H.run_attention(sage, w, d)
    assert bool(torch.isfinite(out).all())
    q, k, v = wl.segment(w, inp, 0)
    ref = orc.attn(orc.prologue(q, k, v, w.dtype), True, wl.default_sm_scale(w))
    got = out.cpu().numpy()[0]
    assert H.cosine(got, ref) >= 0.999
    assert float(np.max(np.abs(got - ref))) <= H.ATOL_ORACLE


def test_prologue_is_deterministic(sage):
    w = wl.WORKLOADS["gqa_causal_b4_l8192"].replace(B=1, Lq=1000, Lk=1000)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    # every field the prologue writes (the V region is sized for the FP16-PV
    # variant's fp16 V; the e4m3 path leaves its second half untouched)
    a = H.run_prologue(sage, w, d)
    fa = _workspace_fields(sage, a)
    b = H.run_prologue(sage, w, d)
    fb = _workspace_fields(sage, b)
    for name in fa:
        assert torch.equal(fa[name], fb[name]), name


def test_quantized_entry_points_match_fused_call(sage):
    w = _small("split", B=2, Hq=4, Hkv=2, Lq=300, Lk=400, D=128, layout=wl.NHD, seed=60,
               causal=True)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    fused = H.run_attention(sage, w, d)
    qt = sage.quant_prologue(d["q"], d["k"], d["v"], "NHD")
    out = torch.empty_like(fused)
    sage.attn_quantized(qt, out, "NHD", True, wl.default_sm_scale(w))
    assert torch.equal(out, fused)


def test_default_scale_is_inverse_sqrt_d(sage):
    w = _small("scale", D=80, seed=61)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    a = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    sage.attn_fwd(d["q"], d["k"], d["v"], a, "HND", False, None)
    sage.attn_fwd(d["q"], d["k"], d["v"], b, "HND", False, float(np.float32(1) / np.sqrt(np.float32(80))))
    assert torch.equal(a, b)


def test_empty_keys_give_zeros(sage):
    q = torch.randn(1, 2, 10, 64, dtype=torch.float16, device="cuda")
    k = torch.randn(1, 2, 0, 64, dtype=torch.float16, device="cuda")
    out = torch.full((1, 2, 10, 64), 7.0, device="cuda")
    sage.attn_fwd(q, k, k, out, "HND")
    assert bool((out == 0).all())


def test_inconsistent_cu_seqlens_reported(sage):
    q = torch.randn(300, 2, 64, dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, 200, 100], dtype=torch.int32, device="cuda")   # not monotonic
    out = torch.zeros(300, 2, 64, device="cuda")
    ws = sage.alloc_workspace(sage.workspace_bytes_varlen(2, 300, 300, 2, 2, 64))
    sage.attn_fwd_varlen(q, q, q, out, cu, cu, 200, 200, ws=ws)
    assert sage.device_status(ws) == sage.ERR_INVALID_ARG


def test_inconsistent_cu_seqlens_reported_packed_lists(sage):
    """The same with sizes for which the prologue's work lists run over the
    sequences' own tiles (a declared maximum far above the mean length): the
    offsets are checked on the device and the call reports them."""
    q = torch.randn(300, 2, 64, dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, 100, 50, 150, 300], dtype=torch.int32, device="cuda")  # 100 > 50
    out = torch.zeros(300, 2, 64, device="cuda")
    ws = sage.alloc_workspace(sage.workspace_bytes_varlen(4, 300, 300, 2, 2, 64))
    sage.attn_fwd_varlen(q, q, q, out, cu, cu, 1000, 1000, ws=ws)
    assert sage.device_status(ws) == sage.ERR_INVALID_ARG


# ------------------------------------------------- the prologue's two-launch plan
# The prologue can also run as two launches (Q tiles and K/V statistics,
# then K/V tiles); the automatic plan is one launch.  A test hook forces either
# plan, so the
# small shapes check the two-launch plan bit-exactly against the oracle and
# the bench shape checks that both plans write identical workspaces.
TWO_LAUNCH = ["d1", "d128_ragged", "d80", "causal_lq_gt_lk", "gqa_nhd", "varlen_small",
              "varlen_empty_keys"]


@pytest.fixture
def two_launches(sage):
    sage.set_prologue_launches(2)
    yield
    sage.set_prologue_launches(0)


@pytest.mark.parametrize("name", TWO_LAUNCH)
def test_two_launch_prologue_bit_exact(sage, orc, two_launches, name):
    w = next(x for x in SMALL if x.name == name)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    before = sage.launch_count()
    _, ws = _check_prologue(sage, orc, w, inp, d)
    assert sage.launch_count() - before == (2 if max(wl_lk(w)) > 0 else 1)
    out = H.run_attention(sage, w, d).cpu().numpy()
    samples = [(s, (0, w.Hq), (0, lq)) for s, (lq, lk) in enumerate(w.seg_lengths()) if lq > 0]
    worst, cmin = _check_rows(orc, w, inp, out, samples, ws.oracle)
    assert worst <= H.ATOL_ORACLE, worst
    assert cmin >= H.COS_EXACT, cmin


def wl_lk(w):
    return [lk for lq, lk in w.seg_lengths()]


def _workspace_fields(sage, qt):
    nstat = qt.nseg * qt.Hkv * qt.Dp
    shapes = {"q16": (torch.int16, (qt.q_rows, qt.Dp)), "k16": (torch.int16, (qt.k_rows, qt.Dp)),
              "v8": (torch.uint8, (qt.v_rows, qt.v_cols)), "s_q": (torch.float32, (qt.q_rows,)),
              "s_k": (torch.float32, (qt.k_rows // 128,)), "s_v": (torch.float32, (nstat,)),
              "k_mean": (torch.float32, (nstat,))}
    return {f: sage.ws_view(qt, f, dt, sh).clone() for f, (dt, sh) in shapes.items()}


def test_prologue_plans_agree_at_bench_size(sage):
    w = wl.WORKLOADS["b2_h24_l4096_d128"]
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    got = []
    for n in (1, 2):
        sage.set_prologue_launches(n)
        try:
            before = sage.launch_count()
            qt = H.run_prologue(sage, w, d)
            torch.cuda.synchronize()
            assert sage.launch_count() - before == n
            assert sage.device_status(qt._ws) == sage.OK
            got.append(_workspace_fields(sage, qt))
        finally:
            sage.set_prologue_launches(0)
    for f in got[0]:
        assert torch.equal(got[0][f], got[1][f]), f
