"""The allocation-free statistics entry point, sage_kv_stats_noalloc.

Some callers may not allocate device memory at all, not even a workspace:
code running inside a host framework that owns every device allocation and
forbids its extensions to allocate, or a latency-critical loop that cannot
pay for cudaMalloc's implicit device synchronisation.  This entry point keeps
its scratch accumulators in a static device array inside the library.

The test calls it on several problems in a row (a large one, then smaller
ones, so stale accumulators from an earlier call would show), one of them
with a head dimension that forces element-wise loads (D=100) and one whose
channels are padded (D=40, padded to 64), and compares every result, bit for
bit, with the K channel means and V channel scales written by the
workspace-based prologue; padded channels must be exactly zero and the
call's device status word must read OK.  This file is named so that pytest
collects it last.
"""
import numpy as np
import pytest

from quantized_attention_smooth_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _case(name, B, Hkv, Lk, D, dtype, layout, seed):
    w = wl.Workload(name, B=B, Hq=Hkv, Hkv=Hkv, Lq=128, Lk=Lk, D=D, dtype=dtype,
                    layout=layout, causal=False, seed=seed, k_offset_sigma=3.0)
    inp = wl.make_inputs(w)
    dt = torch.float16 if dtype == wl.F16 else torch.bfloat16

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt).cuda()

    return w, dev(inp["q"]), dev(inp["k"]), dev(inp["v"])


CASES = [
    ("b2_h24_l4096_d128", 2, 24, 4096, 128, wl.F16, wl.HND, 1101),
    ("b3_h4_l1000_d80_nhd", 3, 4, 1000, 80, wl.BF16, wl.NHD, 1102),
    ("b1_h3_l777_d100_nhd_elementwise", 1, 3, 777, 100, wl.F16, wl.NHD, 1103),
    ("b2_h2_l300_d40_padded", 2, 2, 300, 40, wl.BF16, wl.HND, 1104),
]


def test_noalloc_statistics_match_the_prologue_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_smooth_gb300 import sage
    for name, B, Hkv, Lk, D, dtype, layout, seed in CASES:
        w, q, k, v = _case(name, B, Hkv, Lk, D, dtype, layout, seed)
        lay = "HND" if layout == wl.HND else "NHD"
        Dp = 64 if D <= 64 else 128
        n = B * Hkv * Dp
        qt = sage.quant_prologue(q, k, v, lay)             # workspace-based path
        ref_mean = sage.ws_view(qt, "k_mean", torch.float32, (n,)).clone()
        ref_sv = sage.ws_view(qt, "s_v", torch.float32, (n,)).clone()
        k_mean = torch.full((n,), float("nan"), device="cuda")
        s_v = torch.full((n,), float("nan"), device="cuda")
        sage.kv_stats_noalloc(k, v, lay, k_mean, s_v)
        assert sage.kv_stats_noalloc_status() == sage.OK, (name, sage.last_error())
        assert torch.equal(k_mean.view(torch.int32), ref_mean.view(torch.int32)), name
        assert torch.equal(s_v.view(torch.int32), ref_sv.view(torch.int32)), name
        if Dp > D:                                          # padded channels
            assert torch.all(k_mean.view(B * Hkv, Dp)[:, D:] == 0), name
            assert torch.all(s_v.view(B * Hkv, Dp)[:, D:] == 0), name


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_smooth_gb300 import sage
    k = torch.zeros(2, 65, 8, 128, dtype=torch.float16, device="cuda")   # 2*65*128 > 16384
    out = torch.zeros(2 * 65 * 128, device="cuda")
    with pytest.raises(sage.SageError, match="static scratch"):
        sage.kv_stats_noalloc(k, k, "HND", out, out)
