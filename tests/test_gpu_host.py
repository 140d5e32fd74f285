"""The host-buffer call (sage_attn_fwd_host): q, k, v and out in page-locked
host memory, chunked and pipelined by the library.  Attention never mixes
heads or batch entries, so its output must equal sage_attn_fwd's bit for bit
on the same inputs, whatever the chunking."""
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
    base = dict(B=2, Hq=4, Hkv=2, Lq=300, Lk=333, D=128, dtype=wl.F16, layout=wl.HND,
                causal=False, seed=900, k_offset_sigma=2.0)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    (_w("hnd_chunk1"), 1),
    (_w("hnd_auto"), 0),
    (_w("nhd_bf16_gqa_causal", B=3, Hq=6, Hkv=3, Lq=256, Lk=256, layout=wl.NHD,
        dtype=wl.BF16, causal=True, seed=901), 2),          # 2 does not divide 3
    (_w("d40_ragged_nhd", B=1, Hq=2, Hkv=2, Lq=130, Lk=700, D=40, layout=wl.NHD, seed=902), 1),
    (_w("hnd_causal_lq_lt_lk", B=2, Hq=2, Hkv=1, Lq=200, Lk=450, D=64, causal=True,
        seed=903), 0),
]


def _host(x):
    return x.cpu().pin_memory()


def _compare(sage, w, chunk):
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    lay = "HND" if w.layout == wl.HND else "NHD"
    scale = wl.default_sm_scale(w)
    ref = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    sage.attn_fwd(d["q"], d["k"], d["v"], ref, lay, w.causal, scale)
    hq, hk, hv = _host(d["q"]), _host(d["k"]), _host(d["v"])
    out = torch.full(hq.shape, float("nan"), dtype=torch.float32).pin_memory()
    sage.attn_fwd_host(hq, hk, hv, out, lay, w.causal, scale, chunk_kv_heads=chunk)
    torch.cuda.synchronize()
    assert torch.equal(out, ref.cpu())


@pytest.mark.parametrize("w,chunk", CASES, ids=[w.name for w, _ in CASES])
def test_host_call_equals_device_call(sage, w, chunk):
    _compare(sage, w, chunk)


def test_host_call_at_bench_size(sage):
    _compare(sage, wl.WORKLOADS["b2_h24_l4096_d128"], 0)


def test_host_call_pv16_equals_device_call(sage):
    w = _w("pv16_nhd_bf16", B=2, Hq=4, Hkv=2, Lq=300, Lk=333, layout=wl.NHD, dtype=wl.BF16,
           seed=904)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    scale = wl.default_sm_scale(w)
    ref = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    sage.attn_fwd_pv16(d["q"], d["k"], d["v"], ref, "NHD", w.causal, scale)
    hq, hk, hv = _host(d["q"]), _host(d["k"]), _host(d["v"])
    out = torch.full(hq.shape, float("nan"), dtype=torch.float32).pin_memory()
    sage.attn_fwd_host(hq, hk, hv, out, "NHD", w.causal, scale, chunk_kv_heads=1, pv16=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref.cpu())


def test_failure_in_an_early_chunk_stays_visible(sage):
    """A bounded wait that runs out in the first of four chunks (the library's
    failure-injection hook, limited to one attention launch) must still show
    in the workspace's status word after the later chunks have run; the next
    call clears it."""
    w = _w("fault_chunks", B=2, Hq=4, Hkv=2, Lq=256, Lk=384, seed=905)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    hq, hk, hv = _host(d["q"]), _host(d["k"]), _host(d["v"])
    out = torch.empty(hq.shape, dtype=torch.float32).pin_memory()
    ws = sage.alloc_workspace(sage.workspace_bytes_host(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, 1))
    scale = wl.default_sm_scale(w)
    try:
        sage.set_fault(skip_kv_tile=1, timeout_ns=50_000_000, launches=1)
        sage.attn_fwd_host(hq, hk, hv, out, "HND", False, scale, ws=ws, chunk_kv_heads=1)
        status = sage.device_status(ws)                    # synchronises
    finally:
        sage.set_fault(-1, 0)
    assert status == sage.ERR_DEVICE_TIMEOUT
    sage.attn_fwd_host(hq, hk, hv, out, "HND", False, scale, ws=ws, chunk_kv_heads=1)
    assert sage.device_status(ws) == sage.OK


@pytest.mark.parametrize("fail_at", [0, 1, 3])
def test_failed_chunk_leaves_earlier_chunks_complete(sage, fail_at):
    """A chunk that fails (the library's test hook) ends the host-buffer call
    with an error.  The caller's stream still waits for the earlier chunks'
    copies: once it is synchronised their rows are in host memory, equal to
    the device call's, and no later row was written; the next call runs
    normally.  Chunk c of B=2, Hkv=2 at one kv head per chunk is batch entry
    c // 2, query heads 2 (c % 2) and 2 (c % 2) + 1."""
    w = _w("fail_chunk", Lq=256, Lk=384, seed=906)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    scale = wl.default_sm_scale(w)
    ref = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    sage.attn_fwd(d["q"], d["k"], d["v"], ref, "HND", False, scale)
    ref = ref.cpu()
    hq, hk, hv = _host(d["q"]), _host(d["k"]), _host(d["v"])
    out = torch.full(hq.shape, float("nan"), dtype=torch.float32).pin_memory()
    try:
        sage.set_host_fail_chunk(fail_at)
        with pytest.raises(sage.SageError) as err:
            sage.attn_fwd_host(hq, hk, hv, out, "HND", False, scale, chunk_kv_heads=1)
    finally:
        sage.set_host_fail_chunk(-1)
    assert err.value.status == sage.ERR_INVALID_ARG
    torch.cuda.current_stream().synchronize()
    for c in range(4):
        b, h0 = c // 2, 2 * (c % 2)
        rows = out[b, h0:h0 + 2]
        if c < fail_at:
            assert torch.equal(rows, ref[b, h0:h0 + 2]), c
        else:
            assert torch.isnan(rows).all(), c
    sage.attn_fwd_host(hq, hk, hv, out, "HND", False, scale, chunk_kv_heads=1)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def _vw(name, lq, lk, **kw):
    base = dict(B=0, Hq=4, Hkv=2, Lq=0, Lk=0, D=64, dtype=wl.F16, layout=wl.NHD,
                causal=False, seed=910, k_offset_sigma=1.5, seqlens_q=lq, seqlens_k=lk)
    base.update(kw)
    return wl.Workload(name, **base)


VARLEN_CASES = [
    (_vw("varlen_d40_ragged", (1, 130, 257, 128), (5, 128, 300, 1), D=40), 1),
    (_vw("varlen_bf16_gqa_causal", (200, 64, 333), (200, 64, 333), Hq=6, Hkv=3, D=128,
         dtype=wl.BF16, causal=True, seed=911), 2),            # 2 does not divide 3
    (_vw("varlen_empty_key_sequence", (130, 7, 256), (140, 0, 129), D=80, seed=912), 0),
    (_vw("varlen_many_sequences", tuple(int(x) for x in np.random.default_rng(914).integers(1, 300, 80)),
         tuple(int(x) for x in np.random.default_rng(915).integers(0, 300, 80)), Hq=6, Hkv=3,
         seed=914), 0),
]


def _compare_varlen(sage, w, chunk):
    """sage_attn_fwd_varlen_host against sage_attn_fwd_varlen on the same
    packed inputs: equal bit for bit, and nothing left in the status word."""
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    ref = H.run_attention(sage, w, d)
    hq, hk, hv = _host(d["q"]), _host(d["k"]), _host(d["v"])
    out = torch.full(hq.shape, float("nan"), dtype=torch.float32).pin_memory()
    cu_q, cu_k = torch.from_numpy(inp["cu_q"]), torch.from_numpy(inp["cu_k"])
    ws = sage.alloc_workspace(sage.workspace_bytes_varlen_host(
        w.nseg, sum(w.seqlens_q), sum(w.seqlens_k), w.Hq, w.Hkv, w.D, chunk))
    sage.attn_fwd_varlen_host(hq, hk, hv, out, cu_q, cu_k, max(w.seqlens_q), max(w.seqlens_k),
                              w.causal, wl.default_sm_scale(w), chunk_kv_heads=chunk, ws=ws)
    assert sage.device_status(ws) == sage.OK                # synchronises
    assert torch.equal(out, ref.cpu())


@pytest.mark.parametrize("w,chunk", VARLEN_CASES, ids=[w.name for w, _ in VARLEN_CASES])
def test_varlen_host_call_equals_device_call(sage, w, chunk):
    _compare_varlen(sage, w, chunk)


def test_varlen_host_call_at_full_size(sage):
    _compare_varlen(sage, wl.WORKLOADS["varlen_d80"], 0)


def test_varlen_failure_in_an_early_chunk_stays_visible(sage):
    """The packed call keeps the status word across chunks as the dense one
    does: a bounded wait that runs out in the first of two chunks shows after
    the call, and the next call clears it."""
    w = _vw("varlen_fault_chunks", (300, 200), (400, 260), Hq=2, Hkv=2, seed=913)
    inp = wl.make_inputs(w)
    d = H.device_inputs(w, inp)
    hq, hk, hv = _host(d["q"]), _host(d["k"]), _host(d["v"])
    out = torch.empty(hq.shape, dtype=torch.float32).pin_memory()
    cu_q, cu_k = torch.from_numpy(inp["cu_q"]), torch.from_numpy(inp["cu_k"])
    ws = sage.alloc_workspace(sage.workspace_bytes_varlen_host(2, 500, 660, 2, 2, w.D, 1))
    scale = wl.default_sm_scale(w)
    try:
        sage.set_fault(skip_kv_tile=1, timeout_ns=50_000_000, launches=1)
        sage.attn_fwd_varlen_host(hq, hk, hv, out, cu_q, cu_k, 300, 400, False, scale,
                                  chunk_kv_heads=1, ws=ws)
        status = sage.device_status(ws)                    # synchronises
    finally:
        sage.set_fault(-1, 0)
    assert status == sage.ERR_DEVICE_TIMEOUT
    sage.attn_fwd_varlen_host(hq, hk, hv, out, cu_q, cu_k, 300, 400, False, scale,
                              chunk_kv_heads=1, ws=ws)
    assert sage.device_status(ws) == sage.OK
