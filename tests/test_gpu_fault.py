"""Device-side failure detection without a GPU fault.

The attention kernel's waits are bounded.  The library's failure-injection
hook makes the K producer skip one key tile, so the tensor-core issuer waits
for a tile that never arrives; after the (here short) limit the kernel must
raise the workspace status word, drain its copies and MMAs, release its
tensor memory and exit, leaving the context usable.  Nothing here traps,
faults or hangs the GPU: every wait involved ends by its limit."""
from __future__ import annotations

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


def _inputs():
    w = wl.Workload("fault", B=1, Hq=2, Hkv=2, Lq=512, Lk=512, D=64, dtype=wl.F16,
                    layout=wl.HND, causal=False, seed=91, k_offset_sigma=2.0)
    return w, H.device_inputs(w, wl.make_inputs(w))


def test_wait_that_runs_out_is_reported_and_the_context_recovers(sage):
    w, d = _inputs()
    scale = wl.default_sm_scale(w)
    ws = sage.alloc_workspace(sage.workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D))
    good = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    sage.attn_fwd(d["q"], d["k"], d["v"], good, "HND", False, scale, ws=ws)
    torch.cuda.synchronize()
    assert sage.device_status(ws) == sage.OK

    qt = sage.quant_prologue(d["q"], d["k"], d["v"], "HND", ws=ws)
    out = torch.zeros_like(good)
    try:
        sage.set_fault(skip_kv_tile=1, timeout_ns=50_000_000)      # 50 ms limit
        sage.attn_quantized(qt, out, "HND", False, scale)
        status = sage.device_status(ws)                            # synchronises
    finally:
        sage.set_fault(-1, 0)
    assert status == sage.ERR_DEVICE_TIMEOUT

    # the context is still usable: the same call now succeeds and gives the
    # same output as before the failure
    again = torch.empty_like(good)
    sage.attn_fwd(d["q"], d["k"], d["v"], again, "HND", False, scale, ws=ws)
    torch.cuda.synchronize()
    assert sage.device_status(ws) == sage.OK
    assert torch.equal(again, good)
