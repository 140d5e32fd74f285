"""The tensor-rate measurement the benchmark divides by (sage_debug_tc_rate):
back-to-back M=128 N=128 tcgen05 MMAs of the attention kernel's two kinds on
every SM.  An e4m3 MMA (K=32) does twice the work of an fp16 one (K=16) in
about the same time on this tensor core, and the rates sit in the range of
the chip's dense 16-bit / 8-bit figures; the bounded wait never runs out."""
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_tensor_rates_are_measured_and_plausible():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    from quantized_attention_smooth_gb300 import sage
    stream = torch.cuda.current_stream()
    rates = bench.tensor_rates(torch, sage, stream, torch.device("cuda", 0), n_mma=1 << 13,
                               reps=3)
    r16, r8 = rates[0], rates[1]
    assert 500.0 < r16 < 5000.0, r16          # TFLOP/s
    assert 1.6 < r8 / r16 < 2.4, (r16, r8)


def test_tensor_rate_call_refuses_bad_arguments():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_smooth_gb300 import sage
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(sage.SageError, match="kind"):
        sage.debug_tc_rate(2, 16, status)
    with pytest.raises(sage.SageError, match="n_mma"):
        sage.debug_tc_rate(0, 0, status)
