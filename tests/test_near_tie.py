"""The parity tests' near-tie criterion (helpers.near_tie_rows), on the CPU.

A row of the 96-sequence packed stress shape (segment 15, query head 1, row
12) has a key whose 448 P in the oracle's arithmetic is 183.99998, next to
the e4m3 rounding boundary 184 (the midpoint of 176 and 192): an exp2 a few
ulp away from the oracle's rounds that P~ code the other way.  The criterion
must flag that row and almost no other."""
import numpy as np
import pytest

from quantized_attention_smooth_gb300 import workloads as wl
from tests import helpers as H


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _segment_15(orc):
    from tests.test_gpu_parity import SMALL
    w = [x for x in SMALL if x.name == "varlen_many"][0]
    inp = wl.make_inputs(w)
    q, k, v = wl.segment(w, inp, 15)
    return w, orc.prologue(q, k, v, w.dtype)


def test_the_stress_row_is_a_near_tie(orc):
    w, pro = _segment_15(orc)
    assert H.near_tie_rows(orc, pro, 1, [12], w.causal, wl.default_sm_scale(w)) == [True]


def test_near_ties_are_rare(orc):
    w, pro = _segment_15(orc)
    flags = H.near_tie_rows(orc, pro, 1, list(range(pro["Lq"])), w.causal,
                            wl.default_sm_scale(w))
    assert sum(flags) <= 3, sum(flags)


def test_boundary_values_are_flagged_and_others_not(orc):
    """The e4m3 encoder changes code across the window only at a rounding
    boundary (the midpoint of two neighbouring e4m3 values: 184 between 176
    and 192, 100 between 96 and 104), not at the representable values."""
    f32 = np.float32
    for v, tie in ((184.0, True), (176.0, False), (192.0, False), (100.0, True),
                   (104.0, False), (96.0, False)):
        x = f32(v)
        lo = orc.e4m3_encode(np.array([x * (1.0 - H.NEAR_TIE)], f32))
        hi = orc.e4m3_encode(np.array([x * (1.0 + H.NEAR_TIE)], f32))
        assert bool(lo[0] != hi[0]) == tie, v
