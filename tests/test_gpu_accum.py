"""Precision of the FP8 PV accumulator, measured through the attention
kernel's own PV instructions (sage_debug_pv_accum: tcgen05 kind::f8f6f4,
e4m3 x e4m3, M=128, N=Dp, K=32 per instruction, accumulating in tensor
memory).

The stable-diffusion.cpp "SageAttention" kernel table pairs the FP8 PV
products with an FP32 buffer; these tests state what the tensor core's own
accumulator actually keeps, against exact sums computed on the host (every
product of two e4m3 values is a multiple of 2^-18 below 2^18, so float64
sums of up to 2^15 of them are exact):

* a 24-bit significand (the fp32 width): a product 2^-s of the largest
  addend survives exactly for every s <= 23, in the same instruction, in the
  next instruction and in the next key tile;
* inside one instruction the addends are aligned to the largest one with 25
  fraction bits: parts below 2^-25 of it are dropped, and the sum is cut
  (not rounded) to 24 bits;
* over long key spans the error stays within what those two rules allow
  per instruction (2^-19 of its largest addend plus 2^-22 of its result),
  summed over the instructions: at 32768 keys that is ~1e-5 of the output,
  far below the e4m3 quantisation error of P~ and V.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sage():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_attention_smooth_gb300 import sage as s
    return s


def _e4m3_values():
    v = np.zeros(256)
    for c in range(256):
        e, m = (c >> 3) & 15, c & 7
        mag = m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10)
        v[c] = -mag if c & 0x80 else mag
    v[0x7F] = v[0xFF] = np.nan
    return v


E4M3 = _e4m3_values()


def _pow2(e):
    """e4m3 code of 2^e, -9 <= e <= 8."""
    return (e + 7) << 3 if e >= -6 else 1 << (e + 9)


def _run(sage, p, v):
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = sage.debug_pv_accum(torch.from_numpy(np.ascontiguousarray(p)).cuda(),
                              torch.from_numpy(np.ascontiguousarray(v)).cuda(), status)
    torch.cuda.synchronize()
    assert sage.device_status(status) == sage.OK, sage.last_error()
    return out.cpu().numpy().astype(np.float64)


def _exact(p, v):
    return np.einsum("trj,tcj->rc", E4M3[p], E4M3[v])


DP = 128
ROW_EXP = np.array([8 - (r % 18) for r in range(128)])     # 2^a on row r
COL_EXP = np.array([8 - (c % 18) for c in range(DP)])      # 2^b on column c


@pytest.mark.parametrize("place", [(0, 1, 0), (1, 0, 0), (0, 31, 0), (0, 32, 0), (0, 127, 0),
                                   (0, 1, 1)],
                         ids=["same_instr", "small_first", "same_instr_last", "next_instr",
                              "last_instr", "next_tile"])
@pytest.mark.parametrize("sign", [1, -1], ids=["plus", "minus"])
def test_single_small_addend_kept_to_24_bits(sage, place, sign):
    """2^16 + sign*2^(16-s): exact for s <= 23, within one unit of the last
    of 24 bits beyond."""
    kb, ks, ts = place
    p = np.zeros((ts + 1, 128, 128), np.uint8)
    v = np.zeros((ts + 1, DP, 128), np.uint8)
    p[0, :, kb] = _pow2(8)
    v[0, :, kb] = _pow2(8)
    p[ts, :, ks] = [_pow2(int(a)) for a in ROW_EXP]
    v[ts, :, ks] = [_pow2(int(b)) | (0x80 if sign < 0 else 0) for b in COL_EXP]
    hw, ex = _run(sage, p, v), _exact(p, v)
    s = 16 - (ROW_EXP[:, None] + COL_EXP[None, :])
    keep = s <= 23
    assert np.array_equal(hw[keep], ex[keep]), "a product >= 2^-23 of the largest was not kept"
    assert np.all(np.abs(hw[~keep] - ex[~keep]) <= 2.0 ** -7)


@pytest.mark.parametrize("s", range(18, 30))
def test_small_addends_aligned_then_truncated(sage, s):
    """One product 2^16 and 31 products 2^(16-s) in one instruction: the
    small ones count only while 2^(16-s) >= 2^-9 (25 fraction bits below the
    leading bit), and their sum is cut to the 24-bit grid of 2^16 (2^-7)."""
    a = 16 - s + 9
    a, b = (8, 16 - s - 8) if a > 8 else (a, -9)
    p = np.zeros((1, 128, 128), np.uint8)
    v = np.zeros((1, DP, 128), np.uint8)
    p[0, :, 0], v[0, :, 0] = _pow2(8), _pow2(8)
    p[0, :, 1:32], v[0, :, 1:32] = _pow2(a), _pow2(b)
    hw = _run(sage, p, v)
    small = 2.0 ** (16 - s)
    kept = 31 * small if small >= 2.0 ** -9 else 0.0
    model = 65536.0 + np.floor(kept / 2.0 ** -7) * 2.0 ** -7
    assert np.all(hw == model), (s, hw[0, 0], model)


def _random_codes(rng, shape, scale, signed):
    """e4m3 codes of seeded values (round to nearest on the code grid)."""
    x = rng.standard_normal(shape) * scale if signed else rng.random(shape) ** 4 * scale
    finite = np.array([c for c in range(127) if np.isfinite(E4M3[c])])
    mags = E4M3[finite]
    order = np.argsort(mags)
    mags, finite = mags[order], finite[order]
    idx = np.clip(np.searchsorted(mags, np.abs(x)), 1, len(mags) - 1)
    lo = np.abs(x) - mags[idx - 1] <= mags[idx] - np.abs(x)
    code = np.where(lo, finite[idx - 1], finite[idx]).astype(np.uint8)
    return code | ((x < 0) * 0x80).astype(np.uint8)


@pytest.mark.parametrize("ntiles", [1, 8, 64, 256])
def test_long_key_span_error_bound(sage, ntiles):
    """Softmax-like P~ in [0, 448] and signed V over up to 32768 keys: the
    accumulated error is within 2^-19 of each instruction's largest addend
    (running sum or product) plus 2^-22 of its result, summed over the
    instructions."""
    rng = np.random.default_rng(1000 + ntiles)
    p = _random_codes(rng, (ntiles, 128, 128), 448.0, False)
    v = _random_codes(rng, (ntiles, DP, 128), 100.0, True)
    hw = _run(sage, p, v)
    P, V = E4M3[p], E4M3[v]
    # per instruction i (32 keys): exact partial sums [i][row][col], and an
    # upper bound of its largest product, max|P| x max|V| over its keys
    Pi = np.moveaxis(P.reshape(ntiles, 128, 4, 32), 2, 1).reshape(ntiles * 4, 128, 32)
    Vi = np.moveaxis(V.reshape(ntiles, DP, 4, 32), 2, 1).reshape(ntiles * 4, DP, 32)
    part = np.einsum("irk,ick->irc", Pi, Vi)
    acc = np.cumsum(part, axis=0)
    prev = np.concatenate([np.zeros((1, 128, DP)), acc[:-1]], axis=0)
    top = np.abs(Pi).max(axis=2)[:, :, None] * np.abs(Vi).max(axis=2)[:, None, :]
    # per instruction: < 33 x 2^-25 of the largest addend from the alignment,
    # plus the cut of the result to 24 bits (< 2^-23 of it; 2^-22 for slack)
    bound = (2.0 ** -19 * np.maximum(np.abs(prev), top) + 2.0 ** -22 * np.abs(acc)).sum(axis=0)
    err = np.abs(hw - acc[-1])
    assert np.all(err <= bound), float(np.max(err / bound))
    assert np.all(np.isfinite(hw))
