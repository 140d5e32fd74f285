"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module holds shapes and random-number recipes only: no step of the
quantized-attention method lives here.  Both the CUDA path and the CPU oracle
receive the very same bits produced below.

Recipe: numpy PCG64 seeded per workload; q, k, v ~ N(0, 1) drawn in float32;
k gets a per-channel offset that is shared by every token (either drawn from
N(0, sigma) per channel, or a fixed value on a few outlier channels); the sum
is rounded once to fp16 or bf16.  Varlen workloads draw their sequence
lengths uniformly from a closed range with their own seed.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

F16, BF16 = 0, 1
HND, NHD = 0, 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                     # batch (ignored when seqlens is set)
    Hq: int
    Hkv: int
    Lq: int                    # per-batch lengths (ignored when seqlens is set)
    Lk: int
    D: int
    dtype: int                 # F16 or BF16
    layout: int                # HND or NHD (varlen is always packed (T, H, D))
    causal: bool
    seed: int
    k_offset_sigma: float = 0.0          # per-channel N(0, sigma) offset on k
    k_outliers: tuple = ()               # channels that get +k_outlier_value
    k_outlier_value: float = 0.0
    sm_scale: float | None = None        # None: 1/sqrt(D)
    seqlens_q: tuple | None = None       # varlen: packed sequences
    seqlens_k: tuple | None = None

    @property
    def varlen(self) -> bool:
        return self.seqlens_q is not None

    @property
    def nseg(self) -> int:
        return len(self.seqlens_q) if self.varlen else self.B

    def seg_lengths(self):
        if self.varlen:
            return list(zip(self.seqlens_q, self.seqlens_k))
        return [(self.Lq, self.Lk)] * self.B

    def ops(self, dim: int | None = None, causal_effective: bool = False) -> float:
        """4*Lq*Lk*D per (segment, head); causal_effective halves Lq*Lk."""
        d = self.D if dim is None else dim
        tot = 0.0
        for lq, lk in self.seg_lengths():
            pairs = lq * lk
            if self.causal and causal_effective:
                pairs = sum(min(i + 1, lk) for i in range(lq)) if lq <= 4096 else \
                    _causal_pairs(lq, lk)
            tot += 4.0 * self.Hq * pairs * d
        return tot

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _causal_pairs(lq: int, lk: int) -> int:
    # sum_{i<lq} min(i+1, lk)
    a = min(lq, lk)
    s = a * (a + 1) // 2
    if lq > lk:
        s += (lq - lk) * lk
    return s


def _varlen_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


_C5_LENS = _varlen_lengths(1005, 8, 1024, 16384)

# The five workloads: a small smoke case, the RTX 5070 measurement shape,
# causal GQA prefill, video-DiT self/cross attention, and the padding/varlen
# stress case.
WORKLOADS = {
    "small_d64": Workload("small_d64", B=1, Hq=2, Hkv=2, Lq=256, Lk=256, D=64,
                          dtype=F16, layout=HND, causal=False, seed=1001,
                          k_offset_sigma=2.0, sm_scale=1.0 / 8.0),
    "b2_h24_l4096_d128": Workload("b2_h24_l4096_d128", B=2, Hq=24, Hkv=24,
                                  Lq=4096, Lk=4096, D=128, dtype=F16,
                                  layout=HND, causal=False, seed=1002,
                                  k_offset_sigma=3.0),
    "gqa_causal_b4_l8192": Workload("gqa_causal_b4_l8192", B=4, Hq=32, Hkv=8,
                                    Lq=8192, Lk=8192, D=128, dtype=BF16,
                                    layout=NHD, causal=True, seed=1003,
                                    k_outliers=(7, 42, 77, 119),
                                    k_outlier_value=15.0),
    "dit_self_l32768": Workload("dit_self_l32768", B=1, Hq=40, Hkv=40,
                                Lq=32768, Lk=32768, D=128, dtype=BF16,
                                layout=HND, causal=False, seed=1004,
                                k_offset_sigma=4.0),
    "dit_cross_l32768x512": Workload("dit_cross_l32768x512", B=1, Hq=40,
                                     Hkv=40, Lq=32768, Lk=512, D=128,
                                     dtype=BF16, layout=HND, causal=False,
                                     seed=1004, k_offset_sigma=4.0),
    "varlen_d80": Workload("varlen_d80", B=0, Hq=16, Hkv=16, Lq=0, Lk=0, D=80,
                           dtype=F16, layout=NHD, causal=False, seed=1005,
                           k_outliers=(5, 33, 61, 79), k_outlier_value=20.0,
                           seqlens_q=_C5_LENS, seqlens_k=_C5_LENS),
    "varlen_d40": Workload("varlen_d40", B=0, Hq=16, Hkv=16, Lq=0, Lk=0, D=40,
                           dtype=F16, layout=NHD, causal=False, seed=1005,
                           k_outliers=(3, 17, 29, 38), k_outlier_value=20.0,
                           seqlens_q=_C5_LENS, seqlens_k=_C5_LENS),
}


def to_bits(x32: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 to fp16/bf16 (nearest even) and return the uint16 bits."""
    if dtype == F16:
        return x32.astype(np.float16).view(np.uint16)
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_float(bits: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def make_inputs(w: Workload) -> dict:
    """q, k, v as uint16 bit arrays in the workload's caller layout.

    Dense HND: (B, H, L, D); dense NHD: (B, L, H, D); varlen: packed (T, H, D)
    with int32 cu_seqlens.
    """
    rng = np.random.default_rng(w.seed)
    if w.varlen:
        Tq, Tk = sum(w.seqlens_q), sum(w.seqlens_k)
        qs, ks = (Tq, w.Hq, w.D), (Tk, w.Hkv, w.D)
    elif w.layout == HND:
        qs, ks = (w.B, w.Hq, w.Lq, w.D), (w.B, w.Hkv, w.Lk, w.D)
    else:
        qs, ks = (w.B, w.Lq, w.Hq, w.D), (w.B, w.Lk, w.Hkv, w.D)
    q = rng.standard_normal(qs, dtype=np.float32)
    k = rng.standard_normal(ks, dtype=np.float32)
    v = rng.standard_normal(ks, dtype=np.float32)
    off = np.zeros(w.D, dtype=np.float32)
    if w.k_offset_sigma:
        off += rng.normal(0.0, w.k_offset_sigma, size=w.D).astype(np.float32)
    for c in w.k_outliers:
        off[c] += np.float32(w.k_outlier_value)
    k += off
    out = dict(q=to_bits(q, w.dtype), k=to_bits(k, w.dtype), v=to_bits(v, w.dtype))
    del q, k, v
    if w.varlen:
        out["cu_q"] = np.concatenate([[0], np.cumsum(w.seqlens_q)]).astype(np.int32)
        out["cu_k"] = np.concatenate([[0], np.cumsum(w.seqlens_k)]).astype(np.int32)
    return out


def segment(w: Workload, inp: dict, s: int):
    """One segment's q, k, v as [H, L, D] bit arrays (layout permutation only)."""
    if w.varlen:
        cq, ck = inp["cu_q"], inp["cu_k"]
        q = inp["q"][cq[s]:cq[s + 1]].transpose(1, 0, 2)
        k = inp["k"][ck[s]:ck[s + 1]].transpose(1, 0, 2)
        v = inp["v"][ck[s]:ck[s + 1]].transpose(1, 0, 2)
    elif w.layout == HND:
        q, k, v = inp["q"][s], inp["k"][s], inp["v"][s]
    else:
        q = inp["q"][s].transpose(1, 0, 2)
        k = inp["k"][s].transpose(1, 0, 2)
        v = inp["v"][s].transpose(1, 0, 2)
    return (np.ascontiguousarray(q), np.ascontiguousarray(k),
            np.ascontiguousarray(v))


def out_segment(w: Workload, out: np.ndarray, s: int, cu_q=None) -> np.ndarray:
    """View of one segment of a caller-layout output as [H, L, D]."""
    if w.varlen:
        return out[cu_q[s]:cu_q[s + 1]].transpose(1, 0, 2)
    if w.layout == HND:
        return out[s]
    return out[s].transpose(1, 0, 2)


def default_sm_scale(w: Workload) -> float:
    return w.sm_scale if w.sm_scale is not None else float(np.float32(1.0) / np.sqrt(np.float32(w.D)))
