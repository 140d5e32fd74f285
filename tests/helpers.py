"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
read the library's workspace back in the oracle's per-segment layout, and
compare outputs.  Nothing here computes a step of the method."""
from __future__ import annotations

import numpy as np

from quantized_attention_smooth_gb300 import workloads as wl

ATOL_ORACLE = 2e-3      # max-abs difference to the oracle (fp32 outputs)
COS_EXACT = 0.999       # cosine similarity to fp64 exact attention
# An element beyond ATOL_ORACLE is accepted only in a row where the oracle's
# own 448 P of some key lies within NEAR_TIE of an e4m3 rounding boundary: the
# kernel's exp2 (a few ulp from the oracle's) may round that P~ code the other
# way.  Such a flip moves the output by at most one e4m3 step of that key's
# weight times |v - o|; FLIP_CAP bounds what the tests accept.
NEAR_TIE = 2.0 ** -19
FLIP_CAP = 2e-2


def torch_dtype(dtype):
    import torch
    return torch.float16 if dtype == wl.F16 else torch.bfloat16


def to_device(bits: np.ndarray, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(dtype)).cuda()


def device_inputs(w: wl.Workload, inp: dict):
    import torch
    d = dict(q=to_device(inp["q"], w.dtype), k=to_device(inp["k"], w.dtype),
             v=to_device(inp["v"], w.dtype))
    if w.varlen:
        d["cu_q"] = torch.from_numpy(inp["cu_q"]).cuda()
        d["cu_k"] = torch.from_numpy(inp["cu_k"]).cuda()
    return d


def run_prologue(sage, w: wl.Workload, d: dict):
    if w.varlen:
        return sage.quant_prologue_varlen(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"],
                                          max(w.seqlens_q), max(w.seqlens_k))
    return sage.quant_prologue(d["q"], d["k"], d["v"], w.layout)


def out_tensor(w: wl.Workload, d: dict):
    import torch
    return torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device="cuda")


def workspace_for(sage, w: wl.Workload):
    if w.varlen:
        n = sage.workspace_bytes_varlen(w.nseg, sum(w.seqlens_q), sum(w.seqlens_k), w.Hq,
                                        w.Hkv, w.D)
    else:
        n = sage.workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D)
    return sage.alloc_workspace(n)


def run_attention(sage, w: wl.Workload, d: dict, out=None, ws=None):
    out = out_tensor(w, d) if out is None else out
    scale = wl.default_sm_scale(w)
    if w.varlen:
        sage.attn_fwd_varlen(d["q"], d["k"], d["v"], out, d["cu_q"], d["cu_k"],
                             max(w.seqlens_q), max(w.seqlens_k), w.causal, scale, ws=ws)
    else:
        sage.attn_fwd(d["q"], d["k"], d["v"], out, w.layout, w.causal, scale, ws=ws)
    return out


class Workspace:
    """The quantized tensors of a prologue call, on the host."""

    def __init__(self, sage, qt, w: wl.Workload, inp: dict):
        import torch
        self.w, self.qt = w, qt
        Dp = qt.Dp
        self.q16 = sage.ws_view(qt, "q16", torch.int16, (qt.q_rows, Dp)).cpu().numpy()
        self.k16 = sage.ws_view(qt, "k16", torch.int16, (qt.k_rows, Dp)).cpu().numpy()
        self.v8 = sage.ws_view(qt, "v8", torch.uint8, (qt.v_rows, qt.v_cols)).cpu().numpy()
        self.s_q = sage.ws_view(qt, "s_q", torch.float32, (qt.q_rows,)).cpu().numpy()
        self.s_k = sage.ws_view(qt, "s_k", torch.float32, (qt.k_rows // 128,)).cpu().numpy()
        nstat = qt.nseg * qt.Hkv * Dp
        self.s_v = sage.ws_view(qt, "s_v", torch.float32, (nstat,)).cpu().numpy().reshape(
            qt.nseg, qt.Hkv, Dp)
        self.k_mean = sage.ws_view(qt, "k_mean", torch.float32, (nstat,)).cpu().numpy().reshape(
            qt.nseg, qt.Hkv, Dp)
        self.cu_q = inp.get("cu_q")
        self.cu_k = inp.get("cu_k")

    def _base(self, s, cu, H, head_rows):
        if self.w.varlen:
            return 128 * (s + int(cu[s]) // 128)
        return s * H * head_rows

    def segment(self, s):
        """Quantized tensors of segment s in the oracle's layout."""
        qt, w = self.qt, self.w
        Dp = qt.Dp
        lens = w.seg_lengths()[s]
        Lq, Lk = lens
        qb = self._base(s, self.cu_q, qt.Hq, qt.q_head_rows)
        kb = self._base(s, self.cu_k, qt.Hkv, qt.k_head_rows)
        qrows = np.stack([np.arange(Lq) + qb + h * qt.q_head_rows for h in range(qt.Hq)])
        krows = np.stack([np.arange(Lk) + kb + h * qt.k_head_rows for h in range(qt.Hkv)])
        q8 = self.q16[qrows].view(np.float16).astype(np.float32)
        k8 = self.k16[krows].view(np.float16).astype(np.float32)
        assert np.all(q8 == np.rint(q8)) and np.all(k8 == np.rint(k8))
        nkb = (Lk + 127) // 128
        sk_idx = np.stack([(kb + h * qt.k_head_rows) // 128 + np.arange(nkb)
                           for h in range(qt.Hkv)])
        vrow0 = 0 if w.varlen else s * qt.Hkv * Dp
        vcol0 = kb if w.varlen else 0
        v8 = np.stack([self.v8[vrow0 + h * Dp: vrow0 + (h + 1) * Dp, vcol0: vcol0 + Lk].T
                       for h in range(qt.Hkv)])
        return dict(q8=q8.astype(np.int8), s_q=self.s_q[qrows], k8=k8.astype(np.int8),
                    s_k=self.s_k[sk_idx], v8=np.ascontiguousarray(v8), s_v=self.s_v[s],
                    k_mean=self.k_mean[s], qrows=qrows, krows=krows)

    def padding_is_zero(self, s):
        """Every row of the 128-token tiles past the segment end is zero."""
        qt, w = self.qt, self.w
        Lq, Lk = w.seg_lengths()[s]
        qb = self._base(s, self.cu_q, qt.Hq, qt.q_head_rows)
        kb = self._base(s, self.cu_k, qt.Hkv, qt.k_head_rows)
        ok = True
        for h in range(qt.Hq):
            r0 = qb + h * qt.q_head_rows
            ok &= bool(np.all(self.q16[r0 + Lq: r0 + (Lq + 127) // 128 * 128] == 0))
            ok &= bool(np.all(self.s_q[r0 + Lq: r0 + (Lq + 127) // 128 * 128] == 0))
        for h in range(qt.Hkv):
            r0 = kb + h * qt.k_head_rows
            ok &= bool(np.all(self.k16[r0 + Lk: r0 + (Lk + 127) // 128 * 128] == 0))
            vrow0 = (0 if w.varlen else s * qt.Hkv * qt.Dp) + h * qt.Dp
            vcol0 = kb if w.varlen else 0
            ok &= bool(np.all(self.v8[vrow0: vrow0 + qt.Dp,
                                      vcol0 + Lk: vcol0 + (Lk + 127) // 128 * 128] == 0))
        return ok


def compare_prologue(orc_seg: dict, gpu_seg: dict, D: int):
    """Bit-exact comparison of every quantized tensor; returns mismatch counts."""
    res = {}
    for name in ("q8", "s_q", "k8", "s_k", "v8", "s_v", "k_mean"):
        a, b = orc_seg[name], gpu_seg[name]
        assert a.shape == b.shape, (name, a.shape, b.shape)
        if a.dtype == np.float32:
            res[name] = int(np.sum(a.view(np.uint32) != b.view(np.uint32)))
        else:
            res[name] = int(np.sum(a != b))
    return res


def near_tie_rows(orc, pro, h, rows, causal, sm_scale):
    """For query head h of one segment: which of `rows` have a key whose 448 P,
    in the oracle's arithmetic (fp32 dequantised logits, running maximum per
    128-key block, exp2), lies within NEAR_TIE of an e4m3 rounding boundary."""
    f32 = np.float32
    Hq, Hkv, Lk = pro["Hq"], pro["Hkv"], pro["Lk"]
    hk = h // (Hq // Hkv)
    scale_log2 = f32(f32(sm_scale) * f32(1.4426950408889634))
    k8 = pro["k8"][hk].astype(np.int64)
    out = []
    for i in rows:
        S = k8 @ pro["q8"][h, i].astype(np.int64)
        m = f32(-np.inf)
        tie = False
        for b in range((Lk + 127) // 128):
            j0, j1 = 128 * b, min(Lk, 128 * b + 128)
            c = f32(f32(pro["s_q"][h, i] * pro["s_k"][hk, b]) * scale_log2)
            x = (S[j0:j1].astype(f32) * c).astype(f32)
            if causal:
                x[np.arange(j0, j1) > i] = -np.inf
            if not np.isfinite(x).any():
                continue
            m_new = f32(max(m, x.max()))
            d = (x - m_new).astype(f32)
            v448 = (f32(448.0) * np.exp2(d.astype(np.float64)).astype(f32)).astype(f32)
            lo = orc.e4m3_encode((v448 * (1.0 - NEAR_TIE)).astype(f32))
            hi = orc.e4m3_encode((v448 * (1.0 + NEAR_TIE)).astype(f32))
            tie |= bool(np.any(lo != hi))
            m = m_new
        out.append(tie)
    return out


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
