// Quantisation prologue (HBM-bound), sm_103a.
//
// What it computes follows stable-diffusion.cpp's "SageAttention" page (the
// FP8-path paragraph: smooth K, quantise V per channel, pad and permute V for
// FP8 tensor cores; "Use": head_dim zero-padded to 64/128), the SageAttention
// overview's Core features (INT8 Q/K, smoothing) and the SageAttention-RDNA4
// v0.4.0 notes (key mean summed in fp64, 64-bit offsets).
//
// Kernels, in launch order (the first three once per group of kv heads whose
// K and V fit comfortably in L2, so that the second pass over K and V reads
// L2 rather than HBM; the first pass marks its lines evict-last):
//   kv_stats     per (segment, kv head, 256-token chunk): exact per-channel
//                sums of K (int64 fixed point at 2^-24 for fp16, fp64 for
//                bf16) and per-channel max |V| (as ordered float bits),
//                accumulated with atomics.
//   kv_finalize  per (segment, kv head, channel): K mean, V scale and its
//                reciprocal multiplier.
//   kv_quant     per (segment, kv head, 128-token block), K and V blocks in
//                separate CTAs: smoothed K -> int8 codes (stored as exact
//                fp16 integers, the tensor-core operand) with one scale per
//                block; V -> e4m3 per channel, transposed to channel-major
//                through shared memory.
//   q_quant      per (segment, q head, 128-token tile): Q -> int8 codes with
//                one scale per token.
// Every 128-token tile of the workspace is written in full (zeros past the
// sequence end and past D), so the attention kernel never reads stale bytes.
//
// Loads are 128-bit (8 elements) when D % 8 == 0 and the tensors are 16-byte
// aligned, otherwise element-wise.  Rounding is explicit (__fmul_rn,
// __fdiv_rn, __float2int_rn) so the codes match a plain IEEE restatement.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "sage_device.cuh"
#include "sage_geom.h"
#include "sage_kernels.h"

namespace sage {

namespace {

constexpr int kThreads = 256;
constexpr int kStatsChunk = 256;

__device__ __forceinline__ float to_f32(uint16_t bits, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

// L2 cache policies: keep the first pass over K/V resident for the second.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld16(const void* p, uint64_t pol) {
  uint4 u;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "l"(p), "l"(pol));
  return u;
}

// Loads channels c0..c0+7 of one token row (zeros for channels >= D).
template <bool kVec>
__device__ __forceinline__ void load8(const uint16_t* row, int c0, int D,
                                      bool bf16, float (&x)[8], uint64_t pol) {
  if (kVec) {
    if (c0 < D) {
      const uint4 u = ld16(row + c0, pol);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = to_f32(static_cast<uint16_t>(w[i] & 0xFFFFu), bf16);
        x[2 * i + 1] = to_f32(static_cast<uint16_t>(w[i] >> 16), bf16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      x[i] = (c0 + i < D) ? to_f32(row[c0 + i], bf16) : 0.0f;
  }
}

// Two int8 codes clamp(rint(x * inv), -127, 127) as a pair of exact fp16
// integers (low half: x0).  rint uses the 1.5*2^23 addend (ties to even,
// exact for |x * inv| < 2^22); the fp16 conversion of integers is exact.
__device__ __forceinline__ uint32_t code_f16x2(float x0, float x1, float inv) {
  const float r0 = fminf(fmaxf((__fmul_rn(x0, inv) + 12582912.0f) - 12582912.0f, -127.0f), 127.0f);
  const float r1 = fminf(fmaxf((__fmul_rn(x1, inv) + 12582912.0f) - 12582912.0f, -127.0f), 127.0f);
  const __half2 hv = __floats2half2_rn(r0, r1);
  return *reinterpret_cast<const uint32_t*>(&hv);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// ---------------------------------------------------------------- stats
template <bool kVec, bool kBf16>
__global__ void __launch_bounds__(kThreads)
kv_stats_kernel(SegGeo g, const uint16_t* __restrict__ k,
                const uint16_t* __restrict__ v, void* ksum,
                uint32_t* __restrict__ vmax, uint32_t* status, int h_base) {
  const int64_t s = blockIdx.z, h = h_base + blockIdx.y;
  int64_t start = 0, len = g.Lk;
  if (g.varlen && !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len)) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBadSeqlens);
    return;
  }
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kStatsChunk;
  if (t0 >= len) return;
  const int64_t t1 = min(len, t0 + kStatsChunk);
  const int G = static_cast<int>(g.Dp / 8);
  const int lc = threadIdx.x % G, r = threadIdx.x / G, R = kThreads / G;
  const int c0 = lc * 8;
  const int64_t base = (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                       h * g.k_head_stride;

  // fp16 keys: exact sums in units of 2^-24, each key split into two exact
  // int32 parts (hi in units of 2^20, lo in [-2^19, 2^19]) with fp32
  // round-to-integer arithmetic; this keeps the FP64 pipe (slow on GB300) out
  // of the loop.  bf16 keys: fp64 sums.
  int hs[8], ls[8];
  double dsum[8];
  float am[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) { hs[i] = 0; ls[i] = 0; dsum[i] = 0.0; am[i] = 0.0f; }
  const uint64_t keep = policy_evict_last();

#pragma unroll 4
  for (int64_t t = t0 + r; t < t1; t += R) {
    float kx[8], vx[8];
    load8<kVec>(k + base + t * g.k_tok_stride, c0, static_cast<int>(g.D), kBf16, kx, keep);
    load8<kVec>(v + base + t * g.k_tok_stride, c0, static_cast<int>(g.D), kBf16, vx, keep);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (kBf16) {
        dsum[i] += static_cast<double>(kx[i]);
      } else {
        const float tr = fmaf(kx[i], 16.0f, 12582912.0f);     // 1.5*2^23 + rint(16 k)
        const float hi_f = tr - 12582912.0f;
        const float lo_f = fmaf(kx[i], 16777216.0f, hi_f * -1048576.0f);
        hs[i] += __float_as_int(tr) - 0x4B400000;
        ls[i] += __float_as_int(lo_f + 12582912.0f) - 0x4B400000;
      }
      am[i] = fmaxf(am[i], fabsf(vx[i]));
    }
  }

  __shared__ long long red_i[kThreads][8];
  __shared__ float red_a[kThreads][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    red_i[threadIdx.x][i] = kBf16 ? __double_as_longlong(dsum[i])
                                  : static_cast<long long>(hs[i]) * 1048576ll + ls[i];
    red_a[threadIdx.x][i] = am[i];
  }
  __syncthreads();
  if (r == 0) {
    long long isum[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) isum[i] = red_i[threadIdx.x][i];
    for (int rr = 1; rr < R; ++rr) {
      const int src = rr * G + lc;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (kBf16) dsum[i] += __longlong_as_double(red_i[src][i]);
        else isum[i] += red_i[src][i];
        am[i] = fmaxf(am[i], red_a[src][i]);
      }
    }
    const int64_t o = (s * g.Hkv + h) * g.Dp + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (c0 + i >= g.D) break;
      if (kBf16) atomicAdd(reinterpret_cast<double*>(ksum) + o + i, dsum[i]);
      else atomicAdd(reinterpret_cast<unsigned long long*>(ksum) + o + i,
                     static_cast<unsigned long long>(isum[i]));
      atomicMax(vmax + o + i, __float_as_uint(am[i]));   // am >= +0
    }
  }
}

__global__ void kv_finalize_kernel(SegGeo g, const void* ksum,
                                   const uint32_t* vmax, float* k_mean,
                                   float* s_v, float* v_inv, int h_base, int h_count) {
  // thread -> (segment, kv head in [h_base, h_base + h_count), channel)
  const int64_t per_seg = static_cast<int64_t>(h_count) * g.Dp;
  const int64_t n = g.nseg * per_seg;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n) return;
  const int64_t s = idx / per_seg;
  const int64_t i = (s * g.Hkv + h_base) * g.Dp + idx % per_seg;
  int64_t len = g.Lk;
  if (g.varlen) {
    len = static_cast<int64_t>(g.cu_k[s + 1]) - g.cu_k[s];
    if (len < 0) len = 0;
  }
  double S;
  if (g.dtype == 1) S = reinterpret_cast<const double*>(ksum)[i];
  else S = __ll2double_rn(reinterpret_cast<const long long*>(ksum)[i]) *
           5.9604644775390625e-08;   // 2^-24, exact
  k_mean[i] = len > 0 ? __double2float_rn(__ddiv_rn(S, static_cast<double>(len))) : 0.0f;
  const float a = __uint_as_float(vmax[i]);
  s_v[i] = __fdiv_rn(a, 448.0f);
  v_inv[i] = a > 0.0f ? __fdiv_rn(448.0f, a) : 0.0f;
}

// ---------------------------------------------------------- K/V quant
// One CTA quantises one 128-token block of K (role 0) or of V (role 1) of one
// (segment, kv head); blocks are numbered ((s * h_count + hh) * nkb + kb) * 2
// + role over the current head group.
template <bool kVec, bool kBf16>
__global__ void __launch_bounds__(kThreads)
kv_quant_kernel(SegGeo g, const uint16_t* __restrict__ k,
                const uint16_t* __restrict__ v,
                const float* __restrict__ k_mean,
                const float* __restrict__ v_inv, uint16_t* __restrict__ k16,
                float* __restrict__ s_k, uint8_t* __restrict__ v8,
                int h_base, int h_count, int nkb) {
  const int role = blockIdx.x & 1;
  const int64_t blk = blockIdx.x >> 1;
  const int64_t kb = blk % nkb;
  const int64_t hh = (blk / nkb) % h_count;
  const int64_t s = blk / (static_cast<int64_t>(nkb) * h_count);
  const int64_t h = h_base + hh;
  int64_t start = 0, len = g.Lk;
  if (g.varlen && !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len)) return;
  const int64_t t0 = kb * kBlockN;
  if (t0 >= len) return;
  const int G = static_cast<int>(g.Dp / 8);
  const int lc = threadIdx.x % G, r = threadIdx.x / G, R = kThreads / G;
  const int c0 = lc * 8;
  const int P = kBlockN / R;                 // 8 (Dp 128) or 4 (Dp 64)
  const int D = static_cast<int>(g.D);
  const int64_t in_base = (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                          h * g.k_head_stride;
  const int64_t stat = (s * g.Hkv + h) * g.Dp + c0;
  const uint64_t last_use = policy_evict_first();

  if (role == 0) {
    // ---- K: smoothing and one int8 scale per 128-token block
    __shared__ float red[kThreads / 32];
    const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hkv, g.k_head_rows) +
                         h * g.k_head_rows + t0;
    float mean[8], kh[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mean[i] = (c0 + i < D) ? k_mean[stat + i] : 0.0f;
    float am = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p >= P) break;
      const int64_t t = t0 + r + p * R;
      float x[8];
      if (t < len) load8<kVec>(k + in_base + t * g.k_tok_stride, c0, D, kBf16, x, last_use);
      else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        kh[p][i] = (t < len && c0 + i < D) ? __fsub_rn(x[i], mean[i]) : 0.0f;
        am = fmaxf(am, fabsf(kh[p][i]));
      }
    }
    am = warp_max(am);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
    __syncthreads();
    am = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) am = fmaxf(am, red[w]);
    const float kinv = am > 0.0f ? __fdiv_rn(127.0f, am) : 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p >= P) break;
      const int64_t rr = r + p * R;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = code_f16x2(kh[p][2 * i], kh[p][2 * i + 1], kinv);
      *reinterpret_cast<uint4*>(k16 + (row0 + rr) * g.Dp + c0) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (threadIdx.x == 0) s_k[row0 / kBlockN] = __fdiv_rn(am, 127.0f);
  } else {
    // ---- V: e4m3 per channel, transposed to [channel][token].  A thread
    // quantises 8 channels of 4 consecutive tokens and packs, per channel, the
    // 4 token bytes into one word; word (c, w) of the shared tile sits at
    // c * 32 + (w ^ (c / 8 % 32)) so that writes and row reads spread banks.
    __shared__ uint32_t vt[128 * 32];
    float vinv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) vinv[i] = (c0 + i < D) ? v_inv[stat + i] : 0.0f;
    const int RG = kThreads / G;                 // 4-token groups per pass
    for (int tw = r; tw < kBlockN / 4; tw += RG) {
      uint32_t word[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) word[i] = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t t = t0 + 4 * tw + e;
        float x[8];
        if (t < len) load8<kVec>(v + in_base + t * g.k_tok_stride, c0, D, kBf16, x, last_use);
        else {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const uint32_t two = pack_e4m3x2(__fmul_rn(x[i], vinv[i]),
                                           __fmul_rn(x[i + 1], vinv[i + 1]));
          word[i] |= (two & 0xFFu) << (8 * e);
          word[i + 1] |= (two >> 8) << (8 * e);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + i;
        vt[c * 32 + (tw ^ ((c >> 3) & 31))] = word[i];
      }
    }
    __syncthreads();
    const int64_t vrow0 = (g.varlen ? 0 : s * g.Hkv * g.Dp) + h * g.Dp;
    const int64_t vcol0 = (g.varlen ? ws_seg_base(1, s, start, 0, 0) : 0) + t0;
    const int words = static_cast<int>(g.Dp) * (kBlockN / 4);
    for (int wi = threadIdx.x; wi < words; wi += kThreads) {
      const int c = wi / (kBlockN / 4), tw = wi % (kBlockN / 4);
      const uint32_t val = vt[c * 32 + (tw ^ ((c >> 3) & 31))];
      *reinterpret_cast<uint32_t*>(v8 + (vrow0 + c) * g.v_cols + vcol0 + 4 * tw) = val;
    }
  }
}

// ------------------------------------------------------------- Q quant
template <bool kVec, bool kBf16>
__global__ void __launch_bounds__(kThreads)
q_quant_kernel(SegGeo g, const uint16_t* __restrict__ q,
               uint16_t* __restrict__ q16, float* __restrict__ s_q,
               uint32_t* status) {
  const int64_t s = blockIdx.z, h = blockIdx.y;
  int64_t start = 0, len = g.Lq;
  if (g.varlen && !seg_range(g.cu_q, s, g.total_q, g.max_q, &start, &len)) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) atomicOr(status, kStatusBadSeqlens);
    return;
  }
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kBlockM;
  if (t0 >= len) return;
  const int G = static_cast<int>(g.Dp / 8);
  const int lc = threadIdx.x % G, r = threadIdx.x / G, R = kThreads / G;
  const int c0 = lc * 8;
  const int D = static_cast<int>(g.D);
  const int64_t in_base = (g.varlen ? start * g.q_tok_stride : s * g.q_seg_stride) +
                          h * g.q_head_stride;
  const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hq, g.q_head_rows) +
                       h * g.q_head_rows + t0;
  const uint64_t once = policy_evict_first();
  for (int rr = r; rr < kBlockM; rr += R) {
    const int64_t t = t0 + rr;
    float x[8];
    if (t < len) load8<kVec>(q + in_base + t * g.q_tok_stride, c0, D, kBf16, x, once);
    else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    }
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(x[i]));
    for (int o = G / 2; o > 0; o >>= 1)
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
    const float inv = am > 0.0f ? __fdiv_rn(127.0f, am) : 0.0f;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = code_f16x2(x[2 * i], x[2 * i + 1], inv);
    *reinterpret_cast<uint4*>(q16 + (row0 + rr) * g.Dp + c0) =
        make_uint4(w[0], w[1], w[2], w[3]);
    if (lc == 0) s_q[row0 + rr] = __fdiv_rn(am, 127.0f);
  }
}

// K and V of one head group are read twice (stats, then quantisation); the
// group is sized so that both passes fit in L2 with room to spare.
constexpr int64_t kL2GroupBytes = 48ll << 20;

template <bool kVec, bool kBf16>
cudaError_t launch_prologue_t(const SegGeo& g, const PrologueBuffers& b,
                              cudaStream_t st) {
  const dim3 blk(kThreads);
  const int64_t maxk = g.varlen ? g.max_k : g.Lk;
  const int64_t maxq = g.varlen ? g.max_q : g.Lq;
  if (maxk > 0) {
    const int64_t tokens = g.varlen ? g.total_k : g.nseg * g.Lk;
    const int64_t head_bytes = tokens * g.D * 2 * 2;          // K and V, one kv head
    int64_t group = head_bytes > 0 ? kL2GroupBytes / head_bytes : g.Hkv;
    if (group < 1) group = 1;
    if (group > g.Hkv) group = g.Hkv;
    const int nkb = static_cast<int>((maxk + kBlockN - 1) / kBlockN);
    for (int64_t h0 = 0; h0 < g.Hkv; h0 += group) {
      const int hc = static_cast<int>(g.Hkv - h0 < group ? g.Hkv - h0 : group);
      dim3 gs(static_cast<unsigned>((maxk + kStatsChunk - 1) / kStatsChunk),
              static_cast<unsigned>(hc), static_cast<unsigned>(g.nseg));
      kv_stats_kernel<kVec, kBf16><<<gs, blk, 0, st>>>(g, b.k, b.v, b.ksum, b.vmax,
                                                        b.status, static_cast<int>(h0));
      const int64_t nstat = g.nseg * hc * g.Dp;
      kv_finalize_kernel<<<static_cast<unsigned>((nstat + 255) / 256), 256, 0, st>>>(
          g, b.ksum, b.vmax, b.k_mean, b.s_v, b.v_inv, static_cast<int>(h0), hc);
      const int64_t nblk = g.nseg * hc * static_cast<int64_t>(nkb) * 2;
      kv_quant_kernel<kVec, kBf16><<<static_cast<unsigned>(nblk), blk, 0, st>>>(
          g, b.k, b.v, b.k_mean, b.v_inv, b.k16, b.s_k, b.v8, static_cast<int>(h0), hc, nkb);
    }
  }
  if (maxq > 0) {
    dim3 gq(static_cast<unsigned>((maxq + kBlockM - 1) / kBlockM),
            static_cast<unsigned>(g.Hq), static_cast<unsigned>(g.nseg));
    q_quant_kernel<kVec, kBf16><<<gq, blk, 0, st>>>(g, b.q, b.q16, b.s_q, b.status);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const SegGeo& g, const PrologueBuffers& b,
                            bool vec, cudaStream_t st) {
  const bool bf16 = g.dtype == 1;
  if (vec) return bf16 ? launch_prologue_t<true, true>(g, b, st)
                       : launch_prologue_t<true, false>(g, b, st);
  return bf16 ? launch_prologue_t<false, true>(g, b, st)
              : launch_prologue_t<false, false>(g, b, st);
}

// ------------------------------------------- statistics without allocation
// Scratch of the allocation-free statistics entry point: the status word,
// then per-channel K sums (8 B), V maxima (4 B) and V multipliers (4 B) for
// at most kStaticStatEntries (segment, kv head, channel) triples.  It lives
// in the module image, so every device that loads this library holds it
// until the process exits; concurrent calls share it.
namespace {
constexpr size_t kStaticHeader = 256;
__device__ __align__(256) unsigned char g_stats_scratch[
    kStaticHeader + kStaticStatEntries * (8 + 4 + 4)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

template <bool kVec, bool kBf16>
void launch_stats_only(const SegGeo& g, const uint16_t* k, const uint16_t* v,
                       void* ksum, uint32_t* vmax, float* k_mean, float* s_v,
                       float* v_inv, uint32_t* status, cudaStream_t st) {
  if (g.Lk > 0) {
    dim3 gs(static_cast<unsigned>((g.Lk + kStatsChunk - 1) / kStatsChunk),
            static_cast<unsigned>(g.Hkv), static_cast<unsigned>(g.nseg));
    kv_stats_kernel<kVec, kBf16><<<gs, kThreads, 0, st>>>(g, k, v, ksum, vmax, status, 0);
  }
  const int64_t nstat = g.nseg * g.Hkv * g.Dp;
  kv_finalize_kernel<<<static_cast<unsigned>((nstat + 255) / 256), 256, 0, st>>>(
      g, ksum, vmax, k_mean, s_v, v_inv, 0, static_cast<int>(g.Hkv));
}
}  // namespace

cudaError_t launch_kv_stats_static(const SegGeo& g, const uint16_t* k,
                                   const uint16_t* v, float* k_mean, float* s_v,
                                   bool vec, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned char* base = nullptr;
  {
    // one-time set-up per device, with that device current: the host-side
    // name of the array is not a device address, so look the address up
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_stats_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_addr[dev] = p;
    }
    base = static_cast<unsigned char*>(g_scratch_addr[dev]);
  }
  const int64_t n = g.nseg * g.Hkv * g.Dp;
  if (n > kStaticStatEntries) return cudaErrorInvalidValue;
  uint32_t* status = reinterpret_cast<uint32_t*>(base);
  void* ksum = base + kStaticHeader;
  uint32_t* vmax = reinterpret_cast<uint32_t*>(base + kStaticHeader + kStaticStatEntries * 8);
  float* v_inv = reinterpret_cast<float*>(base + kStaticHeader + kStaticStatEntries * 12);
  // the previous call's sums and maxima are still there: clear them
  e = cudaMemsetAsync(base, 0, kStaticHeader + kStaticStatEntries * 12, st);
  if (e != cudaSuccess) return e;
  const bool bf16 = g.dtype == 1;
  if (vec) {
    if (bf16) launch_stats_only<true, true>(g, k, v, ksum, vmax, k_mean, s_v, v_inv, status, st);
    else launch_stats_only<true, false>(g, k, v, ksum, vmax, k_mean, s_v, v_inv, status, st);
  } else {
    if (bf16) launch_stats_only<false, true>(g, k, v, ksum, vmax, k_mean, s_v, v_inv, status, st);
    else launch_stats_only<false, false>(g, k, v, ksum, vmax, k_mean, s_v, v_inv, status, st);
  }
  return cudaGetLastError();
}

}  // namespace sage
