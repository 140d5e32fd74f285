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
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Read-only 16-byte load with an L2 policy.  Not volatile: the compiler may
// schedule it early (the inputs are never written by the prologue).
__device__ __forceinline__ uint4 ld16(const void* p, uint64_t pol) {
  uint4 u;
  asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "l"(p), "l"(pol));
  return u;
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

// Channels c0..c0+7 of one token row as four packed 16-bit pairs (zeros for
// channels >= D).
template <bool kVec>
__device__ __forceinline__ uint4 load8_raw(const uint16_t* row, int c0, int D, uint64_t pol) {
  if constexpr (kVec) {
    return c0 < D ? ld16(row + c0, pol) : make_uint4(0u, 0u, 0u, 0u);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (c0 + 2 * i < D) ? row[c0 + 2 * i] : 0u;
      const uint32_t hi = (c0 + 2 * i + 1 < D) ? row[c0 + 2 * i + 1] : 0u;
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
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
                uint32_t* __restrict__ vmax, uint32_t* status, int h_base,
                uint32_t* done, float* k_mean, float* s_v, float* v_inv) {
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

  const int D = static_cast<int>(g.D);
  for (int64_t tb = t0 + r; tb < t1; tb += 8 * R) {
    uint4 kr[8], vr[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {                // 16 loads in flight per thread
      const int64_t t = tb + u * R;
      const bool in = t < t1;
      kr[u] = in ? load8_raw<kVec>(k + base + t * g.k_tok_stride, c0, D, keep)
                 : make_uint4(0u, 0u, 0u, 0u);
      vr[u] = in ? load8_raw<kVec>(v + base + t * g.k_tok_stride, c0, D, keep)
                 : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t kw[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      const uint32_t vw[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float kx = to_f32(static_cast<uint16_t>(kw[i >> 1] >> (16 * (i & 1))), kBf16);
        const float vx = to_f32(static_cast<uint16_t>(vw[i >> 1] >> (16 * (i & 1))), kBf16);
        if (kBf16) {
          dsum[i] += static_cast<double>(kx);
        } else {
          const float tr = fmaf(kx, 16.0f, 12582912.0f);      // 1.5*2^23 + rint(16 k)
          const float hi_f = tr - 12582912.0f;
          const float lo_f = fmaf(kx, 16777216.0f, hi_f * -1048576.0f);
          hs[i] += __float_as_int(tr) - 0x4B400000;
          ls[i] += __float_as_int(lo_f + 12582912.0f) - 0x4B400000;
        }
        am[i] = fmaxf(am[i], fabsf(vx));
      }
    }
  }

  // reduce the rows: lanes holding the same channels first (warp shuffles),
  // then the eight warps through shared memory, one channel per thread
  long long part[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    part[i] = kBf16 ? __double_as_longlong(dsum[i])
                    : static_cast<long long>(hs[i]) * 1048576ll + ls[i];
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const long long other = __shfl_xor_sync(0xFFFFFFFFu, part[i], o);
      if (kBf16) part[i] = __double_as_longlong(__longlong_as_double(part[i]) +
                                                __longlong_as_double(other));
      else part[i] += other;
      am[i] = fmaxf(am[i], __shfl_xor_sync(0xFFFFFFFFu, am[i], o));
    }
  }
  __shared__ long long red_i[kThreads / 32][128];
  __shared__ float red_a[kThreads / 32][128];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane < G) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      red_i[wid][c0 + i] = part[i];
      red_a[wid][c0 + i] = am[i];
    }
  }
  __syncthreads();
  const int64_t obase = (s * g.Hkv + h) * g.Dp;
  if (threadIdx.x < g.D) {
    const int c = threadIdx.x;
    long long si = 0;
    double sd = 0.0;
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      if (kBf16) sd += __longlong_as_double(red_i[w][c]);
      else si += red_i[w][c];
      a = fmaxf(a, red_a[w][c]);
    }
    if (kBf16) atomicAdd(reinterpret_cast<double*>(ksum) + obase + c, sd);
    else atomicAdd(reinterpret_cast<unsigned long long*>(ksum) + obase + c,
                   static_cast<unsigned long long>(si));
    atomicMax(vmax + obase + c, __float_as_uint(a));   // a >= +0
    if (done != nullptr) __threadfence();
  }
  if (done == nullptr) return;
  // The last CTA of this (segment, kv head) turns the sums into the K mean
  // and the V scales (the finalize step) while the sums are hot in L2.
  __shared__ int last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t chunks = static_cast<uint32_t>((len + kStatsChunk - 1) / kStatsChunk);
    last = atomicAdd(done + s * g.Hkv + h, 1u) == chunks - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int c = threadIdx.x; c < g.Dp; c += kThreads) {
    const int64_t i = (s * g.Hkv + h) * g.Dp + c;
    double S;
    if (kBf16) S = __longlong_as_double(__ldcg(reinterpret_cast<const long long*>(ksum) + i));
    else S = __ll2double_rn(__ldcg(reinterpret_cast<const long long*>(ksum) + i)) *
             5.9604644775390625e-08;   // 2^-24, exact
    k_mean[i] = __double2float_rn(__ddiv_rn(S, static_cast<double>(len)));
    const float a = __uint_as_float(__ldcg(vmax + i));
    s_v[i] = __fdiv_rn(a, 448.0f);
    v_inv[i] = a > 0.0f ? __fdiv_rn(448.0f, a) : 0.0f;
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

// ------------------------------------------------------------- Q quant
// One 128-token tile of Q of query head h in segment s.
template <bool kVec, bool kBf16>
__device__ __forceinline__ void quant_q_tile(const SegGeo& g, const uint16_t* __restrict__ q,
                                             uint16_t* __restrict__ q16,
                                             float* __restrict__ s_q, uint32_t* status,
                                             int64_t s, int64_t h, int64_t qt) {
  int64_t start = 0, len = g.Lq;
  if (g.varlen && !seg_range(g.cu_q, s, g.total_q, g.max_q, &start, &len)) {
    if (threadIdx.x == 0 && qt == 0 && h == 0) atomicOr(status, kStatusBadSeqlens);
    return;
  }
  const int64_t t0 = qt * kBlockM;
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
  const int P = kBlockM / R;                   // rows per thread: 8 (Dp 128) or 4 (Dp 64)
  uint4 raw[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) {                // all loads first: one round trip
    if (p >= P) break;
    const int64_t t = t0 + r + p * R;
    raw[p] = t < len ? load8_raw<kVec>(q + in_base + t * g.q_tok_stride, c0, D, once)
                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    if (p >= P) break;
    const int64_t rr = r + p * R;
    const uint32_t w[4] = {raw[p].x, raw[p].y, raw[p].z, raw[p].w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      x[i] = to_f32(static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1))), kBf16);
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(x[i]));
    for (int o = G / 2; o > 0; o >>= 1)
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
    const float inv = am > 0.0f ? __fdiv_rn(127.0f, am) : 0.0f;
    *reinterpret_cast<uint4*>(q16 + (row0 + rr) * g.Dp + c0) =
        make_uint4(code_f16x2(x[0], x[1], inv), code_f16x2(x[2], x[3], inv),
                   code_f16x2(x[4], x[5], inv), code_f16x2(x[6], x[7], inv));
    if (lc == 0) s_q[row0 + rr] = __fdiv_rn(am, 127.0f);
  }
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
                int h_base, int h_count, int nkb,
                const uint16_t* __restrict__ q, uint16_t* __restrict__ q16,
                float* __restrict__ s_q, uint32_t* status, int nqt) {
  const int64_t nkv = static_cast<int64_t>(g.nseg) * h_count * nkb * 2;
  if (static_cast<int64_t>(blockIdx.x) >= nkv) {
    // Q tiles of the query heads that read this group's kv heads
    const int64_t grp = g.Hq / g.Hkv;
    const int64_t qb = blockIdx.x - nkv;
    const int64_t qt = qb % nqt;
    const int64_t hq = h_base * grp + (qb / nqt) % (h_count * grp);
    const int64_t sq = qb / (static_cast<int64_t>(nqt) * h_count * grp);
    quant_q_tile<kVec, kBf16>(g, q, q16, s_q, status, sq, hq, qt);
    return;
  }
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
    // ---- K: smoothing and one int8 scale per 128-token block.  The raw
    // values stay packed (16-bit) in registers; k - mean is recomputed (the
    // same IEEE subtraction) in the amax and in the quantisation pass.
    __shared__ float red[kThreads / 32];
    const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hkv, g.k_head_rows) +
                         h * g.k_head_rows + t0;
    float mean[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mean[i] = (c0 + i < D) ? k_mean[stat + i] : 0.0f;
    uint4 raw[8];
    bool valid[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p >= P) break;
      const int64_t t = t0 + r + p * R;
      valid[p] = t < len;
      raw[p] = valid[p] ? load8_raw<kVec>(k + in_base + t * g.k_tok_stride, c0, D, last_use)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
    float am = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p >= P) break;
      const uint32_t w[4] = {raw[p].x, raw[p].y, raw[p].z, raw[p].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x = to_f32(static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1))), kBf16);
        const float kh = (valid[p] && c0 + i < D) ? __fsub_rn(x, mean[i]) : 0.0f;
        am = fmaxf(am, fabsf(kh));
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
      const uint32_t w[4] = {raw[p].x, raw[p].y, raw[p].z, raw[p].w};
      float kh[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x = to_f32(static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1))), kBf16);
        kh[i] = (valid[p] && c0 + i < D) ? __fsub_rn(x, mean[i]) : 0.0f;
      }
      *reinterpret_cast<uint4*>(k16 + (row0 + rr) * g.Dp + c0) =
          make_uint4(code_f16x2(kh[0], kh[1], kinv), code_f16x2(kh[2], kh[3], kinv),
                     code_f16x2(kh[4], kh[5], kinv), code_f16x2(kh[6], kh[7], kinv));
    }
    if (threadIdx.x == 0) s_k[row0 / kBlockN] = __fdiv_rn(am, 127.0f);
  } else {
    // ---- V: e4m3 per channel, transposed to [channel][token].  A thread
    // quantises 8 channels of 4 consecutive tokens and packs, per channel, the
    // 4 token bytes into one word; word (c, w) of the shared tile sits at
    // c * 32 + (w ^ 4 * (c / 8 % 8)), which spreads the writes over banks and
    // keeps every group of four words (16 bytes of a row) contiguous.
    __shared__ __align__(16) uint32_t vt[128 * 32];
    float vinv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) vinv[i] = (c0 + i < D) ? v_inv[stat + i] : 0.0f;
    const int RG = kThreads / G;                 // 4-token groups per pass
    const int NTW = (kBlockN / 4) / RG;          // groups per thread: 2 (Dp 128) or 1
    uint4 raw[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a) {                // all loads first: one round trip
      if (a >= NTW) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t t = t0 + 4 * (r + a * RG) + e;
        raw[a][e] = t < len ? load8_raw<kVec>(v + in_base + t * g.k_tok_stride, c0, D, last_use)
                            : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      if (a >= NTW) break;
      const int tw = r + a * RG;
      uint32_t word[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) word[i] = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w[4] = {raw[a][e].x, raw[a][e].y, raw[a][e].z, raw[a][e].w};
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float x0 = to_f32(static_cast<uint16_t>(w[i >> 1] & 0xFFFFu), kBf16);
          const float x1 = to_f32(static_cast<uint16_t>(w[i >> 1] >> 16), kBf16);
          const uint32_t two = pack_e4m3x2(__fmul_rn(x0, vinv[i]), __fmul_rn(x1, vinv[i + 1]));
          word[i] |= (two & 0xFFu) << (8 * e);
          word[i + 1] |= (two >> 8) << (8 * e);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + i;
        vt[c * 32 + (tw ^ (((c >> 3) & 7) << 2))] = word[i];
      }
    }
    __syncthreads();
    const int64_t vrow0 = (g.varlen ? 0 : s * g.Hkv * g.Dp) + h * g.Dp;
    const int64_t vcol0 = (g.varlen ? ws_seg_base(1, s, start, 0, 0) : 0) + t0;
    const int quads = static_cast<int>(g.Dp) * (kBlockN / 16);   // 16-byte pieces
    for (int qi = threadIdx.x; qi < quads; qi += kThreads) {
      const int c = qi / (kBlockN / 16), tw = 4 * (qi % (kBlockN / 16));
      const uint4 val = *reinterpret_cast<const uint4*>(&vt[c * 32 + (tw ^ (((c >> 3) & 7) << 2))]);
      *reinterpret_cast<uint4*>(v8 + (vrow0 + c) * g.v_cols + vcol0 + 4 * tw) = val;
    }
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
  const int nqt = static_cast<int>((maxq + kBlockM - 1) / kBlockM);
  const int64_t grp = g.Hq / g.Hkv;
  const int64_t tokens = g.varlen ? g.total_k : g.nseg * g.Lk;
  const int64_t head_bytes = tokens * g.D * 2 * 2;            // K and V, one kv head
  int64_t group = head_bytes > 0 ? kL2GroupBytes / head_bytes : g.Hkv;
  if (group < 1) group = 1;
  if (group > g.Hkv) group = g.Hkv;
  const int nkb = maxk > 0 ? static_cast<int>((maxk + kBlockN - 1) / kBlockN) : 0;
  for (int64_t h0 = 0; h0 < g.Hkv; h0 += group) {
    const int hc = static_cast<int>(g.Hkv - h0 < group ? g.Hkv - h0 : group);
    if (maxk > 0) {
      dim3 gs(static_cast<unsigned>((maxk + kStatsChunk - 1) / kStatsChunk),
              static_cast<unsigned>(hc), static_cast<unsigned>(g.nseg));
      kv_stats_kernel<kVec, kBf16><<<gs, blk, 0, st>>>(g, b.k, b.v, b.ksum, b.vmax, b.status,
                                                        static_cast<int>(h0), b.done,
                                                        b.k_mean, b.s_v, b.v_inv);
    }
    // K/V blocks of this head group, then the Q tiles of its query heads
    const int64_t nblk = g.nseg * hc * static_cast<int64_t>(nkb) * 2 +
                         g.nseg * hc * grp * static_cast<int64_t>(nqt);
    if (nblk > 0)
      kv_quant_kernel<kVec, kBf16><<<static_cast<unsigned>(nblk), blk, 0, st>>>(
          g, b.k, b.v, b.k_mean, b.v_inv, b.k16, b.s_k, b.v8, static_cast<int>(h0), hc, nkb,
          b.q, b.q16, b.s_q, b.status, nqt);
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
    kv_stats_kernel<kVec, kBf16><<<gs, kThreads, 0, st>>>(g, k, v, ksum, vmax, status, 0,
                                                           nullptr, nullptr, nullptr, nullptr);
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
