// Quantisation prologue (HBM-bound), sm_103a.
//
// What it computes follows stable-diffusion.cpp's "SageAttention" page (the
// FP8-path paragraph: smooth K, quantise V per channel, pad and permute V for
// FP8 tensor cores; "Use": head_dim zero-padded to 64/128), the SageAttention
// overview's Core features (INT8 Q/K, smoothing) and the SageAttention-RDNA4
// v0.4.0 notes (key mean summed in fp64, 64-bit offsets).
//
// Kernels, in launch order:
//   kv_stats     per (segment, kv head, 512-token chunk): exact per-channel
//                sums of K (int64 fixed point at 2^-24 for fp16, fp64 for
//                bf16) and per-channel max |V| (as ordered float bits),
//                accumulated with atomics.
//   kv_finalize  per (segment, kv head, channel): K mean, V scale and its
//                reciprocal multiplier.
//   kv_quant     per (segment, kv head, 128-token block): smoothed K -> int8
//                codes (stored as exact fp16 integers, the tensor-core
//                operand) with one scale per block; V -> e4m3 per channel,
//                transposed to channel-major through shared memory.
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
constexpr int kStatsChunk = 512;

__device__ __forceinline__ float to_f32(uint16_t bits, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

// Loads channels c0..c0+7 of one token row (zeros for channels >= D).
template <bool kVec>
__device__ __forceinline__ void load8(const uint16_t* row, int c0, int D,
                                      bool bf16, float (&x)[8]) {
  if (kVec) {
    if (c0 < D) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + c0);
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

__device__ __forceinline__ uint16_t code_f16(float x, float inv) {
  float r = static_cast<float>(__float2int_rn(__fmul_rn(x, inv)));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return __half_as_ushort(__float2half_rn(r));   // exact: |r| <= 127
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
                uint32_t* __restrict__ vmax, uint32_t* status) {
  const int64_t s = blockIdx.z, h = blockIdx.y;
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

  long long isum[8];
  double dsum[8];
  float am[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) { isum[i] = 0; dsum[i] = 0.0; am[i] = 0.0f; }

#pragma unroll 4
  for (int64_t t = t0 + r; t < t1; t += R) {
    float kx[8], vx[8];
    load8<kVec>(k + base + t * g.k_tok_stride, c0, static_cast<int>(g.D), kBf16, kx);
    load8<kVec>(v + base + t * g.k_tok_stride, c0, static_cast<int>(g.D), kBf16, vx);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (kBf16) dsum[i] += static_cast<double>(kx[i]);
      else isum[i] += __float2ll_rn(kx[i] * 16777216.0f);   // exact: k * 2^24
      am[i] = fmaxf(am[i], fabsf(vx[i]));
    }
  }

  __shared__ long long red_i[kThreads][8];
  __shared__ float red_a[kThreads][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    red_i[threadIdx.x][i] = kBf16 ? __double_as_longlong(dsum[i]) : isum[i];
    red_a[threadIdx.x][i] = am[i];
  }
  __syncthreads();
  if (r == 0) {
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
                                   float* s_v, float* v_inv) {
  const int64_t n = g.nseg * g.Hkv * g.Dp;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t s = i / (g.Hkv * g.Dp);
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
constexpr int kVPitch = 132;   // bytes per channel row of the V transpose tile

template <bool kVec, bool kBf16>
__global__ void __launch_bounds__(kThreads)
kv_quant_kernel(SegGeo g, const uint16_t* __restrict__ k,
                const uint16_t* __restrict__ v,
                const float* __restrict__ k_mean,
                const float* __restrict__ v_inv, uint16_t* __restrict__ k16,
                float* __restrict__ s_k, uint8_t* __restrict__ v8,
                uint32_t* status) {
  const int64_t s = blockIdx.z, h = blockIdx.y;
  int64_t start = 0, len = g.Lk;
  if (g.varlen && !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len)) return;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kBlockN;
  if (t0 >= len) return;
  const int G = static_cast<int>(g.Dp / 8);
  const int lc = threadIdx.x % G, r = threadIdx.x / G, R = kThreads / G;
  const int c0 = lc * 8;
  const int P = kBlockN / R;                 // 8 (Dp 128) or 4 (Dp 64)
  const int D = static_cast<int>(g.D);
  const int64_t in_base = (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                          h * g.k_head_stride;
  const int64_t stat = (s * g.Hkv + h) * g.Dp + c0;
  const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hkv, g.k_head_rows) +
                       h * g.k_head_rows + t0;

  __shared__ float red[kThreads / 32];
  __shared__ __align__(16) uint8_t vt[128 * kVPitch];

  // ---- K: smoothing and one int8 scale per 128-token block
  float mean[8], kh[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mean[i] = (c0 + i < D) ? k_mean[stat + i] : 0.0f;
  float am = 0.0f;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    if (p >= P) break;
    const int64_t t = t0 + r + p * R;
    float x[8];
    if (t < len) load8<kVec>(k + in_base + t * g.k_tok_stride, c0, D, kBf16, x);
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
      w[i] = static_cast<uint32_t>(code_f16(kh[p][2 * i], kinv)) |
             (static_cast<uint32_t>(code_f16(kh[p][2 * i + 1], kinv)) << 16);
    *reinterpret_cast<uint4*>(k16 + (row0 + rr) * g.Dp + c0) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (threadIdx.x == 0) s_k[row0 / kBlockN] = __fdiv_rn(am, 127.0f);

  // ---- V: e4m3 per channel, transposed to [channel][token]
  float vinv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) vinv[i] = (c0 + i < D) ? v_inv[stat + i] : 0.0f;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    if (p >= P) break;
    const int64_t rr = r + p * R;
    const int64_t t = t0 + rr;
    float x[8];
    if (t < len) load8<kVec>(v + in_base + t * g.k_tok_stride, c0, D, kBf16, x);
    else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint32_t two = pack_e4m3x2(__fmul_rn(x[i], vinv[i]),
                                       __fmul_rn(x[i + 1], vinv[i + 1]));
      vt[(c0 + i) * kVPitch + rr] = static_cast<uint8_t>(two & 0xFFu);
      vt[(c0 + i + 1) * kVPitch + rr] = static_cast<uint8_t>(two >> 8);
    }
  }
  __syncthreads();
  const int64_t vrow0 = (g.varlen ? 0 : s * g.Hkv * g.Dp) + h * g.Dp;
  const int64_t vcol0 = (g.varlen ? ws_seg_base(1, s, start, 0, 0) : 0) + t0;
  const int words = static_cast<int>(g.Dp) * (kBlockN / 4);
  for (int wi = threadIdx.x; wi < words; wi += kThreads) {
    const int c = wi / (kBlockN / 4), x4 = wi % (kBlockN / 4);
    const uint32_t val = *reinterpret_cast<const uint32_t*>(&vt[c * kVPitch + 4 * x4]);
    *reinterpret_cast<uint32_t*>(v8 + (vrow0 + c) * g.v_cols + vcol0 + 4 * x4) = val;
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
  for (int rr = r; rr < kBlockM; rr += R) {
    const int64_t t = t0 + rr;
    float x[8];
    if (t < len) load8<kVec>(q + in_base + t * g.q_tok_stride, c0, D, kBf16, x);
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
      w[i] = static_cast<uint32_t>(code_f16(x[2 * i], inv)) |
             (static_cast<uint32_t>(code_f16(x[2 * i + 1], inv)) << 16);
    *reinterpret_cast<uint4*>(q16 + (row0 + rr) * g.Dp + c0) =
        make_uint4(w[0], w[1], w[2], w[3]);
    if (lc == 0) s_q[row0 + rr] = __fdiv_rn(am, 127.0f);
  }
}

template <bool kVec, bool kBf16>
cudaError_t launch_prologue_t(const SegGeo& g, const PrologueBuffers& b,
                              cudaStream_t st) {
  const dim3 blk(kThreads);
  const int64_t maxk = g.varlen ? g.max_k : g.Lk;
  const int64_t maxq = g.varlen ? g.max_q : g.Lq;
  if (maxk > 0) {
    dim3 gs(static_cast<unsigned>((maxk + kStatsChunk - 1) / kStatsChunk),
            static_cast<unsigned>(g.Hkv), static_cast<unsigned>(g.nseg));
    kv_stats_kernel<kVec, kBf16><<<gs, blk, 0, st>>>(g, b.k, b.v, b.ksum, b.vmax, b.status);
  }
  const int64_t nstat = g.nseg * g.Hkv * g.Dp;
  kv_finalize_kernel<<<static_cast<unsigned>((nstat + 255) / 256), 256, 0, st>>>(
      g, b.ksum, b.vmax, b.k_mean, b.s_v, b.v_inv);
  if (maxk > 0) {
    dim3 gk(static_cast<unsigned>((maxk + kBlockN - 1) / kBlockN),
            static_cast<unsigned>(g.Hkv), static_cast<unsigned>(g.nseg));
    kv_quant_kernel<kVec, kBf16><<<gk, blk, 0, st>>>(
        g, b.k, b.v, b.k_mean, b.v_inv, b.k16, b.s_k, b.v8, b.status);
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
    kv_stats_kernel<kVec, kBf16><<<gs, kThreads, 0, st>>>(g, k, v, ksum, vmax, status);
  }
  const int64_t nstat = g.nseg * g.Hkv * g.Dp;
  kv_finalize_kernel<<<static_cast<unsigned>((nstat + 255) / 256), 256, 0, st>>>(
      g, ksum, vmax, k_mean, s_v, v_inv);
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
