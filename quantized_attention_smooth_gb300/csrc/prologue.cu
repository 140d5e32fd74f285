// Quantisation prologue (HBM-bound), sm_103a.
//
// What it computes follows stable-diffusion.cpp's "SageAttention" page (the
// FP8-path paragraph: smooth K, quantise V per channel, pad and permute V for
// FP8 tensor cores; "Use": head_dim zero-padded to 64/128), the SageAttention
// overview's Core features (INT8 Q/K, smoothing) and the SageAttention-RDNA4
// v0.4.0 notes (key mean summed in fp64, 64-bit offsets).
//
// One persistent kernel.  Its CTAs take work items, in order, from a counter
// in the workspace.  A unit is one (segment, kv head); its items are
//   stats  256 tokens of K and V: exact per-channel sums of K (int64 fixed
//          point at 2^-24 for fp16, fp64 for bf16) and per-channel max |V|,
//          added to the unit's accumulators with atomics.  The unit's last
//          stats item turns them into the K mean, the V scale and its
//          reciprocal multiplier and raises the unit's ready flag.
//   Q      128 tokens of one query head that reads this kv head: int8 codes
//          (stored as exact fp16 integers, the tensor-core operand), one
//          scale per token.
//   K      128 tokens: smoothed K (k - mean, fp32) -> int8 codes, one scale
//          per block.  Waits for the ready flag.
//   V      128 tokens: e4m3 per channel, transposed to channel-major through
//          shared memory.  Waits for the ready flag.
// The list puts a unit's K and V items `lag` units after its stats and Q
// items, far enough that its statistics are normally done before a CTA takes
// them and near enough that the unit's K and V are still in L2 (the stats
// pass marks them evict-last).  Items are taken in list order by running
// CTAs only, so every item waited on is already held by a running CTA and
// the waits always end; they are bounded all the same (timeout -> status
// bit).  Every 128-token tile of the workspace is written in full (zeros
// past the sequence end and past D), so the attention kernel never reads
// stale bytes.
//
// Loads are 128-bit (8 elements) when D % 8 == 0 and the tensors are 16-byte
// aligned, otherwise element-wise.  Rounding is explicit (__fmul2_rn,
// __fdiv_rn, round-to-nearest-even additions) so the codes match a plain
// IEEE restatement.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "sage_device.cuh"
#include "sage_geom.h"
#include "sage_kernels.h"

namespace sage {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 256;                 // tokens per stats item
// fp32 2^23 + 2^22 + 0x6600: adding it rounds to an integer n (ties to even)
// and leaves 0x6600 + n, the fp16 bits of 1536 + n, in the low 16 bits.
constexpr float kCodeMagic = 12609024.0f;
constexpr float kRintMagic = 12582912.0f;   // 1.5 * 2^23

// Work list of one call (host-computed).
struct Plan {
  int64_t units;      // nseg * Hkv
  int64_t lag;        // units between a unit's stats/Q items and its K/V items
  int64_t total;      // items
  int32_t n_stats;    // stats items per unit
  int32_t n_q;        // Q items per unit (query heads of the kv head x tiles)
  int32_t n_kv;       // K and V items per unit (2 per 128-token block)
  int32_t nqt;        // 128-token tiles per query head
};

struct ProParams {
  SegGeo g;
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* q16;
  uint16_t* k16;
  uint8_t* v8;
  float* s_q;
  float* s_k;
  float* s_v;
  float* k_mean;
  float* v_inv;
  void* ksum;                 // int64 (fp16) or double (bf16) per (unit, channel)
  uint32_t* vmax;             // float bits per (unit, channel)
  uint32_t* done;             // stats items finished per unit
  uint32_t* ready;            // per unit: statistics final
  unsigned long long* next;   // work counter
  uint32_t* status;
  uint64_t timeout_ns;
  float one;                  // 1.0, opaque to the compiler (see code2)
  Plan plan;
};

enum ItemKind { kItemStats = 0, kItemQ = 1, kItemKV = 2 };

struct Item {
  int kind;
  int64_t unit;
  int32_t sub;
};

// Item i of the list.  Slots 0 .. lag-1 hold stats and Q items of units
// 0 .. lag-1; slot j >= lag holds those of unit j and then the K/V items of
// unit j - lag; the last lag slots hold K/V items only.
__device__ __forceinline__ Item decode(const Plan& P, int64_t i) {
  const int64_t a = P.n_stats + P.n_q;
  const int64_t per = a + P.n_kv;
  Item it;
  int64_t off;
  if (i < P.lag * a) {
    it.unit = i / a;
    off = i - it.unit * a;
  } else {
    i -= P.lag * a;
    const int64_t mid = (P.units - P.lag) * per;
    if (i >= mid) {
      i -= mid;
      const int64_t j = i / P.n_kv;
      it.kind = kItemKV;
      it.unit = P.units - P.lag + j;
      it.sub = static_cast<int32_t>(i - j * P.n_kv);
      return it;
    }
    const int64_t j = i / per;
    off = i - j * per;
    if (off >= a) {
      it.kind = kItemKV;
      it.unit = j;
      it.sub = static_cast<int32_t>(off - a);
      return it;
    }
    it.unit = P.lag + j;
  }
  if (off < P.n_stats) {
    it.kind = kItemStats;
    it.sub = static_cast<int32_t>(off);
  } else {
    it.kind = kItemQ;
    it.sub = static_cast<int32_t>(off - P.n_stats);
  }
  return it;
}

// ------------------------------------------------------------ memory ops
// L2 cache policies: keep the stats pass over K/V resident for the K/V items.
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

// The same load, kept by the compiler where written: a second pass re-reads
// its rows (from L1) instead of holding them in registers across a barrier.
__device__ __forceinline__ uint4 ld16_again(const void* p) {
  uint4 u;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "l"(p));
  return u;
}

// Channels c0..c0+7 of one token row as packed 16-bit values (zeros for
// channels >= D).
template <bool kVec, bool kAgain = false>
__device__ __forceinline__ uint4 load8(const uint16_t* row, int c0, int D, uint64_t pol) {
  if constexpr (kVec) {
    if constexpr (kAgain) return c0 < D ? ld16_again(row + c0) : make_uint4(0u, 0u, 0u, 0u);
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

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// ------------------------------------------------------------- numerics
__device__ __forceinline__ uint32_t word(const uint4& u, int i) {
  return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w;
}

// Two packed 16-bit inputs -> two fp32 (exact).  .x is the low half.
template <bool kBf16>
__device__ __forceinline__ float2 cvt2(uint32_t w) {
  if constexpr (kBf16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
  }
}

// Magnitude bits (sign cleared, low 16 bits) -> fp32 value.
template <bool kBf16>
__device__ __forceinline__ float mag_f32(uint32_t m) {
  if constexpr (kBf16) return __uint_as_float(m << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(m)));
}

// Max magnitude (bits) of the eight 16-bit values of a load.  Magnitudes of
// finite fp16/bf16 values order like their bit patterns.
__device__ __forceinline__ uint32_t max_mag8(const uint4& u) {
  const uint32_t m = __vmaxu2(__vmaxu2(u.x & 0x7FFF7FFFu, u.y & 0x7FFF7FFFu),
                              __vmaxu2(u.z & 0x7FFF7FFFu, u.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

// Two int8 codes rint(x * inv) (ties to even) as a pair of exact fp16
// integers, .x in the low half.  |x| <= amax and inv = fl(127 / amax) keep
// |x * inv| below 127.5, so no clamp is needed.  The product must be rounded
// to fp32 before the rounding addition, but the code generator fuses a packed
// multiply followed by a packed add into one packed FMA (rint of the exact
// product), explicit .rn or not.  The addition is therefore written as the
// FMA p * one + magic with `one` a runtime 1.0, which leaves nothing to fuse
// and rounds exactly like p + magic.
__device__ __forceinline__ uint32_t code2(float2 x, float inv, float one) {
  const float2 p = __fmul2_rn(x, make_float2(inv, inv));
  const float2 t = __ffma2_rn(p, make_float2(one, one), make_float2(kCodeMagic, kCodeMagic));
  const uint32_t h = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x5410);
  __half2 hv;
  memcpy(&hv, &h, 4);
  hv = __hsub2(hv, __floats2half2_rn(1536.0f, 1536.0f));
  uint32_t r;
  memcpy(&r, &hv, 4);
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Row maxima of P rows spread over G = 2P lanes (one value per lane and row):
// each exchange halves the values a lane keeps, so lane l ends with the
// maximum of row (l % G) / 2 over the G lanes.
template <int P>
__device__ __forceinline__ uint32_t row_max_transposed(uint32_t (&a)[P], int lane) {
#pragma unroll
  for (int n = P; n > 1; n >>= 1) {
    const int h = n / 2;
    const bool upper = (lane & n) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const uint32_t send = upper ? a[i] : a[i + h];
      const uint32_t keep = upper ? a[i + h] : a[i];
      a[i] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, n));
    }
  }
  return max(a[0], __shfl_xor_sync(0xFFFFFFFFu, a[0], 1));
}

// --------------------------------------------------------------- smem
struct StatsSmem {
  long long part[kThreads / 32][128];
  uint32_t vmax[kThreads / 32][128];
};
struct Smem {
  union {
    StatsSmem st;
    uint32_t vt[128 * 32];            // V tile, [channel][4-token word]
    float red[kThreads / 32];
  } u;
  long long next[2];
  int flag;
};

// Thread 0 waits (bounded) for a unit's ready flag; the CTA learns the
// outcome through shared memory.  Returns false on timeout.
__device__ __forceinline__ bool wait_ready(const ProParams& p, int64_t unit, Smem& sm) {
  if (threadIdx.x == 0) {
    const uint32_t* f = p.ready + unit;
    int ok = ld_acquire(f) != 0u;
    if (!ok) {
      const uint64_t t0 = global_timer_ns();
      while (true) {
        __nanosleep(128);
        if (ld_acquire(f) != 0u) { ok = 1; break; }
        if (global_timer_ns() - t0 > p.timeout_ns) {
          atomicOr(p.status, kStatusTimeout);
          break;
        }
      }
    }
    sm.flag = ok;
  }
  __syncthreads();
  return sm.flag != 0;
}

// ---------------------------------------------------------------- stats
template <bool kVec, bool kBf16, int DP>
__device__ __forceinline__ void stats_item(const ProParams& p, int64_t unit, int chunk,
                                           Smem& sm) {
  constexpr int G = DP / 8, R = kThreads / G, TPT = kChunk / R;   // TPT 16 or 8
  const SegGeo& g = p.g;
  const int64_t s = unit / g.Hkv, h = unit % g.Hkv;
  int64_t start = 0, len = g.Lk;
  if (g.varlen && !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len)) {
    if (threadIdx.x == 0 && chunk == 0) atomicOr(p.status, kStatusBadSeqlens);
    len = 0;
  }
  const int64_t chunks = len > 0 ? (len + kChunk - 1) / kChunk : 1;
  if (chunk >= chunks) return;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const int D = static_cast<int>(g.D);
  const int64_t base = (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                       h * g.k_head_stride;
  const uint16_t* kb = p.k + base;
  const uint16_t* vb = p.v + base;
  const int64_t t0 = static_cast<int64_t>(chunk) * kChunk;
  const int64_t t1 = min(len, t0 + kChunk);
  const uint64_t keep = policy_evict_last();

  // fp16 keys: per thread at most 16 tokens, each split exactly into
  // hi = rint(16 k) and lo = k - hi / 16 (a multiple of 2^-24, |lo| <= 1/32);
  // 16 of either sum exactly in fp32 (|sum hi| < 2^24, |sum lo| * 2^24 <=
  // 2^23).  The FP64 pipe (slow on GB300) stays out of the loop.  bf16 keys:
  // fp64 sums.
  float2 hs[4], ls[4];
  double ds[8];
  uint32_t vm[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hs[i] = make_float2(0.0f, 0.0f);
    ls[i] = make_float2(0.0f, 0.0f);
    vm[i] = 0u;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) ds[i] = 0.0;

#pragma unroll
  for (int j0 = 0; j0 < TPT; j0 += 4) {
    uint4 kr[4], vr[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {             // 8 loads in flight per thread
      const int64_t t = t0 + r + static_cast<int64_t>(R) * (j0 + u);
      const bool in = t < t1;
      kr[u] = in ? load8<kVec>(kb + t * g.k_tok_stride, c0, D, keep) : make_uint4(0u, 0u, 0u, 0u);
      vr[u] = in ? load8<kVec>(vb + t * g.k_tok_stride, c0, D, keep) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        vm[i] = __vmaxu2(vm[i], word(vr[u], i) & 0x7FFF7FFFu);
        const float2 x = cvt2<kBf16>(word(kr[u], i));
        if constexpr (kBf16) {
          ds[2 * i] += static_cast<double>(x.x);
          ds[2 * i + 1] += static_cast<double>(x.y);
        } else {
          const float2 tr = __ffma2_rn(x, make_float2(16.0f, 16.0f),
                                       make_float2(kRintMagic, kRintMagic));
          const float2 hi = __fadd2_rn(tr, make_float2(-kRintMagic, -kRintMagic));
          const float2 lo = __ffma2_rn(hi, make_float2(-0.0625f, -0.0625f), x);
          hs[i] = __fadd2_rn(hs[i], hi);
          ls[i] = __fadd2_rn(ls[i], lo);
        }
      }
    }
  }

  // combine the rows: lanes holding the same channels (warp shuffles), then
  // the eight warps through shared memory, one channel per thread
  long long part[8];
  uint32_t am[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (kBf16) {
      part[2 * i] = __double_as_longlong(ds[2 * i]);
      part[2 * i + 1] = __double_as_longlong(ds[2 * i + 1]);
    } else {
      part[2 * i] = static_cast<long long>(__float2int_rn(hs[i].x)) * 1048576ll +
                    __float2int_rn(ls[i].x * 16777216.0f);
      part[2 * i + 1] = static_cast<long long>(__float2int_rn(hs[i].y)) * 1048576ll +
                        __float2int_rn(ls[i].y * 16777216.0f);
    }
    am[2 * i] = vm[i] & 0xFFFFu;
    am[2 * i + 1] = vm[i] >> 16;
  }
#pragma unroll
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const long long other = __shfl_xor_sync(0xFFFFFFFFu, part[i], o);
      if constexpr (kBf16)
        part[i] = __double_as_longlong(__longlong_as_double(part[i]) +
                                       __longlong_as_double(other));
      else
        part[i] += other;
      am[i] = max(am[i], __shfl_xor_sync(0xFFFFFFFFu, am[i], o));
    }
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane < G) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sm.u.st.part[wid][c0 + i] = part[i];
      sm.u.st.vmax[wid][c0 + i] = am[i];
    }
  }
  __syncthreads();
  const int64_t obase = unit * DP;
  if (threadIdx.x < D) {
    const int c = threadIdx.x;
    long long si = 0;
    double sd = 0.0;
    uint32_t a = 0u;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      if constexpr (kBf16) sd += __longlong_as_double(sm.u.st.part[w][c]);
      else si += sm.u.st.part[w][c];
      a = max(a, sm.u.st.vmax[w][c]);
    }
    if constexpr (kBf16) atomicAdd(static_cast<double*>(p.ksum) + obase + c, sd);
    else atomicAdd(static_cast<unsigned long long*>(p.ksum) + obase + c,
                   static_cast<unsigned long long>(si));
    atomicMax(p.vmax + obase + c, __float_as_uint(mag_f32<kBf16>(a)));
    __threadfence();
  }
  // The unit's last stats item turns the sums into the K mean and the V
  // scales while they are hot in L2, then raises the ready flag.
  __syncthreads();
  if (threadIdx.x == 0)
    sm.flag = atomicAdd(p.done + unit, 1u) == static_cast<uint32_t>(chunks - 1);
  __syncthreads();
  const bool last = sm.flag != 0;
  __syncthreads();                             // sm.flag is reused by the next item
  if (!last) return;
  __threadfence();
  for (int c = threadIdx.x; c < DP; c += kThreads) {
    const int64_t i = obase + c;
    double S;
    if constexpr (kBf16)
      S = __longlong_as_double(__ldcg(static_cast<const long long*>(p.ksum) + i));
    else
      S = __ll2double_rn(__ldcg(static_cast<const long long*>(p.ksum) + i)) *
          5.9604644775390625e-08;   // 2^-24, exact
    p.k_mean[i] = len > 0 ? __double2float_rn(__ddiv_rn(S, static_cast<double>(len))) : 0.0f;
    const float a = __uint_as_float(__ldcg(p.vmax + i));
    p.s_v[i] = __fdiv_rn(a, 448.0f);
    p.v_inv[i] = a > 0.0f ? __fdiv_rn(448.0f, a) : 0.0f;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) st_release(p.ready + unit, 1u);
}

// ------------------------------------------------------------------- Q
template <bool kVec, bool kBf16, int DP>
__device__ __forceinline__ void q_item(const ProParams& p, int64_t unit, int sub) {
  constexpr int G = DP / 8, R = kThreads / G, P = kBlockM / R;   // P 8 or 4
  const SegGeo& g = p.g;
  const int64_t grp = g.Hq / g.Hkv;
  const int64_t s = unit / g.Hkv;
  const int64_t hq = (unit % g.Hkv) * grp + sub / p.plan.nqt;
  const int64_t qt = sub % p.plan.nqt;
  int64_t start = 0, len = g.Lq;
  if (g.varlen && !seg_range(g.cu_q, s, g.total_q, g.max_q, &start, &len)) {
    if (threadIdx.x == 0 && sub == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  const int64_t t0 = qt * kBlockM;
  if (t0 >= len) return;
  const int lane = threadIdx.x & 31;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const int D = static_cast<int>(g.D);
  const uint16_t* qb = p.q + (g.varlen ? start * g.q_tok_stride : s * g.q_seg_stride) +
                       hq * g.q_head_stride;
  const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hq, g.q_head_rows) +
                       hq * g.q_head_rows + t0;
  const uint64_t once = policy_evict_first();
  uint4 raw[P];
#pragma unroll
  for (int i = 0; i < P; ++i) {                // all loads first: one round trip
    const int64_t t = t0 + r + R * i;
    raw[i] = t < len ? load8<kVec>(qb + t * g.q_tok_stride, c0, D, once)
                     : make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t am[P];
#pragma unroll
  for (int i = 0; i < P; ++i) am[i] = max_mag8(raw[i]);
  // lane l now holds the max of row (l % G) / 2; even lanes form the
  // multiplier 127 / amax, odd lanes the scale amax / 127 (one division each)
  const float amax = mag_f32<kBf16>(row_max_transposed<P>(am, lane));
  const bool odd = (lc & 1) != 0;
  const float quo = __fdiv_rn(odd ? amax : 127.0f, odd ? 127.0f : amax);
  const float mine = amax > 0.0f ? quo : 0.0f;
  if (odd) p.s_q[row0 + r + R * (lc >> 1)] = mine;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const float inv = __shfl_sync(0xFFFFFFFFu, mine, (lane & ~(G - 1)) | (2 * i));
    uint4 o;
    o.x = code2(cvt2<kBf16>(raw[i].x), inv, p.one);
    o.y = code2(cvt2<kBf16>(raw[i].y), inv, p.one);
    o.z = code2(cvt2<kBf16>(raw[i].z), inv, p.one);
    o.w = code2(cvt2<kBf16>(raw[i].w), inv, p.one);
    *reinterpret_cast<uint4*>(p.q16 + (row0 + r + R * i) * DP + c0) = o;
  }
}

// ------------------------------------------------------------------- K
template <bool kVec, bool kBf16, int DP>
__device__ __forceinline__ void k_item(const ProParams& p, int64_t unit, int kb_idx,
                                       Smem& sm) {
  constexpr int G = DP / 8, R = kThreads / G, P = kBlockN / R;
  const SegGeo& g = p.g;
  const int64_t s = unit / g.Hkv, h = unit % g.Hkv;
  int64_t start = 0, len = g.Lk;
  if (g.varlen && !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len)) return;
  const int64_t t0 = static_cast<int64_t>(kb_idx) * kBlockN;
  if (t0 >= len) return;
  if (!wait_ready(p, unit, sm)) return;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const int D = static_cast<int>(g.D);
  const uint16_t* kb = p.k + (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                       h * g.k_head_stride;
  const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hkv, g.k_head_rows) +
                       h * g.k_head_rows + t0;
  float2 nmean[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    nmean[i] = make_float2(-__ldcg(p.k_mean + unit * DP + c0 + 2 * i),
                           -__ldcg(p.k_mean + unit * DP + c0 + 2 * i + 1));
  const uint64_t last_use = policy_evict_first();
  // smoothing k - mean (fp32) is recomputed in both passes; the second pass
  // re-reads its rows; rows past the sequence end count as zero
  float am = 0.0f;
  {
    uint4 raw[P];
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int64_t t = t0 + r + R * i;
      raw[i] = t < len ? load8<kVec>(kb + t * g.k_tok_stride, c0, D, last_use)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < P; ++i) {
      float ar = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 kh = __fadd2_rn(cvt2<kBf16>(word(raw[i], j)), nmean[j]);
        ar = fmaxf(ar, fmaxf(fabsf(kh.x), fabsf(kh.y)));
      }
      if (t0 + r + R * i < len) am = fmaxf(am, ar);
    }
  }
  am = warp_max(am);
  if ((threadIdx.x & 31) == 0) sm.u.red[threadIdx.x >> 5] = am;
  __syncthreads();
  am = sm.u.red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) am = fmaxf(am, sm.u.red[w]);
  const float kinv = am > 0.0f ? __fdiv_rn(127.0f, am) : 0.0f;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int64_t t = t0 + r + R * i;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (t < len) {
      const uint4 x = load8<kVec, true>(kb + t * g.k_tok_stride, c0, D, last_use);
      o.x = code2(__fadd2_rn(cvt2<kBf16>(x.x), nmean[0]), kinv, p.one);
      o.y = code2(__fadd2_rn(cvt2<kBf16>(x.y), nmean[1]), kinv, p.one);
      o.z = code2(__fadd2_rn(cvt2<kBf16>(x.z), nmean[2]), kinv, p.one);
      o.w = code2(__fadd2_rn(cvt2<kBf16>(x.w), nmean[3]), kinv, p.one);
    }
    *reinterpret_cast<uint4*>(p.k16 + (row0 + r + R * i) * DP + c0) = o;
  }
  if (threadIdx.x == 0) p.s_k[row0 / kBlockN] = __fdiv_rn(am, 127.0f);
}

// ------------------------------------------------------------------- V
// A thread quantises 8 channels of 4 consecutive tokens and packs, per
// channel, the 4 token bytes into one word; word (c, w) of the shared tile
// sits at c * 32 + (w ^ 4 * (c / 8 % 8)), which spreads the writes over banks
// and keeps every group of four words (16 bytes of a row) contiguous.
template <bool kVec, bool kBf16, int DP>
__device__ __forceinline__ void v_item(const ProParams& p, int64_t unit, int kb_idx,
                                       Smem& sm) {
  constexpr int G = DP / 8, RG = kThreads / G, NTW = (kBlockN / 4) / RG;   // NTW 2 or 1
  const SegGeo& g = p.g;
  const int64_t s = unit / g.Hkv, h = unit % g.Hkv;
  int64_t start = 0, len = g.Lk;
  if (g.varlen && !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len)) return;
  const int64_t t0 = static_cast<int64_t>(kb_idx) * kBlockN;
  if (t0 >= len) return;
  if (!wait_ready(p, unit, sm)) return;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const int D = static_cast<int>(g.D);
  const uint16_t* vb = p.v + (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                       h * g.k_head_stride;
  float vinv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) vinv[i] = __ldcg(p.v_inv + unit * DP + c0 + i);
  const uint64_t last_use = policy_evict_first();
  uint4 raw[NTW][4];
#pragma unroll
  for (int a = 0; a < NTW; ++a) {               // all loads first: one round trip
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t t = t0 + 4 * (r + a * RG) + e;
      raw[a][e] = t < len ? load8<kVec>(vb + t * g.k_tok_stride, c0, D, last_use)
                          : make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int a = 0; a < NTW; ++a) {
    const int tw = r + a * RG;
#pragma unroll
    for (int j = 0; j < 4; ++j) {               // channels c0 + 2j, c0 + 2j + 1
      const float2 x0 = cvt2<kBf16>(word(raw[a][0], j));
      const float2 x1 = cvt2<kBf16>(word(raw[a][1], j));
      const float2 x2 = cvt2<kBf16>(word(raw[a][2], j));
      const float2 x3 = cvt2<kBf16>(word(raw[a][3], j));
      const float2 i0 = make_float2(vinv[2 * j], vinv[2 * j]);
      const float2 i1 = make_float2(vinv[2 * j + 1], vinv[2 * j + 1]);
      const float2 a01 = __fmul2_rn(make_float2(x0.x, x1.x), i0);
      const float2 a23 = __fmul2_rn(make_float2(x2.x, x3.x), i0);
      const float2 b01 = __fmul2_rn(make_float2(x0.y, x1.y), i1);
      const float2 b23 = __fmul2_rn(make_float2(x2.y, x3.y), i1);
      const uint32_t wa = __byte_perm(pack_e4m3x2(a01.x, a01.y), pack_e4m3x2(a23.x, a23.y), 0x5410);
      const uint32_t wb = __byte_perm(pack_e4m3x2(b01.x, b01.y), pack_e4m3x2(b23.x, b23.y), 0x5410);
      const int ca = c0 + 2 * j, cb = ca + 1;
      sm.u.vt[ca * 32 + (tw ^ (((ca >> 3) & 7) << 2))] = wa;
      sm.u.vt[cb * 32 + (tw ^ (((cb >> 3) & 7) << 2))] = wb;
    }
  }
  __syncthreads();
  const int64_t vrow0 = (g.varlen ? 0 : s * g.Hkv * DP) + h * DP;
  const int64_t vcol0 = (g.varlen ? ws_seg_base(1, s, start, 0, 0) : 0) + t0;
  constexpr int kQuads = DP * (kBlockN / 16);   // 16-byte pieces
#pragma unroll
  for (int qi = threadIdx.x; qi < kQuads; qi += kThreads) {
    const int c = qi / (kBlockN / 16), tw = 4 * (qi % (kBlockN / 16));
    const uint4 val = *reinterpret_cast<const uint4*>(&sm.u.vt[c * 32 + (tw ^ (((c >> 3) & 7) << 2))]);
    *reinterpret_cast<uint4*>(p.v8 + (vrow0 + c) * g.v_cols + vcol0 + 4 * tw) = val;
  }
}

// --------------------------------------------------------------- kernel
template <bool kVec, bool kBf16, int DP>
__global__ void __launch_bounds__(kThreads, 3)
prologue_kernel(const __grid_constant__ ProParams p) {
  __shared__ __align__(16) Smem sm;
  if (threadIdx.x == 0) sm.next[0] = static_cast<long long>(atomicAdd(p.next, 1ull));
  __syncthreads();
  long long cur = sm.next[0];
  int buf = 1;
  while (cur < p.plan.total) {
    // take the next item now; its index is needed only after this one
    unsigned long long nxt = 0;
    if (threadIdx.x == 0) nxt = atomicAdd(p.next, 1ull);
    const Item it = decode(p.plan, cur);
    if (it.kind == kItemStats) {
      stats_item<kVec, kBf16, DP>(p, it.unit, it.sub, sm);
    } else if (it.kind == kItemQ) {
      q_item<kVec, kBf16, DP>(p, it.unit, it.sub);
    } else if ((it.sub & 1) == 0) {
      k_item<kVec, kBf16, DP>(p, it.unit, it.sub >> 1, sm);
    } else {
      v_item<kVec, kBf16, DP>(p, it.unit, it.sub >> 1, sm);
    }
    if (threadIdx.x == 0) sm.next[buf] = static_cast<long long>(nxt);
    __syncthreads();
    cur = sm.next[buf];
    buf ^= 1;
  }
}

// Work list of a call: n_q = n_kv = 0 gives statistics only.
Plan make_plan(const SegGeo& g, bool with_quant, int64_t grid) {
  Plan P{};
  const int64_t maxk = g.varlen ? g.max_k : g.Lk;
  const int64_t maxq = g.varlen ? g.max_q : g.Lq;
  P.units = g.nseg * g.Hkv;
  P.n_stats = static_cast<int32_t>(maxk > 0 ? (maxk + kChunk - 1) / kChunk : 1);
  P.nqt = static_cast<int32_t>((maxq + kBlockM - 1) / kBlockM);
  if (with_quant) {
    P.n_q = static_cast<int32_t>(g.Hq / g.Hkv) * P.nqt;
    P.n_kv = static_cast<int32_t>(2 * ((maxk + kBlockN - 1) / kBlockN));
  }
  const int64_t per = P.n_stats + P.n_q + P.n_kv;
  if (P.n_kv == 0) {
    P.lag = P.units;                      // no K/V items: everything in the first phase
  } else {
    // at least twice the CTAs in flight between a unit's stats and its K/V
    // items, while the K and V of the units in between stay well inside L2
    const int64_t unit_bytes = 4 * maxk * g.D;
    int64_t lag = (2 * grid + per - 1) / per;
    const int64_t l2_budget = 40ll << 20;
    if (unit_bytes > 0 && lag * unit_bytes > l2_budget) lag = l2_budget / unit_bytes;
    if (lag < 1) lag = 1;
    if (lag > P.units) lag = P.units;
    P.lag = lag;
  }
  P.total = P.units * per;
  return P;
}

template <bool kVec, bool kBf16, int DP>
cudaError_t launch_t(ProParams& prm, bool with_quant, cudaStream_t st) {
  static int per_sm[64] = {};                  // resident CTAs per SM, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (per_sm[dev] == 0) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prologue_kernel<kVec, kBf16, DP>,
                                                      kThreads, 0);
    if (e != cudaSuccess) return e;
    per_sm[dev] = n > 0 ? n : 1;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int64_t grid = static_cast<int64_t>(sms) * per_sm[dev];
  prm.plan = make_plan(prm.g, with_quant, grid);
  if (grid > prm.plan.total) grid = prm.plan.total;
  if (grid <= 0) return cudaSuccess;
  prologue_kernel<kVec, kBf16, DP><<<static_cast<unsigned>(grid), kThreads, 0, st>>>(prm);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_any(ProParams& prm, bool vec, bool with_quant, cudaStream_t st) {
  const bool bf16 = prm.g.dtype == 1;
  const bool d64 = prm.g.Dp == 64;
  if (vec) {
    if (bf16) return d64 ? launch_t<true, true, 64>(prm, with_quant, st)
                         : launch_t<true, true, 128>(prm, with_quant, st);
    return d64 ? launch_t<true, false, 64>(prm, with_quant, st)
               : launch_t<true, false, 128>(prm, with_quant, st);
  }
  if (bf16) return d64 ? launch_t<false, true, 64>(prm, with_quant, st)
                       : launch_t<false, true, 128>(prm, with_quant, st);
  return d64 ? launch_t<false, false, 64>(prm, with_quant, st)
             : launch_t<false, false, 128>(prm, with_quant, st);
}

}  // namespace

cudaError_t launch_prologue(const SegGeo& g, const PrologueBuffers& b,
                            bool vec, cudaStream_t st) {
  ProParams prm{};
  prm.g = g;
  prm.q = b.q; prm.k = b.k; prm.v = b.v;
  prm.q16 = b.q16; prm.k16 = b.k16; prm.v8 = b.v8;
  prm.s_q = b.s_q; prm.s_k = b.s_k; prm.s_v = b.s_v;
  prm.k_mean = b.k_mean; prm.v_inv = b.v_inv;
  prm.ksum = b.ksum; prm.vmax = b.vmax; prm.done = b.done; prm.ready = b.ready;
  prm.next = b.next; prm.status = b.status; prm.timeout_ns = b.timeout_ns;
  prm.one = 1.0f;
  return launch_any(prm, vec, true, st);
}

// ------------------------------------------- statistics without allocation
// Scratch of the allocation-free statistics entry point: a header (status
// word, work counter, per-unit done counters and ready flags), then
// per-channel K sums (8 B), V maxima (4 B) and V multipliers (4 B) for at
// most kStaticStatEntries (segment, kv head, channel) triples.  It lives in
// the module image, so every device that loads this library holds it until
// the process exits; concurrent calls share it.
namespace {
constexpr int64_t kMaxStaticUnits = kStaticStatEntries / 64;
constexpr size_t kStaticHeader = 256 + 2 * 4 * kMaxStaticUnits;
__device__ __align__(256) unsigned char g_stats_scratch[
    kStaticHeader + kStaticStatEntries * (8 + 4 + 4)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

cudaError_t launch_kv_stats_static(const SegGeo& g, const uint16_t* k,
                                   const uint16_t* v, float* k_mean, float* s_v,
                                   bool vec, uint64_t timeout_ns, cudaStream_t st) {
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
  const int64_t units = g.nseg * g.Hkv;
  if (units * g.Dp > kStaticStatEntries) return cudaErrorInvalidValue;
  // the previous call's counters, sums and maxima are still there: clear them
  e = cudaMemsetAsync(base, 0, kStaticHeader + kStaticStatEntries * 12, st);
  if (e != cudaSuccess) return e;
  ProParams prm{};
  prm.g = g;
  prm.k = k; prm.v = v;
  prm.k_mean = k_mean; prm.s_v = s_v;
  prm.status = reinterpret_cast<uint32_t*>(base);
  prm.next = reinterpret_cast<unsigned long long*>(base + 8);
  prm.done = reinterpret_cast<uint32_t*>(base + 256);
  prm.ready = reinterpret_cast<uint32_t*>(base + 256 + 4 * kMaxStaticUnits);
  prm.ksum = base + kStaticHeader;
  prm.vmax = reinterpret_cast<uint32_t*>(base + kStaticHeader + kStaticStatEntries * 8);
  prm.v_inv = reinterpret_cast<float*>(base + kStaticHeader + kStaticStatEntries * 12);
  prm.timeout_ns = timeout_ns;
  prm.one = 1.0f;
  return launch_any(prm, vec, false, st);
}

}  // namespace sage
