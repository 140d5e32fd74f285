// Quantisation prologue (HBM-bound), sm_103a.
//
// What it computes follows stable-diffusion.cpp's "SageAttention" page (the
// FP8-path paragraph: smooth K, quantise V per channel, pad and permute V for
// FP8 tensor cores; "Use": head_dim zero-padded to 64/128), the SageAttention
// overview's Core features (INT8 Q/K, smoothing) and the SageAttention-RDNA4
// v0.4.0 notes (key mean summed in fp64, 64-bit offsets).
//
// One persistent kernel, three CTAs per SM, launched cooperatively (every CTA
// resident).  A CTA has eight consumer warps, a producer warp and a helper
// warp around a ring of two 32 KB shared-memory stages.  The producer takes
// work items from a counter in the workspace and copies each item's 128-token
// input tile into a free stage with a tensor copy (TMA), zero-padded to Dp
// channels; the consumers quantise the tile in the stage and release it.  A
// unit is one (segment, kv head); its items are
//   stats K   128 keys: exact per-channel sums (int64 fixed point at 2^-24
//             for fp16, fp64 for bf16), added to the unit's accumulators;
//   stats V   128 values: per-channel max |v|, likewise;
//   Q         128 tokens of one query head that reads this kv head: int8
//             codes (stored as exact fp16 integers, the tensor-core operand),
//             one scale per token;
//   K         128 keys: smoothed K (k - mean, fp32) -> int8 codes, one scale
//             per block (the unit's K sums are copied next to the tile and
//             turned into the mean there);
//   V         128 values: e4m3 per channel (the unit's maxima are copied
//             next to the tile and turned into multipliers there),
//             transposed to channel-major;
//   final     (statistics-only calls) the unit's K mean and V scales.
// The units are cut into groups of about 100 MB of K and V, and each group
// has two lists: A (its stats tiles) and B (its K and V tiles, or its final
// items, which need the group's statistics).  A items never wait.  Once a
// CTA's consumers are done with every A item of group g it has taken, its
// helper warp arrives at the group's barrier (a counter, one release per
// CTA and group); B items of the group are taken only after every CTA has
// arrived, so they find the group's sums complete and their K and V, read
// by the A list with an evict-last hint, still in L2.  Few large groups
// measured faster than many small ones (fewer barrier rounds; the Q list
// fills the waits).  Beyond L2, the part of K and V that does not stay there
// is read again from HBM.  The Q tiles depend on nothing: they form one more
// list, taken only when neither of the others has an item ready, so they
// fill the barrier waits and the end.  A unit's items are its tiles up to
// the longest sequence's count; packed sequences whose lists would then be
// a quarter empty or more take lists over each sequence's own tiles instead
// (packed_lists, vdecode).  Nothing waits inside a list, and
// every wait is bounded (timeout -> status bit).  Every 128-token
// tile of the workspace is written in full (zeros past the sequence end and
// past D), so the attention kernel never reads stale bytes.
//
// Without 16-byte aligned rows (D % 8 != 0 or unaligned tensors) the same
// kernel runs with element-wise global loads instead of tensor copies.
// Rounding is explicit (packed .rn multiplies, __fdiv_rn, round-to-nearest-
// even additions) so the codes match a plain IEEE restatement.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "sage_device.cuh"
#include "sage_geom.h"
#include "sage_kernels.h"

namespace sage {

namespace {

constexpr int kConsumers = 256;              // eight consumer warps
constexpr int kProducerWarp = 8;
constexpr int kHelperWarp = 9;
constexpr int kThreads = kConsumers + 64;
constexpr int kStages = 2;                   // three CTAs per SM: more tiles in work at once
constexpr int kQueue = 8;                    // finished stats tiles awaiting the helper
constexpr int kMaxGroups = 64;               // counters per list in the workspace
constexpr int64_t kGroupBytes = 100ll << 20; // K and V bytes of a group (target)
constexpr int64_t kL2Hold = 128ll << 20;     // K and V bytes held in L2 between reads
constexpr int kTileBytes = 128 * 128 * 2;    // 128 rows of up to 128 16-bit values
constexpr uint32_t kSleepNs = 20000;         // suspend hint of barrier waits
constexpr int kCuSmem = 256;                 // packed sequences: offsets held in shared memory
// fp32 2^23 + 2^22 + 0x6600: adding it rounds to an integer n (ties to even)
// and leaves 0x6600 + n, the fp16 bits of 1536 + n, in the low 16 bits.
constexpr float kCodeMagic = 12609024.0f;
constexpr float kRintMagic = 12582912.0f;    // 1.5 * 2^23

enum ItemKind {
  kStatsK = 0, kStatsV = 1, kQ = 2, kK = 3, kV = 4, kEnd = 5, kGroupEnd = 6, kFinal = 7
};

// Work of one call (host-computed; every count fits in 31 bits).  The units
// are cut into groups.  Each group has two item lists with their own
// counters: A (stats tiles, no dependencies) and B (K and V tiles, or one
// final item per unit in a statistics-only call; they need the group's
// sums).  A CTA whose consumers are done with its last A item of group g
// says so at group g's barrier; once every CTA has, the group's sums are
// complete and its B items may be taken.  A items never wait, and may run
// `lead` groups ahead of the B items, which bounds the K and V held in L2
// between their two reads.  Q tiles form a single list of their own.
struct Plan {
  int32_t units;      // nseg * Hkv
  int32_t group;      // units per group
  int32_t groups;
  int32_t lead;       // groups the A list may run ahead of the B list
  int32_t n_stats;    // stats items per unit (K and V tiles alternate)
  int32_t n_q;        // Q items per unit (query heads of the kv head x tiles)
  int32_t n_kv;       // K and V items per unit (K and V tiles alternate)
  int32_t n_b;        // B items per unit: n_kv, or 1 (final) without quantisation
  int32_t nqt;        // 128-token tiles per query head
  int32_t open;       // the statistics are final already (no A list, no barriers)
  int32_t q_first;    // Q items before A items
};

// What a launch does (see make_plan).
enum PlanMode : int {
  kPlanAll = 0,       // statistics, Q, then K and V once a group's statistics are final
  kPlanStats = 1,     // statistics and the final items only
  kPlanStatsQ = 2,    // Q first, then statistics and the final items
  kPlanKV = 3,        // K and V from final statistics
};

struct ProParams {
  SegGeo g;
  CUtensorMap mq, mk, mv;     // 3D maps of q, k, v (tensor-copy path)
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
  unsigned int* cnt_a;        // [kMaxGroups] A-list counters
  unsigned int* cnt_b;        // [kMaxGroups] B-list counters
  unsigned int* gbar;         // [kMaxGroups] CTAs done with the group's A list
  unsigned int* cnt_q;        // Q-list counter
  uint32_t* status;
  uint64_t timeout_ns;
  int32_t q_hnd, k_hnd;       // 1: tiles are (head, token) planes; 0: token-major
  float one;                  // 1.0, opaque to the compiler (see code2)
  int32_t v16;                // V written as fp16 (FP16-PV variant) instead of e4m3
  Plan plan;
};

struct Slot {
  int32_t kind, sub, unit, nvalid;
};

struct alignas(1024) PSmem {
  unsigned char tile[kStages][kTileBytes];
  alignas(16) unsigned char aux[kStages][1024];   // K items: the unit's K sums; V: its maxima
  float coef[128];            // the current item's K mean or V multipliers
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t qfull[kQueue];
  uint64_t qempty[kQueue];
  int32_t queue[kQueue];      // unit of a finished stats tile, or a marker
  int32_t qinfo[kQueue];      // stats tile: 2 * stage + (1 for V)
  Slot slot[kStages];
  float red[8];
  int abort;
  // packed instances (at most kCuSmem sequences): cu_seqlens_k and _q,
  // copied at the start (every item looks up its sequence's offsets; from
  // global memory each lookup is an L2 round trip on the producer's path)
  int32_t cu_k[kCuSmem + 1];
  int32_t cu_q[kCuSmem + 1];
};

__device__ __forceinline__ int group_units(const Plan& P, int g) {
  return min(P.units - g * P.group, P.group);
}

// Item i of group g's A list (the stats tiles of each unit, K and V tiles
// alternating).
__device__ __forceinline__ void decode_a(const Plan& P, int g, int i, int* kind, int* unit,
                                         int* sub) {
  const int u = i / P.n_stats, off = i - u * P.n_stats;
  *unit = g * P.group + u;
  *kind = (off & 1) ? kStatsV : kStatsK;
  *sub = off >> 1;
}

// Item i of the Q list (the Q tiles of each unit in turn).
__device__ __forceinline__ void decode_q(const Plan& P, int i, int* kind, int* unit, int* sub) {
  const int u = i / P.n_q;
  *unit = u;
  *kind = kQ;
  *sub = i - u * P.n_q;
}

// Item i of group g's B list (K and V tiles alternate; without quantisation
// one final item per unit).
__device__ __forceinline__ void decode_b(const Plan& P, int g, int i, int* kind, int* unit,
                                         int* sub) {
  const int u = i / P.n_b, off = i - u * P.n_b;
  *unit = g * P.group + u;
  *kind = P.n_kv == 0 ? kFinal : (off & 1) ? kV : kK;
  *sub = P.n_kv == 0 ? 0 : off >> 1;
}

// Packed sequences.  Lists sized by the longest sequence would carry every
// shorter sequence's missing tiles as empty items (41 % of them for 8
// sequences of 2k-16k tokens), each still claimed and decoded.  The packed
// lists run over virtual tiles instead: sequence s owns tiles vt(s) ..
// vt(s + 1) - 1, vt(s) = s + floor(cu[s] / 128), which is its workspace base
// over 128 (ws_seg_base).  That is at least its real tile count and at most
// one more, so a list carries at most one or two empty items per sequence.
// Units stay sequence-major (unit = s Hkv + h); a list holds m items per
// virtual tile and unit (K and V: 2; Q: the kv head's query heads).  The
// entries are clamped to [0, total] and vt(nseg) comes from the host's
// total, so every list stays within the sizes the host checked even for
// inconsistent offsets (which check_offsets reports).
__device__ __forceinline__ int vtile(const int32_t* cu, int s, int nseg, int64_t total) {
  if (s <= 0) return 0;
  int64_t c = s >= nseg ? total : static_cast<int64_t>(cu[s]);
  c = c < 0 ? 0 : (c > total ? total : c);
  return s + static_cast<int>(c >> 7);
}

// First item of unit u in a packed list (u = nseg Hkv: the list's end).
__device__ __forceinline__ int vstart(const int32_t* cu, int nseg, int64_t total, int Hkv,
                                      int m, int u) {
  const int s = u / Hkv, h = u - s * Hkv;
  const int v0 = vtile(cu, s, nseg, total);
  const int w = s < nseg ? vtile(cu, s + 1, nseg, total) - v0 : 0;
  return m * (Hkv * v0 + h * w);
}

// The sequence of the last item a producer decoded from a list: its
// virtual tiles v0 .. v0 + w - 1.  A producer's claims from a list increase
// by about one item per CTA, so the next item is mostly in the same
// sequence and needs no search (each search step is a dependent load).
struct SeqCache {
  int s = 0, v0 = 0, w = 0;
};

// Item i of a packed list: its unit, virtual tile t within the unit's
// sequence and place j in [0, m).  False for inconsistent offsets.
__device__ __forceinline__ bool vdecode(const int32_t* cu, int nseg, int64_t total, int Hkv,
                                        int m, int i, SeqCache& c, int* unit, int* t, int* j) {
  const int q = i / m;                 // (virtual tile, kv head) slot
  *j = i - q * m;
  if (q < Hkv * c.v0 || q >= Hkv * (c.v0 + c.w)) {
    int lo = 0, hi = nseg;             // the last sequence s with Hkv vt(s) <= q
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (Hkv * vtile(cu, mid, nseg, total) <= q) lo = mid;
      else hi = mid;
    }
    c.s = lo;
    c.v0 = vtile(cu, lo, nseg, total);
    c.w = vtile(cu, lo + 1, nseg, total) - c.v0;
  }
  const int r = q - Hkv * c.v0;
  if (c.w <= 0 || r < 0 || r >= Hkv * c.w) return false;
  const int h = r / c.w;
  *unit = c.s * Hkv + h;
  *t = r - h * c.w;
  return true;
}

// ------------------------------------------------------------ memory ops
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

__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, int32_t z, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
         "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, int32_t z, int32_t w,
                                                 uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
         "r"(w), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Contiguous global -> shared copy (16-byte aligned ends) completing on bar.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}


// Barrier of the eight consumer warps (the other two warps run on their own).
__device__ __forceinline__ void csync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// mbarrier wait that lets the warp sleep until the phase completes (or the
// hint runs out) instead of polling; bounded like mbar_wait.
__device__ __forceinline__ bool mbar_sleep_wait(uint64_t* bar, uint32_t parity,
                                                volatile int* abort, uint32_t* status,
                                                uint64_t timeout_ns) {
  uint64_t t0 = 0;
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepNs) : "memory");
    if (ok) return true;
    if (abort != nullptr && *abort) return false;
    const uint64_t now = global_timer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > timeout_ns) {
      if (abort != nullptr) *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
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

// Max magnitude (bits) of the eight 16-bit values of a row piece.
// Magnitudes of finite fp16/bf16 values order like their bit patterns.
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

// Segment bounds (dense: the whole sequence) from offsets cu (g.cu_k or
// g.cu_q, or their shared-memory copies); false on bad cu_seqlens.
__device__ __forceinline__ bool key_range(const SegGeo& g, const int32_t* cu, int64_t s,
                                          int64_t* start, int64_t* len) {
  *start = 0;
  *len = g.Lk;
  return !g.varlen || seg_range(cu, s, g.total_k, g.max_k, start, len);
}
__device__ __forceinline__ bool query_range(const SegGeo& g, const int32_t* cu, int64_t s,
                                            int64_t* start, int64_t* len) {
  *start = 0;
  *len = g.Lq;
  return !g.varlen || seg_range(cu, s, g.total_q, g.max_q, start, len);
}

// Rows of the current 128-token tile for one thread: row r + R * i as
// channels c0..c0+7.  Tensor-copy path: the stage holds 128 rows of Dp
// values (zeros past D), read with constant offsets.  Fallback: element-wise
// global loads of token t0 + r + R * i (zeros past D).
template <bool kTma, int DP>
struct TileRows {
  const unsigned char* at;      // kTma: stage + (r * DP + c0) * 2
  const uint16_t* row0;         // !kTma: row r of the tile, channel 0
  int64_t tok_stride;           // !kTma
  int c0, D;                    // !kTma
  template <int R>
  __device__ __forceinline__ uint4 get(int i) const {
    if constexpr (kTma) {
      return *reinterpret_cast<const uint4*>(at + i * (R * DP * 2));
    } else {
      if (c0 >= D) return make_uint4(0u, 0u, 0u, 0u);
      const uint16_t* row = row0 + static_cast<int64_t>(i) * R * tok_stride;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = (c0 + 2 * j < D) ? row[c0 + 2 * j] : 0u;
        const uint32_t hi = (c0 + 2 * j + 1 < D) ? row[c0 + 2 * j + 1] : 0u;
        w[j] = lo | (hi << 16);
      }
      return make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
};

// ------------------------------------------------------------- stats K
template <bool kBf16, int DP, class Rows>
__device__ __forceinline__ void stats_k(int nvalid, const Rows& rows, unsigned char* scratch) {
  constexpr int G = DP / 8, R = kConsumers / G, P = kBlockN / R;   // P 8 or 4 rows
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const bool full = nvalid == kBlockN;
  // fp16 keys: a thread holds at most 8 rows of a channel, each split exactly
  // into hi = rint(16 k) and lo = k - hi / 16 (a multiple of 2^-24, |lo| <=
  // 1/32); up to 16 of either sum exactly in fp32 (|sum hi| < 2^24, |sum lo|
  // * 2^24 <= 2^23).  The FP64 pipe (slow on GB300) stays out of the loop.
  static_assert(!kBf16, "bf16 keys take stats_k_bf16");
  long long part[8];
  {
    float2 hs[4], ls[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hs[j] = make_float2(0.0f, 0.0f);
      ls[j] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < P; ++i) {
      if (full || r + R * i < nvalid) {
        const uint4 u = rows.template get<R>(i);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 x = cvt2<false>(word(u, j));
          const float2 tr = __ffma2_rn(x, make_float2(16.0f, 16.0f),
                                       make_float2(kRintMagic, kRintMagic));
          const float2 hi = __fadd2_rn(tr, make_float2(-kRintMagic, -kRintMagic));
          const float2 lo = __ffma2_rn(hi, make_float2(-0.0625f, -0.0625f), x);
          hs[j] = __fadd2_rn(hs[j], hi);
          ls[j] = __fadd2_rn(ls[j], lo);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      part[2 * j] = static_cast<long long>(__float2int_rn(hs[j].x)) * 1048576ll +
                    __float2int_rn(ls[j].x * 16777216.0f);
      part[2 * j + 1] = static_cast<long long>(__float2int_rn(hs[j].y)) * 1048576ll +
                        __float2int_rn(ls[j].y * 16777216.0f);
    }
  }
  // lanes holding the same channels (warp shuffles), then one row per warp
  // in shared memory (the stage, once every row has been read); the helper
  // warp adds the eight rows and the result to the unit's sums
#pragma unroll
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) part[j] += __shfl_xor_sync(0xFFFFFFFFu, part[j], o);
  }
  long long (*tab)[DP] = reinterpret_cast<long long (*)[DP]>(scratch);
  csync();                                     // every row read: the stage is free
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane < G) {
#pragma unroll
    for (int j = 0; j < 8; ++j) tab[wid][c0 + j] = part[j];
  }
}

// bf16 keys.  A bf16 value is (128 + m) 2^(E - 134) with E its exponent
// field (m < 128), so when the nonzero values of a thread's rows of a
// channel lie within 13 binades (E_max - E_min <= 13) and E_max <= 250,
// every partial sum is a multiple of 2^(E_min - 134) below 2^(E_min - 110)
// in magnitude: the fp32 sum of at most 8 of them is exact.  Otherwise
// (rare: a value near zero next to large ones, subnormals, huge values) the
// thread sums that channel in fp64 (exact for 8 values), adds it to the
// unit's sum itself and fences the reduction.  The exact fp32 partials go
// to the stage, one row per thread of a channel group; then one thread per
// channel puts them on the integer grid 2^(g - 150), g = (largest exponent
// field) - 34, where each is below 2^58 and their sum below 2^63, and adds
// them exactly (a partial further below, subnormal or not finite goes to
// the unit's sum in fp64 by itself, fenced).  The helper warp turns the
// integer sums into fp64 reductions (flush_stats).
template <int DP, class Rows>
__device__ __forceinline__ void stats_k_bf16(const ProParams& p, int unit, int nvalid,
                                             const Rows& rows, unsigned char* scratch) {
  constexpr int G = DP / 8, R = kConsumers / G, P = kBlockN / R;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const bool full = nvalid == kBlockN;
  float2 fs[4];
  uint32_t emax[4], emin[4];       // packed exponent fields (max, min over nonzero)
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    fs[j] = make_float2(0.0f, 0.0f);
    emax[j] = 0u;
    emin[j] = 0x00FF00FFu;
  }
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if (full || r + R * i < nvalid) {
      const uint4 u = rows.template get<R>(i);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = word(u, j);
        fs[j] = __fadd2_rn(fs[j], cvt2<true>(w));
        const uint32_t e2 = (w >> 7) & 0x00FF00FFu;
        const uint32_t zero = __vcmpeq2(w & 0x7FFF7FFFu, 0u);   // 0xFFFF in zero halves
        emax[j] = __vmaxu2(emax[j], e2);
        emin[j] = __vminu2(emin[j], e2 | (zero & 0x00FF00FFu));
      }
    }
  }
  float part[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t hi = h ? (emax[j] >> 16) : (emax[j] & 0xFFFFu);
      const uint32_t lo = h ? (emin[j] >> 16) : (emin[j] & 0xFFFFu);
      float v = h ? fs[j].y : fs[j].x;
      if (hi > 250u || (lo <= hi && hi - lo > 13u)) {
        double d = 0.0;
        for (int i = 0; i < P; ++i) {
          if (full || r + R * i < nvalid) {
            const float2 x = cvt2<true>(word(rows.template get<R>(i), j));
            d += static_cast<double>(h ? x.y : x.x);
          }
        }
        atomicAdd(static_cast<double*>(p.ksum) + static_cast<int64_t>(unit) * DP + c0 + 2 * j + h,
                  d);
        __threadfence();
        v = 0.0f;
      }
      part[2 * j + h] = v;
    }
  }
  float (*tab)[DP] = reinterpret_cast<float (*)[DP]>(scratch);
  csync();                                     // every row read: the stage is free
  float4* dst = reinterpret_cast<float4*>(&tab[r][c0]);
  dst[0] = make_float4(part[0], part[1], part[2], part[3]);
  dst[1] = make_float4(part[4], part[5], part[6], part[7]);
  csync();                                     // the table is complete
  if (threadIdx.x < DP) {
    const int c = threadIdx.x;
    int emax = 0;
#pragma unroll 8
    for (int w = 0; w < R; ++w)
      emax = max(emax, static_cast<int>((__float_as_uint(tab[w][c]) >> 23) & 0xFFu));
    const int g = emax - 34;
    long long acc = 0;
    bool fenced = false;
#pragma unroll 8
    for (int w = 0; w < R; ++w) {
      const uint32_t b = __float_as_uint(tab[w][c]);
      const int e = static_cast<int>((b >> 23) & 0xFFu);
      if ((b & 0x7FFFFFFFu) == 0u) continue;
      if (e == 0 || e == 255 || e < g) {
        atomicAdd(static_cast<double*>(p.ksum) + static_cast<int64_t>(unit) * DP + c,
                  static_cast<double>(__uint_as_float(b)));
        fenced = true;
        continue;
      }
      const long long v = static_cast<long long>((b & 0x7FFFFFu) | 0x800000u) << (e - g);
      acc += (b >> 31) ? -v : v;
    }
    if (fenced) __threadfence();
    long long* accs = reinterpret_cast<long long*>(scratch + R * DP * 4);
    int* gs = reinterpret_cast<int*>(scratch + R * DP * 4 + DP * 8);
    accs[c] = acc;
    gs[c] = g;
  }
}

// ------------------------------------------------------------- stats V
// Per-channel max |v| of the tile, one row of packed pairs per warp in the
// stage; the helper warp takes the maximum over the rows.
template <bool kBf16, int DP, class Rows>
__device__ __forceinline__ void stats_v(int nvalid, const Rows& rows, unsigned char* scratch) {
  constexpr int G = DP / 8, R = kConsumers / G, P = kBlockN / R;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const bool full = nvalid == kBlockN;
  uint32_t vm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if (full || r + R * i < nvalid) {
      const uint4 u = rows.template get<R>(i);
#pragma unroll
      for (int j = 0; j < 4; ++j) vm[j] = __vmaxu2(vm[j], word(u, j) & 0x7FFF7FFFu);
    }
  }
#pragma unroll
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) vm[j] = __vmaxu2(vm[j], __shfl_xor_sync(0xFFFFFFFFu, vm[j], o));
  }
  uint32_t (*tab)[DP / 2] = reinterpret_cast<uint32_t (*)[DP / 2]>(scratch);
  csync();                                     // every row read: the stage is free
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane < G) {
#pragma unroll
    for (int j = 0; j < 4; ++j) tab[wid][c0 / 2 + j] = vm[j];
  }
}

// ------------------------------------------------------------------- Q
// out: q16 row of this thread's first row (r), channel c0.
template <bool kBf16, int DP, class Rows>
__device__ __forceinline__ void q_tile(const ProParams& p, int nvalid, const Rows& rows,
                                       uint16_t* out, float* sq) {
  constexpr int G = DP / 8, R = kConsumers / G, P = kBlockM / R;   // P 8 or 4
  const int lane = threadIdx.x & 31;
  const int lc = threadIdx.x % G, r = threadIdx.x / G;
  const bool full = nvalid == kBlockM;
  uint4 raw[P];
#pragma unroll
  for (int i = 0; i < P; ++i)
    raw[i] = (full || r + R * i < nvalid) ? rows.template get<R>(i) : make_uint4(0u, 0u, 0u, 0u);
  uint32_t am[P];
#pragma unroll
  for (int i = 0; i < P; ++i) am[i] = max_mag8(raw[i]);
  // lane l now holds the max of row (l % G) / 2; even lanes form the
  // multiplier 127 / amax, odd lanes the scale amax / 127 (one division each)
  const float amax = mag_f32<kBf16>(row_max_transposed<P>(am, lane));
  const bool odd = (lc & 1) != 0;
  const float quo = __fdiv_rn(odd ? amax : 127.0f, odd ? 127.0f : amax);
  const float mine = amax > 0.0f ? quo : 0.0f;
  if (odd) sq[r + R * (lc >> 1)] = mine;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const float inv = __shfl_sync(0xFFFFFFFFu, mine, (lane & ~(G - 1)) | (2 * i));
    uint4 o;
    o.x = code2(cvt2<kBf16>(raw[i].x), inv, p.one);
    o.y = code2(cvt2<kBf16>(raw[i].y), inv, p.one);
    o.z = code2(cvt2<kBf16>(raw[i].z), inv, p.one);
    o.w = code2(cvt2<kBf16>(raw[i].w), inv, p.one);
    *reinterpret_cast<uint4*>(out + i * (R * DP)) = o;
  }
}

// ------------------------------------------------------------------- K
// out: k16 row of this thread's first row (r), channel c0; mean: the unit's
// K mean (shared memory).
template <bool kBf16, int DP, class Rows>
__device__ __forceinline__ void k_tile(const ProParams& p, int nvalid, const Rows& rows,
                                       const float* mean, uint16_t* out, float* sk,
                                       float* red) {
  constexpr int G = DP / 8, R = kConsumers / G, P = kBlockN / R;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const bool full = nvalid == kBlockN;
  float2 nmean[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) nmean[j] = make_float2(-mean[c0 + 2 * j], -mean[c0 + 2 * j + 1]);
  // smoothing k - mean (fp32) is recomputed in the second pass from the
  // tile; rows past the sequence end count as zero
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    if (full || r + R * i < nvalid) {
      const uint4 u = rows.template get<R>(i);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 kh = __fadd2_rn(cvt2<kBf16>(word(u, j)), nmean[j]);
        am = fmaxf(am, fmaxf(fabsf(kh.x), fabsf(kh.y)));
      }
    }
  }
  am = warp_max(am);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
  csync();
  am = red[0];
#pragma unroll
  for (int w = 1; w < kConsumers / 32; ++w) am = fmaxf(am, red[w]);
  const float kinv = am > 0.0f ? __fdiv_rn(127.0f, am) : 0.0f;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (full || r + R * i < nvalid) {
      const uint4 u = rows.template get<R>(i);
      o.x = code2(__fadd2_rn(cvt2<kBf16>(u.x), nmean[0]), kinv, p.one);
      o.y = code2(__fadd2_rn(cvt2<kBf16>(u.y), nmean[1]), kinv, p.one);
      o.z = code2(__fadd2_rn(cvt2<kBf16>(u.z), nmean[2]), kinv, p.one);
      o.w = code2(__fadd2_rn(cvt2<kBf16>(u.w), nmean[3]), kinv, p.one);
    }
    *reinterpret_cast<uint4*>(out + i * (R * DP)) = o;
  }
  if (threadIdx.x == 0) *sk = __fdiv_rn(am, 127.0f);
}

// ------------------------------------------------------------------- V
// A thread quantises 8 channels of 4 consecutive tokens and packs, per
// channel, the 4 token bytes into one word; word (c, w) of the transposed
// tile sits at c * 32 + (w ^ 4 * (c / 8 % 8)), which spreads the writes over
// banks and keeps every group of four words (16 bytes of a row) contiguous.
// The transposed tile overwrites the stage once every row has been read.
// out: v8 at (channel 0 of the unit, first token of the tile).
template <bool kTma, bool kBf16, int DP>
__device__ __forceinline__ void v_tile(const ProParams& p, int nvalid, const TileRows<kTma, DP>& rows,
                                       const float* vinv_s, uint8_t* out, uint32_t* vt) {
  constexpr int G = DP / 8, RG = kConsumers / G, NTW = (kBlockN / 4) / RG;   // NTW 2 or 1
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const bool full = nvalid == kBlockN;
  float vinv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) vinv[j] = vinv_s[c0 + j];
  // thread (lc, r) reads tokens 4 (r + a RG) + e: rows 4r + e + 4 RG a
  TileRows<kTma, DP> rv = rows;
  if constexpr (kTma) rv.at = rows.at + 3 * r * DP * 2;          // row r -> row 4r
  else rv.row0 = rows.row0 + static_cast<int64_t>(3 * r) * rows.tok_stride;
  uint4 raw[NTW][4];
#pragma unroll
  for (int a = 0; a < NTW; ++a) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 4 * (r + a * RG) + e;
      raw[a][e] = (full || t < nvalid) ? rv.template get<1>(e + 4 * RG * a)
                                       : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  csync();                                      // every row read: the stage is free
  const int swz = ((c0 >> 3) & 7) << 2;         // the same for the 8 channels of c0
#pragma unroll
  for (int a = 0; a < NTW; ++a) {
    uint32_t* w0 = vt + c0 * 32 + ((r + a * RG) ^ swz);
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
      w0[(2 * j) * 32] = __byte_perm(pack_e4m3x2(a01.x, a01.y), pack_e4m3x2(a23.x, a23.y), 0x5410);
      w0[(2 * j + 1) * 32] = __byte_perm(pack_e4m3x2(b01.x, b01.y), pack_e4m3x2(b23.x, b23.y), 0x5410);
    }
  }
  csync();
  constexpr int kQuads = DP * (kBlockN / 16);   // 16-byte pieces
  const int64_t vcols = p.g.v_cols;
#pragma unroll
  for (int qi = threadIdx.x; qi < kQuads; qi += kConsumers) {
    const int c = qi / (kBlockN / 16), tw = 4 * (qi % (kBlockN / 16));
    const uint4 val = *reinterpret_cast<const uint4*>(&vt[c * 32 + (tw ^ (((c >> 3) & 7) << 2))]);
    *reinterpret_cast<uint4*>(out + c * vcols + 4 * tw) = val;
  }
}

// V for the FP16-PV variant: the same transposition without scaling, to
// fp16 (bf16 inputs rounded to nearest even).  A channel row of the tile is
// 64 words of two tokens; word w of channel c sits at c * 64 + (w ^ 8 * (c /
// 8 % 8)), keeping every 16-byte group whole.
// out: v16 at (channel 0 of the unit, first token of the tile).
template <bool kTma, bool kBf16, int DP>
__device__ __forceinline__ void v_tile16(const ProParams& p, int nvalid,
                                         const TileRows<kTma, DP>& rows, uint16_t* out,
                                         uint32_t* vt) {
  constexpr int G = DP / 8, RG = kConsumers / G, NTW = (kBlockN / 4) / RG;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  const bool full = nvalid == kBlockN;
  TileRows<kTma, DP> rv = rows;
  if constexpr (kTma) rv.at = rows.at + 3 * r * DP * 2;          // row r -> row 4r
  else rv.row0 = rows.row0 + static_cast<int64_t>(3 * r) * rows.tok_stride;
  uint4 raw[NTW][4];
#pragma unroll
  for (int a = 0; a < NTW; ++a) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 4 * (r + a * RG) + e;
      raw[a][e] = (full || t < nvalid) ? rv.template get<1>(e + 4 * RG * a)
                                       : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  csync();                                      // every row read: the stage is free
  const int swz = ((c0 >> 3) & 7) << 3;         // the same for the 8 channels of c0
#pragma unroll
  for (int a = 0; a < NTW; ++a) {
    const int q = r + a * RG;                   // tokens 4q .. 4q + 3
#pragma unroll
    for (int j = 0; j < 4; ++j) {               // channels c0 + 2j, c0 + 2j + 1
      uint32_t h[4];                            // fp16 pair (channel 2j low, 2j + 1 high)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (kBf16) {
          const float2 x = cvt2<true>(word(raw[a][e], j));
          const __half2 hv = __floats2half2_rn(x.x, x.y);
          memcpy(&h[e], &hv, 4);
        } else {
          h[e] = word(raw[a][e], j);
        }
      }
      uint2* lo = reinterpret_cast<uint2*>(vt + (c0 + 2 * j) * 64 + ((2 * q) ^ swz));
      uint2* hi = reinterpret_cast<uint2*>(vt + (c0 + 2 * j + 1) * 64 + ((2 * q) ^ swz));
      *lo = make_uint2(__byte_perm(h[0], h[1], 0x5410), __byte_perm(h[2], h[3], 0x5410));
      *hi = make_uint2(__byte_perm(h[0], h[1], 0x7632), __byte_perm(h[2], h[3], 0x7632));
    }
  }
  csync();
  constexpr int kChunks = DP * (kBlockN * 2 / 16);   // 16-byte pieces
  const int64_t vcols = p.g.v_cols;
#pragma unroll
  for (int ci = threadIdx.x; ci < kChunks; ci += kConsumers) {
    const int c = ci / (kBlockN * 2 / 16), w4 = 4 * (ci % (kBlockN * 2 / 16));
    const uint4 val = *reinterpret_cast<const uint4*>(&vt[c * 64 + (w4 ^ (((c >> 3) & 7) << 3))]);
    *reinterpret_cast<uint4*>(out + c * vcols + 2 * w4) = val;
  }
}

// ---------------------------------------------------------- statistics
// A unit's K mean of one channel from its exact sum (fp16: int64 fixed point
// at 2^-24; bf16: fp64): the fp64 quotient by the key count, rounded to fp32.
template <bool kBf16>
__device__ __forceinline__ float k_mean_of(long long raw, int64_t len) {
  if (len <= 0) return 0.0f;
  double S;
  if constexpr (kBf16) S = __longlong_as_double(raw);
  else S = __ll2double_rn(raw) * 5.9604644775390625e-08;   // 2^-24, exact
  return __double2float_rn(__ddiv_rn(S, static_cast<double>(len)));
}

// Per-channel V scale amax / 448 and multiplier 448 / amax (0 for a zero
// channel) from the unit's maximum (float bits).
__device__ __forceinline__ float v_scale_of(uint32_t m) {
  return __fdiv_rn(__uint_as_float(m), 448.0f);
}
__device__ __forceinline__ float v_mul_of(uint32_t m) {
  const float a = __uint_as_float(m);
  return a > 0.0f ? __fdiv_rn(448.0f, a) : 0.0f;
}

// ------------------------------------------------------------- consumers
template <bool kTma, bool kBf16, int DP, bool kPacked>
__device__ __forceinline__ void consume(const ProParams& p, const Slot& it, int stage,
                                        PSmem& sm) {
  constexpr int G = DP / 8;
  const SegGeo& g = p.g;
  const int32_t* cuk = kPacked ? sm.cu_k : g.cu_k;   // packed: the shared copies
  const int32_t* cuq = kPacked ? sm.cu_q : g.cu_q;
  const int64_t s = it.unit / g.Hkv, h = it.unit % g.Hkv;
  const int lc = threadIdx.x % G, r = threadIdx.x / G, c0 = lc * 8;
  TileRows<kTma, DP> rows;
  rows.at = sm.tile[stage] + (r * DP + c0) * 2;
  rows.c0 = c0;
  rows.D = static_cast<int>(g.D);
  int64_t start = 0, len = 0;
  if (it.kind == kQ) {
    const int64_t hq = h * (g.Hq / g.Hkv) + it.sub / p.plan.nqt;
    const int64_t t0 = static_cast<int64_t>(it.sub % p.plan.nqt) * kBlockM;
    query_range(g, cuq, s, &start, &len);
    if constexpr (!kTma) {
      rows.row0 = p.q + (g.varlen ? start * g.q_tok_stride : s * g.q_seg_stride) +
                  hq * g.q_head_stride + (t0 + r) * g.q_tok_stride;
      rows.tok_stride = g.q_tok_stride;
    }
    const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hq, g.q_head_rows) +
                         hq * g.q_head_rows + t0;
    q_tile<kBf16, DP>(p, it.nvalid, rows, p.q16 + (row0 + r) * DP + c0, p.s_q + row0);
    return;
  }
  const bool seg_ok = key_range(g, cuk, s, &start, &len);
  const int64_t t0 = static_cast<int64_t>(it.sub) * kBlockN;
  if constexpr (!kTma) {
    const uint16_t* src = (it.kind == kStatsK || it.kind == kK) ? p.k : p.v;
    rows.row0 = src + (g.varlen ? start * g.k_tok_stride : s * g.k_seg_stride) +
                h * g.k_head_stride + (t0 + r) * g.k_tok_stride;
    rows.tok_stride = g.k_tok_stride;
  }
  if (it.kind == kStatsK) {
    if constexpr (kBf16) stats_k_bf16<DP>(p, it.unit, it.nvalid, rows, sm.tile[stage]);
    else stats_k<kBf16, DP>(it.nvalid, rows, sm.tile[stage]);
  } else if (it.kind == kStatsV) {
    stats_v<kBf16, DP>(it.nvalid, rows, sm.tile[stage]);
  } else if (it.kind == kK) {
    // the unit's K mean from its sums (copied next to the tile); the item of
    // the first block also stores it
    if (threadIdx.x < DP) {
      const int c = threadIdx.x;
      const float m = k_mean_of<kBf16>(reinterpret_cast<const long long*>(sm.aux[stage])[c], len);
      sm.coef[c] = m;
      if (it.sub == 0) p.k_mean[static_cast<int64_t>(it.unit) * DP + c] = m;
    }
    csync();
    const int64_t row0 = ws_seg_base(g.varlen, s, start, g.Hkv, g.k_head_rows) +
                         h * g.k_head_rows + t0;
    k_tile<kBf16, DP>(p, it.nvalid, rows, sm.coef, p.k16 + (row0 + r) * DP + c0,
                      p.s_k + row0 / kBlockN, sm.red);
  } else if (it.kind == kV) {
    // the unit's V multipliers from its maxima; the first block's item also
    // stores the scales
    if (threadIdx.x < DP) {
      const int c = threadIdx.x;
      const uint32_t mx = reinterpret_cast<const uint32_t*>(sm.aux[stage])[c];
      const float mul = v_mul_of(mx);
      sm.coef[c] = mul;
      if (it.sub == 0) {
        p.s_v[static_cast<int64_t>(it.unit) * DP + c] = v_scale_of(mx);
        p.v_inv[static_cast<int64_t>(it.unit) * DP + c] = mul;
      }
    }
    csync();
    const int64_t vrow0 = (g.varlen ? 0 : s * g.Hkv * DP) + h * DP;
    const int64_t vcol0 = (g.varlen ? ws_seg_base(1, s, start, 0, 0) : 0) + t0;
    if (p.v16)
      v_tile16<kTma, kBf16, DP>(p, it.nvalid, rows,
                                reinterpret_cast<uint16_t*>(p.v8) + vrow0 * g.v_cols + vcol0,
                                reinterpret_cast<uint32_t*>(sm.tile[stage]));
    else
      v_tile<kTma, kBf16, DP>(p, it.nvalid, rows, sm.coef, p.v8 + vrow0 * g.v_cols + vcol0,
                              reinterpret_cast<uint32_t*>(sm.tile[stage]));
  } else {
    // final item (statistics only): the unit's K mean and V scales, read from
    // L2 (the group's barrier, acquired by the producer, orders them)
    if (threadIdx.x < DP) {
      const int64_t i = static_cast<int64_t>(it.unit) * DP + threadIdx.x;
      p.k_mean[i] = k_mean_of<kBf16>(__ldcg(static_cast<const long long*>(p.ksum) + i),
                                     seg_ok ? len : 0);
      const uint32_t mx = __ldcg(p.vmax + i);
      p.s_v[i] = v_scale_of(mx);
      p.v_inv[i] = v_mul_of(mx);
    }
  }
}

// Markers the consumers hand to the helper: the end, and the end of group
// g's A list (kMarkGroup - g).
constexpr int kMarkEnd = -1;
constexpr int kMarkGroup = -2;

// Group g's barrier (helper lane 0): this CTA's consumers are done with
// every A item of the group it took.  Their sums and maxima (relaxed
// reductions, ordered before the hand-over by the consumers' barrier and
// the queue's mbarrier) are released with the count.
__device__ __forceinline__ void group_arrive(const ProParams& p, int g) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(p.gbar + g) : "memory");
}

// A finished stats tile's per-warp rows (in its stage) -> the unit's K sums
// or V maxima (relaxed reductions, one per channel and lane).
template <bool kBf16, int DP>
__device__ __forceinline__ void flush_stats(const ProParams& p, int unit, bool is_v,
                                            const unsigned char* scratch) {
  const int lane = threadIdx.x & 31;
  const int64_t base = static_cast<int64_t>(unit) * DP;
#pragma unroll
  for (int i = 0; i < DP / 32; ++i) {
    const int c = lane + 32 * i;
    if (c >= p.g.D) break;
    if (is_v) {
      const uint32_t (*tab)[DP / 2] = reinterpret_cast<const uint32_t (*)[DP / 2]>(scratch);
      uint32_t m = 0u;
#pragma unroll
      for (int w = 0; w < kConsumers / 32; ++w) m = __vmaxu2(m, tab[w][c >> 1]);
      m = (c & 1) ? (m >> 16) : (m & 0xFFFFu);
      atomicMax(p.vmax + base + c, __float_as_uint(mag_f32<kBf16>(m)));
    } else if constexpr (kBf16) {
      // the channel's exact integer sum on the grid 2^(g - 150) (stats_k_bf16)
      constexpr int R = kConsumers / (DP / 8);
      const long long acc = reinterpret_cast<const long long*>(scratch + R * DP * 4)[c];
      const int g = reinterpret_cast<const int*>(scratch + R * DP * 4 + DP * 8)[c];
      if (acc != 0) {
        // exact when |acc| < 2^53; 2^(g - 150) is a normal double (g >= -33)
        const double scale = __longlong_as_double(static_cast<long long>(g - 150 + 1023) << 52);
        atomicAdd(static_cast<double*>(p.ksum) + base + c, __ll2double_rn(acc) * scale);
      }
    } else {
      const long long (*tab)[DP] = reinterpret_cast<const long long (*)[DP]>(scratch);
      {
        long long si = 0;
#pragma unroll
        for (int w = 0; w < kConsumers / 32; ++w) si += tab[w][c];
        atomicAdd(static_cast<unsigned long long*>(p.ksum) + base + c,
                  static_cast<unsigned long long>(si));
      }
    }
  }
}

// The helper warp takes what the consumers hand over, in order.  A finished
// stats tile: it adds the tile's rows to the unit's sums and maxima, then
// releases the tile's stage.  A group marker: the CTA is done with the
// group's A list, so every lane fences its own reductions (each lane orders
// what it issued itself) and lane 0 arrives at the group's barrier.  The
// fences wait for outstanding writes, which is why they run here and not on
// a consumer thread.  The helper never waits for other CTAs.
template <bool kBf16, int DP>
__device__ __forceinline__ void helper(const ProParams& p, PSmem& sm) {
  const int lane = threadIdx.x & 31;
  int q = 0;
  uint32_t qph = 0;
  while (true) {
    if (!mbar_sleep_wait(&sm.qfull[q], qph, &sm.abort, p.status, p.timeout_ns)) return;
    const int unit = sm.queue[q];
    const int info = sm.qinfo[q];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.qempty[q]);
    if (++q == kQueue) {
      q = 0;
      qph ^= 1u;
    }
    if (unit == kMarkEnd) return;
    if (unit <= kMarkGroup) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      __syncwarp();
      if (lane == 0) group_arrive(p, kMarkGroup - unit);
      continue;
    }
    const int stage = info >> 1;
    flush_stats<kBf16, DP>(p, unit, (info & 1) != 0, sm.tile[stage]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);     // the stage may be refilled
  }
}

// Consumer thread 0 hands a finished stats tile (unit >= 0) or a marker to
// the helper warp.
__device__ __forceinline__ bool hand_over(const ProParams& p, PSmem& sm, int unit, int info,
                                          int* q, uint32_t* ph) {
  if (!mbar_sleep_wait(&sm.qempty[*q], *ph ^ 1u, &sm.abort, p.status, p.timeout_ns))
    return false;
  sm.queue[*q] = unit;
  sm.qinfo[*q] = info;
  mbar_arrive(&sm.qfull[*q]);
  if (++*q == kQueue) {
    *q = 0;
    *ph ^= 1u;
  }
  return true;
}

// Packed sequences: each CTA's helper warp checks its share of the offsets
// (the lists over virtual tiles cover every tile only for consistent ones)
// and reports an inconsistent entry in the status word.
__device__ __forceinline__ void check_offsets(const ProParams& p) {
  const SegGeo& g = p.g;
  const int64_t per = (g.nseg + gridDim.x - 1) / gridDim.x;
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t s1 = s0 + per < g.nseg ? s0 + per : g.nseg;
  bool bad = false;
  for (int64_t s = s0 + (threadIdx.x & 31); s < s1; s += 32) {
    int64_t start, len;
    bad |= !seg_range(g.cu_k, s, g.total_k, g.max_k, &start, &len) ||
           !seg_range(g.cu_q, s, g.total_q, g.max_q, &start, &len);
  }
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0)
    atomicOr(p.status, kStatusBadSeqlens);
}

// -------------------------------------------------------------- producer
// kPacked: packed sequences, whose lists run over virtual tiles (vdecode;
// packed_lists chooses).  It is a template parameter so that the other
// instances keep the plain per-unit lists with no trace of it: with the
// packed code in a shared instance the dense prologue ran 8 % slower
// without executing any of it.
template <bool kTma, bool kBf16, int DP, bool kPacked>
__device__ __forceinline__ void produce(const ProParams& p, PSmem& sm) {
  const SegGeo& g = p.g;
  const Plan& P = p.plan;
  const int lane = threadIdx.x & 31;
  const uint64_t keep = policy_evict_last(), once = policy_evict_first();
  int stage = 0;
  uint32_t upar = 0;       // bit s: parity of the uses of stage s so far
  uint32_t tma = 0;        // bit s: stage s was last filled by a tensor copy
  bool ok = true;
  int ga = P.n_stats > 0 ? 0 : P.groups;   // group of the A list being taken
  int gb = 0;              // group of the B list being taken
  bool b_open = P.open != 0;   // group gb's statistics are final
  uint32_t poll = 0;       // group gb's barrier count, read on the previous turn
  bool polled = false;
  int a_idx = 0, b_idx = 0, q_idx = 0;  // claims taken ahead (lane 0), valid when *_pend
  bool a_pend = false, b_pend = false, q_pend = false;
  bool q_left = P.n_q > 0;   // the Q list may still have items
  const uint32_t grid = gridDim.x;
  uint64_t idle0 = 0;
  // packed lists: the first item and size of groups ga and gb (over
  // virtual tiles), the Q list's size, and the sequence of the last A, B and
  // Q item decoded (B holds one final item per unit without K/V items)
  const bool pk_b = kPacked && P.n_kv > 0;
  const int nseg = static_cast<int>(g.nseg), hkv = static_cast<int>(g.Hkv);
  const int32_t* cuk = kPacked ? sm.cu_k : g.cu_k;   // packed: the shared copies
  const int32_t* cuq = kPacked ? sm.cu_q : g.cu_q;
  const int gq = static_cast<int>(g.Hq / g.Hkv);
  int a_first = 0, a_size = 0, b_first = 0, b_size = 0, q_size = 0;
  SeqCache ca, cb, cq;
  auto kv_first = [&](int gi) {
    return vstart(cuk, nseg, g.total_k, hkv, 2, min(gi * P.group, P.units));
  };
  auto set_a = [&]() {
    if constexpr (kPacked) {
      if (ga < P.groups) {
        a_first = kv_first(ga);
        a_size = kv_first(ga + 1) - a_first;
      }
    }
  };
  auto set_b = [&]() {
    if constexpr (kPacked) {
      if (gb < P.groups) {
        b_first = pk_b ? kv_first(gb) : 0;
        b_size = pk_b ? kv_first(gb + 1) - b_first : group_units(P, gb) * P.n_b;
      }
    }
  };
  if constexpr (kPacked) {
    set_a();
    set_b();
    q_size = P.n_q > 0 ? vstart(cuq, nseg, g.total_q, hkv, gq, P.units) : 0;
  }
  // a packed item outside its sequence's tiles (inconsistent offsets)
  auto bad_offsets = [&]() {
    if (lane == 0) atomicOr(p.status, kStatusBadSeqlens);
  };
  while (ok) {
    // ---- choose the next item: a B item if its group is final, else an A
    // item (at most `lead` groups ahead of the B list), else a Q item, else
    // poll and wait
    Slot it{-1, 0, 0, 0};
    bool marker = false;
    while (gb < P.groups) {
      if (!b_open) {
        if (polled) {
          polled = false;
          if (__shfl_sync(0xFFFFFFFFu, poll, 0) >= grid) {
            b_open = true;
            if (lane == 0) {
              // acquire the group's statistics; the copy engine (async proxy)
              // reads them below
              asm volatile("fence.acq_rel.gpu;" ::: "memory");
              asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            __syncwarp();
          }
        }
        if (!b_open) break;
      }
      if (!b_pend && lane == 0) b_idx = static_cast<int>(atomicAdd(p.cnt_b + gb, 1u));
      const int idx = __shfl_sync(0xFFFFFFFFu, b_idx, 0);
      b_pend = false;
      if (idx < (kPacked ? b_size : group_units(P, gb) * P.n_b)) {
        if (pk_b) {
          int u, t, j;
          if (vdecode(cuk, nseg, g.total_k, hkv, 2, b_first + idx, cb, &u, &t, &j)) {
            it.kind = j ? kV : kK;
            it.unit = u;
            it.sub = t;
          } else {
            bad_offsets();
          }
        } else {
          decode_b(P, gb, idx, &it.kind, &it.unit, &it.sub);
        }
        // claim the group's next B item now; it is used on the next turn
        if (lane == 0) b_idx = static_cast<int>(atomicAdd(p.cnt_b + gb, 1u));
        b_pend = true;
        break;
      }
      ++gb;
      b_open = P.open != 0;
      set_b();
    }
    // the Q list: a lambda, taken before or after the A list
    auto take_q = [&]() {
      if (it.kind < 0 && q_left) {
        if (!q_pend && lane == 0) q_idx = static_cast<int>(atomicAdd(p.cnt_q, 1u));
        const int idx = __shfl_sync(0xFFFFFFFFu, q_idx, 0);
        q_pend = false;
        if (idx < (kPacked ? q_size : P.units * P.n_q)) {
          if constexpr (kPacked) {
            int u, t, j;
            if (!vdecode(cuq, nseg, g.total_q, hkv, gq, idx, cq, &u, &t, &j)) {
              bad_offsets();
            } else if (t < P.nqt) {      // else the sequence's spare virtual tile
              it.kind = kQ;
              it.unit = u;
              it.sub = j * P.nqt + t;
            }
          } else {
            decode_q(P, idx, &it.kind, &it.unit, &it.sub);
          }
          if (lane == 0) q_idx = static_cast<int>(atomicAdd(p.cnt_q, 1u));
          q_pend = true;
        } else {
          q_left = false;
        }
      }
    };
    if (P.q_first) take_q();
    if (it.kind < 0 && ga < P.groups && ga <= gb + P.lead) {
      if (!a_pend && lane == 0) a_idx = static_cast<int>(atomicAdd(p.cnt_a + ga, 1u));
      const int idx = __shfl_sync(0xFFFFFFFFu, a_idx, 0);
      a_pend = false;
      if (idx < (kPacked ? a_size : group_units(P, ga) * P.n_stats)) {
        if constexpr (kPacked) {
          int u, t, j;
          if (vdecode(cuk, nseg, g.total_k, hkv, 2, a_first + idx, ca, &u, &t, &j)) {
            it.kind = j ? kStatsV : kStatsK;
            it.unit = u;
            it.sub = t;
          } else {
            bad_offsets();
          }
        } else {
          decode_a(P, ga, idx, &it.kind, &it.unit, &it.sub);
        }
        // claim the group's next A item now (A items never wait, so holding
        // the claim cannot hold up a barrier)
        if (lane == 0) a_idx = static_cast<int>(atomicAdd(p.cnt_a + ga, 1u));
        a_pend = true;
      } else {
        it.kind = kGroupEnd;                  // this CTA is done with group ga's A list
        it.unit = ga;
        marker = true;
        ++ga;
        set_a();
      }
    }
    if (!P.q_first) take_q();
    if (it.kind < 0) {
      if (ga >= P.groups && gb >= P.groups && !q_left) {
        it.kind = kEnd;
        marker = true;
      } else {
        // nothing to take yet: read group gb's barrier count for the next turn
        if (!polled && gb < P.groups && !b_open) {
          if (lane == 0)
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];"
                         : "=r"(poll) : "l"(p.gbar + gb) : "memory");
          polled = true;
        }
        if (idle0 == 0) idle0 = global_timer_ns();
        else if (global_timer_ns() - idle0 > p.timeout_ns) {
          if (lane == 0) atomicOr(p.status, kStatusTimeout);
          sm.abort = 1;
          ok = false;
          break;
        }
        __nanosleep(64);
        continue;
      }
    }
    idle0 = 0;
    if (!polled && gb < P.groups && !b_open) {
      // keep the barrier read in flight while this item is set up
      if (lane == 0)
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];"
                     : "=r"(poll) : "l"(p.gbar + gb) : "memory");
      polled = true;
    }

    // every decoded item must name a unit of the plan: anything else is an
    // internal error, reported and skipped rather than followed
    if (!marker && (it.unit < 0 || it.unit >= P.units)) {
      if (lane == 0) atomicOr(p.status, kStatusBadItem);
      continue;
    }
    // a final item loads nothing: it is passed on like a marker
    if (it.kind == kFinal) marker = true;
    int64_t s = 0, h = 0, start = 0, len = 0, t0 = 0;
    if (!marker) {
      s = it.unit / g.Hkv;
      h = it.unit % g.Hkv;
      bool seg_ok;
      if (it.kind == kQ) {
        seg_ok = query_range(g, cuq, s, &start, &len);
        h = h * (g.Hq / g.Hkv) + it.sub / P.nqt;        // query head
        t0 = static_cast<int64_t>(it.sub % P.nqt) * kBlockM;
      } else {
        seg_ok = key_range(g, cuk, s, &start, &len);
        t0 = static_cast<int64_t>(it.sub) * kBlockN;
      }
      if (!seg_ok) {
        if (lane == 0 && it.sub == 0) atomicOr(p.status, kStatusBadSeqlens);
        len = 0;
      }
      if (t0 >= len) continue;               // nothing to load or quantise
      it.nvalid = static_cast<int32_t>(len - t0 < kBlockN ? len - t0 : kBlockN);
    }
    // wait until the consumers have released this stage's previous item
    if (!mbar_sleep_wait(&sm.empty[stage], ((upar >> stage) & 1u) ^ 1u, &sm.abort, p.status,
                         p.timeout_ns)) {
      ok = false;
      break;
    }
    if (lane == 0) sm.slot[stage] = it;
    __syncwarp();
    if (marker) {
      if (lane == 0) mbar_arrive(&sm.full[stage]);
      tma &= ~(1u << stage);
      upar ^= 1u << stage;
      stage = stage + 1 == kStages ? 0 : stage + 1;
      if (it.kind == kEnd) break;
      continue;
    }
    if (lane == 0) {
      const bool kv = it.kind == kK || it.kind == kV;
      const uint32_t aux_bytes = it.kind == kK ? DP * 8 : it.kind == kV ? DP * 4 : 0;
      if constexpr (kTma) {
        const CUtensorMap* map = it.kind == kQ ? &p.mq
                               : (it.kind == kStatsK || it.kind == kK) ? &p.mk : &p.mv;
        const int hnd = it.kind == kQ ? p.q_hnd : p.k_hnd;
        const int64_t H = it.kind == kQ ? g.Hq : g.Hkv;
        const int64_t L = it.kind == kQ ? g.Lq : g.Lk;
        int32_t y, zc;
        if (hnd) {
          y = static_cast<int32_t>(t0);
          zc = static_cast<int32_t>(s * H + h);
        } else {
          y = static_cast<int32_t>(h);
          zc = static_cast<int32_t>((g.varlen ? start : s * L) + t0);
        }
        mbar_expect_tx(&sm.full[stage], static_cast<uint32_t>(kBlockN * DP * 2) + aux_bytes);
        if (g.strided)           // views: (channel, token, head, batch) maps
          tma_load_4d_hint(sm.tile[stage], map, 0, static_cast<int32_t>(t0),
                           static_cast<int32_t>(h), static_cast<int32_t>(s), &sm.full[stage],
                           it.kind <= kStatsV ? keep : once);
        else
        tma_load_3d_hint(sm.tile[stage], map, 0, y, zc, &sm.full[stage],
                         it.kind <= kStatsV ? keep : once);
      } else {
        mbar_expect_tx(&sm.full[stage], aux_bytes);
      }
      if (kv) {
        // the unit's K sums or V maxima, complete since its group's barrier
        const void* src =
            it.kind == kK
                ? static_cast<const void*>(static_cast<const long long*>(p.ksum) +
                                           static_cast<int64_t>(it.unit) * DP)
                : static_cast<const void*>(p.vmax + static_cast<int64_t>(it.unit) * DP);
        bulk_load(sm.aux[stage], src, aux_bytes, &sm.full[stage]);
      }
    }
    if constexpr (kTma) tma |= 1u << stage;
    upar ^= 1u << stage;
    stage = stage + 1 == kStages ? 0 : stage + 1;
  }
  if (!ok) {
    // let every copy already issued land before the CTA can exit
    for (int st = 0; st < kStages; ++st)
      if (tma & (1u << st))
        mbar_wait(&sm.full[st], ((upar >> st) & 1u) ^ 1u, nullptr, p.status, p.timeout_ns);
  }
}

// --------------------------------------------------------------- kernel
template <bool kTma, bool kBf16, int DP, bool kPacked>
__global__ void __launch_bounds__(kThreads, 3)
prologue_kernel(const __grid_constant__ ProParams p) {
  extern __shared__ uint8_t smem_raw[];
  PSmem& sm = *reinterpret_cast<PSmem*>(align1024(smem_raw));
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kQueue; ++s) {
      mbar_init(&sm.qfull[s], 1);
      mbar_init(&sm.qempty[s], 1);
    }
    sm.abort = 0;
    mbar_fence_init();
  }
  if constexpr (kPacked) {          // at most kCuSmem sequences (launch_any)
    for (int i = threadIdx.x; i <= p.g.nseg; i += kThreads) {
      sm.cu_k[i] = p.g.cu_k[i];
      sm.cu_q[i] = p.g.cu_q[i];
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp == kProducerWarp) {
    if constexpr (kTma) {
      if ((threadIdx.x & 31) == 0) {
        tma_prefetch_desc(&p.mq);
        tma_prefetch_desc(&p.mk);
        tma_prefetch_desc(&p.mv);
      }
    }
    produce<kTma, kBf16, DP, kPacked>(p, sm);
    return;
  }
  if (warp == kHelperWarp) {
    if constexpr (kPacked) check_offsets(p);
    helper<kBf16, DP>(p, sm);
    return;
  }
  int stage = 0, q = 0;
  uint32_t phase = 0, qph = 0;
  while (true) {
    if (!mbar_sleep_wait(&sm.full[stage], phase, &sm.abort, p.status, p.timeout_ns)) break;
    const Slot it = sm.slot[stage];
    if (it.kind == kEnd) break;
    if (it.kind != kGroupEnd) consume<kTma, kBf16, DP, kPacked>(p, it, stage, sm);
    csync();                                    // every consumer is done with the stage
    if (threadIdx.x == 0) {
      if (it.kind <= kStatsV) {
        // the helper adds the tile's rows to the unit's statistics and then
        // releases the stage
        hand_over(p, sm, it.unit, 2 * stage + (it.kind == kStatsV ? 1 : 0), &q, &qph);
      } else {
        mbar_arrive(&sm.empty[stage]);
        if (it.kind == kGroupEnd) hand_over(p, sm, kMarkGroup - it.unit, 0, &q, &qph);
      }
    }
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  if (threadIdx.x == 0) hand_over(p, sm, kMarkEnd, 0, &q, &qph);   // the helper may stop
}

constexpr size_t kSmemBytes = sizeof(PSmem) + 1024;   // + alignment slack

// Work of a launch (PlanMode): without K/V items the B list holds one final
// item per unit; without statistics (kPlanKV) the B list is open at once.
bool make_plan(const SegGeo& g, int mode, Plan* out) {
  Plan P{};
  const int64_t maxk = g.varlen ? g.max_k : g.Lk;
  const int64_t maxq = g.varlen ? g.max_q : g.Lq;
  const int64_t nkb = (maxk + kBlockN - 1) / kBlockN;
  const int64_t units = g.nseg * g.Hkv;
  const bool stats = mode != kPlanKV;
  const int64_t n_stats = stats ? (nkb > 0 ? 2 * nkb : 1) : 0;
  const int64_t nqt = (maxq + kBlockM - 1) / kBlockM;
  const int64_t n_q = (mode == kPlanAll || mode == kPlanStatsQ) ? (g.Hq / g.Hkv) * nqt : 0;
  const int64_t n_kv = (mode == kPlanAll || mode == kPlanKV) ? 2 * nkb : 0;
  const int64_t per = n_stats + n_q + (n_kv > 0 ? n_kv : 1);
  if (units * per >= (int64_t(1) << 31)) return false;
  if (g.varlen) {
    // packed lists: 2 (K and V) or Hq / Hkv (Q) items per virtual tile and
    // kv head, nseg + total / 128 virtual tiles
    const int64_t vk = g.nseg + g.total_k / kBlockN + 1, vq = g.nseg + g.total_q / kBlockM + 1;
    if (2 * g.Hkv * vk >= (int64_t(1) << 31) || g.Hq * vq >= (int64_t(1) << 31)) return false;
  }
  int64_t group = units, lead = 1;
  if (n_kv > 0 && stats) {
    // a group's K and V are read by its A list and again (from L2) by its B
    // list, which runs up to `lead` groups behind: lead + 1 groups must fit
    const int64_t unit_bytes = 4 * maxk * g.D;
    group = unit_bytes > 0 ? kGroupBytes / unit_bytes : units;
    if (group < 1) group = 1;
    if (group > units) group = units;
    if ((units + group - 1) / group > kMaxGroups) group = (units + kMaxGroups - 1) / kMaxGroups;
    const int64_t gbytes = group * unit_bytes;
    lead = gbytes > 0 ? kL2Hold / gbytes - 1 : 1;
    if (lead < 1) lead = 1;
  }
  const int64_t groups = units > 0 ? (units + group - 1) / group : 0;
  P.units = static_cast<int32_t>(units);
  P.group = static_cast<int32_t>(group);
  P.groups = static_cast<int32_t>(groups);
  P.lead = static_cast<int32_t>(lead < groups ? lead : (groups > 0 ? groups : 1));
  P.n_stats = static_cast<int32_t>(n_stats);
  P.n_q = static_cast<int32_t>(n_q);
  P.n_kv = static_cast<int32_t>(n_kv);
  P.n_b = static_cast<int32_t>(n_kv > 0 ? n_kv : 1);
  P.nqt = static_cast<int32_t>(nqt);
  P.open = stats ? 0 : 1;
  P.q_first = mode == kPlanStatsQ ? 1 : 0;
  *out = P;
  return true;
}

// 3D map of a q/k/v input: (channel, token, head plane) for head-major
// tensors, (channel, head, token) for token-major ones.  Boxes are 128 rows
// of Dp channels; channels past D are zero-filled by the copy.
bool input_map(CUtensorMap* map, const uint16_t* base, int64_t D, int64_t Dp, int64_t H,
               int64_t L, int64_t ntok, bool hnd) {
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  dims[0] = static_cast<uint64_t>(D);
  strides[0] = static_cast<uint64_t>(D) * 2;
  box[0] = static_cast<uint32_t>(Dp);
  if (hnd) {
    dims[1] = static_cast<uint64_t>(L);
    dims[2] = static_cast<uint64_t>(ntok / L * H);
    strides[1] = static_cast<uint64_t>(L * D) * 2;
    box[1] = 128;
    box[2] = 1;
  } else {
    dims[1] = static_cast<uint64_t>(H);
    dims[2] = static_cast<uint64_t>(ntok);
    strides[1] = static_cast<uint64_t>(H * D) * 2;
    box[1] = 1;
    box[2] = 128;
  }
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(base),
                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 4D map of a strided view: (channel, token, head, batch) with the caller's
// strides (elements, each a multiple of 8); boxes are 128 tokens of Dp
// channels, channels past D zero-filled.
bool view_map(CUtensorMap* map, const uint16_t* base, int64_t D, int64_t Dp, int64_t L,
              int64_t H, int64_t B, int64_t tok, int64_t head, int64_t batch) {
  uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(L),
                      static_cast<uint64_t>(H), static_cast<uint64_t>(B)};
  uint64_t strides[3] = {static_cast<uint64_t>(tok) * 2, static_cast<uint64_t>(head) * 2,
                         static_cast<uint64_t>(batch) * 2};
  uint32_t box[4] = {static_cast<uint32_t>(Dp), 128, 1, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<uint16_t*>(base),
                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <bool kTma, bool kBf16, int DP, bool kPacked>
cudaError_t launch_t(ProParams& prm, int mode, cudaStream_t st) {
  // resident CTAs per SM, per device (filled once; every thread computes
  // the same value, so relaxed atomics suffice)
  static std::atomic<int> per_sm[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (per_sm[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(prologue_kernel<kTma, kBf16, DP, kPacked>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prologue_kernel<kTma, kBf16, DP, kPacked>,
                                                      kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    per_sm[dev].store(n > 0 ? n : 1, std::memory_order_relaxed);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (!make_plan(prm.g, mode, &prm.plan)) return cudaErrorInvalidValue;
  if (prm.plan.groups <= 0) return cudaSuccess;
  // every CTA is resident at once (the group barriers count them all): a
  // cooperative launch of exactly the resident CTAs
  const unsigned grid = static_cast<unsigned>(sms * per_sm[dev].load(std::memory_order_relaxed));
  void* args[] = {&prm};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(prologue_kernel<kTma, kBf16, DP, kPacked>),
                                  dim3(grid), dim3(kThreads), args, kSmemBytes, st);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaGetLastError();
}

// Packed sequences take the lists over virtual tiles (vdecode) when at least
// a quarter of the items in lists sized by the longest sequence would be
// empty, estimated from the host's sizes: the listed tiles are nseq
// ceil(max_k / 128) and the real ones at most total_k / 128 + nseq.  Each
// packed item costs the producer a little more (5-7 % with equal lengths,
// no empty items to save); with 8 sequences of 2k-16k tokens (41 % empty)
// the packed lists were 9 % faster at Dp = 64 and as fast at Dp = 128.
// The offsets then sit in shared memory, which bounds the sequences.
bool packed_lists(const SegGeo& g) {
  if (!g.varlen || g.nseg > kCuSmem) return false;
  const int64_t listed = g.nseg * ((g.max_k + kBlockN - 1) / kBlockN);
  const int64_t real_max = g.total_k / kBlockN + g.nseg;
  return 4 * real_max <= 3 * listed;
}

cudaError_t launch_any(ProParams& prm, bool vec, int mode, cudaStream_t st) {
  const SegGeo& g = prm.g;
  const bool bf16 = g.dtype == 1;
  const bool d64 = g.Dp == 64;
  if (vec) {
    // tensor maps of the inputs (a tensor with no tokens is never read)
    prm.q_hnd = !g.varlen && g.q_tok_stride == g.D;
    prm.k_hnd = !g.varlen && g.k_tok_stride == g.D;
    const int64_t ntq = g.varlen ? g.total_q : g.nseg * g.Lq;
    const int64_t ntk = g.varlen ? g.total_k : g.nseg * g.Lk;
    if (g.strided) {
      if ((prm.q != nullptr && ntq > 0 &&
           !view_map(&prm.mq, prm.q, g.D, g.Dp, g.Lq, g.Hq, g.nseg, g.q_tok_stride,
                     g.q_head_stride, g.q_seg_stride)) ||
          (ntk > 0 && (!view_map(&prm.mk, prm.k, g.D, g.Dp, g.Lk, g.Hkv, g.nseg, g.k_tok_stride,
                                 g.k_head_stride, g.k_seg_stride) ||
                       !view_map(&prm.mv, prm.v, g.D, g.Dp, g.Lk, g.Hkv, g.nseg, g.k_tok_stride,
                                 g.k_head_stride, g.k_seg_stride))))
        return cudaErrorInvalidValue;
    } else {
      if (prm.q != nullptr && ntq > 0 &&
          !input_map(&prm.mq, prm.q, g.D, g.Dp, g.Hq, g.Lq, ntq, prm.q_hnd))
        return cudaErrorInvalidValue;
      if (ntk > 0 && (!input_map(&prm.mk, prm.k, g.D, g.Dp, g.Hkv, g.Lk, ntk, prm.k_hnd) ||
                      !input_map(&prm.mv, prm.v, g.D, g.Dp, g.Hkv, g.Lk, ntk, prm.k_hnd)))
        return cudaErrorInvalidValue;
    }
    if (packed_lists(g)) {
      if (bf16) return d64 ? launch_t<true, true, 64, true>(prm, mode, st)
                           : launch_t<true, true, 128, true>(prm, mode, st);
      return d64 ? launch_t<true, false, 64, true>(prm, mode, st)
                 : launch_t<true, false, 128, true>(prm, mode, st);
    }
    if (bf16) return d64 ? launch_t<true, true, 64, false>(prm, mode, st)
                         : launch_t<true, true, 128, false>(prm, mode, st);
    return d64 ? launch_t<true, false, 64, false>(prm, mode, st)
               : launch_t<true, false, 128, false>(prm, mode, st);
  }
  if (bf16) return d64 ? launch_t<false, true, 64, false>(prm, mode, st)
                       : launch_t<false, true, 128, false>(prm, mode, st);
  return d64 ? launch_t<false, false, 64, false>(prm, mode, st)
             : launch_t<false, false, 128, false>(prm, mode, st);
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
  prm.ksum = b.ksum; prm.vmax = b.vmax;
  prm.cnt_a = b.sync; prm.cnt_b = b.sync + kMaxGroups; prm.gbar = b.sync + 2 * kMaxGroups;
  prm.cnt_q = b.sync + 3 * kMaxGroups;
  prm.status = b.status; prm.timeout_ns = b.timeout_ns;
  prm.v16 = b.v16;
  prm.one = 1.0f;
  // One launch keeps a few groups of K and V in L2 between their two reads
  // (the A list runs ahead of the B list).  Two launches (the Q tiles, the K
  // and V statistics and the final items; then the K and V tiles from the
  // final statistics, with counters of their own) re-read K and V from DRAM.
  // With three CTAs per SM one launch measured as fast or faster at every
  // size tried (134 MB to 402 MB of K and V), so two launches run only when
  // a test asks for them.
  const bool two = b.launches == 2;
  if (!two) return launch_any(prm, vec, kPlanAll, st);
  cudaError_t e = launch_any(prm, vec, kPlanStatsQ, st);
  if (e != cudaSuccess) return e;
  if ((g.varlen ? g.max_k : g.Lk) <= 0) return cudaSuccess;    // no keys to quantise
  ProParams kv = prm;
  kv.cnt_a = b.sync + 4 * kMaxGroups; kv.cnt_b = b.sync + 5 * kMaxGroups;
  kv.gbar = b.sync + 6 * kMaxGroups; kv.cnt_q = b.sync + 7 * kMaxGroups;
  return launch_any(kv, vec, kPlanKV, st);
}

// ------------------------------------------- statistics without allocation
// Scratch of the allocation-free statistics entry point: a header (status
// word, list counters and group-barrier counters), then
// per-channel K sums (8 B), V maxima (4 B) and V multipliers (4 B) for at
// most kStaticStatEntries (segment, kv head, channel) triples.  It lives in
// the module image, so every device that loads this library holds it until
// the process exits; concurrent calls share it.
namespace {
constexpr size_t kStaticHeader = 256 + 16 * kMaxGroups;
__device__ __align__(256) unsigned char g_stats_scratch[
    kStaticHeader + kStaticStatEntries * (8 + 4 + 4)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

cudaError_t read_kv_stats_static_status(uint32_t* word, cudaStream_t st) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_stats_scratch, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e;
}

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
  prm.cnt_a = reinterpret_cast<unsigned int*>(base + 256);
  prm.cnt_b = prm.cnt_a + kMaxGroups;
  prm.gbar = prm.cnt_a + 2 * kMaxGroups;
  prm.cnt_q = prm.cnt_a + 3 * kMaxGroups;
  prm.ksum = base + kStaticHeader;
  prm.vmax = reinterpret_cast<uint32_t*>(base + kStaticHeader + kStaticStatEntries * 8);
  prm.v_inv = reinterpret_cast<float*>(base + kStaticHeader + kStaticStatEntries * 12);
  prm.timeout_ns = timeout_ns;
  prm.one = 1.0f;
  return launch_any(prm, vec, kPlanStats, st);
}

}  // namespace sage
