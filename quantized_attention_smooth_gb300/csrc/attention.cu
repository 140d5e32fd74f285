// Fused quantised attention forward on sm_103a tensor cores (tcgen05).
//
// Method (stable-diffusion.cpp "SageAttention" kernel table: INT8 Q/K, FP8 PV
// with an FP32 buffer; SageAttention overview, Core features): per query
// tile of 128 rows and key tile of 128 keys,
//   S   = q8 . k8^T                      exact integers
//   x   = S * ((s_q * s_k) * sm_scale * log2 e)   base-2 logits, -inf masked
//   m'  = max(m, rowmax x);  P = 2^(x - m');  l = l * 2^(m - m') + sum P
//   O   = O * 2^(m - m') + e4m3(448 P) . v~
// and finally out = O * s_v / (448 l) in fp32 for the caller's D channels.
// The kernel carries 448 P and 448 l (the FP16-PV variant: P and l).
//
// GB300 mapping.  sm_103a has no INT8 tcgen05 MMA, so QK^T runs as
// kind::f16 on operands that hold the int8 codes as exact fp16 integers;
// each product is < 2^14 and a 128-term row sum < 2^21, so the fp32
// accumulator holds the exact INT32 result.  PV runs as kind::f8f6f4 (e4m3 x
// e4m3 -> fp32) with both operands in shared memory.
//
// One CTA owns one (segment, query head) and TWO 128-row query tiles that
// share every K/V tile.  16 warps:
//   warps 0-3   softmax of query tile 0 (one row per thread, TMEM lane = row)
//   warps 4-7   softmax of query tile 1
//   warps 8-11  correction: rescale O in TMEM when the row max grows (while
//               the softmax is still exponentiating), then the epilogue
//   warp 12     TMA producer of both Q tiles and the K ring
//   warp 13     tcgen05 issuer of query tile 0 (one thread) and TMEM owner
//   warp 14     TMA producer of the V ring
//   warp 15     tcgen05 issuer of query tile 1 (one thread)
// TMEM (512 columns): S0 | S1 | O0 | O1.  P~ (e4m3) goes to shared memory in
// the 128-byte swizzled K-major layout, so S_t is free as soon as the softmax
// has loaded it into registers: QK^T of the next key tile then runs on the
// tensor core while the softmax is still exponentiating the current one.
// Per query tile t and key tile j the hand-offs are:
//   MMA --s_full--> softmax --s_free--> MMA (next QK^T into S_t)
//                   softmax --alpha_ready[j&1]--> correction --pv_ready--> MMA
//                   softmax (P~ in smem) -------------------pv_ready--> MMA
//   MMA (PV done) --o_done--> correction (rescale), softmax (P~ buffer free)
// K and V stages are released by one arrival per active query tile.  Every
// wait is bounded: a wait that runs out raises the workspace status word and
// an abort flag, all roles drain their in-flight copies and MMAs, and the CTA
// frees its TMEM and exits.

#include <cuda_fp16.h>

#include <atomic>

#include "sage_device.cuh"
#include "sage_geom.h"
#include "sage_kernels.h"

namespace sage {
namespace {

constexpr int kKStages = 2;   // K ring (released after the second QK^T)
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2_448 = 8.80735492205760410750f;
constexpr int kAtomBytes = 128 * 128;   // 128 rows x 128 bytes (swizzle atom column)
constexpr unsigned kFull = 0xFFFFFFFFu;
// register split (launch: 512 threads x 128): 2 x 128 x 192 + 128 x 80 + 128 x 48
constexpr int kSoftmaxRegs = 192;
constexpr int kCorrRegs = 80;
constexpr int kMiscRegs = 48;

// Shared memory of one CTA.  kV16: the FP16-PV variant (fp16 P~ and V; its
// larger operands leave room for one K and one V stage only).
template <int DP, bool kV16 = false>
struct Layout {
  static constexpr int kTiles = 2;                     // query tiles per CTA
  static constexpr int kKSt = kV16 ? 1 : kKStages;     // K ring
  static constexpr int kVStages = kV16 ? 1 : 3;        // V ring (released after a PV)
  static constexpr int kQBytes = kBlockM * DP * 2;     // one query tile
  static constexpr int kKBytes = kBlockN * DP * 2;
  static constexpr int kVBytes = DP * kBlockN * (kV16 ? 2 : 1);
  static constexpr int kPBytes = kBlockM * kBlockN * (kV16 ? 2 : 1);   // P~ of one tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTiles * kQBytes;
  static constexpr int kVOff = kKOff + kKSt * kKBytes;
  static constexpr int kPOff = kVOff + kVStages * kVBytes;
  static constexpr int kBarOff = kPOff + kTiles * kPBytes;
  // q_full, k_full[SK], k_empty[SK], v_full[SV], v_empty[SV], then per tile:
  // s_full, s_free, alpha_ready[2], pv_ready, o_done, l_ready, drain, epi_full, epi_free;
  // sv_ready
  static constexpr int kNumBars = 1 + 2 * kKSt + 2 * kVStages + 2 * 10 + 1;
  static constexpr int kAlphaOff = (kBarOff + kNumBars * 8 + 15) / 16 * 16;
  static constexpr int kLOff = kAlphaOff + 4 * kBlockM * 4;
  static constexpr int kSvOff = kLOff + 2 * kBlockM * 4;
  static constexpr int kMiscOff = kSvOff + DP * 4;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// S (128x128 fp32 in TMEM) = Q tile . K tile^T, K dimension DP in steps of 16.
// q_lo / k_lo: low descriptor words of the 1024-byte aligned operand tiles.
template <int DP>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo) {
  constexpr uint32_t idesc = make_idesc(kFmtF16, kFmtF16, kBlockM, kBlockN);
#pragma unroll
  for (int kk = 0; kk < DP / 16; ++kk) {
    const uint32_t off = ((kk / 4) * kAtomBytes + (kk % 4) * 32) >> 4;
    mma_f16_ss_lo(d_tmem, q_lo + off, k_lo + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (128xDP fp32 in TMEM) (+)= P~ (128x128 e4m3, smem) . V~ tile^T
// (V~ stored DP rows x 128 keys), K dimension 128 keys in steps of 32.
template <int DP>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_lo, uint32_t v_lo,
                                         bool accumulate) {
  constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, kBlockM, DP);
#pragma unroll
  for (int kk = 0; kk < kBlockN / 32; ++kk)
    mma_f8_ss_lo(o_tmem, p_lo + ((kk * 32) >> 4), v_lo + ((kk * 32) >> 4), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
}

// FP16-PV: O (128xDP fp32 in TMEM) (+)= P~ (128x128 fp16, smem, two 64-key
// swizzle atoms) . V16 tile^T (DP rows x 128 keys fp16, two 64-key atoms),
// K dimension 128 keys in steps of 16.
template <int DP>
__device__ __forceinline__ void issue_pv16(uint32_t o_tmem, uint32_t p_lo, uint32_t v_lo,
                                           bool accumulate) {
  constexpr uint32_t idesc = make_idesc(kFmtF16, kFmtF16, kBlockM, DP);
#pragma unroll
  for (int kk = 0; kk < kBlockN / 16; ++kk) {
    const uint32_t p_off = ((kk / 4) * kAtomBytes + (kk % 4) * 32) >> 4;
    const uint32_t v_off = ((kk / 4) * (DP * 128) + (kk % 4) * 32) >> 4;
    mma_f16_ss_lo(o_tmem, p_lo + p_off, v_lo + v_off, idesc,
                  (accumulate || kk > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag, uint32_t* status,
                                         uint64_t timeout_ns) {
  bool ok = mbar_wait(bar, parity, abort_flag, status, timeout_ns);
  return __all_sync(kFull, ok);
}

template <int DP, bool kV16>
__global__ void __launch_bounds__(kThreads, 1)
attn_kernel(const __grid_constant__ CUtensorMap tm_q,
            const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v,
            const __grid_constant__ CUtensorMap tm_o, const AttnParams p) {
  using L = Layout<DP, kV16>;
  constexpr int kKStages = L::kKSt;
  constexpr int kVStages = L::kVStages;
  // Shared memory, 1024-byte aligned for the swizzled tiles.  At Dp = 64 the
  // base is declared aligned (the driver places dynamic shared memory after
  // its 1 KB per-block reservation; a base off the grid is reported and the
  // CTA does nothing): the code generator then keeps that instance free of
  // register spills, 4 % faster.  At Dp = 128 the same declaration makes it
  // spill, so that instance rounds the base up at run time.
  uint8_t* smem;
  if constexpr (DP == 64) {
    extern __shared__ __align__(1024) uint8_t smem_al[];
    if ((smem_u32(smem_al) & 1023u) != 0) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadItem);
      return;
    }
    smem = smem_al;
  } else {
    extern __shared__ uint8_t smem_raw[];
    smem = align1024(smem_raw);
  }
  const SegGeo& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which query tiles: a pair (heaviest causal pairs first), or, for
  // the balanced dense launch (flat_pairs >= 0), a 1D list of pairs in
  // (segment, head, pair) order followed by the single tiles of the pairs
  // that would have formed the last partial wave
  int64_t s, h, qt0;
  int ntile = 2;
  if (p.flat_pairs >= 0) {
    const int64_t npairs = ((g.Lq + kBlockM - 1) / kBlockM + 1) / 2;
    int64_t pu = blockIdx.x, sub = 0;
    if (pu >= p.flat_pairs) {
      sub = (pu - p.flat_pairs) & 1;
      pu = p.flat_pairs + (pu - p.flat_pairs) / 2;
      ntile = 1;
    }
    const int64_t sh = pu / npairs;
    h = sh % g.Hq;
    s = sh / g.Hq;
    qt0 = 2 * (pu % npairs) + sub;
  } else {
    s = blockIdx.z;
    h = blockIdx.y;
    qt0 = 2 * static_cast<int64_t>(p.causal ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x);
  }
  int64_t qstart = 0, len_q = g.Lq, kstart = 0, len_k = g.Lk;
  if (g.varlen) {
    const bool okq = seg_range(g.cu_q, s, g.total_q, g.max_q, &qstart, &len_q);
    const bool okk = seg_range(g.cu_k, s, g.total_k, g.max_k, &kstart, &len_k);
    if (!okq || !okk) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
  }
  if (qt0 * kBlockM >= len_q) return;
  // query rows this CTA owns: a single tile leaves the next one to its neighbour
  const int64_t qlim = ntile == 2 ? len_q : min(len_q, (qt0 + 1) * kBlockM);
  const int64_t hk = h / (g.Hq / g.Hkv);
  const int nk_all = static_cast<int>((len_k + kBlockN - 1) / kBlockN);
  int n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int64_t qt = qt0 + t;
    if (qt * kBlockM >= qlim) n_t[t] = 0;
    else n_t[t] = (p.causal && nk_all > qt + 1) ? static_cast<int>(qt + 1) : nk_all;
  }
  const int n_max = n_t[0] > n_t[1] ? n_t[0] : n_t[1];
  const int64_t q_row0 = ws_seg_base(g.varlen, s, qstart, g.Hq, g.q_head_rows) +
                         h * g.q_head_rows + qt0 * kBlockM;
  const int64_t k_row0 = ws_seg_base(g.varlen, s, kstart, g.Hkv, g.k_head_rows) +
                         hk * g.k_head_rows;
  const int64_t v_row0 = (g.varlen ? 0 : s * g.Hkv * DP) + hk * DP;
  const int64_t v_col0 = g.varlen ? ws_seg_base(1, s, kstart, 0, 0) : 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* s_full = v_empty + kVStages;      // [2]
  uint64_t* s_free = s_full + 2;              // [2]
  // the softmax may run one key tile ahead of the correction (S is released
  // early), so the row rescale factors and their barrier alternate by j & 1
  uint64_t* alpha_ready = s_free + 2;         // [2 tiles][2 key-tile parities]
  uint64_t* pv_ready = alpha_ready + 4;       // [2] softmax (128) + correction (128)
  uint64_t* o_done = pv_ready + 2;            // [2]
  uint64_t* l_ready = o_done + 2;             // [2]
  uint64_t* drain = l_ready + 2;              // [2]
  // epilogue staging: a chunk's rows are in shared memory; a reused staging
  // buffer has been read by its tensor store
  uint64_t* epi_full = drain + 2;             // [2]
  uint64_t* epi_free = epi_full + 2;          // [2]
  uint64_t* sv_ready = epi_free + 2;          // the V scales are in shared memory
  float* alpha_s = reinterpret_cast<float*>(smem + L::kAlphaOff);   // [2][2][128]
  float* l_s = reinterpret_cast<float*>(smem + L::kLOff);           // [2][128]
  float* sv_cache = reinterpret_cast<float*>(smem + L::kSvOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  // V tile j (channel-major: DP rows x 128 keys) into a ring stage: one box of
  // e4m3, or two 64-key boxes of fp16 (one 128-byte swizzle atom each)
  auto load_v = [&](uint8_t* dst, int j, uint64_t* bar) {
    if constexpr (kV16) {
      for (int a = 0; a < 2; ++a)
        tma_load_2d(dst + a * (DP * 128), &tm_v,
                    static_cast<int32_t>(v_col0 + j * kBlockN + 64 * a),
                    static_cast<int32_t>(v_row0), bar);
    } else {
      tma_load_2d(dst, &tm_v, static_cast<int32_t>(v_col0 + j * kBlockN),
                  static_cast<int32_t>(v_row0), bar);
    }
  };

  // The producers set up their own rings and issue the copies that need no
  // free slot (Q, the first K and V tiles) at once, so those loads overlap
  // the rest of the set-up.
  const uint32_t active = n_t[1] > 0 ? 2u : 1u;   // query tiles reading K/V
  int k_last = -1, v_last = -1;                    // last tile each producer issued
  if (warp == 12 && lane == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], active);
    }
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    if (n_max > 0) mbar_expect_tx(q_full, (n_t[1] > 0 ? 2 : 1) * L::kQBytes);
    for (int t = 0; t < 2; ++t) {
      if (n_t[t] == 0) continue;
      for (int a = 0; a < DP / 64; ++a)
        tma_load_2d(smem + L::kQOff + t * L::kQBytes + a * kAtomBytes, &tm_q, a * 64,
                    static_cast<int32_t>(q_row0 + t * kBlockM), q_full);
    }
    for (int j = 0; j < n_max && j < kKStages; ++j) {
      if (j == p.skip_kv_tile) continue;   // failure injection (tests only)
      mbar_expect_tx(&k_full[j], L::kKBytes);
      for (int a = 0; a < DP / 64; ++a)
        tma_load_2d(smem + L::kKOff + j * L::kKBytes + a * kAtomBytes, &tm_k, a * 64,
                    static_cast<int32_t>(k_row0 + j * kBlockN), &k_full[j]);
      k_last = j;
    }
  }
  if (warp == 14 && lane == 0) {
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], active);
    }
    mbar_fence_init();
    tma_prefetch_desc(&tm_v);
    for (int j = 0; j < n_max && j < kVStages; ++j) {
      mbar_expect_tx(&v_full[j], L::kVBytes);
      load_v(smem + L::kVOff + j * L::kVBytes, j, &v_full[j]);
      v_last = j;
    }
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(sv_ready, DP);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], kBlockM);
      mbar_init(&alpha_ready[2 * t], kBlockM);
      mbar_init(&alpha_ready[2 * t + 1], kBlockM);
      mbar_init(&pv_ready[t], 2 * kBlockM);
      mbar_init(&o_done[t], 1);
      mbar_init(&l_ready[t], kBlockM);
      mbar_init(&epi_full[t], kBlockM);
      mbar_init(&epi_free[t], 1);
      mbar_init(&drain[t], 1);
    }
    mbar_fence_init();
  }
  if (warp == 13) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int wg = warp >> 2;

  // Epilogue of query tile t by one warpgroup (thread r holds row r; the
  // thread with r == 0 issues the tensor stores and counts them in stores):
  // out = O * s_v / (448 l), the caller's D channels only.  Tensor stores
  // where their clipping is exact (dense outputs end at Lq; full tiles of a
  // packed sequence), from staging chunks of 128 rows x 32 fp32 in the
  // 128-byte swizzle layout, held in Q_t and P~_t, which the tensor cores no
  // longer read; per-row stores otherwise.  False if a bounded wait ran out.
  auto epilogue = [&](int t, int r, uint32_t lane_off, int& stores) -> bool {
    const int64_t qtile = qt0 + t;
    if (qtile * kBlockM >= qlim) return true;              // not this CTA's tile
    const int D = static_cast<int>(g.D);
    const int64_t seg_off = g.varlen ? qstart * p.out_tok_stride : s * p.out_seg_stride;
    const int64_t qi = qtile * kBlockM + r;
    float* orow = p.out + seg_off + h * p.out_head_stride + qi * p.out_tok_stride;
    const bool valid = qi < len_q;
    if (n_t[t] == 0) {            // no visible key (empty key sequence): zeros
      if (valid)
        for (int c = 0; c < D; ++c) orow[c] = 0.0f;
      return true;
    }
    // l_ready completes once, when the softmax has finished the tile; by then
    // it has waited for every PV but the last, so o_done's parity names the
    // last PV exactly, even for a warpgroup that has not followed its phases
    if (!wait_all(&l_ready[t], 0, abort_flag, p.status, p.timeout_ns) ||
        !wait_all(&o_done[t], (n_t[t] - 1) & 1, abort_flag, p.status, p.timeout_ns))
      return false;
    if (!wait_all(sv_ready, 0, abort_flag, p.status, p.timeout_ns)) return false;
    tc_fence_after();
    const float l448 = l_s[t * kBlockM + r];
    const float inv = l448 > 0.0f ? __fdiv_rn(1.0f, l448) : 0.0f;
    const uint32_t to = tbase + lane_off + 256 + t * DP;
    if (p.out_tma != 0 && (!g.varlen || (qtile + 1) * kBlockM <= len_q)) {
      // 16 KB staging buffers: the pieces of Q_t, then those of P~_t
      constexpr int kQBufs = L::kQBytes / 16384, kBufs = kQBufs + L::kPBytes / 16384;
      uint8_t* const q_t = smem + L::kQOff + t * L::kQBytes;
      uint8_t* const p_t = smem + L::kPOff + t * L::kPBytes;
      for (int cc = 0; cc < DP / 32 && 32 * cc < D; ++cc) {
        const int bi = cc % kBufs;
        uint8_t* buf = bi < kQBufs ? q_t + bi * 16384 : p_t + (bi - kQBufs) * 16384;
        if (cc >= kBufs) {        // the store of chunk cc - kBufs must have read it
          if (r == 0) {
            bulk_wait_read<kBufs - 1>();
            mbar_arrive(&epi_free[t]);
          }
          if (!wait_all(&epi_free[t], (cc - kBufs) & 1, abort_flag, p.status, p.timeout_ns))
            return false;
        }
        uint4* row = reinterpret_cast<uint4*>(buf + r * 128);
#pragma unroll
        for (int half = 0; half < 2; ++half) {     // 16 columns at a time
          uint32_t o[16];
          tmem_ld16(to + 32 * cc + 16 * half, o);
          tmem_ld_wait();
          reg_fence(o);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int c = 32 * cc + 16 * half + 4 * k4;
            uint4 v;
            v.x = __float_as_uint(__uint_as_float(o[4 * k4]) * sv_cache[c] * inv);
            v.y = __float_as_uint(__uint_as_float(o[4 * k4 + 1]) * sv_cache[c + 1] * inv);
            v.z = __float_as_uint(__uint_as_float(o[4 * k4 + 2]) * sv_cache[c + 2] * inv);
            v.w = __float_as_uint(__uint_as_float(o[4 * k4 + 3]) * sv_cache[c + 3] * inv);
            row[(4 * half + k4) ^ (r & 7)] = v;
          }
        }
        fence_proxy_async_smem();
        // every row of the chunk is staged (all threads wait, so none can
        // arrive twice in one phase)
        mbar_arrive(&epi_full[t]);
        if (!wait_all(&epi_full[t], cc & 1, abort_flag, p.status, p.timeout_ns)) return false;
        if (r == 0) {
          const int32_t row0 = static_cast<int32_t>(qtile * kBlockM);
          if (p.out_tma == 3)
            tma_store_3d(&tm_o, buf, 32 * cc, static_cast<int32_t>(h),
                         static_cast<int32_t>(qstart) + row0);
          else if (p.out_tma == 1)
            tma_store_4d(&tm_o, buf, 32 * cc, row0, static_cast<int32_t>(h),
                         static_cast<int32_t>(s));
          else
            tma_store_4d(&tm_o, buf, 32 * cc, static_cast<int32_t>(h), row0,
                         static_cast<int32_t>(s));
          bulk_commit();
          ++stores;
        }
      }
      return true;
    }
    const bool vec = (D % 4 == 0) && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
#pragma unroll 1
    for (int cc = 0; cc < DP / 16; ++cc) {
      uint32_t o[16];
      tmem_ld16(to + 16 * cc, o);
      tmem_ld_wait();
      reg_fence(o);
      if (!valid) continue;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = 16 * cc + i;
        if (vec && (i & 3) == 0 && c < D) {
          float4 v4;
          v4.x = __uint_as_float(o[i]) * sv_cache[c] * inv;
          v4.y = __uint_as_float(o[i + 1]) * sv_cache[c + 1] * inv;
          v4.z = __uint_as_float(o[i + 2]) * sv_cache[c + 2] * inv;
          v4.w = __uint_as_float(o[i + 3]) * sv_cache[c + 3] * inv;
          *reinterpret_cast<float4*>(orow + c) = v4;
        } else if (!vec && c < D) {
          orow[c] = __uint_as_float(o[i]) * sv_cache[c] * inv;
        }
      }
    }
    return true;
  };

  if (wg == 3) {
    regs_decrease<kMiscRegs>();
    if (warp == 12 && lane == 0) {
      // ============================================== TMA producer: K (Q and
      // the first kKStages tiles went out during set-up)
      int last = k_last;
      for (int j = kKStages; j < n_max; ++j) {
        const int st = j % kKStages;
        if (j >= kKStages &&
            !mbar_wait(&k_empty[st], ((j / kKStages) - 1) & 1, abort_flag, p.status,
                       p.timeout_ns))
          break;
        if (j == p.skip_kv_tile) continue;   // failure injection (tests only)
        mbar_expect_tx(&k_full[st], L::kKBytes);
        uint8_t* kdst = smem + L::kKOff + st * L::kKBytes;
        for (int a = 0; a < DP / 64; ++a)
          tma_load_2d(kdst + a * kAtomBytes, &tm_k, a * 64,
                      static_cast<int32_t>(k_row0 + j * kBlockN), &k_full[st]);
        last = j;
      }
      // no copy may still be in flight when the CTA exits
      if (n_max > 0) mbar_wait(q_full, 0, nullptr, p.status, p.timeout_ns);
      for (int j = max(0, last - kKStages + 1); j <= last; ++j)
        if (j != p.skip_kv_tile)
          mbar_wait(&k_full[j % kKStages], (j / kKStages) & 1, nullptr, p.status,
                    p.timeout_ns);
    } else if (warp == 14 && lane == 0) {
      // ============================================== TMA producer: V (the
      // first kVStages tiles went out during set-up)
      int last = v_last;
      for (int j = kVStages; j < n_max; ++j) {
        const int st = j % kVStages;
        if (j >= kVStages &&
            !mbar_wait(&v_empty[st], ((j / kVStages) - 1) & 1, abort_flag, p.status,
                       p.timeout_ns))
          break;
        mbar_expect_tx(&v_full[st], L::kVBytes);
        load_v(smem + L::kVOff + st * L::kVBytes, j, &v_full[st]);
        last = j;
      }
      for (int j = max(0, last - kVStages + 1); j <= last; ++j)
        mbar_wait(&v_full[j % kVStages], (j / kVStages) & 1, nullptr, p.status, p.timeout_ns);
    } else if ((warp == 13 || warp == 15) && lane == 0 && n_t[warp == 13 ? 0 : 1] > 0) {
      // ============================================== tcgen05 issuer of tile t
      const int t = warp == 13 ? 0 : 1;
      const int n = n_t[t];
      const uint32_t qa = sdesc_sw128_lo(smem_u32(smem + L::kQOff + t * L::kQBytes));
      const uint32_t ka0 = sdesc_sw128_lo(smem_u32(smem + L::kKOff));
      const uint32_t va0 = sdesc_sw128_lo(smem_u32(smem + L::kVOff));
      const uint32_t pa = sdesc_sw128_lo(smem_u32(smem + L::kPOff + t * L::kPBytes));
      const uint32_t ts = tbase + t * 128, to = tbase + 256 + t * DP;
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, p.timeout_ns) &&
                mbar_wait(&k_full[0], 0, abort_flag, p.status, p.timeout_ns);
      bool issued = false;
      if (ok) {
        tc_fence_after();
        issue_qk<DP>(ts, qa, ka0);
        tc_commit(&s_full[t]);
        tc_commit(&k_empty[0]);
        issued = true;
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          // next QK^T into S_t as soon as the softmax has read S_t(j)
          const int sk = (j + 1) % kKStages;
          ok = mbar_wait(&s_free[t], j & 1, abort_flag, p.status, p.timeout_ns) &&
               mbar_wait(&k_full[sk], ((j + 1) / kKStages) & 1, abort_flag, p.status,
                         p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          issue_qk<DP>(ts, qa, ka0 + sk * (L::kKBytes >> 4));
          tc_commit(&s_full[t]);
          tc_commit(&k_empty[sk]);
        }
        const int sv = j % kVStages;
        ok = mbar_wait(&v_full[sv], (j / kVStages) & 1, abort_flag, p.status, p.timeout_ns) &&
             mbar_wait(&pv_ready[t], j & 1, abort_flag, p.status, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
        if constexpr (kV16) issue_pv16<DP>(to, pa, va0 + sv * (L::kVBytes >> 4), j > 0);
        else issue_pv<DP>(to, pa, va0 + sv * (L::kVBytes >> 4), j > 0);
        tc_commit(&o_done[t]);
        tc_commit(&v_empty[sv]);
      }
      // key tiles the other query tile reads but this one does not (causal
      // tile 0 skips the last one): release them once they have landed
      for (int j = n; ok && j < n_max; ++j) {
        ok = mbar_wait(&k_full[j % kKStages], (j / kKStages) & 1, abort_flag, p.status,
                       p.timeout_ns) &&
             mbar_wait(&v_full[j % kVStages], (j / kVStages) & 1, abort_flag, p.status,
                       p.timeout_ns);
        if (!ok) break;
        mbar_arrive(&k_empty[j % kKStages]);
        mbar_arrive(&v_empty[j % kVStages]);
      }
      if (issued) {   // every MMA must finish before TMEM is released
        tc_commit(&drain[t]);
        mbar_wait(&drain[t], 0, nullptr, p.status, p.timeout_ns);
      }
    }
    // tile 1's epilogue, alongside tile 0's on the correction warps (lanes
    // without a role wait here for their lane 0 instead of spinning)
    __syncwarp();
    const int r3 = threadIdx.x - 3 * kBlockM;
    int stores = 0;
    epilogue(1, r3, static_cast<uint32_t>((warp & 3) * 32) << 16, stores);
    if (r3 == 0 && stores > 0) bulk_wait_all();
  } else if (wg == 2) {
    // ================================================ correction + tile 0's epilogue
    regs_decrease<kCorrRegs>();
    const int r = threadIdx.x - 256;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    if (r < DP) {             // the V scales for the epilogue, off the set-up path
      sv_cache[r] = kV16 ? 1.0f : p.s_v[(s * g.Hkv + hk) * DP + r];
      mbar_arrive(sv_ready);
    }
    bool ok = true;
    for (int j = 0; ok && j < n_max; ++j) {
      for (int t = 0; t < 2; ++t) {
        if (j >= n_t[t]) continue;
        ok = wait_all(&alpha_ready[2 * t + (j & 1)], (j >> 1) & 1, abort_flag, p.status,
                      p.timeout_ns);
        if (!ok) break;
        if (j > 0) {
          // O_t holds PV of key tiles < j once PV(j-1) is done
          ok = wait_all(&o_done[t], (j - 1) & 1, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          const float alpha = alpha_s[(2 * t + (j & 1)) * kBlockM + r];
          if (__any_sync(kFull, alpha < 1.0f)) {
            const uint32_t to = tbase + lane_off + 256 + t * DP;
            // 16-column chunks, the next chunk's load in flight while this
            // one is scaled; a buffer is reloaded only after its store
            // has completed
            constexpr int NC = DP / 16;
            const float2 a2 = make_float2(alpha, alpha);
            uint32_t ob[2][16];
            tmem_ld16(to, ob[0]);
            tmem_ld_wait();
            reg_fence(ob[0]);
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
              uint32_t (&cur)[16] = ob[cc & 1];
              if (cc + 1 < NC) {
                if (cc >= 1) tmem_st_wait();
                tmem_ld16(to + 16 * (cc + 1), ob[(cc + 1) & 1]);
              }
#pragma unroll
              for (int i = 0; i < 16; i += 2) {     // packed multiplies, same rounding
                const float2 v = __fmul2_rn(
                    make_float2(__uint_as_float(cur[i]), __uint_as_float(cur[i + 1])), a2);
                cur[i] = __float_as_uint(v.x);
                cur[i + 1] = __float_as_uint(v.y);
              }
              tmem_st16(to + 16 * cc, cur);
              if (cc + 1 < NC) {
                tmem_ld_wait();
                reg_fence(ob[(cc + 1) & 1]);
              }
            }
            tmem_st_wait();
          }
        }
        tc_fence_before();
        mbar_arrive(&pv_ready[t]);
      }
    }
    int stores = 0;                 // tensor stores issued (thread r == 0)
    if (ok) ok = epilogue(0, r, lane_off, stores);
    // the tensor stores must be complete before the CTA ends
    if (r == 0 && stores > 0) bulk_wait_all();
  } else {
    // ================================================ softmax of tile wg
    regs_increase<kSoftmaxRegs>();
    const int t = wg;
    const int r = threadIdx.x - t * kBlockM;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tbase + lane_off + t * 128;
    // this row of the P~ tile: 128 bytes, 16-byte chunks swizzled by row % 8
    uint8_t* prow = smem + L::kPOff + t * L::kPBytes + r * 128;
    const int rsw = r & 7;
    const int64_t qi = (qt0 + t) * kBlockM + r;          // query index in segment
    const int n = n_t[t];
    const float* skp = p.s_k + k_row0 / kBlockN;
    const float sq = n > 0 ? p.s_q[q_row0 + t * kBlockM + r] : 0.0f;
    const int64_t kend = p.causal ? (len_k < qi + 1 ? len_k : qi + 1) : len_k;
    float m = -INFINITY, l448 = 0.0f;
    float sk_next = n > 0 ? skp[0] : 0.0f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const float sk = sk_next;
      if (j + 1 < n) sk_next = skp[j + 1];
      ok = wait_all(&s_full[t], j & 1, abort_flag, p.status, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
      tmem_ld32(ts, sr[0]);
      tmem_ld32(ts + 32, sr[1]);
      tmem_ld32(ts + 64, sr[2]);
      tmem_ld32(ts + 96, sr[3]);
      tmem_ld_wait();
      reg_fence(sr[0]);
      reg_fence(sr[1]);
      reg_fence(sr[2]);
      reg_fence(sr[3]);
      tc_fence_before();
      mbar_arrive(&s_free[t]);                           // S_t may be overwritten

      // c > 0 keeps -inf * c = -inf for masked keys even when a scale is 0
      const float c = fmaxf((sq * sk) * p.scale_log2, 1e-30f);
      const int64_t key0 = static_cast<int64_t>(j) * kBlockN;
      if (key0 + kBlockN > kend) {
        const int64_t lim64 = kend - key0;
        const int lim = lim64 < 0 ? 0 : static_cast<int>(lim64);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) sr[i >> 5][i & 31] = 0xFF800000u;   // -inf
      }
      // row max of the exact integer scores, four independent chains
      float mx0 = __uint_as_float(sr[0][0]), mx1 = __uint_as_float(sr[1][0]);
      float mx2 = __uint_as_float(sr[2][0]), mx3 = __uint_as_float(sr[3][0]);
#pragma unroll
      for (int i = 1; i < 32; ++i) {
        mx0 = fmaxf(mx0, __uint_as_float(sr[0][i]));
        mx1 = fmaxf(mx1, __uint_as_float(sr[1][i]));
        mx2 = fmaxf(mx2, __uint_as_float(sr[2][i]));
        mx3 = fmaxf(mx3, __uint_as_float(sr[3][i]));
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      const float m_new = fmaxf(m, m_tile);
      const float alpha = fast_exp2(m - m_new);          // 0 on the first tile
      alpha_s[(2 * t + (j & 1)) * kBlockM + r] = alpha;
      mbar_arrive(&alpha_ready[2 * t + (j & 1)]);        // correction may rescale O now

      // The oracle's rounding order: the logit x = RN(S c), then
      // d = RN(x - m'), then P = 2^d and P~ = e4m3(448 P) (the FP16-PV
      // variant rounds P itself to fp16).  The subtraction is an FMA with
      // the run-time multiplier `one` = 1, so it cannot be fused with the
      // product: a fused S c - m' would skip the logit's own rounding, which
      // at |x| ~ 1e4 is worth ~5e-4 in the exponent and flips e4m3 codes.
      // 448 P is taken as 2^(RN(d + log2 448)): for the d that carry weight
      // (|d| < 24) that rounding moves P by at most 2^-20 ln 2 relative, a
      // few times the exp2 unit's own error, and it costs one packed add
      // where a multiply after the exp2 measured 2 % slower.  Packed fp32
      // pairs; the two packed sums keep four chains (element i goes to
      // chain i % 4).
      const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_new, -m_new);
      const float2 one2 = make_float2(p.one, p.one);
      const float2 kL448 = make_float2(kLog2_448, kLog2_448);
      // The row is encoded and stored in parts (64 keys at Dp = 128, 32 at
      // Dp = 64), so only a part of it is live in registers: fewer spills, 1-4 %
      // faster than the whole row at once.  The wait for the previous PV comes
      // before the first part's store; at Dp = 64 the shorter PV is done by
      // the end of the first quarter, at Dp = 128 only by mid-row.
      float2 a01 = make_float2(0.0f, 0.0f), a23 = make_float2(0.0f, 0.0f);
      constexpr int kParts = DP == 64 ? 4 : 2;
      constexpr int kPartQ = 32 / kParts;                    // groups of 4 keys per part
      constexpr int kPartW = (kV16 ? 64 : 32) / kParts;      // packed words per part
      constexpr int kPartC = (kV16 ? 16 : 8) / kParts;       // 16-byte chunks per part
#pragma unroll
      for (int part = 0; part < kParts; ++part) {
        uint32_t w[kPartW];
#pragma unroll
        for (int qq = 0; qq < kPartQ; ++qq) {
          const int q4 = kPartQ * part + qq;
          const int i = 4 * q4;
          const uint32_t* src = &sr[i >> 5][i & 31];
          const float2 x01 = __fmul2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])), c2);
          const float2 x23 = __fmul2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])), c2);
          float2 d01 = __ffma2_rn(x01, one2, nm2);
          float2 d23 = __ffma2_rn(x23, one2, nm2);
          if constexpr (!kV16) {                             // log2 of 448 P
            d01 = __fadd2_rn(d01, kL448);
            d23 = __fadd2_rn(d23, kL448);
          }
          const float2 p01 = make_float2(fast_exp2(d01.x), fast_exp2(d01.y));
          const float2 p23 = make_float2(fast_exp2(d23.x), fast_exp2(d23.y));
          if constexpr (kV16) {
            const __half2 h01 = __floats2half2_rn(p01.x, p01.y);
            const __half2 h23 = __floats2half2_rn(p23.x, p23.y);
            w[2 * qq] = *reinterpret_cast<const uint32_t*>(&h01);
            w[2 * qq + 1] = *reinterpret_cast<const uint32_t*>(&h23);
          } else {
            w[qq] = pack_e4m3x2(p01.x, p01.y) | (pack_e4m3x2(p23.x, p23.y) << 16);
          }
          a01 = __fadd2_rn(a01, p01);
          a23 = __fadd2_rn(a23, p23);
        }
        // the P~ buffer is free once PV(j-1) has read it
        if (part == 0 && j > 0) {
          ok = wait_all(&o_done[t], (j - 1) & 1, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
        }
        // 16-byte chunks of the row, swizzled by row % 8 within each 64-key
        // (fp16) or 128-key (e4m3) atom
#pragma unroll
        for (int cc = 0; cc < kPartC; ++cc) {
          const int c16 = kPartC * part + cc;
          *reinterpret_cast<uint4*>(prow + (c16 / 8) * kAtomBytes + (((c16 % 8) ^ rsw) << 4)) =
              make_uint4(w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
        }
      }
      if (!ok) break;
      const float a0 = a01.x, a1 = a01.y, a2 = a23.x, a3 = a23.y;
      fence_proxy_async_smem();
      l448 = l448 * alpha + ((a0 + a1) + (a2 + a3));
      m = m_new;
      mbar_arrive(&pv_ready[t]);
    }
    if (ok && n > 0) {
      l_s[t * kBlockM + r] = l448;
      mbar_arrive(&l_ready[t]);
    }
  }

  // ---- teardown: all roles have drained; release tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ------------------------------------------------- debug: one QK^T tile
template <int DP>
__global__ void __launch_bounds__(128, 1)
debug_qk_kernel(const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k, int64_t q_row0,
                int64_t k_row0, int32_t* out, uint32_t* status,
                uint64_t timeout_ns) {
  using L = Layout<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* ld_full = bars;
  uint64_t* mma_done = bars + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  if (threadIdx.x == 0) {
    mbar_init(ld_full, 1);
    mbar_init(mma_done, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_expect_tx(ld_full, L::kQBytes + L::kKBytes);
    for (int a = 0; a < DP / 64; ++a) {
      tma_load_2d(smem + L::kQOff + a * kAtomBytes, &tm_q, a * 64,
                  static_cast<int32_t>(q_row0), ld_full);
      tma_load_2d(smem + L::kKOff + a * kAtomBytes, &tm_k, a * 64,
                  static_cast<int32_t>(k_row0), ld_full);
    }
    ok = mbar_wait(ld_full, 0, nullptr, status, timeout_ns);
    if (ok) {
      tc_fence_after();
      issue_qk<DP>(tbase, sdesc_sw128_lo(smem_u32(smem + L::kQOff)),
                   sdesc_sw128_lo(smem_u32(smem + L::kKOff)));
      tc_commit(mma_done);
      ok = mbar_wait(mma_done, 0, nullptr, status, timeout_ns);
    }
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    tc_fence_after();
    const int r = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t v[32];
      tmem_ld32(tbase + lane_off + 32 * cc, v);
      tmem_ld_wait();
      reg_fence(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        int32_t iv;
        asm("cvt.rzi.s32.f32 %0, %1;" : "=r"(iv) : "f"(__uint_as_float(v[i])));
        out[r * 128 + 32 * cc + i] = iv;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

// ------------------------------------------------ debug: PV accumulation
// O (128 x DP fp32 in TMEM) = sum over ntiles of P~_t . V~_t^T through the
// attention kernel's own PV instructions (issue_pv: kind::f8f6f4, e4m3
// operands in the 128-byte swizzled K-major shared-memory layout, K = 32
// per MMA, the first MMA overwriting).  p8: [ntiles][128 rows][128 keys],
// v8: [ntiles][DP channels][128 keys], e4m3 codes; 16-byte aligned rows.
// One CTA of 128 threads: each tile is staged by plain loads with the
// swizzle the softmax uses for P~, then one thread issues the MMAs and
// waits (bounded) for them before the next tile overwrites the operands.
template <int DP>
__global__ void __launch_bounds__(128, 1)
debug_pv_kernel(const uint8_t* p8, const uint8_t* v8, int64_t ntiles, float* out,
                uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ps = smem;                                  // 128 x 128 e4m3
  uint8_t* vs = smem + kBlockM * kBlockN;              // DP x 128 e4m3
  uint64_t* mma_done = reinterpret_cast<uint64_t*>(vs + DP * kBlockN);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  const int warp = threadIdx.x >> 5, r = threadIdx.x;
  if (r == 0) {
    mbar_init(mma_done, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  bool ok = true;
  for (int64_t t = 0; ok && t < ntiles; ++t) {
    const uint4* prow = reinterpret_cast<const uint4*>(p8 + (t * kBlockM + r) * kBlockN);
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(ps + r * 128 + ((c ^ (r & 7)) << 4)) = prow[c];
    if (r < DP) {
      const uint4* vrow = reinterpret_cast<const uint4*>(v8 + (t * DP + r) * kBlockN);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(vs + r * 128 + ((c ^ (r & 7)) << 4)) = vrow[c];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (r == 0) {
      tc_fence_after();
      issue_pv<DP>(tbase, sdesc_sw128_lo(smem_u32(ps)), sdesc_sw128_lo(smem_u32(vs)), t > 0);
      tc_commit(mma_done);
      ok = mbar_wait(mma_done, static_cast<uint32_t>(t & 1), nullptr, status, timeout_ns);
    }
    ok = __syncthreads_and(ok);                        // operands read before reuse
  }
  if (ok) {
    tc_fence_after();
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int cc = 0; cc < DP / 32; ++cc) {
      uint32_t v[32];
      tmem_ld32(tbase + lane_off + 32 * cc, v);
      tmem_ld_wait();
      reg_fence(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) out[r * DP + 32 * cc + i] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

// ------------------------------------------------ tensor-core rate
// One CTA per SM; one thread issues n back-to-back M=128 N=128 MMAs of the
// attention kernel's two kinds (kind 0: fp16 operands, K=16, as QK^T; kind
// 1: e4m3 operands, K=32, as PV) from zeroed shared-memory operands into one
// TMEM accumulator, commits once and waits (bounded).  Timed by the caller
// around the launch, it gives the tensor pipe's rate at the clock the GPU
// runs at that moment.
template <int kKind>
__global__ void __launch_bounds__(128, 1)
tc_rate_kernel(int64_t n, uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + 2 * kAtomBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  for (int i = threadIdx.x; i < 2 * kAtomBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    mbar_fence_init();
  }
  if (threadIdx.x < 32) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t a_lo = sdesc_sw128_lo(smem_u32(smem));
    const uint32_t b_lo = sdesc_sw128_lo(smem_u32(smem + kAtomBytes));
    constexpr uint32_t idesc = kKind == 0 ? make_idesc(kFmtF16, kFmtF16, kBlockM, kBlockN)
                                          : make_idesc(kFmtE4M3, kFmtE4M3, kBlockM, kBlockN);
    for (int64_t i = 0; i < n; ++i) {
      const uint32_t off = static_cast<uint32_t>(i & 3) * 2;   // 32-byte K slices of the atom
      if constexpr (kKind == 0) mma_f16_ss_lo(tbase, a_lo + off, b_lo + off, idesc, i > 0);
      else mma_f8_ss_lo(tbase, a_lo + off, b_lo + off, idesc, i > 0);
    }
    tc_commit(done);
    mbar_wait(done, 0, nullptr, status, timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

__global__ void debug_e4m3_kernel(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = static_cast<uint8_t>(pack_e4m3x2(in[i], 0.0f) & 0xFFu);
}

template <int DP, bool kV16>
cudaError_t launch_attention_t(const AttnMaps& maps, const AttnParams& p,
                               cudaStream_t st) {
  using L = Layout<DP, kV16>;
  // the shared-memory limit is a per-device attribute of the kernel (set
  // once; concurrent first calls set the same value)
  static std::atomic<bool> configured[64] = {};
  int cdev = 0;
  cudaError_t ce = cudaGetDevice(&cdev);
  if (ce != cudaSuccess) return ce;
  if (cdev < 0 || cdev >= 64) return cudaErrorInvalidDevice;
  if (!configured[cdev].load(std::memory_order_relaxed)) {
    ce = cudaFuncSetAttribute(attn_kernel<DP, kV16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (ce != cudaSuccess) return ce;
    configured[cdev].store(true, std::memory_order_relaxed);
  }
  const int64_t maxq = p.g.varlen ? p.g.max_q : p.g.Lq;
  const int64_t nqt = (maxq + kBlockM - 1) / kBlockM;      // query tiles, two per CTA
  dim3 grid(static_cast<unsigned>((nqt + 1) / 2), static_cast<unsigned>(p.g.Hq),
            static_cast<unsigned>(p.g.nseg));
  AttnParams prm = p;
  prm.flat_pairs = -1;
  if (kV16 && p.g.varlen) return cudaErrorInvalidValue;    // dense problems only
  if (!p.g.varlen && !p.causal) {
    // Uniform pairs run in waves of one CTA per SM.  When the last wave is
    // at most half full, its pairs run as single tiles instead (launched
    // last), which shortens that wave to one tile's time.
    static std::atomic<int> sms[64] = {};       // resident CTAs per device, filled once
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && sms[dev].load(std::memory_order_relaxed) == 0) {
      int n = 0, per = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, attn_kernel<DP, kV16>, kThreads,
                                                        L::kAlloc);
      if (e != cudaSuccess) return e;
      sms[dev].store(n * (per > 0 ? per : 1), std::memory_order_relaxed);
    }
    const int64_t wave = (dev >= 0 && dev < 64) ? sms[dev].load(std::memory_order_relaxed) : 0;
    const int64_t pairs = static_cast<int64_t>(grid.x) * grid.y * grid.z;
    const int64_t tail = wave > 0 ? pairs % wave : 0;
    if (tail > 0 && 2 * tail <= wave && pairs + tail < (int64_t(1) << 31)) {
      prm.flat_pairs = pairs - tail;
      grid = dim3(static_cast<unsigned>(pairs + tail), 1, 1);
    }
  }
  attn_kernel<DP, kV16><<<grid, kThreads, L::kAlloc, st>>>(maps.q, maps.k, maps.v, maps.o,
                                                            prm);
  note_launch();
  return cudaGetLastError();
}

template <int DP>
cudaError_t launch_debug_qk_t(const AttnMaps& maps, const AttnParams& p,
                              int64_t q_row0, int64_t k_row0, int32_t* out,
                              cudaStream_t st) {
  static std::atomic<bool> configured[64] = {};   // per-device kernel attribute
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(debug_qk_kernel<DP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<DP>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  debug_qk_kernel<DP><<<1, 128, Layout<DP>::kAlloc, st>>>(maps.q, maps.k, q_row0, k_row0,
                                                          out, p.status, p.timeout_ns);
  note_launch();
  return cudaGetLastError();
}

template <int DP>
cudaError_t launch_debug_pv_t(const uint8_t* p8, const uint8_t* v8, int64_t ntiles, float* out,
                              uint32_t* status, uint64_t timeout_ns, cudaStream_t st) {
  constexpr int kSmem = kBlockM * kBlockN + DP * kBlockN + 16 + 1024;
  debug_pv_kernel<DP><<<1, 128, kSmem, st>>>(p8, v8, ntiles, out, status, timeout_ns);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnMaps& maps, const AttnParams& p,
                             cudaStream_t st) {
  if (p.v16)
    return p.g.Dp == 64 ? launch_attention_t<64, true>(maps, p, st)
                        : launch_attention_t<128, true>(maps, p, st);
  return p.g.Dp == 64 ? launch_attention_t<64, false>(maps, p, st)
                      : launch_attention_t<128, false>(maps, p, st);
}

cudaError_t launch_debug_qk(const AttnMaps& maps, const AttnParams& p,
                            int64_t q_row0, int64_t k_row0, int32_t* out,
                            cudaStream_t st) {
  return p.g.Dp == 64 ? launch_debug_qk_t<64>(maps, p, q_row0, k_row0, out, st)
                      : launch_debug_qk_t<128>(maps, p, q_row0, k_row0, out, st);
}

cudaError_t launch_debug_e4m3(const float* in, uint8_t* out, int64_t n,
                              cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256 < 152 * 16 ? (n + 255) / 256 : 152 * 16;
  debug_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(in, out, n);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_tc_rate(int kind, int64_t n_mma, uint32_t* status, uint64_t timeout_ns,
                           cudaStream_t st) {
  // more shared memory than two CTAs can hold: exactly one CTA per SM
  constexpr int kSmem = 120 * 1024;
  static std::atomic<bool> configured[64] = {};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(tc_rate_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc_rate_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_relaxed);
  }
  if (kind == 0) tc_rate_kernel<0><<<sms, 128, kSmem, st>>>(n_mma, status, timeout_ns);
  else tc_rate_kernel<1><<<sms, 128, kSmem, st>>>(n_mma, status, timeout_ns);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_debug_pv(const uint8_t* p8, const uint8_t* v8, int64_t ntiles, int64_t Dp,
                            float* out, uint32_t* status, uint64_t timeout_ns,
                            cudaStream_t st) {
  return Dp == 64 ? launch_debug_pv_t<64>(p8, v8, ntiles, out, status, timeout_ns, st)
                  : launch_debug_pv_t<128>(p8, v8, ntiles, out, status, timeout_ns, st);
}

}  // namespace sage
