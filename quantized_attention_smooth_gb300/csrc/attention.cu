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
//
// GB300 mapping.  sm_103a has no INT8 tcgen05 MMA, so QK^T runs as
// kind::f16 on operands that hold the int8 codes as exact fp16 integers;
// each product is < 2^14 and a 128-term row sum < 2^21, so the fp32
// accumulator holds the exact INT32 result.  PV runs as kind::f8f6f4 (e4m3 x
// e4m3 -> fp32) with P~ read straight from tensor memory.  One CTA owns one
// (segment, query head, 128-row tile):
//   warp 4      TMA producer: Q once, then a 3-stage K/V ring
//   warp 5      tcgen05 issuer (one thread) and TMEM owner
//   warps 0-3   softmax, one row per thread (TMEM lane = row); they also
//               rescale O in TMEM and run the epilogue
// TMEM (512 columns): S0 | S1 (double-buffered S) | O (Dp) | P~0 | P~1.
// Every wait is bounded: a wait that runs out raises the workspace status
// word and an abort flag, all roles drain their in-flight copies and MMAs,
// and the CTA frees its TMEM and exits.

#include "sage_device.cuh"
#include "sage_geom.h"
#include "sage_kernels.h"

namespace sage {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
__host__ __device__ constexpr uint32_t col_s(int b) { return b ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_p(int b) { return b ? 416u : 384u; }
constexpr int kAtomBytes = 128 * 128;   // 128 rows x 128 bytes (swizzle atom column)
constexpr unsigned kFull = 0xFFFFFFFFu;

template <int DP>
struct Layout {
  static constexpr int kQBytes = kBlockM * DP * 2;
  static constexpr int kKBytes = kBlockN * DP * 2;
  static constexpr int kVBytes = DP * kBlockN;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kStages * kKBytes;
  static constexpr int kBarOff = kVOff + kStages * kVBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_done, drain
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSvOff = kMiscOff + 16;
  static constexpr int kBytes = kSvOff + DP * 4;
  // at least ~116 KB so that one CTA (and its 512 TMEM columns) owns an SM
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// S (128x128 fp32 in TMEM) = Q tile . K tile^T, K dimension DP in steps of 16.
template <int DP>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem,
                                         uint32_t k_smem) {
  constexpr uint32_t idesc = make_idesc(kFmtF16, kFmtF16, kBlockM, kBlockN);
#pragma unroll
  for (int kk = 0; kk < DP / 16; ++kk) {
    const uint32_t off = (kk / 4) * kAtomBytes + (kk % 4) * 32;
    mma_f16_ss(d_tmem, sdesc_sw128(q_smem + off), sdesc_sw128(k_smem + off),
               idesc, kk > 0 ? 1u : 0u);
  }
}

// O (128xDP fp32 in TMEM) (+)= P~ (128x128 e4m3 in TMEM) . V~ tile^T
// (V~ stored DP rows x 128 keys), K dimension 128 keys in steps of 32.
template <int DP>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem,
                                         uint32_t v_smem, bool accumulate) {
  constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, kBlockM, DP);
#pragma unroll
  for (int kk = 0; kk < kBlockN / 32; ++kk)
    mma_f8_ts(o_tmem, p_tmem + kk * 8, sdesc_sw128(v_smem + kk * 32), idesc,
              (accumulate || kk > 0) ? 1u : 0u);
}

template <int DP>
__global__ void __launch_bounds__(kThreads, 1)
attn_kernel(const __grid_constant__ CUtensorMap tm_q,
            const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = Layout<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const SegGeo& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which tile (heaviest causal tiles first)
  const int64_t s = blockIdx.z, h = blockIdx.y;
  const int64_t qt = p.causal ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;
  int64_t qstart = 0, len_q = g.Lq, kstart = 0, len_k = g.Lk;
  if (g.varlen) {
    const bool okq = seg_range(g.cu_q, s, g.total_q, g.max_q, &qstart, &len_q);
    const bool okk = seg_range(g.cu_k, s, g.total_k, g.max_k, &kstart, &len_k);
    if (!okq || !okk) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
  }
  if (qt * kBlockM >= len_q) return;
  const int64_t hk = h / (g.Hq / g.Hkv);
  int n_kv = static_cast<int>((len_k + kBlockN - 1) / kBlockN);
  if (p.causal && n_kv > qt + 1) n_kv = static_cast<int>(qt + 1);
  const int64_t q_row0 = ws_seg_base(g.varlen, s, qstart, g.Hq, g.q_head_rows) +
                         h * g.q_head_rows + qt * kBlockM;
  const int64_t k_row0 = ws_seg_base(g.varlen, s, kstart, g.Hkv, g.k_head_rows) +
                         hk * g.k_head_rows;
  const int64_t v_row0 = (g.varlen ? 0 : s * g.Hkv * DP) + hk * DP;
  const int64_t v_col0 = g.varlen ? ws_seg_base(1, s, kstart, 0, 0) : 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float* sv_cache = reinterpret_cast<float*>(smem + L::kSvOff);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kBlockM);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
  if (threadIdx.x < DP) sv_cache[threadIdx.x] = p.s_v[(s * g.Hkv + hk) * DP + threadIdx.x];
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 4) {
    // ================================================= TMA producer
    if (lane == 0) {
      mbar_expect_tx(q_full, L::kQBytes);
      for (int a = 0; a < DP / 64; ++a)
        tma_load_2d(smem + L::kQOff + a * kAtomBytes, &tm_q, a * 64,
                    static_cast<int32_t>(q_row0), q_full);
      int last = -1;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        if (j >= kStages &&
            !mbar_wait(&kv_empty[st], ((j / kStages) - 1) & 1, abort_flag,
                       p.status, p.timeout_ns))
          break;
        if (j == p.skip_kv_tile) continue;   // failure injection (tests only)
        mbar_expect_tx(&kv_full[st], L::kKBytes + L::kVBytes);
        uint8_t* kdst = smem + L::kKOff + st * L::kKBytes;
        for (int a = 0; a < DP / 64; ++a)
          tma_load_2d(kdst + a * kAtomBytes, &tm_k, a * 64,
                      static_cast<int32_t>(k_row0 + j * kBlockN), &kv_full[st]);
        tma_load_2d(smem + L::kVOff + st * L::kVBytes, &tm_v,
                    static_cast<int32_t>(v_col0 + j * kBlockN),
                    static_cast<int32_t>(v_row0), &kv_full[st]);
        last = j;
      }
      // no copy may still be in flight when the CTA exits
      mbar_wait(q_full, 0, nullptr, p.status, p.timeout_ns);
      for (int j = max(0, last - kStages + 1); j <= last; ++j)
        if (j != p.skip_kv_tile)
          mbar_wait(&kv_full[j % kStages], (j / kStages) & 1, nullptr, p.status,
                    p.timeout_ns);
    }
  } else if (warp == 5) {
    // ================================================= tcgen05 issuer
    if (lane == 0) {
      const uint32_t qa = smem_u32(smem + L::kQOff);
      const uint32_t ka0 = smem_u32(smem + L::kKOff);
      const uint32_t va0 = smem_u32(smem + L::kVOff);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, p.timeout_ns);
      bool issued = false;
      if (ok && n_kv > 0) {
        ok = mbar_wait(&kv_full[0], 0, abort_flag, p.status, p.timeout_ns);
        if (ok) {
          tc_fence_after();
          issue_qk<DP>(tbase + col_s(0), qa, ka0);
          tc_commit(&s_full[0]);
          issued = true;
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          if (j + 1 < n_kv) {
            const int st1 = (j + 1) % kStages;
            ok = mbar_wait(&kv_full[st1], ((j + 1) / kStages) & 1, abort_flag,
                           p.status, p.timeout_ns);
            if (!ok) break;
            tc_fence_after();
            issue_qk<DP>(tbase + col_s((j + 1) & 1), qa, ka0 + st1 * L::kKBytes);
            tc_commit(&s_full[(j + 1) & 1]);
          }
          ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.status,
                         p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          const int st = j % kStages;
          issue_pv<DP>(tbase + kColO, tbase + col_p(j & 1), va0 + st * L::kVBytes,
                       j > 0);
          tc_commit(&kv_empty[st]);
          tc_commit(o_done);
        }
      }
      if (issued) {   // every MMA must finish before TMEM is released
        tc_commit(drain);
        mbar_wait(drain, 0, nullptr, p.status, p.timeout_ns);
      }
    }
  } else {
    // ================================================= softmax warps 0-3
    const int r = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int64_t qi = qt * kBlockM + r;          // query index in segment
    const float sq = p.s_q[q_row0 + r];
    const float* skp = p.s_k + k_row0 / kBlockN;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      ok = mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag, p.status, p.timeout_ns);
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
      const uint32_t ts = tbase + lane_off + col_s(b);
      tmem_ld32(ts, sr[0]);
      tmem_ld32(ts + 32, sr[1]);
      tmem_ld32(ts + 64, sr[2]);
      tmem_ld32(ts + 96, sr[3]);
      tmem_ld_wait();
      reg_fence(sr[0]);
      reg_fence(sr[1]);
      reg_fence(sr[2]);
      reg_fence(sr[3]);

      const float c = (sq * skp[j]) * p.scale_log2;
      const int64_t key0 = static_cast<int64_t>(j) * kBlockN;
      const bool need_mask = (key0 + kBlockN > len_k) ||
                             (p.causal && key0 + kBlockN - 1 > qt * kBlockM);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        float xv = __uint_as_float(sr[i >> 5][i & 31]) * c;
        if (need_mask) {
          const int64_t key = key0 + i;
          if (key >= len_k || (p.causal && key > qi)) xv = -INFINITY;
        }
        sr[i >> 5][i & 31] = __float_as_uint(xv);
        mx = fmaxf(mx, xv);
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = fast_exp2(m - m_new);
      float psum = 0.0f;
      uint32_t pw[32];
#pragma unroll
      for (int w4 = 0; w4 < 32; ++w4) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 4 * w4 + e;
          pv[e] = fast_exp2(__uint_as_float(sr[i >> 5][i & 31]) - m_new);
          psum += pv[e];
        }
        pw[w4] = pack_e4m3x2(448.0f * pv[0], 448.0f * pv[1]) |
                 (pack_e4m3x2(448.0f * pv[2], 448.0f * pv[3]) << 16);
      }
      tmem_st32(tbase + lane_off + col_p(b), pw);
      tmem_st_wait();
      l = l * alpha + psum;
      if (j > 0) {
        // O holds PV of tiles < j once that PV is done; rescale it in place
        ok = mbar_wait(o_done, (j - 1) & 1, abort_flag, p.status, p.timeout_ns);
        ok = __all_sync(kFull, ok);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(kFull, alpha < 1.0f)) {
#pragma unroll 1
          for (int cc = 0; cc < DP / 32; ++cc) {
            uint32_t o[32];
            const uint32_t to = tbase + lane_off + kColO + 32 * cc;
            tmem_ld32(to, o);
            tmem_ld_wait();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(to, o);
          }
          tmem_st_wait();
        }
      }
      m = m_new;
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }

    if (ok && n_kv > 0) {
      ok = mbar_wait(o_done, (n_kv - 1) & 1, abort_flag, p.status, p.timeout_ns);
      ok = __all_sync(kFull, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.0f ? __fdiv_rn(1.0f, 448.0f * l) : 0.0f;
      const bool valid = qi < len_q;
      const int D = static_cast<int>(g.D);
      const int64_t seg_off = g.varlen ? qstart * p.out_tok_stride : s * p.out_seg_stride;
      float* orow = p.out + seg_off + h * p.out_head_stride + qi * p.out_tok_stride;
      const bool vec = (D % 4 == 0) && ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
#pragma unroll 1
      for (int cc = 0; cc < DP / 32; ++cc) {
        uint32_t o[32];
        if (n_kv > 0) {
          tmem_ld32(tbase + lane_off + kColO + 32 * cc, o);
          tmem_ld_wait();
          reg_fence(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (valid) {
          if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const int c = 32 * cc + i;
              if (c < D) {
                float4 v4;
                v4.x = __uint_as_float(o[i]) * sv_cache[c] * inv;
                v4.y = __uint_as_float(o[i + 1]) * sv_cache[c + 1] * inv;
                v4.z = __uint_as_float(o[i + 2]) * sv_cache[c + 2] * inv;
                v4.w = __uint_as_float(o[i + 3]) * sv_cache[c + 3] * inv;
                *reinterpret_cast<float4*>(orow + c) = v4;
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int c = 32 * cc + i;
              if (c < D) orow[c] = __uint_as_float(o[i]) * sv_cache[c] * inv;
            }
          }
        }
      }
    }
  }

  // ---- teardown: all roles have drained; release tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
      issue_qk<DP>(tbase, smem_u32(smem + L::kQOff), smem_u32(smem + L::kKOff));
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

__global__ void debug_e4m3_kernel(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = static_cast<uint8_t>(pack_e4m3x2(in[i], 0.0f) & 0xFFu);
}

template <int DP>
cudaError_t launch_attention_t(const AttnMaps& maps, const AttnParams& p,
                               cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(
        attn_kernel<DP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<DP>::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t maxq = p.g.varlen ? p.g.max_q : p.g.Lq;
  dim3 grid(static_cast<unsigned>((maxq + kBlockM - 1) / kBlockM),
            static_cast<unsigned>(p.g.Hq), static_cast<unsigned>(p.g.nseg));
  attn_kernel<DP><<<grid, kThreads, Layout<DP>::kAlloc, st>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

template <int DP>
cudaError_t launch_debug_qk_t(const AttnMaps& maps, const AttnParams& p,
                              int64_t q_row0, int64_t k_row0, int32_t* out,
                              cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(
        debug_qk_kernel<DP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<DP>::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  debug_qk_kernel<DP><<<1, 128, Layout<DP>::kAlloc, st>>>(maps.q, maps.k, q_row0, k_row0,
                                                          out, p.status, p.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnMaps& maps, const AttnParams& p,
                             cudaStream_t st) {
  return p.g.Dp == 64 ? launch_attention_t<64>(maps, p, st)
                      : launch_attention_t<128>(maps, p, st);
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
  return cudaGetLastError();
}

}  // namespace sage
