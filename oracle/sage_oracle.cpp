// Quantized-attention oracle: a plain, slow, CPU restatement of the
// SageAttention2-style forward pass (smoothed INT8 Q/K, FP8 P and V), of its
// FP16-PV variant (the same INT8 Q/K, fp16 P and V), and of exact fp64
// attention to measure both against.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg load this library.  The product path (the CUDA
// library under quantized_attention_smooth_gb300/) never calls it, links it or
// shares a line of code with it.
//
// Sources of the method (web pages, cited by title and section):
//  [SD]  stable-diffusion.cpp, docs "SageAttention": kernel-selection table
//        (per-thread INT8 Q/K, FP8 PV, FP32 buffer), the FP8-path paragraph
//        (smooth K, per-channel V, pad and permute V, FP32 output) and the
//        "Use" section (head_dim 1..128 zero-padded to 64/128, original
//        softmax scale kept, output cropped).
//  [OV]  "SageAttention: Quantized Attention Library" overview, "Core features"
//        (INT8 QK^T per-token/per-thread, FP8 PV, smoothing of outliers).
//  [RD]  SageAttention-RDNA4 releases, v0.4.0 "Hand-written prologue"
//        (key mean summed in fp64) and v0.2.0 (one Q scale per token).
//  [RM]  SageAttention README translation, usage section (layouts, causal,
//        GQA, different q/kv lengths).
//  [WH]  SageAttention 2.2.0 sm_120a wheel page, accuracy section (masking
//        relies on real -inf; compare against float64 attention).
//
// Readings taken where the pages are silent (each one is listed in the
// design notes of the repository):
//  * Q: one INT8 scale per token; K (after smoothing): one scale per block of
//    128 consecutive tokens of one (segment, kv-head); V: one FP8 scale per
//    channel over all tokens of one (segment, kv-head).
//  * int8 code = clamp(rint(x * (127/amax)), -127, 127), ties to even, scale
//    stored as amax/127; FP8: e4m3(v * (448/amax_c)) rounded to nearest even
//    with saturation to +-448, scale amax_c/448.  amax == 0 gives zero codes
//    and a zero scale.
//  * K mean: the exact sum of the channel over the tokens, rounded once to
//    fp64, divided by the token count in fp64, rounded to fp32; smoothing is
//    the fp32 subtraction k - mean.
//  * Online softmax over 128-key tiles in base 2: x = S_int * ((s_q*s_k) *
//    (sm_scale*log2 e)), exact running max, P = exp2(x - m), the row sum l
//    accumulates the unquantized fp32 P, P~ = e4m3(448 * P).
//  * Output = O * s_v[c] / (448 * l) for the first D channels (cropped);
//    a row with no visible key (l == 0) outputs zeros.
//  * Causal mask, top-left aligned: key j is visible to query i iff j <= i.
//  * GQA: query head h reads kv head h / (Hq / Hkv).
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fPIC -shared -pthread
// (no fast-math: every fp32 operation above is one IEEE round-to-nearest op).

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kKeyBlock = 128;          // K quantisation block and softmax tile
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kFp8Max = 448.0f;       // largest finite e4m3 magnitude
constexpr float kInt8Max = 127.0f;

// ---------------------------------------------------------------- decoding
float decode_f16(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  float mag;
  if (e == 0) mag = std::ldexp(static_cast<float>(m), -24);
  else if (e == 31) mag = m ? NAN : INFINITY;
  else mag = std::ldexp(static_cast<float>(m + 1024), e - 25);
  return s ? -mag : mag;
}

float decode_bf16(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

float decode_in(uint16_t bits, int dtype) {
  return dtype == 0 ? decode_f16(bits) : decode_bf16(bits);
}

// ------------------------------------------------------------------ e4m3
// e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
// S.1111.111 is NaN, largest finite 1.75 * 2^8 = 448, subnormals m * 2^-9.
float e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  float mag = (e == 0) ? std::ldexp(static_cast<float>(m), -9)
                       : std::ldexp(static_cast<float>(8 + m), e - 10);
  return s ? -mag : mag;
}

// Round to the nearest e4m3 value, ties to the even code, saturating at 448.
uint8_t e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  float a = std::fabs(x);
  if (a >= kFp8Max) return sign | 0x7E;
  if (a < 0.015625f) {                       // below 2^-6: subnormal grid 2^-9
    float q = std::nearbyint(a * 512.0f);    // 0..8; 8 is the first normal
    return sign | static_cast<uint8_t>(q);
  }
  int E;
  float f = std::frexp(a, &E);               // a = f * 2^E, f in [0.5, 1)
  int e = E - 1;                             // a = (2f) * 2^e, 2f in [1, 2)
  float q = std::nearbyint((2.0f * f - 1.0f) * 8.0f);
  int qi = static_cast<int>(q);
  if (qi == 8) { qi = 0; e += 1; }
  int code = ((e + 7) << 3) | qi;
  if (code > 0x7E) code = 0x7E;
  return sign | static_cast<uint8_t>(code);
}

// ------------------------------------------------------------------ fp16
// IEEE binary16: sign, 5 exponent bits (bias 15), 10 mantissa bits; largest
// finite 65504, subnormals m * 2^-24.  Round to nearest, ties to even;
// magnitudes from 65520 (the tie above 65504) round to infinity.
uint16_t fp16_encode(float x) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  if (std::isnan(x)) return 0x7E00;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 65520.0) return sign | 0x7C00;
  if (a == 0.0) return sign;
  int E;
  std::frexp(a, &E);                       // a = f * 2^E, f in [0.5, 1)
  const int e = std::max(E - 1, -14);      // binade exponent, subnormals below 2^-14
  const double ulp = std::ldexp(1.0, e - 10);
  const double r = std::nearbyint(a / ulp);   // exact quotient, ties to even
  const double v = r * ulp;
  if (v >= 65520.0) return sign | 0x7C00;
  if (v < std::ldexp(1.0, -14))            // subnormal: m * 2^-24
    return sign | static_cast<uint16_t>(std::ldexp(v, 24));
  int Ev;
  const double f = std::frexp(v, &Ev);     // v = f * 2^Ev
  const int biased = Ev - 1 + 15;
  const uint16_t mant = static_cast<uint16_t>((f * 2.0 - 1.0) * 1024.0);
  return sign | static_cast<uint16_t>(biased << 10) | mant;
}

// ------------------------------------------------------------ quantisers
int8_t int8_code(float x, float inv) {
  float r = std::nearbyint(x * inv);
  if (r > kInt8Max) r = kInt8Max;
  if (r < -kInt8Max) r = -kInt8Max;
  return static_cast<int8_t>(r);
}

// Exact sum of n fp32 values (stride apart), rounded once to fp64.
// Each nonzero value is M * 2^e with |M| < 2^24; the significands are added
// in 128-bit integers aligned to the smallest exponent.  Returns false if the
// span of exponents does not fit the accumulator (never for fp16 inputs).
bool exact_sum(const float* x, int64_t n, int64_t stride, double* out) {
  int emin = INT_MAX, emax = INT_MIN;
  for (int64_t t = 0; t < n; ++t) {
    float v = x[t * stride];
    if (v == 0.0f) continue;
    int E;
    std::frexp(v, &E);
    emin = std::min(emin, E - 24);
    emax = std::max(emax, E - 24);
  }
  if (emin == INT_MAX) { *out = 0.0; return true; }
  int count_bits = 0;
  while ((int64_t(1) << count_bits) < n + 1) ++count_bits;
  if ((emax - emin) + 25 + count_bits > 126) return false;
  __int128 acc = 0;
  for (int64_t t = 0; t < n; ++t) {
    float v = x[t * stride];
    if (v == 0.0f) continue;
    int E;
    float f = std::frexp(v, &E);
    int64_t M = static_cast<int64_t>(std::ldexp(f, 24));  // exact integer
    acc += static_cast<__int128>(M) << ((E - 24) - emin);
  }
  *out = std::ldexp(static_cast<double>(acc), emin);
  return true;
}

int64_t padded_dim(int64_t D) { return D <= 64 ? 64 : 128; }

template <class Fn>
void parallel_for(int64_t n, int nthreads, Fn fn) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  nthreads = static_cast<int>(std::min<int64_t>(nthreads, n));
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w) {
    pool.emplace_back([=] {
      for (int64_t i = w; i < n; i += nthreads) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int oracle_padded_dim(int64_t D) { return static_cast<int>(padded_dim(D)); }

uint8_t oracle_e4m3_encode(float x) { return e4m3_encode(x); }
uint16_t oracle_fp16_encode(float x) { return fp16_encode(x); }
float oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }

void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  const int64_t block = 1 << 16;
  parallel_for((n + block - 1) / block, 0, [&](int64_t b) {
    const int64_t end = std::min(n, (b + 1) * block);
    for (int64_t i = b * block; i < end; ++i) out[i] = e4m3_encode(x[i]);
  });
}

// Exact mean of n values: fp32(fp64(exact sum) / n).  Returns 0 on success.
int oracle_exact_mean(const float* x, int64_t n, float* mean) {
  double s;
  if (!exact_sum(x, n, 1, &s)) return 1;
  *mean = n > 0 ? static_cast<float>(s / static_cast<double>(n)) : 0.0f;
  return 0;
}

// Prologue for one segment (one batch entry or one packed sequence).
// Inputs are raw fp16 (dtype 0) or bf16 (dtype 1) bits, [H][L][D] contiguous.
// Outputs, all for the padded head dim Dp = 64 (D <= 64) or 128:
//   q8 [Hq][Lq][Dp], s_q [Hq][Lq]
//   k_mean [Hkv][Dp], k8 [Hkv][Lk][Dp], s_k [Hkv][ceil(Lk/128)]
//   v_amax [Hkv][Dp], s_v [Hkv][Dp], v8 (e4m3 codes) [Hkv][Lk][Dp]
// Returns 0 on success, 1 if an exact key sum does not fit the accumulator,
// 2 on a bad argument.
int oracle_prologue(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    int dtype, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                    int64_t D, int8_t* q8, float* s_q, float* k_mean,
                    int8_t* k8, float* s_k, float* v_amax, float* s_v,
                    uint8_t* v8) {
  if (D < 1 || D > 128 || Hq < 1 || Hkv < 1 || Hq % Hkv) return 2;
  const int64_t Dp = padded_dim(D);

  // a) head-dim padding with zeros, decoded to fp32 (exact)
  std::vector<float> qp(Hq * Lq * Dp, 0.0f), kp(Hkv * Lk * Dp, 0.0f),
      vp(Hkv * Lk * Dp, 0.0f);
  for (int64_t h = 0; h < Hq; ++h)
    for (int64_t t = 0; t < Lq; ++t)
      for (int64_t c = 0; c < D; ++c)
        qp[(h * Lq + t) * Dp + c] = decode_in(q[(h * Lq + t) * D + c], dtype);
  for (int64_t h = 0; h < Hkv; ++h)
    for (int64_t t = 0; t < Lk; ++t)
      for (int64_t c = 0; c < D; ++c) {
        kp[(h * Lk + t) * Dp + c] = decode_in(k[(h * Lk + t) * D + c], dtype);
        vp[(h * Lk + t) * Dp + c] = decode_in(v[(h * Lk + t) * D + c], dtype);
      }

  // b) K column means over all tokens of the head (smoothing, [SD], [RD])
  for (int64_t h = 0; h < Hkv; ++h)
    for (int64_t c = 0; c < Dp; ++c) {
      double s;
      if (!exact_sum(&kp[h * Lk * Dp + c], Lk, Dp, &s)) return 1;
      k_mean[h * Dp + c] =
          Lk > 0 ? static_cast<float>(s / static_cast<double>(Lk)) : 0.0f;
    }

  // c) V column absolute maxima
  for (int64_t h = 0; h < Hkv; ++h)
    for (int64_t c = 0; c < Dp; ++c) {
      float a = 0.0f;
      for (int64_t t = 0; t < Lk; ++t)
        a = std::max(a, std::fabs(vp[(h * Lk + t) * Dp + c]));
      v_amax[h * Dp + c] = a;
    }

  // d) Q: one int8 scale per token
  for (int64_t h = 0; h < Hq; ++h)
    for (int64_t t = 0; t < Lq; ++t) {
      const float* row = &qp[(h * Lq + t) * Dp];
      float a = 0.0f;
      for (int64_t c = 0; c < Dp; ++c) a = std::max(a, std::fabs(row[c]));
      float inv = a > 0.0f ? kInt8Max / a : 0.0f;
      for (int64_t c = 0; c < Dp; ++c)
        q8[(h * Lq + t) * Dp + c] = int8_code(row[c], inv);
      s_q[h * Lq + t] = a / kInt8Max;
    }

  // e) smoothed K: one int8 scale per block of 128 tokens
  const int64_t nkb = (Lk + kKeyBlock - 1) / kKeyBlock;
  std::vector<float> khat(Dp * kKeyBlock);
  for (int64_t h = 0; h < Hkv; ++h)
    for (int64_t b = 0; b < nkb; ++b) {
      int64_t t0 = b * kKeyBlock, t1 = std::min(Lk, t0 + kKeyBlock);
      float a = 0.0f;
      for (int64_t t = t0; t < t1; ++t)
        for (int64_t c = 0; c < Dp; ++c) {
          float x = kp[(h * Lk + t) * Dp + c] - k_mean[h * Dp + c];
          khat[(t - t0) * Dp + c] = x;
          a = std::max(a, std::fabs(x));
        }
      float inv = a > 0.0f ? kInt8Max / a : 0.0f;
      for (int64_t t = t0; t < t1; ++t)
        for (int64_t c = 0; c < Dp; ++c)
          k8[(h * Lk + t) * Dp + c] = int8_code(khat[(t - t0) * Dp + c], inv);
      s_k[h * nkb + b] = a / kInt8Max;
    }

  // f) V: one e4m3 scale per channel, largest magnitude mapped to 448
  for (int64_t h = 0; h < Hkv; ++h)
    for (int64_t c = 0; c < Dp; ++c) {
      float a = v_amax[h * Dp + c];
      float inv = a > 0.0f ? kFp8Max / a : 0.0f;
      for (int64_t t = 0; t < Lk; ++t)
        v8[(h * Lk + t) * Dp + c] = e4m3_encode(vp[(h * Lk + t) * Dp + c] * inv);
      s_v[h * Dp + c] = a / kFp8Max;
    }
  return 0;
}

// Quantised attention for one segment, rows [r0, r1) of query heads
// [h0, h1), from the prologue's outputs.  out is [Hq][Lq][D] fp32; only the
// requested rows are written.  sm_scale is the softmax scale on the natural
// logits (the caller resolves its default).  nthreads <= 0: all cores.
int oracle_attn(const int8_t* q8, const float* s_q, const int8_t* k8,
                const float* s_k, const uint8_t* v8, const float* s_v,
                int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D,
                int causal, float sm_scale, int64_t h0, int64_t h1,
                int64_t r0, int64_t r1, float* out, int nthreads) {
  if (D < 1 || D > 128 || Hq % Hkv) return 2;
  const int64_t Dp = padded_dim(D);
  const int64_t group = Hq / Hkv;
  const int64_t nkb = (Lk + kKeyBlock - 1) / kKeyBlock;
  const float scale_log2 = sm_scale * kLog2e;
  const int64_t nrows = r1 - r0;
  const int64_t items = (h1 - h0) * nrows;

  parallel_for(items, nthreads, [&](int64_t it) {
    const int64_t h = h0 + it / nrows;
    const int64_t i = r0 + it % nrows;
    const int64_t hk = h / group;
    const int8_t* qi = &q8[(h * Lq + i) * Dp];
    const float sq = s_q[h * Lq + i];
    float m = -INFINITY, l = 0.0f;
    std::vector<float> O(Dp, 0.0f), x(kKeyBlock), acc(Dp);
    std::vector<uint8_t> pt(kKeyBlock);
    for (int64_t b = 0; b < nkb; ++b) {
      const int64_t j0 = b * kKeyBlock, j1 = std::min(Lk, j0 + kKeyBlock);
      const float c = (sq * s_k[hk * nkb + b]) * scale_log2;   // dequant factor
      float mt = -INFINITY;
      bool visible = false;
      for (int64_t j = j0; j < j1; ++j) {
        if (causal && j > i) { x[j - j0] = -INFINITY; continue; }
        const int8_t* kj = &k8[(hk * Lk + j) * Dp];
        int32_t S = 0;                                          // INT32 QK^T
        for (int64_t d = 0; d < Dp; ++d)
          S += static_cast<int32_t>(qi[d]) * static_cast<int32_t>(kj[d]);
        x[j - j0] = static_cast<float>(S) * c;
        mt = std::max(mt, x[j - j0]);
        visible = true;
      }
      if (!visible) continue;                                   // fully masked
      const float m_new = std::max(m, mt);
      const float alpha = std::exp2(m - m_new);                 // 0 on first tile
      float psum = 0.0f;
      for (int64_t j = j0; j < j1; ++j) {
        float p = std::exp2(x[j - j0] - m_new);
        psum += p;
        pt[j - j0] = e4m3_encode(kFp8Max * p);
      }
      l = l * alpha + psum;
      for (int64_t d = 0; d < Dp; ++d) acc[d] = 0.0f;
      for (int64_t j = j0; j < j1; ++j) {
        const float pj = e4m3_value(pt[j - j0]);
        const uint8_t* vj = &v8[(hk * Lk + j) * Dp];
        for (int64_t d = 0; d < Dp; ++d) acc[d] += pj * e4m3_value(vj[d]);
      }
      for (int64_t d = 0; d < Dp; ++d) O[d] = O[d] * alpha + acc[d];
      m = m_new;
    }
    float* o = &out[(h * Lq + i) * D];
    for (int64_t d = 0; d < D; ++d)
      o[d] = l > 0.0f ? (O[d] * s_v[hk * Dp + d]) / (kFp8Max * l) : 0.0f;
  });
  return 0;
}

// V for the FP16-PV variant ([OV] API list: "INT8 QK^T, FP16 PV"): each
// input value rounded to fp16 (exact for fp16 inputs), channels padded to Dp
// with zeros.  v16 is [Hkv][Lk][Dp] binary16 bits.
int oracle_v16(const uint16_t* v, int dtype, int64_t Hkv, int64_t Lk, int64_t D,
               uint16_t* v16) {
  if (D < 1 || D > 128) return 2;
  const int64_t Dp = padded_dim(D);
  for (int64_t h = 0; h < Hkv; ++h)
    for (int64_t t = 0; t < Lk; ++t)
      for (int64_t c = 0; c < Dp; ++c)
        v16[(h * Lk + t) * Dp + c] =
            c < D ? fp16_encode(decode_in(v[(h * Lk + t) * D + c], dtype)) : 0;
  return 0;
}

// FP16-PV variant of the quantised attention: the same INT8 QK^T, dequant,
// masking and online softmax as oracle_attn, then P~ = fp16(P) (no 448
// scaling), O accumulates P~ * V16 in fp32 per 128-key tile, and the output
// is O / l for the first D channels (a row with no visible key outputs zeros).
int oracle_attn_pv16(const int8_t* q8, const float* s_q, const int8_t* k8,
                     const float* s_k, const uint16_t* v16, int64_t Hq, int64_t Hkv,
                     int64_t Lq, int64_t Lk, int64_t D, int causal, float sm_scale,
                     int64_t h0, int64_t h1, int64_t r0, int64_t r1, float* out,
                     int nthreads) {
  if (D < 1 || D > 128 || Hq % Hkv) return 2;
  const int64_t Dp = padded_dim(D);
  const int64_t group = Hq / Hkv;
  const int64_t nkb = (Lk + kKeyBlock - 1) / kKeyBlock;
  const float scale_log2 = sm_scale * kLog2e;
  const int64_t nrows = r1 - r0;
  parallel_for((h1 - h0) * nrows, nthreads, [&](int64_t it) {
    const int64_t h = h0 + it / nrows;
    const int64_t i = r0 + it % nrows;
    const int64_t hk = h / group;
    const int8_t* qi = &q8[(h * Lq + i) * Dp];
    const float sq = s_q[h * Lq + i];
    float m = -INFINITY, l = 0.0f;
    std::vector<float> O(Dp, 0.0f), x(kKeyBlock), acc(Dp), pt(kKeyBlock);
    for (int64_t b = 0; b < nkb; ++b) {
      const int64_t j0 = b * kKeyBlock, j1 = std::min(Lk, j0 + kKeyBlock);
      const float c = (sq * s_k[hk * nkb + b]) * scale_log2;
      float mt = -INFINITY;
      bool visible = false;
      for (int64_t j = j0; j < j1; ++j) {
        if (causal && j > i) { x[j - j0] = -INFINITY; continue; }
        const int8_t* kj = &k8[(hk * Lk + j) * Dp];
        int32_t S = 0;
        for (int64_t d = 0; d < Dp; ++d)
          S += static_cast<int32_t>(qi[d]) * static_cast<int32_t>(kj[d]);
        x[j - j0] = static_cast<float>(S) * c;
        mt = std::max(mt, x[j - j0]);
        visible = true;
      }
      if (!visible) continue;
      const float m_new = std::max(m, mt);
      const float alpha = std::exp2(m - m_new);
      float psum = 0.0f;
      for (int64_t j = j0; j < j1; ++j) {
        const float p = std::exp2(x[j - j0] - m_new);
        psum += p;
        pt[j - j0] = decode_f16(fp16_encode(p));
      }
      l = l * alpha + psum;
      for (int64_t d = 0; d < Dp; ++d) acc[d] = 0.0f;
      for (int64_t j = j0; j < j1; ++j) {
        const uint16_t* vj = &v16[(hk * Lk + j) * Dp];
        for (int64_t d = 0; d < Dp; ++d) acc[d] += pt[j - j0] * decode_f16(vj[d]);
      }
      for (int64_t d = 0; d < Dp; ++d) O[d] = O[d] * alpha + acc[d];
      m = m_new;
    }
    float* o = &out[(h * Lq + i) * D];
    for (int64_t d = 0; d < D; ++d) o[d] = l > 0.0f ? O[d] / l : 0.0f;
  });
  return 0;
}

// Exact (unquantised) attention in fp64 from the raw inputs of one segment:
// softmax(q k^T * sm_scale) v with the same masking and head map.
int oracle_attn_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      int dtype, int64_t Hq, int64_t Hkv, int64_t Lq,
                      int64_t Lk, int64_t D, int causal, double sm_scale,
                      int64_t h0, int64_t h1, int64_t r0, int64_t r1,
                      double* out, int nthreads) {
  if (Hq % Hkv) return 2;
  const int64_t group = Hq / Hkv;
  const int64_t nrows = r1 - r0;
  parallel_for((h1 - h0) * nrows, nthreads, [&](int64_t it) {
    const int64_t h = h0 + it / nrows;
    const int64_t i = r0 + it % nrows;
    const int64_t hk = h / group;
    std::vector<double> s(Lk), qi(D), o(D, 0.0);
    for (int64_t d = 0; d < D; ++d) qi[d] = decode_in(q[(h * Lq + i) * D + d], dtype);
    double mx = -INFINITY;
    const int64_t jend = causal ? std::min<int64_t>(Lk, i + 1) : Lk;
    for (int64_t j = 0; j < jend; ++j) {
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d)
        acc += qi[d] * static_cast<double>(decode_in(k[(hk * Lk + j) * D + d], dtype));
      s[j] = acc * sm_scale;
      mx = std::max(mx, s[j]);
    }
    double den = 0.0;
    for (int64_t j = 0; j < jend; ++j) {
      double w = std::exp(s[j] - mx);
      den += w;
      for (int64_t d = 0; d < D; ++d)
        o[d] += w * static_cast<double>(decode_in(v[(hk * Lk + j) * D + d], dtype));
    }
    for (int64_t d = 0; d < D; ++d)
      out[(h * Lq + i) * D + d] = den > 0.0 ? o[d] / den : 0.0;
  });
  return 0;
}

}  // extern "C"
