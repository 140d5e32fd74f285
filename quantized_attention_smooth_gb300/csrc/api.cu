// C ABI of the library: argument validation, workspace layout, TMA tensor
// maps and kernel launches.  The library allocates nothing and never
// synchronises the host (sage_device_status excepted, which exists to read
// the device status word back).

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "sage.h"
#include "sage_geom.h"
#include "sage_kernels.h"

using namespace sage;

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void sage::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
uint64_t sage::launch_count() { return g_launches.load(std::memory_order_relaxed); }

namespace {

thread_local std::string g_last_error;
std::atomic<int> g_skip_kv_tile{-1};
std::atomic<int> g_prologue_launches{0};
std::atomic<unsigned long long> g_timeout_ns{0};
// attention launches the failure-injection hook still applies to (-1: all)
std::atomic<int> g_fault_launches{-1};
std::atomic<int> g_host_fail_chunk{-1};
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;   // 1 s

// Bound of every device-side wait of the next launches.
uint64_t wait_timeout_ns() {
  const unsigned long long t = g_timeout_ns.load();
  return t ? t : kDefaultTimeoutNs;
}

sage_status fail(sage_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

sage_status ok() {
  g_last_error.clear();
  return SAGE_OK;
}

sage_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SAGE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t padded_dim(int64_t D) { return D <= 64 ? 64 : 128; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of every workspace buffer.
struct WsLayout {
  size_t status, ksum, vmax, sync, zero_end, k_mean, s_v, v_inv, s_q, s_k, q16, k16,
      v8, total;
};

WsLayout ws_layout(const SegGeo& g) {
  const int64_t nstat = g.nseg * g.Hkv * g.Dp;
  const int64_t q_rows = (g.varlen ? 1 : g.nseg) * g.Hq * g.q_head_rows;
  const int64_t k_rows = (g.varlen ? 1 : g.nseg) * g.Hkv * g.k_head_rows;
  const int64_t v_rows = (g.varlen ? 1 : g.nseg) * g.Hkv * g.Dp;
  WsLayout w{};
  size_t o = 0;
  w.status = o; o += 256;
  w.ksum = o; o = align256(o + nstat * 8);
  w.vmax = o; o = align256(o + nstat * 4);
  w.sync = o; o = align256(o + 8 * 64 * 4);   // two launches' list counters
  // means and scales start at zero: a segment without keys keeps them so
  w.k_mean = o; o = align256(o + nstat * 4);
  w.s_v = o; o = align256(o + nstat * 4);
  w.v_inv = o; o = align256(o + nstat * 4);
  w.zero_end = o;
  w.s_q = o; o = align256(o + q_rows * 4);
  w.s_k = o; o = align256(o + (k_rows / 128) * 4);
  w.q16 = o; o = align256(o + q_rows * g.Dp * 2);
  w.k16 = o; o = align256(o + k_rows * g.Dp * 2);
  w.v8 = o; o = align256(o + v_rows * g.v_cols * 2);   // e4m3, or fp16 (FP16-PV)
  w.total = o;
  return w;
}

bool check_dims(int64_t Hq, int64_t Hkv, int64_t D, sage_status* st) {
  if (D < 1 || D > 128) {
    *st = fail(SAGE_ERR_UNSUPPORTED, "head_dim D=%lld outside 1..128", (long long)D);
    return false;
  }
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) {
    *st = fail(SAGE_ERR_INVALID_ARG, "Hq=%lld must be a positive multiple of Hkv=%lld",
               (long long)Hq, (long long)Hkv);
    return false;
  }
  return true;
}

// Geometry of a dense call.
SegGeo dense_geo(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                 int64_t D, int dtype, int layout) {
  SegGeo g{};
  g.nseg = B; g.Hq = Hq; g.Hkv = Hkv; g.Lq = Lq; g.Lk = Lk; g.D = D;
  g.Dp = padded_dim(D);
  g.dtype = dtype; g.varlen = 0;
  g.max_q = static_cast<int32_t>(Lq > INT32_MAX ? INT32_MAX : Lq);
  g.max_k = static_cast<int32_t>(Lk > INT32_MAX ? INT32_MAX : Lk);
  if (layout == SAGE_HND) {
    g.q_seg_stride = Hq * Lq * D; g.q_head_stride = Lq * D; g.q_tok_stride = D;
    g.k_seg_stride = Hkv * Lk * D; g.k_head_stride = Lk * D; g.k_tok_stride = D;
  } else {
    g.q_seg_stride = Lq * Hq * D; g.q_head_stride = D; g.q_tok_stride = Hq * D;
    g.k_seg_stride = Lk * Hkv * D; g.k_head_stride = D; g.k_tok_stride = Hkv * D;
  }
  g.q_head_rows = round_up(Lq, 128);
  g.k_head_rows = round_up(Lk, 128);
  g.v_cols = g.k_head_rows;
  return g;
}

// Dense geometry of strided views: q_strides / kv_strides are {batch, head,
// token} in elements (channel stride 1).  Refuses, with the reason, views
// the prologue cannot read.
sage_status strided_geo(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D,
                        int dtype, const int64_t* qs, const int64_t* kvs, SegGeo* g) {
  if (qs == nullptr || kvs == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "q_strides and kv_strides must be host int64[3] arrays");
  for (int i = 0; i < 3; ++i) {
    if (qs[i] <= 0 || kvs[i] <= 0)
      return fail(SAGE_ERR_UNSUPPORTED,
                  "strided views need positive strides (q {%lld, %lld, %lld}, k/v {%lld, "
                  "%lld, %lld}); zero (broadcast) or negative strides are not served",
                  (long long)qs[0], (long long)qs[1], (long long)qs[2], (long long)kvs[0],
                  (long long)kvs[1], (long long)kvs[2]);
    if (qs[i] >= (int64_t(1) << 39) || kvs[i] >= (int64_t(1) << 39))
      return fail(SAGE_ERR_UNSUPPORTED,
                  "a stride of 2^39 elements or more is not served (tensor-copy limit)");
  }
  *g = dense_geo(B, Hq, Hkv, Lq, Lk, D, dtype, SAGE_HND);
  g->strided = 1;
  g->q_seg_stride = qs[0]; g->q_head_stride = qs[1]; g->q_tok_stride = qs[2];
  g->k_seg_stride = kvs[0]; g->k_head_stride = kvs[1]; g->k_tok_stride = kvs[2];
  return SAGE_OK;
}

SegGeo varlen_geo(int64_t nseq, int64_t total_q, int64_t total_k, int max_q,
                  int max_k, int64_t Hq, int64_t Hkv, int64_t D, int dtype,
                  const int32_t* cu_q, const int32_t* cu_k) {
  SegGeo g{};
  g.nseg = nseq; g.Hq = Hq; g.Hkv = Hkv; g.Lq = 0; g.Lk = 0; g.D = D;
  g.Dp = padded_dim(D);
  g.dtype = dtype; g.varlen = 1;
  g.cu_q = cu_q; g.cu_k = cu_k;
  g.total_q = total_q; g.total_k = total_k;
  g.max_q = max_q; g.max_k = max_k;
  g.q_seg_stride = 0; g.q_head_stride = D; g.q_tok_stride = Hq * D;
  g.k_seg_stride = 0; g.k_head_stride = D; g.k_tok_stride = Hkv * D;
  g.q_head_rows = 128 * (nseq + total_q / 128);
  g.k_head_rows = 128 * (nseq + total_k / 128);
  g.v_cols = g.k_head_rows;
  return g;
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

sage_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(SAGE_ERR_UNSUPPORTED,
                "device %d is sm_%d%d; this build runs on sm_103 (GB300) only", dev,
                major, minor);
  return SAGE_OK;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn();

}  // namespace

bool sage::encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes,
                        const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return fn(map, dt, rank, base, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

namespace {

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, void* base,
               uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {row_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_tiled(map, dt, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

sage_status make_maps(const sage_quantized* qt, AttnMaps* maps) {
  if (!encode_2d(&maps->q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qt->q16, qt->Dp, qt->q_rows,
                 qt->Dp * 2, 64, 128) ||
      !encode_2d(&maps->k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qt->k16, qt->Dp, qt->k_rows,
                 qt->Dp * 2, 64, 128) ||
      !(qt->v_fp16
            ? encode_2d(&maps->v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qt->v8, qt->v_cols,
                        qt->v_rows, qt->v_cols * 2, 64, static_cast<uint32_t>(qt->Dp))
            : encode_2d(&maps->v, CU_TENSOR_MAP_DATA_TYPE_UINT8, qt->v8, qt->v_cols,
                        qt->v_rows, qt->v_cols, 128, static_cast<uint32_t>(qt->Dp))))
    return fail(SAGE_ERR_CUDA, "cuTensorMapEncodeTiled failed or unavailable");
  return SAGE_OK;
}

SegGeo geo_of(const sage_quantized* qt) {
  SegGeo g{};
  g.nseg = qt->nseg; g.Hq = qt->Hq; g.Hkv = qt->Hkv; g.Lq = qt->Lq; g.Lk = qt->Lk;
  g.D = qt->D; g.Dp = qt->Dp; g.dtype = qt->dtype; g.varlen = qt->varlen;
  g.cu_q = qt->cu_q; g.cu_k = qt->cu_k; g.total_q = qt->total_q; g.total_k = qt->total_k;
  g.max_q = qt->max_q; g.max_k = qt->max_k;
  g.q_head_rows = qt->q_head_rows; g.k_head_rows = qt->k_head_rows; g.v_cols = qt->v_cols;
  return g;
}

void fill_quantized(const SegGeo& g, const WsLayout& w, uint8_t* ws, sage_quantized* qt) {
  std::memset(qt, 0, sizeof(*qt));
  qt->nseg = g.nseg; qt->Hq = g.Hq; qt->Hkv = g.Hkv; qt->Lq = g.Lq; qt->Lk = g.Lk;
  qt->D = g.D; qt->Dp = g.Dp; qt->dtype = g.dtype; qt->varlen = g.varlen;
  qt->total_q = g.total_q; qt->total_k = g.total_k; qt->max_q = g.max_q; qt->max_k = g.max_k;
  qt->q_head_rows = g.q_head_rows; qt->k_head_rows = g.k_head_rows;
  qt->q_rows = (g.varlen ? 1 : g.nseg) * g.Hq * g.q_head_rows;
  qt->k_rows = (g.varlen ? 1 : g.nseg) * g.Hkv * g.k_head_rows;
  qt->v_rows = (g.varlen ? 1 : g.nseg) * g.Hkv * g.Dp;
  qt->v_cols = g.v_cols;
  qt->cu_q = g.cu_q; qt->cu_k = g.cu_k;
  qt->q16 = ws + w.q16; qt->k16 = ws + w.k16; qt->v8 = ws + w.v8;
  qt->s_q = reinterpret_cast<float*>(ws + w.s_q);
  qt->s_k = reinterpret_cast<float*>(ws + w.s_k);
  qt->s_v = reinterpret_cast<float*>(ws + w.s_v);
  qt->k_mean = reinterpret_cast<float*>(ws + w.k_mean);
  qt->stats = ws + w.ksum;
  qt->status = reinterpret_cast<uint32_t*>(ws + w.status);
}

// Shared tail of both prologue entry points (arguments already validated).
// keep_status: leave the device status word as it is (the host-buffer
// pipeline's later chunks, so that a failure of an earlier chunk stays
// visible to sage_device_status); otherwise it is cleared with the rest.
sage_status run_prologue(const SegGeo& g, const void* q, const void* k, const void* v,
                         void* ws, size_t ws_bytes, sage_quantized* qt,
                         cudaStream_t st, bool v16 = false, bool keep_status = false) {
  const WsLayout w = ws_layout(g);
  if (ws == nullptr || !aligned(ws, 256))
    return fail(SAGE_ERR_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
  if (ws_bytes < w.total)
    return fail(SAGE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  if (g.q_head_rows * g.Hq * (g.varlen ? 1 : g.nseg) >= (int64_t(1) << 31) ||
      g.k_head_rows * g.Hkv * (g.varlen ? 1 : g.nseg) >= (int64_t(1) << 31) ||
      g.v_cols >= (int64_t(1) << 31))
    return fail(SAGE_ERR_UNSUPPORTED, "problem exceeds 2^31 workspace rows");
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  fill_quantized(g, w, wsb, qt);
  qt->v_fp16 = v16 ? 1 : 0;
  const size_t zero_from = keep_status ? w.ksum : 0;   // the status word lies below ksum
  cudaError_t e = cudaMemsetAsync(wsb + zero_from, 0, w.zero_end - zero_from, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  PrologueBuffers b{};
  b.q = static_cast<const uint16_t*>(q);
  b.k = static_cast<const uint16_t*>(k);
  b.v = static_cast<const uint16_t*>(v);
  b.q16 = reinterpret_cast<uint16_t*>(wsb + w.q16);
  b.k16 = reinterpret_cast<uint16_t*>(wsb + w.k16);
  b.v8 = wsb + w.v8;
  b.s_q = reinterpret_cast<float*>(wsb + w.s_q);
  b.s_k = reinterpret_cast<float*>(wsb + w.s_k);
  b.s_v = reinterpret_cast<float*>(wsb + w.s_v);
  b.k_mean = reinterpret_cast<float*>(wsb + w.k_mean);
  b.v_inv = reinterpret_cast<float*>(wsb + w.v_inv);
  b.ksum = wsb + w.ksum;
  b.vmax = reinterpret_cast<uint32_t*>(wsb + w.vmax);
  b.sync = reinterpret_cast<unsigned int*>(wsb + w.sync);
  b.timeout_ns = wait_timeout_ns();
  b.status = reinterpret_cast<uint32_t*>(wsb + w.status);
  // tensor copies need 16-byte aligned rows: base, channel count and every
  // stride (for views) in whole 16-byte units
  const bool vec = (g.D % 8 == 0) && aligned(q, 16) && aligned(k, 16) && aligned(v, 16) &&
                   g.q_seg_stride % 8 == 0 && g.q_head_stride % 8 == 0 &&
                   g.q_tok_stride % 8 == 0 && g.k_seg_stride % 8 == 0 &&
                   g.k_head_stride % 8 == 0 && g.k_tok_stride % 8 == 0;
  b.v16 = v16 ? 1 : 0;
  b.launches = g_prologue_launches.load();
  e = launch_prologue(g, b, vec, st);
  if (e != cudaSuccess) return cuda_fail(e, "prologue launch");
  return ok();
}

sage_status check_common(const void* q, const void* k, const void* v, int dtype) {
  if (dtype != SAGE_F16 && dtype != SAGE_BF16)
    return fail(SAGE_ERR_INVALID_ARG, "dtype %d is neither SAGE_F16 nor SAGE_BF16", dtype);
  if (q == nullptr || k == nullptr || v == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "q, k and v must be non-null device pointers");
  if (!aligned(q, 2) || !aligned(k, 2) || !aligned(v, 2))
    return fail(SAGE_ERR_INVALID_ARG, "q, k and v must be 2-byte aligned");
  return SAGE_OK;
}

float resolve_scale(float sm_scale, int64_t D) {
  return sm_scale > 0.0f ? sm_scale : 1.0f / sqrtf(static_cast<float>(D));
}

sage_status launch_attn(const sage_quantized* qt, float* out, int layout, int is_causal,
                        float sm_scale, cudaStream_t st) {
  AttnMaps maps{};
  sage_status s = make_maps(qt, &maps);
  if (s != SAGE_OK) return s;
  AttnParams p{};
  p.g = geo_of(qt);
  p.s_q = qt->s_q; p.s_k = qt->s_k; p.s_v = qt->s_v;
  p.out = out;
  if (qt->varlen) {
    p.out_seg_stride = 0; p.out_head_stride = qt->D; p.out_tok_stride = qt->Hq * qt->D;
  } else if (layout == SAGE_HND) {
    p.out_seg_stride = qt->Hq * qt->Lq * qt->D; p.out_head_stride = qt->Lq * qt->D;
    p.out_tok_stride = qt->D;
  } else {
    p.out_seg_stride = qt->Lq * qt->Hq * qt->D; p.out_head_stride = qt->D;
    p.out_tok_stride = qt->Hq * qt->D;
  }
  p.scale_log2 = resolve_scale(sm_scale, qt->D) * 1.44269504088896340736f;
  p.one = 1.0f;
  p.causal = is_causal ? 1 : 0;
  // the output as a tensor-store target (32-column boxes of 128 rows): rows
  // of a dense tile are clipped at Lq, columns at D; needs 16-byte rows
  p.out_tma = 0;
  if (qt->D % 4 == 0 && aligned(out, 16)) {
    const uint64_t D = static_cast<uint64_t>(qt->D), Hq = static_cast<uint64_t>(qt->Hq);
    uint64_t dims[4], strides[3];
    uint32_t box[4];
    uint32_t rank = 4;
    int kind;
    if (qt->varlen) {
      rank = 3;
      kind = 3;
      dims[0] = D; dims[1] = Hq; dims[2] = static_cast<uint64_t>(qt->total_q);
      strides[0] = D * 4; strides[1] = Hq * D * 4;
      box[0] = 32; box[1] = 1; box[2] = 128;
    } else if (layout == SAGE_HND) {
      kind = 1;
      const uint64_t Lq = static_cast<uint64_t>(qt->Lq);
      dims[0] = D; dims[1] = Lq; dims[2] = Hq; dims[3] = static_cast<uint64_t>(qt->nseg);
      strides[0] = D * 4; strides[1] = Lq * D * 4; strides[2] = Hq * Lq * D * 4;
      box[0] = 32; box[1] = 128; box[2] = 1; box[3] = 1;
    } else {
      kind = 2;
      const uint64_t Lq = static_cast<uint64_t>(qt->Lq);
      dims[0] = D; dims[1] = Hq; dims[2] = Lq; dims[3] = static_cast<uint64_t>(qt->nseg);
      strides[0] = D * 4; strides[1] = Hq * D * 4; strides[2] = Lq * Hq * D * 4;
      box[0] = 32; box[1] = 1; box[2] = 128; box[3] = 1;
    }
    if (encode_tiled(&maps.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, out, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      p.out_tma = kind;
  }
  p.v16 = qt->v_fp16;
  p.skip_kv_tile = g_skip_kv_tile.load();
  if (p.skip_kv_tile >= 0) {                  // a limited fault: count this launch
    int left = g_fault_launches.load();
    while (left >= 0) {
      if (left == 0) {
        p.skip_kv_tile = -1;
        break;
      }
      if (g_fault_launches.compare_exchange_weak(left, left - 1)) break;
    }
  }
  p.timeout_ns = wait_timeout_ns();
  p.status = qt->status;
  cudaError_t e = launch_attention(maps, p, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return ok();
}

int64_t out_elems_dense(int64_t B, int64_t Hq, int64_t Lq, int64_t D) {
  return B * Hq * Lq * D;
}

}  // namespace

namespace {

// Dense prologue entry points (e4m3 V, or fp16 V for the FP16-PV variant).
sage_status dense_prologue(const void* q, const void* k, const void* v, int dtype, int layout,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                           int64_t D, void* ws, size_t ws_bytes, sage_quantized* qt,
                           sage_stream_t stream, bool v16) {
  if (qt == nullptr) return fail(SAGE_ERR_INVALID_ARG, "qt must not be null");
  sage_status s = SAGE_OK;
  if (layout != SAGE_HND && layout != SAGE_NHD)
    return fail(SAGE_ERR_INVALID_ARG, "layout %d is neither SAGE_HND nor SAGE_NHD", layout);
  if (B < 0 || Lq < 0 || Lk < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative size (B=%lld Lq=%lld Lk=%lld)",
                (long long)B, (long long)Lq, (long long)Lk);
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if ((s = check_common(q, k, v, dtype)) != SAGE_OK) return s;
  if (B == 0 || Lq == 0 || Lk == 0)
    return fail(SAGE_ERR_INVALID_ARG, "the prologue needs B, Lq and Lk > 0");
  return run_prologue(dense_geo(B, Hq, Hkv, Lq, Lk, D, dtype, layout), q, k, v, ws,
                      ws_bytes, qt, reinterpret_cast<cudaStream_t>(stream), v16);
}

// Dense one-call entry points: prologue and attention, or zeros for an empty
// key set.
sage_status dense_fwd(const void* q, const void* k, const void* v, float* out, int64_t B,
                      int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D, int layout,
                      int is_causal, float sm_scale, int dtype, void* ws, size_t ws_bytes,
                      sage_stream_t stream, bool v16, bool keep_status = false) {
  sage_status s = SAGE_OK;
  if (layout != SAGE_HND && layout != SAGE_NHD)
    return fail(SAGE_ERR_INVALID_ARG, "layout %d is neither SAGE_HND nor SAGE_NHD", layout);
  if (B < 0 || Lq < 0 || Lk < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative size (B=%lld Lq=%lld Lk=%lld)",
                (long long)B, (long long)Lq, (long long)Lk);
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if (B == 0 || Lq == 0) return ok();                 // nothing to compute
  // an empty key tensor may legitimately have null data pointers
  if ((s = check_common(q, Lk == 0 ? q : k, Lk == 0 ? q : v, dtype)) != SAGE_OK) return s;
  if (out == nullptr || !aligned(out, 4))
    return fail(SAGE_ERR_INVALID_ARG, "out must be a 4-byte aligned device pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (Lk == 0) {                                      // empty softmax: zeros
    if ((s = check_device()) != SAGE_OK) return s;
    cudaError_t e = cudaMemsetAsync(out, 0, out_elems_dense(B, Hq, Lq, D) * 4, st);
    return e == cudaSuccess ? ok() : cuda_fail(e, "cudaMemsetAsync");
  }
  sage_quantized qt;
  s = run_prologue(dense_geo(B, Hq, Hkv, Lq, Lk, D, dtype, layout), q, k, v, ws, ws_bytes,
                   &qt, st, v16, keep_status);
  if (s != SAGE_OK) return s;
  if (qt.nseg > 65535 || qt.Hq > 65535)
    return fail(SAGE_ERR_UNSUPPORTED, "more than 65535 segments or heads");
  return launch_attn(&qt, out, layout, is_causal, sm_scale, st);
}

// The varlen prologue; keep_status leaves the workspace's status word as it
// is (the host-buffer pipeline's later chunks).
sage_status varlen_prologue(const void* q, const void* k, const void* v, int dtype,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int64_t nseq, int64_t total_q, int64_t total_k, int max_q,
                            int max_k, int64_t Hq, int64_t Hkv, int64_t D, void* ws,
                            size_t ws_bytes, sage_quantized* qt, sage_stream_t stream,
                            bool keep_status) {
  if (qt == nullptr) return fail(SAGE_ERR_INVALID_ARG, "qt must not be null");
  sage_status s = SAGE_OK;
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if ((s = check_common(q, k, v, dtype)) != SAGE_OK) return s;
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4))
    return fail(SAGE_ERR_INVALID_ARG, "cu_seqlens_q/k must be aligned device pointers");
  if (nseq < 1 || total_q < 1 || total_k < 1 || max_q < 1 || max_k < 1)
    return fail(SAGE_ERR_INVALID_ARG,
                "varlen prologue needs nseq, totals and maxima > 0 (nseq=%lld)",
                (long long)nseq);
  if (nseq > 65535) return fail(SAGE_ERR_UNSUPPORTED, "nseq=%lld > 65535", (long long)nseq);
  return run_prologue(varlen_geo(nseq, total_q, total_k, max_q, max_k, Hq, Hkv, D, dtype,
                                 cu_seqlens_q, cu_seqlens_k),
                      q, k, v, ws, ws_bytes, qt, reinterpret_cast<cudaStream_t>(stream),
                      /*v16=*/false, keep_status);
}

// Packed varlen prologue and attention in one call; keep_status as above.
sage_status varlen_fwd(const void* q, const void* k, const void* v, float* out,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t nseq,
                       int64_t total_q, int64_t total_k, int max_q, int max_k, int64_t Hq,
                       int64_t Hkv, int64_t D, int is_causal, float sm_scale, int dtype,
                       void* ws, size_t ws_bytes, sage_stream_t stream, bool keep_status) {
  sage_status s = SAGE_OK;
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if (nseq < 0 || total_q < 0 || total_k < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative varlen size");
  if (nseq == 0 || total_q == 0) return ok();
  if (out == nullptr || !aligned(out, 4))
    return fail(SAGE_ERR_INVALID_ARG, "out must be a 4-byte aligned device pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (total_k == 0) {
    if ((s = check_common(q, q, q, dtype)) != SAGE_OK) return s;
    if ((s = check_device()) != SAGE_OK) return s;
    cudaError_t e = cudaMemsetAsync(out, 0, total_q * Hq * D * 4, st);
    return e == cudaSuccess ? ok() : cuda_fail(e, "cudaMemsetAsync");
  }
  sage_quantized qt;
  s = varlen_prologue(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, nseq, total_q, total_k,
                      max_q, max_k, Hq, Hkv, D, ws, ws_bytes, &qt, stream, keep_status);
  if (s != SAGE_OK) return s;
  return launch_attn(&qt, out, SAGE_NHD, is_causal, sm_scale, st);
}

}  // namespace


// ------------------------------------------------ host-buffer pipeline
// sage_attn_fwd_host cuts a dense problem into (batch, kv-head group) chunks
// and pipelines them: the copy of chunk i+1 into device staging runs on one
// stream while chunk i's prologue and attention run on the caller's stream
// and chunk i-1's output is copied back on a third.  Two staging slots
// alternate; events order every reuse.  Attention never mixes heads or
// batches, so the result is the same as one sage_attn_fwd call.
// sage_attn_fwd_varlen_host does the same for packed sequences: its chunks
// are kv-head groups of the whole packed tensor (every sequence), and the
// cumulative offsets are copied once into the workspace.
namespace {

// A host-buffer problem: dense (B entries of Lq query and Lk key rows) or
// packed varlen (one entry of total_q and total_k rows, nseq sequences).
struct HostShape {
  int64_t B, Hq, Hkv, Lq, Lk, D;
  bool varlen;
  int64_t nseq;              // varlen only
  int max_q, max_k;          // varlen only
};

HostShape dense_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D) {
  return HostShape{B, Hq, Hkv, Lq, Lk, D, false, 0, 0, 0};
}

struct HostPlan {
  int64_t chunk_kv;          // kv heads per chunk
  int64_t group;             // query heads per kv head
  size_t ws_bytes;           // prologue workspace of one chunk (offset 0)
  size_t q_bytes, kv_bytes, out_bytes;   // one chunk's q, k (= v), out
  size_t cu;                 // varlen: offset of the device copy of cu_seqlens_q, then _k
  size_t slot[2];            // offsets of the two staging slots
  size_t total;
};

int sm_count_of_current_device() {
  static std::atomic<int> sms[64] = {};          // per device, filled once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// chunk_kv <= 0 picks enough kv heads for one wave of query-tile pairs per
// chunk (one per SM), so that each chunk's attention still fills the GPU, or
// one fewer when that still fills 90 % of the wave; chunks whose attention
// outlasts their copies are sized for whole waves instead.
// Packed sequences take four waves: a chunk's attention lasts at least as
// long as a pair of its longest sequence, so a chunk of few heads leaves
// most SMs idle behind that pair (measured on 8 sequences of 2k-16k tokens,
// 16 heads: 4 or 2 kv heads per chunk 20-54 % faster than copying in,
// computing and copying back; 1 head 11 % and 41 %).
HostPlan host_plan(const HostShape& h, int64_t chunk_kv) {
  HostPlan P{};
  P.group = h.Hq / h.Hkv;
  if (chunk_kv <= 0) {
    // query tiles per query head (packed sequences: at most one ragged tile each)
    const int64_t qtiles = (h.Lq + 127) / 128 + (h.varlen ? h.nseq : 0);
    const int64_t pairs = P.group * ((qtiles + 1) / 2);
    const int64_t sms = sm_count_of_current_device() > 0 ? sm_count_of_current_device() : 152;
    const int64_t want = (h.varlen ? 4 : 1) * sms;
    chunk_kv = pairs > 0 ? (want + pairs - 1) / pairs : h.Hkv;
    // A dense chunk one kv head smaller that still fills 90 % of the wave
    // keeps its pairs out of a second, nearly empty wave (B=2 H=24 L=4096:
    // 9 kv heads, 144 pairs, 1.047 ms per call against 1.111 ms for 10).
    if (!h.varlen && chunk_kv > 1 && 10 * (chunk_kv - 1) * pairs >= 9 * want) --chunk_kv;
    // A dense chunk whose attention outlasts its copies (long key spans: more
    // than ~7000 flops per copied byte, about 1.4 PFLOP/s of attention over a
    // 200 GB/s link) is sized for whole waves of pairs instead, the smallest
    // that wastes at most 5 % of its last wave (L=32768: 7 kv heads, 896 pairs
    // in 6 waves, 14.06 ms per call against 15.45 ms for 2 heads).
    const double flops = 4.0 * P.group * h.Lq * h.Lk;              // per kv head, / D
    const double bytes = 6.0 * P.group * h.Lq + 4.0 * h.Lk;        // q, k, v in, out; / D
    if (!h.varlen && pairs > 0 && flops > 7000.0 * bytes) {
      for (int64_t c = chunk_kv; c <= h.Hkv; ++c) {
        const int64_t n = c * pairs, waves = (n + sms - 1) / sms;
        if (20 * (waves * sms - n) <= n) {                         // waste <= 5 %
          chunk_kv = c;
          break;
        }
      }
    }
  }
  P.chunk_kv = chunk_kv < 1 ? 1 : (chunk_kv > h.Hkv ? h.Hkv : chunk_kv);
  const int64_t hq = P.chunk_kv * P.group;
  P.q_bytes = static_cast<size_t>(hq * h.Lq * h.D * 2);
  P.kv_bytes = static_cast<size_t>(P.chunk_kv * h.Lk * h.D * 2);
  P.out_bytes = static_cast<size_t>(hq * h.Lq * h.D * 4);
  P.ws_bytes = align256(
      h.varlen ? sage_workspace_bytes_varlen(h.nseq, h.Lq, h.Lk, hq, P.chunk_kv, h.D)
               : sage_workspace_bytes(1, hq, P.chunk_kv, h.Lq, h.Lk, h.D));
  P.cu = P.ws_bytes;
  const size_t cu_bytes = h.varlen ? 2 * align256(static_cast<size_t>(h.nseq + 1) * 4) : 0;
  const size_t per_slot = align256(P.q_bytes) + 2 * align256(P.kv_bytes) + align256(P.out_bytes);
  P.slot[0] = P.ws_bytes + cu_bytes;
  P.slot[1] = P.slot[0] + per_slot;
  P.total = P.slot[1] + per_slot;
  return P;
}

// Host-side check of a host cu_seqlens array: starts at 0, ends at total,
// and every length lies in 0..maxlen.
bool check_cu_host(const int32_t* cu, int64_t nseq, int64_t total, int maxlen,
                   const char* name, sage_status* st) {
  if (cu[0] != 0 || cu[nseq] != total) {
    *st = fail(SAGE_ERR_INVALID_ARG, "%s must start at 0 and end at %lld", name,
               (long long)total);
    return false;
  }
  for (int64_t i = 0; i < nseq; ++i) {
    const int64_t len = static_cast<int64_t>(cu[i + 1]) - cu[i];
    if (len < 0 || len > maxlen) {
      *st = fail(SAGE_ERR_INVALID_ARG, "%s: sequence %lld has length %lld outside 0..%d", name,
                 (long long)i, (long long)len, maxlen);
      return false;
    }
  }
  return true;
}

// Copy streams and events of the pipeline, created once per device and kept
// for the process (like the kernels' attributes); calls on one device enqueue
// one at a time.
struct HostRuntime {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, loaded[2] = {}, computed[2] = {}, stored[2] = {};
};

HostRuntime g_host_rt[64];

cudaError_t host_runtime_init(HostRuntime& rt) {
  if (rt.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&rt.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&rt.out, cudaStreamNonBlocking);
  cudaEvent_t* evs[] = {&rt.start, &rt.loaded[0], &rt.loaded[1], &rt.computed[0],
                        &rt.computed[1], &rt.stored[0], &rt.stored[1]};
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e == cudaSuccess) {
    rt.ready = true;
    return e;
  }
  // a partial set is released, so a later call starts from nothing
  for (cudaEvent_t* ev : evs)
    if (*ev != nullptr) {
      cudaEventDestroy(*ev);
      *ev = nullptr;
    }
  if (rt.in != nullptr) cudaStreamDestroy(rt.in);
  if (rt.out != nullptr) cudaStreamDestroy(rt.out);
  rt.in = rt.out = nullptr;
  return e;
}

// One chunk's rows of a dense tensor between host and device staging:
// contiguous for HND, a pitched copy (Lq rows of the chunk's heads) for NHD.
cudaError_t copy_chunk(void* dst, const void* src, bool to_device, bool hnd, int64_t b,
                       int64_t h0, int64_t hn, int64_t H, int64_t L, int64_t D,
                       size_t elem, cudaStream_t st) {
  const cudaMemcpyKind kind = to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost;
  if (hnd) {
    const size_t off = static_cast<size_t>((b * H + h0) * L * D) * elem;
    const size_t n = static_cast<size_t>(hn * L * D) * elem;
    return to_device
               ? cudaMemcpyAsync(dst, static_cast<const char*>(src) + off, n, kind, st)
               : cudaMemcpyAsync(static_cast<char*>(dst) + off, src, n, kind, st);
  }
  const size_t host_pitch = static_cast<size_t>(H * D) * elem;
  const size_t dev_pitch = static_cast<size_t>(hn * D) * elem;
  const size_t off = static_cast<size_t>((b * L * H + h0) * D) * elem;
  return to_device
             ? cudaMemcpy2DAsync(dst, dev_pitch, static_cast<const char*>(src) + off, host_pitch,
                                 dev_pitch, static_cast<size_t>(L), kind, st)
             : cudaMemcpy2DAsync(static_cast<char*>(dst) + off, host_pitch, src, dev_pitch,
                                 dev_pitch, static_cast<size_t>(L), kind, st);
}

}  // namespace

namespace {

// The host-buffer pipeline (see sage_attn_fwd_host and
// sage_attn_fwd_varlen_host); v16 runs the FP16-PV kernels (dense only).
// Arguments are checked by the callers.
sage_status host_pipeline(const void* q, const void* k, const void* v, float* out,
                          const HostShape& h, const int32_t* cu_q, const int32_t* cu_k,
                          int layout, int is_causal, float sm_scale, int dtype,
                          int64_t chunk_kv_heads, void* ws, size_t ws_bytes,
                          sage_stream_t stream, bool v16) {
  sage_status s = SAGE_OK;
  if ((s = check_device()) != SAGE_OK) return s;
  const HostPlan P = host_plan(h, chunk_kv_heads);
  if (ws == nullptr || !aligned(ws, 256))
    return fail(SAGE_ERR_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
  if (ws_bytes < P.total)
    return fail(SAGE_ERR_WORKSPACE, "workspace has %zu bytes, the host-buffer call needs %zu",
                ws_bytes, P.total);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(SAGE_ERR_UNSUPPORTED, "device index %d", dev);
  HostRuntime& rt = g_host_rt[dev];
  std::lock_guard<std::mutex> lock(rt.mu);
  if ((e = host_runtime_init(rt)) != cudaSuccess) return cuda_fail(e, "pipeline streams");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const bool hnd = layout == SAGE_HND;
  // the staging and the workspace may still be in use by the caller's
  // earlier work on its stream
  e = cudaEventRecord(rt.start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(rt.in, rt.start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "pipeline start");
  // Every exit from here on first makes the caller's stream wait for the copies
  // already enqueued, so that it never completes while one of them still
  // reads the staging or writes the caller's host output.
  const char* where = nullptr;
  int32_t* dcu_q = reinterpret_cast<int32_t*>(base + P.cu);
  int32_t* dcu_k = reinterpret_cast<int32_t*>(
      base + P.cu + align256(static_cast<size_t>(h.nseq + 1) * 4));
  if (h.varlen) {
    // the offsets, once, ahead of the first chunk's inputs on the copy stream
    const size_t n = static_cast<size_t>(h.nseq + 1) * 4;
    e = cudaMemcpyAsync(dcu_q, cu_q, n, cudaMemcpyHostToDevice, rt.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dcu_k, cu_k, n, cudaMemcpyHostToDevice, rt.in);
    if (e != cudaSuccess) where = "pipeline offsets";
  }
  int64_t i = 0;
  for (int64_t b = 0; b < h.B && where == nullptr && s == SAGE_OK; ++b) {
    for (int64_t g0 = 0; g0 < h.Hkv; g0 += P.chunk_kv, ++i) {
      const int64_t gn = h.Hkv - g0 < P.chunk_kv ? h.Hkv - g0 : P.chunk_kv;
      const int64_t h0 = g0 * P.group, hn = gn * P.group;
      const int sl = static_cast<int>(i & 1);
      uint8_t* dq = base + P.slot[sl];
      uint8_t* dk = dq + align256(P.q_bytes);
      uint8_t* dv = dk + align256(P.kv_bytes);
      float* dout = reinterpret_cast<float*>(dv + align256(P.kv_bytes));
      // inputs: after the slot's previous chunk has been computed
      e = cudaStreamWaitEvent(rt.in, rt.computed[sl], 0);
      if (e == cudaSuccess)
        e = copy_chunk(dq, q, true, hnd, b, h0, hn, h.Hq, h.Lq, h.D, 2, rt.in);
      if (e == cudaSuccess)
        e = copy_chunk(dk, k, true, hnd, b, g0, gn, h.Hkv, h.Lk, h.D, 2, rt.in);
      if (e == cudaSuccess)
        e = copy_chunk(dv, v, true, hnd, b, g0, gn, h.Hkv, h.Lk, h.D, 2, rt.in);
      if (e == cudaSuccess) e = cudaEventRecord(rt.loaded[sl], rt.in);
      // compute: after the inputs landed and the slot's previous output left
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st, rt.loaded[sl], 0);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st, rt.stored[sl], 0);
      if (e != cudaSuccess) {
        where = "pipeline copy-in";
        break;
      }
      // the first chunk clears the device status word, the others keep it,
      // so a bounded wait that ran out in any chunk stays visible
      if (i == g_host_fail_chunk.load()) {
        s = fail(SAGE_ERR_INVALID_ARG, "chunk %lld failed (test hook)", (long long)i);
        break;
      }
      if (h.varlen)
        s = varlen_fwd(dq, dk, dv, dout, dcu_q, dcu_k, h.nseq, h.Lq, h.Lk, h.max_q, h.max_k,
                       hn, gn, h.D, is_causal, sm_scale, dtype, base, P.ws_bytes, stream,
                       /*keep_status=*/i > 0);
      else
        s = dense_fwd(dq, dk, dv, dout, 1, hn, gn, h.Lq, h.Lk, h.D, layout, is_causal,
                      sm_scale, dtype, base, P.ws_bytes, stream, v16, /*keep_status=*/i > 0);
      if (s != SAGE_OK) break;
      e = cudaEventRecord(rt.computed[sl], st);
      // output: after the chunk was computed
      if (e == cudaSuccess) e = cudaStreamWaitEvent(rt.out, rt.computed[sl], 0);
      if (e == cudaSuccess)
        e = copy_chunk(out, dout, false, hnd, b, h0, hn, h.Hq, h.Lq, h.D, 4, rt.out);
      if (e == cudaSuccess) e = cudaEventRecord(rt.stored[sl], rt.out);
      if (e != cudaSuccess) {
        where = "pipeline copy-out";
        break;
      }
    }
  }
  // the caller's stream completes once every output is in host memory (and,
  // after a failure, once every copy enqueued so far has finished; rt.start,
  // whose first record the copy stream has already waited for, marks the end
  // of the copy-in stream)
  cudaError_t ej = cudaEventRecord(rt.start, rt.in);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, rt.start, 0);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, rt.stored[0], 0);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, rt.stored[1], 0);
  if (where != nullptr) return cuda_fail(e, where);
  if (s != SAGE_OK) return s;
  return ej == cudaSuccess ? ok() : cuda_fail(ej, "pipeline end");
}

// Dense host-buffer call: argument checks, then the pipeline.
sage_status host_fwd(const void* q, const void* k, const void* v, float* out, int64_t B,
                     int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D, int layout,
                     int is_causal, float sm_scale, int dtype, int64_t chunk_kv_heads,
                     void* ws, size_t ws_bytes, sage_stream_t stream, bool v16) {
  sage_status s = SAGE_OK;
  if (layout != SAGE_HND && layout != SAGE_NHD)
    return fail(SAGE_ERR_INVALID_ARG, "layout %d is neither SAGE_HND nor SAGE_NHD", layout);
  if (B < 0 || Lq < 0 || Lk < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative size (B=%lld Lq=%lld Lk=%lld)",
                (long long)B, (long long)Lq, (long long)Lk);
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if (dtype != SAGE_F16 && dtype != SAGE_BF16)
    return fail(SAGE_ERR_INVALID_ARG, "dtype %d is neither SAGE_F16 nor SAGE_BF16", dtype);
  if (B == 0 || Lq == 0) return ok();                 // nothing to compute
  if (Lk == 0)
    return fail(SAGE_ERR_INVALID_ARG, "the host-buffer call needs Lk > 0");
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "null host buffer");
  return host_pipeline(q, k, v, out, dense_shape(B, Hq, Hkv, Lq, Lk, D), nullptr, nullptr,
                       layout, is_causal, sm_scale, dtype, chunk_kv_heads, ws, ws_bytes,
                       stream, v16);
}

// Packed varlen host-buffer call: argument and offset checks, then the pipeline.
sage_status varlen_host_fwd(const void* q, const void* k, const void* v, float* out,
                            const int32_t* cu_q, const int32_t* cu_k, int64_t nseq,
                            int64_t total_q, int64_t total_k, int max_q, int max_k,
                            int64_t Hq, int64_t Hkv, int64_t D, int is_causal, float sm_scale,
                            int dtype, int64_t chunk_kv_heads, void* ws, size_t ws_bytes,
                            sage_stream_t stream) {
  sage_status s = SAGE_OK;
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if (dtype != SAGE_F16 && dtype != SAGE_BF16)
    return fail(SAGE_ERR_INVALID_ARG, "dtype %d is neither SAGE_F16 nor SAGE_BF16", dtype);
  if (nseq < 0 || total_q < 0 || total_k < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative varlen size");
  if (nseq == 0 || total_q == 0) return ok();         // nothing to compute
  if (total_k == 0)
    return fail(SAGE_ERR_INVALID_ARG, "the host-buffer call needs total_k > 0");
  if (nseq > 65535) return fail(SAGE_ERR_UNSUPPORTED, "nseq=%lld > 65535", (long long)nseq);
  if (max_q < 1 || max_k < 1)
    return fail(SAGE_ERR_INVALID_ARG, "max_q and max_k must be positive");
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || cu_q == nullptr ||
      cu_k == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "null host buffer");
  if (!check_cu_host(cu_q, nseq, total_q, max_q, "cu_seqlens_q", &s) ||
      !check_cu_host(cu_k, nseq, total_k, max_k, "cu_seqlens_k", &s))
    return s;
  const HostShape h{1, Hq, Hkv, total_q, total_k, D, true, nseq, max_q, max_k};
  return host_pipeline(q, k, v, out, h, cu_q, cu_k, SAGE_NHD, is_causal, sm_scale, dtype,
                       chunk_kv_heads, ws, ws_bytes, stream, false);
}

}  // namespace

extern "C" {

size_t sage_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                            int64_t D) {
  if (B < 0 || Lq < 0 || Lk < 0 || D < 1 || D > 128 || Hq < 1 || Hkv < 1 || Hq % Hkv)
    return 0;
  return ws_layout(dense_geo(B, Hq, Hkv, Lq, Lk, D, 0, SAGE_HND)).total;
}

size_t sage_workspace_bytes_varlen(int64_t nseq, int64_t total_q, int64_t total_k,
                                   int64_t Hq, int64_t Hkv, int64_t D) {
  if (nseq < 0 || total_q < 0 || total_k < 0 || D < 1 || D > 128 || Hq < 1 || Hkv < 1 ||
      Hq % Hkv)
    return 0;
  return ws_layout(varlen_geo(nseq, total_q, total_k, 0, 0, Hq, Hkv, D, 0, nullptr,
                              nullptr)).total;
}

sage_status sage_quant_prologue(const void* q, const void* k, const void* v, int dtype,
                                int layout, int64_t B, int64_t Hq, int64_t Hkv,
                                int64_t Lq, int64_t Lk, int64_t D, void* ws,
                                size_t ws_bytes, sage_quantized* qt,
                                sage_stream_t stream) {
  return dense_prologue(q, k, v, dtype, layout, B, Hq, Hkv, Lq, Lk, D, ws, ws_bytes, qt,
                        stream, false);
}

sage_status sage_quant_prologue_pv16(const void* q, const void* k, const void* v, int dtype,
                                     int layout, int64_t B, int64_t Hq, int64_t Hkv,
                                     int64_t Lq, int64_t Lk, int64_t D, void* ws,
                                     size_t ws_bytes, sage_quantized* qt,
                                     sage_stream_t stream) {
  return dense_prologue(q, k, v, dtype, layout, B, Hq, Hkv, Lq, Lk, D, ws, ws_bytes, qt,
                        stream, true);
}

sage_status sage_quant_prologue_varlen(const void* q, const void* k, const void* v,
                                       int dtype, const int32_t* cu_seqlens_q,
                                       const int32_t* cu_seqlens_k, int64_t nseq,
                                       int64_t total_q, int64_t total_k, int max_q,
                                       int max_k, int64_t Hq, int64_t Hkv, int64_t D,
                                       void* ws, size_t ws_bytes, sage_quantized* qt,
                                       sage_stream_t stream) {
  return varlen_prologue(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, nseq, total_q, total_k,
                         max_q, max_k, Hq, Hkv, D, ws, ws_bytes, qt, stream, false);
}

sage_status sage_quant_prologue_strided(const void* q, const void* k, const void* v,
                                        int dtype, int64_t B, int64_t Hq, int64_t Hkv,
                                        int64_t Lq, int64_t Lk, int64_t D,
                                        const int64_t* q_strides, const int64_t* kv_strides,
                                        void* ws, size_t ws_bytes, sage_quantized* qt,
                                        sage_stream_t stream) {
  if (qt == nullptr) return fail(SAGE_ERR_INVALID_ARG, "qt must not be null");
  sage_status s = SAGE_OK;
  if (B < 0 || Lq < 0 || Lk < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative size (B=%lld Lq=%lld Lk=%lld)",
                (long long)B, (long long)Lq, (long long)Lk);
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  if ((s = check_common(q, k, v, dtype)) != SAGE_OK) return s;
  if (B == 0 || Lq == 0 || Lk == 0)
    return fail(SAGE_ERR_INVALID_ARG, "the prologue needs B, Lq and Lk > 0");
  SegGeo g;
  if ((s = strided_geo(B, Hq, Hkv, Lq, Lk, D, dtype, q_strides, kv_strides, &g)) != SAGE_OK)
    return s;
  return run_prologue(g, q, k, v, ws, ws_bytes, qt, reinterpret_cast<cudaStream_t>(stream));
}

sage_status sage_attn_quantized(const sage_quantized* qt, float* out, int layout,
                                int is_causal, float sm_scale, sage_stream_t stream) {
  if (qt == nullptr || qt->q16 == nullptr || qt->status == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "qt is null or was not filled by the prologue");
  if (out == nullptr || !aligned(out, 4))
    return fail(SAGE_ERR_INVALID_ARG, "out must be a 4-byte aligned device pointer");
  if (!qt->varlen && layout != SAGE_HND && layout != SAGE_NHD)
    return fail(SAGE_ERR_INVALID_ARG, "layout %d is neither SAGE_HND nor SAGE_NHD", layout);
  if (qt->nseg > 65535 || qt->Hq > 65535)
    return fail(SAGE_ERR_UNSUPPORTED, "more than 65535 segments or heads");
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  return launch_attn(qt, out, layout, is_causal, sm_scale,
                     reinterpret_cast<cudaStream_t>(stream));
}

sage_status sage_attn_fwd(const void* q, const void* k, const void* v, float* out,
                          int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                          int64_t D, int layout, int is_causal, float sm_scale, int dtype,
                          void* ws, size_t ws_bytes, sage_stream_t stream) {
  return dense_fwd(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, layout, is_causal, sm_scale, dtype,
                   ws, ws_bytes, stream, false);
}

sage_status sage_attn_fwd_pv16(const void* q, const void* k, const void* v, float* out,
                               int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                               int64_t D, int layout, int is_causal, float sm_scale,
                               int dtype, void* ws, size_t ws_bytes, sage_stream_t stream) {
  return dense_fwd(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, layout, is_causal, sm_scale, dtype,
                   ws, ws_bytes, stream, true);
}

sage_status sage_attn_fwd_strided(const void* q, const void* k, const void* v, float* out,
                                  int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                                  int64_t D, const int64_t* q_strides,
                                  const int64_t* kv_strides, int layout, int is_causal,
                                  float sm_scale, int dtype, void* ws, size_t ws_bytes,
                                  sage_stream_t stream) {
  sage_status s = SAGE_OK;
  if (layout != SAGE_HND && layout != SAGE_NHD)
    return fail(SAGE_ERR_INVALID_ARG, "layout %d is neither SAGE_HND nor SAGE_NHD", layout);
  if (B < 0 || Lq < 0 || Lk < 0)
    return fail(SAGE_ERR_INVALID_ARG, "negative size (B=%lld Lq=%lld Lk=%lld)",
                (long long)B, (long long)Lq, (long long)Lk);
  if (!check_dims(Hq, Hkv, D, &s)) return s;
  SegGeo g;
  if ((s = strided_geo(B, Hq, Hkv, Lq, Lk, D, dtype, q_strides, kv_strides, &g)) != SAGE_OK)
    return s;
  if (B == 0 || Lq == 0) return ok();                 // nothing to compute
  if ((s = check_common(q, Lk == 0 ? q : k, Lk == 0 ? q : v, dtype)) != SAGE_OK) return s;
  if (out == nullptr || !aligned(out, 4))
    return fail(SAGE_ERR_INVALID_ARG, "out must be a 4-byte aligned device pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (Lk == 0) {                                      // empty softmax: zeros
    if ((s = check_device()) != SAGE_OK) return s;
    cudaError_t e = cudaMemsetAsync(out, 0, out_elems_dense(B, Hq, Lq, D) * 4, st);
    return e == cudaSuccess ? ok() : cuda_fail(e, "cudaMemsetAsync");
  }
  sage_quantized qt;
  if ((s = run_prologue(g, q, k, v, ws, ws_bytes, &qt, st)) != SAGE_OK) return s;
  if (qt.nseg > 65535 || qt.Hq > 65535)
    return fail(SAGE_ERR_UNSUPPORTED, "more than 65535 segments or heads");
  return launch_attn(&qt, out, layout, is_causal, sm_scale, st);
}

sage_status sage_attn_fwd_varlen(const void* q, const void* k, const void* v, float* out,
                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                 int64_t nseq, int64_t total_q, int64_t total_k, int max_q,
                                 int max_k, int64_t Hq, int64_t Hkv, int64_t D,
                                 int is_causal, float sm_scale, int dtype, void* ws,
                                 size_t ws_bytes, sage_stream_t stream) {
  return varlen_fwd(q, k, v, out, cu_seqlens_q, cu_seqlens_k, nseq, total_q, total_k, max_q,
                    max_k, Hq, Hkv, D, is_causal, sm_scale, dtype, ws, ws_bytes, stream, false);
}

sage_status sage_debug_qk_int32(const sage_quantized* qt, int64_t seg, int64_t hq,
                                int64_t qtile, int64_t ktile, int32_t* out,
                                sage_stream_t stream) {
  if (qt == nullptr || qt->q16 == nullptr || out == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "null argument");
  if (qt->varlen) return fail(SAGE_ERR_UNSUPPORTED, "debug tiles are for dense calls only");
  if (seg < 0 || seg >= qt->nseg || hq < 0 || hq >= qt->Hq || qtile < 0 ||
      qtile * 128 >= qt->q_head_rows || ktile < 0 || ktile * 128 >= qt->k_head_rows)
    return fail(SAGE_ERR_INVALID_ARG, "tile index out of range");
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  AttnMaps maps;
  if ((s = make_maps(qt, &maps)) != SAGE_OK) return s;
  AttnParams p{};
  p.g = geo_of(qt);
  p.status = qt->status;
  p.timeout_ns = kDefaultTimeoutNs;
  const int64_t hk = hq / (qt->Hq / qt->Hkv);
  const int64_t q_row0 = (seg * qt->Hq + hq) * qt->q_head_rows + qtile * 128;
  const int64_t k_row0 = (seg * qt->Hkv + hk) * qt->k_head_rows + ktile * 128;
  cudaError_t e = launch_debug_qk(maps, p, q_row0, k_row0, out,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "debug qk launch");
  return ok();
}

sage_status sage_debug_pv_accum(const uint8_t* p8, const uint8_t* v8, int64_t ntiles,
                                int64_t Dp, float* out, uint32_t* status,
                                sage_stream_t stream) {
  if (p8 == nullptr || v8 == nullptr || out == nullptr || status == nullptr)
    return fail(SAGE_ERR_INVALID_ARG, "null argument");
  if (Dp != 64 && Dp != 128) return fail(SAGE_ERR_INVALID_ARG, "Dp must be 64 or 128");
  if (ntiles < 1 || ntiles > 4096)
    return fail(SAGE_ERR_INVALID_ARG, "ntiles must be 1..4096 (got %lld)", (long long)ntiles);
  if (!aligned(p8, 16) || !aligned(v8, 16) || !aligned(out, 4) || !aligned(status, 4))
    return fail(SAGE_ERR_INVALID_ARG, "p8 and v8 must be 16-byte aligned, out and status 4");
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(status, 0, 4, st);
  if (e == cudaSuccess) e = launch_debug_pv(p8, v8, ntiles, Dp, out, status, kDefaultTimeoutNs, st);
  if (e != cudaSuccess) return cuda_fail(e, "debug pv launch");
  return ok();
}

sage_status sage_debug_tc_rate(int kind, int64_t n_mma, uint32_t* status,
                               sage_stream_t stream) {
  if (kind != 0 && kind != 1) return fail(SAGE_ERR_INVALID_ARG, "kind must be 0 or 1");
  if (n_mma < 1 || n_mma > (int64_t(1) << 22))
    return fail(SAGE_ERR_INVALID_ARG, "n_mma must be 1..2^22");
  if (status == nullptr || !aligned(status, 4))
    return fail(SAGE_ERR_INVALID_ARG, "status must be a 4-byte aligned device pointer");
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(status, 0, 4, st);
  if (e == cudaSuccess) e = launch_tc_rate(kind, n_mma, status, kDefaultTimeoutNs, st);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core rate launch");
  return ok();
}

sage_status sage_debug_e4m3(const float* in, uint8_t* out, int64_t n, sage_stream_t stream) {
  if (n < 0 || (n > 0 && (in == nullptr || out == nullptr)))
    return fail(SAGE_ERR_INVALID_ARG, "bad buffers");
  if (n == 0) return ok();
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  cudaError_t e = launch_debug_e4m3(in, out, n, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "debug e4m3 launch");
}

void sage_debug_set_fault(int skip_kv_tile, uint64_t timeout_ns) {
  g_skip_kv_tile.store(skip_kv_tile);
  g_timeout_ns.store(timeout_ns);
}

void sage_debug_set_fault_launches(int launches) {
  g_fault_launches.store(launches < 0 ? -1 : launches);
}

void sage_debug_set_prologue_launches(int launches) {
  g_prologue_launches.store(launches == 1 || launches == 2 ? launches : 0);
}

void sage_debug_set_host_fail_chunk(int chunk) {
  g_host_fail_chunk.store(chunk < 0 ? -1 : chunk);
}

}  // extern "C"

namespace {
// The sage_status a device status word stands for.
sage_status status_of_word(uint32_t word) {
  if (word & kStatusTimeout)
    return fail(SAGE_ERR_DEVICE_TIMEOUT, "a device-side wait ran out (status 0x%x)", word);
  if (word & kStatusBadSeqlens)
    return fail(SAGE_ERR_INVALID_ARG, "cu_seqlens inconsistent with totals/maxima");
  if (word & kStatusBadItem)
    return fail(SAGE_ERR_UNSUPPORTED, "internal error: a prologue work item fell outside "
                "the call's plan and was skipped");
  return ok();
}
}  // namespace

extern "C" {

sage_status sage_device_status(const void* ws, sage_stream_t stream) {
  if (ws == nullptr) return fail(SAGE_ERR_INVALID_ARG, "null workspace");
  uint32_t word = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  return status_of_word(word);
}

sage_status sage_kv_stats_noalloc_status(sage_stream_t stream) {
  sage_status s = check_device();
  if (s != SAGE_OK) return s;
  uint32_t word = 0;
  cudaError_t e = read_kv_stats_static_status(&word, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reading the static scratch's status word");
  return status_of_word(word);
}

sage_status sage_kv_stats_noalloc(const void* k, const void* v, int dtype, int layout,
                                  int64_t B, int64_t Hkv, int64_t Lk, int64_t D,
                                  float* k_mean, float* s_v, sage_stream_t stream) {
  sage_status s = SAGE_OK;
  if (layout != SAGE_HND && layout != SAGE_NHD)
    return fail(SAGE_ERR_INVALID_ARG, "layout %d is neither SAGE_HND nor SAGE_NHD", layout);
  if (!check_dims(Hkv, Hkv, D, &s)) return s;
  if ((s = check_common(k, k, v, dtype)) != SAGE_OK) return s;
  if (B < 1 || Lk < 1)
    return fail(SAGE_ERR_INVALID_ARG, "B and Lk must be positive (B=%lld Lk=%lld)",
                (long long)B, (long long)Lk);
  if (k_mean == nullptr || s_v == nullptr || !aligned(k_mean, 4) || !aligned(s_v, 4))
    return fail(SAGE_ERR_INVALID_ARG, "k_mean and s_v must be 4-byte aligned device pointers");
  const int64_t entries = B * Hkv * padded_dim(D);
  if (entries > kStaticStatEntries)
    return fail(SAGE_ERR_UNSUPPORTED,
                "B*Hkv*Dp = %lld exceeds the %lld channel slots of the static scratch",
                (long long)entries, (long long)kStaticStatEntries);
  if ((s = check_device()) != SAGE_OK) return s;
  const SegGeo g = dense_geo(B, Hkv, Hkv, 1, Lk, D, dtype, layout);
  const bool vec = (D % 8 == 0) && aligned(k, 16) && aligned(v, 16);
  cudaError_t e = launch_kv_stats_static(g, static_cast<const uint16_t*>(k),
                                         static_cast<const uint16_t*>(v), k_mean, s_v, vec,
                                         wait_timeout_ns(),
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "static-scratch statistics");
  return ok();
}

size_t sage_workspace_bytes_host(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                                 int64_t D, int64_t chunk_kv_heads) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || D < 1 || D > 128 ||
      Hq % Hkv != 0)
    return 0;
  return host_plan(dense_shape(B, Hq, Hkv, Lq, Lk, D), chunk_kv_heads).total;
}

size_t sage_workspace_bytes_varlen_host(int64_t nseq, int64_t total_q, int64_t total_k,
                                        int64_t Hq, int64_t Hkv, int64_t D,
                                        int64_t chunk_kv_heads) {
  if (nseq <= 0 || nseq > 65535 || total_q <= 0 || total_k <= 0 || D < 1 || D > 128 ||
      Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return 0;
  const HostShape h{1, Hq, Hkv, total_q, total_k, D, true, nseq, 0, 0};
  return host_plan(h, chunk_kv_heads).total;
}

sage_status sage_attn_fwd_varlen_host(const void* q, const void* k, const void* v, float* out,
                                      const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, int64_t nseq,
                                      int64_t total_q, int64_t total_k, int max_q, int max_k,
                                      int64_t Hq, int64_t Hkv, int64_t D, int is_causal,
                                      float sm_scale, int dtype, int64_t chunk_kv_heads,
                                      void* ws, size_t ws_bytes, sage_stream_t stream) {
  return varlen_host_fwd(q, k, v, out, cu_seqlens_q, cu_seqlens_k, nseq, total_q, total_k,
                         max_q, max_k, Hq, Hkv, D, is_causal, sm_scale, dtype, chunk_kv_heads,
                         ws, ws_bytes, stream);
}

sage_status sage_attn_fwd_host(const void* q, const void* k, const void* v, float* out,
                               int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                               int64_t D, int layout, int is_causal, float sm_scale,
                               int dtype, int64_t chunk_kv_heads, void* ws, size_t ws_bytes,
                               sage_stream_t stream) {
  return host_fwd(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, layout, is_causal, sm_scale, dtype,
                  chunk_kv_heads, ws, ws_bytes, stream, false);
}

sage_status sage_attn_fwd_host_pv16(const void* q, const void* k, const void* v, float* out,
                                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                                    int64_t D, int layout, int is_causal, float sm_scale,
                                    int dtype, int64_t chunk_kv_heads, void* ws,
                                    size_t ws_bytes, sage_stream_t stream) {
  return host_fwd(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, layout, is_causal, sm_scale, dtype,
                  chunk_kv_heads, ws, ws_bytes, stream, true);
}

const char* sage_last_error(void) { return g_last_error.c_str(); }

uint64_t sage_launch_count(void) { return launch_count(); }

}  // extern "C"
