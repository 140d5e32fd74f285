// Host-side launch interface of the kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sage_geom.h"

namespace sage {

// cuTensorMapEncodeTiled (looked up once through the runtime): 16-bit or
// 8-bit elements, no interleave, 256-byte L2 promotion, zero fill.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle);

// Counts one kernel launch of this library (process-wide, all devices).
void note_launch();
uint64_t launch_count();

struct PrologueBuffers {
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
  void* ksum;        // int64 (fp16 inputs) or double (bf16), [nseg][Hkv][Dp]
  uint32_t* vmax;    // float bits, [nseg][Hkv][Dp]
  int32_t launches;           // 0: one or two launches by size; 1 or 2: that many (tests)
  unsigned int* sync;         // 2 x 4 x 64 counters (A lists, B lists, group barriers, Q list
                              // of each of the prologue's two launches), zeroed
  uint32_t* status;
  uint64_t timeout_ns;        // bound of every wait
  int32_t v16;                // write V as fp16 (FP16-PV variant) instead of e4m3
};

cudaError_t launch_prologue(const SegGeo& g, const PrologueBuffers& b,
                            bool vec, cudaStream_t st);

// Largest nseg * Hkv * Dp served by the allocation-free statistics call.
constexpr int64_t kStaticStatEntries = 16384;

// K channel means and V channel scales of a dense call, with the scratch
// accumulators in a static device array instead of a caller workspace.
cudaError_t launch_kv_stats_static(const SegGeo& g, const uint16_t* k,
                                   const uint16_t* v, float* k_mean, float* s_v,
                                   bool vec, uint64_t timeout_ns, cudaStream_t st);

// Reads (synchronising st) the status word at the start of that static
// array on the current device.
cudaError_t read_kv_stats_static_status(uint32_t* word, cudaStream_t st);

struct AttnParams {
  SegGeo g;
  const float* s_q;
  const float* s_k;
  const float* s_v;
  float* out;
  // output addressing in elements; varlen segments start at cu_q[s]*tok
  int64_t out_seg_stride, out_head_stride, out_tok_stride;
  float scale_log2;          // sm_scale * log2(e)
  float one;                 // 1.0f: the multiplier of the FMA that subtracts the row
                             // max from a rounded logit (a run-time value, so the
                             // compiler cannot fuse that subtraction with the product)
  int32_t causal;
  int32_t skip_kv_tile;      // failure-injection hook, -1 = off
  int32_t v16;               // FP16-PV variant: V and P~ in fp16, single-stage K and V rings
  int32_t out_tma;           // output map: 0 none (per-row stores), 1 dense HND,
                             // 2 dense NHD, 3 packed (varlen)
  int32_t flat_pairs;        // >= 0: 1D grid of this many pairs, then single tiles;
                             // -1: (pair, head, segment) grid (set by the launcher)
  uint64_t timeout_ns;
  uint32_t* status;
};

struct AttnMaps {
  CUtensorMap q, k, v;
  CUtensorMap o;             // fp32 output, 32-column boxes of 128 rows (see out_tma)
};

cudaError_t launch_attention(const AttnMaps& maps, const AttnParams& p,
                             cudaStream_t st);

cudaError_t launch_debug_qk(const AttnMaps& maps, const AttnParams& p,
                            int64_t q_row0, int64_t k_row0, int32_t* out,
                            cudaStream_t st);

cudaError_t launch_debug_pv(const uint8_t* p8, const uint8_t* v8, int64_t ntiles, int64_t Dp,
                            float* out, uint32_t* status, uint64_t timeout_ns,
                            cudaStream_t st);

cudaError_t launch_tc_rate(int kind, int64_t n_mma, uint32_t* status, uint64_t timeout_ns,
                           cudaStream_t st);

cudaError_t launch_debug_e4m3(const float* in, uint8_t* out, int64_t n,
                              cudaStream_t st);

}  // namespace sage
