// Geometry of one call, shared by the host launcher and the kernels: where a
// (segment, head, token) lives in the caller's tensors and in the workspace.
// A segment is a batch entry (dense) or a packed sequence (varlen).
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define SAGE_HD __host__ __device__ __forceinline__
#else
#define SAGE_HD inline
#endif

namespace sage {

// Status bits of the workspace's device status word.
constexpr uint32_t kStatusTimeout = 1u;      // a bounded wait ran out
constexpr uint32_t kStatusBadSeqlens = 2u;   // cu_seqlens inconsistent
constexpr uint32_t kStatusBadItem = 4u;      // a work item decoded outside the call's plan

struct SegGeo {
  int64_t nseg, Hq, Hkv, Lq, Lk, D, Dp;
  int32_t dtype, varlen;
  int32_t strided;            // dense inputs given as arbitrary views (per-tensor strides)
  const int32_t* cu_q;
  const int32_t* cu_k;
  int64_t total_q, total_k;
  int32_t max_q, max_k;
  // caller tensors, in elements
  int64_t q_seg_stride, q_head_stride, q_tok_stride;
  int64_t k_seg_stride, k_head_stride, k_tok_stride;   // shared by k and v
  // workspace rows
  int64_t q_head_rows, k_head_rows, v_cols;
};

SAGE_HD int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

#ifdef __CUDACC__
// Segment bounds; for varlen, validates cu_seqlens entries against the
// totals and the declared maxima.  Returns false (and sets the status bit)
// on an inconsistent entry.
__device__ __forceinline__ bool seg_range(const int32_t* cu, int64_t s,
                                          int64_t total, int32_t maxlen,
                                          int64_t* start, int64_t* len) {
  const int64_t a = cu[s], b = cu[s + 1];
  if (a < 0 || b < a || b > total || b - a > maxlen) return false;
  *start = a;
  *len = b - a;
  return true;
}
#endif

// Workspace row of token 0 of head 0 of a segment (rows of Dp elements).
SAGE_HD int64_t ws_seg_base(int varlen, int64_t s, int64_t start, int64_t H,
                            int64_t head_rows) {
  return varlen ? 128 * (s + start / 128) : s * H * head_rows;
}

}  // namespace sage
