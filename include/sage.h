/*
 * sage.h - C ABI of the GB300 (sm_103a) smoothed quantized attention library.
 *
 * The method (SageAttention2/2++-style quantized attention) is described on
 * these pages, cited below by title and section:
 *   [SD] stable-diffusion.cpp, docs "SageAttention": kernel-selection table
 *        (per-thread INT8 Q/K, FP8 PV, FP32 buffer), FP8-path paragraph
 *        (smooth K, per-channel V, pad and permute V, FP32 output), "Use"
 *        section (head_dim 1..128 zero-padded to 64/128, original softmax
 *        scale, cropped output, GQA, different q/kv lengths, batches) and
 *        the error convention (an unavailable feature reports an error).
 *   [OV] "SageAttention: Quantized Attention Library", Core features
 *        (INT8 QK^T per token/thread, FP8 PV, K smoothing, varlen, GQA).
 *   [RM] SageAttention README translation, usage section (q, k, v fp16/bf16,
 *        tensor_layout "HND" (B,H,L,D) or "NHD" (B,L,H,D), is_causal).
 *   [RD] SageAttention-RDNA4 releases, v0.4.0 (hand-written prologue, key
 *        mean summed in fp64, 64-bit offsets) and v0.3.0 (fused q/k/v views;
 *        a refusal carries its reason).
 *   [WH] SageAttention 2.2.0 sm_120a wheel page, accuracy section (the
 *        backends' errors against float64 attention).
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers of the current CUDA device and
 *    are owned by the caller (the host-buffer calls sage_attn_fwd_host,
 *    sage_attn_fwd_host_pv16 and sage_attn_fwd_varlen_host take host
 *    buffers instead).  The library allocates no memory, never synchronises
 *    the host and enqueues all work on the caller's stream (the host-buffer
 *    calls add copies on two streams of their own, ordered by events).
 *  - Arguments are validated on the host before anything is enqueued; a bad
 *    argument returns an error and launches nothing.  The reason is kept in
 *    a thread-local string returned by sage_last_error().
 *  - Inputs q, k, v are fp16 or bf16, densely packed (the *_strided calls
 *    also take views with their own strides).
 *    Dense calls take HND (B,H,L,D) or NHD (B,L,H,D); varlen calls take
 *    packed (T,H,D) with int32 cumulative sequence offsets.
 *  - The output is fp32 in the same layout as q, with the caller's D
 *    (padding channels are never written).
 *  - D is 1..128; Hq must be a multiple of Hkv (query head h reads kv head
 *    h / (Hq/Hkv)).  sm_scale <= 0 selects 1/sqrt(D).
 *  - is_causal masks key j for query i when j > i (top-left alignment).
 *  - Failures detected on the device (a bounded wait that ran out, an
 *    inconsistent cu_seqlens array) are recorded in a status word at the
 *    start of the workspace; sage_device_status() reads it.
 */
#ifndef SAGE_H_
#define SAGE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SAGE_API __attribute__((visibility("default")))
#else
#define SAGE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* sage_stream_t;

typedef enum {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = 1,    /* bad pointer, size, enum or alignment      */
  SAGE_ERR_UNSUPPORTED = 2,    /* valid request this build does not serve   */
  SAGE_ERR_WORKSPACE = 3,      /* workspace too small or misaligned         */
  SAGE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed         */
  SAGE_ERR_DEVICE_TIMEOUT = 5  /* a device-side bounded wait ran out        */
} sage_status;

enum { SAGE_HND = 0, SAGE_NHD = 1 };
enum { SAGE_F16 = 0, SAGE_BF16 = 1 };

/* Quantised operands produced by the prologue; every pointer points into
 * the caller's workspace.  Layout (Dp = 64 if D <= 64 else 128; all token
 * counts padded to multiples of 128 per (segment, head), padding zeroed):
 *   q16  : [q_rows][Dp] fp16 holding the int8 codes of Q (exact integers)
 *   k16  : [k_rows][Dp] fp16 holding the int8 codes of smoothed K
 *          (sm_103a has no 8-bit integer tensor-core MMA, so QK^T runs on
 *          the 16-bit kind, whose operands these are: each int8 code n,
 *          -127..127, is stored as the exact fp16 value n, so q16 and k16
 *          are the quantised Q and K codes themselves, one-to-one)
 *   v8   : [v_rows][v_cols] e4m3 codes of V, channel-major ("permuted"):
 *          row = (segment base) + kv_head*Dp + channel, column = token
 *   s_q  : [q_rows] fp32, one scale per query token
 *   s_k  : [k_rows/128] fp32, one scale per 128-token key block
 *   s_v  : [nseg][Hkv][Dp] fp32, one scale per value channel
 *   k_mean: [nseg][Hkv][Dp] fp32, the per-channel token mean of K
 * Row of token t of head h in segment s: dense  (s*H + h)*L_pad + t,
 *                                        varlen h*T_pad + base(s) + t with
 * base(s) = 128*(s + cu[s]/128) and T_pad = 128*(nseg + total/128).       */
typedef struct {
  int64_t nseg, Hq, Hkv, Lq, Lk, D, Dp;
  int32_t dtype, varlen;
  int64_t total_q, total_k;         /* varlen packed token totals        */
  int32_t max_q, max_k;             /* varlen length upper bounds        */
  int64_t q_head_rows, k_head_rows; /* L_pad (dense) or T_pad (varlen)   */
  int64_t q_rows, k_rows, v_rows, v_cols;
  const int32_t* cu_q;              /* varlen only (device), else NULL   */
  const int32_t* cu_k;
  void* q16;
  void* k16;
  void* v8;
  float* s_q;
  float* s_k;
  float* s_v;
  float* k_mean;
  void* stats;                      /* per-channel accumulators          */
  uint32_t* status;                 /* device status word (workspace+0)  */
  int32_t v_fp16;                   /* 1: v8 holds fp16 V (FP16-PV), no s_v */
} sage_quantized;

/* Workspace bytes for a dense call (HND or NHD).  Returns 0 for invalid
 * sizes.  The workspace must be 256-byte aligned. */
SAGE_API size_t sage_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq,
                            int64_t Lk, int64_t D);

/* Workspace bytes for a packed varlen call with nseq sequences and total_q
 * query / total_k key tokens. */
SAGE_API size_t sage_workspace_bytes_varlen(int64_t nseq, int64_t total_q,
                                   int64_t total_k, int64_t Hq, int64_t Hkv,
                                   int64_t D);

/* Quantisation prologue ([SD] FP8-path paragraph; [OV] Core features; [RD]
 * v0.4.0): pads D to Dp, smooths K by its exact per-channel token mean
 * (the sum is exact, rounded once to fp64), quantises Q to int8 per token
 * and smoothed K per 128-token block, V to e4m3 per channel (largest
 * magnitude -> 448), and writes V channel-major for the tensor cores.
 * Fills *qt with pointers into ws.  q,k,v: dense tensors in `layout`. */
SAGE_API sage_status sage_quant_prologue(const void* q, const void* k, const void* v,
                                int dtype, int layout, int64_t B, int64_t Hq,
                                int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D,
                                void* ws, size_t ws_bytes, sage_quantized* qt,
                                sage_stream_t stream);

/* Varlen prologue: q (total_q,Hq,D), k/v (total_k,Hkv,D); cu_seqlens_q/k are
 * device int32 arrays of nseq+1 non-decreasing offsets starting at 0 and
 * ending at total_q/total_k; max_q/max_k bound every sequence length. */
SAGE_API sage_status sage_quant_prologue_varlen(
    const void* q, const void* k, const void* v, int dtype,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t nseq,
    int64_t total_q, int64_t total_k, int max_q, int max_k, int64_t Hq,
    int64_t Hkv, int64_t D, void* ws, size_t ws_bytes, sage_quantized* qt,
    sage_stream_t stream);

/* Prologue on strided views ([RD] v0.3.0, "Fused q/k/v views"): q, k and v
 * may be views into larger tensors, such as the three slices of one fused
 * projection, whose token stride is then 3*H*D instead of H*D.
 *   q_strides : host int64[3], q's {batch, head, token} strides in elements;
 *   kv_strides: host int64[3], the same for k and v, which share them;
 *   the channel stride is 1 and every other stride must be positive.
 * Views with a 16-byte aligned base, strides that are multiples of 8
 * elements and D % 8 == 0 are copied by the tensor engine; any other
 * positive strides are read element by element.  A view this call cannot
 * serve is refused before any launch with SAGE_ERR_UNSUPPORTED (or
 * SAGE_ERR_INVALID_ARG for missing strides) and the reason in
 * sage_last_error(); nothing falls back silently.  The workspace
 * (sage_workspace_bytes) and the quantised operands are those of
 * sage_quant_prologue. */
SAGE_API sage_status sage_quant_prologue_strided(
    const void* q, const void* k, const void* v, int dtype, int64_t B, int64_t Hq,
    int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D, const int64_t* q_strides,
    const int64_t* kv_strides, void* ws, size_t ws_bytes, sage_quantized* qt,
    sage_stream_t stream);

/* FP16-PV prologue ([OV] API list, sageattn_qk_int8_pv_fp16_cuda: INT8
 * QK^T, FP16 PV; [WH] accuracy table: the most accurate backend).  As
 * sage_quant_prologue, except that V is kept in fp16 instead of e4m3: each
 * value rounded to nearest even (exact for fp16 inputs), no per-channel
 * scale, stored channel-major like the e4m3 V (2 bytes per element; the
 * workspace of sage_workspace_bytes has room for it).  Sets qt->v_fp16 = 1,
 * which makes sage_attn_quantized run the FP16-PV kernel.  Dense inputs. */
SAGE_API sage_status sage_quant_prologue_pv16(const void* q, const void* k, const void* v,
                                     int dtype, int layout, int64_t B, int64_t Hq,
                                     int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D,
                                     void* ws, size_t ws_bytes, sage_quantized* qt,
                                     sage_stream_t stream);

/* Fused attention on quantised operands ([SD] kernel table: INT8 QK^T,
 * FP8 PV with an fp32 accumulator; [OV] Core features): per 128x128 tile,
 * exact integer S = q8 k8^T on the tensor cores, logits S*s_q*s_k*sm_scale
 * in base 2, -inf masking, online softmax in fp32, P quantised to e4m3 as
 * 448*P, O += P~ V~ accumulated in fp32 tensor memory, and
 * out = O * s_v / (448 * l) in fp32.  `layout` is the dense output layout
 * (ignored for varlen, which writes packed (total_q,Hq,D)). */
/* (With qt->v_fp16 set, the FP16-PV kernel runs instead: the same INT8
 * QK^T and online softmax, P~ = fp16(P) without the 448 scaling, O += P~ V16
 * in fp32 tensor memory, out = O / l.) */
SAGE_API sage_status sage_attn_quantized(const sage_quantized* qt, float* out,
                                int layout, int is_causal, float sm_scale,
                                sage_stream_t stream);

/* Prologue + attention in one call (dense). */
SAGE_API sage_status sage_attn_fwd(const void* q, const void* k, const void* v,
                          float* out, int64_t B, int64_t Hq, int64_t Hkv,
                          int64_t Lq, int64_t Lk, int64_t D, int layout,
                          int is_causal, float sm_scale, int dtype, void* ws,
                          size_t ws_bytes, sage_stream_t stream);

/* Prologue + FP16-PV attention in one call (dense; see
 * sage_quant_prologue_pv16). */
SAGE_API sage_status sage_attn_fwd_pv16(const void* q, const void* k, const void* v,
                               float* out, int64_t B, int64_t Hq, int64_t Hkv,
                               int64_t Lq, int64_t Lk, int64_t D, int layout,
                               int is_causal, float sm_scale, int dtype, void* ws,
                               size_t ws_bytes, sage_stream_t stream);

/* Host-buffer call: sage_attn_fwd on q, k, v and out in HOST memory (dense
 * HND or NHD, same arguments and conventions), with the host<->device copies
 * inside.  The operation is sage_attn_fwd's (the prologue of
 * sage_quant_prologue, then sage_attn_quantized; [SD] kernel table, [OV]
 * Core features); the chunking and copy pipeline are this library's own and
 * have no counterpart on the pages.  The problem is cut into chunks of (one batch entry, chunk_kv_heads
 * kv heads with their query heads); 0 picks enough kv heads for one wave of
 * query-tile pairs per chunk.  Chunk i+1's inputs are copied into device
 * staging while chunk i is computed on `stream` and chunk i-1's output is
 * copied back, on two copy streams the library creates once per device and
 * keeps.  Attention never mixes heads or batch entries, so the output equals
 * one sage_attn_fwd call's.
 *   ws: device workspace of sage_workspace_bytes_host(...) bytes (the chunk
 *       prologue's workspace and two staging slots).
 *   Host buffers should be page-locked for the copies to overlap; the call
 *   returns once everything is enqueued, and `stream` completes when every
 *   output row is in `out`.  Calls on one device enqueue one at a time.
 *   Lk = 0 is refused (use sage_attn_fwd); B = 0 or Lq = 0 does nothing.
 *   Device-side failures of every chunk accumulate in the status word at
 *   the start of ws (the first chunk clears it, later chunks keep it), so
 *   sage_device_status(ws, stream) after the call reports a bounded wait
 *   that ran out in any chunk. */
SAGE_API size_t sage_workspace_bytes_host(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq,
                                          int64_t Lk, int64_t D, int64_t chunk_kv_heads);
SAGE_API sage_status sage_attn_fwd_host(const void* q, const void* k, const void* v,
                                        float* out, int64_t B, int64_t Hq, int64_t Hkv,
                                        int64_t Lq, int64_t Lk, int64_t D, int layout,
                                        int is_causal, float sm_scale, int dtype,
                                        int64_t chunk_kv_heads, void* ws, size_t ws_bytes,
                                        sage_stream_t stream);

/* The same host-buffer pipeline around the FP16-PV variant
 * (sage_attn_fwd_pv16); same workspace size. */
SAGE_API sage_status sage_attn_fwd_host_pv16(const void* q, const void* k, const void* v,
                                             float* out, int64_t B, int64_t Hq, int64_t Hkv,
                                             int64_t Lq, int64_t Lk, int64_t D, int layout,
                                             int is_causal, float sm_scale, int dtype,
                                             int64_t chunk_kv_heads, void* ws,
                                             size_t ws_bytes, sage_stream_t stream);

/* Host-buffer call for packed sequences: sage_attn_fwd_varlen on q, k, v
 * (packed (T,H,D)) and out (packed (total_q,Hq,D) fp32) in HOST memory, with
 * cu_seqlens_q and cu_seqlens_k (nseq + 1 int32 each) in host memory too.
 * The operation is sage_attn_fwd_varlen's ([OV] "variable-length sequences
 * via sageattn_varlen"); the pipeline is sage_attn_fwd_host's, with chunks
 * of chunk_kv_heads kv heads (and their query heads) of the whole packed
 * tensor, every sequence at once; 0 picks enough kv heads for four waves
 * of query-tile pairs per chunk (a chunk lasts at least as long as a pair of
 * its longest sequence).  The offsets are checked on the host (start at
 * 0, end at the totals, every length in 0..max) and copied once into the
 * workspace, so they may live in ordinary host memory; a bad array returns
 * SAGE_ERR_INVALID_ARG and enqueues nothing.  The output equals one
 * sage_attn_fwd_varlen call's.
 *   ws: device workspace of sage_workspace_bytes_varlen_host(...) bytes (0
 *       for invalid sizes).
 *   nseq = 0 or total_q = 0 does nothing; total_k = 0 is refused (use
 *   sage_attn_fwd_varlen).  The status word behaves as for
 *   sage_attn_fwd_host. */
SAGE_API size_t sage_workspace_bytes_varlen_host(int64_t nseq, int64_t total_q,
                                                 int64_t total_k, int64_t Hq, int64_t Hkv,
                                                 int64_t D, int64_t chunk_kv_heads);
SAGE_API sage_status sage_attn_fwd_varlen_host(
    const void* q, const void* k, const void* v, float* out, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, int64_t nseq, int64_t total_q, int64_t total_k, int max_q,
    int max_k, int64_t Hq, int64_t Hkv, int64_t D, int is_causal, float sm_scale, int dtype,
    int64_t chunk_kv_heads, void* ws, size_t ws_bytes, sage_stream_t stream);

/* Prologue + attention in one call on strided views (see
 * sage_quant_prologue_strided); out is dense fp32 in `layout`. */
SAGE_API sage_status sage_attn_fwd_strided(
    const void* q, const void* k, const void* v, float* out, int64_t B, int64_t Hq,
    int64_t Hkv, int64_t Lq, int64_t Lk, int64_t D, const int64_t* q_strides,
    const int64_t* kv_strides, int layout, int is_causal, float sm_scale, int dtype,
    void* ws, size_t ws_bytes, sage_stream_t stream);

/* Prologue + attention in one call (packed varlen, [OV] "variable-length
 * sequences via sageattn_varlen"). */
SAGE_API sage_status sage_attn_fwd_varlen(
    const void* q, const void* k, const void* v, float* out,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t nseq,
    int64_t total_q, int64_t total_k, int max_q, int max_k, int64_t Hq,
    int64_t Hkv, int64_t D, int is_causal, float sm_scale, int dtype,
    void* ws, size_t ws_bytes, sage_stream_t stream);

/* Debug: the exact INT32 QK^T tile (128x128, row-major) of query tile
 * `qtile` and key tile `ktile` of head `hq` in segment `seg`, computed with
 * the attention kernel's own tensor-core path and converted from the fp32
 * accumulator with round-toward-zero.  out: device int32[128*128]. */
SAGE_API sage_status sage_debug_qk_int32(const sage_quantized* qt, int64_t seg,
                                int64_t hq, int64_t qtile, int64_t ktile,
                                int32_t* out, sage_stream_t stream);

/* Debug: the precision of the PV accumulator ([SD] kernel table: the FP8
 * PV products accumulate into an fp32 buffer).  Computes
 *   out[r][c] = sum over t < ntiles, j < 128 of P~_t[r][j] * V~_t[c][j]
 * with the attention kernel's own PV instructions (tcgen05 kind::f8f6f4,
 * e4m3 x e4m3, M=128, N=Dp, K=32 per instruction, accumulating in tensor
 * memory; the first instruction overwrites), so that tests can compare the
 * hardware's sums with exact ones.
 *   p8    : device e4m3 codes [ntiles][128 rows][128 keys], 16-byte aligned;
 *   v8    : device e4m3 codes [ntiles][Dp channels][128 keys] (the prologue's
 *           channel-major V), 16-byte aligned;
 *   ntiles: 1..4096 key tiles of 128 keys; Dp: 64 or 128;
 *   out   : device fp32 [128][Dp];
 *   status: a device word the call clears and the kernel sets if its bounded
 *           wait runs out (read it with sage_device_status(status, stream)). */
SAGE_API sage_status sage_debug_pv_accum(const uint8_t* p8, const uint8_t* v8, int64_t ntiles,
                                         int64_t Dp, float* out, uint32_t* status,
                                         sage_stream_t stream);

/* Measurement: the tensor pipe's rate for the attention kernel's two MMA
 * kinds, at the clock the GPU runs at the time (no counterpart on the
 * pages; the benchmark reports its kernel against it).  Launches one CTA
 * per SM, in which one thread issues n_mma back-to-back tcgen05 MMAs of
 * shape M=128 N=128 into one tensor-memory accumulator: kind 0 = fp16
 * operands, K=16 (2*128*128*16 flops each, the QK^T kind); kind 1 = e4m3
 * operands, K=32 (twice that, the PV kind).  Operands are zeros; nothing is
 * returned but the time the caller measures around the call (events on
 * `stream`).  n_mma: 1..2^22.  status: a device word the call clears and
 * the kernel sets if its bounded wait runs out (sage_device_status). */
SAGE_API sage_status sage_debug_tc_rate(int kind, int64_t n_mma, uint32_t* status,
                                        sage_stream_t stream);

/* Debug: the attention kernel's fp32 -> e4m3 conversion (round to nearest
 * even, saturating to +-448) applied to n device floats. */
SAGE_API sage_status sage_debug_e4m3(const float* in, uint8_t* out, int64_t n,
                            sage_stream_t stream);

/* Debug hook for failure-detection tests: the next attention launches skip
 * loading key/value tile `skip_kv_tile` (-1: off) so that the consumer's
 * bounded wait runs out after `timeout_ns` (0: default of one second). */
SAGE_API void sage_debug_set_fault(int skip_kv_tile, uint64_t timeout_ns);

/* Debug hook: the fault set by sage_debug_set_fault applies to the next
 * `launches` attention launches only (so that a test can fail one chunk of
 * a host-buffer call); -1, the default, applies it to every launch. */
SAGE_API void sage_debug_set_fault_launches(int launches);

/* Test hook: the prologue entry points run as one launch (1), as two
 * launches (2: Q tiles and K/V statistics, then K/V tiles), or choose (0,
 * the default: one launch, measured as fast or faster at every size).  Other
 * values mean 0.  The results are identical either way; the hook lets tests
 * cover both plans at any size. */
SAGE_API void sage_debug_set_prologue_launches(int launches);

/* Test hook: the host-buffer calls (sage_attn_fwd_host, _host_pv16,
 * sage_attn_fwd_varlen_host) treat chunk `chunk` (0-based, in order) as if
 * its launch had failed: they enqueue nothing for it or after it and return
 * SAGE_ERR_INVALID_ARG, after making the caller's stream wait for the
 * copies of the earlier chunks, as they do on any failure.  -1, the
 * default, turns it off. */
SAGE_API void sage_debug_set_host_fail_chunk(int chunk);

/* Reads (synchronising `stream`) the device status word of workspace ws:
 * SAGE_OK, SAGE_ERR_DEVICE_TIMEOUT, SAGE_ERR_INVALID_ARG, or
 * SAGE_ERR_UNSUPPORTED for an internal inconsistency the prologue caught
 * (a work item outside the call's plan, skipped).  The prologue clears it;
 * the kernels only set bits. */
SAGE_API sage_status sage_device_status(const void* ws, sage_stream_t stream);

/* Allocation-free smoothing statistics (the pages have no counterpart: an
 * addition of this library).  For callers that may not allocate device
 * memory at all, not even a workspace: code running inside a host framework
 * that owns every device allocation and forbids its extensions to allocate,
 * or a latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation and unbounded cost.  Computes, for a dense K and V (HND
 * or NHD, fp16/bf16), the same per-channel K token mean and V scale
 * (max |v| / 448) as sage_quant_prologue, into caller-owned k_mean and s_v,
 * each [B][Hkv][Dp] fp32 (Dp = 64 if D <= 64 else 128; padded channels 0).
 * Its scratch accumulators live in one static device array inside the
 * library, sized for B*Hkv*Dp <= 16384 channel slots (about 256 KB, held by
 * every GPU that loads the library until the process exits); larger
 * problems return SAGE_ERR_UNSUPPORTED.  The first call on each device looks
 * up the array's device address (a one-time set-up); make that first call
 * before any stream capture.  Every call clears and reuses the same array,
 * so calls that overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.  It calls no cudaMalloc or
 * cudaFree.  Failures on the device (a bounded wait that ran out, for
 * instance because an overlapping call took the array's counters) are
 * recorded in a status word at the start of the array, which every call
 * clears; sage_kv_stats_noalloc_status reads it. */
SAGE_API sage_status sage_kv_stats_noalloc(const void* k, const void* v, int dtype,
                                           int layout, int64_t B, int64_t Hkv,
                                           int64_t Lk, int64_t D, float* k_mean,
                                           float* s_v, sage_stream_t stream);

/* Reads (synchronising `stream`) the device status word of the last
 * sage_kv_stats_noalloc call on the current device: SAGE_OK, or
 * SAGE_ERR_DEVICE_TIMEOUT when a bounded wait ran out (k_mean and s_v may
 * then be partial), or SAGE_ERR_UNSUPPORTED for an internal inconsistency.
 * Like the statistics call, it allocates nothing; the pages have no
 * counterpart. */
SAGE_API sage_status sage_kv_stats_noalloc_status(sage_stream_t stream);

/* Reason of the last failure on this thread ("" if none). */
SAGE_API const char* sage_last_error(void);

/* Instrumentation (no counterpart in the pages): the number of kernels this
 * library has launched in this process, all devices and threads, counted on
 * the host as each launch is issued.  The difference across a region gives
 * the kernels issued inside it.  Never fails. */
SAGE_API uint64_t sage_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SAGE_H_ */
