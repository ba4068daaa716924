/* gla.h - C ABI of the GB300 Simple GLA mixer library (libgla.so).
 *
 * What it computes.  Source: "Beyond the KV cache: Training and serving i14's Laplace 3B linear
 * attention model on AWS Trainium2 with native PyTorch" (AWS blog post; Spanish and Chinese
 * copies carry the later sections and the figure captions).
 *   - Section "i14 and the Laplace 3B architecture", paragraph "GLA mixer": every head h keeps a
 *     d_k x d_v = 96 x 192 matrix state, decayed by a fixed per-head factor lambda_h and written
 *     with the rank-1 outer product of the current key and value; the readout queries the state.
 *     The equation images are missing from the text; this library computes
 *         S_t = lambda_h * S_{t-1} + k_t v_t^T ,      o_t = S_t^T (scale * q_t)
 *     with the readout after the update, S_0 = h0 (zeros when h0 is NULL) and hT = S_T.
 *   - Section "Challenge 1: Using native PyTorch on Trainium for GLA": the chunked form with
 *     128-token chunks (intra-chunk masked linear attention plus the carried state; the state
 *     advances with lambda^C, the decay compounded over the chunk).  gla_chunk_fwd computes that
 *     form; its result equals the recurrence above up to rounding.
 *   - Section "Challenge 3" (backward through the sequential state updates): gla_chunk_bwd is the
 *     adjoint of the recurrence.  lambda is fixed at initialisation, not learned ("Decay
 *     schedule"), so there is no gradient for it.
 *   - Section "Optimizing inference on Trainium2" (a wrapper reads and writes each sequence's
 *     recurrent state in a pool, one fixed page per sequence): gla_decode_step advances a pool of
 *     states by one token in place.
 *
 * Conventions shared by every entry point.
 *   - Sizes: only d_k = 96 and d_v = 192 are implemented; other values return
 *     GLA_ERR_UNSUPPORTED.  H >= 1.  Chunk size is 128 tokens (GLA_CHUNK).
 *   - Pointers are DEVICE pointers owned by the caller, 16-byte aligned (else GLA_ERR_ALIGN),
 *     except where a comment says "host".  The library never allocates, frees or keeps them.
 *   - Layouts are dense, C order, token-major:
 *       q, k     [n_seq, T, H, 96]   (or packed [T_total, H, 96] with cu_seqlens)
 *       v, o, dO [n_seq, T, H, 192]  (or packed [T_total, H, 192])
 *       h0, hT, dhT, dh0, state  [n_seq (or pool rows), H, 96, 192], always fp32
 *       log_lambda [H] fp32: natural log of lambda_h, <= 0 (-inf allowed: lambda = 0)
 *   - dtype (gla_dtype) is the type of q, k, v, o, dO, dq, dk, dv.  GLA_BF16 runs the tensor-core
 *     kernels (bf16 operands, fp32 accumulation and fp32 state); results are rounded to bf16
 *     nearest-even.  GLA_F32 runs the all-fp32 CUDA-core kernels.
 *   - scale multiplies q (1/sqrt(96) in the Laplace 3B configuration).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Argument errors are detected on the host before anything is launched and return a negative
 *     gla_status; nothing aborts the process.  Faults found while a kernel runs (a bounded wait
 *     that timed out, a pool slot out of range) set a sticky per-device error word that
 *     gla_get_device_error() reports.
 *   - Empty work is valid: n_seq = 0, T = 0 or sequences of length 0 launch nothing for them;
 *     a length-0 sequence gives hT = h0 (zeros if h0 is NULL) and dh0 = dhT.
 *   - The library looks up the device addresses of its own device variables (the error word,
 *     the hand-over flags, the array of gla_chunk_fwd_noalloc) once per device and keeps them,
 *     and creates a few CUDA objects per device that live until the process exits (the
 *     backward's two side streams; the host-buffer forward's two copy streams and its events),
 *     so resetting a device (cudaDeviceReset) after the library's first call on it is not
 *     supported.
 */
#ifndef GLA_H_
#define GLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gla_stream_t; /* identical to cudaStream_t */

typedef enum {
  GLA_OK = 0,
  GLA_ERR_NULL = -1,        /* a required pointer is NULL */
  GLA_ERR_SHAPE = -2,       /* negative size, bad cu_seqlens, pool slot out of range, or
                               n_seq * H * 96 or the token count reaches 2^31 */
  GLA_ERR_DTYPE = -3,       /* dtype is not a gla_dtype */
  GLA_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned */
  GLA_ERR_UNSUPPORTED = -5, /* d_k != 96, d_v != 192, or no sm_103 device current */
  GLA_ERR_WORKSPACE = -6,   /* workspace missing or smaller than gla_workspace_bytes() */
  GLA_ERR_LAUNCH = -7,      /* the CUDA runtime refused a launch */
  GLA_ERR_TIMEOUT = -8,     /* a bounded device-side wait gave up (kernel returned early) */
  GLA_ERR_BOUNDS = -9       /* debug-bounds build only: a device index fell outside its buffer
                               (the access was skipped; see gla_debug_bounds) */
} gla_status;

typedef enum { GLA_BF16 = 0, GLA_F32 = 1 } gla_dtype;

#define GLA_DK 96
#define GLA_DV 192
#define GLA_CHUNK 128

/* Bytes of device workspace that gla_chunk_fwd / gla_chunk_bwd need for `n_seq` packed
 * (cu_seqlens) sequences of H heads.  The workspace holds the longest-first schedule of the
 * (sequence, head) work.  Calls without cu_seqlens need none (pass NULL, 0). */
size_t gla_workspace_bytes(int n_seq, int H);

/* Chunked forward.
 *   q, k, v      inputs (layouts above), dtype `dtype`.
 *   log_lambda   [H] fp32 device.
 *   h0           [n_seq, H, 96, 192] fp32, or NULL for zero initial states.
 *   scale        multiplies q.
 *   o            output, same dtype and layout as v.
 *   hT           [n_seq, H, 96, 192] fp32 final states, or NULL to skip.
 *   cu_seqlens   NULL: n_seq sequences of T tokens each, layout [n_seq, T, H, d].
 *                else: [n_seq + 1] int32 device array of packed offsets, cu_seqlens[0] = 0,
 *                non-decreasing, cu_seqlens[n_seq] = T (the packed total); its values are read on
 *                the device only (no host synchronisation), so the caller guarantees them.
 *   workspace    >= gla_workspace_bytes(n_seq, H) bytes when cu_seqlens != NULL, else unused.
 * Returns GLA_OK once the work is queued on `stream`. */
int gla_chunk_fwd(const void* q, const void* k, const void* v, const float* log_lambda,
                  const float* h0, float scale, void* o, float* hT, const int32_t* cu_seqlens,
                  int n_seq, int T, int H, int dk, int dv, int dtype, void* workspace,
                  size_t ws_bytes, gla_stream_t stream);

/* Chunked forward with the self-augmentation step ("Beyond the KV cache", section "i14 and the
 * Laplace 3B architecture", the paragraph after the state readout): every output row also gains
 * a gated copy of its own value,
 *     o_t += sigmoid(q_t . (a_h * k_t)) v_t,
 * with a_h the head's aug_balance (a learned rescaling of the key's channels; a = 0 gives the
 * half-strength copy 0.5 v_t).  The query enters the gate unscaled.
 *   aug          [H, 96] fp32 device (non-NULL, 16-byte aligned); a NULL aug returns GLA_ERR_NULL.
 *   every other argument, and the results, as in gla_chunk_fwd (hT is not affected: the copy
 *   adds to the output only).
 * gla_chunk_bwd differentiates the mixer without this step. */
int gla_chunk_fwd_aug(const void* q, const void* k, const void* v, const float* log_lambda,
                      const float* h0, float scale, const float* aug, void* o, float* hT,
                      const int32_t* cu_seqlens, int n_seq, int T, int H, int dk, int dv, int dtype,
                      void* workspace, size_t ws_bytes, gla_stream_t stream);

/* Bytes of device workspace that gla_chunk_bwd needs; n_seq, T, H as in that call, packed != 0
 * when cu_seqlens is given, dtype the gla_dtype.  In bf16 mode the workspace holds fp32 partial
 * sums of dq and dk (2 x T_total x H x 96 x 4 bytes) plus the packed schedule; in fp32 mode only
 * the packed schedule (0 extra bytes for fixed-length calls). */
size_t gla_bwd_workspace_bytes(int n_seq, int T, int H, int packed, int dtype);

/* Chunked backward: gradients of L(o, hT) given dO = dL/do and dhT = dL/dhT.
 *   q, k, v, log_lambda, h0, scale, cu_seqlens, n_seq, T, H, dtype: as in gla_chunk_fwd
 *                (h0 NULL = zeros).
 *   dO           same dtype and layout as v.
 *   dhT          [n_seq, H, 96, 192] fp32, or NULL for zero.
 *   dq, dk       outputs, layout of q; dv output, layout of v; all of dtype `dtype`.
 *   dh0          [n_seq, H, 96, 192] fp32 output, or NULL to skip.
 *   workspace    >= gla_bwd_workspace_bytes(n_seq, T, H, cu_seqlens != NULL, dtype) bytes.
 * The forward state is recomputed on chip; nothing from gla_chunk_fwd is needed.  In bf16 mode dv
 * and dh0 come from one reverse scan, dq and dk from scans over each 64-column tile of d_v whose
 * fp32 partial sums meet in the workspace before the final bf16 rounding. */
int gla_chunk_bwd(const void* q, const void* k, const void* v, const float* log_lambda,
                  const float* h0, float scale, const void* dO, const float* dhT, void* dq,
                  void* dk, void* dv, float* dh0, const int32_t* cu_seqlens, int n_seq, int T,
                  int H, int dk_size, int dv_size, int dtype, void* workspace, size_t ws_bytes,
                  gla_stream_t stream);

/* One decode step for N sequences, in place on a state pool.
 *   q, k         [N, H, 96]; v, o [N, H, 192]; dtype `dtype`.
 *   state        [pool_rows, H, 96, 192] fp32, updated in place: S <- lambda S + k v^T.
 *   slot         [N] int32 device array: sequence n uses pool row slot[n]; NULL = row n
 *                (then pool_rows >= N is required).  Rows must be distinct.  A slot outside
 *                [0, pool_rows) skips that sequence (state and o untouched) and records
 *                GLA_ERR_SHAPE in the device error word.
 *   o            readout o = S^T (scale q), taken after the update. */
int gla_decode_step(const void* q, const void* k, const void* v, const float* log_lambda,
                    float scale, float* state, const int32_t* slot, int pool_rows, void* o, int N,
                    int H, int dk, int dv, int dtype, gla_stream_t stream);

/* One decode step with the self-augmentation step: as gla_decode_step, and the output also gains
 * sigmoid(q . (a_h * k)) v (see gla_chunk_fwd_aug); aug [H, 96] fp32 device, non-NULL and
 * 16-byte aligned.  The state update is the same. */
int gla_decode_step_aug(const void* q, const void* k, const void* v, const float* log_lambda,
                        float scale, const float* aug, float* state, const int32_t* slot,
                        int pool_rows, void* o, int N, int H, int dk, int dv, int dtype,
                        gla_stream_t stream);

/* Per-tier Head RMSNorm and SiLU output gate ("Beyond the KV cache", section "i14 and the
 * Laplace 3B architecture": the per-head outputs pass through a Head RMSNorm within each decay
 * tier, then are gated by SiLU(g_t)).  For every row t and head h:
 *     y[t,h,:] = o[t,h,:] / sqrt(mean_c o[t,h,c]^2 + eps) * weight[tier[h],:] * SiLU(g[t,h,:]),
 * SiLU(x) = x sigmoid(x); the RMS runs over the head's 192 channels.
 *   o, g, y      [rows, H, 192], dtype `dtype` (o is a chunked-forward or decode output, g the
 *                gate stream); y may not alias o or g.
 *   weight       [n_tiers, 192] fp32 device, the gain of each tier's norm.
 *   tier         [H] int32 device: the tier of each head; a value outside [0, n_tiers) leaves
 *                that head's rows untouched and records GLA_ERR_SHAPE in the device error word.
 *   eps          >= 0, added to the mean square (not stated on the pages).
 * H <= 4096 (else GLA_ERR_UNSUPPORTED).  Pointers 16-byte aligned (tier 4-byte).  Returns GLA_OK once the work is queued on `stream`. */
int gla_head_norm_gate(const void* o, const void* g, const float* weight, const int32_t* tier,
                       int n_tiers, float eps, void* y, long long rows, int H, int dv, int dtype,
                       gla_stream_t stream);

/* One decode step whose readout goes straight through the per-tier Head RMSNorm and the SiLU
 * output gate ("Beyond the KV cache", section "i14 and the Laplace 3B architecture": the per-head
 * outputs pass through a Head RMSNorm within each decay tier, then the SiLU(g_t) gate; heads are
 * grouped into tiers that share a norm, section "Decay schedule's reach").  The state update is
 * that of gla_decode_step (aug NULL) or gla_decode_step_aug (aug non-NULL) on an fp32 pool; the
 * readout o (fp32, before any rounding) is not stored but normalised and gated in the same
 * kernel, and
 *     y[n,h,:] = o / sqrt(mean_c o_c^2 + eps) * weight[tier[h],:] * SiLU(g[n,h,:])
 * is written, as gla_head_norm_gate would compute from o.
 *   g            [N, H, 192] gate stream, dtype `dtype`, 16-byte aligned.
 *   weight       [n_tiers, 192] fp32, 16-byte aligned; tier [H] int32 (4-byte aligned).  A tier
 *                outside [0, n_tiers) leaves that head's y untouched (the state is still updated)
 *                and records GLA_ERR_SHAPE in the device error word.
 *   eps          >= 0; n_tiers >= 1 (else GLA_ERR_SHAPE).
 *   y            [N, H, 192] output, dtype `dtype`; may not alias g.
 * Every other argument as in gla_decode_step_aug. */
int gla_decode_step_norm_gate(const void* q, const void* k, const void* v, const float* log_lambda,
                              float scale, const float* aug, float* state, const int32_t* slot,
                              int pool_rows, const void* g, const float* weight, const int32_t* tier,
                              int n_tiers, float eps, void* y, int N, int H, int dk, int dv, int dtype,
                              gla_stream_t stream);

/* One decode step on a state pool stored in bf16 (no counterpart in the paper: a storage
 * variant that halves the state stream).  As gla_decode_step (aug NULL) or gla_decode_step_aug
 * (aug non-NULL), with `state` a [pool_rows, H, 96, 192] bf16 pool: each state is widened to
 * fp32, updated and read out in fp32 (the readout uses the update before rounding), and written
 * back rounded to bf16 (to nearest, ties to even).  The rounding error is kept in the state and
 * carried by later steps (relative 2^-9 per element per step, decayed by lambda), so long decodes
 * drift from the fp32-state result; the fp32 pool is the reference path. */
int gla_decode_step_bf16_state(const void* q, const void* k, const void* v, const float* log_lambda,
                               float scale, const float* aug, void* state, const int32_t* slot,
                               int pool_rows, void* o, int N, int H, int dk, int dv, int dtype,
                               gla_stream_t stream);

/* Decode step on a state pool stored as MXFP8 (no counterpart in the paper: a storage variant
 * that quarters the state stream; the pages keep fp32 states).  Format: OCP Microscaling (MX)
 * v1.0 MXFP8, E4M3 elements (OCP 8-bit floating point: bias 7, largest finite 448) with one E8M0
 * scale byte b (value 2^(b - 127)) per block of 32 consecutive values of a state row:
 *   state_codes   [pool_rows, H, 96, 192] uint8 E4M3 codes, 16-byte aligned;
 *   state_scales  [pool_rows, H, 96, 6] uint8 E8M0 scales of the blocks (columns 32j .. 32j+31),
 *                 16-byte aligned.
 * Each state is widened exactly to fp32, updated (S <- lambda S + k v^T) and read out
 * (o = S^T (scale q), from the update before it is stored) in fp32, and written back quantised:
 * per block, shared exponent se = floor(log2(max |x|)) - 8, plus one where the block maximum
 * would otherwise exceed 448 (the MX rule alone saturates such maxima to 448; here nothing
 * saturates), clamped to [-127, 127] (-127 for an all-zero block); codes = x 2^-se rounded to
 * E4M3, to nearest, ties to even.  The quantisation error (up to 2^-4 relative per element per
 * step, decayed by lambda) stays in the state, so long decodes drift from the fp32 result much
 * more than with the bf16 pool; the fp32 pool is the reference path.  Every other argument as in
 * gla_decode_step (aug NULL) or gla_decode_step_aug (aug non-NULL). */
int gla_decode_step_mxfp8_state(const void* q, const void* k, const void* v, const float* log_lambda,
                                float scale, const float* aug, uint8_t* state_codes, uint8_t* state_scales,
                                const int32_t* slot, int pool_rows, void* o, int N, int H, int dk, int dv,
                                int dtype, gla_stream_t stream);

/* Conversions between fp32 state rows and MXFP8 (the format of gla_decode_step_mxfp8_state), for
 * building a pool from fp32 states (a prefill's hT) and reading one back.  `rows` rows of 192
 * values: x [rows, 192] fp32, codes [rows, 192] uint8, scales [rows, 6] uint8; all 16-byte
 * aligned.  Quantisation as in gla_decode_step_mxfp8_state; dequantisation is exact. */
int gla_state_to_mxfp8(const float* x, uint8_t* codes, uint8_t* scales, long long rows, gla_stream_t stream);
int gla_state_from_mxfp8(const uint8_t* codes, const uint8_t* scales, float* x, long long rows,
                         gla_stream_t stream);

/* Sequence-split forward for long sequences (no counterpart in the paper).  A sequence's work
 * otherwise sits on one CTA per (head, 64-column tile of d_v), so one long sequence among few
 * keeps most SMs idle.  Here each sequence is cut into segments of at most seg_chunks chunks
 * (128 tokens each), and the forward runs in three steps: every segment from a zero state (its
 * final state U_i), a scan per (sequence, head) that chains them (S_in of the next segment =
 * lambda^(L_i) S_in + U_i; hT after the last), and every segment again from its S_in, writing o.
 * Same results as gla_chunk_fwd (the sums are only reassociated), about twice its reads of q, k
 * and v; worth it when the longest sequences dominate the call.
 *   cu_seqlens_host  [n_seq + 1] host array of packed offsets (cu_seqlens_host[0] = 0,
 *                    non-decreasing, cu_seqlens_host[n_seq] = T): the segments are planned on the
 *                    host, so no device offsets are needed (a fixed-length batch passes 0, T,
 *                    2T, ... with T = n_seq * T_seq and the [n_seq, T_seq, H, d] layout).
 *   aug              NULL, or aug_balance [H, 96] (the self-augmentation step of gla_chunk_fwd_aug).
 *   seg_chunks       >= 1, chunks per segment; 0: chosen by gla_split_choose_seg_chunks.  When
 *                    every sequence fits one segment the call is gla_chunk_fwd (or _aug).
 *   workspace        >= gla_split_workspace_bytes(cu_seqlens_host, n_seq, H, seg_chunks) bytes,
 *                    256-byte aligned: the plan, the segment states (two fp32 [segments, H, 96,
 *                    192] arrays) and the packed schedule.
 * Every other argument as in gla_chunk_fwd.  The plan is copied to the device with pageable
 * host-to-device copies (which may wait for the stream's earlier work).
 * gla_split_workspace_bytes returns 0 for a NULL cu_seqlens_host, n_seq < 0, H < 1, seg_chunks
 * < 0 or decreasing offsets.
 * gla_split_choose_seg_chunks: the segment length that seg_chunks = 0 uses, from a cost model of
 * the packed forward (one CTA per (segment, head, d_v tile) unit on each of 152 SMs, longest
 * units first, a unit costing its chunks plus a start-up cost; the split's two passes against the
 * plain forward's one), over lengths that cut the longest sequence into 2 .. 64 equal parts.
 * Returns 0 when no split is estimated faster, GLA_ERR_NULL / GLA_ERR_SHAPE on bad arguments.
 * Host only (no device needed). */
size_t gla_split_workspace_bytes(const int32_t* cu_seqlens_host, int n_seq, int H, int seg_chunks);
int gla_split_choose_seg_chunks(const int32_t* cu_seqlens_host, int n_seq, int H);
int gla_chunk_fwd_split(const void* q, const void* k, const void* v, const float* log_lambda,
                        const float* h0, float scale, const float* aug, void* o, float* hT,
                        const int32_t* cu_seqlens_host, int n_seq, int T, int H, int dk, int dv,
                        int dtype, int seg_chunks, void* workspace, size_t ws_bytes,
                        gla_stream_t stream);

/* The forward without any device allocation (no counterpart in the paper).  For callers that
 * cannot allocate device memory per call, such as a serving engine whose memory is all handed to
 * its own pool at start-up: same arguments and results as gla_chunk_fwd, minus the workspace.
 * The longest-first schedule of packed sequences lives instead in a library-owned device array of
 * GLA_NOALLOC_MAX_SEQS int32 (64 KB), kept by every GPU that loads the library until exit.
 *   Arguments are checked as in gla_chunk_fwd (the same status codes, including GLA_ERR_SHAPE for
 *   n_seq * H * 96 or the token count at 2^31 or beyond); then n_seq > GLA_NOALLOC_MAX_SEQS with
 *   cu_seqlens returns GLA_ERR_WORKSPACE (nothing launched).
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress); make
 *   that first call before any stream capture on the device.
 *   Calls share the array: calls that overlap on the GPU (unordered streams) race on it.  Calls
 *   ordered on one stream do not; each rewrites the entries it uses before reading them. */
#define GLA_NOALLOC_MAX_SEQS 16384
int gla_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* log_lambda,
                          const float* h0, float scale, void* o, float* hT,
                          const int32_t* cu_seqlens, int n_seq, int T, int H, int dk, int dv,
                          int dtype, gla_stream_t stream);

/* The chunked forward on HOST buffers ("Beyond the KV cache", section "Challenge 1: Using native
 * PyTorch on Trainium for GLA": sequences are independent, and within one the scan carries only
 * the state across a chunk boundary): q, k, v are read from host memory and o, hT written back
 * to host memory, the copies pipelined with the compute inside the call.  The batch is cut into
 * `pieces`: sub-batches of whole sequences (pieces <= n_seq), or, with pieces > n_seq, each
 * sequence cut into pieces / n_seq parts of a whole number of 128-token chunks (fewer when T does
 * not divide so), a part starting from the final state of the one before, which is the state the
 * uncut scan carries across that boundary: the results equal gla_chunk_fwd's on the same values.
 * Piece i is copied in on a library stream while piece i - 1 runs on `stream` and piece i - 2 is
 * copied out on another library stream; `stream` completes after the last copy out, so the host
 * outputs may be read once `stream` has been synchronised.
 *   q, k, v      HOST [n_seq, T, H, 96 / 192] of dtype `dtype` (page-locked memory lets the copies
 *                overlap the compute; pageable memory works, without the overlap).
 *   h0           HOST [n_seq, H, 96, 192] fp32, or NULL for zeros.
 *   o, hT        HOST outputs (o as v; hT [n_seq, H, 96, 192] fp32, or NULL to skip).
 *   log_lambda   DEVICE [H] fp32, 16-byte aligned.
 *   pieces       >= 1.
 *   workspace    DEVICE, 256-byte aligned, >= gla_chunk_fwd_host_workspace_bytes(n_seq, T, H,
 *                dtype) bytes: the staged batch (q, k, v, o) and three sets of states.
 * Fixed-length batches only.  Returns GLA_OK once the work is queued; argument errors as in
 * gla_chunk_fwd, GLA_ERR_WORKSPACE for a missing or short workspace, GLA_ERR_LAUNCH if a copy or
 * an event could not be queued.  Calls on one device are issued one at a time (a library mutex);
 * their work may still overlap on the GPU, so calls on streams that are not ordered with each
 * other need workspaces of their own (calls on one stream may share one).
 * gla_chunk_fwd_host_workspace_bytes returns 0 for n_seq < 0, T < 0, H < 1 or an unknown dtype. */
size_t gla_chunk_fwd_host_workspace_bytes(int n_seq, int T, int H, int dtype);
int gla_chunk_fwd_host(const void* q, const void* k, const void* v, const float* log_lambda,
                       const float* h0, float scale, void* o, float* hT, int n_seq, int T, int H,
                       int dk, int dv, int dtype, int pieces, void* workspace, size_t ws_bytes,
                       gla_stream_t stream);

/* Synchronises `stream`, then returns and clears the current device's sticky error word:
 * GLA_OK, GLA_ERR_TIMEOUT or GLA_ERR_SHAPE (or, in the debug-bounds build, GLA_ERR_BOUNDS);
 * GLA_ERR_LAUNCH if the stream itself failed.
 * There is one word per device, shared by every caller of the library on that device: the first
 * fault recorded since the last read is kept, and whichever caller reads next sees and clears it. */
int gla_get_device_error(gla_stream_t stream);

/* 1 in the library's debug-bounds build (libgla_debug.so, compiled with GLA_DEBUG_BOUNDS), 0 in
 * the release build (libgla.so).  The debug-bounds build is the same library with device-side
 * index checks at the kernels' computed global accesses (state rows, output and gradient rows,
 * partial-sum rows, packed-order and segment lookups, hand-over flags, TMA coordinates): an index
 * outside its buffer records GLA_ERR_BOUNDS in the device error word and the access is skipped.
 * It stands in for a memory checker; its results equal the release build's. */
int gla_debug_bounds(void);

/* Upper bound, in nanoseconds, of every device-side wait on an mbarrier (default 2e9).  A wait
 * that exceeds it records GLA_ERR_TIMEOUT, drains the copies its CTA has in flight, releases
 * tensor memory and returns.  Meant for tests of that path; applies to the current device. */
int gla_set_wait_limit_ns(unsigned long long ns);

/* Human-readable name of a gla_status value. */
const char* gla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GLA_H_ */
