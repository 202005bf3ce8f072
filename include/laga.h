/*
 * laga.h -- C ABI of the GB300 (sm_103a) per-rank LAGA compute.
 *
 * LAGA (Latent All-Gather Attention), from "A Training-Memory Regression in
 * MLA Sequence Parallelism: Why Megatron-Core Forbids Absorption, and LAGA --
 * a Communication-Efficient Fix" (arXiv 2607.17644v1).  After the latent
 * all-gather (Algorithm 1 step 3) each rank holds the full-sequence latent
 * c = [latent (d_kv) | k_pe (d_rope)] and its head shard of q.  This library
 * runs the rest of the rank's attention on one GPU:
 *
 *   a1  L = LayerNorm(latent) * gamma           (Section 2.1, Alg. 1 step 1)
 *   a2  RoPE of k_pe (shared by all heads) and of q_rope   (Section 5.3)
 *   a3  KV = L . W_kv_b[:, shard]  -> k_nope | v per head  (Alg. 1 step 4,
 *                                                          Section 5.1 eq.)
 *   a4  causal attention, scores = (q_nope||q_rope)(k_nope||k_pe)^T/sqrt(d),
 *       out = softmax(scores) v                        (Alg. 1 step 5)
 *   a5-a7 the backward of all of the above: dq, dc, dW_kv_b shard, dgamma
 *       (Section 5.2)
 *
 * Conventions (the page leaves these open; each is the plainest reading):
 *   - d = d_nope + d_rope; causal means key j is visible to query i iff j<=i.
 *   - LayerNorm: biased variance, gain gamma, no bias, eps = ln_eps (or its
 *     RMS variant, dims->norm = LAGA_NORM_RMS).
 *   - RoPE rotates pairs (i, i + d_rope/2) by the angle whose cos/sin the
 *     caller passes in cos/sin [S, d_rope/2] (fp32, positions 0..S-1 of the
 *     gathered sequence).  q is passed raw; the library rotates q_rope and
 *     k_pe itself; dq and dc are gradients with respect to the raw inputs.
 *   - W_kv_b is [d_kv, n_h_total * (d_nope + d_v)] row-major; the columns of
 *     head i are [k_nope (d_nope) | v (d_v)]; this call's shard is heads
 *     [head_offset, head_offset + n_h_shard).
 *
 * Ownership and execution.  The caller allocates every buffer (device
 * memory unless stated otherwise).  The library never allocates device
 * memory, never frees and never synchronises (except laga_sync_check); every
 * call only validates its arguments on the host and enqueues kernels on
 * `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 * The library owns no stream and no event: the one entry point that uses a
 * second stream, laga_bwd_overlap, takes it and its two events from the
 * caller.  Outputs are overwritten, not accumulated.  Summing the partial dc and dgamma of several head shards
 * is the caller's job (the reduce-scatter / all-reduce of Section 5.2).
 *
 * Errors.  All argument, size and alignment checks happen before the first
 * launch; on any error nothing is enqueued.  Device pointers must be 16-byte
 * aligned.  A launch failure returns LAGA_ERR_CUDA.  Device-side waits are
 * bounded; one that gives up records LAGA_ERR_TIMEOUT in a device flag that
 * laga_sync_check() (or the next laga_fwd/laga_bwd on the same device)
 * reports.  No C++ exception crosses this ABI.
 */
#ifndef LAGA_H
#define LAGA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LAGA_OK = 0,
  LAGA_ERR_ARG = 1,          /* bad size, NULL pointer, unknown enum value   */
  LAGA_ERR_ALIGN = 2,        /* a pointer is not 16-byte aligned             */
  LAGA_ERR_WORKSPACE = 3,    /* workspace smaller than laga_workspace_bytes  */
  LAGA_ERR_UNSUPPORTED = 4,  /* valid but not built: e.g. causal = 0        */
  LAGA_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed            */
  LAGA_ERR_TIMEOUT = 6       /* a bounded device wait gave up                */
} laga_status;

/* Which form of Section 3 to run on one rank.
 *  LAGA      latent gathered, K/V rebuilt per head shard, K/V layout
 *            [B, S, H, d_nope + d_v] (token-major).
 *  EXPLICIT  same arithmetic, K/V in the head-major layout [B, H, S, ...]
 *            that the explicit form's all-to-all produces (Section 3.2, B1);
 *            at SP = 1 results are bit-identical to LAGA (Proposition 1).
 *  ABSORBED  q_absorbed = W^k^T q_nope, attention over the latent, latent
 *            accumulator, V up-projection afterwards (Section 3.2, B2); the
 *            memory-trap contrast path, not a performance path.
 *  LAGA_FUSED  the LAGA form with the up-projection fused into the
 *            key-stationary backward (the fused up-projection kernel the
 *            paper leaves to future work, Section 4.7 and Section 8): the
 *            dK/dV kernel rebuilds each key tile's k_nope and v from L and
 *            W_kv_b on the tensor cores, so the forward's K/V is scratch
 *            (LAGA_WS_FWD) instead of a saved activation, and LAGA_WS_SAVED
 *            shrinks by B * S * n_h_shard * (d_nope + d_v) * 2 bytes (with
 *            d_nope + d_v padded to 256).  Same arithmetic as LAGA: results
 *            are identical to it. */
typedef enum {
  LAGA_FORM_LAGA = 0,
  LAGA_FORM_EXPLICIT = 1,
  LAGA_FORM_ABSORBED = 2,
  LAGA_FORM_LAGA_FUSED = 3
} laga_form;

/* Normalisation of the latent (step a1).  The paper's "LN" is LayerNorm:
 * mean-subtracted, biased variance, gain gamma, no bias.  LAGA_NORM_RMS is
 * its RMS variant, an extension of the method: no mean subtraction,
 * L = x * gamma / sqrt(mean(x^2) + eps). */
typedef enum { LAGA_NORM_LAYER = 0, LAGA_NORM_RMS = 1 } laga_norm;

/* Element type of q, c, W_kv_b, O, dO and dq.  Compute is bf16 operands with
 * fp32 accumulation in both cases; fp32 I/O is rounded to bf16 on-device. */
typedef enum { LAGA_BF16 = 0, LAGA_FP32 = 1 } laga_dtype;

typedef struct {
  int B;            /* batch, >= 1                                            */
  int S;            /* full (gathered) sequence length, >= 1                  */
  int n_h_total;    /* heads whose columns W_kv_b holds                        */
  int head_offset;  /* first head of this shard                                */
  int n_h_shard;    /* heads in this shard (n_h / SP); offset+shard <= total   */
  int d_nope;       /* multiples of 16; d_nope, d_v <= 128, d_rope <= 64 even, */
  int d_rope;       /* d_kv <= 512.  DeepSeek-V3: 128 / 64 / 128 / 512.        */
  int d_v;
  int d_kv;
  float scale;      /* softmax scale; 0 selects 1/sqrt(d_nope + d_rope)        */
  float ln_eps;     /* LayerNorm epsilon (1e-5 in the workloads)               */
  int causal;       /* must be 1                                               */
  laga_dtype io_dtype;
  laga_form form;
  laga_norm norm;   /* latent norm of step a1 (LAGA_NORM_LAYER = 0)          */
} laga_dims;

/* Workspace passes. */
#define LAGA_WS_SAVED 0   /* written by laga_fwd, read by laga_bwd: keep it    */
#define LAGA_WS_BWD 1     /* transient scratch of laga_bwd                     */
#define LAGA_WS_FWD 2     /* transient scratch of laga_fwd_scratch: read and   */
                          /* written only by that call's kernels (0 bytes     */
                          /* except for LAGA_FORM_LAGA_FUSED)                 */

/* Bytes of workspace `pass` needs for these dims (0 if the dims are
 * invalid).  Host-only, no CUDA call. */
size_t laga_workspace_bytes(const laga_dims* dims, int pass);

/* Enumerate the named tensors inside workspace `pass` (activation
 * accounting).  index runs from 0; returns LAGA_ERR_ARG past the last one.
 * *name is a static string, *offset/*bytes are byte offsets inside the
 * workspace.  Host-only. */
laga_status laga_workspace_tensor(const laga_dims* dims, int pass, int index,
                                  const char** name, size_t* offset, size_t* bytes);

/* Forward, steps a1-a4.
 *   q      [B, S, n_h_shard, d_nope + d_rope]  io dtype, raw (un-rotated)
 *   c      [B, S, d_kv + d_rope]                io dtype, [latent | k_pe]
 *   w_kvb  [d_kv, n_h_total * (d_nope + d_v)]   io dtype, full matrix
 *   gamma  [d_kv] fp32;  cos, sin [S, d_rope/2] fp32
 *   o      [B, S, n_h_shard, d_v]               io dtype (output)
 *   lse    [B, n_h_shard, S] fp32 natural-log row log-sum-exp (output)
 *   ws_saved / saved_bytes: LAGA_WS_SAVED workspace; must stay unchanged
 *          until the matching laga_bwd. */
laga_status laga_fwd(const laga_dims* dims, const void* q, const void* c, const void* w_kvb,
                     const float* gamma, const float* cos, const float* sin,
                     void* o, float* lse, void* ws_saved, size_t saved_bytes, void* stream);

/* laga_fwd with a forward scratch: ws_fwd / fwd_bytes is a LAGA_WS_FWD
 * workspace, free for other use once the call's kernels on `stream` are
 * done.  ws_fwd may be NULL when laga_workspace_bytes(dims, LAGA_WS_FWD) is
 * 0; LAGA_FORM_LAGA_FUSED needs it (laga_fwd returns LAGA_ERR_WORKSPACE for
 * that form).  Otherwise as laga_fwd. */
laga_status laga_fwd_scratch(const laga_dims* dims, const void* q, const void* c,
                             const void* w_kvb, const float* gamma, const float* cos,
                             const float* sin, void* o, float* lse, void* ws_saved,
                             size_t saved_bytes, void* ws_fwd, size_t fwd_bytes, void* stream);

/* Backward, steps a5-a7, for the loss sum(O * dO).
 *   q, c, w_kvb, gamma, cos, sin, o, lse: exactly as given to / returned by
 *          the matching laga_fwd;  d_o [B, S, n_h_shard, d_v] io dtype
 *   dq     [B, S, n_h_shard, d_nope + d_rope]   io dtype (output)
 *   dc     [B, S, d_kv + d_rope] fp32: this shard's partial (output)
 *   dw     [d_kv, n_h_shard * (d_nope + d_v)] fp32: gradient of this
 *          shard's columns of W_kv_b (output)
 *   dgamma [d_kv] fp32: this shard's partial (output)
 *   ws_saved: the forward's saved workspace (read only)
 *   ws_bwd / bwd_bytes: LAGA_WS_BWD scratch.
 * Every kernel is enqueued on `stream`, in order. */
laga_status laga_bwd(const laga_dims* dims, const void* q, const void* c, const void* w_kvb,
                     const float* gamma, const float* cos, const float* sin,
                     const void* o, const float* lse, const void* d_o,
                     void* dq, float* dc, float* dw, float* dgamma,
                     const void* ws_saved, size_t saved_bytes,
                     void* ws_bwd, size_t bwd_bytes, void* stream);

/* laga_bwd with the two independent kernels of the attention backward on
 * two streams, an opt-in for callers that own a second stream.  Arguments
 * as for laga_bwd, plus:
 *   aux_stream  a cudaStream_t of the caller's, different from `stream`
 *   fork_event, join_event  two cudaEvent_t of the caller's (created on the
 *               device of `stream`; timing may be disabled)
 * The call records fork_event on `stream` and makes aux_stream wait for it;
 * the query-stationary dQ kernel then runs on aux_stream beside the key-
 * stationary dK/dV kernel and the up-projection and norm backward on
 * `stream`; join_event, recorded on aux_stream after the dQ kernel, is
 * waited on by `stream` before the call returns.  So all of the call's work
 * is ordered before anything enqueued on `stream` afterwards, and work the
 * caller enqueues on aux_stream afterwards follows the dQ kernel.  The
 * events and aux_stream must not be used by another call until this one's
 * work is enqueued (the library keeps no lock).  While per-kernel profiling
 * is on, every kernel runs on `stream`.  For the absorbed and fused forms
 * this is laga_bwd (the fused form's dQ kernel reads the K/V that its dK/dV
 * kernel rebuilds).  LAGA_ERR_ARG if an event is NULL or
 * aux_stream == stream. */
laga_status laga_bwd_overlap(const laga_dims* dims, const void* q, const void* c,
                             const void* w_kvb, const float* gamma, const float* cos,
                             const float* sin, const void* o, const float* lse, const void* d_o,
                             void* dq, float* dc, float* dw, float* dgamma, const void* ws_saved,
                             size_t saved_bytes, void* ws_bwd, size_t bwd_bytes, void* stream,
                             void* aux_stream, void* fork_event, void* join_event);

/* Synchronise `stream` and report a launch error or a device wait that gave
 * up since the last check on this device (and clear the flag). */
laga_status laga_sync_check(void* stream);

/* Diagnostic of the error path above; the paper has no counterpart.
 * Enqueues one single-thread kernel whose bounded wait (about 17 ms) on an
 * mbarrier that nothing arrives on gives up, so the next laga_sync_check()
 * on this device reports LAGA_ERR_TIMEOUT.  No fault, no unbounded spin.
 * Returns LAGA_ERR_CUDA if the launch fails. */
laga_status laga_selftest_wait_timeout(void* stream);

/* Diagnostic of the tensor-core issue rate; the paper has no counterpart.
 * Launches n_cta CTAs (one per SM when n_cta <= the SM count); in each, one
 * thread issues n_instr tcgen05.mma of M = 128, K = 16, N = n (bf16
 * operands, fp32 TMEM accumulator) back to back and times them with the SM
 * clock, from the first issue to the completion of the last.
 *   form   bits 0-1  0: A and B in shared memory; 1: A in TMEM, B in shared
 *                    memory; 2: the two alternating
 *          bit 2     B MN-major (64-wide N boxes) instead of K-major
 *          bits 3-5  while the MMAs run, the CTA's other seven warps (one on
 *                    the issuing thread's SM sub-partition)
 *                    0: idle; 1: stream TMEM loads from other columns;
 *                    2: stream 16-byte shared-memory stores;
 *                    3: stream 16 KB bulk copies (TMA) into shared memory;
 *                    4: stream TMEM stores to other columns;
 *                    5: exponentials and FMAs in registers;
 *                    6: broadcast shared-memory loads (all lanes one address)
 *          bit 6     operands spread like N(0,1) draws instead of small
 *                    repeating values
 *   n_acc, run  instruction k accumulates into accumulator (k / run) % n_acc
 *          (n_acc = 1: one dependent chain; n_acc > 1: independent
 *          accumulators interleaved in runs of `run` instructions)
 *   cycles [n_cta] device array (output): SM clocks per CTA; 0 if the
 *          bounded wait for completion gave up
 * LAGA_ERR_ARG for n not a multiple of 16 in [16, 256] (of 64 with an
 * MN-major B), n_acc * n beyond the free TMEM columns (512; 496 with A in
 * TMEM; 448 with background TMEM loads or stores), n_instr outside [1, 2^20] or not a
 * multiple of 48, 48 not a multiple of n_acc * run, or n_cta outside
 * [1, 4096].  Asynchronous on `stream`. */
laga_status laga_diag_mma_rate(int form, int n, int n_acc, int run, int n_instr, int n_cta,
                               unsigned long long* cycles, void* stream);

/* Static text for a status code. */
const char* laga_status_string(laga_status status);

/* Number of kernel launches the last laga_fwd / laga_bwd call on this host
 * thread enqueued (0 after an error).  For launch accounting. */
int laga_last_launch_count(void);

/* LayerNorm + RoPE backward (the backward of steps a1-a2 alone) for callers
 * that cannot allocate device memory, e.g. a runtime that has reserved the
 * whole device for its own pool and forbids cudaMalloc during a step, or an
 * embedding that owns only the tensors it passes in.  The paper has no
 * counterpart of this entry point; it exists for such callers.
 *
 * Instead of a caller workspace it uses a fixed scratch array inside the
 * library (296 x 512 fp32 = 592 KiB per device, held from the first call on
 * that device until the process exits) and calls no cudaMalloc, cudaFree or
 * allocating library routine.  The first call on a device looks up the
 * scratch's device address (once, with that device current); make that
 * first call before any stream capture.  All calls share the scratch: calls
 * whose kernels may overlap on the GPU race on it and must be ordered by the
 * caller.  Each call rewrites all the scratch it reads, so no state carries
 * over between calls.
 *   c           [B, S, d_kv + d_rope]       io dtype, as given to laga_fwd
 *   gamma       [d_kv] fp32; cos, sin [S, d_rope/2] fp32
 *   d_latent    [B, S, d_kv] fp32: gradient with respect to the normalised
 *               latent L = LayerNorm(latent) * gamma
 *   d_kpe_rot   [B, S, n_h_shard, d_rope] fp32: each head's gradient with
 *               respect to the RoPE'd k_pe (summed over heads in head order)
 *   dc          [B, S, d_kv + d_rope] fp32 (output), dgamma [d_kv] fp32 (output)
 * The statistics of the latent norm (dims->norm) are recomputed from c.  d_kv above 512 does not
 * fit the scratch and returns LAGA_ERR_WORKSPACE; other errors as for
 * laga_bwd. */
laga_status laga_norm_rope_bwd_noalloc(const laga_dims* dims, const void* c, const float* gamma,
                                       const float* cos, const float* sin,
                                       const float* d_latent, const float* d_kpe_rot,
                                       float* dc, float* dgamma, void* stream);

/* Per-kernel timing for measurement.  While enabled, every kernel the
 * library launches is bracketed by two CUDA events recorded on its own
 * stream; laga_profile_read() waits for those events and returns, per kernel
 * name, the summed elapsed milliseconds and the launch count since the last
 * laga_profile_reset().  Names are static strings.  Returns the number of
 * distinct kernels (at most max are written).  Off by default. */
void laga_profile_enable(int on);
void laga_profile_reset(void);
int laga_profile_read(const char** names, double* total_ms, int* launches, int max);

#ifdef __cplusplus
}
#endif

#endif /* LAGA_H */
