/*
 * replayssm.h -- C ABI of libreplayssm, the GB300 (sm_103a) ReplaySSM decode path.
 *
 * The operations follow "ReplaySSM: Cache SSM Inputs, Not State" (Tri Dao's
 * blog post, as summarised on papercache).  Instead of reading and writing the
 * fp32 SSM state S (nheads, d, n) every token, each sequence keeps a
 * checkpoint S_0 plus a ring buffer of its last L inputs; outputs come from
 * S_0 and the buffer, and a flush folds the buffer into S_0 when it fills.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every call returns an rssm_status (RSSM_OK = 0, negative on error).  On a
 *    non-zero status nothing was launched.
 *  - Calls are asynchronous on the caller's stream and never synchronise.
 *    Pass a cudaStream_t (NULL = the legacy default stream).  The calling
 *    thread's current CUDA device must own every pointer.  Consecutive calls
 *    on one stream may overlap on the GPU (programmatic dependent launch),
 *    but a call reads nothing the previous call writes before the previous
 *    call's kernels have completed, so one call's output may be passed as the
 *    next call's input.
 *  - The caller owns all memory.  Every pointer is a DEVICE pointer,
 *    contiguous, row-major in the documented layout.  S, S0, snapshot slots,
 *    k, q and ring_k must be 16-byte aligned; every other array must be
 *    aligned to its element size.  The library allocates nothing and keeps
 *    no state between calls.
 *  - dtypes: RSSM_F32 (float) or RSSM_BF16 (bfloat16).  The checkpoint and
 *    state are always float32; the step size Delta, the gate g and beta are
 *    float32.  Ring entries of v/k use the input dtype.
 *  - One call handles one layer.  A stack of layers is a loop of calls.
 *  - Inconsistent per-sequence bookkeeping found ON THE DEVICE (a committed
 *    count out of range, a draft window that does not fit, an accepted count
 *    out of range) sets a bit in the caller's sticky int32 error word *err
 *    (RSSM_EBIT_*) and that sequence is skipped; kernels never trap and never
 *    spin.  Read *err after synchronising; clear it yourself.
 *  - Every wait inside a kernel is bounded (about one second) and sets
 *    RSSM_EBIT_TIMEOUT when it runs out.  In the precompute kernel of a
 *    two-launch call (a workspace is given) the affected sequence is skipped
 *    as a whole: its pointers, checkpoint and committed ring entries stay as
 *    they were (the outputs of its heads are undefined: each is either left
 *    untouched or what the ordinary call writes).
 *    A wait that runs out in any other kernel leaves the affected sequences'
 *    outputs and state undefined: restore them from a checkpoint.  The
 *    environment variable RSSM_WAIT_LIMIT_NS (nanoseconds, read at every
 *    call) replaces the precompute kernels' limit; 0 makes those waits count
 *    as run out at once, which exercises the recovery path in tests.
 *  - Supported shapes (checked on the host, RSSM_ERR_UNSUPPORTED otherwise):
 *    n (Mamba-2 state size) and dk (GDN key size) in {16, 32, 64, 128};
 *    d and dv multiples of 4 with 4 <= d <= 256;
 *    1 <= L <= 32; 1 <= T <= 8 and T <= L; H % G == 0; Hv % Hk == 0; B >= 1.
 *
 * Ring buffer and checkpoint layout (HBM)
 * ---------------------------------------
 *  Mamba-2 (rssm_m2_replay), per layer:
 *    S0       float [B][H][d][n]
 *    ring_v   in_dtype [B][H][L][d]
 *    ring_k   in_dtype [B][G][L][n]      (k is shared by the H/G heads of a group)
 *    ring_dt  float [B][H][L]
 *    start, count, flag, sync   int32 [B]
 *  Entry j (1-based) of sequence b's window sits in ring slot
 *  (start[b] + j - 1) mod L; count[b] entries are committed.  Head i uses
 *  group i / (H/G).  `sync` is a per-sequence arrival counter the kernels use
 *  to hand the pointer update to the last of a sequence's thread blocks; it
 *  must be zero before the first call and every call leaves it zero.
 *
 *  GDN (rssm_gdn_replay), per layer:
 *    S0       float [B][Hv][dv][dk]
 *    ring_u   u_dtype [B][Hv][L][dv]   (cached corrections u)
 *    ring_k   in_dtype [B][Hk][L][dk]
 *    ring_g   float [B][Hv][L]         (log decays g)
 *    start, count, flag, sync   int32 [B]
 */
#ifndef REPLAYSSM_H_
#define REPLAYSSM_H_

#include <stdint.h>

#if defined(__GNUC__)
#define RSSM_API __attribute__((visibility("default")))
#else
#define RSSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *rssm_stream_t; /* identical to cudaStream_t */
typedef int32_t rssm_status;

#define RSSM_OK 0
#define RSSM_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad dims, T > L ... */
#define RSSM_ERR_UNSUPPORTED (-2) /* valid but not a supported shape/dtype      */
#define RSSM_ERR_CUDA (-3)        /* the launch itself failed                     */

#define RSSM_F32 0
#define RSSM_BF16 1

/* sticky device error bits (OR-ed into *err) */
#define RSSM_EBIT_COUNT_RANGE 1 /* start/count outside [0, L-1] at a decode step   */
#define RSSM_EBIT_WINDOW 2      /* count + T > L at a verify round                  */
#define RSSM_EBIT_ACCEPTED 4    /* accepted outside [0, T] or count + accepted > L  */
#define RSSM_EBIT_CUR 8         /* snapshot slot index outside [0, T]              */
#define RSSM_EBIT_TIMEOUT 16    /* a bounded wait inside a pipelined kernel ran out */
#define RSSM_EBIT_BOUNDS 32     /* an index check of the bounds-checked build
                                   (compiled with -DRSSM_CHECKED) failed     */

/* kinds of replay_seq_bytes / gdn_replay_seq_bytes */
#define RSSM_SEQ_REPLAY 0   /* checkpoint S_0, ring buffer, pointers, workspace share */
#define RSSM_SEQ_SNAPSHOT 1 /* the baseline: T + 1 full state slots and a slot index  */

typedef struct {
  int32_t B, H, G, d, n, L;
  int32_t in_dtype; /* dtype of v, k, q and of ring_v, ring_k */
  int32_t y_dtype;  /* dtype of y */
} rssm_m2_dims;

typedef struct {
  float *S0;
  void *ring_v;
  void *ring_k;
  float *ring_dt;
  int32_t *start, *count, *flag, *sync;
  int32_t *err; /* one int32 */
  float *work;        /* optional workspace, 16-byte aligned, or NULL (see
                         replay_decode_step) */
  int64_t work_bytes; /* its size; a call uses it only if it holds at least
                         replay_decode_workspace_bytes() */
} rssm_m2_replay;

typedef struct {
  int32_t B, Hv, Hk, dk, dv, L;
  int32_t in_dtype; /* dtype of q, k, v and of ring_k */
  int32_t u_dtype;  /* dtype of ring_u (RSSM_F32 recommended) */
  int32_t y_dtype;
} rssm_gdn_dims;

typedef struct {
  float *S0;
  void *ring_u;
  void *ring_k;
  float *ring_g;
  int32_t *start, *count, *flag, *sync;
  int32_t *err;
  float *work;        /* optional workspace, 16-byte aligned, or NULL (see
                         gdn_replay_decode) */
  int64_t work_bytes; /* its size; a call with T drafts (T = 1: decode) uses it
                         only if it holds gdn_replay_workspace_bytes(dims, T) */
} rssm_gdn_replay;

/* ------------------------------------------------------------------------ */
/* Mamba-2                                                                   */
/* ------------------------------------------------------------------------ */

/* Baseline decode step ("Background -- memory bound" recurrence; "Algorithm --
 * Mamba-2 standard decode", baseline): per head a = exp(A_i Delta),
 * S <- a S + Delta v k^T, y = S q, reading and writing the whole state.
 *   S   float [B][H][d][n]  (in/out)     v  in_dtype [B][H][d]
 *   k,q in_dtype [B][G][n]               dt float [B][H]      A float [H]
 *   y   y_dtype [B][H][d] (out)                                               */
RSSM_API rssm_status ssm_state_update_baseline(const rssm_m2_dims *dims, float *S, const void *v, const void *k,
                                      const void *q, const float *dt, const float *A, void *y,
                                      rssm_stream_t stream);

/* ReplaySSM output-only decode step ("Relaxed requirement: output-only decode";
 * "Algorithm -- Mamba-2 standard decode"): with h = count[b], append
 * (v, Delta, k) at slot (start + h) mod L and write
 *   y = abar (S_0 q) + sum_{j=1}^{h+1} s_j (k_j^T q) v_j,
 *   abar = prod_{i<=h+1} a_i,  s_j = Delta_j prod_{j<i<=h+1} a_i,  a_i = exp(A Delta_i);
 * then count <- h+1 and flag <- (count == L).  S_0 is only read.  Inputs as for
 * the baseline.  A sequence whose start/count is out of range is skipped and
 * sets RSSM_EBIT_COUNT_RANGE.
 * With st->work non-NULL the step runs as two launches ("Kernel design
 * details": a small precompute kernel for the ring-dependent terms, then a
 * main kernel streaming S_0); the workspace holds per (sequence, head) the
 * precomputed terms between them and carries nothing from one call to the
 * next.  With st->work NULL one launch does both (same results).             */
RSSM_API rssm_status replay_decode_step(const rssm_m2_dims *dims, const rssm_m2_replay *st, const void *v,
                               const void *k, const void *q, const float *dt, const float *A, void *y,
                               rssm_stream_t stream);

/* Bytes of the optional decode workspace (rssm_m2_replay.work) for dims:
 * B * H * 4 * ceil((d + L + 4) / 4) floats.  Returns 0 for invalid dims.
 * Host only; launches nothing.                                                */
RSSM_API int64_t replay_decode_workspace_bytes(const rssm_m2_dims *dims);

/* Bytes of the optional workspace for replay_spec_verify with up to T drafts:
 * B * H * 4 * ceil((16 + P d) / 4) with P = 1 for T = 1, 4 for T <= 4, 8 for
 * T <= 8.  0 for invalid arguments.  Host only.                               */
RSSM_API int64_t replay_verify_workspace_bytes(const rssm_m2_dims *dims, int32_t T);

/* Device bytes that one sequence holds per Mamba-2 layer, for the accounting
 * of "Results -- speculative decoding" (maximum decode concurrency at a fixed
 * HBM budget, Fig. 11): the budget divided by layers x this figure is the
 * largest batch that fits.
 *   kind RSSM_SEQ_REPLAY: S_0 (4 H d n), the v/k/Delta rings
 *     (L (H d + G n) elements + 4 H L), the four int32 words start, count,
 *     flag, sync, and this sequence's share of the workspace: the larger of
 *     the decode and the verify workspace for window T >= 1, the decode
 *     workspace for T = 0.
 *   kind RSSM_SEQ_SNAPSHOT: the baseline, (T + 1) state slots of 4 H d n
 *     bytes and the int32 slot index for T >= 1; one state for T = 0.
 * Buffers shared by the whole batch (the error word) are not counted.
 * 0 for invalid arguments (dims as replay_decode_step, 0 <= T <= 8, kind one
 * of the two).  Host only; launches nothing.                                 */
RSSM_API int64_t replay_seq_bytes(const rssm_m2_dims *dims, int32_t T, int32_t kind);

/* Flush ("Algorithm -- Mamba-2 standard decode", flush): for every sequence
 * with flag[b] != 0 and c = count[b] committed entries,
 *   S_0 <- abar S_0 + sum_{j=1}^{c} s_j v_j k_j^T
 * then start <- (start + c) mod L, count <- 0, flag <- 0.  Other sequences are
 * untouched.  The flag array is plain data: setting it from the host flushes
 * any sequence at any time without changing later outputs.                   */
RSSM_API rssm_status replay_flush(const rssm_m2_dims *dims, const rssm_m2_replay *st, const float *A,
                         rssm_stream_t stream);

/* Decode step with the flush fused in ("Algorithm -- Mamba-2 standard decode":
 * append, output, and if the buffer is full, flush): the same outputs as
 * replay_decode_step followed by replay_flush, in one launch.  A sequence
 * whose buffer fills with this token (count reaches L) has all L entries
 * folded into S_0 from the tile this launch already holds, using this step's
 * decay weights; it ends with count = 0 and flag = 0 (start is unchanged,
 * since start + L = start mod L).  Other sequences end as after
 * replay_decode_step.  Like replay_decode_step, the call overwrites every
 * valid sequence's flag, so an early flush requested through the flag array
 * must be carried out with replay_flush before this call.
 * Arguments as replay_decode_step.                                            */
RSSM_API rssm_status replay_decode_step_fused(const rssm_m2_dims *dims, const rssm_m2_replay *st, const void *v,
                                              const void *k, const void *q, const float *dt, const float *A,
                                              void *y, rssm_stream_t stream);

/* replay_decode_step_fused with a workspace owned by the library, so that
 * the call allocates nothing and needs no caller buffer beyond the state.
 * The pages have no counterpart: this is an interface variant of
 * replay_decode_step_fused, with the same outputs and state updates.
 * st->work is ignored; the two-launch kernels use a file-scope device array
 * of 8 MiB (2,097,152 floats) inside the library, whose address in the
 * current context is looked up on every call (no allocation).  Requires
 * B * H * 4 * ceil((d + L + 4) / 4) <= 2,097,152 (RSSM_ERR_UNSUPPORTED
 * otherwise, before anything is launched).  All calls on one device share
 * that array, so they must be ordered (one stream, or synchronised streams):
 * calls that overlap on the GPU race on it.
 * Arguments as replay_decode_step.                                            */
RSSM_API rssm_status replay_decode_step_fused_noalloc(const rssm_m2_dims *dims, const rssm_m2_replay *st,
                                                      const void *v, const void *k, const void *q,
                                                      const float *dt, const float *A, void *y,
                                                      rssm_stream_t stream);

/* Speculative verify of T drafts ("Algorithm -- speculative decoding"): with
 * h = count[b] (requires h + T <= L, else RSSM_EBIT_WINDOW and the sequence is
 * skipped), write the T drafts tentatively at slots (start + h + s - 1) mod L
 * and, for s = 1..T with p_s = h + s,
 *   Y_s = abar_s (S_0 q_s) + sum_{j<=p_s} w_{j,s} (k_j^T q_s) v_j.
 * count is unchanged; flag <- (h + 2T > L) (early flush one window ahead).
 * With st->work holding replay_verify_workspace_bytes(dims, T) bytes (and L a
 * multiple of 4) the round runs as a precompute launch per (sequence, group)
 * and a launch streaming S_0 once per (sequence, head) for all T drafts;
 * otherwise as one launch per (sequence, head).  Same results.
 *   v  in_dtype [B][T][H][d]   k, q in_dtype [B][T][G][n]   dt float [B][T][H]
 *   y  y_dtype [B][T][H][d]                                                   */
RSSM_API rssm_status replay_spec_verify(const rssm_m2_dims *dims, const rssm_m2_replay *st, int32_t T,
                               const void *v, const void *k, const void *q, const float *dt,
                               const float *A, void *y, rssm_stream_t stream);

/* Speculative verify preceded by the pending flush ("Algorithm -- speculative
 * decoding", flush decision: the early flush that the previous round flagged):
 * replay_flush then replay_spec_verify, issued as those two calls on the
 * stream, so that a speculative round is this call and replay_spec_commit and
 * the flush that round r flags is carried out by round r + 1.  (A fold inside
 * the verify's S_0 stream doubled that kernel's instructions and measured
 * slower than the persistent flush pipeline followed by the verify, so no
 * fused launch is kept.)  Requires st->sync (zero, left zero), as
 * replay_flush.  Workspace and arguments as replay_spec_verify.              */
RSSM_API rssm_status replay_spec_verify_fused(const rssm_m2_dims *dims, const rssm_m2_replay *st, int32_t T,
                                              const void *v, const void *k, const void *q, const float *dt,
                                              const float *A, void *y, rssm_stream_t stream);

/* Device-side commit ("Supplementary design for CUDA Graphs", device commit):
 * count[b] += accepted[b] for b < B; rejected drafts are rolled back by not
 * moving the pointer over them.  accepted outside [0, T] or count + accepted > L
 * sets RSSM_EBIT_ACCEPTED and leaves that sequence unchanged.  Shared by the
 * Mamba-2 and GDN paths.  accepted, count: int32 [B].                       */
RSSM_API rssm_status replay_spec_commit(int32_t B, int32_t T, int32_t L, const int32_t *accepted, int32_t *count,
                               int32_t *err, rssm_stream_t stream);

/* Baseline speculative verify ("Algorithm -- speculative decoding", baseline):
 * each sequence owns T+1 state slots; starting from slot cur[b], apply the T
 * drafts serially (baseline recurrence), writing draft s's state to slot
 * (cur + s) mod (T+1) and its output to y.
 *   slots float [B][T+1][H][d][n]   cur int32 [B]   inputs/outputs as replay_spec_verify. */
RSSM_API rssm_status ssm_spec_verify_baseline(const rssm_m2_dims *dims, int32_t T, float *slots, const int32_t *cur,
                                     const void *v, const void *k, const void *q, const float *dt,
                                     const float *A, void *y, int32_t *err, rssm_stream_t stream);

/* Baseline commit: cur[b] <- (cur[b] + accepted[b]) mod (T+1). */
RSSM_API rssm_status ssm_spec_commit_baseline(int32_t B, int32_t T, const int32_t *accepted, int32_t *cur,
                                     int32_t *err, rssm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Gated DeltaNet                                                            */
/* ------------------------------------------------------------------------ */

/* Baseline GDN decode (appendix "GDN -- standard decode", baseline): per value
 * head alpha = exp(g), u = beta (v - alpha S k), S <- alpha S + u k^T, y = S q.
 *   S float [B][Hv][dv][dk] (in/out)   q, k in_dtype [B][Hk][dk]
 *   v in_dtype [B][Hv][dv]             beta, g float [B][Hv]    y y_dtype [B][Hv][dv] */
RSSM_API rssm_status gdn_state_update_baseline(const rssm_gdn_dims *dims, float *S, const void *q, const void *k,
                                      const void *v, const float *beta, const float *g, void *y,
                                      rssm_stream_t stream);

/* GDN replay decode (appendix "GDN -- standard decode", cache u): with
 * h = count[b], S_h = (prod alpha_j) S_0 + sum_j (prod_{i>j} alpha_i) u_j k_j^T
 * (never materialised: S_h k and S_h q are formed from S_0 k, S_0 q and the
 * buffer), u = beta (v - alpha S_h k), y = alpha S_h q + u (k . q); append
 * (u, k, g); count <- h+1; flag <- (count == L).
 * With a large enough st->work (bf16 inputs, d_k 64 or 128, L a multiple of
 * 4) the step runs as a precompute launch per (sequence, key head) and a
 * launch streaming S_0 per (sequence, value head, row block) ("Kernel design
 * details"); otherwise as one launch per (sequence, value head).  The
 * workspace carries nothing from one call to the next.                       */
RSSM_API rssm_status gdn_replay_decode(const rssm_gdn_dims *dims, const rssm_gdn_replay *st, const void *q,
                              const void *k, const void *v, const float *beta, const float *g, void *y,
                              rssm_stream_t stream);

/* GDN decode step with the flush fused in: the same outputs as
 * gdn_replay_decode followed by gdn_replay_flush.  A sequence whose buffer
 * fills with this token has all L entries (this token's u included) folded
 * into S_0 by the same launches; it ends with count = 0, flag = 0.  Falls
 * back to the two calls when the workspace path does not apply.
 * Arguments as gdn_replay_decode.                                             */
RSSM_API rssm_status gdn_replay_decode_fused(const rssm_gdn_dims *dims, const rssm_gdn_replay *st, const void *q,
                                             const void *k, const void *v, const float *beta, const float *g,
                                             void *y, rssm_stream_t stream);

/* Bytes of the optional GDN workspace (rssm_gdn_replay.work) for calls with
 * up to T drafts (T = 1 for decode): B * Hv * 4 * ceil((180 + 2 P dv) / 4)
 * with P = 1 for T = 1, 4 for T <= 4, 8 for T <= 8.  0 for invalid
 * arguments.  Host only.                                                      */
RSSM_API int64_t gdn_replay_workspace_bytes(const rssm_gdn_dims *dims, int32_t T);

/* The same accounting for a GDN layer: RSSM_SEQ_REPLAY counts S_0
 * (4 Hv dv dk), the u/k/g rings (L (Hv dv of u_dtype + Hk dk of in_dtype)
 * + 4 Hv L), the four int32 pointer words and this sequence's share of
 * gdn_replay_workspace_bytes for max(T, 1); RSSM_SEQ_SNAPSHOT counts T + 1
 * state slots and the slot index (one state for T = 0).  0 for invalid
 * arguments.  Host only.                                                     */
RSSM_API int64_t gdn_replay_seq_bytes(const rssm_gdn_dims *dims, int32_t T, int32_t kind);

/* GDN flush: S_0 <- (prod alpha_j) S_0 + sum_j (prod_{i>j} alpha_i) u_j k_j^T
 * over the committed entries of flagged sequences; pointer reset as the Mamba-2
 * flush.                                                                      */
RSSM_API rssm_status gdn_replay_flush(const rssm_gdn_dims *dims, const rssm_gdn_replay *st, rssm_stream_t stream);

/* GDN chunked speculative verify (appendix "GDN -- speculative decoding"):
 * with G_s = sum_{r<=s} g_r,
 *   R_s = beta_s (v_s - e^{G_s} S_h k_s),
 *   A_{s,s'} = beta_s e^{G_s - G_s'} (k_s . k_s')  (s' < s),
 *   u_s = R_s - sum_{s'<s} A_{s,s'} u_s'   (T x T lower-triangular solve),
 *   y_s = e^{G_s} S_h q_s + sum_{s'<=s} e^{G_s - G_s'} (k_s' . q_s) u_s'.
 * Drafts (u_s, k_s, g_s) are written tentatively; count is unchanged;
 * flag <- (h + 2T > L).  Commit with replay_spec_commit.
 *   q, k in_dtype [B][T][Hk][dk]  v in_dtype [B][T][Hv][dv]  beta, g float [B][T][Hv]
 *   y y_dtype [B][T][Hv][dv]                                                  */
RSSM_API rssm_status gdn_replay_verify(const rssm_gdn_dims *dims, const rssm_gdn_replay *st, int32_t T, const void *q,
                              const void *k, const void *v, const float *beta, const float *g, void *y,
                              rssm_stream_t stream);

/* GDN chunked verify preceded by the pending flush: the same outputs and
 * state as gdn_replay_flush followed by gdn_replay_verify, issued as those two
 * calls on the stream.  (A fold inside the verify's S_0 stream was measured
 * slower than the persistent flush and verify pipelines back to back at
 * B = 256, Hv = 32, L = 16, T = 4, so no fused launch is kept.)  A speculative
 * round is this call and replay_spec_commit.  Requires st->sync (zero, left
 * zero), as gdn_replay_flush.  Workspace and arguments as gdn_replay_verify. */
RSSM_API rssm_status gdn_replay_verify_fused(const rssm_gdn_dims *dims, const rssm_gdn_replay *st, int32_t T,
                                             const void *q, const void *k, const void *v, const float *beta,
                                             const float *g, void *y, rssm_stream_t stream);

/* Baseline GDN speculative verify: serial correction-form updates per draft
 * with a full snapshot per draft (T+1 slots, as ssm_spec_verify_baseline).
 *   slots float [B][T+1][Hv][dv][dk]   cur int32 [B].  Commit with
 *   ssm_spec_commit_baseline.                                                 */
RSSM_API rssm_status gdn_spec_verify_baseline(const rssm_gdn_dims *dims, int32_t T, float *slots, const int32_t *cur,
                                     const void *q, const void *k, const void *v, const float *beta,
                                     const float *g, void *y, int32_t *err, rssm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Convolution state: the step before the SSM in a Mamba-2 layer             */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t B;        /* sequences */
  int32_t dx;       /* channels of the x sub-projection (H d: the SSM's v) */
  int32_t dbc;      /* channels of each of B and C (G n: the SSM's k and q) */
  int32_t W;        /* convolution width, 2..8; the state keeps W - 1 columns */
  int32_t io_dtype; /* dtype of state, u and the outputs: RSSM_BF16 or RSSM_F32 */
  int32_t silu;     /* 1: SiLU on the outputs, 0: none */
} rssm_conv_dims;

/* Decode step of the convolution state ("Disaggregated Serving for Hybrid
 * SSM Models", Mamba state layout: a per-sequence state of shape (conv_dim,
 * state_len) in the DS layout, conv_dim = dx + 2 dbc, state_len = W - 1; the
 * arithmetic is not on the pages -- this library reads it as the causal
 * depthwise convolution of width W).  Per sequence b and channel c, with
 * the state's columns oldest first and the new input u:
 *   z = bias[c] + sum_{w<W-1} weight[c][w] state[b][c][w] + weight[c][W-1] u[b][c]
 *   out = silu(z) = z / (1 + exp(-z))  (or z),  state[b][c] <- (state[b][c][1..], u[b][c])
 * in fp32; out is rounded to io_dtype and split by channel into x, B, C.
 *   state  io_dtype [B][dx + 2 dbc][W - 1]   (in/out, DS layout)
 *   u      io_dtype [B][dx + 2 dbc]          (the in-projection's x|B|C columns)
 *   weight float [dx + 2 dbc][W]   bias float [dx + 2 dbc] or NULL
 *   out_x  io_dtype [B][dx]   out_b, out_c io_dtype [B][dbc]  (NULL if dbc = 0)
 * The outputs have the layouts of replay_decode_step's v (H = dx / d heads)
 * and k, q (G = dbc / n groups).  The caller owns all memory; pointers are
 * device pointers aligned to their element size.  RSSM_ERR_INVALID_ARG for
 * null or misaligned pointers or dims out of range (B, dx >= 1, dbc >= 0,
 * 2 <= W <= 8, silu 0 or 1).                                                 */
RSSM_API rssm_status conv_state_update(const rssm_conv_dims *dims, void *state, const void *u, const float *weight,
                                       const float *bias, void *out_x, void *out_b, void *out_c,
                                       rssm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Utilities                                                                  */
/* ------------------------------------------------------------------------ */

/* Library version, e.g. 200 for 0.2.0.  Host-only; never fails. */
RSSM_API int32_t rssm_version(void);

/* Element counts of one layer's arrays, for allocation (host only).
 * Mamba-2: S0 = B H d n, ring_v = B H L d, ring_k = B G L n, ring_dt = B H L,
 * per_seq = B (each of start, count, flag, sync).  GDN: S0 = B Hv dv dk,
 * ring_u = B Hv L dv, ring_k = B Hk L dk, ring_g = B Hv L, per_seq = B.
 * RSSM_ERR_INVALID_ARG for null pointers or invalid dims (as the calls).     */
typedef struct {
  int64_t S0, ring_vec, ring_k, ring_decay, per_seq;
} rssm_layout;
RSSM_API rssm_status rssm_m2_layout_sizes(const rssm_m2_dims *dims, rssm_layout *out);
RSSM_API rssm_status rssm_gdn_layout_sizes(const rssm_gdn_dims *dims, rssm_layout *out);

/* Read the sticky device error word (`err` of a state, one int32 in device
 * memory) into *value: an asynchronous copy on `stream`, then a wait for the
 * stream -- the one call of this library that synchronises.  The word is not
 * cleared.  RSSM_ERR_INVALID_ARG for null pointers, RSSM_ERR_CUDA if the copy
 * or the wait fails (rssm_last_cuda_error tells which).                     */
RSSM_API rssm_status rssm_read_error(const int32_t *err, int32_t *value, rssm_stream_t stream);

/* Static description of a status code.  Host-only; never fails. */
RSSM_API const char *rssm_status_string(rssm_status s);

/* Text of the last CUDA error seen by a call on this thread that returned
 * RSSM_ERR_CUDA ("" if none).  Host-only. */
RSSM_API const char *rssm_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H_ */
