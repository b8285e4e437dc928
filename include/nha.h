/*
 * libnha -- Native Hybrid Attention (NHA) layer operator, forward and backward,
 * for NVIDIA GB300 (sm_103a).  C ABI: plain pointers and sizes only.
 *
 * The operator ("Native Hybrid Attention for Efficient Sequence Modeling",
 * Paper-Notes page, section 关键设计/层内混合, the K^long_t recurrence and the
 * o_t = softmax(q_t K^H_t^T / sqrt(d)) V^H_t equation; "整体框架" for the
 * memory shapes; the chunkwise form in section "Chunkwise 并行计算"):
 *
 *   per (b,h), tokens t = 0..T-1, slots i = 0..m-1,
 *     alpha_t = exp(log_alpha_t),  u_t = 1 - alpha_t   (computed as -expm1)
 *     long memory after token j:
 *        K^long_j = Diag(alpha_j) K^long_{j-1} + u_j (x) k_j,  V^long likewise,
 *        zero before token 0;
 *     query t reads the long memory after token j = t - w (token shift: only
 *     tokens that have left the window are absorbed); when t < w no token has
 *     left yet and all m slot logits are masked;
 *     slot logits   L_{t,i} = q_t . K^long_{t-w}[i] / sqrt(d)   (no position code)
 *     window logits S_{t,s} = rope(q_t, t) . rope(k_s, s) / sqrt(d),
 *                   s in [max(0, t-w+1), t]
 *     p = one softmax over [L_t | S_t];  lse_t = log of its partition
 *     o_t = sum_i p_{t,i} V^long_{t-w}[i] + sum_s p_{t,s} v_s
 *   RoPE: rotate-half pairing (i, i + d/2), theta_i = rope_base^(-2i/d),
 *   absolute 0-based positions.  w = 0 is a pure gated-slot RNN; w >= T is
 *   causal softmax attention (w > T is treated as T).
 *
 * Layout: q, k, v, o, dout, dq, dk, dv are contiguous row-major [B, H, T, d]
 * in the element type `dtype`; log_alpha and dlog_alpha are [B, H, T, m] fp32;
 * lse is [B, H, T] fp32.  Every pointer is a DEVICE pointer, 16-byte aligned.
 *
 * Supported: d in {64, 128}; m in {16, 32, 64}; C == 64 (the chunk length of
 * the chunkwise-parallel form; results depend on C only through rounding);
 * 0 <= T <= 262144; w >= 0; B*H*T*max(d,m) < 2^31.
 * Numerical range: within any chunk of C consecutive tokens, the per-slot sum
 * of log_alpha must be >= -160 (the intra-chunk gate factorisation is exact in
 * fp32 only inside that range).
 *
 * Ownership: the caller allocates every buffer, including the workspace
 * (size from nha_workspace_bytes).  The library never allocates or frees
 * device memory and never synchronises; work is enqueued on `stream` (a
 * cudaStream_t; NULL means the legacy default stream).  The bf16 path also
 * runs independent kernels on an internal non-blocking stream, one per host
 * thread and device with four events, created on the first bf16 call and
 * kept until the process exits: that stream waits on `stream` before its
 * kernels and `stream` waits on it after them (events), so all results are
 * complete when the work enqueued on `stream` is, and stream capture records
 * the fork and join as graph edges.  Make the first bf16 call of a host
 * thread outside stream capture.  Outputs are fully overwritten, never
 * accumulated.
 *
 * Errors: every entry point returns a status and never throws.  Arguments are
 * validated before anything is enqueued; a failed launch maps to
 * NHA_ERR_CUDA.  Faults inside kernels surface at the caller's next
 * synchronisation.  nha_last_error() gives a thread-local message for the
 * last failing call on this thread.
 *
 * Re-entrancy: reentrant; the process-wide state is lazily set kernel
 * attributes and the per-thread side streams above.  Calls on different
 * streams with different workspaces may run concurrently.
 */
#ifndef NHA_H_
#define NHA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NHA_OK = 0,
    NHA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, negative size, bad enum */
    NHA_ERR_UNSUPPORTED = 2,      /* valid but outside the supported d, m, C, T set */
    NHA_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required */
    NHA_ERR_CUDA = 4,             /* a CUDA runtime call or kernel launch failed */
    NHA_ERR_INTERNAL = 5          /* host-side fault injection or an internal check */
} nha_status_t;

typedef enum { NHA_DTYPE_F32 = 0, NHA_DTYPE_BF16 = 1 } nha_dtype_t;

/* Bytes of device workspace nha_forward (backward = 0) or nha_backward
 * (backward = 1) needs for this shape.  Returns 0 for an invalid or
 * unsupported shape (nha_forward / nha_backward then report why). */
size_t nha_workspace_bytes(int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dtype,
                           int backward);

/* Forward.  Writes o [B,H,T,d] (dtype) and lse [B,H,T] (fp32, natural log of
 * the softmax partition, kept for nha_backward). */
nha_status_t nha_forward(const void* q, const void* k, const void* v, const float* log_alpha,
                         void* o, float* lse, int B, int H, int T, int d, int m, int w, int C,
                         nha_dtype_t dtype, float rope_base, void* workspace, size_t ws_bytes,
                         void* stream);

/* Backward of loss = <o, dout>.  Takes the forward's o and lse.  Writes
 * dq, dk, dv [B,H,T,d] (dtype; gradients w.r.t. the un-rotated q and k) and
 * dlog_alpha [B,H,T,m] (fp32). */
nha_status_t nha_backward(const void* q, const void* k, const void* v, const float* log_alpha,
                          const void* o, const float* lse, const void* dout, void* dq, void* dk,
                          void* dv, float* dlog_alpha, int B, int H, int T, int d, int m, int w,
                          int C, nha_dtype_t dtype, float rope_base, void* workspace,
                          size_t ws_bytes, void* stream);

/* ---- Extended calls: optional inputs and outputs ----
 *
 * nha_forward_ex / nha_backward_ex are nha_forward / nha_backward with an
 * optional nha_extras_t (NULL, or a zero-initialised struct, gives exactly
 * the plain calls).  Every pointer in it is optional (NULL = not used) and, if
 * given, a DEVICE pointer with the layout stated beside it.
 *
 * fwd_workspace (backward only): the workspace the forward of the same
 * inputs ran with (nha_forward or nha_forward_ex, same shape, dtype and
 * rope_base), untouched since.  The backward then reads the chunk states,
 * gate totals, RoPE table and rotated q, k the forward left there instead of
 * forming them again, and its own workspace shrinks accordingly
 * (nha_workspace_bytes_ex with the same extras).  This is the usual
 * saved-for-backward context of a training step: keep the forward's
 * workspace alive until the backward has been enqueued after it.
 *
 * Slot states (fp32 [B, H, m, d] each, K and V parts given together):
 *   h0_k, h0_v   initial states: the long memory before token 0 (the ai.info
 *                page, Future Directions: learned initial slot states).  The
 *                memory is then never empty: no slot logit is masked, and the
 *                queries t < w read h0 itself (no gate applies to it before
 *                token 0).  Forward and backward take the same h0.
 *   hT_k, hT_v   forward output: the final states, the long memory after the
 *                last token that left the window (token T - w - 1), i.e. the
 *                state nha_decode_step continues from at t = T; h0 (or zero)
 *                when w >= T.  A sequence cut into segments continues exactly
 *                when each later segment runs on [the previous w tokens; its
 *                own tokens] with the previous segment's hT as h0 and drops
 *                the outputs of those first w queries (window logits depend
 *                on positions only through t - s, so each segment may count
 *                positions from its own start).
 *   dhT_k, dhT_v backward input: the gradient of the loss with respect to hT
 *                (the loss is then <o, dout> + <hT, dhT>).
 *   dh0_k, dh0_v backward output: the gradient with respect to h0 (needs h0).
 *
 * windows: DEVICE array [H] of int32, or NULL: head h (of every batch entry)
 * has its own window min(max(windows[h], 0), w), so w is the largest window;
 * all heads still run in the same launches (the ai.info page: randomised
 * window sizes in training, per-layer / per-head window schedules).  The
 * workspace is then laid out for the smallest possible window (w = 0), so
 * pass the same extras to nha_workspace_bytes_ex; forward and backward (and
 * a forward workspace the backward reuses) must see the same windows.  The
 * host cannot check device values: a value outside [0, w] is clamped.
 *
 * windows_per_sequence: 0, or 1 when windows holds B * H entries, entry
 * b * H + h for head h of batch entry b (per-sequence windows).
 *
 * cu_seqlens: DEVICE array [B + 1] of int32 offsets, or NULL (varlen
 * batches: sequences of different lengths in one call).  Batch entry b is
 * then a sequence of
 * T_b = cu_seqlens[b + 1] - cu_seqlens[b] tokens (clamped to [0, T]) held in
 * rows t < T_b of its T rows in every token array (q, k, v, log_alpha, o,
 * lse, dout, dq, dk, dv, dlog_alpha), and is computed exactly as a call of
 * T_b tokens would compute it: its own window clamp min(w, T_b), hT the
 * state after its token T_b - w - 1, h0 / dh0 / dhT per sequence.  Tiles
 * overlapping rows t >= T_b read them as padding, so those rows of every
 * input must hold finite values (zeros will do), o and lse included when the
 * backward reads them; the forward and backward leave those rows of their
 * outputs unspecified.  The workspace is laid out as for per-head windows
 * (pass the same extras to nha_workspace_bytes_ex).  nha_varlen_pad /
 * nha_varlen_unpad move packed sequences into and out of this layout. */
typedef struct {
    const void* fwd_workspace; /* backward: the forward's workspace, read only */
    size_t fwd_ws_bytes;       /* its size in bytes */
    const float* h0_k;
    const float* h0_v;
    float* hT_k;
    float* hT_v;
    const float* dhT_k;
    const float* dhT_v;
    float* dh0_k;
    float* dh0_v;
    const int* windows; /* DEVICE [H] (or [B * H]) int32 windows, or NULL */
    int* status;        /* DEVICE int32, or NULL: the call's status word (below) */
    int windows_per_sequence; /* 1: windows holds B * H entries */
    const int* cu_seqlens;    /* DEVICE [B + 1] int32 sequence offsets, or NULL */
} nha_extras_t;

/* Packed <-> padded token rows for cu_seqlens calls.
 *   packed: [H, Ttot, width]: the B sequences concatenated along the token
 *           axis, sequence b in rows cu_seqlens[b] .. cu_seqlens[b + 1] - 1
 *           (the layout of a B = 1 call over all Ttot tokens);
 *   padded: [B, H, T, width]: sequence b in rows t < T_b of batch entry b.
 * width elements of elem_bytes bytes (2 or 4) per row, width * elem_bytes a
 * multiple of 4; both arrays DEVICE, 4-byte aligned, on `stream`.
 * nha_varlen_pad writes every padded row: rows t < T_b from the packed
 * array, the rest zero.  nha_varlen_unpad writes packed rows only, those of
 * rows t < T_b.  A row whose packed index falls outside [0, Ttot) is skipped
 * (zero in the padded array); T_b is clamped to [0, T] as in the calls. */
nha_status_t nha_varlen_pad(const void* packed, void* padded, const int* cu_seqlens, int B, int H, int T,
                            int Ttot, int width, int elem_bytes, void* stream);
nha_status_t nha_varlen_unpad(const void* padded, void* packed, const int* cu_seqlens, int B, int H, int T,
                              int Ttot, int width, int elem_bytes, void* stream);

/* Device-side status of a call.  Conditions only the GPU sees cannot be
 * returned by the call itself (it returns once the work is enqueued), so
 * every forward / backward keeps a status word: it sets the word to zero on
 * its stream first, and its kernels OR in these bits.  The word is
 * extras->status when given (read it after the stream has finished the
 * call), else a word in the workspace.
 *   NHA_STATUS_TIMEOUT     a tensor-core kernel's bounded wait on its copies or
 *                          MMAs gave up (about 2 s); its outputs are NaN or
 *                          incomplete and the call's results are void.
 *   NHA_STATUS_GATE_RANGE  the per-slot sum of log_alpha over some chunk of C
 *                          tokens is below -160, outside the range where the
 *                          intra-chunk gate factorisation is exact in fp32; the
 *                          results may hold inf or NaN (see "Numerical range"). */
#define NHA_STATUS_TIMEOUT 1
#define NHA_STATUS_GATE_RANGE 2

/* Sets *status (DEVICE int32) to zero, then runs one bounded wait on a
 * barrier that nothing arrives at, giving up after `cycles` SM clock cycles
 * (0 < cycles <= 2^32): *status becomes NHA_STATUS_TIMEOUT.  Checks, on the
 * GPU, the path by which kernels report a wait that ran out, without any
 * copy or tensor-core work in flight. */
nha_status_t nha_selftest_wait(int* status, long long cycles, void* stream);

/* Workspace bytes of nha_forward_ex (backward = 0) / nha_backward_ex
 * (backward = 1) with these extras; 0 for an invalid or unsupported shape. */
size_t nha_workspace_bytes_ex(int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dtype,
                              int backward, const nha_extras_t* extras);

nha_status_t nha_forward_ex(const void* q, const void* k, const void* v, const float* log_alpha,
                            void* o, float* lse, int B, int H, int T, int d, int m, int w, int C,
                            nha_dtype_t dtype, float rope_base, const nha_extras_t* extras,
                            void* workspace, size_t ws_bytes, void* stream);

nha_status_t nha_backward_ex(const void* q, const void* k, const void* v, const float* log_alpha,
                             const void* o, const float* lse, const void* dout, void* dq, void* dk,
                             void* dv, float* dlog_alpha, int B, int H, int T, int d, int m, int w,
                             int C, nha_dtype_t dtype, float rope_base, const nha_extras_t* extras,
                             void* workspace, size_t ws_bytes, void* stream);

/* ---- Segments of one sequence (sequence parallelism) ----
 *
 * A sequence cut into segments [a_r, b_r) continues exactly when segment r runs
 * nha_forward_ex on [the w tokens before a_r; its own tokens] with h0 = the
 * long memory after token a_r - w - 1, and drops the first w outputs (see
 * hT above).  That h0 follows from per-segment summaries by an associative
 * scan: with S_r the final state of segment r's run started from zero states
 * and A_r the product of the gates of the tokens that left its window,
 *   h0_{r+1} = A_r o h0_r + S_r   (o: per slot, broadcast over d),
 * so every segment can form its summary at once and the scan is the only
 * exchange.  In the backward the state adjoint runs the other way:
 *   g_r = dh0_r + A_r o g_{r+1},  and segment r's dhT is g_{r+1}.
 * (The Paper-Notes page, 局限, leaves contexts beyond 128K unvalidated; this is
 * the exchange a sequence split across ranks needs.) */

/* decay[b,h,i] = exp(sum of log_alpha[b,h,j,i] over j < T - w) (1 when T <= w):
 * A_r above for a run of T tokens.  log_alpha [B,H,T,m] fp32, decay [B,H,m]
 * fp32, DEVICE pointers (log_alpha unused when T <= w). */
nha_status_t nha_gate_total(const float* log_alpha, float* decay, int B, int H, int T, int m, int w,
                            void* stream);

/* out = decay o prev + cur for the K and V parts ([B,H,m,d] fp32 each, decay
 * [B,H,m] broadcast over d): one step of the scan above, forward or
 * backward.  out may be the same arrays as cur. */
nha_status_t nha_state_combine(const float* decay, const float* prev_k, const float* prev_v,
                               const float* cur_k, const float* cur_v, float* out_k, float* out_v,
                               int B, int H, int m, int d, void* stream);

/* ---- Recurrent decode step ----
 *
 * The operator above taken for one new token t of every (b, h) (same page,
 * section 关键设计/层内混合; section 局限 names this recurrent inference mode
 * as the part its authors left unoptimised).  Per (b, h):
 *   1. if t >= w, token j = t - w leaves the window and enters the long memory
 *      with its own gate:  K^long = Diag(alpha_j) K^long + u_j (x) k_j, V^long
 *      likewise (state_k, state_v updated in place); while t < w the slot
 *      logits are masked and the states are left untouched;
 *   2. slot logits q_t . K^long[i] / sqrt(d) (no position code); window logits
 *      rope(q_t, t) . rope(k_s, s) / sqrt(d) for s in [max(0, t-w+1), t];
 *   3. o_t = one softmax over [slots | window] applied to [V^long | v_s];
 *   4. token t (raw k, v and log_alpha) is written into ring entry t mod w.
 * Calling it for t = 0, 1, ..., T-1 from zero states gives the o of
 * nha_forward on the same sequence (up to rounding).
 *
 * Layout (all DEVICE pointers, 16-byte aligned, contiguous row-major):
 *   q, k, v, o     [B, H, d]     element type `dtype` (token t)
 *   log_alpha      [B, H, m]     fp32 (token t)
 *   state_k/_v     [B, H, m, d]  fp32, in/out: K^long, V^long after token
 *                                t - w - 1 on entry, after t - w on return;
 *                                zero before the first token is absorbed
 *   ring_k/_v      [B, H, w, d]  element type, in/out: token s in entry s mod w
 *   ring_la        [B, H, w, m]  fp32, in/out, same indexing
 * Entries of the ring are read only for tokens s in [max(0, t-w), t-1], which
 * earlier calls wrote; with w = 0 the ring pointers are not used (may be NULL).
 * All heads share the position t.  Supported d, m as above; 0 <= t < 262144;
 * 0 <= w <= 262144.  Ownership, errors and streams as for nha_forward; the
 * call needs no workspace and runs on `stream` alone.  Two calls on the same
 * state and ring must be ordered (same stream, or an event between them). */
nha_status_t nha_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                             float* state_k, float* state_v, void* ring_k, void* ring_v, float* ring_la,
                             int t, int B, int H, int d, int m, int w, nha_dtype_t dtype, float rope_base,
                             void* stream);

/* nha_decode_step with launch flags (0 gives exactly nha_decode_step).
 *
 * Every decode launch may start before the kernel enqueued just before it on
 * `stream` has finished (programmatic dependent launch): it reads and writes
 * nothing before that kernel is done, so only its setup overlaps.
 * NHA_DECODE_OVERLAP: the caller states that the kernel enqueued just before
 * this call writes none of this call's state_k, state_v, ring_k, ring_v,
 * ring_la (they belong to another layer, as in a stack of layers decoding
 * one token each in turn).  The step then starts streaming its slot states
 * and window ring in while that kernel is still running, and waits for it
 * only before reading q, k, v, log_alpha and before writing.  Wrong when the
 * previous kernel updates the same state (two steps of one layer back to
 * back): leave the flag off there.  Unknown flag bits are rejected. */
#define NHA_DECODE_OVERLAP 1u
nha_status_t nha_decode_step_ex(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                                float* state_k, float* state_v, void* ring_k, void* ring_v, float* ring_la, int t,
                                int B, int H, int d, int m, int w, nha_dtype_t dtype, float rope_base, unsigned flags,
                                void* stream);

/* nha_decode_step with a position per sequence and, optionally, a window per
 * head.  Sequence b's heads decode token positions[b] (positions: DEVICE
 * array [B] of int32, read by the kernel, so a captured CUDA graph can be
 * replayed while the caller advances the positions on the device);
 * sequences at different positions share one launch (continuous batching).
 * windows (DEVICE array [H] of int32, or NULL for w everywhere): head h keeps
 * a window of windows[h] tokens, 0 <= windows[h] <= w, in the first
 * windows[h] entries of its w-entry ring (token s in entry s mod windows[h];
 * a window of 0 makes that head a pure slot RNN); per-head windows in one
 * launch (the pages' non-uniform window schedules, Future Directions).
 * A head whose position lies outside [0, 262144) or whose window lies outside
 * [0, w] gets o = NaN and its state and ring are left untouched (the host
 * cannot check device values).  Everything else as nha_decode_step. */
nha_status_t nha_decode_step_varlen(const void* q, const void* k, const void* v, const float* log_alpha,
                                    void* o, float* state_k, float* state_v, void* ring_k, void* ring_v,
                                    float* ring_la, const int* positions, const int* windows, int B, int H,
                                    int d, int m, int w, nha_dtype_t dtype, float rope_base, void* stream);

/* Decode state after a prompt of T tokens (the same recurrence and token shift
 * as above): writes state_k, state_v = K^long, V^long after token T - w - 1
 * (zero when T <= w) and puts token s of the prompt (raw k, v and log_alpha)
 * into ring entry s mod w for s in [max(0, T-w), T-1]; other ring entries
 * are left as they are (the decode step never reads them before writing
 * them).  nha_decode_step(..., t = T, ...) then continues the sequence: its
 * o equals that of nha_forward on the prompt extended by token T.
 * Layout: k, v [B, H, T, d] (dtype), log_alpha [B, H, T, m] fp32, the state
 * as for nha_decode_step; all fully written except the ring entries named
 * above.  With T = 0, k, v and log_alpha are not read (may be NULL); with
 * w = 0 the ring pointers are not used.  0 <= T <= 262144; d, m, w as for
 * nha_decode_step.  windows: as for nha_decode_step_varlen (DEVICE array [H]
 * or NULL); a head with a window outside [0, w] gets NaN states and no ring
 * writes.  No workspace; runs on `stream`. */
nha_status_t nha_decode_prefill(const void* k, const void* v, const float* log_alpha, float* state_k,
                                float* state_v, void* ring_k, void* ring_v, float* ring_la,
                                const int* windows, int B, int H, int T, int d, int m, int w,
                                nha_dtype_t dtype, void* stream);

/* ---- Forward without device allocation (the pages have no counterpart) ----
 *
 * Some callers cannot allocate device memory: plugins that receive only
 * their input and output buffers from a host framework, or processes whose
 * device memory belongs to an allocator they may not call.  nha_forward_noalloc is nha_forward with
 * its workspace taken from a fixed scratch array of NHA_NOALLOC_SCRATCH_BYTES
 * compiled into the library (every GPU that loads the library keeps that
 * array until the process exits).  It allocates and frees nothing.
 *
 * Limit: shapes whose forward workspace (nha_workspace_bytes(..., 0)) exceeds
 * NHA_NOALLOC_SCRATCH_BYTES are rejected with NHA_ERR_WORKSPACE before any
 * work is enqueued.  The workspace grows as w shrinks (more tokens leave the
 * window), so compare nha_workspace_bytes(..., 0) for the shape and window at
 * hand against NHA_NOALLOC_SCRATCH_BYTES.
 * Set-up: the first call on a device (and the first call after that device's
 * context was replaced, e.g. by cudaDeviceReset) looks up the scratch's
 * device address in the current context (cudaGetSymbolAddress).
 * Sharing: all calls use the same scratch, which keeps the last call's
 * contents (the forward overwrites every part it reads, so nothing has to
 * start at zero).  Calls whose execution overlaps on the GPU (different
 * streams, or concurrent host threads) race on it: serialise them. */
#define NHA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

nha_status_t nha_forward_noalloc(const void* q, const void* k, const void* v, const float* log_alpha,
                                 void* o, float* lse, int B, int H, int T, int d, int m, int w, int C,
                                 nha_dtype_t dtype, float rope_base, void* stream);

/* ---- Instrumentation (the pages have no counterpart; used by the benchmark) ---- */

/* Number of kernels this library has launched in this process so far. */
unsigned long long nha_launch_count(void);

typedef struct {
    char name[64];    /* kernel name */
    int launches;     /* launches recorded in the session */
    double total_ms;  /* sum of their CUDA-event durations */
} nha_profile_record_t;

/* Opens a profiling session: until nha_profile_end, every kernel launch is
 * bracketed by CUDA events recorded on its own stream (this adds two event
 * records per launch).  Process-wide; not for concurrent sessions. */
nha_status_t nha_profile_begin(void);

/* Closes the session, waits for its events and writes up to `cap`
 * per-kernel records to `out`.  Returns the number of distinct kernels seen,
 * or -1 if an event could not be read. */
int nha_profile_end(nha_profile_record_t* out, int cap);

/* Static description of a status code. */
const char* nha_status_string(nha_status_t status);

/* Message of the last failing call on the calling thread ("" if none). */
const char* nha_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NHA_H_ */
