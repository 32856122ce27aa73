/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunked gated delta rule forward library (libgdn.so).
 *
 * The operation (per value head, h a K x V state):
 *     h_t = exp(g_t) (I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T,     o_t = h_t^T q_t.
 * It is computed chunk by chunk (C tokens) through the affine chunk map of the page
 * "Add context parallelism to the Gated Delta Net (Qwen3-Next / Qwen3.5)" (MaxText PR #5040),
 * section "Why":
 *     h_out = (gamma I - k_tilde^T w) h + k_tilde^T u = M h + U,
 *     o     = (q_g - attn_i w) h + attn_i u,
 * and long sequences are split into segments that run in parallel on the GPU's SMs by the
 * three phases of its section "Implementation": (1) a zero-state pass per segment carrying
 * M_r in low-rank form, (2) an exclusive prefix scan over (M_r, U_r), (3) a re-emit pass from
 * the true incoming state.  Chunk factors (derived from the recurrence; the page names them
 * without defining them):
 *     G_t = inclusive within-chunk cumulative sum of g;   gamma = exp(G_last)
 *     A[t][j] = beta_t exp(G_t - G_j) (k_t . k_j), j < t;  T = (I + A)^-1
 *     w = T diag(beta exp(G)) K,   u = T diag(beta) V,   k_tilde_j = exp(G_last - G_j) k_j,
 *     q_g_t = exp(G_t) q_t,   attn_i[t][j] = exp(G_t - G_j) (q_t . k_j), j <= t.
 *
 * CONVENTIONS (every entry point)
 *   Ownership   the caller allocates every buffer; the library allocates nothing, keeps no
 *               state between calls and never frees caller memory.
 *   Pointers    all tensor arguments are DEVICE pointers of the current CUDA device; the
 *               problem struct is a HOST pointer read before the call returns.
 *   Execution   asynchronous on `stream` (0 = legacy default stream).  Buffers must stay
 *               valid until the stream reaches the work.
 *   Layouts     row-major, contiguous, no padding between rows:
 *                 q, k      [T, hk, K]      io dtype
 *                 v, out    [T, hv, V]      io dtype
 *                 g, beta   [T, hv]         fp32 (g = natural-log decay, beta = write strength)
 *                 h0, h_final [N, hv, K, V] fp32 (the state layout [Hv, K, V] f32 of the page
 *                           "RFC(qwen35): TP Phase2", section "Partition Contract", per sequence)
 *                 cu_seqlens int32 [N+1]    cu[0] = 0, non-decreasing, cu[N] = T
 *                 w [T, hv, K], u [T, hv, V], gcum [T, hv] fp32 (token aligned)
 *                 M [N*P, hv, K, K], U and h_in [N*P, hv, K, V] fp32; segment (n, r) -> n*P + r
 *               Value head j reads key head j / (hv / hk) (grouped order).
 *   Segments    each sequence's Nc = ceil(L / C) chunks are split into P contiguous,
 *               in-order segments; the first (Nc mod P) segments get one extra chunk; a
 *               segment past Nc is empty (identity map).  A reordered (load-balanced) split
 *               cannot be expressed: the section "Limitation: load balancing must be off"
 *               requires contiguous, in-order pieces.
 *   Tails       a sequence whose length is not a multiple of C ends in a short chunk; it is
 *               computed as if padded with g = 0, q = k = v = 0 (the padding bullet of
 *               "Implementation"), and nothing is written past the sequence.
 *   Validation  host-side checks run before any launch; on failure nothing is enqueued and
 *               GDN_ERR_INVALID_ARGUMENT or GDN_ERR_UNSUPPORTED is returned.  cu_seqlens is
 *               checked ON THE DEVICE (the host never reads it): a bad table leaves the
 *               outputs of the affected sequences unwritten and records
 *               GDN_ERR_DEVICE_INPUT in the status word, read by gdn_device_status().
 *   Supported   io dtype bf16 or fp32; K, V in {64, 128}; C = 64; hv % hk == 0; P >= 1;
 *               16-byte aligned tensor pointers.
 *   Kernels     the problem decides, with no caller-side selection: gdn_forward and the *_fused
 *               stage calls run on the tcgen05 tensor-core kernels for bf16 I/O with K = V = 128
 *               and on the fp32 CUDA-core kernels otherwise; the stage calls that take the
 *               materialised fp32 factors (gdn_chunk_prepare, gdn_segment_summary,
 *               gdn_chunk_emit) run on the fp32 CUDA-core kernels for every I/O dtype.
 *   Precision   fp32 I/O runs on fp32 CUDA-core kernels.  bf16 I/O with K = V = 128 runs on the
 *               tensor cores: K K^T and Q K^T on the bf16 inputs as given, every later product
 *               on fp16 operands (inputs converted exactly in range), fp32 accumulation, an
 *               fp32 triangular solve and an fp32 state.  q, k, v, the state and the corrected
 *               values delta must stay below 65504 in magnitude; a value that does not is
 *               reported as GDN_ERR_DEVICE_RANGE.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned pointer          */
    GDN_ERR_UNSUPPORTED = 2,      /* valid but not built: dtype, K, V, C outside the set  */
    GDN_ERR_WORKSPACE = 3,        /* workspace null or smaller than gdn_workspace_size()  */
    GDN_ERR_CUDA = 4,             /* a CUDA launch or runtime call failed                 */
    GDN_ERR_DEVICE_TIMEOUT = 5,   /* a bounded device-side wait expired                   */
    GDN_ERR_DEVICE_INPUT = 6,     /* the device found cu_seqlens inconsistent             */
    GDN_ERR_DEVICE_RANGE = 7      /* a tensor-core operand left the fp16 range (|x| > 65504) */
} gdn_status;

typedef enum gdn_dtype { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

typedef struct gdn_problem {
    int64_t total_tokens;     /* T >= 0: tokens of the packed stream                     */
    int32_t num_seqs;         /* N >= 1                                                  */
    int32_t hk, hv;           /* key heads, value heads (hv % hk == 0)                   */
    int32_t k_dim, v_dim;     /* K, V                                                    */
    int32_t chunk;            /* C (64)                                                  */
    int32_t segments_per_seq; /* P >= 1                                                  */
    int32_t io_dtype;         /* gdn_dtype of q, k, v and out                            */
} gdn_problem;

/* Status text (static storage; never NULL). */
const char* gdn_status_string(gdn_status s);

/* Checks a problem description on the host (no device work). */
gdn_status gdn_check_problem(const gdn_problem* p);

/* Bytes of device workspace gdn_forward needs for problem p (0 when p is invalid).  The
 * workspace holds the status word, the segment summaries (M_r, U_r), the incoming states
 * h_in, on the SIMT path the materialised chunk factors, and on the tcgen05 path with P > 1
 * per-chunk factor records: -w^T, fp16 K, u^T and the state update's decay, 49,664 bytes per
 * 64-token window and value head.  The U summary writes them; the M summary and phase 3 read
 * them and skip the preparation ("Implementation": phase 3 re-emits with the factors the
 * zero-state pass already computed).  A workspace without room for the records is accepted:
 * every phase then computes its own factors. */
size_t gdn_workspace_size(const gdn_problem* p);

/* Whole forward pass ("Implementation": the three phases; with P = 1 the single-pass form,
 * "the single-device path is the same computation, just reassembled").
 *   q, k, v, g, beta   inputs (layouts above)
 *   h0                 initial states [N, hv, K, V] fp32, or NULL for zeros
 *   cu_seqlens         device int32 [N+1]; may be NULL only when N == 1 (then [0, T])
 *   out                [T, hv, V] io dtype
 *   h_final            [N, hv, K, V] fp32, or NULL to skip
 *   workspace          device buffer of ws_bytes >= gdn_workspace_size(p), 16-byte aligned;
 *                      its first 4 bytes are the status word (reset by this call)
 * Returns GDN_OK once the work is enqueued. */
gdn_status gdn_forward(const gdn_problem* p, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* h0,
                       const int32_t* cu_seqlens, void* out, float* h_final, void* workspace,
                       size_t ws_bytes, cudaStream_t stream);

/* gdn_forward with a per-phase clock: it records CUDA events on `stream` around its launches,
 * waits for the last, and writes four elapsed times in milliseconds to phase_ms[0..3] (a host
 * array): phase 1 (the segment summaries), the prefix scan, phase 3, and the first of phase 1's
 * two kernels (the U half when the workspace holds factor records, else the M half).  A phase
 * that does not run (the summaries and the scan with P = 1) reads 0.  It runs the same kernels
 * as gdn_forward; the wait makes it synchronous.  For measurement only.  Errors: those of
 * gdn_forward, GDN_ERR_INVALID_ARGUMENT for a NULL phase_ms, GDN_ERR_CUDA if an event call
 * fails. */
gdn_status gdn_forward_timed(const gdn_problem* p, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* h0,
                             const int32_t* cu_seqlens, void* out, float* h_final,
                             void* workspace, size_t ws_bytes, cudaStream_t stream,
                             float* phase_ms);

/* gdn_forward with explicit limits, for tests of the device-side failure detection.
 *   wait_cycles   limit of every bounded device wait, in SM clock cycles (0 = the default of
 *                 about a second; a wait that expires records GDN_ERR_DEVICE_TIMEOUT in the
 *                 status word, and the kernel still lets its own copies and products land
 *                 before it releases its memory and exits, so the context stays usable)
 *   fault         0 = none; 1 = the tensor-core chunk kernels' chain never signals its first
 *                 hand-off, so the wait for it expires (the same fault in every CTA)
 * The outputs of a call that reports a device error are unspecified.  Errors: those of
 * gdn_forward; GDN_ERR_INVALID_ARGUMENT for a negative wait_cycles or an unknown fault. */
gdn_status gdn_forward_with_limits(const gdn_problem* p, const void* q, const void* k,
                                   const void* v, const float* g, const float* beta,
                                   const float* h0, const int32_t* cu_seqlens, void* out,
                                   float* h_final, void* workspace, size_t ws_bytes,
                                   cudaStream_t stream, long long wait_cycles, int fault);

/* Phase "prepare": the WY/UT factors of every chunk ("Implementation": the WY factors that
 * phase 3 reuses; "Why": w and u of the chunk map).  Writes w [T, hv, K], u [T, hv, V]
 * (fp32) and gcum [T, hv] (fp32, inclusive within-chunk cumulative log-decay; a chunk's
 * gamma is exp of its last row).  dev_status: device int32 status word or NULL. */
gdn_status gdn_chunk_prepare(const gdn_problem* p, const void* k, const void* v, const float* g,
                             const float* beta, const int32_t* cu_seqlens, void* w, void* u,
                             float* gcum, int32_t* dev_status, cudaStream_t stream);

/* Phase 1: zero-state pass per segment carrying the composed transition ("Implementation",
 * phase 1 and the low-rank composition M_new = gamma M - k_tilde^T (w M)).  From M = I, U = 0,
 * per chunk: U <- gamma U + k_tilde^T (u - w U), M <- gamma M - k_tilde^T (w M).
 * Reads k, w, u, gcum (as written by gdn_chunk_prepare); writes M [N*P, hv, K, K] and
 * U [N*P, hv, K, V] (fp32) for every segment, empty ones as (I, 0). */
gdn_status gdn_segment_summary(const gdn_problem* p, const void* k, const void* w, const void* u,
                               const float* gcum, const int32_t* cu_seqlens, float* M, float* U,
                               int32_t* dev_status, cudaStream_t stream);

/* Phase 2: exclusive prefix scan over the segment summaries ("Implementation", phase 2;
 * "Why": affine maps compose associatively).  h_in[n*P] = h0[n] (zeros when h0 is NULL),
 * h_in[n*P + r + 1] = M[n*P + r] h_in[n*P + r] + U[n*P + r]; h_final[n] is the map of the
 * last segment applied once more (NULL to skip).  Pure fp32; needs no cu_seqlens. */
gdn_status gdn_state_prefix_scan(const gdn_problem* p, const float* M, const float* U,
                                 const float* h0, float* h_in, float* h_final,
                                 cudaStream_t stream);

/* Phase 3: re-emit from the true incoming states, reusing the chunk factors
 * ("Implementation", phase 3; "Why": o = (q_g - attn_i w) h + attn_i u).  Per chunk:
 * delta = u - w h, o = q_g h + attn_i delta, h <- gamma h + k_tilde^T delta.
 * h_in [N*P, hv, K, V] fp32 (NULL = zeros); writes out and, from each sequence's last
 * segment, h_final (NULL to skip). */
gdn_status gdn_chunk_emit(const gdn_problem* p, const void* q, const void* k, const void* w,
                          const void* u, const float* gcum, const float* h_in,
                          const int32_t* cu_seqlens, void* out, float* h_final,
                          int32_t* dev_status, cudaStream_t stream);

/* Phase 1 with the chunk factors recomputed on chip (no materialised w, u): the same M_r,
 * U_r as gdn_chunk_prepare followed by gdn_segment_summary, read straight from k, v, g, beta.
 * With skip_last != 0 the last segment of each sequence is not summarised (the forward pass
 * never reads it).  Tensor-core family only (bf16, K = V = 128); GDN_ERR_UNSUPPORTED
 * otherwise. */
gdn_status gdn_segment_summary_fused(const gdn_problem* p, const void* k, const void* v,
                                     const float* g, const float* beta,
                                     const int32_t* cu_seqlens, float* M, float* U,
                                     int skip_last, int32_t* dev_status, cudaStream_t stream);

/* Phase 3 with the chunk factors recomputed on chip: the same out and h_final as
 * gdn_chunk_prepare followed by gdn_chunk_emit.  h_in [N*P, hv, K, V] fp32 or NULL (zeros).
 * Tensor-core family only (bf16, K = V = 128); GDN_ERR_UNSUPPORTED otherwise. */
gdn_status gdn_chunk_emit_fused(const gdn_problem* p, const void* q, const void* k,
                                const void* v, const float* g, const float* beta,
                                const float* h_in, const int32_t* cu_seqlens, void* out,
                                float* h_final, int32_t* dev_status, cudaStream_t stream);

/* Reads (synchronously: it waits for `stream`) the status word at `status_word` -- a
 * dev_status pointer or a gdn_forward workspace -- and clears it when `reset` != 0.
 * Returns the recorded status (GDN_OK when none), or GDN_ERR_CUDA if the read failed. */
gdn_status gdn_device_status(const void* status_word, int reset, cudaStream_t stream);

/* gdn_forward for callers that cannot allocate device memory (for example a plug-in whose host
 * framework owns all device memory, or a serving loop with a fixed memory plan that forbids
 * allocations after start-up).  It takes no workspace: its scratch is a 64 MiB array in the
 * library's own device memory, which every GPU that loads the library holds until the process
 * exits.  There is no counterpart on the source pages; this is a deployment convenience.
 *   - Same arguments, results and errors as gdn_forward, minus the workspace.  What must fit in
 *     64 MiB is the workspace without the optional per-chunk factor tiles: the status word and,
 *     with P > 1, the segment summaries and incoming states (192 KiB per segment and value head
 *     at K = V = 128, so N * P * hv <= 341).  A problem needing more is rejected with
 *     GDN_ERR_WORKSPACE before anything is enqueued; one whose full gdn_workspace_size() exceeds
 *     64 MiB but whose minimum fits runs without the factor tiles.
 *   - It allocates nothing (no cudaMalloc, no allocating library call).
 *   - All calls on a device share the one array, which keeps the last call's contents (each
 *     call clears the status word; nothing else needs to start at zero).  Calls whose work
 *     overlaps on the GPU (different streams without ordering, or concurrent host threads)
 *     race on it: order them on one stream.
 *   - The first call on a device looks up the array's device address with that device current
 *     and caches it; make that first call before any stream capture.
 *   - The status word is the array's first word; it is not exposed, so read a device-side
 *     error by repeating the call through gdn_forward with a workspace if one is reported. */
gdn_status gdn_forward_static_scratch(const gdn_problem* p, const void* q, const void* k,
                                      const void* v, const float* g, const float* beta,
                                      const float* h0, const int32_t* cu_seqlens, void* out,
                                      float* h_final, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------- */
/* Backward: gradients of the forward pass.                                                 */

/* Bytes of device workspace gdn_backward needs for problem p (0 when p is invalid): the status
 * word, the state entering and the gradient of the state leaving every chunk (fp32, 2 * 4 * K *
 * V bytes per chunk and value head each way), per-value-head dq and dk (fp32), and the
 * intermediates of 304 concurrent per-chunk blocks. */
size_t gdn_backward_workspace_size(const gdn_problem* p);

/* Gradients of L = <dout, out> + <dh_final, h_final> through the forward of gdn_forward
 * (the same problem, inputs and h0) with respect to q, k, v, g, beta and h0.  The page "Add
 * context parallelism to the Gated Delta Net" holds the layer's backward to parity (sections
 * "Tests" and "Measured results"); its formulas follow from the chunk map of section "Why".
 *   dout        [T, hv, V] io dtype            dh_final  [N, hv, K, V] fp32, or NULL (zeros)
 *   dq, dk      [T, hk, K] io dtype (a key head's gradient sums over the value heads reading it)
 *   dv          [T, hv, V] io dtype            dg, dbeta [T, hv] fp32
 *   dh0         [N, hv, K, V] fp32, or NULL to skip
 *   workspace   ws_bytes >= gdn_backward_workspace_size(p), 16-byte aligned; its first 4 bytes
 *               are the status word (reset by this call)
 * segments_per_seq is not used.  The state recurrences and the triangular factors are fp32
 * arithmetic on CUDA cores; the per-chunk products run on the tensor cores with fp32
 * accumulation, their operands rounded to TF32 for bf16 I/O and split into two TF32 parts
 * (fp32 accuracy) for fp32 I/O.  Tails, padding, cu_seqlens checks and errors as for
 * gdn_forward.  Returns GDN_OK once the work is enqueued. */
gdn_status gdn_backward(const gdn_problem* p, const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* h0,
                        const int32_t* cu_seqlens, const void* dout, const float* dh_final,
                        void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------- */
/* Prologue: the layer-side steps that produce q, k, v, g, beta from the projections.          */

typedef struct gdn_prologue_problem {
    int64_t total_tokens;     /* T >= 0                                                     */
    int32_t num_seqs;         /* N >= 1                                                     */
    int32_t hk, hv;           /* key heads, value heads (hv % hk == 0)                      */
    int32_t k_dim, v_dim;     /* K, V: multiples of 8 up to 128                             */
    int32_t conv_width;       /* W in [1, 4]: taps of the causal conv                       */
    int32_t activation;       /* 0: none, 1: SiLU after the conv                            */
    int32_t io_dtype;         /* gdn_dtype of x, the conv states, a, b, q, k, v             */
} gdn_prologue_problem;

/* The layer prologue ahead of the recurrence (page "Add context parallelism to the Gated Delta
 * Net", section "Implementation", layer-side bullets: a causal depthwise conv over the q | k | v
 * channels with a halo of conv_kernel_dim - 1 tokens; page "RFC(qwen35): TP Phase2", section
 * "Partition Contract": a per-request conv state of qkv_dim x (conv_kernel_dim - 1) inputs).
 * With Ch = 2 hk K + hv V channels (q's, then k's, then v's):
 *     y_t[c] = sum_{i < W} conv_w[c][i] x_{t-W+1+i}[c]     (inputs before a sequence's start
 *              come from conv_state_in[n][c][0 .. W-2], oldest first, or are 0 when it is NULL)
 *     y -> SiLU(y) when activation = 1;  q, k = their channels / max(L2 norm, 1e-6) per head;
 *     v = its channels;  g = -exp(A_log) softplus(a + dt_bias);  beta = sigmoid(b)
 * (the optional SiLU, the L2 normalisation and the g, beta maps are readings: the pages name
 * these steps without formulas).
 *   x [T, Ch] io dtype;  conv_w [Ch, W] fp32;  conv_state_in, conv_state_out [N, Ch, W-1] io dtype
 *   (either may be NULL; out may alias in: it receives each sequence's last W-1 inputs, older
 *   entries shifting in when a sequence is shorter);  a, b [T, hv] io dtype;  A_log, dt_bias
 *   [hv] fp32;  outputs q, k [T, hk, K], v [T, hv, V] io dtype, g, beta [T, hv] fp32, in the
 *   layouts gdn_forward reads.  x, q, k, v 16-byte aligned.  cu_seqlens as for gdn_forward
 *   (device-checked; dev_status records GDN_ERR_DEVICE_INPUT).  HBM-bound elementwise kernels. */
gdn_status gdn_prologue(const gdn_prologue_problem* p, const void* x, const float* conv_w,
                        const void* conv_state_in, const void* a, const void* b,
                        const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                        void* q, void* k, void* v, float* g, float* beta, void* conv_state_out,
                        int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------- */
/* Decode: one token per request over a pool of per-slot recurrent states.                   */

typedef struct gdn_decode_problem {
    int32_t batch;            /* B >= 0 rows (requests), one token each                     */
    int32_t slots;            /* S >= 1 states in the pool                                  */
    int32_t hk, hv;           /* key heads, value heads (hv % hk == 0)                      */
    int32_t k_dim, v_dim;     /* K, V in {64, 128}                                          */
    int32_t io_dtype;         /* gdn_dtype of q, k, v and out                               */
} gdn_decode_problem;

/* Checks a decode problem description on the host (no device work). */
gdn_status gdn_check_decode_problem(const gdn_decode_problem* p);

/* One decode step (page "RFC(qwen35): TP Phase2": section "Execution Contract" -- the decode
 * kernels run against the head and state shapes and update only request-local recurrent
 * state; section "Partition Contract" -- the state is [Hv, K, V] f32 per request; section
 * "Request-State Lifecycle" -- requests live in slots that are reused).  Row b is the next
 * token of the request whose state is state[slot[b]]; per value head j (key head
 * j / (hv / hk)), with h that state:
 *     h <- exp(g) (I - beta k k^T) h + beta k v^T,     out = h^T q
 * -- the token recurrence of gdn_forward, one token long, continuing from the slot's state.
 *   q, k        [B, hk, K] io dtype          v, out   [B, hv, V] io dtype
 *   g, beta     [B, hv] fp32                 state    [S, hv, K, V] fp32, updated in place
 *   slot        device int32 [B]: the state slot of each row.  A negative entry marks a
 *               padding row: its out row is set to 0 and no state is read or written.
 *   dev_status  device int32 status word, or NULL
 * Slots are checked on the device: a row whose slot is >= S, or is named by another row too,
 * is skipped (its state and out row are left untouched) and GDN_ERR_DEVICE_INPUT is recorded in
 * dev_status; the other rows are computed.  A slot is started from a prefill by passing
 * state + slot * hv * K * V as gdn_forward's h_final (one sequence), or from zero by clearing
 * it; nothing of a previous request survives either.  All tensor pointers 16-byte aligned.
 * Runs on fp32 CUDA-core arithmetic (the step is bound by the state's HBM traffic: 2 * 4 * K * V
 * bytes per row and value head).  Returns GDN_OK once the work is enqueued. */
gdn_status gdn_decode_step(const gdn_decode_problem* p, const void* q, const void* k,
                           const void* v, const float* g, const float* beta,
                           const int32_t* slot, float* state, void* out, int32_t* dev_status,
                           cudaStream_t stream);

/* Text of the last CUDA error that made an entry point return GDN_ERR_CUDA on the calling
 * host thread ("no CUDA error" when there was none).  Static storage. */
const char* gdn_last_error_string(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
