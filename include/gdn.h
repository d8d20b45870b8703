/*
 * gdn.h -- C ABI of libgdn: the gated-delta SSM (Gated DeltaNet) layer step on
 * NVIDIA GB300 (sm_103a).
 *
 * CONVENTIONS (every entry point)
 *   Memory      Every array argument is DEVICE memory owned by the caller
 *               (allocated by whatever allocator the caller uses). The library
 *               never allocates, frees, or keeps a pointer past the call.
 *   Streams     Work is enqueued on `stream` (NULL = the legacy default
 *               stream). No entry point synchronises; results are ready when
 *               the stream reaches them. Calls other than
 *               gdn_prefill_chunked_noalloc may be captured into CUDA
 *               graphs. gdn_decode_step, gdn_decode_step_bf16_state,
 *               gdn_decode_step_select, gdn_verify_k2 and gdn_verify_kn
 *               with n_draft 2..8 launch as
 *               programmatic dependents of the previous kernel in the
 *               stream: their blocks may become resident while that kernel
 *               finishes. Before it has completed they read only the layer
 *               parameters (gdn_params: conv weights, dt, A_log, norm
 *               weight), which that kernel must therefore not write; every
 *               other argument (activations, state, conv history, snapshots,
 *               accepted counts) is read after it, in stream order. (A
 *               launch of at most one wave also asks for its state rows to
 *               be brought into L2 before then, which reads nothing.)
 *   Errors      Host-side validation runs before anything is launched. A
 *               call that returns anything but GDN_OK has enqueued nothing,
 *               except GDN_ERR_CUDA, where the launch itself failed;
 *               gdn_last_cuda_error() then names the CUDA error.
 *   Reentrancy  The library holds no mutable global state besides the
 *               last-error text (per host thread) and the device-side error
 *               bits (see gdn_check_device): calls from several host threads
 *               and streams are safe as long as their buffers do not overlap.
 *   Precision   Parameters, recurrent state, conv history and all outputs are
 *               float32 (gdn_decode_step_bf16_state excepted); activations are
 *               float32 or bf16 (gdn_dtype). All arithmetic is float32.
 *
 * SHAPES (gdn_dims)
 *   B   = n_seq, Hq = n_qk_heads, Hv = n_v_heads (a multiple of Hq; r = Hv/Hq),
 *   d   = head_dim = d_k = d_v (128 is supported), W = d_conv (2..8),
 *   conv_dim = (2 Hq + Hv) d.
 *   V head h reads QK head floor(h / r) (consecutive V heads share a QK head).
 *   Supported: d == 128, 2 <= W <= 8, 1 <= r <= 8, Hv*d*d*4 bytes per sequence.
 *
 * LAYOUTS (elements, row-major, innermost last)
 *   state      float [B][Hv][d][d]: state[b][h][j][i] = S_h[i][j] with i the
 *              key index and j the value index, so each value row j is
 *              contiguous over i (the transposed layout of "fm_kernel_ssm.h",
 *              section "Delta-rule recurrence").
 *   conv_state float [B][conv_dim][W-1], oldest tap first, holding RAW inputs
 *              ("fm_kernel_ssm.h", "Causal depthwise conv1d + SiLU").
 *   x          act   [B][T] rows of x_stride elements; the first conv_dim
 *              entries of a row are the token's [Q | K | V] projection
 *              ("ssm_mamba.rs", conv1d_update_l2norm_strided: input rows may
 *              be farther apart than conv_dim, e.g. a fused qkvz row).
 *   z          act   [B][T] rows of z_stride elements, first Hv*d used.
 *   alpha, beta_logit act [B][T] rows of gate_stride elements, first Hv used.
 *   out        float [B][T][Hv][d], dense.
 *   Token index t of sequence b is row (b*T + t) for every row-strided input.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as CUDA's cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, stride too small, misalignment */
    GDN_ERR_UNSUPPORTED = 2,  /* a valid shape this library has no kernel for (d != 128, W > 8, r > 8) */
    GDN_ERR_CUDA = 3,         /* the launch failed; see gdn_last_cuda_error() */
    GDN_ERR_DEVICE = 4        /* a kernel's bounded wait gave up (see gdn_check_device) */
} gdn_status;

typedef enum gdn_dtype {
    GDN_F32 = 0,
    GDN_BF16 = 1
} gdn_dtype;

typedef struct gdn_dims {
    int32_t n_seq;        /* B  >= 1 */
    int32_t n_qk_heads;   /* Hq >= 1 */
    int32_t n_v_heads;    /* Hv, a multiple of Hq */
    int32_t head_dim;     /* d (128) */
    int32_t d_conv;       /* W, 2..8 */
    int32_t reserved;     /* must be 0 */
    int64_t x_stride;     /* elements between token rows of x, >= conv_dim */
    int64_t z_stride;     /* elements between token rows of z, >= Hv*d */
    int64_t gate_stride;  /* elements between token rows of alpha / beta_logit, >= Hv */
} gdn_dims;

/* Per-layer parameters, all float32 device arrays. */
typedef struct gdn_params {
    const float *conv_w;  /* [conv_dim][W], tap W-1 multiplies the current token */
    const float *dt;      /* [Hv] decay-gate bias */
    const float *A_log;   /* [Hv]; the decay rate is a = -exp(A_log) */
    const float *norm_w;  /* [d] gated-RMSNorm gain, shared by every V head */
    float l2_eps;         /* added to sum(x^2) in the Q/K L2 norm (e.g. 1e-6) */
    float rms_eps;        /* added to mean(y^2) in the gated RMSNorm (e.g. 1e-6) */
} gdn_params;

/*
 * Decay gate. "fm_kernel_ssm.h", section "Decay gate"; the guarded softplus
 * as in "scr_state.hpp" log_gate:
 *   g[r][h] = -exp(A_log[h]) * softplus(alpha[r][h] + dt[h]),
 *   softplus(v) = v for v > 20, else log1p(exp(v)).
 * g is returned pre-exp (negative, so exp(g) is in (0, 1)).
 *   alpha  [rows] rows of alpha_stride elements (dtype alpha_dtype), first n_heads used
 *   dt, A_log [n_heads] float; g [rows][n_heads] float, dense.
 * Errors: GDN_ERR_INVALID_ARG for null pointers, rows or n_heads < 1,
 * alpha_stride < n_heads.
 */
gdn_status gdn_decay_gate(const void *alpha, gdn_dtype alpha_dtype, int64_t alpha_stride,
                          const float *dt, const float *A_log, float *g,
                          int32_t rows, int32_t n_heads, gdn_stream_t stream);

/*
 * Causal depthwise conv1d + SiLU over n_tokens tokens of every sequence, with
 * the per-head L2 norm of the Q and K channels fused in.
 * "fm_kernel_ssm.h", section "Causal depthwise conv1d + SiLU" (single step
 * and the n-token scan); "ssm_mamba.rs", conv1d_update_l2norm (L2 on the Q/K
 * channels after SiLU, V channels SiLU only) and its _strided form.
 * Per channel c and token t, with the window [hist[c][0..W-2], x[t][c]]:
 *   out[t][c] = silu(sum_tau window[tau] * conv_w[c][tau]); then the history
 *   drops its oldest entry and appends the RAW x[t][c]. For c in the Q or K
 *   part, each head's d outputs are divided by sqrt(sum out^2 + l2_eps).
 *   conv_state [B][conv_dim][W-1] updated in place (ends holding the last
 *              W-1 raw inputs); x as in LAYOUTS (dims->x_stride);
 *   out        float [B][n_tokens][conv_dim] dense: [Q^ | K^ | V].
 * dims->z_stride and gate_stride are not used. With n_tokens > 1 the tokens
 * are computed in parallel ("ssm_mamba.rs", token-parallel prefill conv1d:
 * the window slides over inputs, so no output depends on another), bit for
 * bit equal to n_tokens single-token calls. n_tokens <= 2,097,120.
 * Errors: INVALID_ARG (null, n_tokens < 1, bad dims), UNSUPPORTED (d, W),
 * CUDA (n_tokens above the limit).
 */
gdn_status gdn_conv_update(float *conv_state, const void *x, gdn_dtype x_dtype,
                           const float *conv_w, float *out, const gdn_dims *dims,
                           int32_t n_tokens, float l2_eps, gdn_stream_t stream);

/*
 * One decode step of the gated-delta recurrence, state updated in place.
 * "fm_kernel_ssm.h", section "Delta-rule recurrence". Per V head h (QK head
 * hk = h / r) and value row j, with decay = exp(g[b][h]):
 *   row_j <- decay * row_j;  pred = row_j . k_hk;  delta = beta (v_h[j] - pred);
 *   row_j <- row_j + delta k_hk;  y[b][h][j] = scale * (row_j . q_hk)   (updated row).
 * q and k must already be L2-normalised, beta already a sigmoid, g pre-exp.
 *   q, k  float, sequence b's head hk at q + b*qkv_stride + hk*d (same for k)
 *   v     float, sequence b's head h  at v + b*qkv_stride + h*d
 *   g, beta float [B][Hv]; y float [B][Hv][d].
 * With the dense output of gdn_conv_update: q = out, k = out + Hq*d,
 * v = out + 2*Hq*d, qkv_stride = conv_dim.
 * Errors: INVALID_ARG (null, bad dims, qkv_stride too small), UNSUPPORTED (d, r).
 */
gdn_status gdn_recurrence_decode(float *state, const float *q, const float *k,
                                 const float *v, int64_t qkv_stride,
                                 const float *g, const float *beta, float *y,
                                 const gdn_dims *dims, float scale, gdn_stream_t stream);

/*
 * Gated RMSNorm per V head. "fm_kernel_ssm.h", section "Gated RMSNorm":
 *   inv = 1 / sqrt(mean_j y[j]^2 + eps);  out[j] = ((y[j] * inv) * w[j]) * silu(z[j]).
 * w [head_dim] is shared by every head.
 *   y, out float [rows][n_v_heads][head_dim] (out may alias y);
 *   z      rows of z_stride elements (dtype z_dtype), first n_v_heads*head_dim used.
 * Errors: INVALID_ARG (null, sizes < 1, z_stride too small), UNSUPPORTED (head_dim != 128).
 */
gdn_status gdn_gated_norm(const float *y, const float *norm_w, const void *z,
                          gdn_dtype z_dtype, int64_t z_stride, float *out,
                          int32_t rows, int32_t n_v_heads, int32_t head_dim,
                          float eps, gdn_stream_t stream);

/*
 * The fused layer step for one token of every sequence, in ONE launch:
 * conv + SiLU + Q/K L2 norm, decay gate and beta = sigmoid(beta_logit), the
 * recurrence (scale = 1/sqrt(d)), and the gated RMSNorm. Each state element
 * is read once and written once. Same arithmetic as gdn_conv_update ->
 * gdn_decay_gate -> gdn_recurrence_decode -> gdn_gated_norm, bit for bit.
 * ("fm_kernel_ssm.h" sections "Decay gate" through "Delta-rule recurrence";
 * "ssm_mamba.rs" conv1d_update_l2norm_strided for the batched, strided form.)
 *   state, conv_state updated in place; x, z, alpha, beta_logit as in LAYOUTS
 *   with T = 1; out float [B][Hv][d].
 * Errors: INVALID_ARG, UNSUPPORTED as above.
 */
gdn_status gdn_decode_step(float *state, float *conv_state, const void *x, const void *z,
                           const void *alpha, const void *beta_logit, gdn_dtype act_dtype,
                           const gdn_params *params, float *out, const gdn_dims *dims,
                           gdn_stream_t stream);

/*
 * gdn_decode_step with the recurrent state and the output stored as bf16: a
 * serving option that halves the state traffic of a decode step. None of the
 * source pages defines such a variant (their state is float32); it is offered
 * outside the float32 tolerances. Each state row is widened exactly to float32, stepped
 * with the same float32 arithmetic as gdn_decode_step (the readout uses the
 * updated row before it is rounded), and rounded to nearest even when stored;
 * each output value is rounded to nearest even.
 *   state  bf16 [B][Hv][d][d] (same layout as the float32 state), in place
 *   out    bf16 [B][Hv][d]
 *   conv_state, x, z, alpha, beta_logit, params, dims as for gdn_decode_step
 *          (the conv history stays float32).
 * Errors: INVALID_ARG, UNSUPPORTED as for gdn_decode_step.
 */
gdn_status gdn_decode_step_bf16_state(void *state, float *conv_state, const void *x,
                                      const void *z, const void *alpha, const void *beta_logit,
                                      gdn_dtype act_dtype, const gdn_params *params, void *out,
                                      const gdn_dims *dims, gdn_stream_t stream);

/*
 * K=2 draft verification ("ssm_mamba.rs", gdn_verify_fused_conv_k2 and
 * gdn_verify_fused_norm_k2): both positions of every sequence in ONE launch.
 * Position 0 then position 1 are applied exactly as two gdn_decode_step calls
 * would apply them (bit for bit), while each state row is read once:
 *   state_snap, conv_snap  <- state and conv window after position 0
 *   state, conv_state      <- after position 1 (the committed result)
 *   out float [B][2][Hv][d] (both positions).
 * Inputs are [B][2] token rows (row b*2 + p). state_snap has the layout of
 * state, conv_snap that of conv_state; neither may overlap the others.
 * Errors: INVALID_ARG, UNSUPPORTED as above.
 */
gdn_status gdn_verify_k2(float *state, float *conv_state, float *state_snap, float *conv_snap,
                         const void *x, const void *z, const void *alpha,
                         const void *beta_logit, gdn_dtype act_dtype,
                         const gdn_params *params, float *out, const gdn_dims *dims,
                         gdn_stream_t stream);

/*
 * Commit or roll back after gdn_verify_k2 ("ssm_mamba.rs",
 * gdn_verify_fused_conv_k2: the position-0 snapshot is the rollback point).
 * Per sequence b with n_accept[b] (device int32 [B]):
 *   1 -> state[b] <- state_snap[b], conv_state[b] <- conv_snap[b]
 *        (bit-exact state after one decode step);
 *   2 -> nothing (state already holds both positions);
 *   otherwise sequence b is left unchanged and bit 16 is set in the
 *   device-side error word (see gdn_check_device).
 * Errors: INVALID_ARG (null, bad dims), UNSUPPORTED (d).
 */
gdn_status gdn_verify_commit(float *state, float *conv_state, const float *state_snap,
                             const float *conv_snap, const int32_t *n_accept,
                             const gdn_dims *dims, gdn_stream_t stream);

/*
 * The single-token step that follows a K-token verify (gdn_verify_k2, K = 2,
 * or gdn_verify_kn, K = n_draft) with the rollback folded in ("ssm_mamba.rs",
 * gdn_verify_fused_conv_k2: the position-0 snapshot is the rollback point,
 * and the generic form issues no copies). Sequence b starts from the state
 * after its n = n_accept[b] accepted tokens (device int32 [B]):
 *   n < K   state_snap entry n-1 (float [B][K-1][Hv][d][d]) and conv_snap
 *           entry n-1 (float [B][E][conv_dim][W-1], E = conv_snap_entries:
 *           K-1 for gdn_verify_k2's snapshots, K for gdn_verify_kn's);
 *   n = K   state and conv_state;
 *   otherwise state and conv_state, and bit 16 is set in the device-side
 *           error word (see gdn_check_device).
 * The step's results go to state, conv_state and out exactly as in
 * gdn_decode_step, so this call equals gdn_verify_commit (gdn_verify_commit_kn)
 * followed by gdn_decode_step, bit for bit, without the commit's copy. With
 * K = 1 the snapshots are not read (may be NULL). The snapshots are only read
 * and may not overlap state or conv_state.
 * Errors: INVALID_ARG (null, n_draft < 1, conv_snap_entries not K-1 or K,
 * overlapping snapshots, bad dims), UNSUPPORTED as gdn_decode_step.
 */
gdn_status gdn_decode_step_select(float *state, float *conv_state, const float *state_snap,
                                  const float *conv_snap, int32_t conv_snap_entries,
                                  const int32_t *n_accept, int32_t n_draft, const void *x,
                                  const void *z, const void *alpha, const void *beta_logit,
                                  gdn_dtype act_dtype, const gdn_params *params, float *out,
                                  const gdn_dims *dims, gdn_stream_t stream);

/*
 * Sequential scan of the recurrence over n_tokens tokens of every sequence
 * ("fm_kernel_ssm.h", "Delta-rule recurrence": the naive sequential scan,
 * kept as the permanent correctness reference for the chunked path). Each
 * state row stays in registers across the tokens and is written back once;
 * per token the arithmetic is gdn_recurrence_decode's, so the result equals
 * n_tokens gdn_recurrence_decode calls bit for bit.
 *   q, k, v  token t of sequence b is row b*n_tokens + t: its QK head hk at
 *            q + row*qkv_stride + hk*d (same for k), V head h at
 *            v + row*qkv_stride + h*d
 *   g, beta  float [B][n_tokens][Hv] (g pre-exp, beta already a sigmoid)
 *   y        float [B][n_tokens][Hv][d]
 * Errors: INVALID_ARG (null, n_tokens < 1, bad dims, qkv_stride too small),
 * UNSUPPORTED (d, r).
 */
gdn_status gdn_recurrence_scan(float *state, const float *q, const float *k, const float *v,
                               int64_t qkv_stride, const float *g, const float *beta, float *y,
                               const gdn_dims *dims, int32_t n_tokens, float scale,
                               gdn_stream_t stream);

/*
 * The fused layer step applied to n_tokens tokens of every sequence one token
 * at a time, in ONE launch, with the state rows held in registers throughout:
 * equal bit for bit to n_tokens gdn_decode_step calls. It is the on-device
 * sequential reference for gdn_prefill_chunked at lengths beyond a CPU
 * check ("fm_kernel_ssm.h", "Delta-rule recurrence").
 *   state, conv_state updated in place; x, z, alpha, beta_logit as in LAYOUTS
 *   with T = n_tokens; out float [B][n_tokens][Hv][d].
 * Errors: INVALID_ARG (null, n_tokens < 1, bad dims), UNSUPPORTED (d, W, r).
 */
gdn_status gdn_layer_scan(float *state, float *conv_state, const void *x, const void *z,
                          const void *alpha, const void *beta_logit, gdn_dtype act_dtype,
                          const gdn_params *params, float *out, const gdn_dims *dims,
                          int32_t n_tokens, gdn_stream_t stream);

/*
 * Draft verification of K = n_draft positions per sequence, every sequence in
 * ONE launch ("ssm_mamba.rs", gdn_verify_fused_conv_kn and
 * gdn_verify_fused_conv_kn_batched: all positions in one launch, every
 * per-position rollback snapshot written inline, the committed window
 * duplicated as the last snapshot so the caller issues no copies; here the
 * recurrent state is snapshotted as well). Positions are applied exactly as
 * K gdn_decode_step calls would apply them, bit for bit.
 *   state, conv_state <- after position K-1 (the committed result)
 *   state_snap float [B][K-1][Hv][d][d]: entry p = state after position p,
 *              p = 0..K-2 (the state after K-1 is `state` itself, so it is
 *              not duplicated: that would cost a full extra state write);
 *              may be NULL when K == 1
 *   conv_snap  float [B][K][conv_dim][W-1]: entry p = conv window after
 *              position p; entry K-1 duplicates the committed conv_state
 *   out float [B][K][Hv][d]; inputs are [B][K] token rows (row b*K + p).
 * The snapshot arrays may not overlap state, conv_state or each other.
 * For K = 2..8 the positions run in the fused step kernel (each state row
 * read once and held in registers across the positions); longer drafts run
 * in the layer scan of gdn_layer_scan. Both give the same bits.
 * Errors: INVALID_ARG (null, n_draft < 1, bad dims), UNSUPPORTED (d, W, r).
 */
gdn_status gdn_verify_kn(float *state, float *conv_state, float *state_snap, float *conv_snap,
                         const void *x, const void *z, const void *alpha,
                         const void *beta_logit, gdn_dtype act_dtype,
                         const gdn_params *params, float *out, const gdn_dims *dims,
                         int32_t n_draft, gdn_stream_t stream);

/*
 * Commit or roll back after gdn_verify_kn with the same n_draft = K. Per
 * sequence b with n = n_accept[b] (device int32 [B]), the number of
 * positions kept:
 *   n == K      nothing (state and conv_state already hold all K);
 *   1 <= n < K  state[b] <- state_snap[b][n-1], conv_state[b] <- conv_snap[b][n-1]
 *               (bit-exact state after n decode steps);
 *   otherwise   sequence b is left unchanged and bit 16 is set in the
 *               device-side error word (see gdn_check_device).
 * Errors: INVALID_ARG (null, n_draft < 1, bad dims), UNSUPPORTED (d).
 */
gdn_status gdn_verify_commit_kn(float *state, float *conv_state, const float *state_snap,
                                const float *conv_snap, const int32_t *n_accept,
                                const gdn_dims *dims, int32_t n_draft, gdn_stream_t stream);

/*
 * Workspace bytes gdn_prefill_chunked needs for these dims and n_tokens: per
 * (sequence, 64-token chunk) a 34 KB image per V head (the chunk's
 * (I + A)^-1, decayed Q K^T and gates) and a 64 KB image per QK head (its
 * normalised Q and K rows as tensor-core operands), i.e.
 * n_seq * ceil(n_tokens / 64) * (34816 * n_v_heads + 65536 * n_qk_heads).
 * Returns 0 for invalid dims, n_tokens < 1 or chunk != 64.
 */
size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t n_tokens, int32_t chunk);

/*
 * Chunked prefill over n_tokens tokens of every sequence: the same function
 * as n_tokens gdn_decode_step calls, evaluated chunk by chunk
 * ("fm_kernel_ssm.h", "Delta-rule recurrence": the sequential scan is the
 * reference the chunked path is validated against; "ssm_mamba.rs",
 * "Mamba-2 SSD chunked prefill scan": 64-token chunks joined by
 * ceil(T/64) sequential state links).
 *   state, conv_state updated in place (state after the last token);
 *   x, z, alpha, beta_logit as in LAYOUTS with T = n_tokens;
 *   out float [B][n_tokens][Hv][d].
 *   workspace  caller-owned device scratch of at least
 *              gdn_prefill_workspace_bytes(dims, n_tokens, chunk) bytes,
 *              16-byte aligned; its contents on entry do not matter and are
 *              meaningless on return. Calls that overlap on the GPU need
 *              separate workspaces.
 * Runs as three launches on `stream`: every chunk's state-independent
 * operands (its normalised Q and K rows, (I + A)^-1 transform, decayed Q K^T
 * and gates) in parallel into the workspace, the sequential pass over the
 * chunks of each (sequence, V head), and the conv-history update.
 * chunk must be 64. x, params->conv_w and out must be 16-byte aligned, with x
 * rows a multiple of 16 bytes apart (x_stride * element size). Agrees with the
 * sequential scan within float32 rounding, not bit for bit.
 * Errors: INVALID_ARG (null, n_tokens < 1, bad dims, alignment, workspace too
 * small), UNSUPPORTED (d, W, chunk != 64).
 */
gdn_status gdn_prefill_chunked(float *state, float *conv_state, const void *x, const void *z,
                               const void *alpha, const void *beta_logit, gdn_dtype act_dtype,
                               const gdn_params *params, float *out, const gdn_dims *dims,
                               int32_t n_tokens, int32_t chunk, void *workspace,
                               size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_prefill_chunked for callers that cannot allocate device memory, e.g. a
 * runtime that hands out every byte of device memory from a plan fixed at
 * start-up and exposes no allocator to the libraries it loads, or a loop with
 * latency bounds that an allocation (which may synchronise the device) would
 * break. None of the source pages has a counterpart: it is a packaging of
 * gdn_prefill_chunked, same arguments and results, without the workspace.
 *
 * The workspace is a fixed 16 MiB array inside the library (a static device
 * variable): every GPU on which the library is loaded holds it until the
 * process exits, and it serves calls whose gdn_prefill_workspace_bytes is at
 * most 16 MiB (e.g. one sequence of 2048 tokens with 2 QK and 4 V heads, or
 * 16 x 64 tokens with 4 QK and 8 V heads). Larger calls return
 * GDN_ERR_UNSUPPORTED (the reason is in gdn_last_cuda_error()) and launch
 * nothing. The library itself allocates nothing either.
 *
 * The first call on a device resolves the array's device address on the
 * current device; make that first call before any stream capture. Every call
 * on a device shares the one array and leaves its contents behind: nothing in
 * it needs to start at zero (each call writes every image it reads first), but
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race on it and must be ordered by the caller.
 * Errors: as gdn_prefill_chunked, plus GDN_ERR_UNSUPPORTED beyond the limit.
 */
gdn_status gdn_prefill_chunked_noalloc(float *state, float *conv_state, const void *x,
                                       const void *z, const void *alpha, const void *beta_logit,
                                       gdn_dtype act_dtype, const gdn_params *params, float *out,
                                       const gdn_dims *dims, int32_t n_tokens, int32_t chunk,
                                       gdn_stream_t stream);

/*
 * Every wait inside a kernel on a bulk copy, a tensor-core operation,
 * another warp group of the same CTA or data pushed by another CTA of the
 * same cluster is bounded by the GPU's global timer
 * (2 s); a kernel whose wait gives up sets a bit in a device-side error word,
 * stops its remaining work, waits (bounded again) for the copies and products
 * it already issued, frees its tensor memory and returns instead of hanging:
 *   bit 1   the chunked prefill's sequential pass gave up a wait
 *   bit 2   the chunked prefill's per-chunk transform pass gave up a wait
 *   bit 8   a copy or product the prefill issued did not finish in its drain
 *   bit 16  gdn_verify_commit saw an accepted count outside 1..2, or
 *           gdn_verify_commit_kn / gdn_decode_step_select one outside 1..K
 *   bit 32  (checked build only, libgdn_checked.so) a kernel's index
 *           arithmetic left the range its arguments allow
 *   bit 64  the multi-token conv gave up its tile-copy wait
 *   bit 128 a row slice of a fused decode / verify step gave up waiting for
 *           the gated-norm partial sums of the head's other row slices (that
 *           head's outputs are not valid)
 * The one wait not bounded by the library is the hardware's tensor-memory
 * allocation at the start of the prefill kernels, which lasts until CTAs of
 * other launches on the same SM release their columns. This call waits for
 * all work on the device (it synchronises), reads the word into *code (may be
 * NULL) and clears it. Returns GDN_OK when no bit was set, GDN_ERR_DEVICE when
 * one was, GDN_ERR_CUDA if the read failed.
 */
gdn_status gdn_check_device(int32_t *code);

/* Text of the last CUDA error seen by a call on this host thread ("" if none). */
const char *gdn_last_cuda_error(void);

/* Name of a status code. */
const char *gdn_status_string(gdn_status status);

/* Library version string. */
const char *gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
