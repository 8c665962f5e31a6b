/*
 * ttt.h — C ABI of the B300 chunked test-time-training (TTT) scan library.
 *
 * The TTT layer keeps, per (batch row, head), a state that is the weights of a
 * small model and, for each chunk of b tokens, takes one gradient step on the
 * key -> value reconstruction loss, with every gradient of the chunk taken at
 * the chunk-start weights; it reads out z_t = f(q_t; W_t) with the weights
 * after token t's own gradient.
 *   - "5 · TestingTime 训练与长上下文" (PaperTrace), section 1.1: the layer's
 *     three parts (initial state W0, update rule, output rule); chunks of
 *     b = 16 whose gradients are taken at the chunk-start weights; the dual
 *     form that turns the chunk's outer products into matrix products.
 *   - same page, section 2.3: f_W(k) = W k, loss 1/2 ||W k - v||^2,
 *     gradient (W k - v) k^T (the delta rule); section 2.1: read-out
 *     y_t = f(q_t; W_t); section 2.4: state reset per sequence.
 *   - "Test-Time Training (TTT) guide" (diosapp), section 3: TTT-Linear and
 *     TTT-MLP (two layers, hidden width 4x the input, GELU), mini-batch TTT
 *     and the dual form.
 *
 * Conventions for every call
 *   Row vectors: z = q W, W[i][j] with i the input and j the output index
 *   (the pages' W k is k W^T here). Dual form of one chunk c, Wa = state at
 *   its start:  E = K_c Wa - V_c;  Z_c = Q_c Wa - eta tril(Q_c K_c^T) E
 *   (diagonal included: update, then read);  W = Wa - eta K_c^T E.
 *   Gradients of a chunk are summed (an averaged step equals eta / b).
 *   A final chunk shorter than b follows the same rule.
 *
 *   Memory: every pointer is device memory owned by the caller, contiguous
 *   row-major, 16-byte aligned. The library allocates nothing; the caller
 *   passes a workspace of ttt_workspace_bytes() bytes.
 *
 *   Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream) and the call returns without waiting. Argument
 *   errors are returned before anything is enqueued. Errors a kernel detects
 *   (a wait that ran out of time) are written to a status word inside the
 *   workspace; ttt_last_device_status() reads it.
 *
 *   Inputs are never modified. Outputs (and the workspace) may overlap
 *   neither an input nor one another: a call whose buffers do returns
 *   TTT_ERR_ARG before anything is enqueued. Inputs may alias each other.
 */
#ifndef TTT_B300_H
#define TTT_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TTT_API __attribute__((visibility("default")))
#else
#define TTT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TTT_OK = 0,
  TTT_ERR_ARG = -1,          /* bad pointer, size, alignment or workspace */
  TTT_ERR_UNSUPPORTED = -2,  /* a valid request the library does not serve (e.g. d > 64) */
  TTT_ERR_CUDA = -3,         /* a CUDA runtime call failed (launch, copy, no device) */
  TTT_ERR_TIMEOUT = -4,      /* a kernel's bounded wait ran out (reported via the workspace) */
  TTT_ERR_DEVICE_CHECK = -5  /* a kernel's own consistency check failed */
} ttt_status;

typedef enum {
  TTT_F32 = 0,   /* Q, K, V, Z are float32 */
  TTT_BF16 = 1   /* Q, K, V, Z are bfloat16 (state and arithmetic stay fp32-accumulated) */
} ttt_dtype;

typedef enum { TTT_VARIANT_LINEAR = 0, TTT_VARIANT_MLP = 1 } ttt_variant;

/* Inner-model variants of TTT-Linear (the ttt_linear_*_fwd calls below). */
typedef enum {
  TTT_INNER_BIAS = 1,
  TTT_INNER_TOKEN_ETA = 2,
  TTT_INNER_LN = 3,
  TTT_INNER_MOMENTUM = 4
} ttt_inner_variant;

/* Options for the *_ex calls. Zero-initialise, then set fields. */
typedef struct {
  uint64_t wait_timeout_ns; /* limit for every wait inside a kernel; 0 = 2 s */
  int32_t inject_stall;     /* test hook: 1 = the load pipeline never fills, so the
                               consumers' bounded wait must run out (TTT_ERR_TIMEOUT);
                               2 = TTT-MLP on two CTAs per unit: the second CTA never
                               sends its G partials, so the first CTA's exchange wait
                               must run out (TTT_ERR_TIMEOUT) */
  int32_t force_path;       /* 0 = automatic; 1 = general fp32 SIMT kernel;
                               2 = tensor-core kernel, one pass per sequence;
                               3 = tensor-core kernels, segment-parallel form.
                               2 and 3 return TTT_ERR_UNSUPPORTED where they cannot
                               serve (they need bf16, d = 64, b % 16 == 0). */
  int32_t seg_len;          /* segment-parallel form only: tokens per segment, a
                               multiple of b and of 16; 0 = chosen automatically */
  void* phase_events;       /* optional instrumentation, NULL = none: an array of 4
                               cudaEvent_t (created by the caller) that TTT-Linear
                               records on `stream` before its first kernel, after the
                               affine-map kernel, after the combine kernel and after
                               the read-out kernel. On the one-pass path the first
                               three are recorded back to back. Given events, the
                               segment-parallel form runs in one piece (no overlap). */
  int32_t pieces;           /* segment-parallel form only: 0 = automatic; 1 = the
                               three kernels one after another over all segments;
                               n > 1 = the segments are cut into n pieces and the
                               affine maps of piece p + 1 run beside the read-out of
                               piece p (a second stream inside the call) */
} ttt_options;

/* How a TTT-Linear call with these arguments runs (filled by ttt_linear_plan). */
typedef struct {
  int32_t path;       /* 1 = fp32 SIMT kernel, 2 = tensor-core one pass, 3 = segment-parallel */
  int32_t seg_len;    /* tokens per segment (the whole sequence on paths 1 and 2) */
  int32_t seg_count;  /* segments per (batch row, head) */
  int32_t kernels;    /* kernels one call enqueues (besides a 16-byte status reset) */
  int32_t affine;     /* path 3: 1 = affine maps by warp-level MMAs (16-token tiles),
                         2 = by tcgen05 tensor cores (64-token steps); else 0 */
  int32_t pieces;     /* path 3: pieces the segments are cut into (1 = no overlap); else 1 */
} ttt_plan;

/* Bytes of workspace a call with these sizes needs on the current device
 * (>= 256; a status word lives at its start). variant: TTT_VARIANT_LINEAR or
 * TTT_VARIANT_MLP. TTT-Linear with bf16 operands may run in the
 * segment-parallel form, whose per-segment affine maps and start states live
 * in the workspace (3 d^2 floats per segment boundary); the size covers that
 * whatever the dtype. Returns 0 for invalid sizes. */
TTT_API size_t ttt_workspace_bytes(int B, int H, int T, int d, int b, int variant);

/* As ttt_workspace_bytes, for a call made with these options (a forced path
 * or segment length may need more, or less). opt may be NULL. */
TTT_API size_t ttt_workspace_bytes_ex(int B, int H, int T, int d, int b, int variant,
                                      const ttt_options* opt);

/*
 * TTT-Linear forward over whole sequences.
 *
 * How it runs. With bf16 operands, d = 64 and b % 16 == 0 the tensor-core
 * kernels serve the call. When there are too few (batch row, head) units to
 * fill the GPU, the sequence is cut into segments of whole chunks and run in
 * the segment-parallel form: one chunk's step W <- W - eta K_c^T (K_c W - V_c)
 * is the affine map W <- A_c W + B_c (A_c = I - eta K_c^T K_c,
 * B_c = eta K_c^T V_c), so each segment's composed map is computed on its own,
 * the maps are chained from W0 to give every segment's start state, and the
 * segments are then read out side by side. Exact algebra on the chunk update
 * ("5 · TestingTime 训练与长上下文", section 4); results agree with the one-pass
 * form within bf16 rounding. Three kernels are enqueued, three per piece
 * when the segments are cut into pieces whose affine maps overlap the
 * previous piece's read-out (ttt_options.pieces; work on a second stream
 * that the call joins back into `stream`); otherwise one.
 *   Q, K, V  [B][H][T][d], dtype dt.  eta [H] float32 (per-head inner learning rate).
 *   W0       [H][d][d] float32: initial state per head, shared by the batch
 *            (an outer-loop parameter); every batch row restarts from it.
 *   Z        [B][H][T][d], dtype dt: z_t = q_t W_t.
 *   W_out    [B][H][d][d] float32: state after the last token (resume point
 *            when T % b == 0).
 *   Sizes: B >= 1, H >= 1, T >= 0, 1 <= d <= 64, b >= 1.
 * Returns TTT_ERR_ARG for null/misaligned pointers, bad sizes or a short
 * workspace; TTT_ERR_CUDA if a launch fails.
 */
TTT_API ttt_status ttt_linear_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                          const float* eta, const float* W0, int B, int H, int T, int d, int b,
                          void* Z, float* W_out, void* workspace, size_t ws_bytes, void* stream);

/* The plan ttt_linear_fwd(_ex) follows for these arguments on the current
 * device; nothing is enqueued. Same argument errors as the forward call. */
TTT_API ttt_status ttt_linear_plan(int B, int H, int T, int d, int b, ttt_dtype dt, const ttt_options* opt,
                                   ttt_plan* out);

TTT_API ttt_status ttt_linear_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                             const float* eta, const float* W0, int B, int H, int T, int d, int b,
                             void* Z, float* W_out, void* workspace, size_t ws_bytes, void* stream,
                             const ttt_options* opt);

/*
 * TTT-MLP forward: f(x) = gelu(x W1) W2 with tanh-GELU (Hendrycks and Gimpel
 * 2016), hidden width m = 4 d ("Test-Time Training (TTT) guide", section 3).
 * With bf16 operands, d = 64 and b % 16 == 0 a tensor-core kernel serves the
 * call: for b = 16 a cluster of two CTAs per (batch row, head), each holding half
 * of the hidden units and exchanging its partial sums of G and Z with the other
 * through distributed shared memory; otherwise one CTA per (batch row, head).
 * ttt_options.force_path: 1 forces the fp32 SIMT kernel, 2 the one-CTA tensor
 * kernel, 3 the two-CTA kernel (b = 16 only; TTT_ERR_UNSUPPORTED elsewhere).
 *   W1_0 [H][d][4d], W2_0 [H][4d][d] float32, shared by the batch.
 *   W1_out [B][H][d][4d], W2_out [B][H][4d][d] float32.
 *   Other arguments as ttt_linear_fwd.
 */
TTT_API ttt_status ttt_mlp_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                       const float* eta, const float* W1_0, const float* W2_0, int B, int H, int T,
                       int d, int b, void* Z, float* W1_out, float* W2_out, void* workspace,
                       size_t ws_bytes, void* stream);

TTT_API ttt_status ttt_mlp_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                          const float* eta, const float* W1_0, const float* W2_0, int B, int H,
                          int T, int d, int b, void* Z, float* W1_out, float* W2_out,
                          void* workspace, size_t ws_bytes, void* stream, const ttt_options* opt);

/*
 * TTT-MLP forward that allocates nothing and takes no workspace. (No
 * counterpart on the pages: it exists for callers that cannot allocate
 * device memory, for example code inside a region that must not synchronise
 * the device, under a memory pool that hands out only the tensors it
 * manages, or a plain C host that owns just its inputs and outputs.) The
 * workspace ttt_mlp_fwd needs comes from a fixed array inside the library
 * instead: a status word, and 8 MiB for the per-unit chunk-start copies of
 * W1, W2 that only the fp32 SIMT kernel keeps in memory.
 *   - Limit: the tensor-core kernel (bf16, d = 64, b % 16 == 0) keeps those
 *     copies on chip and takes any number of units; when the SIMT kernel
 *     serves the call, at d = 64 at most 64 (batch row, head) units fit.
 *     Larger requests return TTT_ERR_UNSUPPORTED before anything is enqueued.
 *   - Every GPU that loads the library holds that array until the process exits.
 *   - All calls on a device share it: calls whose kernels overlap on the GPU
 *     race and give wrong results, so order them (one stream, or events).
 *   - The first call on a device looks up the array's address with that
 *     device current; make that first call before any stream capture.
 *   - A wait that runs out inside the kernel is recorded in the array's own
 *     status word: read it with ttt_mlp_noalloc_last_device_status().
 * Arguments and results as ttt_mlp_fwd; TTT_ERR_CUDA if the lookup fails.
 */
TTT_API ttt_status ttt_mlp_fwd_noalloc(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                       const float* eta, const float* W1_0, const float* W2_0, int B,
                                       int H, int T, int d, int b, void* Z, float* W1_out,
                                       float* W2_out, void* stream);

/* Waits for `stream`, then reads and clears the status word of the fixed array
 * that ttt_mlp_fwd_noalloc uses on the current device: TTT_OK, or the first
 * error a kernel of the latest such call recorded (TTT_ERR_TIMEOUT). (No
 * counterpart on the pages.) Allocates nothing. */
TTT_API ttt_status ttt_mlp_noalloc_last_device_status(void* stream);

/*
 * One TTT-Linear decode token per (batch row, head), in O(d^2) per head.
 *   q, k, v, z [B][H][d], dtype dt.  eta [H].
 *   W_anchor [B][H][d][d] float32 in/out: state at the start of the current chunk.
 *   W_run    [B][H][d][d] float32 in/out: state after the tokens seen so far.
 *   pos = tokens already seen; this token is number pos.
 *   e = k W_anchor - v;  W_run -= eta k^T e;  z = q W_run;
 *   if (pos + 1) % b == 0 then W_anchor = W_run (the chunk is complete).
 * After ttt_linear_fwd over T tokens with T % b == 0, W_anchor = W_run =
 * W_out and pos = T continue the sequence exactly.
 */
TTT_API ttt_status ttt_linear_decode_step(const void* q, const void* k, const void* v, ttt_dtype dt,
                                  const float* eta, float* W_anchor, float* W_run, int B, int H,
                                  int d, int pos, int b, void* z, void* stream);

/* N decode tokens per (batch row, head) in one launch: tokens pos .. pos + N - 1,
 * each exactly as ttt_linear_decode_step (the chunk-start anchor moves whenever
 * a token completes a chunk). q, k, v, z [B][H][N][d], dtype dt; W_anchor, W_run
 * as above (in/out). N = 0 enqueues nothing. Calling it equals N calls of
 * ttt_linear_decode_step with positions pos, pos + 1, ..., and amortises the
 * launch over the N tokens. */
TTT_API ttt_status ttt_linear_decode(const void* q, const void* k, const void* v, ttt_dtype dt,
                                     const float* eta, float* W_anchor, float* W_run, int B, int H,
                                     int N, int d, int pos, int b, void* z, void* stream);

/*
 * Inner-model variants of TTT-Linear. The pages name these ingredients without
 * formulas; each call states the reading it computes. The four plain calls run
 * one fp32 CUDA kernel per call (linear_variants.cu): one CTA per (batch row, head),
 * the state in shared memory, any d <= 64 and any b, Q/K/V/Z fp32 or bf16
 * (dt). They take no workspace (the kernel has no waits and no status word).
 * Q, K, V, Z, eta, W0, W_out and the per-call arrays follow ttt_linear_fwd's
 * conventions; per-head vectors are [H][d] float32, shared by the batch rows.
 * Errors: TTT_ERR_ARG for null/misaligned pointers, bad sizes or outputs that
 * overlap an input or each other; TTT_ERR_UNSUPPORTED for d > 64;
 * TTT_ERR_CUDA if the launch fails.
 *
 * ttt_linear_bias_fwd: f(k) = k W + beta ("Test-Time Training (TTT) guide",
 * section 3, writes f(W, x) = W x + b). (W, beta) are trained together by the
 * chunk rule on 1/2 ||k W + beta - v||^2: e = k W_a + beta_a - v at the
 * chunk-start weights, W -= eta k^T e, beta -= eta e; read-out
 * z_t = q_t W_t + beta_t. beta0 [H][d] in, beta_out [B][H][d] out.
 */
TTT_API ttt_status ttt_linear_bias_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                       const float* eta, const float* W0, const float* beta0, int B,
                                       int H, int T, int d, int b, void* Z, float* W_out,
                                       float* beta_out, void* stream);

/* ttt_linear_token_eta_fwd: a learning rate per token ("5 · TestingTime
 * 训练与长上下文", section 3.1, lists a learnable learning rate). eta_tok
 * [B][H][T] float32 >= 0 scales token t's gradient in the chunk rule:
 * W -= eta_t k_t^T (k_t W_a - v_t); read-out z_t = q_t W_t. */
TTT_API ttt_status ttt_linear_token_eta_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                            const float* eta_tok, const float* W0, int B, int H, int T,
                                            int d, int b, void* Z, float* W_out, void* stream);

/*
 * The bias and the per-token rate on the tensor-core kernels. Both variants are
 * the plain chunk rule on changed inputs, padded to 64 features:
 *   bias (d <= 63): q' = [q | 1 | 0], k' = [k | 1 | 0], v' = [v | 0] and
 *     W0' = [[W0, 0]; [beta0, 0]; [0, 0]]; the state's row d is beta, its
 *     padded columns stay 0, and z' = [q W + beta | 0];
 *   per-token rate (d <= 64): k' = sqrt(eta_t) k, v' = sqrt(eta_t) v, eta = 1;
 *     q is unchanged (zero-padded when d < 64).
 * The *_ex calls take a workspace of ttt_linear_variant_workspace_bytes(variant,
 * dt, B, H, T, d, b) bytes (16-byte aligned, disjoint from every input and
 * output): a status word, the changed inputs and the inner ttt_linear_fwd's own
 * workspace. With bf16 operands and b % 16 == 0 they write the changed inputs
 * (one elementwise kernel), run ttt_linear_fwd's kernels on them (one pass or
 * segment-parallel, by its automatic plan) and copy Z, W_out and beta_out out
 * of the padded results; otherwise (fp32, b % 16 != 0, d too large for the
 * padding) they run the fp32 variant kernel like the plain calls, and the
 * workspace holds only the status word. Results equal the plain calls' up to
 * rounding: k' and v' are rounded to bf16 again after the scaling.
 * ttt_last_device_status(workspace, stream) reports the inner forward's bounded
 * waits and, for the per-token rate, TTT_ERR_DEVICE_CHECK when some eta_t < 0
 * (that unit's results are then undefined).
 * ttt_linear_variant_workspace_bytes returns 0 for bad sizes or an unknown
 * variant; for TTT_INNER_LN and TTT_INNER_MOMENTUM it is the status word alone.
 */
TTT_API size_t ttt_linear_variant_workspace_bytes(int variant, ttt_dtype dt, int B, int H, int T, int d, int b);

TTT_API ttt_status ttt_linear_bias_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                          const float* eta, const float* W0, const float* beta0, int B,
                                          int H, int T, int d, int b, void* Z, float* W_out, float* beta_out,
                                          void* workspace, size_t ws_bytes, void* stream);

TTT_API ttt_status ttt_linear_token_eta_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                               const float* eta_tok, const float* W0, int B, int H, int T,
                                               int d, int b, void* Z, float* W_out, void* workspace,
                                               size_t ws_bytes, void* stream);

/* ttt_linear_ln_fwd: a layer norm and a residual inside f (same page, section
 * 3.1): f(k) = k + LN(k W), LN(y) = gamma (y - mean y) / sqrt(var y + 1e-6)
 * + beta over the d features of a token (biased variance), gamma, beta [H][d].
 * Trained by the chunk rule on 1/2 ||f(k) - v||^2 (gradient through LN at the
 * chunk-start W); read-out z_t = q_t + LN(q_t W_t). */
TTT_API ttt_status ttt_linear_ln_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                     const float* eta, const float* W0, const float* gamma,
                                     const float* beta, int B, int H, int T, int d, int b, void* Z,
                                     float* W_out, void* stream);

/* ttt_linear_ln_fwd_ex: the same layer; with bf16 operands, d = 64 and b a
 * multiple of 16 it runs on the tensor cores (one CTA per (batch row, head), W resident as fp32
 * accumulator fragments, bf16 operands of every product; each token's layer-norm
 * statistics summed over the 64 features across the CTA's warps), in the chunk's
 * form: Y = K W_a, x = (Y - mean) / s, g = gamma (K + gamma x + beta - V),
 * E = (g - mean(g) - x mean(g x)) / s, X = Q W_a - eta tril(Q K^T) E,
 * Z = Q + LN(X), W = W_a - eta K^T E. Otherwise it runs the fp32 variant kernel
 * like the plain call. workspace: ttt_linear_variant_workspace_bytes(
 * TTT_INNER_LN, ...) bytes (the status word; 16-byte aligned, disjoint from every
 * input and output); ttt_last_device_status reports the tensor kernel's bounded
 * waits. opt may be NULL; its fields as for ttt_linear_momentum_fwd_ex. */
TTT_API ttt_status ttt_linear_ln_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                        const float* eta, const float* W0, const float* gamma,
                                        const float* beta, int B, int H, int T, int d, int b, void* Z,
                                        float* W_out, void* workspace, size_t ws_bytes, void* stream,
                                        const ttt_options* opt);

/* ttt_linear_momentum_fwd: momentum gradient descent with chunk-start
 * gradients ("推理时的“临阵磨枪”：Test-Time Training如何教会AI“边做边学”",
 * sections 2.3 and 5.1, keep a momentum state beside W; the page leaves its
 * update function undefined). Per token t of a chunk with start state W_a:
 * g_t = k_t^T (k_t W_a - v_t), M = beta M + (1 - beta) g_t, W -= alpha M,
 * z_t = q_t W. M starts at zero for every sequence and carries across chunks.
 * alpha, beta [H]; M_out [B][H][d][d] the final momentum. */
TTT_API ttt_status ttt_linear_momentum_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                           const float* alpha, const float* beta, const float* W0, int B,
                                           int H, int T, int d, int b, void* Z, float* W_out, float* M_out,
                                           void* stream);

/* ttt_linear_momentum_fwd_ex: the same layer; with bf16 operands, d = 64 and
 * b a multiple of 16 it runs on the tensor cores (one CTA per (batch row, head),
 * W and M resident as fp32 accumulator fragments; bf16 operands of every
 * product; a chunk walked in 16-token tiles, each tile's E from the chunk-start
 * W), in the closed form of a run of tokens: E = K W_a - V,
 *   Z = Q W_a - alpha c .* (Q M_a) - alpha (tril(Q K^T) .* D) E,
 *   c_s = beta + ... + beta^s,  D[s][i] = 1 - beta^(s-i+1),
 * and at the chunk end (n tokens) W = W_a - alpha (c_n M_a + K^T (d .* E)),
 * M = beta^n M_a + (1 - beta) K^T (w .* E), d_i = 1 - beta^(n-i+1),
 * w_i = beta^(n-i). Otherwise it runs the fp32 variant kernel like the plain
 * call. workspace: ttt_linear_variant_workspace_bytes(TTT_INNER_MOMENTUM, ...)
 * bytes (the status word; 16-byte aligned, disjoint from every input and
 * output); ttt_last_device_status(workspace, stream) reports the tensor
 * kernel's bounded waits. opt may be NULL: wait_timeout_ns and inject_stall
 * as for ttt_linear_fwd_ex; force_path 1 = the fp32 kernel, 2 = the tensor
 * kernel (TTT_ERR_UNSUPPORTED where it cannot serve, and for T = 0), 3 =
 * TTT_ERR_UNSUPPORTED (no segment-parallel form). */
TTT_API ttt_status ttt_linear_momentum_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                              const float* alpha, const float* beta, const float* W0, int B,
                                              int H, int T, int d, int b, void* Z, float* W_out, float* M_out,
                                              void* workspace, size_t ws_bytes, void* stream,
                                              const ttt_options* opt);

/*
 * Backward of ttt_linear_fwd: the vector-Jacobian product of (Z, W_out) with
 * respect to (Q, K, V, eta, W0), for training the outer loop ("5 · TestingTime
 * 训练与长上下文", section 2.2: W0 and the projections that make Q, K, V are
 * outer-loop parameters). Per chunk c with start state W:
 *   E = K_c W - V_c,  S = tril(Q_c K_c^T),  Z_c = Q_c W - eta S E,  W' = W - eta K_c^T E,
 * reversed from G = dW_out (G: gradient of the next chunk's start state).
 *   Q, K, V, dZ [B][H][T][d] of dtype dt; eta [H]; W0 [H][d][d];
 *   dW_out [B][H][d][d]. Outputs dQ, dK, dV [B][H][T][d] of dtype dt, deta [H] and
 *   dW0 [H][d][d] float32 (summed over the batch rows, which share eta and W0).
 *   Kernels: bf16 with d = 64 and b = 16 runs on the tensor cores (state and
 *   products fp32-accumulated, W checkpointed every 64 tokens in the workspace);
 *   when B * H leaves SMs idle the sequence is cut into segments of whole
 *   64-token blocks, one CTA each, whose start states come from the forward's
 *   segment maps and whose end gradients come from the affine form of the
 *   read-out (G_start = A_s^T G_end + sum over the segment of Zhat^T dZ);
 *   every other case with d <= 64 runs the fp32 SIMT kernel (fp32 or bf16
 *   operands; chunks longer than 64 tokens are walked in 32-token blocks, with
 *   the chunk's E and dE kept in the workspace); d > 64 returns
 *   TTT_ERR_UNSUPPORTED.
 *   workspace: ttt_linear_bwd_workspace_bytes(B, H, T, d, b) bytes (a status
 *   word, the kept states, per-unit partial sums and, for b > 64, one chunk's
 *   E and dE per unit), 16-byte aligned. A wait in the
 *   tensor-core kernel that runs out records TTT_ERR_TIMEOUT there
 *   (ttt_last_device_status).
 * All pointers are device memory, 16-byte aligned, caller-owned; work is
 * enqueued on `stream`. Argument errors return before anything is enqueued.
 */
TTT_API size_t ttt_linear_bwd_workspace_bytes(int B, int H, int T, int d, int b);

TTT_API ttt_status ttt_linear_bwd(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                  const float* eta, const float* W0, int B, int H, int T, int d, int b,
                                  const void* dZ, const float* dW_out, void* dQ, void* dK, void* dV,
                                  float* deta, float* dW0, void* workspace, size_t ws_bytes,
                                  void* stream);

/*
 * Backward of ttt_mlp_fwd: the vector-Jacobian product of (Z, W1_out, W2_out)
 * with respect to (Q, K, V, eta, W1_0, W2_0), for training the outer loop
 * ("5 · TestingTime 训练与长上下文", section 2.2). Per chunk with start weights
 * P1 [d][m], P2 [m][d] (m = 4d) the forward is
 *   U = K P1, A = s(U), G = A P2 - V, D = (G P2^T) .* s'(U),
 *   Z = s(Q P1 - eta tril(Q K^T) D) P2 - eta tril(Aq A^T) G,
 *   P1' = P1 - eta K^T D,  P2' = P2 - eta A^T G   (s: tanh-GELU),
 * reversed chunk by chunk from dW1_out, dW2_out (s'' enters through D).
 *   Q, K, V, dZ [B][H][T][d] of dtype dt; eta [H]; W1_0 [H][d][m]; W2_0
 *   [H][m][d]; dW1_out [B][H][d][m]; dW2_out [B][H][m][d]. Outputs dQ, dK, dV
 *   [B][H][T][d] of dtype dt; deta [H], dW1 [H][d][m], dW2 [H][m][d] float32,
 *   summed over the batch rows (which share eta and the initial weights).
 *   d <= 64, any b (a final partial chunk included). One fp32 CUDA kernel, one
 *   CTA per (batch row, head), plus a reduction over the batch rows: a parity
 *   form, whose workspace keeps every chunk-start (W1, W2) and one chunk's
 *   matrices per unit.
 *   workspace: ttt_mlp_bwd_workspace_bytes(B, H, T, d, b) bytes, 16-byte aligned.
 *   Errors: TTT_ERR_ARG for null/misaligned pointers, bad sizes, a short
 *   workspace or outputs that overlap an input or each other;
 *   TTT_ERR_UNSUPPORTED for d > 64.
 */
TTT_API size_t ttt_mlp_bwd_workspace_bytes(int B, int H, int T, int d, int b);

TTT_API ttt_status ttt_mlp_bwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                               const float* W1_0, const float* W2_0, int B, int H, int T, int d, int b,
                               const void* dZ, const float* dW1_out, const float* dW2_out, void* dQ, void* dK,
                               void* dV, float* deta, float* dW1, float* dW2, void* workspace,
                               size_t ws_bytes, void* stream);

/* Waits for `stream`, then reads and clears the status word of `workspace`.
 * Every call that takes a workspace (the *_fwd calls and ttt_linear_bwd)
 * clears that word when it is enqueued, so this reports the kernels of the
 * latest such call that used this workspace: TTT_OK, or the first error one
 * of them recorded (TTT_ERR_TIMEOUT, TTT_ERR_DEVICE_CHECK). */
TTT_API ttt_status ttt_last_device_status(void* workspace, void* stream);

/* Static description of a status code. */
TTT_API const char* ttt_status_str(ttt_status s);

#ifdef __cplusplus
}
#endif

#endif /* TTT_B300_H */
