/*
 * spec_markov.h -- C ABI of libspecmarkov.so, the token-level hot path of speculative decoding
 * on GB300 (sm_103a): draft proposal over the vocabulary, target verification, TV confidence
 * with prefix survival, and the hardware-aware prefix scheduler.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every array argument is a DEVICE pointer owned by the caller; the library never allocates
 *    device or host memory and never keeps a pointer after the call returns. Scalars are passed
 *    by value; the few host outputs are named *_host below.
 *  - Layouts are dense row-major (C-contiguous) with the shapes given per argument.
 *    R = requests, gamma = proposed positions per request, V = vocabulary, rank = Markov rank.
 *  - Logits and Markov weights are SPEC_F32 or SPEC_BF16. W1 is the Markov embedding [V, rank]
 *    (row x is the low-rank code of previous token x); W2 is the Markov projection stored
 *    [V, rank] (row v holds the rank weights that project onto token v, the weight layout of a
 *    bias-free linear layer rank -> V).
 *  - Temperature: one T scales draft and target logits alike, after the Markov bias is added;
 *    the kernels multiply by the fp32 number 1.0f/T.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising. No call does host I/O on the data.
 *  - Scratch lives in the caller's workspace `ws` of `ws_bytes` bytes (device memory, 256-byte
 *    aligned), sized by spec_workspace_bytes(). Initialise a workspace once with
 *    spec_workspace_init() before its first use. Calls that share a workspace must not run
 *    concurrently on different streams.
 *  - Every entry point returns a spec_status. Arguments are validated on the host before any
 *    launch; a failed validation launches nothing. SPEC_ERR_CUDA reports a launch error.
 *  - Faults found on the device (a token id outside [0, V), a non-finite normaliser, a rejection
 *    whose residual mass is zero) never trap: the kernels set bits in a status word inside the
 *    workspace, read with spec_device_status(). Outputs of an affected request are still
 *    written with valid token ids.
 *
 * Indexing (anchor-first window): x_0 is the anchor (the previous round's bonus token). Draft
 * position k in [1, gamma] reads base-logit row U[r, k-1, :] and the Markov bias
 * W1[x_{k-1}] . W2. Target row i in [0, gamma] scores the token that follows window position i,
 * so x_k is checked against target row k-1 and row l is the bonus row when l tokens survive.
 */
#ifndef SPEC_MARKOV_H
#define SPEC_MARKOV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_ABI_VERSION 1

/* status codes */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG (-1)        /* null pointer, bad size, bad length, misalignment */
#define SPEC_ERR_UNSUPPORTED_DTYPE (-2)  /* dtype code outside {SPEC_F32, SPEC_BF16} */
#define SPEC_ERR_WORKSPACE_TOO_SMALL (-3)
#define SPEC_ERR_CUDA (-4)               /* a CUDA runtime call or launch failed */
#define SPEC_ERR_UNSUPPORTED (-6)        /* a combination the library does not implement */
#define SPEC_ERR_TOO_LARGE (-7)          /* sizes beyond a fixed limit (SPEC_NOALLOC_MAX_ROWS) */

/* dtype codes */
#define SPEC_F32 0
#define SPEC_BF16 1

/* op codes for spec_workspace_bytes */
#define SPEC_OP_PROPOSE 0
#define SPEC_OP_VERIFY_GREEDY 1
#define SPEC_OP_VERIFY_REJECTION 2
#define SPEC_OP_TV_CONFIDENCE 3
#define SPEC_OP_SCHEDULE 4
#define SPEC_OP_TARGET_STATS 5
#define SPEC_OP_MTP_GREEDY 6
#define SPEC_OP_ALL 7 /* a workspace large enough for every op at this size */

/* device status bits (spec_device_status) */
#define SPEC_DEV_BAD_TOKEN 0x1u      /* an anchor or draft token outside [0, V) was read */
#define SPEC_DEV_NONFINITE 0x2u      /* a row's softmax normaliser was NaN or infinite */
#define SPEC_DEV_EMPTY_RESIDUAL 0x4u /* a rejection met zero residual mass (p_t == p_d) */
#define SPEC_DEV_BAD_LENGTH 0x8u     /* a per-request length outside [0, gamma] */
#define SPEC_DEV_TIMEOUT 0x10u       /* a kernel's bounded wait expired; its outputs are invalid */

/* Largest R * gamma the prefix scheduler accepts (its sort runs in one CTA's shared memory). */
#define SPEC_SCHEDULE_MAX_CANDIDATES 16384

/*
 * Workspace size in bytes for `op` at this problem size (SPEC_OP_ALL covers every op). The
 * workspace is device memory owned by the caller, at least 256-byte aligned.
 */
size_t spec_workspace_bytes(int op, int R, int gamma, int V, int rank);

/* Zero the workspace header (the device status word) on `stream`. Call once per workspace. */
int spec_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Copy the device status word of `ws` into *status_host (synchronises `stream`); if `clear`
 * is non-zero the word is then reset to 0. Bits are the SPEC_DEV_* values.
 */
int spec_device_status(void* ws, size_t ws_bytes, void* stream, uint32_t* status_host,
                       int clear);

/* Static description of a status code. */
const char* spec_status_string(int status);

/* SPEC_ABI_VERSION of the loaded library. */
int spec_abi_version(void);

/*
 * Draft proposal over the vocabulary.
 * Defines: "[DeepSeek-6] DSpark", section 3 (semi-autoregressive head: per position,
 *   p_k(v) = softmax_v(U_k(v) + B_k(v)), sampled left to right) and section 4 "Markov Head"
 *   (B(x_{k-1}, .) = W1[x_{k-1}] W2, rank 256); with rank == 0 it is the MTP/NextN greedy
 *   proposal of "Module deepseek_v4_mtp", Forward (draft = argmax(logits)).
 * For k = 1..gamma (serially): s_k = U[r,k-1,:] + W1[x_{k-1}] . W2^T (x_0 = anchors[r]);
 *   greedy (u_draft == NULL or temperature == 0): x_k = argmax_v s_k(v), ties to the lowest id;
 *   sampling: x_k = the smallest v whose cumulative softmax(s_k / T) mass exceeds
 *   u_draft[r,k-1] (inverse CDF in ascending token order).
 * Arguments:
 *   U            [R, gamma, V] draft base logits, dtype u_dtype.
 *   W1, W2       [V, rank] each, dtype w_dtype (ignored when rank == 0).
 *   rank         0 (no Markov head) or the Markov rank (1..1024).
 *   anchors      [R] int32 x_0 (may be NULL when rank == 0).
 *   u_draft      [R, gamma] fp32 uniforms in [0, 1), or NULL for greedy.
 *   temperature  > 0 for sampling, 0 for greedy.
 *   draft_tokens [R, gamma] int32 output.
 *   draft_logp   [R, gamma] fp32 output log p_d(x_k) (optional, NULL to skip).
 *   draft_stats  [R, gamma, 2] fp32 output (m, log Z) of softmax(s_k / T), with
 *                p_d(v) = exp(s_k(v)/T - m - log Z); T = 1 when greedy (optional).
 * fp32 weights use the canonical fp32 chain acc = fmaf(W1[x][i], W2[v][i], acc), i ascending,
 * then s = U + acc in fp32, so greedy ids are reproducible bit for bit. bf16 weights with bf16
 * logits, V % 8 == 0 and rank a multiple of 64 up to 256 run on the tcgen05 tensor cores.
 */
int spec_markov_propose(const void* U, int u_dtype, const void* W1, const void* W2, int w_dtype,
                        int rank, const int32_t* anchors, const float* u_draft,
                        float temperature, int R, int gamma, int V, int32_t* draft_tokens,
                        float* draft_logp, float* draft_stats, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * Draft proposal and the target normalisers of the same window in one call.
 * Defines: as spec_markov_propose followed by spec_target_stats(target, l_dtype, temperature,
 *   R * (gamma + 1), V, target_stats): the proposal of "[DeepSeek-6] DSpark", sections 3-4, and
 *   the p_t normalisers that its rejection verification (section 9) needs.
 * The target normalisers do not depend on the proposal. With bf16 weights on the tensor cores
 * and R <= 256 the proposal runs as one persistent launch whose serial positions leave SMs
 * partly idle, and a share of its CTAs streams the target rows meanwhile. Other shapes run the
 * two operations one after the other.
 * Arguments: as spec_markov_propose (U of dtype l_dtype), plus
 *   target       [R, gamma+1, V] target logits, dtype l_dtype (required).
 *   target_stats [R*(gamma+1), 2] fp32 output (m, log Z) of softmax(target[row,:] / T), for
 *                spec_verify_rejection's target_stats.
 *   temperature  > 0 (the normalisers are those of the tempered target).
 * Errors as spec_markov_propose; SPEC_ERR_INVALID_ARG for a NULL target or target_stats.
 */
int spec_markov_propose_target_stats(const void* U, int l_dtype, const void* W1, const void* W2,
                                     int w_dtype, int rank, const int32_t* anchors,
                                     const float* u_draft, float temperature, int R, int gamma,
                                     int V, int32_t* draft_tokens, float* draft_logp,
                                     float* draft_stats, const void* target, float* target_stats,
                                     void* ws, size_t ws_bytes, void* stream);

/*
 * MTP/NextN greedy proposal and greedy verification of the same window in one call.
 * Defines: "Module deepseek_v4_mtp", Forward (without a Markov head the draft token of
 *   position k is the argmax of the draft logits of position k-1, so the positions are
 *   independent) and "DeepSeek-V4 MTP/NextN 怎样逐步生成候选", sections 三-四 (the verify
 *   window [bonus, d1..d_gamma]: accept the longest prefix of drafts equal to the target
 *   argmax of the row before them, then emit the target argmax of the row after it).
 * Equal to spec_markov_propose(D, dtype, NULL, NULL, 0, 0, NULL, NULL, 0, ...) followed by
 * spec_verify_greedy(target, dtype, draft_tokens, lengths, ...), bit for bit. With 16-byte
 * aligned logits, V a multiple of 8 (bf16) or 4 (fp32), gamma <= 1024 and R <= 2048 it is one
 * streaming launch over both tensors; other shapes run the two operations.
 * Arguments:
 *   D            [R, gamma, V] draft logits (bf16 or fp32, `dtype`); may be NULL if gamma = 0.
 *   target       [R, gamma+1, V] target logits of the same dtype.
 *   lengths      [R] int32 verified lengths l_r in [0, gamma], or NULL for gamma. Target rows
 *                past l_r are not read; all gamma draft tokens are always proposed.
 *   draft_tokens [R, gamma] int32 output: the draft argmax per position (ties: lowest id).
 *   accept_len, out_tokens, next_anchor: as spec_verify_greedy (out_tokens, next_anchor
 *                optional).
 * Workspace: spec_workspace_bytes(SPEC_OP_MTP_GREEDY, R, gamma, V, 0), initialised once with
 * spec_workspace_init (the launch uses per-request counters that it leaves at zero).
 * Errors: SPEC_ERR_INVALID_ARG for bad sizes or NULL required pointers,
 * SPEC_ERR_UNSUPPORTED_DTYPE, SPEC_ERR_WORKSPACE_TOO_SMALL. A row without a finite maximum sets
 * SPEC_DEV_NONFINITE (its argmax is then 0); a length outside [0, gamma] sets
 * SPEC_DEV_BAD_LENGTH and is clamped.
 */
int spec_mtp_greedy(const void* D, const void* target, int dtype, const int32_t* lengths, int R,
                    int gamma, int V, int32_t* draft_tokens, int32_t* accept_len,
                    int32_t* out_tokens, int32_t* next_anchor, void* ws, size_t ws_bytes,
                    void* stream);

/*
 * Greedy verification with a bonus token.
 * Defines: "DeepSeek-V4 MTP/NextN 怎样逐步生成候选", sections 三-四 (verify window
 *   [bonus, d1..d_gamma]; all accepted -> gamma drafts + one new bonus; first mismatch -> one
 *   target token) and "[DeepSeek-6] DSpark", section 1 (accept the longest legal prefix, then
 *   emit one bonus token).
 * With y_i = argmax target[r,i,:] (ties to the lowest id) and l = lengths[r] (gamma if NULL):
 *   n = the largest i <= l with x_j == y_{j-1} for all j <= i; bonus = y_n.
 * Arguments:
 *   target       [R, gamma+1, V] target logits, dtype t_dtype.
 *   draft_tokens [R, gamma] int32.
 *   lengths      [R] int32 in [0, gamma], or NULL.
 *   accept_len   [R] int32 output n.
 *   out_tokens   [R, gamma+1] int32 output x_1..x_n, bonus, then -1 padding (optional).
 *   next_anchor  [R] int32 output bonus (optional).
 */
int spec_verify_greedy(const void* target, int t_dtype, const int32_t* draft_tokens,
                       const int32_t* lengths, int R, int gamma, int V, int32_t* accept_len,
                       int32_t* out_tokens, int32_t* next_anchor, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * Softmax normalisers of target rows: stats[row] = (m, log Z) of softmax(target[row,:] / T).
 * Defines: "[DeepSeek-6] DSpark", section 3 (the exact per-token probabilities that
 *   rejection sampling needs) -- the p_t half of every probability used below.
 * Arguments: target [rows, V] (rows = R * (gamma+1) for a verify window), stats [rows, 2] fp32.
 */
int spec_target_stats(const void* target, int t_dtype, float temperature, int rows, int V,
                      float* stats, void* ws, size_t ws_bytes, void* stream);

/*
 * Lossless rejection-sampling verification with a residual resample or a bonus token.
 * Defines: named in "[DeepSeek-6] DSpark", sections 3 and 9 (exact draft probabilities make
 *   rejection sampling lossless; acceptance is governed by p_d versus p_t); the rule itself is
 *   standard speculative sampling: for k = 1..l accept x_k iff
 *   u_accept[r,k-1] * p_d,k(x_k) < p_t,k-1(x_k) (i.e. with probability min(1, p_t/p_d));
 *   at the first rejection k = n+1 the output token is the inverse-CDF draw with u_resid[r]
 *   from norm(max(0, p_t,n - p_d,n+1)); if all l survive it is drawn from p_t,l.
 * Arguments:
 *   target       [R, gamma+1, V] and U [R, gamma, V], both dtype l_dtype. With gamma = 0 every
 *                final row is a bonus row drawn from p_t alone and U may be NULL.
 *   W1, W2, rank, anchors: as spec_markov_propose (they rebuild p_d for the residual).
 *   draft_tokens [R, gamma] int32 from spec_markov_propose.
 *   draft_logp   [R, gamma] and draft_stats [R, gamma, 2] from the same propose call, at the
 *                same temperature.
 *   target_stats [R*(gamma+1), 2] from spec_target_stats at this temperature, or NULL to have
 *                them computed here.
 *   u_accept     [R, gamma] and u_resid [R] fp32 uniforms in [0, 1).
 *   temperature  > 0.
 *   lengths      [R] int32 in [0, gamma] (tokens to verify per request), or NULL for gamma.
 *   accept_len, out_tokens, next_anchor: as spec_verify_greedy (the output token replaces the
 *                greedy bonus).
 */
int spec_verify_rejection(const void* target, const void* U, int l_dtype, const void* W1,
                          const void* W2, int w_dtype, int rank, const int32_t* anchors,
                          const int32_t* draft_tokens, const float* draft_logp,
                          const float* draft_stats, const float* target_stats,
                          const float* u_accept, const float* u_resid, float temperature,
                          const int32_t* lengths, int R, int gamma, int V, int32_t* accept_len,
                          int32_t* out_tokens, int32_t* next_anchor, void* ws, size_t ws_bytes,
                          void* stream);

/*
 * TV soft labels and prefix survival.
 * Defines: "[DeepSeek-6] DSpark", section 5 (c*_k = 1 - 1/2 ||p_d,k - p_t,k||_1 over the
 *   softmaxed draft and aligned target logits) and section 6 (a_{r,j} = prod_{i<=j} c_{r,i}).
 * c*_{r,k} is evaluated as sum_v min(p_d,k(v), p_t,k-1(v)) (equal in exact arithmetic), with
 * p_d,k conditioned on the proposed prefix; a_{r,j} is the sequential fp32 product over j.
 * Arguments:
 *   U [R, gamma, V], target [R, gamma+1, V] (dtype l_dtype); W1, W2, rank, anchors as propose.
 *   draft_tokens [R, gamma]; draft_stats [R, gamma, 2] from propose at this temperature, or
 *   NULL to recompute them; target_stats as spec_verify_rejection (or NULL).
 *   conf [R, gamma] and survival [R, gamma] fp32 outputs (survival optional).
 */
int spec_tv_confidence(const void* U, const void* target, int l_dtype, const void* W1,
                       const void* W2, int w_dtype, int rank, const int32_t* anchors,
                       const int32_t* draft_tokens, const float* draft_stats,
                       const float* target_stats, float temperature, int R, int gamma, int V,
                       float* conf, float* survival, void* ws, size_t ws_bytes, void* stream);

/*
 * Grammar-masked drafting.
 * Defines: "Module deepseek_v4_mtp", Forward (the draft argmax is grammar-masked when a mask is
 *   given). Reading: `allowed` is a per-request bitmask [R, ceil(V/32)] uint32 (bit v%32 of
 *   word v/32 set = token v may be proposed; NULL = every token). The draft distribution of
 *   every position of request r is the softmax restricted to its allowed tokens (the others
 *   have logit -inf): argmax, sampling, draft_logp and draft_stats, the rejection residual
 *   norm(max(0, p_t - p_d)) and the TV label all use that restricted p_d. The target is never
 *   masked, so rejection verification stays lossless. A request with no allowed token sets
 *   SPEC_DEV_NONFINITE. Arguments otherwise as the unmasked entry points; a proposal made with
 *   a mask must be verified and scored with the same mask.
 */
int spec_markov_propose_masked(const void* U, int u_dtype, const void* W1, const void* W2,
                               int w_dtype, int rank, const int32_t* anchors,
                               const float* u_draft, float temperature, int R, int gamma, int V,
                               int32_t* draft_tokens, float* draft_logp, float* draft_stats,
                               const uint32_t* allowed, void* ws, size_t ws_bytes,
                               void* stream);
int spec_verify_rejection_masked(const void* target, const void* U, int l_dtype, const void* W1,
                                 const void* W2, int w_dtype, int rank, const int32_t* anchors,
                                 const int32_t* draft_tokens, const float* draft_logp,
                                 const float* draft_stats, const float* target_stats,
                                 const float* u_accept, const float* u_resid, float temperature,
                                 const int32_t* lengths, int R, int gamma, int V,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* next_anchor,
                                 const uint32_t* allowed, void* ws, size_t ws_bytes,
                                 void* stream);
int spec_tv_confidence_masked(const void* U, const void* target, int l_dtype, const void* W1,
                              const void* W2, int w_dtype, int rank, const int32_t* anchors,
                              const int32_t* draft_tokens, const float* draft_stats,
                              const float* target_stats, float temperature, int R, int gamma,
                              int V, float* conf, float* survival, const uint32_t* allowed,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * Hardware-aware prefix scheduler.
 * Defines: "[DeepSeek-6] DSpark", section 6: maximise Theta = tau * SPS(B) with
 *   B = sum_r (1 + l_r) and tau = sum_r (1 + sum_{j<=l_r} a_{r,j}), queueing every candidate
 *   (r, j) by a_{r,j} in decreasing order (prefix-closed because a is non-increasing in j).
 * Candidates are ordered by (a desc, r asc, j asc); tau is carried in fixed point
 * q = round-half-even(a * 2^32) so that the prefix sums are exact integers; for
 * K = 0..min(R*gamma, Bmax-R): Theta(K) = double(R * 2^32 + S_K) * sps[R+K]; K* is the smallest
 * K reaching the maximum and l_r counts the selected candidates of request r. The result is
 * bit-identical to any implementation of the same definition.
 * Arguments:
 *   survival [R, gamma] fp32 in [0, 1], non-increasing in j.
 *   sps      [Bmax+1] fp64 steps per second at batch size B (index B), finite and >= 0.
 *   lengths  [R] int32 output; B_out [1] int32 output; theta_out [1] fp64 output
 *            (tau * SPS(B) in natural units). All three are device pointers.
 * Requires R * gamma <= SPEC_SCHEDULE_MAX_CANDIDATES and Bmax >= R.
 */
int spec_schedule_prefix(const float* survival, const double* sps, int Bmax, int R, int gamma,
                         int32_t* lengths, int32_t* B_out, double* theta_out, void* ws,
                         size_t ws_bytes, void* stream);

/*
 * Dynamic top-K prefix selection.
 * Defines: "[DeepSeek-6] DSpark", section 7 (asynchronous scheduling): the verify batch size is
 *   decided from confidences computed steps earlier, and the current step fills that capacity
 *   with its own highest-survival candidates. With capacity B the first
 *   K = clamp(B - R, 0, min(R*gamma, Bmax-R)) candidates of the same queue as
 *   spec_schedule_prefix (a desc, r asc, j asc) are selected, so the selection is prefix-closed
 *   per request and equals spec_schedule_prefix's whenever B is that scheduler's optimum.
 * Arguments as spec_schedule_prefix, plus:
 *   capacity [1] int32 device pointer: the batch size B (typically B_out of an earlier call).
 *            It is read by the kernel, so it may be written by earlier work on `stream`.
 *   theta_out receives Theta at the selected K; B_out receives R + K.
 *   B_opt_out [1] int32 device pointer or NULL: receives the batch size spec_schedule_prefix
 *            would choose for this survival (R + K*), the capacity of a later step. The same
 *            sorted queue serves both, so this costs no second sort.
 * A negative capacity selects K = 0 and sets SPEC_DEV_BAD_LENGTH in the device status word.
 * Returns SPEC_ERR_INVALID_ARG for a null capacity, otherwise as spec_schedule_prefix.
 */
int spec_schedule_topk(const float* survival, const double* sps, int Bmax, int R, int gamma,
                       const int32_t* capacity, int32_t* lengths, int32_t* B_out,
                       double* theta_out, int32_t* B_opt_out, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * Flattened (variable-length) verify batch.
 * Defines: "[DeepSeek-6] DSpark", section 7 (production adaptation): padding every request to
 *   the same query length would spend on padding the verify budget the scheduler just saved,
 *   so the physical batch is the tokens of all requests flattened into independent rows, and
 *   the per-sequence structure travels in a marker tensor.
 * Layout: request r owns the 1 + l_r packed target rows offsets[r] .. offsets[r+1]-1 (its
 *   verify positions 0..l_r, position l_r being the bonus position); B = offsets[R] is the
 *   scheduler's batch size sum_r (1 + l_r). A packed target array is allocated for
 *   R*(gamma+1) rows (the largest batch); only its first B rows are read.
 *
 * spec_flat_layout: from lengths [R] int32 in [0, gamma] (device) writes
 *   offsets  [R+1] int32 (device, required) and the markers
 *   row_req  [R*(gamma+1)] int32 request of each packed row (optional, -1 past B) and
 *   row_pos  [R*(gamma+1)] int32 position of each packed row (optional, -1 past B).
 *   A length outside [0, gamma] is clamped and sets SPEC_DEV_BAD_LENGTH. The workspace is
 *   used for its status word only (ws_bytes >= 256).
 */
int spec_flat_layout(const int32_t* lengths, int R, int gamma, int32_t* offsets,
                     int32_t* row_req, int32_t* row_pos, void* ws, size_t ws_bytes,
                     void* stream);

/*
 * Packing of padded rows into the flattened layout: for every request r and position
 * i <= l_r, row (r, i) of src [R, gamma+1, row_bytes] is copied to packed row offsets[r] + i of
 * dst [R*(gamma+1), row_bytes]. Rows past a request's length are neither read nor written, so
 * the bytes moved are those of the B scheduled rows. It stands in for a target model that
 * writes its logits (or a caller's per-row statistics) straight into the packed layout.
 *   row_bytes  bytes per row, a multiple of 4 (16-byte rows and pointers copy 16 bytes at a
 *              time); lengths and offsets as for spec_flat_layout (device).
 * A length outside [0, gamma] is clamped and sets SPEC_DEV_BAD_LENGTH; so does an offset that
 * would put a row outside the R*(gamma+1) packed rows (that row is not written). The
 * workspace is used for its status word only (ws_bytes >= 256).
 */
int spec_flat_pack(const void* src, int row_bytes, const int32_t* lengths,
                   const int32_t* offsets, int R, int gamma, void* dst, void* ws, size_t ws_bytes,
                   void* stream);

/*
 * Target normalisers of a flattened batch: stats[b] = (m, log Z) of softmax(target[b,:] / T)
 * for the packed rows b < offsets[R]; rows past the batch are neither read nor written.
 * target [R*(gamma+1), V] packed, stats [R*(gamma+1), 2] fp32 (packed like target).
 */
int spec_target_stats_flat(const void* target, int t_dtype, float temperature, int R, int gamma,
                           int V, const int32_t* offsets, float* stats, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * Greedy verification of a flattened batch: as spec_verify_greedy with target row (r, i) at
 * packed row offsets[r] + i. lengths and offsets (from spec_flat_layout of the same lengths)
 * are required; outputs keep the per-request [R, gamma+1] layout. Offsets that put a row
 * outside the R*(gamma+1) packed rows set SPEC_DEV_BAD_LENGTH (the row is then read as row 0).
 */
int spec_verify_greedy_flat(const void* target, int t_dtype, const int32_t* draft_tokens,
                            const int32_t* lengths, const int32_t* offsets, int R, int gamma,
                            int V, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* next_anchor, void* ws, size_t ws_bytes, void* stream);

/*
 * Rejection verification of a flattened batch: as spec_verify_rejection_masked with target
 * row (r, i) at packed row offsets[r] + i; target_stats (optional) is packed the same way
 * (spec_target_stats_flat). lengths and offsets are required; `allowed` may be NULL.
 * U, draft tokens, draft statistics, uniforms and outputs keep their per-request layouts.
 */
int spec_verify_rejection_flat(const void* target, const void* U, int l_dtype, const void* W1,
                               const void* W2, int w_dtype, int rank, const int32_t* anchors,
                               const int32_t* draft_tokens, const float* draft_logp,
                               const float* draft_stats, const float* target_stats,
                               const float* u_accept, const float* u_resid, float temperature,
                               const int32_t* lengths, const int32_t* offsets, int R, int gamma,
                               int V, int32_t* accept_len, int32_t* out_tokens,
                               int32_t* next_anchor, const uint32_t* allowed, void* ws,
                               size_t ws_bytes, void* stream);

/* Largest R * (gamma + 1) that spec_verify_greedy_noalloc accepts. */
#define SPEC_NOALLOC_MAX_ROWS 65536

/*
 * Greedy verification that allocates nothing and takes no workspace.
 * No page defines this entry point: it exists for callers that cannot allocate
 * device memory at the call site (a plug-in inside an engine that reserves all device memory at
 * start-up, a latency-critical loop that must not meet cudaMalloc's implicit synchronisation,
 * a host whose memory is owned by another framework's allocator). It computes exactly what
 * spec_verify_greedy computes, with the same arguments and outputs, except:
 *   - its scratch (a status word and one argmax per target row, 256 + 4 * 65536 bytes) is a
 *     fixed device array inside the library, held by every GPU that loads the library until the
 *     process exits; R * (gamma + 1) above SPEC_NOALLOC_MAX_ROWS returns SPEC_ERR_TOO_LARGE
 *     before any launch;
 *   - the first call on a device looks up that array's device address (once per device, with
 *     that device current); make that first call before any stream capture. The address is
 *     kept for the life of the process: after a cudaDeviceReset of that device it is stale, and
 *     this entry point must not be called on that device again;
 *   - every call on a device shares the one array, so calls whose work overlaps on the GPU
 *     (other streams, other host threads) race and give undefined results: order them;
 *   - the device status bits of this call (SPEC_DEV_*, cleared at the start of every call) are
 *     copied into *device_status (a device pointer, optional) at the end of the call's work.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 */
int spec_verify_greedy_noalloc(const void* target, int t_dtype, const int32_t* draft_tokens,
                               const int32_t* lengths, int R, int gamma, int V,
                               int32_t* accept_len, int32_t* out_tokens, int32_t* next_anchor,
                               uint32_t* device_status, void* stream);

/*
 * TEST-ONLY: never call this outside a test of the timeout path; the next tensor-core pass it
 * stalls produces no result.
 * Test support for the bounded waits (no counterpart on the pages). The next tensor-core
 * Markov pass launched by this process never receives its first W2 tile, so its MMA thread's
 * wait expires (after about 2 s of SM clock): the kernel sets SPEC_DEV_TIMEOUT in the device
 * status word, abandons its work (its partials, and the outputs built from them, are
 * invalid), drains its copies, frees its tensor memory and returns; the CUDA context stays
 * usable. Nothing faults or hangs.
 */
int spec_test_stall_next_markov(void);

/*
 * Tracing (no counterpart on the pages; instrumentation of this library).
 * Kernel classes: SPEC_KCLASS_MARKOV (the Markov producer: tensor-core GEMM fused with the
 * softmax / residual / TV epilogue, or its CUDA-core form), SPEC_KCLASS_STREAM (rank-0 streaming
 * row reductions), SPEC_KCLASS_SELECT (per-row select / sample), SPEC_KCLASS_OTHER (scans,
 * finalisers, the scheduler), SPEC_KCLASS_PROPOSE (the persistent tensor-core proposal: every
 * position with its selects, and the target normalisers of the fused entry point).
 */
#define SPEC_KCLASS_MARKOV 0
#define SPEC_KCLASS_STREAM 1
#define SPEC_KCLASS_SELECT 2
#define SPEC_KCLASS_OTHER 3
#define SPEC_KCLASS_PROPOSE 4
#define SPEC_KCLASS_COUNT 5

/* Number of kernels this process has launched through the library (all classes). */
unsigned long long spec_launch_count(void);

/*
 * Attach caller-created CUDA events (cudaEvent_t handles created with timing enabled) to one
 * kernel class: the i-th launch of that class after this call records begin_events[i] before
 * and end_events[i] after itself on the launch stream, for i < capacity. The records are
 * external (cudaEventRecordExternal), so a launch captured into a CUDA graph keeps them as timing
 * records at each replay. Pass capacity 0 to detach. The events stay owned by the caller.
 * Process-global state; not thread-safe.
 */
int spec_trace_events(int kclass, void* const* begin_events, void* const* end_events,
                      int capacity);

/* Launches of `kclass` recorded into the attached events since spec_trace_events. */
int spec_trace_count(int kclass);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_MARKOV_H */
