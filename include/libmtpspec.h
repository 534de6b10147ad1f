/*
 * libmtpspec — the data-parallel hot path of MTP (multi-token prediction) speculative
 * decoding on one NVIDIA GB300 GPU (sm_103a): the draft head's input stage, greedy
 * drafting, and greedy or speculative-sampling verification of a batch of drafts.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every array pointer is a DEVICE pointer owned by the caller.  The library never
 *    allocates, frees or keeps any of them after the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL: the legacy default stream).  All
 *    work is enqueued on it asynchronously; nothing synchronises the host.
 *  - The return value reports what the host can see before launching: MTPSPEC_OK, or a
 *    negative mtpspec_status for a bad argument, dtype, shape or workspace, or a launch
 *    failure.  Nothing is enqueued when the return value is not MTPSPEC_OK.
 *  - What only the device can see (a draft id outside [0, V), a bad per-row sampling
 *    parameter) is OR-ed into the optional device word `*status` as MTPSPEC_STATUS_*
 *    bits; the caller zeroes that word beforehand.  No kernel traps.
 *  - Row-major, contiguous arrays.  Logits are float32 or bfloat16 (mtpspec_dtype);
 *    bfloat16 arrays are passed as their 16-bit patterns.  Token ids are int32.
 *  - Inputs must be finite or -inf.  NaN logits give unspecified (but in-bounds)
 *    results.
 *
 * Sources, cited by page title and section:
 *  [HB] "14. MTP: speculative decoding with the built-in draft head" (Transformer by
 *       Hand, stage 2), sections "The draft head" and "The speculative decoding loop
 *       (greedy version)".
 *  [DL] "The decoding loop and MTP" (agent-loop-visualizer docs), sections "Why a
 *       hand-written decoding loop" and "MTP speculative decoding".
 *  [ZH] "MPT (MTP, Multi-Token Prediction) 原理详解", sections 二.2 (forward 流程),
 *       三 (stages 0-4) and 四 (worked example).
 *  [PX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 *       (SC'11), Philox4x32-10.
 */
#ifndef LIBMTPSPEC_H
#define LIBMTPSPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MTPSPEC_OK = 0,
    MTPSPEC_ERR_ARG = -1,          /* null pointer, misaligned pointer, bad scalar */
    MTPSPEC_ERR_DTYPE = -2,        /* dtype is not MTPSPEC_F32 / MTPSPEC_BF16 */
    MTPSPEC_ERR_SHAPE = -3,        /* a size is out of the supported range */
    MTPSPEC_ERR_WORKSPACE = -4,    /* workspace null or smaller than required */
    MTPSPEC_ERR_CUDA = -5,         /* a CUDA runtime call or kernel launch failed */
    MTPSPEC_ERR_UNSUPPORTED = -6   /* the current device is not sm_103 */
} mtpspec_status;

typedef enum { MTPSPEC_F32 = 0, MTPSPEC_BF16 = 1 } mtpspec_dtype;

/* Bits OR-ed into the device status word. */
#define MTPSPEC_STATUS_BAD_DRAFT_ID 0x1 /* a draft id outside [0, V); that draft is rejected */
#define MTPSPEC_STATUS_BAD_PARAM 0x2    /* a row with temperature < 0 or NaN, or top_p <= 0 or
                                           NaN; that row is verified greedily */
#define MTPSPEC_STATUS_TIMEOUT 0x4      /* a bounded wait inside a kernel gave up (a copy
                                           engine fault); outputs of that call are invalid */

/* ------------------------------------------------------------------ draft input stage */

/*
 * mtp_draft_input — the MTP draft head's input stage ([HB] "The draft head":
 * fc(cat(norm(e_{t+1}), norm(h_t))); [ZH] 二.2 steps 2-3: eh_proj(cat(enorm(embeds),
 * hnorm(previous_hidden_states)))).  For each of M tokens:
 *     x   = [ rmsnorm(emb_next[t]) * enorm_w ; rmsnorm(hidden[t]) * hnorm_w ]   (2H)
 *     out[t] = eh_proj_w @ x                                                    (H)
 * with rmsnorm(v) = v / sqrt(mean(v^2) + eps).  The normalised activations are rounded
 * to bf16; the projection accumulates in fp32 and rounds its output to bf16.
 *
 *   emb_next, hidden  bf16 [M, H]    embedding of token t+1 and main-model hidden state
 *                                    at position t (after the main model's final norm)
 *   enorm_w, hnorm_w  bf16 [H]       RMSNorm weights
 *   eh_proj_w         bf16 [H, 2H]   row-major (out x in); columns 0..H-1 multiply the
 *                                    embedding half, H..2H-1 the hidden half
 *   out               bf16 [M, H]
 *   M >= 0 tokens, 1 <= H <= 65536 with H % 8 == 0, eps >= 0.
 *   workspace         device scratch of at least mtp_draft_input_workspace_bytes(M, H)
 *                     bytes (may be NULL when that is 0), 256-byte aligned.
 * Every pointer must be 16-byte aligned.  Small M streams the weight once through a
 * fused norm + GEMV; large M normalises into the workspace and runs a tcgen05 GEMM.
 * Returns MTPSPEC_OK (also for M == 0, with nothing enqueued) or an error as above.
 */
int mtp_draft_input(const void *emb_next, const void *hidden, const void *enorm_w,
                    const void *hnorm_w, const void *eh_proj_w, void *out, int64_t M, int64_t H,
                    float eps, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace mtp_draft_input needs for (M, H); 0 on the GEMV path.
 * Returns 0 as well for arguments mtp_draft_input would reject. */
size_t mtp_draft_input_workspace_bytes(int64_t M, int64_t H);

/* ------------------------------------------------------------------ greedy drafting */

/*
 * mtp_greedy_draft — greedy draft tokens: the argmax of each row of draft logits
 * ([HB] "The speculative decoding loop": the draft is the argmax of the draft head's
 * logits; [ZH] 三 stages 1-2, greedy sample of each MTP step), taking the LOWEST id
 * among equal maxima ([DL] "Why a hand-written decoding loop").  bf16 values are
 * compared as stored; -inf is an ordinary value, so an all -inf row gives id 0.
 *
 *   logits   [M, V] of dtype        out_ids  int32 [M]
 *   M >= 0, 1 <= V <= 2^31 - 1.  logits aligned to its element size.
 */
int mtp_greedy_draft(const void *logits, int dtype, int64_t M, int64_t V, int32_t *out_ids,
                     void *stream);

/*
 * mtp_lm_head_greedy — the greedy draft straight from the draft head's output layer,
 * without writing the [M, V] logits ([HB] "The draft head": the block's output passes a
 * normalisation and the output layer shared with the main model, and the draft is the
 * argmax of those logits; [ZH] 二.1 shared_head = the main model's lm_head, 三 stage 1
 * compute_logits then greedy sample).  For each of M tokens:
 *     x        = hidden[t], or rmsnorm(hidden[t]) * norm_w rounded to bf16 when norm_w
 *                is given (rmsnorm as in mtp_draft_input)
 *     logits_v = sum_k lm_head_w[v, k] * x_k       (bf16 products, fp32 accumulation)
 *     out_ids[t]   = the LOWEST v among the largest logits_v ([DL] "Why a hand-written
 *                    decoding loop": argmax takes the lower id)
 *     out_logit[t] = that largest logit (fp32), when out_logit is not NULL.
 * The pick is made on the fp32 sums: where the two largest exact logits lie within the
 * fp32 rounding of the sum, either id may come back.
 *
 *   hidden       bf16 [M, H]    the draft block's output (before the final norm when
 *                               norm_w is given)
 *   norm_w       bf16 [H] or NULL   final RMSNorm weight; eps >= 0 its epsilon
 *   lm_head_w    bf16 [V, H]    row-major (vocabulary x hidden), as nn.Linear(H, V)
 *   out_ids      int32 [M]      out_logit float [M] or NULL
 *   workspace    >= mtp_lm_head_greedy_workspace_bytes(M, H, V) bytes, 256-byte aligned
 *   status       int32 [1] or NULL   MTPSPEC_STATUS_TIMEOUT is OR-ed in if a wait of the
 *                                    GEMM gave up (its ids are then unspecified)
 *   M >= 0 (<= 2^20), 8 <= H <= 65536 with H % 8 == 0, 1 <= V <= 8,388,480.  hidden,
 *   norm_w and lm_head_w 16-byte aligned.  Returns MTPSPEC_OK (also for M == 0, with
 *   nothing enqueued) or an error as above.
 */
int mtp_lm_head_greedy(const void *hidden, const void *norm_w, float eps, const void *lm_head_w,
                       int64_t M, int64_t H, int64_t V, int32_t *out_ids, float *out_logit,
                       void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/* Bytes of device workspace mtp_lm_head_greedy needs for (M, H, V); 0 for arguments it
 * would reject. */
size_t mtp_lm_head_greedy_workspace_bytes(int64_t M, int64_t H, int64_t V);

/*
 * mtp_draft_steps — D serial greedy draft steps of the draft head ([ZH] 三 stages 1-2: the
 * bonus token and the main model's hidden state start the chain; each step embeds the
 * previous token, runs the head, greedy-samples the next draft and passes the token and
 * the head's hidden state to the next step; 二.2 step 1: the input embedding at position 0
 * is zeroed; [HB] "The draft head").  The head's decoder block is not part of this
 * library: its output is taken to be its input.  Step k = 0 .. D-1, with ids = next_ids
 * and h = hidden before step 0:
 *     e   = embed_w[ids[t]], or a zero row where positions[t] + k == 0 (or the id lies
 *           outside [0, V): then MTPSPEC_STATUS_BAD_DRAFT_ID is OR-ed into *status)
 *     y   = mtp_draft_input(e, h)                      (bf16 [M, H])
 *     ids = mtp_lm_head_greedy(y, norm_w, lm_head_w)   -> draft_ids[:, k]
 *     h   = y
 * Every step is one embedding gather, the input stage and the output layer; nothing is
 * allocated or synchronised, so the call can be captured into a CUDA graph.
 *
 *   embed_w     bf16 [V, H]   token embeddings (shared with the main model)
 *   next_ids    int32 [M]     the token after each row's last verified position
 *   positions   int32 [M] or NULL   that token's position (no mask when NULL)
 *   hidden      bf16 [M, H]   the main model's hidden state at the previous position
 *   enorm_w, hnorm_w, eh_proj_w   as in mtp_draft_input
 *   norm_w      bf16 [H] or NULL, lm_head_w bf16 [V, H]   as in mtp_lm_head_greedy
 *   draft_ids   int32 [M, D]  hidden_out bf16 [D, M, H] or NULL (every step's y)
 *   workspace   >= mtp_draft_steps_workspace_bytes(M, H, V) bytes, 256-byte aligned
 *   status      int32 [1] or NULL
 *   M >= 0 (<= 2^20), 8 <= H <= 65536 with H % 8 == 0, 1 <= V <= 8,388,480, 1 <= D <= 64.
 *   Matrices, norm weights and hidden_out 16-byte aligned.
 */
int mtp_draft_steps(const void *embed_w, const int32_t *next_ids, const int32_t *positions,
                    const void *hidden, const void *enorm_w, const void *hnorm_w,
                    const void *eh_proj_w, const void *norm_w, const void *lm_head_w, float eps,
                    int64_t M, int64_t H, int64_t V, int32_t D, int32_t *draft_ids,
                    void *hidden_out, void *workspace, size_t workspace_bytes, int32_t *status,
                    void *stream);

/* Bytes of device workspace mtp_draft_steps needs for (M, H, V); 0 for arguments it would
 * reject. */
size_t mtp_draft_steps_workspace_bytes(int64_t M, int64_t H, int64_t V);

/*
 * mtp_lm_head_topk — the k largest logits of the draft output layer, for a drafter that
 * proposes several candidates per position, again without writing the [M, V] logits
 * ([HB] "The draft head" and [ZH] 三 stage 1: the output layer's logits; [DL] "Why a
 * hand-written decoding loop": top-k keeps the k largest, and a tie goes to the lower id).
 * The logits are those of mtp_lm_head_greedy.
 *   out_ids     int32 [M, k]   the ids of the k largest logits of each token, in
 *                              decreasing order, equal logits by increasing id
 *   out_logits  float [M, k] or NULL   their fp32 logits
 *   1 <= k <= 8 and k <= V; workspace >= mtp_lm_head_topk_workspace_bytes(M, H, V).
 * Other arguments, limits and errors as mtp_lm_head_greedy.  As there, the order is taken
 * on the fp32 sums: ids whose exact logits lie within the fp32 rounding of each other may
 * come back in either order (or, at the k-th place, either may be listed).
 */
int mtp_lm_head_topk(const void *hidden, const void *norm_w, float eps, const void *lm_head_w,
                     int64_t M, int64_t H, int64_t V, int32_t k, int32_t *out_ids,
                     float *out_logits, void *workspace, size_t workspace_bytes, int32_t *status,
                     void *stream);

/* Bytes of device workspace mtp_lm_head_topk needs for (M, H, V) (any k); 0 for
 * arguments it would reject. */
size_t mtp_lm_head_topk_workspace_bytes(int64_t M, int64_t H, int64_t V);

/* ------------------------------------------------------------------ greedy verification */

/*
 * spec_verify_greedy — greedy verification of D drafts per row ([HB] "The speculative
 * decoding loop (greedy version)": a draft is kept when it equals the main model's own
 * argmax, otherwise the main model's token replaces it; [ZH] 三 stage 3 "greedy
 * strategy" and stage 4, 四 steps C-D; [DL] "MTP speculative decoding" item 2: when
 * all guesses hold the last position gives one more token).
 *
 *   target_logits  [B, D+1, V]  row b, position j predicts the token after position j
 *                               of the verified sequence [bonus, d_0, .., d_{D-1}]
 *   draft_ids      int32 [B, D]
 *   out_tokens     int32 [B, D+1]  d_0 .. d_{a-1}, then argmax(target[b, a]) (the
 *                                  correction, or the bonus token when a = D), then -1
 *   num_accepted   int32 [B]       a = the number of leading drafts equal to the argmax
 *                                  at their position (0..D).  Tokens emitted = a + 1;
 *                                  a KV cache of the verified sequence keeps 1 + a
 *                                  entries.
 *   status         int32 [1] or NULL   MTPSPEC_STATUS_BAD_DRAFT_ID for ids outside [0, V)
 *   B >= 0, 1 <= D <= 64, 1 <= V <= 2^31 - 1.
 */
int spec_verify_greedy(const void *target_logits, int dtype, const int32_t *draft_ids, int64_t B,
                       int32_t D, int64_t V, int32_t *out_tokens, int32_t *num_accepted,
                       int32_t *status, void *stream);

/* ------------------------------------------------------------------ sampling verification */

/*
 * spec_verify_sample — speculative-sampling verification ([ZH] 三 stage 3 "rejection
 * sampling" and stage 4; [DL] "Why a hand-written decoding loop" for the filters and
 * "MTP speculative decoding" items 2-3; [HB] "How to explain it": the output
 * distribution is unchanged).  For each row b with temperature tau_b > 0:
 *   p_j = filter(target_logits[b, j]), q_j = filter(draft_logits[b, j]), where filter
 *         is: divide by tau_b, keep logits >= the k-th largest (top-k, ties kept), form
 *         the softmax, keep a token when the mass of strictly larger kept logits is
 *         < top_p (top-p), renormalise;
 *   draft j < D is accepted when d_j is in the support of p_j and (d_j is outside the
 *         support of q_j, or U_acc(b, j) <= p_j(d_j) / q_j(d_j));
 *   at the first rejected position a the token is drawn from
 *         normalize(max(0, p_a - q_a)) (from p_a if that is identically zero);
 *   when all D drafts are accepted the bonus token is drawn from p_D.
 * Draws take the inverse CDF in ascending id order with U_smp(b, j).  U_acc, U_smp are
 * Philox4x32-10 ([PX]) outputs 0 and 1 for key (seed lo, seed hi) and counter
 * (b, j, 0, 0), each mapped to (2 * (word >> 9) + 1) * 2^-24.  A row with tau_b = 0 is
 * verified greedily as in spec_verify_greedy (reported p_target = [d_j == argmax],
 * p_draft = 1).
 * draft_logits may be NULL: a one-hot draft, q_j the point mass on d_j (greedy guesses,
 * [DL] "MTP speculative decoding" items 1 and 3: a guess is kept with its probability
 * under p_j, otherwise the token is drawn from the other candidates).  Then d_j is
 * accepted when it is in the support of p_j and U_acc(b, j) <= p_j(d_j), the residual is
 * p_a with d_a removed, p_draft reports 1 (0 for an id outside [0, V)), and only the
 * target logits are read.
 *
 *   target_logits  [B, D+1, V]     draft_logits [B, D, V] (same dtype) or NULL
 *   draft_ids      int32 [B, D]
 *   temperature    float [B]       0 => greedy row
 *   top_k          int32 [B] or NULL   <= 0 or >= V => off
 *   top_p          float [B] or NULL   >= 1 => off; must be > 0
 *   seed           Philox key
 *   out_tokens, num_accepted   as in spec_verify_greedy
 *   p_target, p_draft  float [B, D] or NULL   p_j(d_j) and q_j(d_j) for every j < D; when
 *                  both are NULL the call may skip the positions behind each row's first
 *                  rejection, and the top-p thresholds of a draft whose acceptance is
 *                  already certain (no output depends on them), which makes it faster; the
 *                  tokens and accepted counts are the same either way
 *   workspace      >= spec_verify_workspace_bytes(B, D, V) bytes, 256-byte aligned;
 *                  no initial contents are needed
 *   status         int32 [1] or NULL
 *   B >= 0, 1 <= D <= 64, 1 <= V <= 2,097,152 (fp32) or 4,194,304 (bf16); a larger V
 *   returns MTPSPEC_ERR_SHAPE.
 *   Two verifiers compute these results.  Up to V = 407,552 (fp32) or 815,104 (bf16) with
 *   draft logits, 651,776 or 1,303,552 with a one-hot draft, a cluster of at most 16 CTAs
 *   stages a unit's rows in shared memory and verifies the unit alone.  Past those limits
 *   (or with the environment variable MTPSPEC_VERIFY_IMPL=chunks) the chunked verifier
 *   cuts each unit's rows into up to 256 chunks of 32 KB of logits, spread over the CTAs
 *   resident on the GPU, which combine their chunks' statistics through the workspace.
 *   Both follow the rule above; the outputs of one verifier are deterministic, those of
 *   the two agree except where a decision sits within rounding of its boundary.
 */
int spec_verify_sample(const void *target_logits, const void *draft_logits, int dtype,
                       const int32_t *draft_ids, const float *temperature, const int32_t *top_k,
                       const float *top_p, uint64_t seed, int64_t B, int32_t D, int64_t V,
                       int32_t *out_tokens, int32_t *num_accepted, float *p_target,
                       float *p_draft, void *workspace, size_t workspace_bytes, int32_t *status,
                       void *stream);

/* Bytes of device workspace spec_verify_sample needs for (B, D, V); 0 for B == 0 or
 * for arguments spec_verify_sample rejects whatever the logit type (V above the bf16
 * limit included).  Up to the cluster limit for fp32 with draft logits (V <= 407,552)
 * this is 16 bytes per unit plus 4 per row; beyond it, or with MTPSPEC_VERIFY_IMPL=chunks
 * set when both calls are made, it adds the chunked verifier's coordination slots: up
 * to 128 slots, each about 80 KB plus 12 bytes per nucleus entry (V / 3 entries, at
 * least 8,192 and at most 65,536). */
size_t spec_verify_workspace_bytes(int64_t B, int32_t D, int64_t V);

/*
 * spec_verify_sample_static — spec_verify_sample without a caller-supplied workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory, such as a serving loop whose device memory is owned entirely
 * by another allocator (a framework's caching pool that must see every allocation), or a
 * latency-critical decode step that must never risk the device-wide synchronisation an
 * allocation can cause.  The per-unit scratch lives in a fixed array inside the library
 * (1 MiB of device memory on every GPU that loads the library, held until the process
 * exits), so this call allocates nothing.
 *   Arguments, outputs and status: as spec_verify_sample.
 *   Limit: B * (D + 1) <= 65536; a larger batch returns MTPSPEC_ERR_SHAPE.
 *   Device: the scratch used is the one on the stream's device (the call makes that
 *   device current, as every entry point does).  The first call on a device does the
 *   set-up: it looks up the array's device address, with that device current.  Make
 *   that first call before any stream capture begins.  While its stream is being
 *   captured, the call does not ask the stream for its device; it takes the current
 *   device, which must then be the stream's.
 *   The looked-up address is kept for the life of the process: after cudaDeviceReset
 *   (or anything else that destroys the device's primary context) this entry point
 *   must not be called again on that device.
 *   All calls on a device share the array and each call overwrites the records it uses:
 *   two calls whose GPU work can overlap (different streams, or threads without stream
 *   ordering between them) race on it and give undefined results.
 */
int spec_verify_sample_static(const void *target_logits, const void *draft_logits, int dtype,
                              const int32_t *draft_ids, const float *temperature,
                              const int32_t *top_k, const float *top_p, uint64_t seed,
                              int64_t B, int32_t D, int64_t V, int32_t *out_tokens,
                              int32_t *num_accepted, float *p_target, float *p_draft,
                              int32_t *status, void *stream);

/* ------------------------------------------------------------------ state around a verification */

/*
 * mtp_state_snapshot — the copy taken before a verification ([HB] the decoding loop's
 * snapshot and "Rolling back": a KV cache needs only its length, which the caller keeps;
 * the linear attention's memory tables and convolution windows are copied):
 *     backup[b] = state[b]   for each of B rows of row_bytes bytes.
 *   state, backup   device [B, row_bytes], 16-byte aligned, not overlapping
 *   B >= 0 (<= 2^24), row_bytes >= 0 with row_bytes % 16 == 0.
 * Returns MTPSPEC_OK (nothing enqueued when there is nothing to copy) or an error.
 */
int mtp_state_snapshot(const void *state, void *backup, int64_t B, int64_t row_bytes,
                       void *stream);

/*
 * mtp_state_fixup — the model state after a verification, from the verifier's accepted
 * counts ([HB] the decoding loop's hit / miss branches and "Rolling back"; [ZH] 三 stage
 * 4).  The verify forward appended D + 1 positions (the carried-in token and the D
 * drafts) after kv_len_before[b].  With a = num_accepted[b]:
 *   a == D (hit):   kv_len = kv_len_before + D + 1; the state is kept; recompute = 0.
 *   a <  D (miss), row_bytes > 0 (a recurrent state):  state[b] = backup[b] (the memory
 *                   tables absorbed rejected drafts and cannot be undone), kv_len =
 *                   kv_len_before (truncated), recompute = 1 + a: the carried-in token and
 *                   the accepted drafts must pass the model again.
 *   a <  D, row_bytes == 0 (attention only):  kv_len = kv_len_before + 1 + a (the kept
 *                   keys do not depend on later positions); recompute = 0.
 *   on a miss, draft_kv_len (the draft head's own cache) = min(draft_kv_len, kv_len).
 * A row with a outside [0, D] is left untouched and ORs MTPSPEC_STATUS_BAD_PARAM into
 * *status.
 *   num_accepted, kv_len_before  int32 [B]      kv_len  int32 [B] (may be kv_len_before)
 *   state   device [B, row_bytes] (in/out)   backup  device [B, row_bytes] from
 *           mtp_state_snapshot; both 16-byte aligned and not overlapping; unused when
 *           row_bytes == 0
 *   draft_kv_len, recompute  int32 [B] or NULL   status  int32 [1] or NULL
 *   B >= 0 (<= 2^24), 1 <= D <= 64, row_bytes >= 0 with row_bytes % 16 == 0.
 */
int mtp_state_fixup(const int32_t *num_accepted, int32_t D, const int32_t *kv_len_before,
                    int32_t *kv_len, void *state, const void *backup, int64_t B,
                    int64_t row_bytes, int32_t *draft_kv_len, int32_t *recompute,
                    int32_t *status, void *stream);

/* ------------------------------------------------------------------ misc */

/* A static, human-readable name for an mtpspec_status value. */
const char *mtpspec_status_string(int code);

/* mtpspec_selftest_wait_timeout — a diagnostic of the kernels' bounded waits (every wait on
 * a copy, a barrier or another CTA gives up after a fixed number of polls and ORs
 * MTPSPEC_STATUS_TIMEOUT into the status word, so that a call that cannot finish returns
 * and leaves the context usable).  It launches one CTA that runs the wait of one kernel
 * family on a barrier or counter that nothing completes, with `limit` polls instead of the
 * kernels' own limit:
 *   which 0  the cluster verifier's two mbarrier wait forms (local, and acquire at cluster
 *            scope);
 *   which 1  the chunked verifier's counter poll in global memory (which also raises its
 *            abort flag);
 *   which 2  the tcgen05 GEMM's stage wait.
 * Each wait must give up; then MTPSPEC_STATUS_TIMEOUT is OR-ed into *status (device memory,
 * int32 [1], not cleared by the call).  1 <= limit <= 2^20.  The pages have no counterpart;
 * this entry point exists so that the timeout path can be tested without a fault.
 * Returns MTPSPEC_OK, MTPSPEC_ERR_ARG or MTPSPEC_ERR_CUDA. */
int mtpspec_selftest_wait_timeout(int which, uint32_t limit, int32_t *status, void *stream);

/* Diagnostics (no counterpart in the pages): the number of kernel launches this library
 * has enqueued, on any stream and device, since it was loaded.  Thread-safe. */
uint64_t mtpspec_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBMTPSPEC_H */
