// Host-side launchers of libmtpspec's kernels (called by the C-ABI entry points in
// api.cu after argument validation).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace mtpspec {

// Adds n to the library's count of kernel launches (read by mtpspec_launch_count).
void count_launches(int n);

// Function attributes persist, so each is set once per device (and the shared-memory
// limit again only when a larger one is asked for): launches recorded by a stream
// capture then make no attribute call.
// Host threads that miss the cache set the attribute one at a time, so the value set on
// the device only grows and the cache never claims more than the device holds.
struct AttrCache {
    std::atomic<int> v[64];
    std::mutex mu;
};
template <typename F>
cudaError_t ensure_attr(F kernel, cudaFuncAttribute attr, int value, AttrCache &c) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (c.v[dev].load(std::memory_order_acquire) >= value) return cudaSuccess;
    std::lock_guard<std::mutex> lock(c.mu);
    if (c.v[dev].load(std::memory_order_relaxed) >= value) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, attr, value);
    if (e == cudaSuccess) c.v[dev].store(value, std::memory_order_release);
    return e;
}

cudaError_t run_greedy_draft(const void *logits, int dtype, int64_t M, int64_t V, int32_t *ids,
                             cudaStream_t stream);

cudaError_t run_verify_greedy(const void *target, int dtype, const int32_t *d, int64_t B,
                              int32_t D, int64_t V, int32_t *tokens, int32_t *num_accepted,
                              int32_t *status, cudaStream_t stream);

}  // namespace mtpspec

namespace mtpspec {

// Per-unit record handed from the unit kernels of spec_verify_sample to its finalize
// kernel: one per (row, position).
struct VerifyUnitRecord {
    int32_t flags;  // bit 0: draft accepted
    int32_t token;  // greedy pick, or the draw (residual / bonus) of this unit, or -1
    float pt;       // p_j(d_j)
    float pd;       // q_j(d_j)
};

struct VerifySampleArgs {
    const void *target;
    const void *draft;
    int dtype;
    const int32_t *draft_ids;
    const float *temperature;
    const int32_t *top_k;
    const float *top_p;
    uint64_t seed;
    int64_t B;
    int32_t D;
    int64_t V;
    int32_t *out_tokens;
    int32_t *num_accepted;
    float *p_target;
    float *p_draft;
    void *workspace;
    int32_t *status;
};

// Greedy rows of a sampling verification (temperature 0, or a bad sampling parameter):
// the argmax of each of their positions, written as unit records.  Rows that sample
// return at once.  Launched as a programmatic dependent of the sampling kernel, so the
// two run concurrently.
cudaError_t run_verify_greedy_rows(const VerifySampleArgs &a, cudaStream_t stream);

// Bytes of workspace a sampling verification of these sizes needs, whichever verifier
// run_verify_sample picks for any logit type and mode.
size_t verify_workspace_bytes(int64_t B, int32_t D, int64_t V);

// Whether one cluster's shared memory can hold a row of V logits of this element size.
bool verify_fits(int64_t V, size_t elem_bytes, bool one_hot);
// Whether either verifier takes V (the cluster kernel, else the chunked one).
bool verify_sample_fits(int64_t V, size_t elem_bytes, bool one_hot);

cudaError_t run_verify_sample(const VerifySampleArgs &a, cudaStream_t stream);

// The per-row finalize over the unit records rec [B, D + 1] (verify_sample.cu).
cudaError_t launch_verify_finalize(const VerifyUnitRecord *rec, const VerifySampleArgs &a,
                                   cudaStream_t stream);

// The chunked verifier (verify_chunked.cu): units cut into vocabulary chunks, several CTAs
// per SM, chunks of a unit coordinated through the workspace.
size_t verify_chunks_workspace_bytes(int64_t B, int32_t D, int64_t V);
bool verify_chunks_fits(int64_t V, size_t elem_bytes);
cudaError_t run_verify_chunks(const VerifySampleArgs &a, cudaStream_t stream);

// Diagnostics of the bounded waits (one CTA each): the cluster verifier's two wait forms,
// the chunked verifier's counter poll and the GEMM's stage wait, each on a barrier or counter
// that nothing completes, with `limit` polls.
cudaError_t run_wait_selftest_clusters(uint32_t limit, int32_t *status, cudaStream_t stream);
cudaError_t run_wait_selftest_chunks(uint32_t limit, int32_t *status, cudaStream_t stream);
cudaError_t run_wait_selftest_gemm(uint32_t limit, int32_t *status, cudaStream_t stream);

// The fixed-scratch variant: per-unit records in the library's static device array
// (a.workspace is ignored).  Units B * (D + 1) must not exceed kStaticVerifyUnits.
constexpr int64_t kStaticVerifyUnits = 65536;
cudaError_t run_verify_sample_static(VerifySampleArgs a, cudaStream_t stream);

}  // namespace mtpspec

namespace mtpspec {

struct DraftInputArgs {
    const void *e, *h, *we, *wh, *W;
    void *y;
    int64_t M, H;
    float eps;
    void *workspace;
};

// Whether (M, H) takes the fused norm + GEMV path (no workspace).
bool draft_input_uses_gemv(int64_t M, int64_t H);
size_t draft_input_workspace_bytes(int64_t M, int64_t H);
cudaError_t run_draft_input(const DraftInputArgs &a, cudaStream_t stream);

// Tensor-core GEMM Y[Mt, H] = B[Mt, K] @ A[H, K]^T (bf16, fp32 accumulate, K = 2H) and its
// workspace (a flag word, then split-K partial sums).  The first gemm_zero_bytes(Mt, H)
// bytes of the workspace must be zeroed before the launch; with pdl the GEMM starts as the
// programmatic dependent of the kernel launched just before it on the stream (its weight
// loads overlap that kernel) and reads B only once that kernel has completed.
size_t gemm_workspace_bytes(int64_t Mt, int64_t H);
size_t gemm_zero_bytes(int64_t Mt, int64_t H);
cudaError_t run_gemm_bf16_nt(const void *A, const void *B, void *Y, int64_t H, int64_t Mt,
                             int64_t K, void *workspace, bool pdl, cudaStream_t stream);

}  // namespace mtpspec

namespace mtpspec {

// The draft head's output layer with the greedy pick (lm_head.cu).
struct LmHeadArgs {
    const void *hidden;   // bf16 [M, H]
    const void *norm_w;   // bf16 [H] or nullptr
    float eps;
    const void *W;        // bf16 [V, H]
    int64_t M, H, V;
    int32_t *ids;         // ids[t * ids_stride], or [M, k] for the top k
    int64_t ids_stride;
    float *logit;         // [M] (or [M, k]) or nullptr
    int32_t k;            // 1: the greedy pick; 2 .. kLmHeadTopK: the k largest
    void *workspace;
    int32_t *status;      // or nullptr
};
size_t lm_head_workspace_bytes(int64_t M, int64_t H, int64_t V, int32_t k = 1);
constexpr int kLmHeadTopK = 8;  // the largest k of the top-k output
cudaError_t run_lm_head_greedy(const LmHeadArgs &a, cudaStream_t stream);

// Pieces it is made of: the RMSNorm of each token's hidden state (draft_input.cu) and the
// tcgen05 GEMM with the argmax epilogue (tcgen05_gemm.cu), which leaves one key
// (order key << 32 | ~id) per (token, 256-id block of the vocabulary) in keys [Mt, o_tiles].
cudaError_t run_head_norm(const void *x, const void *w, void *out, int64_t M, int64_t H, float eps,
                          cudaStream_t stream);
int lm_head_o_tiles(int64_t V);
cudaError_t run_gemm_argmax(const void *W, const void *X, int64_t V, int64_t Mt, int64_t K,
                            unsigned long long *keys, unsigned *err, int topk, cudaStream_t stream);

}  // namespace mtpspec

namespace mtpspec {

// The model state around a verification (state.cu).
cudaError_t run_state_snapshot(const void *state, void *backup, int64_t B, int64_t row_bytes,
                               cudaStream_t stream);
cudaError_t run_state_fixup(const int32_t *num_accepted, int32_t D, const int32_t *kv_before,
                            int32_t *kv_len, void *state, const void *backup, int64_t B,
                            int64_t row_bytes, int32_t *draft_kv_len, int32_t *recompute,
                            int32_t *status, cudaStream_t stream);

}  // namespace mtpspec

namespace mtpspec {

// Serial greedy draft steps (draft_steps.cu).
struct DraftStepsArgs {
    const void *embed;       // bf16 [V, H]
    const int32_t *next_ids; // [M]
    const int32_t *positions;  // [M] or nullptr
    const void *hidden;      // bf16 [M, H]
    const void *enorm_w, *hnorm_w, *eh_proj_w;  // bf16 [H], [H], [H, 2H]
    const void *norm_w;      // bf16 [H] or nullptr
    const void *lm_head_w;   // bf16 [V, H]
    float eps;
    int64_t M, H, V;
    int32_t D;
    int32_t *draft_ids;      // [M, D]
    void *hidden_out;        // bf16 [D, M, H] or nullptr
    void *workspace;
    int32_t *status;
};
size_t draft_steps_workspace_bytes(int64_t M, int64_t H, int64_t V);
cudaError_t run_draft_steps(const DraftStepsArgs &a, cudaStream_t stream);

}  // namespace mtpspec
