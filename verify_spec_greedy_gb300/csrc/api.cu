// The C ABI of libmtpspec: argument validation and launches on the caller's stream.
// Declarations, argument meanings and sources are in include/libmtpspec.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/libmtpspec.h"
#include "kernels.h"

#define MTPSPEC_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int64_t kMaxV = 2147483647;  // ids are int32
constexpr int32_t kMaxD = 64;
constexpr int64_t kMaxRows = 2147483647 / (65 * 16);  // units x cluster CTAs fit a grid
constexpr int64_t kMaxH = 65536;
constexpr int64_t kMaxTokens = 1 << 20;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_size(int dtype) { return dtype == MTPSPEC_F32 ? 4 : 2; }

// Make the stream's device current for this library's runtime and check that it is an
// sm_103 part.  Called only after every host-side check has passed.  A stream that is
// being captured into a graph must not be asked for its device (the query invalidates
// the capture); the capturing thread's current device is used then.
int prepare_device(cudaStream_t stream) {
    int dev = -1;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (stream != nullptr && cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MTPSPEC_ERR_CUDA;
    if (stream != nullptr && cs == cudaStreamCaptureStatusNone) {
        if (cudaStreamGetDevice(stream, &dev) != cudaSuccess) return MTPSPEC_ERR_CUDA;
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess) return MTPSPEC_ERR_CUDA;
        if (cur != dev && cudaSetDevice(dev) != cudaSuccess) return MTPSPEC_ERR_CUDA;
    } else if (cudaGetDevice(&dev) != cudaSuccess) {
        return MTPSPEC_ERR_CUDA;
    }
    static std::mutex mu;
    static int checked[64] = {0};  // 0 unknown, 1 ok, -1 unsupported
    if (dev < 0 || dev >= 64) return MTPSPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (checked[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MTPSPEC_ERR_CUDA;
        checked[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return checked[dev] == 1 ? MTPSPEC_OK : MTPSPEC_ERR_UNSUPPORTED;
}

int launched(cudaError_t e) { return e == cudaSuccess ? MTPSPEC_OK : MTPSPEC_ERR_CUDA; }

}  // namespace

namespace mtpspec {
std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }
}  // namespace mtpspec

MTPSPEC_API int mtpspec_selftest_wait_timeout(int which, uint32_t limit, int32_t *status,
                                              void *stream) {
    if (which < 0 || which > 2) return MTPSPEC_ERR_ARG;
    if (limit < 1 || limit > (1u << 20)) return MTPSPEC_ERR_ARG;
    if (!status || !aligned(status, 4)) return MTPSPEC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    cudaError_t e = which == 0 ? mtpspec::run_wait_selftest_clusters(limit, status, s)
                    : which == 1 ? mtpspec::run_wait_selftest_chunks(limit, status, s)
                                 : mtpspec::run_wait_selftest_gemm(limit, status, s);
    return launched(e);
}

MTPSPEC_API uint64_t mtpspec_launch_count(void) {
    return static_cast<uint64_t>(mtpspec::g_launches.load());
}

MTPSPEC_API const char *mtpspec_status_string(int code) {
    switch (code) {
    case MTPSPEC_OK: return "MTPSPEC_OK";
    case MTPSPEC_ERR_ARG: return "MTPSPEC_ERR_ARG: invalid argument";
    case MTPSPEC_ERR_DTYPE: return "MTPSPEC_ERR_DTYPE: unsupported dtype";
    case MTPSPEC_ERR_SHAPE: return "MTPSPEC_ERR_SHAPE: size out of the supported range";
    case MTPSPEC_ERR_WORKSPACE: return "MTPSPEC_ERR_WORKSPACE: workspace missing or too small";
    case MTPSPEC_ERR_CUDA: return "MTPSPEC_ERR_CUDA: CUDA runtime or launch failure";
    case MTPSPEC_ERR_UNSUPPORTED: return "MTPSPEC_ERR_UNSUPPORTED: device is not sm_103";
    default: return "MTPSPEC: unknown status";
    }
}

MTPSPEC_API int mtp_greedy_draft(const void *logits, int dtype, int64_t M, int64_t V,
                                 int32_t *out_ids, void *stream) {
    if (dtype != MTPSPEC_F32 && dtype != MTPSPEC_BF16) return MTPSPEC_ERR_DTYPE;
    if (M < 0 || V < 1 || V > kMaxV || M > 2147483647 / 16) return MTPSPEC_ERR_SHAPE;
    if (M == 0) return MTPSPEC_OK;
    if (!logits || !out_ids) return MTPSPEC_ERR_ARG;
    if (!aligned(logits, elem_size(dtype)) || !aligned(out_ids, 4)) return MTPSPEC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    return launched(mtpspec::run_greedy_draft(logits, dtype, M, V, out_ids, s));
}

MTPSPEC_API int spec_verify_greedy(const void *target_logits, int dtype, const int32_t *draft_ids,
                                   int64_t B, int32_t D, int64_t V, int32_t *out_tokens,
                                   int32_t *num_accepted, int32_t *status, void *stream) {
    if (dtype != MTPSPEC_F32 && dtype != MTPSPEC_BF16) return MTPSPEC_ERR_DTYPE;
    if (B < 0 || D < 1 || D > kMaxD || V < 1 || V > kMaxV || B > 2147483647 / 16)
        return MTPSPEC_ERR_SHAPE;
    if (B == 0) return MTPSPEC_OK;
    if (!target_logits || !draft_ids || !out_tokens || !num_accepted) return MTPSPEC_ERR_ARG;
    if (!aligned(target_logits, elem_size(dtype)) || !aligned(draft_ids, 4) ||
        !aligned(out_tokens, 4) || !aligned(num_accepted, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    return launched(mtpspec::run_verify_greedy(target_logits, dtype, draft_ids, B, D, V, out_tokens,
                                               num_accepted, status, s));
}

MTPSPEC_API size_t spec_verify_workspace_bytes(int64_t B, int32_t D, int64_t V) {
    if (B <= 0 || D < 1 || D > kMaxD || V < 1 || V > kMaxV || B > kMaxRows) return 0;
    if (!mtpspec::verify_sample_fits(V, 2, true)) return 0;  // too large for any type and mode
    return mtpspec::verify_workspace_bytes(B, D, V);
}

MTPSPEC_API int spec_verify_sample(const void *target_logits, const void *draft_logits, int dtype,
                                   const int32_t *draft_ids, const float *temperature,
                                   const int32_t *top_k, const float *top_p, uint64_t seed,
                                   int64_t B, int32_t D, int64_t V, int32_t *out_tokens,
                                   int32_t *num_accepted, float *p_target, float *p_draft,
                                   void *workspace, size_t workspace_bytes, int32_t *status,
                                   void *stream) {
    if (dtype != MTPSPEC_F32 && dtype != MTPSPEC_BF16) return MTPSPEC_ERR_DTYPE;
    if (B < 0 || D < 1 || D > kMaxD || V < 1 || V > kMaxV || B > kMaxRows) return MTPSPEC_ERR_SHAPE;
    if (!mtpspec::verify_sample_fits(V, elem_size(dtype), draft_logits == nullptr))
        return MTPSPEC_ERR_SHAPE;
    if (B == 0) return MTPSPEC_OK;
    if (!target_logits || !draft_ids || !temperature || !out_tokens || !num_accepted)
        return MTPSPEC_ERR_ARG;
    const size_t es = elem_size(dtype);
    if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(draft_ids, 4) ||
        !aligned(temperature, 4) || !aligned(top_k, 4) || !aligned(top_p, 4) ||
        !aligned(out_tokens, 4) || !aligned(num_accepted, 4) || !aligned(p_target, 4) ||
        !aligned(p_draft, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    if (!workspace || !aligned(workspace, 16) ||
        workspace_bytes < mtpspec::verify_workspace_bytes(B, D, V))
        return MTPSPEC_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    mtpspec::VerifySampleArgs a;
    a.target = target_logits;
    a.draft = draft_logits;
    a.dtype = dtype;
    a.draft_ids = draft_ids;
    a.temperature = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.seed = seed;
    a.B = B;
    a.D = D;
    a.V = V;
    a.out_tokens = out_tokens;
    a.num_accepted = num_accepted;
    a.p_target = p_target;
    a.p_draft = p_draft;
    a.workspace = workspace;
    a.status = status;
    return launched(mtpspec::run_verify_sample(a, s));
}

MTPSPEC_API size_t mtp_draft_input_workspace_bytes(int64_t M, int64_t H) {
    if (M <= 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens) return 0;
    return mtpspec::draft_input_workspace_bytes(M, H);
}

MTPSPEC_API int mtp_draft_input(const void *emb_next, const void *hidden, const void *enorm_w,
                                const void *hnorm_w, const void *eh_proj_w, void *out, int64_t M,
                                int64_t H, float eps, void *workspace, size_t workspace_bytes,
                                void *stream) {
    if (M < 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens) return MTPSPEC_ERR_SHAPE;
    if (!(eps >= 0.0f)) return MTPSPEC_ERR_ARG;
    if (M == 0) return MTPSPEC_OK;
    if (!emb_next || !hidden || !enorm_w || !hnorm_w || !eh_proj_w || !out) return MTPSPEC_ERR_ARG;
    if (!aligned(emb_next, 16) || !aligned(hidden, 16) || !aligned(enorm_w, 16) ||
        !aligned(hnorm_w, 16) || !aligned(eh_proj_w, 16) || !aligned(out, 16))
        return MTPSPEC_ERR_ARG;
    const size_t need = mtpspec::draft_input_workspace_bytes(M, H);
    if (need > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes < need))
        return MTPSPEC_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    mtpspec::DraftInputArgs a;
    a.e = emb_next;
    a.h = hidden;
    a.we = enorm_w;
    a.wh = hnorm_w;
    a.W = eh_proj_w;
    a.y = out;
    a.M = M;
    a.H = H;
    a.eps = eps;
    a.workspace = workspace;
    return launched(mtpspec::run_draft_input(a, s));
}

constexpr int64_t kMaxLmHeadV = 65535LL * 128;  // ids stay well inside int32 tile arithmetic

MTPSPEC_API size_t mtp_lm_head_greedy_workspace_bytes(int64_t M, int64_t H, int64_t V) {
    if (M <= 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens || V < 1 || V > kMaxLmHeadV)
        return 0;
    return mtpspec::lm_head_workspace_bytes(M, H, V);
}

MTPSPEC_API int mtp_lm_head_greedy(const void *hidden, const void *norm_w, float eps,
                                   const void *lm_head_w, int64_t M, int64_t H, int64_t V,
                                   int32_t *out_ids, float *out_logit, void *workspace,
                                   size_t workspace_bytes, int32_t *status, void *stream) {
    if (M < 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens || V < 1 || V > kMaxLmHeadV)
        return MTPSPEC_ERR_SHAPE;
    if (!(eps >= 0.0f)) return MTPSPEC_ERR_ARG;
    if (M == 0) return MTPSPEC_OK;
    if (!hidden || !lm_head_w || !out_ids) return MTPSPEC_ERR_ARG;
    if (!aligned(hidden, 16) || !aligned(norm_w, 16) || !aligned(lm_head_w, 16) ||
        !aligned(out_ids, 4) || !aligned(out_logit, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < mtpspec::lm_head_workspace_bytes(M, H, V))
        return MTPSPEC_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    mtpspec::LmHeadArgs a;
    a.hidden = hidden;
    a.norm_w = norm_w;
    a.eps = eps;
    a.W = lm_head_w;
    a.M = M;
    a.H = H;
    a.V = V;
    a.ids = out_ids;
    a.ids_stride = 1;
    a.logit = out_logit;
    a.k = 1;
    a.workspace = workspace;
    a.status = status;
    return launched(mtpspec::run_lm_head_greedy(a, s));
}

MTPSPEC_API size_t mtp_draft_steps_workspace_bytes(int64_t M, int64_t H, int64_t V) {
    if (M <= 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens || V < 1 || V > kMaxLmHeadV)
        return 0;
    return mtpspec::draft_steps_workspace_bytes(M, H, V);
}

MTPSPEC_API int mtp_draft_steps(const void *embed_w, const int32_t *next_ids, const int32_t *positions,
                                const void *hidden, const void *enorm_w, const void *hnorm_w,
                                const void *eh_proj_w, const void *norm_w, const void *lm_head_w,
                                float eps, int64_t M, int64_t H, int64_t V, int32_t D,
                                int32_t *draft_ids, void *hidden_out, void *workspace,
                                size_t workspace_bytes, int32_t *status, void *stream) {
    if (M < 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens || V < 1 || V > kMaxLmHeadV ||
        D < 1 || D > kMaxD)
        return MTPSPEC_ERR_SHAPE;
    if (!(eps >= 0.0f)) return MTPSPEC_ERR_ARG;
    if (M == 0) return MTPSPEC_OK;
    if (!embed_w || !next_ids || !hidden || !enorm_w || !hnorm_w || !eh_proj_w || !lm_head_w ||
        !draft_ids)
        return MTPSPEC_ERR_ARG;
    if (!aligned(embed_w, 16) || !aligned(hidden, 16) || !aligned(enorm_w, 16) ||
        !aligned(hnorm_w, 16) || !aligned(eh_proj_w, 16) || !aligned(norm_w, 16) ||
        !aligned(lm_head_w, 16) || !aligned(hidden_out, 16) || !aligned(next_ids, 4) ||
        !aligned(positions, 4) || !aligned(draft_ids, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < mtpspec::draft_steps_workspace_bytes(M, H, V))
        return MTPSPEC_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    mtpspec::DraftStepsArgs a;
    a.embed = embed_w;
    a.next_ids = next_ids;
    a.positions = positions;
    a.hidden = hidden;
    a.enorm_w = enorm_w;
    a.hnorm_w = hnorm_w;
    a.eh_proj_w = eh_proj_w;
    a.norm_w = norm_w;
    a.lm_head_w = lm_head_w;
    a.eps = eps;
    a.M = M;
    a.H = H;
    a.V = V;
    a.D = D;
    a.draft_ids = draft_ids;
    a.hidden_out = hidden_out;
    a.workspace = workspace;
    a.status = status;
    return launched(mtpspec::run_draft_steps(a, s));
}

MTPSPEC_API size_t mtp_lm_head_topk_workspace_bytes(int64_t M, int64_t H, int64_t V) {
    if (M <= 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens || V < 1 || V > kMaxLmHeadV)
        return 0;
    return mtpspec::lm_head_workspace_bytes(M, H, V, mtpspec::kLmHeadTopK);
}

MTPSPEC_API int mtp_lm_head_topk(const void *hidden, const void *norm_w, float eps,
                                 const void *lm_head_w, int64_t M, int64_t H, int64_t V, int32_t k,
                                 int32_t *out_ids, float *out_logits, void *workspace,
                                 size_t workspace_bytes, int32_t *status, void *stream) {
    if (M < 0 || H < 8 || H > kMaxH || (H % 8) != 0 || M > kMaxTokens || V < 1 || V > kMaxLmHeadV)
        return MTPSPEC_ERR_SHAPE;
    if (k < 1 || k > mtpspec::kLmHeadTopK || k > V) return MTPSPEC_ERR_SHAPE;
    if (!(eps >= 0.0f)) return MTPSPEC_ERR_ARG;
    if (M == 0) return MTPSPEC_OK;
    if (!hidden || !lm_head_w || !out_ids) return MTPSPEC_ERR_ARG;
    if (!aligned(hidden, 16) || !aligned(norm_w, 16) || !aligned(lm_head_w, 16) ||
        !aligned(out_ids, 4) || !aligned(out_logits, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < mtpspec::lm_head_workspace_bytes(M, H, V, mtpspec::kLmHeadTopK))
        return MTPSPEC_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    mtpspec::LmHeadArgs a;
    a.hidden = hidden;
    a.norm_w = norm_w;
    a.eps = eps;
    a.W = lm_head_w;
    a.M = M;
    a.H = H;
    a.V = V;
    a.ids = out_ids;
    a.ids_stride = k;
    a.logit = out_logits;
    a.k = k;  // k = 1 is the greedy pick, with the same layout of ids and logits
    a.workspace = workspace;
    a.status = status;
    return launched(mtpspec::run_lm_head_greedy(a, s));
}

constexpr int64_t kMaxStateRows = 1LL << 24;

MTPSPEC_API int mtp_state_snapshot(const void *state, void *backup, int64_t B, int64_t row_bytes,
                                   void *stream) {
    if (B < 0 || B > kMaxStateRows || row_bytes < 0 || (row_bytes % 16) != 0) return MTPSPEC_ERR_SHAPE;
    if (B == 0 || row_bytes == 0) return MTPSPEC_OK;
    if (!state || !backup || !aligned(state, 16) || !aligned(backup, 16)) return MTPSPEC_ERR_ARG;
    const char *s0 = static_cast<const char *>(state), *b0 = static_cast<const char *>(backup);
    const int64_t n = B * row_bytes;
    if (s0 < b0 + n && b0 < s0 + n) return MTPSPEC_ERR_ARG;  // overlapping
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    return launched(mtpspec::run_state_snapshot(state, backup, B, row_bytes, s));
}

MTPSPEC_API int mtp_state_fixup(const int32_t *num_accepted, int32_t D, const int32_t *kv_len_before,
                                int32_t *kv_len, void *state, const void *backup, int64_t B,
                                int64_t row_bytes, int32_t *draft_kv_len, int32_t *recompute,
                                int32_t *status, void *stream) {
    if (B < 0 || B > kMaxStateRows || D < 1 || D > kMaxD || row_bytes < 0 || (row_bytes % 16) != 0)
        return MTPSPEC_ERR_SHAPE;
    if (B == 0) return MTPSPEC_OK;
    if (!num_accepted || !kv_len_before || !kv_len) return MTPSPEC_ERR_ARG;
    if (!aligned(num_accepted, 4) || !aligned(kv_len_before, 4) || !aligned(kv_len, 4) ||
        !aligned(draft_kv_len, 4) || !aligned(recompute, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    if (row_bytes > 0) {
        if (!state || !backup || !aligned(state, 16) || !aligned(backup, 16)) return MTPSPEC_ERR_ARG;
        const char *s0 = static_cast<const char *>(state), *b0 = static_cast<const char *>(backup);
        const int64_t n = B * row_bytes;
        if (s0 < b0 + n && b0 < s0 + n) return MTPSPEC_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    return launched(mtpspec::run_state_fixup(num_accepted, D, kv_len_before, kv_len, state, backup,
                                             B, row_bytes, draft_kv_len, recompute, status, s));
}

MTPSPEC_API int spec_verify_sample_static(const void *target_logits, const void *draft_logits,
                                          int dtype, const int32_t *draft_ids,
                                          const float *temperature, const int32_t *top_k,
                                          const float *top_p, uint64_t seed, int64_t B, int32_t D,
                                          int64_t V, int32_t *out_tokens, int32_t *num_accepted,
                                          float *p_target, float *p_draft, int32_t *status,
                                          void *stream) {
    if (dtype != MTPSPEC_F32 && dtype != MTPSPEC_BF16) return MTPSPEC_ERR_DTYPE;
    if (B < 0 || D < 1 || D > kMaxD || V < 1 || V > kMaxV || B > kMaxRows) return MTPSPEC_ERR_SHAPE;
    if (B * (D + 1) > mtpspec::kStaticVerifyUnits) return MTPSPEC_ERR_SHAPE;
    if (!mtpspec::verify_fits(V, elem_size(dtype), draft_logits == nullptr)) return MTPSPEC_ERR_SHAPE;
    if (B == 0) return MTPSPEC_OK;
    if (!target_logits || !draft_ids || !temperature || !out_tokens || !num_accepted)
        return MTPSPEC_ERR_ARG;
    const size_t es = elem_size(dtype);
    if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(draft_ids, 4) ||
        !aligned(temperature, 4) || !aligned(top_k, 4) || !aligned(top_p, 4) ||
        !aligned(out_tokens, 4) || !aligned(num_accepted, 4) || !aligned(p_target, 4) ||
        !aligned(p_draft, 4) || !aligned(status, 4))
        return MTPSPEC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = prepare_device(s);
    if (rc != MTPSPEC_OK) return rc;
    mtpspec::VerifySampleArgs a;
    a.target = target_logits;
    a.draft = draft_logits;
    a.dtype = dtype;
    a.draft_ids = draft_ids;
    a.temperature = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.seed = seed;
    a.B = B;
    a.D = D;
    a.V = V;
    a.out_tokens = out_tokens;
    a.num_accepted = num_accepted;
    a.p_target = p_target;
    a.p_draft = p_draft;
    a.workspace = nullptr;
    a.status = status;
    return launched(mtpspec::run_verify_sample_static(a, s));
}
