// D serial greedy draft steps of the draft head ("MPT (MTP, Multi-Token Prediction) 原理详解"
// 三 stages 1-2: the bonus token and the main model's hidden state start the chain; each
// step embeds the previous token, runs the head and greedy-samples the next draft, then
// passes the token and the head's hidden state to the next step; 二.2 step 1: the input
// embedding at position 0 is zeroed; "14. MTP: speculative decoding with the built-in draft
// head", "The draft head").  The head's decoder block is not part of this library: a step
// passes the input stage's output straight to the final norm and the output layer.
//
// Per step: k_embed_rows (the table rows of the previous ids, zero rows where the position
// is 0 or the id is outside the vocabulary), the input stage (run_draft_input: fused GEMV
// for up to 4 tokens, else RMSNorm + tcgen05 GEMM) and the output layer with the greedy pick
// (run_lm_head_greedy), which writes column k of draft_ids; the next step reads that column
// and this step's hidden state.  Nothing is allocated and nothing waits on the host, so the
// whole call can be captured into one CUDA graph.
#include "common.cuh"
#include "kernels.h"
#include "../../include/libmtpspec.h"

namespace mtpspec {
namespace ds {

constexpr int EMB_THREADS = 128;

// out[t] = embed[ids[t * stride]], or zeros where positions[t] + step == 0 or the id is
// outside [0, V) (which also sets MTPSPEC_STATUS_BAD_DRAFT_ID).  One CTA per token.
__global__ void __launch_bounds__(EMB_THREADS)
k_embed_rows(const uint4 *__restrict__ embed, const int32_t *ids, int64_t stride,
             const int32_t *__restrict__ positions, int step, uint4 *__restrict__ out, int64_t H8,
             int64_t V, int32_t *status) {
    const int64_t t = blockIdx.x;
    const int32_t id = ids[t * stride];
    const bool bad = id < 0 || id >= V;
    const bool zero = bad || (positions && static_cast<int64_t>(positions[t]) + step == 0);
    if (bad && threadIdx.x == 0 && status) atomicOr(status, MTPSPEC_STATUS_BAD_DRAFT_ID);
    const uint4 *src = embed + static_cast<int64_t>(zero ? 0 : id) * H8;
    for (int64_t i = threadIdx.x; i < H8; i += EMB_THREADS)
        out[t * H8 + i] = zero ? make_uint4(0u, 0u, 0u, 0u) : src[i];
}

}  // namespace ds

// Workspace: the embedded rows [M, H], two hidden-state buffers [M, H] (used when the
// caller does not keep every step's), then the input stage's and the output layer's own.
static size_t ds_mh(int64_t M, int64_t H) {
    return (static_cast<size_t>(M) * static_cast<size_t>(H) * 2 + 1023) & ~static_cast<size_t>(1023);
}
static size_t ds_di(int64_t M, int64_t H) {
    return (draft_input_workspace_bytes(M, H) + 1023) & ~static_cast<size_t>(1023);
}

size_t draft_steps_workspace_bytes(int64_t M, int64_t H, int64_t V) {
    return 3 * ds_mh(M, H) + ds_di(M, H) + lm_head_workspace_bytes(M, H, V);
}

cudaError_t run_draft_steps(const DraftStepsArgs &a, cudaStream_t stream) {
    unsigned char *ws = static_cast<unsigned char *>(a.workspace);
    const size_t mh = ds_mh(a.M, a.H);
    uint16_t *e = reinterpret_cast<uint16_t *>(ws);
    uint16_t *ping[2] = {reinterpret_cast<uint16_t *>(ws + mh), reinterpret_cast<uint16_t *>(ws + 2 * mh)};
    void *di_ws = ws + 3 * mh;
    void *lm_ws = ws + 3 * mh + ds_di(a.M, a.H);
    const int32_t *ids_in = a.next_ids;
    int64_t ids_stride = 1;
    const void *h_in = a.hidden;
    for (int32_t k = 0; k < a.D; ++k) {
        ds::k_embed_rows<<<static_cast<unsigned>(a.M), ds::EMB_THREADS, 0, stream>>>(
            static_cast<const uint4 *>(a.embed), ids_in, ids_stride, a.positions, k,
            reinterpret_cast<uint4 *>(e), a.H / 8, a.V, a.status);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        count_launches(1);
        uint16_t *y = a.hidden_out
                          ? static_cast<uint16_t *>(a.hidden_out) + static_cast<int64_t>(k) * a.M * a.H
                          : ping[k & 1];
        DraftInputArgs di;
        di.e = e;
        di.h = h_in;
        di.we = a.enorm_w;
        di.wh = a.hnorm_w;
        di.W = a.eh_proj_w;
        di.y = y;
        di.M = a.M;
        di.H = a.H;
        di.eps = a.eps;
        di.workspace = di_ws;
        err = run_draft_input(di, stream);
        if (err != cudaSuccess) return err;
        LmHeadArgs lh;
        lh.hidden = y;
        lh.norm_w = a.norm_w;
        lh.eps = a.eps;
        lh.W = a.lm_head_w;
        lh.M = a.M;
        lh.H = a.H;
        lh.V = a.V;
        lh.ids = a.draft_ids + k;
        lh.ids_stride = a.D;
        lh.logit = nullptr;
        lh.k = 1;
        lh.workspace = lm_ws;
        lh.status = a.status;
        err = run_lm_head_greedy(lh, stream);
        if (err != cudaSuccess) return err;
        ids_in = a.draft_ids + k;
        ids_stride = a.D;
        h_in = y;
    }
    return cudaSuccess;
}

}  // namespace mtpspec
