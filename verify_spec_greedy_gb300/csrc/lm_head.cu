// The draft head's output layer with the greedy pick: ids[t] = argmax_v (W x_t)_v, the
// lowest id among equal maxima, without writing the [M, V] logits ("14. MTP: speculative
// decoding with the built-in draft head", "The draft head": a normalisation and the output
// layer shared with the main model give the draft logits, and the draft is their argmax;
// "MPT (MTP, Multi-Token Prediction) 原理详解" 二.1 shared_head, 三 stage 1 compute_logits
// and greedy sample; "The decoding loop and MTP", "Why a hand-written decoding loop": the
// lower id wins a tie).
//
// Three launches: the optional RMSNorm of the hidden states into the workspace (bf16, as
// the input stage rounds its activations), the tcgen05 GEMM whose epilogue reduces each
// token's row of a 128-token x 256-id logit tile to one key (order key of the largest logit
// << 32 | ~its lowest id), and the pick below, which takes the largest key of each token
// over the V / 256 tiles.  A larger key is a larger logit, or the same logit at a lower id.
#include "common.cuh"
#include "kernels.h"
#include "../../include/libmtpspec.h"

namespace mtpspec {
namespace lh {

constexpr int PICK_THREADS = 256;

// One warp per token: the largest of its o_tiles keys.
__global__ void __launch_bounds__(PICK_THREADS)
k_lm_head_pick(const unsigned long long *__restrict__ keys, int o_tiles, int64_t M,
               int32_t *__restrict__ ids, int64_t ids_stride, float *__restrict__ logit) {
    pdl_wait_primary();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (PICK_THREADS / 32) + (threadIdx.x >> 5);
    if (t >= M) return;
    const unsigned long long *kr = keys + t * o_tiles;
    unsigned long long best = 0;
    for (int i = lane; i < o_tiles; i += 32) best = max(best, kr[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    if (lane == 0) {
        ids[t * ids_stride] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best));
        if (logit) logit[t] = key_to_float(static_cast<uint32_t>(best >> 32));
    }
}

// One warp per token: the k largest of its o_tiles x TOPK keys.  Each lane keeps the TOPK
// largest of the keys it reads (sorted); then k rounds take the warp's largest head and
// pop it from its lane (keys are distinct: each carries its id).
template <int TOPK>
__global__ void __launch_bounds__(PICK_THREADS)
k_lm_head_pick_topk(const unsigned long long *__restrict__ keys, int o_tiles, int64_t M, int k,
                    int32_t *__restrict__ ids, float *__restrict__ logit) {
    pdl_wait_primary();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (PICK_THREADS / 32) + (threadIdx.x >> 5);
    if (t >= M) return;
    const unsigned long long *kr = keys + t * o_tiles * TOPK;
    const int n = o_tiles * TOPK;
    unsigned long long lst[TOPK];
#pragma unroll
    for (int i = 0; i < TOPK; ++i) lst[i] = 0ull;
    for (int i = lane; i < n; i += 32) {
        const unsigned long long key = kr[i];
        if (key > lst[TOPK - 1]) {
            lst[TOPK - 1] = key;
#pragma unroll
            for (int q = TOPK - 1; q > 0; --q) {
                if (lst[q] > lst[q - 1]) {
                    const unsigned long long tmp = lst[q];
                    lst[q] = lst[q - 1];
                    lst[q - 1] = tmp;
                }
            }
        }
    }
    for (int r = 0; r < k; ++r) {
        unsigned long long m = lst[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const unsigned own = __ballot_sync(0xFFFFFFFFu, m != 0ull && lst[0] == m);
        if (own && lane == __ffs(own) - 1) {
#pragma unroll
            for (int q = 0; q + 1 < TOPK; ++q) lst[q] = lst[q + 1];
            lst[TOPK - 1] = 0ull;
        }
        if (lane == 0) {
            ids[t * k + r] = m ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(m)) : -1;
            if (logit) logit[t * k + r] = key_to_float(static_cast<uint32_t>(m >> 32));
        }
    }
}

}  // namespace lh

// Workspace: a flag word (256 bytes), the normalised hidden states when a norm weight is
// given (M x H bf16, counted always), then the keys [M, o_tiles] (x kLmHeadTopK for a top
// k).
static size_t lm_head_xn_bytes(int64_t M, int64_t H) {
    return (static_cast<size_t>(M) * static_cast<size_t>(H) * 2 + 1023) & ~static_cast<size_t>(1023);
}

size_t lm_head_workspace_bytes(int64_t M, int64_t H, int64_t V, int32_t k) {
    const size_t per = k > 1 ? kLmHeadTopK : 1;  // keys per (token, tile)
    return 256 + lm_head_xn_bytes(M, H) + static_cast<size_t>(M) * lm_head_o_tiles(V) * per * 8;
}

cudaError_t run_lm_head_greedy(const LmHeadArgs &a, cudaStream_t stream) {
    unsigned char *ws = static_cast<unsigned char *>(a.workspace);
    unsigned *flag = a.status ? reinterpret_cast<unsigned *>(a.status) : reinterpret_cast<unsigned *>(ws);
    uint16_t *xn = reinterpret_cast<uint16_t *>(ws + 256);
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(ws + 256 + lm_head_xn_bytes(a.M, a.H));
    const void *X = a.hidden;
    cudaError_t e;
    if (a.norm_w) {
        e = run_head_norm(a.hidden, a.norm_w, xn, a.M, a.H, a.eps, stream);
        if (e != cudaSuccess) return e;
        X = xn;
    }
    e = run_gemm_argmax(a.W, X, a.V, a.M, a.H, keys, flag, a.k > 1 ? kLmHeadTopK : 1, stream);
    if (e != cudaSuccess) return e;
    const int o_tiles = lm_head_o_tiles(a.V);
    const int per = lh::PICK_THREADS / 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.M + per - 1) / per), 1, 1);
    cfg.blockDim = dim3(lh::PICK_THREADS, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.k > 1)
        e = cudaLaunchKernelEx(&cfg, lh::k_lm_head_pick_topk<kLmHeadTopK>,
                               static_cast<const unsigned long long *>(keys), o_tiles, a.M,
                               static_cast<int>(a.k), a.ids, a.logit);
    else
        e = cudaLaunchKernelEx(&cfg, lh::k_lm_head_pick, static_cast<const unsigned long long *>(keys),
                               o_tiles, a.M, a.ids, a.ids_stride, a.logit);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace mtpspec
