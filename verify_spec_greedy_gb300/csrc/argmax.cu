// Greedy drafting and greedy verification: row argmax with the lowest-id tie rule.
//
// Greedy draft ("14. MTP: speculative decoding with the built-in draft head", "The
// speculative decoding loop (greedy version)": the draft is the argmax of the draft
// head's logits) and greedy verification (same section: keep a draft while it equals the
// main model's own argmax, then take the main model's token; "MPT (MTP, Multi-Token
// Prediction) 原理详解" section 三 stages 3-4).  Ties go to the lower id ("The decoding
// loop and MTP", "Why a hand-written decoding loop").
//
// Layout: one thread-block cluster per group of P consecutive logit rows (P = 1 for a
// greedy draft, P = D + 1 for the positions of one verified row).  The C CTAs of the
// cluster split each row's V logits into C contiguous slices and stream them once with
// 16-byte loads; the per-CTA winners meet in CTA 0 through distributed shared memory,
// which writes the ids (draft) or the accepted prefix and tokens (verify).  Reading the
// logits once is the whole cost: the kernel is HBM-bound.
#include "common.cuh"
#include "kernels.h"

namespace mtpspec {

constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxUnroll = 4;
constexpr int kMaxPositions = 65;  // D + 1 with D <= 64

// Argmax of row[lo, hi) over this CTA; every thread returns its partial winner.
template <typename T>
__device__ __forceinline__ ArgMax thread_scan(const T *__restrict__ row, int64_t lo, int64_t hi) {
    constexpr int EPV = elems_per_16B<T>::value;
    ArgMax best{-INFINITY, -1};
    if (hi <= lo) return best;
    const uintptr_t base = reinterpret_cast<uintptr_t>(row + lo);
    int64_t head = static_cast<int64_t>(((16u - (base & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    for (int64_t i = threadIdx.x; i < head; i += blockDim.x) {
        float v = widen(row[lo + i]);
        if (v > best.v || best.i < 0) best = {v, static_cast<int32_t>(lo + i)};
    }
    const int64_t a_lo = lo + head;
    const int64_t nvec = (hi - a_lo) / EPV;
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + a_lo);
    const int64_t stride = static_cast<int64_t>(blockDim.x) * kArgmaxUnroll;
    for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += stride) {
        uint4 raw[kArgmaxUnroll];
#pragma unroll
        for (int u = 0; u < kArgmaxUnroll; ++u) {
            int64_t vi = v0 + static_cast<int64_t>(u) * blockDim.x;
            if (vi < nvec) raw[u] = ld_stream_16B(vp + vi);
        }
#pragma unroll
        for (int u = 0; u < kArgmaxUnroll; ++u) {
            int64_t vi = v0 + static_cast<int64_t>(u) * blockDim.x;
            if (vi < nvec) {
                float f[EPV];
                unpack(raw[u], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (f[e] > best.v || best.i < 0)
                        best = {f[e], static_cast<int32_t>(a_lo + vi * EPV + e)};
                }
            }
        }
    }
    for (int64_t i = a_lo + nvec * EPV + threadIdx.x; i < hi; i += blockDim.x) {
        float v = widen(row[i]);
        if (v > best.v || best.i < 0) best = {v, static_cast<int32_t>(i)};
    }
    return best;
}

// mode 0: greedy draft, out_a[row] = argmax.  mode 1: greedy verify of one row per
// group (P = D + 1), out_a = tokens [B, D+1], out_b = num_accepted [B].
template <typename T>
__global__ void __launch_bounds__(kArgmaxThreads)
k_argmax_groups(const T *__restrict__ logits, int64_t V, int P, int mode,
                const int32_t *__restrict__ draft_ids, int32_t *__restrict__ out_a,
                int32_t *__restrict__ out_b, int32_t *__restrict__ status) {
    __shared__ float red_v[kMaxPositions];
    __shared__ int32_t red_i[kMaxPositions];
    __shared__ float warp_v[kArgmaxThreads / 32];
    __shared__ int32_t warp_i[kArgmaxThreads / 32];
    __shared__ int32_t winners[kMaxPositions];

    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int64_t group = cluster_index();
    // slices are multiples of 16 elements, so interior slice starts keep the row's alignment
    int64_t chunk = (V + C - 1) / C;
    chunk = (chunk + 15) & ~static_cast<int64_t>(15);
    const int64_t lo = min(V, static_cast<int64_t>(rank) * chunk);
    const int64_t hi = min(V, lo + chunk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    for (int p = 0; p < P; ++p) {
        const T *row = logits + (group * P + p) * V;
        ArgMax a = warp_argmax(thread_scan(row, lo, hi));
        if (lane == 0) {
            warp_v[warp] = a.v;
            warp_i[warp] = a.i;
        }
        __syncthreads();
        if (warp == 0) {
            ArgMax b{-INFINITY, -1};
            if (lane < kArgmaxThreads / 32) b = {warp_v[lane], warp_i[lane]};
            b = warp_argmax(b);
            if (lane == 0) {
                red_v[p] = b.v;
                red_i[p] = b.i;
            }
        }
        __syncthreads();
    }
    cluster_sync();

    if (rank == 0) {
        for (int p = threadIdx.x; p < P; p += blockDim.x) {
            ArgMax best{-INFINITY, -1};
            for (uint32_t r = 0; r < C; ++r) {
                ArgMax o;
                o.v = ld_peer_f32(peer_addr(smem_addr(&red_v[p]), r));
                o.i = ld_peer_s32(peer_addr(smem_addr(&red_i[p]), r));
                best = argmax_merge(best, o);
            }
            winners[p] = best.i < 0 ? 0 : best.i;
        }
        __syncthreads();
        if (mode == 0) {
            for (int p = threadIdx.x; p < P; p += blockDim.x) out_a[group * P + p] = winners[p];
        } else if (threadIdx.x == 0) {
            const int D = P - 1;
            const int32_t *d = draft_ids + group * D;
            int32_t *tok = out_a + group * P;
            int bad = 0, a = D;
            for (int j = 0; j < D; ++j) {
                int32_t dj = d[j];
                if (dj < 0 || static_cast<int64_t>(dj) >= V) bad = 1;
                if (a == D && dj != winners[j]) a = j;
            }
            for (int j = 0; j < a; ++j) tok[j] = d[j];
            tok[a] = winners[a];
            for (int j = a + 1; j <= D; ++j) tok[j] = -1;
            out_b[group] = a;
            if (bad && status) atomicOr(status, MTPSPEC_STATUS_BAD_DRAFT_ID);
        }
    }
    // no CTA may exit while CTA 0 still reads its shared memory
    cluster_sync();
}

// Cluster size: enough CTAs per row to keep the slices near 2-4K elements, at most 8; at
// most 4 when there are many rows, which fill the GPU with fewer, longer slices (192 rows of
// 151,936 fp32: 29.4 -> 27.3 us; 1024 rows: 121.5 -> 108.8 us).
static int argmax_cluster_size(int64_t V, int64_t groups) {
    const int cmax = groups >= 64 ? 4 : 8;
    int C = 1;
    while (C < cmax && V / (2 * C) >= 2048) C *= 2;
    return C;
}

template <typename T>
static cudaError_t launch_argmax(const void *logits, int64_t groups, int P, int64_t V, int mode,
                                 const int32_t *d, int32_t *out_a, int32_t *out_b,
                                 int32_t *status, cudaStream_t stream) {
    const int C = argmax_cluster_size(V, groups);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(groups * C), 1, 1);
    cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_argmax_groups<T>,
                                             static_cast<const T *>(logits), V, P, mode, d, out_a,
                                             out_b, status);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_greedy_draft(const void *logits, int dtype, int64_t M, int64_t V, int32_t *ids,
                             cudaStream_t stream) {
    if (dtype == MTPSPEC_F32)
        return launch_argmax<float>(logits, M, 1, V, 0, nullptr, ids, nullptr, nullptr, stream);
    return launch_argmax<uint16_t>(logits, M, 1, V, 0, nullptr, ids, nullptr, nullptr, stream);
}

cudaError_t run_verify_greedy(const void *target, int dtype, const int32_t *d, int64_t B,
                              int32_t D, int64_t V, int32_t *tokens, int32_t *num_accepted,
                              int32_t *status, cudaStream_t stream) {
    if (dtype == MTPSPEC_F32)
        return launch_argmax<float>(target, B, D + 1, V, 1, d, tokens, num_accepted, status,
                                    stream);
    return launch_argmax<uint16_t>(target, B, D + 1, V, 1, d, tokens, num_accepted, status,
                                   stream);
}

}  // namespace mtpspec

namespace mtpspec {

// Greedy rows of a sampling verification: one cluster per row, all D + 1 positions.  A row
// with a positive temperature and a valid top-p belongs to the sampling kernel and is
// skipped.  For a greedy row the record of position j holds the argmax g_j, the flag
// d_j == g_j, p_target = [d_j == g_j] and p_draft = [d_j valid].
template <typename T>
__global__ void __launch_bounds__(kArgmaxThreads)
k_argmax_verify_rows(const T *__restrict__ logits, int64_t V, int D,
                     const float *__restrict__ tau, const float *__restrict__ top_p,
                     const int32_t *__restrict__ draft_ids, VerifyUnitRecord *__restrict__ rec,
                     int32_t *__restrict__ status) {
    __shared__ float red_v[kMaxPositions];
    __shared__ int32_t red_i[kMaxPositions];
    __shared__ float warp_v[kArgmaxThreads / 32];
    __shared__ int32_t warp_i[kArgmaxThreads / 32];

    const int64_t row = cluster_index();
    const float t = tau[row];
    const float p = top_p ? top_p[row] : 1.0f;
    const bool bad = !(t >= 0.0f) || !(p > 0.0f);
    if (!bad && t != 0.0f) return;  // the whole cluster takes this exit together

    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int P = D + 1;
    int64_t chunk = (V + C - 1) / C;
    chunk = (chunk + 15) & ~static_cast<int64_t>(15);
    const int64_t lo = min(V, static_cast<int64_t>(rank) * chunk);
    const int64_t hi = min(V, lo + chunk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int q = 0; q < P; ++q) {
        ArgMax a = warp_argmax(thread_scan(logits + (row * P + q) * V, lo, hi));
        if (lane == 0) {
            warp_v[warp] = a.v;
            warp_i[warp] = a.i;
        }
        __syncthreads();
        if (warp == 0) {
            ArgMax b{-INFINITY, -1};
            if (lane < kArgmaxThreads / 32) b = {warp_v[lane], warp_i[lane]};
            b = warp_argmax(b);
            if (lane == 0) {
                red_v[q] = b.v;
                red_i[q] = b.i;
            }
        }
        __syncthreads();
    }
    cluster_sync();
    if (rank == 0) {
        for (int q = threadIdx.x; q < P; q += blockDim.x) {
            ArgMax best{-INFINITY, -1};
            for (uint32_t r = 0; r < C; ++r) {
                ArgMax o;
                o.v = ld_peer_f32(peer_addr(smem_addr(&red_v[q]), r));
                o.i = ld_peer_s32(peer_addr(smem_addr(&red_i[q]), r));
                best = argmax_merge(best, o);
            }
            const int32_t g = best.i < 0 ? 0 : best.i;
            VerifyUnitRecord u;
            u.token = g;
            if (q < D) {
                const int32_t dj = draft_ids[row * D + q];
                const bool valid = dj >= 0 && static_cast<int64_t>(dj) < V;
                u.flags = dj == g ? 1 : 0;
                u.pt = dj == g ? 1.0f : 0.0f;
                u.pd = valid ? 1.0f : 0.0f;
                if (!valid && status) atomicOr(status, MTPSPEC_STATUS_BAD_DRAFT_ID);
            } else {
                u.flags = 0;
                u.pt = u.pd = 0.0f;
            }
            rec[row * P + q] = u;
        }
        if (threadIdx.x == 0 && bad && status) atomicOr(status, MTPSPEC_STATUS_BAD_PARAM);
    }
    cluster_sync();
}

template <typename T>
static cudaError_t launch_verify_greedy_rows(const VerifySampleArgs &a, cudaStream_t stream) {
    // (beside the sampling verifier's persistent grid, on the SMs it leaves: slices of the
    // original width)
    const int C = argmax_cluster_size(a.V, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B * C), 1, 1);
    cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, k_argmax_verify_rows<T>, static_cast<const T *>(a.target), a.V, a.D, a.temperature,
        a.top_p, a.draft_ids, static_cast<VerifyUnitRecord *>(a.workspace), a.status);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_verify_greedy_rows(const VerifySampleArgs &a, cudaStream_t stream) {
    return a.dtype == MTPSPEC_F32 ? launch_verify_greedy_rows<float>(a, stream)
                                  : launch_verify_greedy_rows<uint16_t>(a, stream);
}

}  // namespace mtpspec
