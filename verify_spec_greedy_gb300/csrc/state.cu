// The model state around a verification ("14. MTP: speculative decoding with the built-in
// draft head", the decoding loop's snapshot / rollback and "Rolling back": a KV cache is
// rolled back by truncation, while the linear attention's memory tables and convolution
// windows are copied before verification and copied back on a miss).
//
// k_state_copy takes the snapshot: one flat copy of B rows of row_bytes, 16-byte streaming
// loads, four vectors in flight per thread, a grid of a few CTAs per SM striding over the
// whole range.  k_state_fixup applies the verifier's accepted counts: grid.y walks the
// rows, grid.x the chunks of a row; the first thread of a row's first chunk writes its
// lengths, and on a miss every chunk copies its slice of the snapshot back.  Rows kept
// whole (a hit) cost one load of their count.  Both are HBM-bound copies.
#include "common.cuh"
#include "kernels.h"
#include "../../include/libmtpspec.h"

namespace mtpspec {
namespace st {

constexpr int THREADS = 256;
constexpr int VPT = 4;                      // 16-byte vectors in flight per thread
constexpr int64_t CHUNK = THREADS * VPT;    // vectors per CTA pass

__device__ __forceinline__ void copy_range(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                           int64_t first, int64_t n, int64_t stride) {
    for (int64_t i = first + threadIdx.x; i < n; i += stride) {
        uint4 v[VPT];
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int64_t k = i + static_cast<int64_t>(u) * THREADS;
            if (k < n) v[u] = ld_stream_16B(src + k);
        }
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int64_t k = i + static_cast<int64_t>(u) * THREADS;
            if (k < n) dst[k] = v[u];
        }
    }
}

__global__ void __launch_bounds__(THREADS)
k_state_copy(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16) {
    copy_range(src, dst, static_cast<int64_t>(blockIdx.x) * CHUNK, n16,
               static_cast<int64_t>(gridDim.x) * CHUNK);
}

__global__ void __launch_bounds__(THREADS)
k_state_fixup(const int32_t *__restrict__ num_accepted, int D, const int32_t *kv_before,
              int32_t *kv_len, uint4 *__restrict__ state, const uint4 *__restrict__ backup,
              int64_t B, int64_t row16, int32_t *__restrict__ draft_kv_len,
              int32_t *__restrict__ recompute, int32_t *__restrict__ status) {
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const int a = num_accepted[b];
        const bool bad = a < 0 || a > D;
        const bool miss = !bad && a < D;
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            if (bad) {
                if (status) atomicOr(status, MTPSPEC_STATUS_BAD_PARAM);
            } else {
                const int before = kv_before[b];
                int kv, rc = 0;
                if (!miss) {
                    kv = before + D + 1;          // every verified position stays
                } else if (row16 > 0) {
                    kv = before;                  // back to the snapshot
                    rc = 1 + a;                   // the carried-in token and the accepted drafts
                } else {
                    kv = before + 1 + a;          // attention only: keep the accepted prefix
                }
                kv_len[b] = kv;
                if (recompute) recompute[b] = rc;
                if (draft_kv_len && miss && draft_kv_len[b] > kv) draft_kv_len[b] = kv;
            }
        }
        if (miss && row16 > 0)
            copy_range(backup + b * row16, state + b * row16,
                       static_cast<int64_t>(blockIdx.x) * CHUNK, row16,
                       static_cast<int64_t>(gridDim.x) * CHUNK);
    }
}

}  // namespace st

cudaError_t run_state_snapshot(const void *state, void *backup, int64_t B, int64_t row_bytes,
                               cudaStream_t stream) {
    const int64_t n16 = B * (row_bytes / 16);
    if (n16 == 0) return cudaSuccess;
    const int64_t chunks = (n16 + st::CHUNK - 1) / st::CHUNK;
    const unsigned grid = static_cast<unsigned>(chunks < 152 * 8 ? chunks : 152 * 8);
    st::k_state_copy<<<grid, st::THREADS, 0, stream>>>(static_cast<const uint4 *>(state),
                                                       static_cast<uint4 *>(backup), n16);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_state_fixup(const int32_t *num_accepted, int32_t D, const int32_t *kv_before,
                            int32_t *kv_len, void *state, const void *backup, int64_t B,
                            int64_t row_bytes, int32_t *draft_kv_len, int32_t *recompute,
                            int32_t *status, cudaStream_t stream) {
    const int64_t row16 = row_bytes / 16;
    const int64_t chunks = row16 > 0 ? (row16 + st::CHUNK - 1) / st::CHUNK : 1;
    const dim3 grid(static_cast<unsigned>(chunks < 2048 ? chunks : 2048),
                    static_cast<unsigned>(B < 65535 ? B : 65535), 1);
    st::k_state_fixup<<<grid, st::THREADS, 0, stream>>>(
        num_accepted, D, kv_before, kv_len, static_cast<uint4 *>(state),
        static_cast<const uint4 *>(backup), B, row16, draft_kv_len, recompute, status);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace mtpspec
