// Y[t, o] = sum_k A[o, k] * B[t, k] in bf16 with fp32 accumulation on the 5th-generation
// tensor cores: the projection of the draft head's input stage for larger token counts
// (A = eh_proj weight [H, 2H], B = the normalised activations [M, 2H]).
//
// The weight is the 128-row MMA operand ("swap AB"), the tokens are the N side, so one
// tile covers 128 output features of up to BN tokens and every weight tile is read once
// per token tile.  Per CTA: a TMA producer warp streams 128 x 64 weight tiles and BN x 64
// activation tiles (128-byte swizzled) through a STAGES-deep shared-memory ring guarded by
// mbarriers; one thread of the MMA warp issues tcgen05.mma (kind::f16, bf16 inputs, fp32
// accumulator in tensor memory) and releases each stage with tcgen05.commit; four epilogue
// warps read the accumulator with tcgen05.ld and store bf16 (or fp32 partial sums when the
// K range is split across CTAs, reduced by a second kernel).  Launched as the programmatic
// dependent of the kernel that writes the activations, the producer loads the weight tiles
// of the first stages, then waits for that kernel, then loads the activation tiles, so the
// weight stream starts while the activations are being written.  Every mbarrier wait is
// bounded; a wait that gives up sets a flag word in the workspace, and the CTA lets its
// copies and MMAs in flight complete before it leaves.
//
// k_head_argmax below is the draft head's output layer with the greedy pick: the same
// pipeline with the tokens as the 128-row operand and 256 vocabulary rows as the N side,
// persistent, with an epilogue that keeps each token's largest logit and its lowest id, so
// the logits never leave the SM.
#include <algorithm>

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace mtpspec {
namespace tg {

constexpr int BM = 128;          // output features per tile (MMA M)
constexpr int BK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int UK = 16;           // K per tcgen05.mma of kind::f16
constexpr int NTHREADS = 192;    // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr uint32_t WAIT_LIMIT = 1u << 18;  // polls: ~3.8 us each when unsuccessful, ~1 s in all
constexpr int A_BYTES = BM * BK * 2;

struct Params {
    uint16_t *y;       // [Mt, H] bf16, when splits == 1
    float *part;       // [splits, Mt, H] fp32 partial sums, when splits > 1
    unsigned long long *keys;  // k_head_argmax: [Mt, o_tiles] (order key << 32 | ~id)
    unsigned *err;     // flag word
    int H, Mt, K;      // H: rows of A (output features, or the vocabulary)
    int kb_total, kb_per_split, splits, o_tiles;
    int pdl;           // k_gemm: B is written by the preceding kernel on the stream
};

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; false if the phase never completed within `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit = WAIT_LIMIT) {
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_test(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with 128-byte swizzle:
// rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked at a stride of 1024 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 8 columns of 32-bit accumulator: this thread's lane, columns col..col+7.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(NTHREADS, 1)
k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
       const Params p) {
    constexpr int B_BYTES = BN * BK * 2;
    constexpr int STAGE = A_BYTES + B_BYTES;
    constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
    extern __shared__ uint8_t smem_dyn[];
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], accb;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int n_issued, n_consumed;  // stage fills sent and consumed (for an abort)

    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BM, t0 = blockIdx.y * BN, split = blockIdx.z;
    const int kb0 = split * p.kb_per_split;
    const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
    const int nkb = max(0, kb1 - kb0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&accb, 1);
        abort_flag = 0;
        n_issued = 0;
        n_consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tmA);
        prefetch_map(&tmB);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0 && lane == 0) {
        // ---- producer: the weight tiles of the first stages, then (once the activations
        // are written) the activation tiles, then both for every later stage
        const int pre = nkb < STAGES ? nkb : STAGES;
        for (int i = 0; i < pre; ++i) {
            mbar_expect_tx(&full[i], STAGE);
            tma_load_2d(ring + i * STAGE, &tmA, (kb0 + i) * BK, o0, &full[i]);
        }
        if (p.pdl) pdl_wait_primary();
        int issued = 0;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
            uint8_t *a = ring + s * STAGE;
            const int kx = (kb0 + i) * BK;
            if (i >= pre) {
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                if (abort_flag) break;
                mbar_expect_tx(&full[s], STAGE);
                tma_load_2d(a, &tmA, kx, o0, &full[s]);
            }
            tma_load_2d(a + A_BYTES, &tmB, kx, t0, &full[s]);
            issued = i + 1;
        }
        n_issued = issued;
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t idesc = instr_desc(BM, BN);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
            if (!mbar_wait(&full[s], ph)) {
                atomicOr(&abort_flag, 1);
                break;
            }
            tc_fence_after();
            const uint32_t a = smem_addr(ring + s * STAGE);
            const uint32_t b = a + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / UK; ++k) {
                // advancing 16 bf16 (32 bytes) along K inside the swizzled 128-byte rows
                mma_bf16(tmem, smem_desc_sw128(a + k * 32), smem_desc_sw128(b + k * 32), idesc,
                         (i > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&empty[s]);
            n_consumed = i + 1;
        }
        mma_commit(&accb);  // arrives once every MMA issued above has completed
    } else if (warp >= 2) {
        // ---- epilogue: TMEM lanes 32*(warp % 4) .. +31 are rows of this warp
        const int q = warp & 3;
        const bool ready = mbar_wait(&accb, 0);
        tc_fence_after();
        if (!ready) atomicOr(&abort_flag, 1);
        const int o = o0 + q * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
        for (int c = 0; c < BN; c += 8) {
            float v[8];
            tmem_ld8(trow + c, v);
            if (!ready || nkb == 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = 0.0f;
            }
            if (o < p.H) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = t0 + c + u;
                    if (t >= p.Mt) break;
                    if (p.splits == 1) {
                        __nv_bfloat16 h = __float2bfloat16_rn(v[u]);
                        p.y[static_cast<size_t>(t) * p.H + o] = *reinterpret_cast<uint16_t *>(&h);
                    } else {
                        p.part[(static_cast<size_t>(split) * p.Mt + t) * p.H + o] = v[u];
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        atomicOr(p.err, MTPSPEC_STATUS_TIMEOUT);
        // let the copies still in flight land, and the MMAs issued complete, before the
        // CTA's shared and tensor memory are released
        for (int i = n_consumed; i < n_issued; ++i)
            if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u)) break;
        mbar_wait(&accb, 0);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// The output layer's argmax GEMM, persistent: logits[t, v] = sum_k X[t, k] W[v, k] with the
// tokens as the 128-row MMA operand and HV = 256 vocabulary rows as the N side.  A tile is
// (token tile, vocabulary tile); CTA c takes tiles c, c + G, ... with the token tiles of one
// vocabulary tile side by side, so the CTAs that share a weight tile run together and it
// leaves HBM once.  Each stage carries 32 KB of weight and the tokens' tile, so four
// stages keep 128 KB of weight in flight per SM.  With at most 64 tokens only their 64
// rows are staged (8 KB): the MMA's rows 64 to 127 then read the start of the weight tile,
// which gives rows of the accumulator that no thread keeps, and five stages fit (160 KB
// of weight in flight).  The accumulator is double-buffered in
// tensor memory (2 x 256 columns): the epilogue of tile j reads one buffer while tile j + 1
// accumulates into the other.  In the epilogue each thread owns one token's row of the
// tile: it scans its 256 logits in id order and keeps the largest order key and the first
// id holding it, then writes one key (order key << 32 | ~id) per (token, vocabulary tile).
// Barriers: the stage ring (full / empty), accf[b] (MMA -> epilogue) and acce[b] (epilogue
// -> MMA).  Every wait is bounded; a wait that gives up raises the CTA's abort flag and
// every role leaves its loop.
constexpr int HT = 128;  // tokens per tile (MMA M)
constexpr int HV = 256;  // vocabulary rows per tile (MMA N)

template <int STAGES, int XROWS, int TOPK>
__global__ void __launch_bounds__(NTHREADS, 1)
k_head_argmax(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
              const Params p, int t_tiles, int n_tiles) {
    static_assert(XROWS == HT || (XROWS == 64 && XROWS * BK * 2 <= HV * BK * 2),
                  "a short token tile is followed by at least as many bytes of weight");
    constexpr int X_BYTES = XROWS * BK * 2;
    constexpr int W_BYTES = HV * BK * 2;
    constexpr int STAGE = X_BYTES + W_BYTES;
    constexpr uint32_t TMEM_COLS = 2 * HV;
    extern __shared__ uint8_t smem_dyn[];
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], accf[2], acce[2];
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort_flag;

    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int nkb = p.kb_total;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4);  // lane 0 of each epilogue warp
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tmX);
        prefetch_map(&tmW);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0 && lane == 0) {
        // ---- producer: every tile's K-blocks through the ring, one global stage counter
        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !abort_flag; tile += G) {
            const int t0 = (tile % t_tiles) * HT, v0 = (tile / t_tiles) * HV;
            for (int i = 0; i < nkb; ++i, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u)) abort_flag = 1;
                if (abort_flag) break;
                uint8_t *a = ring + s * STAGE;
                mbar_expect_tx(&full[s], STAGE);
                tma_load_2d(a, &tmX, i * BK, t0, &full[s]);
                tma_load_2d(a + X_BYTES, &tmW, i * BK, v0, &full[s]);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: tile j accumulates into buffer j & 1 once the epilogue has read it
        constexpr uint32_t idesc = instr_desc(HT, HV);
        int it = 0, j = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !abort_flag; tile += G, ++j) {
            const int b = j & 1;
            if (!mbar_wait(&acce[b], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u)) {
                abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + static_cast<uint32_t>(b * HV);
            for (int i = 0; i < nkb; ++i, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                if (!mbar_wait(&full[s], ph)) abort_flag = 1;
                if (abort_flag) break;
                tc_fence_after();
                const uint32_t a = smem_addr(ring + s * STAGE);
                const uint32_t w = a + X_BYTES;
#pragma unroll
                for (int k = 0; k < BK / UK; ++k)
                    mma_bf16(acc, smem_desc_sw128(a + k * 32), smem_desc_sw128(w + k * 32), idesc,
                             (i > 0 || k > 0) ? 1u : 0u);
                mma_commit(&empty[s]);
            }
            if (abort_flag) break;
            mma_commit(&accf[b]);  // arrives when this tile's MMAs have completed
        }
    } else if (warp >= 2) {
        // ---- epilogue: TMEM lane 32 (warp % 4) + lane is this thread's token
        const int q = warp & 3;
        int j = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += G, ++j) {
            const int b = j & 1;
            const int vt = tile / t_tiles, v0 = vt * HV;
            const int t = (tile % t_tiles) * HT + q * 32 + lane;
            if (abort_flag || !mbar_wait(&accf[b], static_cast<uint32_t>(j >> 1) & 1u)) {
                abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * HV);
            const int nv = min(HV, p.H - v0);  // vocabulary rows of this tile
            if constexpr (TOPK == 1) {
                uint32_t best = 0;  // below every value's order key
                int bv = v0;
                for (int c = 0; c < HV; c += 8) {
                    float v[8];
                    tmem_ld8(trow + c, v);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t key = c + u < nv ? order_key(v[u]) : 0u;
                        if (key > best) {  // strictly larger: the first id keeps a tie
                            best = key;
                            bv = v0 + c + u;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&acce[b])) : "memory");
                if (t < p.Mt)
                    p.keys[static_cast<size_t>(t) * p.o_tiles + vt] =
                        (static_cast<unsigned long long>(best) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(bv));
            } else {
                // the TOPK largest (order key << 32 | ~id), kept sorted in decreasing order:
                // a key that beats the last one replaces it and bubbles up
                unsigned long long lst[TOPK];
#pragma unroll
                for (int i = 0; i < TOPK; ++i) lst[i] = 0ull;
                for (int c = 0; c < HV; c += 8) {
                    float v[8];
                    tmem_ld8(trow + c, v);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const unsigned long long key =
                            c + u < nv ? (static_cast<unsigned long long>(order_key(v[u])) << 32) |
                                             (0xFFFFFFFFu - static_cast<uint32_t>(v0 + c + u))
                                       : 0ull;
                        if (key > lst[TOPK - 1]) {
                            lst[TOPK - 1] = key;
#pragma unroll
                            for (int i = TOPK - 1; i > 0; --i) {
                                if (lst[i] > lst[i - 1]) {
                                    const unsigned long long tmp = lst[i];
                                    lst[i] = lst[i - 1];
                                    lst[i - 1] = tmp;
                                }
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&acce[b])) : "memory");
                if (t < p.Mt) {
                    unsigned long long *kd = p.keys + (static_cast<size_t>(t) * p.o_tiles + vt) * TOPK;
#pragma unroll
                    for (int i = 0; i < TOPK; ++i) kd[i] = lst[i];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) atomicOr(p.err, MTPSPEC_STATUS_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// y = bf16(sum over splits of the fp32 partials), 4 outputs per thread.
__global__ void k_split_reduce(const float *__restrict__ part, uint16_t *__restrict__ y,
                               int64_t n, int splits) {
    pdl_wait_primary();
    const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (i >= n) return;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < splits; ++s) {
        const float4 v = *reinterpret_cast<const float4 *>(part + s * n + i);
        acc[0] += v.x;
        acc[1] += v.y;
        acc[2] += v.z;
        acc[3] += v.w;
    }
    uint16_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        __nv_bfloat16 h = __float2bfloat16_rn(acc[u]);
        o[u] = *reinterpret_cast<uint16_t *>(&h);
    }
    *reinterpret_cast<uint2 *>(y + i) =
        make_uint2(o[0] | (static_cast<uint32_t>(o[1]) << 16), o[2] | (static_cast<uint32_t>(o[3]) << 16));
}

// Diagnostic of the bounded wait: a barrier of two arrivals gets one, so the wait must give
// up after `limit` polls; then MTPSPEC_STATUS_TIMEOUT is OR-ed into the status word, as the
// kernels do.
__global__ void k_wait_selftest(uint32_t limit, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&bar)) : "memory");
    if (!mbar_wait(&bar, 0, limit)) atomicOr(status, MTPSPEC_STATUS_TIMEOUT);
}

}  // namespace tg

cudaError_t run_wait_selftest_gemm(uint32_t limit, int32_t *status, cudaStream_t stream) {
    tg::k_wait_selftest<<<1, 32, 0, stream>>>(limit, status);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2D map of a row-major bf16 matrix [rows, cols] with boxes of box_rows x 64 columns.
static bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(tg::BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct GemmPlan {
    int BN, splits, kb_per_split, kb_total, o_tiles, t_tiles;
};

// SMs of a GB300; the plan depends on the sizes alone, so that the workspace query (which
// needs no GPU) and the launch agree.
constexpr int kPlanSMs = 152;

// Tile widths and K splits.  Up to 256 tokens, one token tile (the narrowest width that
// holds them): the weight, the bulk of the bytes, is streamed once.  Beyond, the width of
// 128, 192 or 256 whose tiles fill the SMs in the fewest waves of the least work (waves x
// width).  Then K is split so that the grid fills one wave (of one CTA an SM, or two for
// tiles up to 64 tokens wide), keeping at least 8 (or 4) K-blocks a split.
static GemmPlan plan_gemm(int64_t H, int64_t Mt, int64_t K) {
    GemmPlan g;
    g.o_tiles = static_cast<int>((H + tg::BM - 1) / tg::BM);
    g.kb_total = static_cast<int>((K + tg::BK - 1) / tg::BK);
    if (Mt <= 256) {
        g.BN = Mt <= 16 ? 16 : (Mt <= 32 ? 32 : (Mt <= 64 ? 64 : (Mt <= 128 ? 128 : (Mt <= 192 ? 192 : 256))));
    } else {
        int64_t best = -1;
        for (int bn : {256, 192, 128}) {
            const int64_t tiles = g.o_tiles * ((Mt + bn - 1) / bn);
            const int64_t cost = ((tiles + kPlanSMs - 1) / kPlanSMs) * bn;
            if (best < 0 || cost < best) {
                best = cost;
                g.BN = bn;
            }
        }
    }
    g.t_tiles = static_cast<int>((Mt + g.BN - 1) / g.BN);
    const int tiles = g.o_tiles * g.t_tiles;
    // token tiles up to 64 wide run two CTAs an SM (rings of 4 to 6 stages), so the weight
    // stream spreads over twice the CTAs, with splits of at least 4 K-blocks
    const int slots = g.BN <= 64 ? 2 * kPlanSMs : kPlanSMs;
    const int minkb = g.BN <= 64 ? 4 : 8;
    int splits = tiles >= slots ? 1 : slots / tiles;
    splits = std::max(1, std::min(splits, g.kb_total / minkb));
    g.kb_per_split = (g.kb_total + splits - 1) / splits;
    g.splits = (g.kb_total + g.kb_per_split - 1) / g.kb_per_split;
    return g;
}

size_t gemm_workspace_bytes(int64_t Mt, int64_t H) {
    const GemmPlan g = plan_gemm(H, Mt, 2 * H);
    const size_t part = g.splits > 1 ? static_cast<size_t>(g.splits) * Mt * H * 4 : 0;
    return 256 + part;  // flag word, then the partial sums
}
size_t gemm_zero_bytes(int64_t Mt, int64_t H) {
    (void)Mt;
    (void)H;
    return 256;  // the flag word's block
}

template <int BN, int STAGES>
static cudaError_t launch_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const tg::Params &p,
                               const GemmPlan &g, bool pdl, cudaStream_t stream) {
    constexpr int smem = STAGES * (tg::A_BYTES + BN * tg::BK * 2) + 1024;
    static AttrCache attr;
    cudaError_t e = ensure_attr(tg::k_gemm<BN, STAGES>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem, attr);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.o_tiles, g.t_tiles, g.splits);
    cfg.blockDim = dim3(tg::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, tg::k_gemm<BN, STAGES>, ma, mb, p);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_gemm_bf16_nt(const void *A, const void *B, void *Y, int64_t H, int64_t Mt,
                             int64_t K, void *workspace, bool pdl, cudaStream_t stream) {
    const GemmPlan g = plan_gemm(H, Mt, K);
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, H, K, tg::BM) || !make_map(&mb, B, Mt, K, g.BN))
        return cudaErrorInvalidValue;
    tg::Params p = {};
    p.y = static_cast<uint16_t *>(Y);
    p.err = static_cast<unsigned *>(workspace);
    p.part = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) + 256);
    p.H = static_cast<int>(H);
    p.Mt = static_cast<int>(Mt);
    p.K = static_cast<int>(K);
    p.kb_total = g.kb_total;
    p.kb_per_split = g.kb_per_split;
    p.splits = g.splits;
    p.pdl = pdl ? 1 : 0;
    cudaError_t e;
    switch (g.BN) {
    case 16: e = launch_gemm<16, 6>(ma, mb, p, g, pdl, stream); break;  // two CTAs an SM
    case 32: e = launch_gemm<32, 5>(ma, mb, p, g, pdl, stream); break;
    case 64: e = launch_gemm<64, 4>(ma, mb, p, g, pdl, stream); break;
    case 128: e = launch_gemm<128, 6>(ma, mb, p, g, pdl, stream); break;
    case 192: e = launch_gemm<192, 5>(ma, mb, p, g, pdl, stream); break;
    default: e = launch_gemm<256, 4>(ma, mb, p, g, pdl, stream); break;
    }
    if (e != cudaSuccess || g.splits == 1) return e;
    const int64_t n = Mt * H;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((n / 4 + 255) / 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tg::k_split_reduce, static_cast<const float *>(p.part),
                           static_cast<uint16_t *>(Y), n, g.splits);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

// The output layer's logits tile by tile with the argmax epilogue: keys [Mt, o_tiles], one
// per (token, block of 256 vocabulary rows).  Token tiles of 128; the persistent grid has
// one CTA per SM (fewer when there are fewer tiles).  No K split.
int lm_head_o_tiles(int64_t V) { return static_cast<int>((V + tg::HV - 1) / tg::HV); }

template <int STAGES, int XROWS, int TOPK>
static cudaError_t launch_head_argmax(const CUtensorMap &mx, const CUtensorMap &mw,
                                      const tg::Params &p, int t_tiles, int n_tiles,
                                      cudaStream_t stream) {
    constexpr int smem = STAGES * (XROWS + tg::HV) * tg::BK * 2 + 1024;
    static AttrCache attr;
    cudaError_t e = ensure_attr(tg::k_head_argmax<STAGES, XROWS, TOPK>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem, attr);
    if (e != cudaSuccess) return e;
    const int grid = n_tiles < kPlanSMs ? n_tiles : kPlanSMs;  // persistent: one CTA per SM
    tg::k_head_argmax<STAGES, XROWS, TOPK><<<grid, tg::NTHREADS, smem, stream>>>(mx, mw, p, t_tiles, n_tiles);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_gemm_argmax(const void *W, const void *X, int64_t V, int64_t Mt, int64_t K,
                            unsigned long long *keys, unsigned *err, int topk, cudaStream_t stream) {
    const bool short_x = Mt <= 64;
    const int t_tiles = static_cast<int>((Mt + tg::HT - 1) / tg::HT);
    const int v_tiles = lm_head_o_tiles(V);
    const int n_tiles = t_tiles * v_tiles;
    CUtensorMap mx, mw;
    if (!make_map(&mx, X, Mt, K, short_x ? 64 : tg::HT) || !make_map(&mw, W, V, K, tg::HV))
        return cudaErrorInvalidValue;
    tg::Params p = {};
    p.keys = keys;
    p.err = err;
    p.H = static_cast<int>(V);
    p.Mt = static_cast<int>(Mt);
    p.K = static_cast<int>(K);
    p.kb_total = static_cast<int>((K + tg::BK - 1) / tg::BK);
    p.kb_per_split = p.kb_total;
    p.splits = 1;
    p.o_tiles = v_tiles;
    if (topk > 1)
        return short_x ? launch_head_argmax<5, 64, kLmHeadTopK>(mx, mw, p, t_tiles, n_tiles, stream)
                       : launch_head_argmax<4, tg::HT, kLmHeadTopK>(mx, mw, p, t_tiles, n_tiles, stream);
    return short_x ? launch_head_argmax<5, 64, 1>(mx, mw, p, t_tiles, n_tiles, stream)
                   : launch_head_argmax<4, tg::HT, 1>(mx, mw, p, t_tiles, n_tiles, stream);
}

}  // namespace mtpspec
