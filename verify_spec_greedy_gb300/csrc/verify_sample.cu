// Speculative-sampling verification: temperature -> top-k -> top-p filtering of target and
// draft logits, the accept test U <= p/q, the residual draw at the first rejection and the
// bonus draw ("MPT (MTP, Multi-Token Prediction) 原理详解", section 三 stage 3 "rejection
// sampling" and stage 4; "The decoding loop and MTP", "Why a hand-written decoding loop" for
// the filters and "MTP speculative decoding" items 2-3 for the drawn replacement and the
// extra token).
//
// Three kernels on the caller's stream:
//  - k_verify_persistent: the sampled rows.  A persistent grid of thread-block clusters,
//    as many as can be resident; cluster g takes units g, g + G, ... (a unit is one
//    (row b, position j) pair of a sampled row).  CTA r of a cluster owns the contiguous
//    vocabulary slice [r*slice, (r+1)*slice).  Each CTA keeps two shared-memory buffers:
//    while it works on one unit, bulk asynchronous copies bring the next unit's slices of
//    the target row (and, for j < D, of the draft row) into the other, so every logit is
//    read from HBM exactly once and the loads overlap the work.
//  - the greedy rows (temperature 0) go to the streaming argmax kernel
//    (run_verify_greedy_rows), launched as a programmatic dependent so that it runs beside
//    the persistent grid.
//  - k_verify_finalize: one thread per row takes the first rejected position.
//
// Work on one unit, all on chip:
//   pass 1   maximum and online softmax sum as the chunks land
//   E1       per-CTA partials meet in every CTA through distributed shared memory
//   pass 2   (top-k / top-p) counts over fine bins of z = (x - max) * log2(e) / tau,
//            R bins per unit of z, only for elements that can hold the boundary; the counts
//            are reduce-scattered and re-broadcast across the cluster (E2)
//   plan     the bins that must hold the boundary, from exact counts (top-k) or from
//            per-bin weight bounds count * 2^(-b/R) (top-p)
//   gather   elements of those bins are pushed to every CTA with their weights, and the
//            exact weight of everything above them is summed (E3); each CTA sorts the
//            candidates (bitonic) and scans them for the exact thresholds.  If the boundary
//            is outside the binned range or too many elements fall in its bins, an exact
//            bisection over the 32-bit value keys replaces this step.
//   accept   p(d), q(d) and U_acc <= p/q (ratio formed with both maxima factored out)
//   draw     only for a rejected draft or the bonus position: draw weights in fixed point
//            (2^31 per unit of probability), per-warp sums in id order, CTA sums exchanged
//            (E4), and the CTA holding the target walks its slice to the token.
//
// Weight sums are formed per thread in fp32 over a fixed set of elements, converted once
// to 64-bit fixed point and reduced as integers, so every sum is deterministic and the same
// in every CTA of a cluster.  Every decision is computed identically in every CTA from
// exchanged data, so all CTAs run the same sequence of cluster barriers.  Exchanges are
// pushes into the peers' shared memory before a barrier.  Every unit starts with barrier
// B1 after its first exchange, so later exchanges of a unit cannot overwrite data a slower
// CTA still reads for the previous unit; the first exchange alternates between two
// buffers by unit parity.  The bulk-copy waits are bounded and raise
// MTPSPEC_STATUS_TIMEOUT when they give up.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mtpspec {
namespace vs {

constexpr int NT = 512;          // threads per CTA
constexpr int NW = NT / 32;      // warps per CTA
constexpr int MAXC = 16;         // largest cluster
constexpr int R = 64;            // histogram bins per unit of z (log2 of the softmax weight)
constexpr int ZR = 24;           // binned range: z in (-ZR, 0], weights in (2^-24, 1]
constexpr int NB = R * ZR;       // bins
constexpr int INCOMING = NB + MAXC;  // reduce-scatter slots per row (C * ceil(NB / C))
constexpr int CAP = 512;         // boundary candidates per row (= NT: one per thread)
constexpr int NCH = 4;           // bulk-copy chunks per row
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr float FX = 2147483648.0f;  // 2^31: fixed-point scale of weights (weights <= 1)
constexpr double INV_FX = 1.0 / 2147483648.0;
constexpr float BOUND_SLACK = 4e-5f;  // relative slack of the per-bin weight bounds
static_assert(CAP == NT, "the candidate sort keeps one candidate per thread");

using UnitResult = VerifyUnitRecord;

struct __align__(8) Cand {
    float v;       // logit
    uint32_t idx;  // token id
};

struct __align__(16) Shared {
    unsigned long long bar[2][2][NCH];  // [buffer][row][chunk] bulk-copy barriers
    // block reductions
    float rf[2][NW];
    float rs[2][NW];
    unsigned long long ru[2][NW];
    unsigned long long scan[NW];
    int32_t scani[NW];
    // E1, by unit parity: partials of every CTA and the draft token's logit per row
    float x_m[2][MAXC][2];
    float x_s[2][MAXC][2];
    float x_d[2][2];
    // per-row state, identical in every CTA of the cluster
    float m[2], Z[2], invZ[2], theta[2], zcut[2];
    int32_t deg[2];           // a row of all -inf: a point mass on id 0
    int32_t mode[2];          // 0 no filter, 1 candidates, 2 exact bisection
    int32_t b1[2], b2[2];
    uint32_t ncand[2];
    unsigned long long tgt[2];
    // histogram of counts (local during pass 2, cluster-wide after E2)
    uint32_t hcnt[2][NB];
    // reduce-scatter inbox, reused for the boundary candidates
    union {
        uint32_t in[2][INCOMING];
        struct {
            Cand c[2][CAP];
            unsigned long long w[2][CAP];
        } cd;
    } u;
    unsigned long long skey[CAP];      // candidate sort keys, then exclusive weight prefix
    float sval[CAP];                   // sorted candidate values
    uint32_t cand_n[2];                // slot allocator, used in CTA 0
    uint32_t lcount[2];                // this CTA's own candidates, then its base slot
    Cand lc[2][CAP];                   // this CTA's own candidates before the push
    uint32_t lw[2][CAP];
    unsigned long long ma_x[MAXC][2];  // per-CTA fixed-point weight above bin b1
    unsigned long long sx[2][2][MAXC];  // exact bisection exchange, by iteration parity
    unsigned long long dr_R[2][MAXC];   // per draw attempt: each CTA's fixed-point weight
    unsigned long long w_sum[NW];
    int32_t flags;  // bit 0: a bulk copy timed out
    int32_t pick[4];
    float fpick[4];
};

__device__ __forceinline__ float ex2(float z) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
    return r;
}
// z = (x - m) * c2, written so that every pass computes it with the same two roundings
__device__ __forceinline__ float zval(float x, float m, float c2) {
    return __fmul_rn(__fsub_rn(x, m), c2);
}
// bin of z in (-ZR, 0]; NB below the range (or NaN)
__device__ __forceinline__ int zbin(float z) {
    if (!(z > -static_cast<float>(ZR))) return NB;
    const int b = static_cast<int>(__fmul_rn(-z, static_cast<float>(R)));
    return b < NB ? b : NB - 1;
}
// a weight (<= 1) in fixed point; the float-to-32-bit conversion is a fast instruction
__device__ __forceinline__ uint32_t fix31(float w) { return __float2uint_rn(__fmul_rn(w, FX)); }
// a per-thread sum in fixed point: a slow 64-bit conversion, used once per thread
__device__ __forceinline__ unsigned long long fix_sum(float s) {
    return __float2ull_rn(__fmul_rn(s, FX));
}

// ---------------------------------------------------------------- Philox4x32-10

// Philox4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32->64 multiplications with
// the round multipliers, half swaps and key mixing; the key advances by the two Weyl
// increments after each round.
__device__ __forceinline__ void philox(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}
// odd multiple of 2^-24 in (0, 1), exact in fp32
__device__ __forceinline__ float word_uniform(uint32_t w) {
    return __uint2float_rn(2u * (w >> 9) + 1u) * 5.9604644775390625e-08f;
}

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2, float c2) {
    if (s2 == 0.0f) return;
    if (s == 0.0f) {
        m = m2;
        s = s2;
        return;
    }
    const float M = fmaxf(m, m2);
    s = s * ex2(__fmul_rn(m - M, c2)) + s2 * ex2(__fmul_rn(m2 - M, c2));
    m = M;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
    return __reduce_add_sync(0xFFFFFFFFu, v);
}

// Sum of one u64 per thread over the block; every thread gets the result.
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long *scratch) {
    v = warp_sum_u64(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long t = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) t += scratch[w];
    return t;
}
// Exclusive prefix sum over the block in thread order.
__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v,
                                                                  unsigned long long *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    unsigned long long before = 0;
    for (int w = 0; w < warp; ++w) before += scratch[w];
    return before + incl - v;
}
// Inclusive prefix maximum over the block in thread order.
__device__ __forceinline__ int32_t block_incl_max_i32(int32_t v, int32_t *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl = max(incl, y);
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int32_t before = -1;
    for (int w = 0; w < warp; ++w) before = max(before, scratch[w]);
    return max(before, incl);
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity) {
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
// Wait for the phase of the given parity; false after WAIT_LIMIT polls.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, uint32_t parity) {
    for (uint32_t it = 0; it < WAIT_LIMIT; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// Order this thread's earlier generic-proxy accesses of shared memory before later
// bulk-copy (async-proxy) writes into it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Visit every element [0, n) of a shared-memory slice as (value, local index), with
// 16-byte vector reads for the aligned body, threads strided over vectors.  Each thread
// always visits the same elements in the same order.
template <typename T, typename F>
__device__ __forceinline__ void for_each_elem(const T *s, int n, F &&f) {
    constexpr int EPV = elems_per_16B<T>::value;
    const int nv = n / EPV;
    const uint4 *v = reinterpret_cast<const uint4 *>(s);
    for (int i = threadIdx.x; i < nv; i += NT) {
        float x[EPV];
        unpack(v[i], x);
#pragma unroll
        for (int e = 0; e < EPV; ++e) f(x[e], i * EPV + e);
    }
    for (int i = nv * EPV + threadIdx.x; i < n; i += NT) f(widen(s[i]), i);
}

// First bin whose cumulative count reaches `need` (NB if none); one warp.
__device__ void count_search(const uint32_t *cnt, uint32_t need, int32_t *out) {
    const int lane = threadIdx.x & 31;
    constexpr int PER = NB / 32;
    uint32_t own = 0;
    for (int t = 0; t < PER; ++t) own += cnt[lane * PER + t];
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += a;
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, incl - own < need && incl >= need);
    if (ball == 0) {
        if (lane == 0) *out = NB;
    } else if (lane == __ffs(ball) - 1) {
        uint32_t acc = incl - own;
        for (int t = 0; t < PER; ++t) {
            acc += cnt[lane * PER + t];
            if (acc >= need) {
                *out = lane * PER + t;
                break;
            }
        }
    }
    __syncwarp();
}

// Bins that must hold the top-p boundary: bin b holds weights in [2^-(b+1)/R, 2^-b/R]
// (relative to the row maximum), so the cumulative weight of bins 0..b lies between two
// bounds.  *first = the first bin whose upper bound reaches `need`, *last = the first bin
// whose lower bound reaches it (NB if none).  One warp.
__device__ void weight_search(const uint32_t *cnt, float need, int32_t *first, int32_t *last) {
    const int lane = threadIdx.x & 31;
    constexpr int PER = NB / 32;
    const float step = ex2(-1.0f / R);
    const float up = 1.0f + BOUND_SLACK, dn = (1.0f - BOUND_SLACK) * step;
    float hi = 0.0f, lo = 0.0f;
    float w = ex2(-static_cast<float>(lane * PER) / R);
    for (int t = 0; t < PER; ++t) {
        const float c = static_cast<float>(cnt[lane * PER + t]);
        hi += c * w * up;
        lo += c * w * dn;
        w *= step;
    }
    float ihi = hi, ilo = lo;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float a = __shfl_up_sync(0xFFFFFFFFu, ihi, o);
        const float c = __shfl_up_sync(0xFFFFFFFFu, ilo, o);
        if (lane >= o) {
            ihi += a;
            ilo += c;
        }
    }
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const float incl = pass == 0 ? ihi : ilo, own = pass == 0 ? hi : lo;
        const float f = pass == 0 ? up : dn;
        int32_t *out = pass == 0 ? first : last;
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, incl - own < need && incl >= need);
        if (ball == 0) {
            if (lane == 0) *out = NB;
        } else if (lane == __ffs(ball) - 1) {
            float acc = incl - own;
            float ww = ex2(-static_cast<float>(lane * PER) / R);
            int res = lane * PER + PER - 1;
            for (int t = 0; t < PER; ++t) {
                acc += static_cast<float>(cnt[lane * PER + t]) * ww * f;
                ww *= step;
                if (acc >= need) {
                    res = lane * PER + t;
                    break;
                }
            }
            *out = res;
        }
    }
    __syncwarp();
}

struct Params {
    const void *T;
    const void *Q;
    const int32_t *d;
    const float *tau;
    const int32_t *topk;
    const float *topp;
    uint64_t seed;
    int64_t B;
    int32_t D;
    int64_t V;
    int64_t slice;
    int32_t nbuf;  // shared-memory data buffers per CTA: 2 (double-buffered) or 1
    int32_t G;     // clusters in the persistent grid
    UnitResult *res;
    int32_t *status;
};

__device__ __forceinline__ bool row_sampled(const Params &P, int64_t b) {
    const float t = P.tau[b];
    const float p = P.topp ? P.topp[b] : 1.0f;
    return t > 0.0f && p > 0.0f;  // rows with tau = 0 or bad parameters are greedy
}

// ---------------------------------------------------------------- the persistent kernel

template <typename T>
__global__ void __launch_bounds__(NT, 1) k_verify_persistent(const Params P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Shared &sh = *reinterpret_cast<Shared *>(smem_raw);
    constexpr int EPV = elems_per_16B<T>::value;
    const size_t data_off = (sizeof(Shared) + 127) & ~static_cast<size_t>(127);
    const size_t row_bytes =
        ((static_cast<size_t>(P.slice) * sizeof(T)) + 127) & ~static_cast<size_t>(127);
    auto sdat = [&](int buf, int row) -> T * {
        return reinterpret_cast<T *>(smem_raw + data_off + (2 * buf + row) * row_bytes);
    };

    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int64_t g = cluster_index();
    const int D = P.D;
    const int64_t V = P.V;
    const int64_t U = P.B * (D + 1);
    const int64_t G = P.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lo64 = static_cast<int64_t>(rank) * P.slice;
    const int64_t rest = V - lo64;
    const int n = static_cast<int>(rest <= 0 ? 0 : (rest < P.slice ? rest : P.slice));
    const int nv = n / EPV;
    const int per_ch = (nv + NCH - 1) / NCH;

    // ---- set-up
    if (tid == 0) {
        for (int bb = 0; bb < 2; ++bb)
            for (int r = 0; r < 2; ++r)
                for (int c = 0; c < NCH; ++c) mbar_init(&sh.bar[bb][r][c], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh.flags = 0;
    }
    __syncthreads();
    cluster_arrive_release();  // peers may touch this CTA's shared memory after the wait below
    pdl_launch_dependents();   // the greedy-row kernel runs beside this grid

    auto row_ptr = [&](int64_t u, int r) -> const T * {
        const int64_t b = u / (D + 1);
        const int j = static_cast<int>(u - b * (D + 1));
        return r == 0 ? static_cast<const T *>(P.T) + (b * (D + 1) + j) * V + lo64
                      : static_cast<const T *>(P.Q) + (b * D + j) * V + lo64;
    };
    auto next_unit = [&](int64_t u) -> int64_t {
        for (u += G; u < U; u += G)
            if (row_sampled(P, u / (D + 1))) return u;
        return -1;
    };
    // thread 0: arm every chunk barrier of buffer `buf` exactly once for unit u, with
    // bulk copies of the 16-byte-aligned bodies of its rows
    auto issue = [&](int64_t u, int buf) {
        const int j = static_cast<int>(u % (D + 1));
        const int nrows = j < D ? 2 : 1;
        for (int r = 0; r < 2; ++r) {
            const T *src = r < nrows ? row_ptr(u, r) : nullptr;
            const bool bulk = r < nrows && nv > 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
            for (int c = 0; c < NCH; ++c) {
                const int v0 = c * per_ch, v1 = min(nv, v0 + per_ch);
                if (bulk && v1 > v0) {
                    const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
                    mbar_expect_tx(&sh.bar[buf][r][c], bytes);
                    bulk_copy_g2s(sdat(buf, r) + v0 * EPV, src + v0 * EPV, bytes, &sh.bar[buf][r][c]);
                } else {
                    mbar_arrive(&sh.bar[buf][r][c]);
                }
            }
        }
    };

    int64_t u = -1;
    if (g < U) u = row_sampled(P, g / (D + 1)) ? g : next_unit(g);
    if (tid == 0 && u >= 0) {
        issue(u, 0);
        if (P.nbuf == 2) {
            const int64_t u1 = next_unit(u);
            if (u1 >= 0) issue(u1, 1);
        }
    }
    bool started = false;

    for (int k = 0; u >= 0; ++k) {
        const int buf = P.nbuf == 2 ? (k & 1) : 0;
        const uint32_t par = static_cast<uint32_t>(P.nbuf == 2 ? (k >> 1) & 1 : k & 1);
        const int ep = k & 1;
        if (P.nbuf == 1 && k > 0 && tid == 0) issue(u, 0);
        T *const sd0 = sdat(buf, 0);
        T *const sd1 = sdat(buf, 1);

        const int64_t b = u / (D + 1);
        const int j = static_cast<int>(u - b * (D + 1));
        const float tau = P.tau[b];
        const int32_t kk = P.topk ? P.topk[b] : 0;
        const float pp = P.topp ? P.topp[b] : 1.0f;
        const bool has_q = j < D;
        const int nrows = has_q ? 2 : 1;
        const bool k_on = kk >= 1 && static_cast<int64_t>(kk) < V;
        const bool p_on = pp < 1.0f;
        const float c2 = __fdiv_rn(1.44269504088896340736f, tau);
        const int32_t d = j < D ? P.d[b * D + j] : -1;
        const bool dvalid = d >= 0 && static_cast<int64_t>(d) < V;
        const bool d_here =
            dvalid && static_cast<int64_t>(d) >= lo64 && static_cast<int64_t>(d) < lo64 + n;

        // the parts the bulk copies do not cover: a ragged tail, or a misaligned row
        for (int r = 0; r < nrows; ++r) {
            const T *src = row_ptr(u, r);
            const bool bulk = nv > 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
            T *dst = r == 0 ? sd0 : sd1;
            for (int i = (bulk ? nv * EPV : 0) + tid; i < n; i += NT) dst[i] = src[i];
        }
        if (tid == 0) {
            sh.cand_n[0] = sh.cand_n[1] = 0;
            sh.lcount[0] = sh.lcount[1] = 0;
            sh.fpick[0] = sh.fpick[1] = -INFINITY;
        }
        for (int i = tid; i < 2 * NB; i += NT) (&sh.hcnt[0][0])[i] = 0;
        __syncthreads();

        // ---- pass 1: maximum + online softmax sum, as the chunks land
        bool timed_out = false;
        auto pass1_row = [&](const T *s, int r, bool active) {
            float tm = -INFINITY, ts = 0.0f;
            const uint4 *vp = reinterpret_cast<const uint4 *>(s);
            for (int c = 0; c < NCH; ++c) {
                if (!mbar_wait_bounded(&sh.bar[buf][r][c], par)) timed_out = true;
                if (!active) continue;
                const int v0 = c * per_ch, v1 = min(nv, v0 + per_ch);
                for (int i = v0 + tid; i < v1; i += NT) {
                    float x[EPV];
                    unpack(vp[i], x);
                    float vm = x[0];
#pragma unroll
                    for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, x[e]);
                    if (vm > tm) {
                        ts *= ex2(__fmul_rn(tm - vm, c2));
                        tm = vm;
                    }
                    if (tm > -INFINITY) {
                        const float nmc = -tm * c2;
                        float a = 0.0f;
#pragma unroll
                        for (int e = 0; e < EPV; ++e) a += ex2(fmaf(x[e], c2, nmc));
                        ts += a;
                    }
                }
            }
            if (active)
                for (int i = nv * EPV + tid; i < n; i += NT) {
                    const float x = widen(s[i]);
                    if (x > -INFINITY) ms_merge(tm, ts, x, 1.0f, c2);
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xFFFFFFFFu, tm, o);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, ts, o);
                ms_merge(tm, ts, m2, s2, c2);
            }
            if (active && lane == 0) {
                sh.rf[r][warp] = tm;
                sh.rs[r][warp] = ts;
            }
        };
        pass1_row(sd0, 0, true);
        pass1_row(sd1, 1, nrows > 1);
        if (timed_out) atomicOr(&sh.flags, 1);
        __syncthreads();
        if (!started) {
            cluster_wait_acquire();  // every CTA of the cluster has started
            started = true;
        }

        // ---- E1: push this CTA's partials (and the draft's logits) to every CTA
        if (tid < nrows) {
            const int r = tid;
            float mv = -INFINITY, sv = 0.0f;
            for (int w = 0; w < NW; ++w) ms_merge(mv, sv, sh.rf[r][w], sh.rs[r][w], c2);
            const float xd =
                d_here ? widen((r == 0 ? sd0 : sd1)[static_cast<int64_t>(d) - lo64]) : 0.0f;
            for (uint32_t c = 0; c < C; ++c) {
                st_peer_f32(peer_addr(smem_addr(&sh.x_m[ep][rank][r]), c), mv);
                st_peer_f32(peer_addr(smem_addr(&sh.x_s[ep][rank][r]), c), sv);
                if (d_here) st_peer_f32(peer_addr(smem_addr(&sh.x_d[ep][r]), c), xd);
            }
        }
        cluster_sync();  // B1

        // ---- row statistics (every CTA, identical)
        if (tid < nrows) {
            const int r = tid;
            float mv = -INFINITY, sv = 0.0f;
            for (uint32_t c = 0; c < C; ++c) ms_merge(mv, sv, sh.x_m[ep][c][r], sh.x_s[ep][c][r], c2);
            float mx = -INFINITY;
            for (uint32_t c = 0; c < C; ++c) mx = fmaxf(mx, sh.x_m[ep][c][r]);
            if (sv > 0.0f && mv != mx) sv *= ex2(__fmul_rn(mv - mx, c2));
            sh.m[r] = mx;
            sh.deg[r] = !(mx > -INFINITY);
            sh.mode[r] = 0;
            sh.theta[r] = -INFINITY;
            sh.Z[r] = sv;
            // for top-p alone, a kept token weighs at least (1 - p) Z / V: the tokens below
            // that level weigh less than (1 - p) Z together
            float zc = -static_cast<float>(ZR);
            if (!k_on && sv > 0.0f) {
                const float lvl = __log2f((1.0f - pp) * sv / static_cast<float>(V));
                zc = fmaxf(zc, lvl - 2.0f / R);
            }
            sh.zcut[r] = zc;
        }
        __syncthreads();

        if (k_on || p_on) {
            // ---- pass 2: counts over fine z bins for the elements that can hold the boundary
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r >= nrows || sh.deg[r]) continue;
                const float m = sh.m[r], zcut = sh.zcut[r];
                uint32_t *h = sh.hcnt[r];
                for_each_elem(r == 0 ? sd0 : sd1, n, [&](float x, int) {
                    const float z = zval(x, m, c2);
                    if (z > zcut) atomicAdd(&h[zbin(z)], 1u);
                });
            }
            __syncthreads();
            // ---- E2a: reduce-scatter, push local bins to their owner CTA
            const int RS = (NB + C - 1) / C;
            for (int idx = tid; idx < nrows * NB; idx += NT) {
                const int r = idx / NB, bn = idx - r * NB;
                const int owner = bn / RS, kq = bn - owner * RS;
                st_peer_u32(peer_addr(smem_addr(&sh.u.in[r][static_cast<int>(rank) * RS + kq]), owner),
                            sh.hcnt[r][bn]);
            }
            cluster_sync();  // B2a
            // ---- E2b: sum the owned bins and broadcast them
            for (int idx = tid; idx < nrows * RS; idx += NT) {
                const int r = idx / RS, kq = idx - r * RS;
                const int bn = static_cast<int>(rank) * RS + kq;
                if (bn >= NB) continue;
                uint32_t cs = 0;
                for (uint32_t c = 0; c < C; ++c) cs += sh.u.in[r][c * RS + kq];
                for (uint32_t c = 0; c < C; ++c)
                    st_peer_u32(peer_addr(smem_addr(&sh.hcnt[r][bn]), c), cs);
            }
            cluster_sync();  // B2b

            // ---- plan per row: the bin range that holds the boundary, or the exact search
            if (warp < nrows) {
                const int r = warp;
                if (!sh.deg[r]) {
                    int32_t b1 = 0, b2 = 0;
                    bool slow = false;
                    if (k_on) {
                        count_search(sh.hcnt[r], static_cast<uint32_t>(kk), &sh.pick[r]);
                        const int32_t bk = sh.pick[r];
                        __syncwarp();
                        slow = bk >= NB;
                        b1 = 0;  // every bin up to the k-th value; top-p then works inside them
                        b2 = bk;
                    } else {
                        weight_search(sh.hcnt[r], pp * sh.Z[r], &sh.pick[r], &sh.pick[2 + r]);
                        b1 = sh.pick[r];
                        b2 = sh.pick[2 + r];
                        __syncwarp();
                        if (b1 >= NB) slow = true;
                        if (b2 >= NB) b2 = NB - 1;
                    }
                    uint32_t inr = 0;
                    if (!slow)
                        for (int t = lane; t < NB; t += 32)
                            if (t >= b1 && t <= b2) inr += sh.hcnt[r][t];
                    inr = warp_sum_u32(inr);
                    if (inr > static_cast<uint32_t>(CAP)) slow = true;
                    if (lane == 0) {
                        sh.mode[r] = slow ? 2 : 1;
                        sh.b1[r] = b1;
                        sh.b2[r] = b2;
                        sh.ncand[r] = inr;
                    }
                }
            }
            __syncthreads();

            // ---- gather the boundary candidates into every CTA, with the exact weight of
            // everything above them (E3)
            const bool any_fast = sh.mode[0] == 1 || (nrows > 1 && sh.mode[1] == 1);
            if (any_fast) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (r >= nrows) break;
                    float above = 0.0f;
                    if (sh.mode[r] == 1) {
                        // compact this CTA's candidates locally, then push them as one block
                        const float m = sh.m[r];
                        const int b1 = sh.b1[r], b2 = sh.b2[r];
                        for_each_elem(r == 0 ? sd0 : sd1, n, [&](float x, int i) {
                            const float z = zval(x, m, c2);
                            const int bn = zbin(z);
                            if (bn < b1) {
                                above += ex2(z);
                            } else if (bn <= b2) {
                                const uint32_t slot = atomicAdd(&sh.lcount[r], 1u);
                                if (slot < static_cast<uint32_t>(CAP)) {
                                    sh.lc[r][slot].v = x;
                                    sh.lc[r][slot].idx = static_cast<uint32_t>(lo64 + i);
                                    sh.lw[r][slot] = fix31(ex2(z));
                                }
                            }
                        });
                    }
                    const unsigned long long ma = block_sum_u64(fix_sum(above), sh.ru[r]);
                    if (sh.mode[r] == 1) {
                        const uint32_t nl = min(sh.lcount[r], static_cast<uint32_t>(CAP));
                        __syncthreads();
                        if (tid == 0)
                            sh.lcount[r] = nl ? atom_peer_add_u32(peer_addr(smem_addr(&sh.cand_n[r]), 0), nl) : 0u;
                        __syncthreads();
                        const uint32_t base = sh.lcount[r];
                        for (uint32_t q = tid; q < nl * C; q += NT) {
                            const uint32_t i = q / C, c = q - i * C, slot = base + i;
                            if (slot < static_cast<uint32_t>(CAP)) {
                                const Cand cv = sh.lc[r][i];
                                st_peer_u64(peer_addr(smem_addr(&sh.u.cd.c[r][slot]), c),
                                            *reinterpret_cast<const unsigned long long *>(&cv));
                                st_peer_u64(peer_addr(smem_addr(&sh.u.cd.w[r][slot]), c), sh.lw[r][i]);
                            }
                        }
                    }
                    if (tid == 0)
                        for (uint32_t c = 0; c < C; ++c)
                            st_peer_u64(peer_addr(smem_addr(&sh.ma_x[rank][r]), c), ma);
                }
                cluster_sync();  // B3
                // ---- exact thresholds: sort the candidates by value (descending) and scan
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (r >= nrows || sh.mode[r] != 1) continue;
                    const int nc = static_cast<int>(sh.ncand[r]);
                    const Cand *cd = sh.u.cd.c[r];
                    const unsigned long long *cw = sh.u.cd.w[r];
                    unsigned long long MA = 0;
                    for (uint32_t c = 0; c < C; ++c) MA += sh.ma_x[c][r];
                    // bitonic sort of (value key, slot), one key per thread; strides below
                    // 32 exchange through shuffles, wider ones through shared memory
                    unsigned long long key =
                        tid < nc ? (static_cast<unsigned long long>(order_key(cd[tid].v)) << 32) |
                                       static_cast<uint32_t>(tid)
                                 : 0ull;
                    for (int kb = 2; kb <= NT; kb <<= 1) {
                        for (int jb = kb >> 1; jb > 0; jb >>= 1) {
                            unsigned long long other;
                            if (jb >= 32) {
                                __syncthreads();
                                sh.skey[tid] = key;
                                __syncthreads();
                                other = sh.skey[tid ^ jb];
                            } else {
                                other = __shfl_xor_sync(0xFFFFFFFFu, key, jb);
                            }
                            const bool lower = (tid & jb) == 0;
                            const bool desc = (tid & kb) == 0;
                            key = (lower == desc) ? max(key, other) : min(key, other);
                        }
                    }
                    const bool real = tid < nc;
                    const uint32_t slot = static_cast<uint32_t>(key);
                    const float v = real ? cd[slot].v : -INFINITY;
                    const unsigned long long w = real ? cw[slot] : 0ull;
                    __syncthreads();
                    sh.sval[tid] = v;
                    // top-k: the k-th largest value (no element lies above the candidates)
                    if (k_on && tid == kk - 1) sh.fpick[r] = v;
                    __syncthreads();
                    const float thk = k_on ? sh.fpick[r] : -INFINITY;
                    const unsigned long long wk = (real && v >= thk) ? w : 0ull;
                    // weight strictly above each value: the exclusive prefix of the weights at
                    // the first position of its tie group (sorted descending)
                    const unsigned long long excl = block_excl_scan_u64(wk, sh.scan);
                    const int32_t headpos = (tid == 0 || sh.sval[tid - 1] != v) ? tid : -1;
                    const int32_t first = block_incl_max_i32(headpos, sh.scani);
                    sh.skey[tid] = excl;
                    const unsigned long long zk = MA + block_sum_u64(wk, sh.ru[r]);
                    if (tid == 0) {
                        const double t = k_on ? static_cast<double>(pp) * static_cast<double>(zk)
                                              : static_cast<double>(pp) * static_cast<double>(sh.Z[r]) *
                                                    static_cast<double>(FX);
                        sh.tgt[r] = static_cast<unsigned long long>(ceil(t));
                    }
                    __syncthreads();
                    const unsigned long long above = MA + sh.skey[first];
                    const bool kept = real && v >= thk && (!p_on || above < sh.tgt[r]);
                    int32_t lastk = kept ? tid : -1;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        lastk = max(lastk, __shfl_xor_sync(0xFFFFFFFFu, lastk, o));
                    __syncthreads();
                    if (lane == 0) sh.scani[warp] = lastk;
                    __syncthreads();
                    int32_t lk = -1;
                    for (int wq = 0; wq < NW; ++wq) lk = max(lk, sh.scani[wq]);
                    const float th = sh.sval[lk < 0 ? 0 : lk];  // the smallest kept value
                    const unsigned long long zf =
                        MA + block_sum_u64((real && v >= th) ? wk : 0ull, sh.ru[r]);
                    if (tid == 0) {
                        sh.theta[r] = th;
                        sh.Z[r] = static_cast<float>(static_cast<double>(zf) * INV_FX);
                    }
                    __syncthreads();
                }
            }

            // ---- exact bisection over value keys (boundary outside the binned range, or too
            // many elements in its bins); both rows advance in lockstep, one barrier a step
            const bool any_slow = sh.mode[0] == 2 || (nrows > 1 && sh.mode[1] == 2);
            if (any_slow) {
                int parity = 0;
                // F(t) per row: count (wt = 0) or fixed-point weight (wt = 1) of the elements
                // with key >= max(t, floor); returns the cluster-wide sums
                auto eval = [&](const uint32_t t[2], const uint32_t fl[2], int wt,
                                unsigned long long out[2]) {
                    unsigned long long acc[2] = {0, 0};
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        if (r >= nrows || sh.mode[r] != 2) continue;
                        const float m = sh.m[r];
                        const uint32_t lim = max(t[r], fl[r]);
                        float a = 0.0f;
                        uint32_t cnum = 0;
                        for_each_elem(r == 0 ? sd0 : sd1, n, [&](float x, int) {
                            if (order_key(x) >= lim) {
                                if (wt) a += ex2(zval(x, m, c2));
                                else ++cnum;
                            }
                        });
                        acc[r] = wt ? fix_sum(a) : static_cast<unsigned long long>(cnum);
                    }
                    const unsigned long long s0 = block_sum_u64(acc[0], sh.ru[0]);
                    const unsigned long long s1 = block_sum_u64(acc[1], sh.ru[1]);
                    if (tid < 2)
                        for (uint32_t c = 0; c < C; ++c)
                            st_peer_u64(peer_addr(smem_addr(&sh.sx[parity][tid][rank]), c),
                                        tid == 0 ? s0 : s1);
                    cluster_sync();
                    for (int r = 0; r < 2; ++r) {
                        unsigned long long sum = 0;
                        for (uint32_t c = 0; c < C; ++c) sum += sh.sx[parity][r][c];
                        out[r] = sum;
                    }
                    parity ^= 1;
                };
                // largest key t with F(t) >= need, by bisection over the 32-bit key space
                auto search = [&](const uint32_t fl[2], int wt, const unsigned long long need[2],
                                  uint32_t res_t[2]) {
                    uint32_t lo[2] = {0u, 0u}, hi[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
                    for (int it = 0; it < 32; ++it) {
                        uint32_t mid[2];
                        for (int r = 0; r < 2; ++r)
                            mid[r] = lo[r] + static_cast<uint32_t>((static_cast<uint64_t>(hi[r]) - lo[r] + 1) / 2);
                        unsigned long long f[2];
                        eval(mid, fl, wt, f);
                        for (int r = 0; r < 2; ++r) {
                            if (lo[r] >= hi[r]) continue;
                            if (f[r] >= need[r]) lo[r] = mid[r];
                            else hi[r] = mid[r] - 1;
                        }
                    }
                    res_t[0] = lo[0];
                    res_t[1] = lo[1];
                };
                uint32_t zero[2] = {0u, 0u}, thk[2] = {0u, 0u}, th[2] = {0u, 0u};
                if (k_on) {
                    const unsigned long long need[2] = {static_cast<unsigned long long>(kk),
                                                        static_cast<unsigned long long>(kk)};
                    search(zero, 0, need, thk);
                }
                th[0] = thk[0];
                th[1] = thk[1];
                if (p_on) {
                    unsigned long long zk[2] = {0, 0};
                    if (k_on) eval(thk, zero, 1, zk);
                    unsigned long long need[2];
                    for (int r = 0; r < 2; ++r) {
                        const double t = k_on ? static_cast<double>(pp) * static_cast<double>(zk[r])
                                              : static_cast<double>(pp) *
                                                    static_cast<double>(sh.Z[r < nrows ? r : 0]) *
                                                    static_cast<double>(FX);
                        need[r] = static_cast<unsigned long long>(ceil(t));
                        if (need[r] == 0) need[r] = 1;
                    }
                    search(thk, 1, need, th);
                }
                unsigned long long zf[2];
                eval(th, zero, 1, zf);
                if (tid < nrows && sh.mode[tid] == 2) {
                    sh.theta[tid] = key_to_float(th[tid]);
                    sh.Z[tid] = static_cast<float>(static_cast<double>(zf[tid]) * INV_FX);
                }
                __syncthreads();
            }
        }
        if (tid < nrows) sh.invZ[tid] = 1.0f / sh.Z[tid];
        __syncthreads();

        // ---- accept test
        uint32_t uw[4] = {static_cast<uint32_t>(b), static_cast<uint32_t>(j), 0u, 0u};
        philox(uw, static_cast<uint32_t>(P.seed), static_cast<uint32_t>(P.seed >> 32));
        const float u_acc = word_uniform(uw[0]), u_smp = word_uniform(uw[1]);

        // membership and probability of a token in the target (0) and draft (1) rows
        const float m0 = sh.m[0], m1 = sh.m[1], th0 = sh.theta[0], th1 = sh.theta[1];
        const float iz0 = sh.invZ[0], iz1 = sh.invZ[1];
        const bool deg0 = sh.deg[0], deg1 = sh.deg[1];
        auto prob0 = [&](float x, int64_t idx) -> float {
            if (deg0) return idx == 0 ? 1.0f : 0.0f;
            return x >= th0 ? ex2(zval(x, m0, c2)) * iz0 : 0.0f;
        };
        auto prob1 = [&](float x, int64_t idx) -> float {
            if (deg1) return idx == 0 ? 1.0f : 0.0f;
            return x >= th1 ? ex2(zval(x, m1, c2)) * iz1 : 0.0f;
        };

        bool accept = false;
        float pt = 0.0f, pd = 0.0f;
        if (j < D && dvalid) {
            const float xt = sh.x_d[ep][0], xq = sh.x_d[ep][1];
            const bool in_p = deg0 ? d == 0 : xt >= th0;
            const bool in_q = deg1 ? d == 0 : xq >= th1;
            pt = prob0(xt, d);
            pd = prob1(xq, d);
            if (!in_p) {
                accept = false;
            } else if (!in_q) {
                accept = true;
            } else {
                float ratio;
                if (deg0 || deg1)
                    ratio = pt / pd;
                else
                    ratio = ex2(__fmul_rn((xt - m0) - (xq - m1), c2)) * (sh.Z[1] / sh.Z[0]);
                accept = u_acc <= ratio;
            }
        }

        // ---- draw (a rejected draft's residual, or the bonus).  Weights in fixed point,
        // summed as integers: the cumulative sums at every level (lane, warp, CTA, cluster)
        // are exact and agree with one another.  Each warp owns a contiguous run of vectors;
        // within it a lane takes consecutive vectors, so (step, lane, element) is ascending
        // id order.
        UnitResult *res = P.res + u;
        const bool draw = (j == D) || !accept;
        if (draw) {
            int wmode = (j == D) ? 1 : 0;  // 0: max(0, p - q), 1: p
            const int nvw = (((n + EPV - 1) / EPV) + NW - 1) / NW;  // vectors per warp
            const int wv0 = warp * nvw, wv1 = wv0 + nvw;
            auto weights = [&](int vi, uint32_t (&w)[EPV]) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) w[e] = 0u;
                const int i0 = vi * EPV;
                if (vi >= wv1 || i0 >= n) return;
                float x[EPV], y[EPV];
                if (i0 + EPV <= n) {
                    unpack(reinterpret_cast<const uint4 *>(sd0)[vi], x);
                    if (wmode == 0) unpack(reinterpret_cast<const uint4 *>(sd1)[vi], y);
                } else {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        x[e] = i0 + e < n ? widen(sd0[i0 + e]) : -INFINITY;
                        y[e] = (wmode == 0 && i0 + e < n) ? widen(sd1[i0 + e]) : -INFINITY;
                    }
                }
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (i0 + e >= n) break;
                    const int64_t gi = lo64 + i0 + e;
                    float p = prob0(x[e], gi);
                    if (p > 0.0f && wmode == 0) p = fmaxf(p - prob1(y[e], gi), 0.0f);
                    w[e] = fix31(p);
                }
            };
            for (int attempt = 0; attempt < 2; ++attempt) {
                unsigned long long acc = 0;
                for (int vq = wv0 + lane; vq < wv1; vq += 32) {
                    uint32_t w[EPV];
                    weights(vq, w);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) acc += w[e];
                }
                acc = warp_sum_u64(acc);
                if (lane == 0) sh.w_sum[warp] = acc;
                __syncthreads();
                if (tid == 0) {
                    unsigned long long cs = 0;
                    for (int wq = 0; wq < NW; ++wq) cs += sh.w_sum[wq];
                    for (uint32_t c = 0; c < C; ++c)
                        st_peer_u64(peer_addr(smem_addr(&sh.dr_R[attempt][rank]), c), cs);
                }
                cluster_sync();  // B4
                const unsigned long long *dR = sh.dr_R[attempt];
                unsigned long long Rt = 0;
                for (uint32_t c = 0; c < C; ++c) Rt += dR[c];
                if (Rt > 0 || wmode == 1) {
                    // smallest id whose cumulative weight exceeds u_smp * R; a cumulative
                    // integer sum S exceeds u_smp * R exactly when S > floor(u_smp * R)
                    const unsigned long long tt = static_cast<unsigned long long>(
                        floor(static_cast<double>(u_smp) * static_cast<double>(Rt)));
                    uint32_t cs = C - 1;
                    unsigned long long before = 0;
                    for (uint32_t c = 0; c < C; ++c) {
                        if (before + dR[c] > tt) {
                            cs = c;
                            break;
                        }
                        before += dR[c];
                    }
                    if (cs == C - 1) {
                        before = 0;
                        for (uint32_t c = 0; c + 1 < C; ++c) before += dR[c];
                    }
                    if (rank == cs) {
                        int ws = NW - 1;
                        unsigned long long wb = before;
                        for (int wq = 0; wq < NW; ++wq) {
                            if (wb + sh.w_sum[wq] > tt) {
                                ws = wq;
                                break;
                            }
                            wb += sh.w_sum[wq];
                        }
                        if (ws == NW - 1) {
                            wb = before;
                            for (int wq = 0; wq + 1 < NW; ++wq) wb += sh.w_sum[wq];
                        }
                        if (warp == ws) {
                            unsigned long long a = wb;
                            int32_t tok = -1, lastpos = -1;
                            for (int v0 = wv0; v0 < wv1 && tok < 0; v0 += 32) {
                                uint32_t w[EPV];
                                weights(v0 + lane, w);
                                unsigned long long own = 0;
#pragma unroll
                                for (int e = 0; e < EPV; ++e) own += w[e];
                                unsigned long long incl = own;
#pragma unroll
                                for (int o = 1; o < 32; o <<= 1) {
                                    const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                                    if (lane >= o) incl += y;
                                }
                                const unsigned hitm =
                                    __ballot_sync(0xFFFFFFFFu, own > 0 && a + incl > tt);
                                const unsigned posm = __ballot_sync(0xFFFFFFFFu, own > 0);
                                // per lane: its first element past the target, its last positive one
                                int first_e = EPV - 1, last_e = 0;
                                {
                                    unsigned long long cum = a + incl - own;
                                    int f = -1;
#pragma unroll
                                    for (int e = 0; e < EPV; ++e) {
                                        cum += w[e];
                                        if (w[e] > 0) last_e = e;
                                        if (f < 0 && w[e] > 0 && cum > tt) f = e;
                                    }
                                    if (f >= 0) first_e = f;
                                }
                                if (posm) {
                                    const int ll = 31 - __clz(posm);
                                    lastpos = (v0 + ll) * EPV + __shfl_sync(0xFFFFFFFFu, last_e, ll);
                                }
                                if (hitm) {
                                    const int hl = __ffs(hitm) - 1;
                                    tok = (v0 + hl) * EPV + __shfl_sync(0xFFFFFFFFu, first_e, hl);
                                }
                                a += __shfl_sync(0xFFFFFFFFu, incl, 31);
                            }
                            if (tok < 0) tok = lastpos < 0 ? 0 : lastpos;
                            if (lane == 0) res->token = static_cast<int32_t>(lo64 + tok);
                        }
                    }
                    break;
                }
                wmode = 1;  // the residual is identically zero: draw from p instead
                __syncthreads();
            }
        }

        if (rank == 0 && tid == 0) {
            res->flags = accept ? 1 : 0;
            res->pt = pt;
            res->pd = pd;
            if (!draw) res->token = -1;
            if (P.status && j < D && !dvalid) atomicOr(P.status, MTPSPEC_STATUS_BAD_DRAFT_ID);
        }

        // ---- this buffer is free: bring in the unit after the next one
        const int64_t un = next_unit(u);
        __syncthreads();
        if (P.nbuf == 2 && tid == 0 && un >= 0) {
            const int64_t un2 = next_unit(un);
            if (un2 >= 0) {
                fence_proxy_async_smem();
                issue(un2, buf);
            }
        } else if (P.nbuf == 1 && tid == 0 && un >= 0) {
            fence_proxy_async_smem();
        }
        u = un;
    }
    if (tid == 0 && (sh.flags & 1) && P.status) atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
    if (!started) {
        cluster_wait_acquire();  // a cluster with no unit still completes its start barrier
    }
}

// One thread per row: the first rejected position decides what the row emits.
__global__ void k_verify_finalize(const UnitResult *__restrict__ res, const int32_t *__restrict__ d,
                                  int64_t B, int32_t D, int32_t *__restrict__ out,
                                  int32_t *__restrict__ num_accepted, float *__restrict__ p_target,
                                  float *__restrict__ p_draft) {
    const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const UnitResult *r = res + b * (D + 1);
    int a = D;
    for (int jj = 0; jj < D; ++jj) {
        const UnitResult u = r[jj];
        if (p_target) p_target[b * D + jj] = u.pt;
        if (p_draft) p_draft[b * D + jj] = u.pd;
        if (a == D && !(u.flags & 1)) a = jj;
    }
    int32_t *o = out + b * (D + 1);
    for (int jj = 0; jj < a; ++jj) o[jj] = d[b * D + jj];
    o[a] = r[a].token;
    for (int jj = a + 1; jj <= D; ++jj) o[jj] = -1;
    num_accepted[b] = a;
}

}  // namespace vs

// ---------------------------------------------------------------- host side

static int verify_cluster_size(int64_t V) {
    if (const char *e = getenv("MTPSPEC_VERIFY_CLUSTER")) {
        const int c = atoi(e);
        if (c >= 1 && c <= vs::MAXC) return c;
    }
    int C = 1;
    while (C < 8 && V / (2 * C) >= 2048) C *= 2;
    return C;
}

static int64_t verify_slice(int64_t V, int C) {
    int64_t s = (V + C - 1) / C;
    return (s + 15) & ~static_cast<int64_t>(15);
}

size_t verify_workspace_bytes(int64_t B, int32_t D) {
    return static_cast<size_t>(B) * static_cast<size_t>(D + 1) * sizeof(vs::UnitResult);
}

constexpr size_t kSmemLimit = 227u * 1024u;

static size_t verify_smem_bytes(int64_t slice, size_t es, int nbuf) {
    const size_t head = (sizeof(vs::Shared) + 127) & ~static_cast<size_t>(127);
    const size_t row = ((static_cast<size_t>(slice) * es) + 127) & ~static_cast<size_t>(127);
    return head + 2 * static_cast<size_t>(nbuf) * row;
}

bool verify_fits(int64_t V, size_t elem_bytes) {
    const int C = verify_cluster_size(V);
    return verify_smem_bytes(verify_slice(V, C), elem_bytes, 1) <= kSmemLimit;
}

// Resident clusters of the persistent kernel for one configuration (cached).
template <typename T>
static int resident_clusters(int C, size_t smem) {
    static std::mutex mu;
    static int cache_c[8] = {0}, cache_v[8] = {0};
    static size_t cache_s[8] = {0};
    static int dev_of[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < 8; ++i)
        if (dev_of[i] == dev && cache_c[i] == C && cache_s[i] == smem) return cache_v[i];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
    cfg.blockDim = dim3(vs::NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, vs::k_verify_persistent<T>, &cfg) != cudaSuccess || n < 1)
        n = 1;
    for (int i = 0; i < 8; ++i)
        if (dev_of[i] == -1 || i == 7) {
            dev_of[i] = dev;
            cache_c[i] = C;
            cache_s[i] = smem;
            cache_v[i] = n;
            break;
        }
    return n;
}

template <typename T>
static cudaError_t launch_verify_persistent(vs::Params p, int C, cudaStream_t stream) {
    p.nbuf = verify_smem_bytes(p.slice, sizeof(T), 2) <= kSmemLimit ? 2 : 1;
    const size_t smem = verify_smem_bytes(p.slice, sizeof(T), p.nbuf);
    cudaError_t e = cudaFuncSetAttribute(vs::k_verify_persistent<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(vs::k_verify_persistent<T>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const int64_t units = p.B * (p.D + 1);
    int64_t G = resident_clusters<T>(C, smem);
    if (G > units) G = units;
    p.G = static_cast<int32_t>(G);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G * C), 1, 1);
    cfg.blockDim = dim3(vs::NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, vs::k_verify_persistent<T>, p);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_verify_sample(const VerifySampleArgs &a, cudaStream_t stream) {
    const int C = verify_cluster_size(a.V);
    vs::Params p;
    p.T = a.target;
    p.Q = a.draft;
    p.d = a.draft_ids;
    p.tau = a.temperature;
    p.topk = a.top_k;
    p.topp = a.top_p;
    p.seed = a.seed;
    p.B = a.B;
    p.D = a.D;
    p.V = a.V;
    p.slice = verify_slice(a.V, C);
    p.nbuf = 2;
    p.G = 1;
    p.res = static_cast<vs::UnitResult *>(a.workspace);
    p.status = a.status;
    // the sampled rows, then (beside them) the greedy rows, then the per-row finalize
    cudaError_t e = a.dtype == MTPSPEC_F32 ? launch_verify_persistent<float>(p, C, stream)
                                           : launch_verify_persistent<uint16_t>(p, C, stream);
    if (e != cudaSuccess) return e;
    e = run_verify_greedy_rows(a, stream);
    if (e != cudaSuccess) return e;
    vs::k_verify_finalize<<<static_cast<unsigned>((a.B + 127) / 128), 128, 0, stream>>>(
        static_cast<const vs::UnitResult *>(a.workspace), a.draft_ids, a.B, a.D, a.out_tokens,
        a.num_accepted, a.p_target, a.p_draft);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace mtpspec

// ---------------------------------------------------------------- fixed-scratch variant

namespace mtpspec {

// Scratch of the fixed-scratch entry point: the per-unit records the two kernels of a
// sampling verification hand over, for up to kStaticVerifyUnits units (B * (D + 1)).  It
// lives in the library's own device memory, so that entry point allocates nothing; every
// GPU that loads the library holds these 1 MiB until the process exits.  All calls on a
// device share it: each call overwrites every record it reads, so nothing needs clearing,
// and calls whose work overlaps on the GPU (other streams, other threads) race on it.
static __device__ __align__(256) unsigned char g_verify_scratch[kStaticVerifyUnits * 16];
static_assert(sizeof(vs::UnitResult) == 16, "one 16-byte record per unit");

static std::mutex g_scratch_mu;
static void *g_scratch_ptr[64] = {nullptr};

cudaError_t run_verify_sample_static(VerifySampleArgs a, cudaStream_t stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void *ptr = nullptr;
    {
        // once per device, with that device current: the device address of the array
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            e = cudaGetSymbolAddress(&ptr, g_verify_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_ptr[dev] = ptr;
        }
        ptr = g_scratch_ptr[dev];
    }
    a.workspace = ptr;
    return run_verify_sample(a, stream);
}

}  // namespace mtpspec
