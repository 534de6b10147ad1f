// Speculative-sampling verification: temperature -> top-k -> top-p filtering of target and
// draft logits, the accept test U <= p/q, the residual draw at the first rejection and the
// bonus draw ("MPT (MTP, Multi-Token Prediction) 原理详解", section 三 stage 3 "rejection
// sampling" and stage 4; "The decoding loop and MTP", "Why a hand-written decoding loop" for
// the filters and "MTP speculative decoding" items 2-3 for the drawn replacement and the
// extra token).
//
// Work unit: one (row b, position j) pair, j = 0..D.  Each unit is one thread-block cluster
// of C CTAs; CTA r owns the contiguous slice [r*slice, (r+1)*slice) of the vocabulary and
// copies its slice of the target row (and, for j < D, of the draft row) into shared memory
// with bulk asynchronous copies, so every logit is read from HBM exactly once.  Everything
// after that runs on chip:
//   pass 1   maximum and online softmax sum (argmax for greedy rows) as the chunks land
//   E1       per-CTA partials meet in every CTA through distributed shared memory
//   pass 2   (top-k / top-p) counts over fine bins of z = (x - max) * log2(e) / tau,
//            R bins per unit of z, only for elements that can hold the boundary; the counts
//            are reduce-scattered and re-broadcast across the cluster (E2)
//   plan     the bins that must hold the boundary, from exact counts (top-k) or from
//            per-bin weight bounds count * 2^(-b/R) (top-p)
//   gather   elements of those bins are pushed to every CTA with their weights, and the
//            exact weight of everything above them is summed (E3); each CTA then finds
//            the thresholds by exact rank / weight-above counts over the candidates.  If
//            the boundary is outside the binned range or too many elements fall in its
//            bins, an exact bisection over the 32-bit value keys replaces this step.
//   accept   p(d), q(d) and U_acc <= p/q (ratio formed with both maxima factored out)
//   draw     only for a rejected draft or the bonus position: draw weights in fixed point
//            (2^31 per unit of probability), per-warp sums in id order, CTA sums exchanged
//            (E4), and the CTA holding the target walks its slice to the token.
// A per-row finalize kernel then takes the first rejected position.
//
// Weight sums are formed per thread in fp32 over a fixed set of elements, converted once
// to 64-bit fixed point and reduced as integers, so every sum is deterministic and the same
// in every CTA of a cluster.  Every decision is computed identically in every CTA from
// exchanged data, so all CTAs run the same sequence of cluster barriers.  Exchanges are
// pushes into the peers' shared memory before a barrier; after the last barrier a CTA only
// reads its own shared memory.  The bulk-copy barrier waits are bounded and raise
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
constexpr int CAP = 512;         // boundary candidates per row
constexpr int NCH = 4;           // bulk-copy chunks per row
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr float FX = 2147483648.0f;  // 2^31: fixed-point scale of weights (weights <= 1)
constexpr double INV_FX = 1.0 / 2147483648.0;
constexpr float BOUND_SLACK = 4e-5f;  // relative slack of the per-bin weight bounds

struct UnitResult {
    int32_t flags;  // bit 0: draft accepted
    int32_t token;  // greedy pick, or the draw (residual / bonus) of this unit, or -1
    float pt;       // p_j(d_j)
    float pd;       // q_j(d_j)
};

struct Cand {
    float v;       // logit
    uint32_t idx;  // token id
};

struct __align__(16) Shared {
    unsigned long long bar[2][NCH];
    // block reductions
    float rf[2][NW];
    float rs[2][NW];
    int32_t ri[2][NW];
    unsigned long long ru[2][NW];
    // E1: partials of every CTA (pushed by each CTA into all peers)
    float x_m[MAXC][2];
    float x_s[MAXC][2];
    int32_t x_i[MAXC][2];
    float x_d[2];  // the draft token's logit in each row, pushed by the CTA that owns it
    // per-row state, identical in every CTA of the cluster
    float c2;                 // log2(e) / tau
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
    uint32_t cand_n[2];                // slot allocator, used in CTA 0
    unsigned long long ma_x[MAXC][2];  // per-CTA fixed-point weight above bin b1
    // exact bisection exchange (double-buffered by iteration parity)
    unsigned long long sx[2][2][MAXC];
    // draws
    unsigned long long dr_R[2][MAXC];  // per draw attempt: each CTA's fixed-point weight
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

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
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
// Wait for phase 0 of a bulk-copy barrier; false after WAIT_LIMIT polls.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar) {
    for (uint32_t it = 0; it < WAIT_LIMIT; ++it)
        if (mbar_try_wait(bar, 0)) return true;
    return false;
}
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
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

// First bin whose cumulative count reaches `need` (NB if none); one warp, lane 0 writes.
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
    UnitResult *res;
    int32_t *status;
};

// ---------------------------------------------------------------- the unit kernel

template <typename T>
__global__ void __launch_bounds__(NT, 2) k_verify_units(const Params P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Shared &sh = *reinterpret_cast<Shared *>(smem_raw);
    constexpr int EPV = elems_per_16B<T>::value;
    const size_t data_off = (sizeof(Shared) + 127) & ~static_cast<size_t>(127);
    const size_t row_bytes =
        ((static_cast<size_t>(P.slice) * sizeof(T)) + 127) & ~static_cast<size_t>(127);
    T *const sd0 = reinterpret_cast<T *>(smem_raw + data_off);
    T *const sd1 = reinterpret_cast<T *>(smem_raw + data_off + row_bytes);

    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int64_t unit = cluster_index();
    const int D = P.D;
    const int64_t b = unit / (D + 1);
    const int j = static_cast<int>(unit - b * (D + 1));
    const int64_t V = P.V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const float tau = P.tau[b];
    const int32_t kk = P.topk ? P.topk[b] : 0;
    const float pp = P.topp ? P.topp[b] : 1.0f;
    const bool bad = !(tau >= 0.0f) || !(pp > 0.0f);
    const bool greedy = bad || tau == 0.0f;
    const bool has_q = !greedy && j < D;
    const int nrows = has_q ? 2 : 1;
    const bool k_on = !greedy && kk >= 1 && static_cast<int64_t>(kk) < V;
    const bool p_on = !greedy && pp < 1.0f;

    const int64_t lo64 = static_cast<int64_t>(rank) * P.slice;
    const int64_t rest = V - lo64;
    const int n = static_cast<int>(rest <= 0 ? 0 : (rest < P.slice ? rest : P.slice));
    const int32_t d = j < D ? P.d[b * D + j] : -1;
    const bool dvalid = d >= 0 && static_cast<int64_t>(d) < V;
    const bool d_here =
        dvalid && static_cast<int64_t>(d) >= lo64 && static_cast<int64_t>(d) < lo64 + n;

    const T *g0 = static_cast<const T *>(P.T) + (b * (D + 1) + j) * V + lo64;
    const T *g1 = has_q ? static_cast<const T *>(P.Q) + (b * D + j) * V + lo64 : nullptr;

    // ---- set-up: barriers, counters, histogram, the temperature scale
    if (tid == 0) {
        for (int r = 0; r < 2; ++r)
            for (int c = 0; c < NCH; ++c) mbar_init(&sh.bar[r][c], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh.cand_n[0] = sh.cand_n[1] = 0;
        sh.flags = 0;
        sh.fpick[0] = sh.fpick[1] = -INFINITY;
        sh.c2 = greedy ? 0.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(tau));
    }
    for (int i = tid; i < 2 * NB; i += NT) (&sh.hcnt[0][0])[i] = 0;
    __syncthreads();
    cluster_arrive_release();  // peers may touch this CTA's shared memory after the wait below
    pdl_launch_dependents();
    const float c2 = sh.c2;

    // ---- loads: bulk copies of the 16-byte-aligned body, plain loads for the rest
    const int nv = n / EPV;
    const bool bulk0 = nv > 0 && (reinterpret_cast<uintptr_t>(g0) & 15u) == 0;
    const bool bulk1 = has_q && nv > 0 && (reinterpret_cast<uintptr_t>(g1) & 15u) == 0;
    const int per_ch = (nv + NCH - 1) / NCH;
    if (tid == 0) {
        for (int r = 0; r < nrows; ++r) {
            if (!(r == 0 ? bulk0 : bulk1)) continue;
            T *dst = r == 0 ? sd0 : sd1;
            const T *src = r == 0 ? g0 : g1;
            for (int c = 0; c < NCH; ++c) {
                const int v0 = c * per_ch, v1 = min(nv, v0 + per_ch);
                if (v1 <= v0) continue;
                const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
                mbar_expect_tx(&sh.bar[r][c], bytes);
                bulk_copy_g2s(dst + v0 * EPV, src + v0 * EPV, bytes, &sh.bar[r][c]);
            }
        }
    }
    for (int i = (bulk0 ? nv * EPV : 0) + tid; i < n; i += NT) sd0[i] = g0[i];
    if (has_q)
        for (int i = (bulk1 ? nv * EPV : 0) + tid; i < n; i += NT) sd1[i] = g1[i];
    __syncthreads();

    // ---- pass 1: argmax (greedy) or maximum + online softmax sum, as the chunks land
    float tm[2] = {-INFINITY, -INFINITY}, ts[2] = {0.0f, 0.0f};
    ArgMax am{-INFINITY, -1};
    bool timed_out = false;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        const T *s = r == 0 ? sd0 : sd1;
        const bool bulk = r == 0 ? bulk0 : bulk1;
        const uint4 *vp = reinterpret_cast<const uint4 *>(s);
        for (int c = 0; c < NCH; ++c) {
            const int v0 = c * per_ch, v1 = min(nv, v0 + per_ch);
            if (bulk && v1 > v0 && !mbar_wait_bounded(&sh.bar[r][c])) timed_out = true;
            for (int i = v0 + tid; i < v1; i += NT) {
                float x[EPV];
                unpack(vp[i], x);
                if (greedy) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (x[e] > am.v || am.i < 0)
                            am = {x[e], static_cast<int32_t>(lo64 + i * EPV + e)};
                } else {
                    float vm = x[0];
#pragma unroll
                    for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, x[e]);
                    if (vm > tm[r]) {
                        ts[r] *= ex2(__fmul_rn(tm[r] - vm, c2));
                        tm[r] = vm;
                    }
                    if (tm[r] > -INFINITY) {
                        float a = 0.0f;
#pragma unroll
                        for (int e = 0; e < EPV; ++e) a += ex2(__fmul_rn(x[e] - tm[r], c2));
                        ts[r] += a;
                    }
                }
            }
        }
        for (int i = nv * EPV + tid; i < n; i += NT) {
            const float x = widen(s[i]);
            if (greedy) {
                if (x > am.v || am.i < 0) am = {x, static_cast<int32_t>(lo64 + i)};
            } else if (x > -INFINITY) {
                ms_merge(tm[r], ts[r], x, 1.0f, c2);
            }
        }
    }
    if (timed_out) atomicOr(&sh.flags, 1);

    // block reduction of the pass-1 partials
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        if (greedy) {
            am = warp_argmax(am);
            if (lane == 0) {
                sh.rf[r][warp] = am.v;
                sh.ri[r][warp] = am.i;
            }
        } else {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xFFFFFFFFu, tm[r], o);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, ts[r], o);
                ms_merge(tm[r], ts[r], m2, s2, c2);
            }
            if (lane == 0) {
                sh.rf[r][warp] = tm[r];
                sh.rs[r][warp] = ts[r];
            }
        }
    }
    __syncthreads();
    cluster_wait_acquire();  // every CTA of the cluster has started

    // ---- E1: push this CTA's partials (and the draft's logits) to every CTA
    if (tid < nrows) {
        const int r = tid;
        float mv = -INFINITY, sv = 0.0f;
        int32_t iv = -1;
        if (greedy) {
            ArgMax a{-INFINITY, -1};
            for (int w = 0; w < NW; ++w) a = argmax_merge(a, ArgMax{sh.rf[r][w], sh.ri[r][w]});
            mv = a.v;
            iv = a.i;
        } else {
            for (int w = 0; w < NW; ++w) ms_merge(mv, sv, sh.rf[r][w], sh.rs[r][w], c2);
        }
        const float xd =
            d_here ? widen((r == 0 ? sd0 : sd1)[static_cast<int64_t>(d) - lo64]) : 0.0f;
        for (uint32_t c = 0; c < C; ++c) {
            st_peer_f32(peer_addr(smem_addr(&sh.x_m[rank][r]), c), mv);
            st_peer_f32(peer_addr(smem_addr(&sh.x_s[rank][r]), c), sv);
            st_peer_u32(peer_addr(smem_addr(&sh.x_i[rank][r]), c), static_cast<uint32_t>(iv));
            if (d_here) st_peer_f32(peer_addr(smem_addr(&sh.x_d[r]), c), xd);
        }
    }
    cluster_sync();  // B1

    UnitResult *res = P.res + unit;
    if (greedy) {
        if (rank == 0 && tid == 0) {
            ArgMax a{-INFINITY, -1};
            for (uint32_t c = 0; c < C; ++c) a = argmax_merge(a, ArgMax{sh.x_m[c][0], sh.x_i[c][0]});
            const int32_t g = a.i < 0 ? 0 : a.i;
            UnitResult out;
            out.token = g;
            out.flags = (j < D && d == g) ? 1 : 0;
            out.pt = (j < D && d == g) ? 1.0f : 0.0f;
            out.pd = (j < D && dvalid) ? 1.0f : 0.0f;
            *res = out;
            if (P.status) {
                if (j < D && !dvalid) atomicOr(P.status, MTPSPEC_STATUS_BAD_DRAFT_ID);
                if (bad && j == 0) atomicOr(P.status, MTPSPEC_STATUS_BAD_PARAM);
                if (sh.flags & 1) atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
            }
        }
        return;
    }

    // ---- row statistics (every CTA, identical)
    if (tid < nrows) {
        const int r = tid;
        float mv = -INFINITY, sv = 0.0f;
        for (uint32_t c = 0; c < C; ++c) ms_merge(mv, sv, sh.x_m[c][r], sh.x_s[c][r], c2);
        float mx = -INFINITY;
        for (uint32_t c = 0; c < C; ++c) mx = fmaxf(mx, sh.x_m[c][r]);
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

    const bool need_filter = k_on || p_on;
    if (need_filter) {
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
            const int owner = bn / RS, k = bn - owner * RS;
            st_peer_u32(peer_addr(smem_addr(&sh.u.in[r][static_cast<int>(rank) * RS + k]), owner),
                        sh.hcnt[r][bn]);
        }
        cluster_sync();  // B2a
        // ---- E2b: sum the owned bins and broadcast them
        for (int idx = tid; idx < nrows * RS; idx += NT) {
            const int r = idx / RS, k = idx - r * RS;
            const int bn = static_cast<int>(rank) * RS + k;
            if (bn >= NB) continue;
            uint32_t cs = 0;
            for (uint32_t c = 0; c < C; ++c) cs += sh.u.in[r][c * RS + k];
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
                    const float m = sh.m[r];
                    const int b1 = sh.b1[r], b2 = sh.b2[r];
                    const uint32_t alloc = peer_addr(smem_addr(&sh.cand_n[r]), 0);
                    for_each_elem(r == 0 ? sd0 : sd1, n, [&](float x, int i) {
                        const float z = zval(x, m, c2);
                        const int bn = zbin(z);
                        if (bn < b1) {
                            above += ex2(z);
                        } else if (bn <= b2) {
                            const uint32_t slot = atom_peer_add_u32(alloc, 1u);
                            if (slot < static_cast<uint32_t>(CAP)) {
                                const uint32_t w = fix31(ex2(z));
                                const uint32_t gi = static_cast<uint32_t>(lo64 + i);
                                for (uint32_t c = 0; c < C; ++c) {
                                    st_peer_f32(peer_addr(smem_addr(&sh.u.cd.c[r][slot].v), c), x);
                                    st_peer_u32(peer_addr(smem_addr(&sh.u.cd.c[r][slot].idx), c), gi);
                                    st_peer_u64(peer_addr(smem_addr(&sh.u.cd.w[r][slot]), c), w);
                                }
                            }
                        }
                    });
                }
                const unsigned long long ma = block_sum_u64(fix_sum(above), sh.ru[r]);
                if (tid == 0)
                    for (uint32_t c = 0; c < C; ++c)
                        st_peer_u64(peer_addr(smem_addr(&sh.ma_x[rank][r]), c), ma);
            }
            cluster_sync();  // B3
            // ---- exact thresholds: rank and weight above each candidate
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r >= nrows || sh.mode[r] != 1) continue;
                const int nc = static_cast<int>(sh.ncand[r]);
                const Cand *cd = sh.u.cd.c[r];
                const unsigned long long *cw = sh.u.cd.w[r];
                unsigned long long MA = 0;
                for (uint32_t c = 0; c < C; ++c) MA += sh.ma_x[c][r];
                // top-k: the k-th largest value (every bin above the candidates is empty)
                float thk = -INFINITY;
                if (k_on) {
                    for (int i = tid; i < nc; i += NT) {
                        const float v = cd[i].v;
                        uint32_t gt = 0, ge = 0;
                        for (int t = 0; t < nc; ++t) {
                            gt += cd[t].v > v;
                            ge += cd[t].v >= v;
                        }
                        if (gt < static_cast<uint32_t>(kk) && ge >= static_cast<uint32_t>(kk))
                            sh.fpick[r] = v;  // every thread that finds it writes the same value
                    }
                    __syncthreads();
                    thk = sh.fpick[r];
                }
                float th = thk;
                if (p_on) {
                    unsigned long long zk = 0;
                    if (k_on) {
                        for (int i = tid; i < nc; i += NT)
                            if (cd[i].v >= thk) zk += cw[i];
                        zk = MA + block_sum_u64(zk, sh.ru[r]);
                    }
                    if (tid == 0) {
                        const double t = k_on ? static_cast<double>(pp) * static_cast<double>(zk)
                                              : static_cast<double>(pp) * static_cast<double>(sh.Z[r]) *
                                                    static_cast<double>(FX);
                        sh.tgt[r] = static_cast<unsigned long long>(ceil(t));
                    }
                    __syncthreads();
                    const unsigned long long tgt = sh.tgt[r];
                    // kept iff the weight strictly above is below the target: the threshold
                    // is the smallest kept value
                    float lowest = INFINITY;
                    for (int i = tid; i < nc; i += NT) {
                        const float v = cd[i].v;
                        if (v < thk) continue;
                        unsigned long long ab = MA;
                        for (int t = 0; t < nc; ++t)
                            if (cd[t].v > v && cd[t].v >= thk) ab += cw[t];
                        if (ab < tgt) lowest = fminf(lowest, v);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        lowest = fminf(lowest, __shfl_xor_sync(0xFFFFFFFFu, lowest, o));
                    if (lane == 0) sh.rf[r][warp] = lowest;
                    __syncthreads();
                    float l = INFINITY;
                    for (int w = 0; w < NW; ++w) l = fminf(l, sh.rf[r][w]);
                    th = l;
                }
                unsigned long long zf = 0;
                for (int i = tid; i < nc; i += NT)
                    if (cd[i].v >= th) zf += cw[i];
                zf = MA + block_sum_u64(zf, sh.ru[r]);
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
                    unsigned long long s = 0;
                    for (uint32_t c = 0; c < C; ++c) s += sh.sx[parity][r][c];
                    out[r] = s;
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
        const float xt = sh.x_d[0], xq = sh.x_d[1];
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

    // ---- draw (a rejected draft's residual, or the bonus).  Weights in fixed point, summed
    // as integers: the cumulative sums at every level (lane, warp, CTA, cluster) are exact
    // and agree with one another.  Each warp owns a contiguous run of vectors; within it a
    // lane takes consecutive vectors, so (step, lane, element) is ascending id order.
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
            for (int v = wv0 + lane; v < wv1; v += 32) {
                uint32_t w[EPV];
                weights(v, w);
#pragma unroll
                for (int e = 0; e < EPV; ++e) acc += w[e];
            }
            acc = warp_sum_u64(acc);
            if (lane == 0) sh.w_sum[warp] = acc;
            __syncthreads();
            if (tid == 0) {
                unsigned long long cs = 0;
                for (int w = 0; w < NW; ++w) cs += sh.w_sum[w];
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
                    for (int w = 0; w < NW; ++w) {
                        if (wb + sh.w_sum[w] > tt) {
                            ws = w;
                            break;
                        }
                        wb += sh.w_sum[w];
                    }
                    if (ws == NW - 1) {
                        wb = before;
                        for (int w = 0; w + 1 < NW; ++w) wb += sh.w_sum[w];
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
                            const unsigned hitm = __ballot_sync(0xFFFFFFFFu, own > 0 && a + incl > tt);
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
        if (P.status) {
            if (j < D && !dvalid) atomicOr(P.status, MTPSPEC_STATUS_BAD_DRAFT_ID);
            if (sh.flags & 1) atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
        }
    } else if (tid == 0 && (sh.flags & 1) && P.status) {
        atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
    }
}

// One thread per row: the first rejected position decides what the row emits.
__global__ void k_verify_finalize(const UnitResult *__restrict__ res, const int32_t *__restrict__ d,
                                  int64_t B, int32_t D, int32_t *__restrict__ out,
                                  int32_t *__restrict__ num_accepted, float *__restrict__ p_target,
                                  float *__restrict__ p_draft) {
    pdl_wait_primary();
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
    while (C < vs::MAXC && V / (2 * C) >= 2048) C *= 2;
    return C;
}

static int64_t verify_slice(int64_t V, int C) {
    int64_t s = (V + C - 1) / C;
    return (s + 15) & ~static_cast<int64_t>(15);
}

size_t verify_workspace_bytes(int64_t B, int32_t D) {
    return static_cast<size_t>(B) * static_cast<size_t>(D + 1) * sizeof(vs::UnitResult);
}

static size_t verify_smem_bytes_es(int64_t slice, size_t es) {
    const size_t head = (sizeof(vs::Shared) + 127) & ~static_cast<size_t>(127);
    const size_t row = ((static_cast<size_t>(slice) * es) + 127) & ~static_cast<size_t>(127);
    return head + 2 * row;
}

bool verify_fits(int64_t V, size_t elem_bytes) {
    const int C = verify_cluster_size(V);
    return verify_smem_bytes_es(verify_slice(V, C), elem_bytes) <= 227u * 1024u;
}

template <typename T>
static cudaError_t launch_verify_sample(const vs::Params &p, int C, cudaStream_t stream) {
    const size_t smem = verify_smem_bytes_es(p.slice, sizeof(T));
    cudaError_t e = cudaFuncSetAttribute(vs::k_verify_units<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(vs::k_verify_units<T>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const int64_t units = p.B * (p.D + 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * C), 1, 1);
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
    return cudaLaunchKernelEx(&cfg, vs::k_verify_units<T>, p);
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
    p.res = static_cast<vs::UnitResult *>(a.workspace);
    p.status = a.status;
    cudaError_t e = a.dtype == MTPSPEC_F32 ? launch_verify_sample<float>(p, C, stream)
                                           : launch_verify_sample<uint16_t>(p, C, stream);
    if (e != cudaSuccess) return e;

    cudaLaunchConfig_t fin = {};
    fin.gridDim = dim3(static_cast<unsigned>((a.B + 127) / 128), 1, 1);
    fin.blockDim = dim3(128, 1, 1);
    fin.stream = stream;
    cudaLaunchAttribute fattr[1];
    fattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    fattr[0].val.programmaticStreamSerializationAllowed = 1;
    fin.attrs = fattr;
    fin.numAttrs = 1;
    return cudaLaunchKernelEx(&fin, vs::k_verify_finalize,
                              static_cast<const vs::UnitResult *>(a.workspace), a.draft_ids, a.B,
                              a.D, a.out_tokens, a.num_accepted, a.p_target, a.p_draft);
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
