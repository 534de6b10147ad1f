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
//   pass 1   per-slice max and online softmax sum (argmax for greedy rows) as chunks land
//   E1       the per-CTA partials meet in every CTA through distributed shared memory
//   pass 2   (top-k/top-p only) histogram of count and fixed-point softmax weight over
//            bins of z = (x - max) * log2(e) / tau, R bins per unit of z; reduce-scattered
//            and re-broadcast across the cluster (E2)
//   gather   the elements of the bins that hold the top-k / top-p boundary are pushed to
//            every CTA (E3); each CTA finds the exact thresholds by radix select on their
//            order-preserving keys.  If the boundary is outside the binned range or its bins
//            hold too many elements, an exact binary search over keys replaces this step.
//   accept   p(d), q(d) and U_acc <= p/q (ratio formed with both maxima factored out)
//   draw     only for a rejected draft or the bonus position: per-warp sums of the draw
//            weights in id order, CTA sums exchanged (E4), and the CTA holding the target
//            walks its slice to the token (inverse CDF in ascending id order).
// A per-row finalize kernel then takes the first rejected position.
//
// Every decision is computed identically in every CTA of a cluster from exchanged data, so
// all CTAs run the same sequence of cluster barriers.  Data exchanges are pushes into the
// peers' shared memory before a barrier; after the last barrier a CTA only reads its own
// shared memory, so it may exit.  The only wait on an asynchronous event is the bulk-copy
// barrier, bounded by an iteration limit that raises MTPSPEC_STATUS_TIMEOUT.
#include "common.cuh"
#include "kernels.h"

namespace mtpspec {
namespace vs {

constexpr int NT = 512;          // threads per CTA
constexpr int NW = NT / 32;      // warps per CTA
constexpr int MAXC = 16;         // largest cluster
constexpr int R = 16;            // histogram bins per unit of z (log2 of the softmax weight)
constexpr int NB = 512;          // binned range: z in (-NB/R, 0] = weights in (2^-32, 1]
constexpr int NBT = NB + 1;      // + one bin for everything below the range
constexpr int INCOMING = NBT + MAXC;  // reduce-scatter slots per row (C * ceil(NBT / C))
constexpr int CAP = 1024;        // boundary candidates per row
constexpr int NCH = 4;           // bulk-copy chunks per row
constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct UnitResult {
    int32_t flags;  // bit 0: draft accepted
    int32_t token;  // greedy pick, or the draw (residual / bonus) of this unit, or -1
    float pt;       // p_j(d_j)
    float pd;       // q_j(d_j)
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
    float m[2], zall[2], invZ[2], Z[2];
    uint32_t theta[2];
    int32_t deg[2];    // row of all -inf: a point mass on id 0
    int32_t mode[2];   // 0 no filter, 1 candidates, 2 exact search
    int32_t blo[2], bhi[2];
    uint32_t ncand[2];
    unsigned long long NA[2], MA[2];
    // histogram (local during pass 2, the cluster-wide histogram after E2)
    uint32_t hcnt[2][NBT];
    unsigned long long hmass[2][NBT];
    // reduce-scatter inbox, reused for the boundary candidates
    union {
        struct {
            uint32_t cnt[2][INCOMING];
            unsigned long long mass[2][INCOMING];
        } in;
        unsigned long long cand[2][CAP];
    } u;
    uint32_t cand_n[2];  // slot allocator, used in CTA 0
    // radix select scratch
    uint32_t s_cnt[256];
    unsigned long long s_mass[256];
    unsigned long long s_bcast[4];
    // exact search exchange (double-buffered by iteration parity)
    unsigned long long sx[2][2][MAXC];
    // draws
    unsigned long long dr_R[2][MAXC];  // per draw attempt: each CTA's fixed-point weight
    unsigned long long w_sum[NW];
    unsigned long long mtot[2];         // exact fixed-point weight of the whole row
    int32_t flags;  // bit 0: a bulk copy timed out
    int32_t pick[4];
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
__device__ __forceinline__ int zbin(float z) {
    if (!(z > -static_cast<float>(NB / R))) return NB;  // below the range (or NaN)
    int b = static_cast<int>(__fmul_rn(-z, static_cast<float>(R)));
    return b < NB ? b : NB - 1;
}
__device__ __forceinline__ unsigned long long fixmass(float e, float scale) {
    return __float2ull_rn(__fmul_rn(e, scale));
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
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
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

// ---------------------------------------------------------------- per-element visitors

// Visit every element [0, n) of a shared-memory slice as (value, local index), with
// 16-byte vector reads for the aligned body, threads strided over vectors.
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

// ---------------------------------------------------------------- radix select

// Among candidates (key << 32 | id) with key >= floor_key, the largest key t such that the
// count (use_mass = false) or the fixed-point weight (use_mass = true) of candidates with
// key >= t reaches `need` (need >= 1 and reachable).  All threads call; returns in all.
__device__ uint32_t radix_select(Shared &sh, const unsigned long long *cand, int n,
                                 uint32_t floor_key, unsigned long long need, bool use_mass,
                                 float m, float c2, float scale) {
    uint32_t prefix = 0, pmask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += NT) {
            sh.s_cnt[i] = 0;
            sh.s_mass[i] = 0;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += NT) {
            const uint32_t key = static_cast<uint32_t>(cand[i] >> 32);
            if (key < floor_key || (key & pmask) != prefix) continue;
            const uint32_t dg = (key >> shift) & 255u;
            if (use_mass) {
                const float x = key_to_float(key);
                atomicAdd(&sh.s_mass[dg], fixmass(ex2(zval(x, m, c2)), scale));
            } else {
                atomicAdd(&sh.s_cnt[dg], 1u);
            }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            // lane l owns digits 255-8l .. 248-8l (descending)
            unsigned long long v[8], tot = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int dg = 255 - (lane * 8 + t);
                v[t] = use_mass ? sh.s_mass[dg] : static_cast<unsigned long long>(sh.s_cnt[dg]);
                tot += v[t];
            }
            unsigned long long incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned long long excl = incl - tot;
            if (excl < need && incl >= need) {
                unsigned long long acc = excl;
                int pick = 0;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (acc + v[t] >= need) {
                        pick = 255 - (lane * 8 + t);
                        break;
                    }
                    acc += v[t];
                }
                sh.s_bcast[0] = static_cast<unsigned long long>(pick);
                sh.s_bcast[1] = need - acc;
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sh.s_bcast[0]) << shift;
        pmask |= 255u << shift;
        need = sh.s_bcast[1];
        __syncthreads();
    }
    return prefix;
}

// Sum of fixed-point weights of candidates with key >= t.
__device__ unsigned long long cand_mass_from(Shared &sh, const unsigned long long *cand, int n,
                                             uint32_t t, float m, float c2, float scale) {
    unsigned long long acc = 0;
    for (int i = threadIdx.x; i < n; i += NT) {
        const uint32_t key = static_cast<uint32_t>(cand[i] >> 32);
        if (key >= t) acc += fixmass(ex2(zval(key_to_float(key), m, c2)), scale);
    }
    acc = warp_sum_u64(acc);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.ru[0][threadIdx.x >> 5] = acc;
    __syncthreads();
    unsigned long long tot = 0;
    for (int w = 0; w < NW; ++w) tot += sh.ru[0][w];
    __syncthreads();
    return tot;
}

// First bin b (0..NB-1) whose cumulative value (bins 0..b) reaches `need`; NB if none.
// One warp; the histogram is the cluster-wide one.  Writes the result to *out.
__device__ void first_bin_reaching(const uint32_t *cnt, const unsigned long long *mass,
                                   bool use_mass, unsigned long long need, int32_t *out) {
    const int lane = threadIdx.x & 31;
    constexpr int PER = (NB + 31) / 32;
    unsigned long long tot = 0;
    for (int t = 0; t < PER; ++t) {
        const int b = lane * PER + t;
        if (b < NB) tot += use_mass ? mass[b] : static_cast<unsigned long long>(cnt[b]);
    }
    unsigned long long incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned long long excl = incl - tot;
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, excl < need && incl >= need);
    if (ball == 0) {
        if (lane == 0) *out = NB;
        return;
    }
    if (lane == __ffs(ball) - 1) {
        unsigned long long acc = excl;
        for (int t = 0; t < PER; ++t) {
            const int b = lane * PER + t;
            acc += use_mass ? mass[b] : static_cast<unsigned long long>(cnt[b]);
            if (acc >= need) {
                *out = b;
                break;
            }
        }
    }
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
    float scale;      // 2^S, the fixed-point weight scale
    float inv_scale;  // 2^-S
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
    const size_t row_bytes = ((static_cast<size_t>(P.slice) * sizeof(T)) + 127) & ~static_cast<size_t>(127);
    T *sdat[2] = {reinterpret_cast<T *>(smem_raw + data_off),
                  reinterpret_cast<T *>(smem_raw + data_off + row_bytes)};

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
    const float c2 = greedy ? 0.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(tau));

    const int64_t lo64 = static_cast<int64_t>(rank) * P.slice;
    const int64_t rest = V - lo64;
    const int n = static_cast<int>(rest <= 0 ? 0 : (rest < P.slice ? rest : P.slice));
    const int32_t d = j < D ? P.d[b * D + j] : -1;
    const bool dvalid = d >= 0 && static_cast<int64_t>(d) < V;
    const bool d_here = dvalid && static_cast<int64_t>(d) >= lo64 && static_cast<int64_t>(d) < lo64 + n;

    const T *grow[2];
    grow[0] = static_cast<const T *>(P.T) + (b * (D + 1) + j) * V + lo64;
    grow[1] = has_q ? static_cast<const T *>(P.Q) + (b * D + j) * V + lo64 : nullptr;

    // ---- set-up: barriers, counters, histogram
    if (tid == 0) {
        for (int r = 0; r < 2; ++r)
            for (int c = 0; c < NCH; ++c) mbar_init(&sh.bar[r][c], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh.cand_n[0] = sh.cand_n[1] = 0;
        sh.flags = 0;
    }
    for (int i = tid; i < 2 * NBT; i += NT) {
        (&sh.hcnt[0][0])[i] = 0;
        (&sh.hmass[0][0])[i] = 0;
    }
    __syncthreads();
    cluster_arrive_release();  // peers may touch this CTA's shared memory after the wait below
    pdl_launch_dependents();

    // ---- loads: bulk copies of the 16-byte-aligned body, plain loads for the rest
    const int nv = n / EPV;
    bool bulk[2] = {false, false};
    for (int r = 0; r < nrows; ++r)
        bulk[r] = nv > 0 && (reinterpret_cast<uintptr_t>(grow[r]) & 15u) == 0;
    if (tid == 0) {
        for (int r = 0; r < nrows; ++r) {
            if (!bulk[r]) continue;
            const int per = (nv + NCH - 1) / NCH;
            for (int c = 0; c < NCH; ++c) {
                const int v0 = c * per, v1 = min(nv, v0 + per);
                if (v1 <= v0) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sh.bar[r][c])) : "memory");
                    continue;
                }
                const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
                mbar_expect_tx(&sh.bar[r][c], bytes);
                bulk_copy_g2s(sdat[r] + v0 * EPV, grow[r] + v0 * EPV, bytes, &sh.bar[r][c]);
            }
        }
    }
    for (int r = 0; r < nrows; ++r) {
        const int from = bulk[r] ? nv * EPV : 0;
        for (int i = from + tid; i < n; i += NT) sdat[r][i] = grow[r][i];
    }
    __syncthreads();

    // ---- pass 1: max (+ online sum when nothing is filtered) or argmax (greedy)
    const bool online = !greedy && !k_on && !p_on;
    float tm[2] = {-INFINITY, -INFINITY}, ts[2] = {0.0f, 0.0f};
    ArgMax am{-INFINITY, -1};
    bool timed_out = false;
    for (int r = 0; r < nrows; ++r) {
        const uint4 *vp = reinterpret_cast<const uint4 *>(sdat[r]);
        const int per = (nv + NCH - 1) / NCH;
        for (int c = 0; c < NCH; ++c) {
            const int v0 = c * per, v1 = min(nv, v0 + per);
            if (bulk[r] && v1 > v0 && !mbar_wait_bounded(&sh.bar[r][c])) timed_out = true;
            for (int i = v0 + tid; i < v1; i += NT) {
                float x[EPV];
                unpack(vp[i], x);
                if (greedy) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (x[e] > am.v || am.i < 0) am = {x[e], static_cast<int32_t>(lo64 + i * EPV + e)};
                } else {
                    float vm = x[0];
#pragma unroll
                    for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, x[e]);
                    if (vm > tm[r]) {
                        ts[r] = ts[r] * ex2(__fmul_rn(tm[r] - vm, c2));
                        tm[r] = vm;
                    }
                    if (online && tm[r] > -INFINITY) {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) ts[r] += ex2(__fmul_rn(x[e] - tm[r], c2));
                    }
                }
            }
        }
        for (int i = nv * EPV + tid; i < n; i += NT) {
            const float x = widen(sdat[r][i]);
            if (greedy) {
                if (x > am.v || am.i < 0) am = {x, static_cast<int32_t>(lo64 + i)};
            } else if (x > -INFINITY) {
                if (online)
                    ms_merge(tm[r], ts[r], x, 1.0f, c2);
                else
                    tm[r] = fmaxf(tm[r], x);
            }
        }
    }
    if (timed_out) atomicOr(&sh.flags, 1);
    if (!online)  // only the maxima matter; a sum of 1 marks a non-empty partial for the merge
        for (int r = 0; r < nrows; ++r) ts[r] = tm[r] > -INFINITY ? 1.0f : 0.0f;

    // block reduction of the pass-1 partials
    for (int r = 0; r < nrows; ++r) {
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
        for (uint32_t c = 0; c < C; ++c) {
            st_peer_f32(peer_addr(smem_addr(&sh.x_m[rank][r]), c), mv);
            st_peer_f32(peer_addr(smem_addr(&sh.x_s[rank][r]), c), sv);
            st_peer_u32(peer_addr(smem_addr(&sh.x_i[rank][r]), c), static_cast<uint32_t>(iv));
            if (d_here)
                st_peer_f32(peer_addr(smem_addr(&sh.x_d[r]), c),
                            widen(sdat[r][static_cast<int64_t>(d) - lo64]));
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
        sh.m[r] = mx;
        sh.zall[r] = sv;
        sh.deg[r] = !(mx > -INFINITY);
        sh.mode[r] = 0;
        sh.theta[r] = 0u;
        sh.Z[r] = sv;
    }
    __syncthreads();

    const bool need_filter = k_on || p_on;
    if (need_filter) {
        // ---- pass 2: histogram of count and fixed-point weight over z bins
        for (int r = 0; r < nrows; ++r) {
            if (sh.deg[r]) continue;
            const float m = sh.m[r];
            uint32_t below = 0;
            unsigned long long below_w = 0;
            for_each_elem(sdat[r], n, [&](float x, int) {
                const float z = zval(x, m, c2);
                const int bn = zbin(z);
                const unsigned long long w = fixmass(ex2(z), P.scale);
                if (bn < NB) {
                    atomicAdd(&sh.hcnt[r][bn], 1u);
                    atomicAdd(&sh.hmass[r][bn], w);
                } else {
                    ++below;
                    below_w += w;
                }
            });
            below = __reduce_add_sync(0xFFFFFFFFu, below);
            below_w = warp_sum_u64(below_w);
            if (lane == 0 && below_w) atomicAdd(&sh.hmass[r][NB], below_w);
            if (lane == 0 && below) atomicAdd(&sh.hcnt[r][NB], below);
        }
        __syncthreads();
        // ---- E2a: reduce-scatter, push local bins to their owner CTA
        const int RS = (NBT + C - 1) / C;
        for (int idx = tid; idx < nrows * NBT; idx += NT) {
            const int r = idx / NBT, bn = idx - r * NBT;
            const int owner = bn / RS, k = bn - owner * RS;
            const int slot = static_cast<int>(rank) * RS + k;
            st_peer_u32(peer_addr(smem_addr(&sh.u.in.cnt[r][slot]), owner), sh.hcnt[r][bn]);
            st_peer_u64(peer_addr(smem_addr(&sh.u.in.mass[r][slot]), owner), sh.hmass[r][bn]);
        }
        cluster_sync();  // B2a
        // ---- E2b: sum the owned bins and broadcast them
        for (int idx = tid; idx < nrows * RS; idx += NT) {
            const int r = idx / RS, k = idx - r * RS;
            const int bn = static_cast<int>(rank) * RS + k;
            if (bn >= NBT) continue;
            uint32_t cs = 0;
            unsigned long long msum = 0;
            for (uint32_t c = 0; c < C; ++c) {
                cs += sh.u.in.cnt[r][c * RS + k];
                msum += sh.u.in.mass[r][c * RS + k];
            }
            for (uint32_t c = 0; c < C; ++c) {
                st_peer_u32(peer_addr(smem_addr(&sh.hcnt[r][bn]), c), cs);
                st_peer_u64(peer_addr(smem_addr(&sh.hmass[r][bn]), c), msum);
            }
        }
        cluster_sync();  // B2b

        // ---- plan per row: the bin range holding the boundary, or the exact search
        if (warp < nrows) {
            const int r = warp;
            if (sh.deg[r]) {
                if (lane == 0) sh.mode[r] = 0;
            } else {
                int32_t bk = -1, blo = 0, bhi = 0;
                bool slow = false;
                if (k_on) {
                    first_bin_reaching(sh.hcnt[r], sh.hmass[r], false,
                                       static_cast<unsigned long long>(kk), &sh.pick[r]);
                    __syncwarp();
                    bk = sh.pick[r];
                    __syncwarp();
                    if (bk >= NB) slow = true;
                    bhi = bk;
                    blo = bk;
                    if (!slow && p_on) {
                        unsigned long long above = 0;  // weight of the bins before bk
                        for (int t = lane; t < bk; t += 32) above += sh.hmass[r][t];
                        above = warp_sum_u64(above);
                        const double tt = static_cast<double>(pp) * static_cast<double>(above);
                        const unsigned long long need = static_cast<unsigned long long>(ceil(tt));
                        if (need == 0) {
                            blo = 0;
                        } else {
                            first_bin_reaching(sh.hcnt[r], sh.hmass[r], true, need, &sh.pick[r]);
                            __syncwarp();
                            blo = min(sh.pick[r], bk);
                            __syncwarp();
                        }
                    }
                } else {  // top-p alone
                    unsigned long long tot = 0;
                    for (int t = lane; t < NBT; t += 32) tot += sh.hmass[r][t];
                    tot = warp_sum_u64(tot);
                    if (lane == 0) sh.mtot[r] = tot;
                    const double tt = static_cast<double>(pp) * static_cast<double>(tot);
                    const unsigned long long need = max(1ull, static_cast<unsigned long long>(ceil(tt)));
                    first_bin_reaching(sh.hcnt[r], sh.hmass[r], true, need, &sh.pick[r]);
                    __syncwarp();
                    blo = bhi = sh.pick[r];
                    __syncwarp();
                    if (blo >= NB) slow = true;
                }
                unsigned long long na = 0, ma = 0, inr = 0;
                if (!slow) {
                    for (int t = lane; t < NB; t += 32) {
                        if (t < blo) {
                            na += sh.hcnt[r][t];
                            ma += sh.hmass[r][t];
                        } else if (t <= bhi) {
                            inr += sh.hcnt[r][t];
                        }
                    }
                    na = warp_sum_u64(na);
                    ma = warp_sum_u64(ma);
                    inr = warp_sum_u64(inr);
                    if (inr > static_cast<unsigned long long>(CAP)) slow = true;
                }
                if (lane == 0) {
                    sh.mode[r] = slow ? 2 : 1;
                    sh.blo[r] = blo;
                    sh.bhi[r] = bhi;
                    sh.NA[r] = na;
                    sh.MA[r] = ma;
                    sh.ncand[r] = static_cast<uint32_t>(inr);
                }
            }
        }
        __syncthreads();

        // ---- gather the boundary candidates into every CTA (E3)
        const bool any_fast = sh.mode[0] == 1 || (nrows > 1 && sh.mode[1] == 1);
        if (any_fast) {
            for (int r = 0; r < nrows; ++r) {
                if (sh.mode[r] != 1) continue;
                const float m = sh.m[r];
                const int blo = sh.blo[r], bhi = sh.bhi[r];
                const uint32_t cnt_addr0 = peer_addr(smem_addr(&sh.cand_n[r]), 0);
                // warp-contiguous traversal so that every lane of a warp iterates together
                const int per_w = (n + NW - 1) / NW;
                const int w0 = warp * per_w, w1 = min(n, w0 + per_w);
                for (int base = w0; base < w1; base += 32) {
                    const int i = base + lane;
                    bool hit = false;
                    uint32_t key = 0;
                    if (i < w1) {
                        const float x = widen(sdat[r][i]);
                        const int bn = zbin(zval(x, m, c2));
                        hit = bn >= blo && bn <= bhi;
                        key = order_key(x);
                    }
                    const unsigned ball = __ballot_sync(0xFFFFFFFFu, hit);
                    if (ball == 0) continue;
                    uint32_t slot0 = 0;
                    if (lane == __ffs(ball) - 1) slot0 = atom_peer_add_u32(cnt_addr0, __popc(ball));
                    slot0 = __shfl_sync(0xFFFFFFFFu, slot0, __ffs(ball) - 1);
                    if (hit) {
                        const uint32_t slot = slot0 + __popc(ball & ((1u << lane) - 1u));
                        const unsigned long long v = (static_cast<unsigned long long>(key) << 32) |
                                                     static_cast<uint32_t>(lo64 + i);
                        if (slot < static_cast<uint32_t>(CAP))
                            for (uint32_t c = 0; c < C; ++c)
                                st_peer_u64(peer_addr(smem_addr(&sh.u.cand[r][slot]), c), v);
                    }
                }
            }
            cluster_sync();  // B3
            // ---- exact thresholds from the candidates
            for (int r = 0; r < nrows; ++r) {
                if (sh.mode[r] != 1) continue;
                const float m = sh.m[r];
                const int nc = static_cast<int>(sh.ncand[r]);
                const unsigned long long *cand = sh.u.cand[r];
                uint32_t thk = 0;
                unsigned long long zk = 0;
                if (k_on) {
                    const unsigned long long need = static_cast<unsigned long long>(kk) - sh.NA[r];
                    thk = radix_select(sh, cand, nc, 0u, need, false, m, c2, P.scale);
                    zk = sh.MA[r] + cand_mass_from(sh, cand, nc, thk, m, c2, P.scale);
                }
                uint32_t th = thk;
                if (p_on) {
                    double tt;
                    if (k_on)
                        tt = static_cast<double>(pp) * static_cast<double>(zk);
                    else
                        tt = static_cast<double>(pp) * static_cast<double>(sh.mtot[r]);
                    unsigned long long need = static_cast<unsigned long long>(ceil(tt));
                    need = need > sh.MA[r] ? need - sh.MA[r] : 1ull;
                    th = radix_select(sh, cand, nc, thk, need, true, m, c2, P.scale);
                }
                const unsigned long long zfx = sh.MA[r] + cand_mass_from(sh, cand, nc, th, m, c2, P.scale);
                if (tid == 0) {
                    sh.theta[r] = th;
                    sh.Z[r] = static_cast<float>(static_cast<double>(zfx) * static_cast<double>(P.inv_scale));
                }
                __syncthreads();
            }
        }

        // ---- exact binary search over keys (boundary outside the binned range, or too
        // many elements in its bins); both rows advance in lockstep, one barrier a step
        const bool any_slow = sh.mode[0] == 2 || (nrows > 1 && sh.mode[1] == 2);
        if (any_slow) {
            int parity = 0;
            // F(t) for each row: count (what = 0) or weight (what = 1) of elements with
            // key >= t and key >= floor; pushed to every CTA; returns the cluster sums
            auto eval = [&](const uint32_t t[2], const uint32_t fl[2], const int what[2],
                            unsigned long long out[2]) {
                unsigned long long acc[2] = {0, 0};
                for (int r = 0; r < nrows; ++r) {
                    if (sh.mode[r] != 2) continue;
                    const float m = sh.m[r];
                    const uint32_t lim = max(t[r], fl[r]);
                    const int wt = what[r];
                    unsigned long long a = 0;
                    for_each_elem(sdat[r], n, [&](float x, int) {
                        if (order_key(x) >= lim)
                            a += wt ? fixmass(ex2(zval(x, m, c2)), P.scale) : 1ull;
                    });
                    acc[r] = warp_sum_u64(a);
                }
                __syncthreads();
                if (lane == 0) {
                    sh.ru[0][warp] = acc[0];
                    sh.ru[1][warp] = acc[1];
                }
                __syncthreads();
                if (tid < 2) {
                    unsigned long long s = 0;
                    for (int w = 0; w < NW; ++w) s += sh.ru[tid][w];
                    for (uint32_t c = 0; c < C; ++c)
                        st_peer_u64(peer_addr(smem_addr(&sh.sx[parity][tid][rank]), c), s);
                }
                cluster_sync();
                for (int r = 0; r < 2; ++r) {
                    unsigned long long s = 0;
                    for (uint32_t c = 0; c < C; ++c) s += sh.sx[parity][r][c];
                    out[r] = s;
                }
                parity ^= 1;
            };
            // largest t with F(t) >= need, by bisection over the 32-bit key space
            auto search = [&](const uint32_t fl[2], const int what[2],
                              const unsigned long long need[2], uint32_t res_t[2]) {
                uint32_t lo[2] = {0u, 0u}, hi[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
                for (int it = 0; it < 32; ++it) {
                    uint32_t mid[2];
                    for (int r = 0; r < 2; ++r)
                        mid[r] = lo[r] + static_cast<uint32_t>((static_cast<uint64_t>(hi[r]) - lo[r] + 1) / 2);
                    unsigned long long f[2];
                    eval(mid, fl, what, f);
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
            int wcnt[2] = {0, 0}, wmass[2] = {1, 1};
            unsigned long long zk[2] = {0, 0};
            if (k_on) {
                unsigned long long need[2] = {static_cast<unsigned long long>(kk),
                                              static_cast<unsigned long long>(kk)};
                search(zero, wcnt, need, thk);
                eval(thk, zero, wmass, zk);
            }
            th[0] = thk[0];
            th[1] = thk[1];
            if (p_on) {
                unsigned long long need[2];
                for (int r = 0; r < 2; ++r) {
                    double tt = k_on ? static_cast<double>(pp) * static_cast<double>(zk[r])
                                     : static_cast<double>(pp) * static_cast<double>(sh.mtot[r < nrows ? r : 0]);
                    need[r] = max(1ull, static_cast<unsigned long long>(ceil(tt)));
                }
                search(thk, wmass, need, th);
            }
            unsigned long long zf[2];
            eval(th, zero, wmass, zf);
            if (tid < nrows && sh.mode[tid] == 2) {
                sh.theta[tid] = th[tid];
                sh.Z[tid] = static_cast<float>(static_cast<double>(zf[tid]) * static_cast<double>(P.inv_scale));
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

    auto member = [&](int r, float x, int64_t idx) -> bool {
        return sh.deg[r] ? idx == 0 : order_key(x) >= sh.theta[r];
    };
    auto prob = [&](int r, float x, int64_t idx) -> float {
        if (!member(r, x, idx)) return 0.0f;
        return sh.deg[r] ? 1.0f : ex2(zval(x, sh.m[r], c2)) * sh.invZ[r];
    };

    bool accept = false;
    float pt = 0.0f, pd = 0.0f;
    if (j < D && dvalid) {
        const float xt = sh.x_d[0], xq = sh.x_d[1];
        const bool in_p = member(0, xt, d), in_q = member(1, xq, d);
        pt = prob(0, xt, d);
        pd = prob(1, xq, d);
        if (!in_p) {
            accept = false;
        } else if (!in_q) {
            accept = true;
        } else {
            float ratio;
            if (sh.deg[0] || sh.deg[1])
                ratio = pt / pd;
            else
                ratio = ex2(__fmul_rn((xt - sh.m[0]) - (xq - sh.m[1]), c2)) * (sh.Z[1] / sh.Z[0]);
            accept = u_acc <= ratio;
        }
    }

    // ---- draw (a rejected draft's residual, or the bonus).  Weights are rounded to fixed
    // point (2^40 per unit of probability) and summed as integers, so the cumulative sums
    // at every level (lane, warp, CTA, cluster) are exact and agree with one another.
    const bool draw = (j == D) || !accept;
    if (draw) {
        int wmode = (j == D) ? 1 : 0;  // 0: max(0, p - q), 1: p
        const int per_w = (((n + NW - 1) / NW) + 31) & ~31;
        const int w0 = min(n, warp * per_w), w1 = min(n, w0 + per_w);
        auto weight = [&](int i) -> unsigned long long {
            const int64_t gi = lo64 + i;
            const float p = prob(0, widen(sdat[0][i]), gi);
            float w = p;
            if (wmode == 0) w = fmaxf(p - prob(1, widen(sdat[1][i]), gi), 0.0f);
            return __float2ull_rn(__fmul_rn(w, 1099511627776.0f));
        };
        for (int attempt = 0; attempt < 2; ++attempt) {
            unsigned long long acc = 0;
            for (int base = w0; base < w1; base += 32) {
                const int i = base + lane;
                if (i < w1) acc += weight(i);
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
                // smallest id whose cumulative weight exceeds u_smp * R: the CTA, then the
                // warp, then the element
                const double t = static_cast<double>(u_smp) * static_cast<double>(Rt);
                uint32_t cs = C - 1;
                unsigned long long before = 0;
                for (uint32_t c = 0; c < C; ++c) {
                    if (static_cast<double>(before + dR[c]) > t) {
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
                        if (static_cast<double>(wb + sh.w_sum[w]) > t) {
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
                        const int v0 = min(n, ws * per_w), v1 = min(n, v0 + per_w);
                        unsigned long long a = wb;
                        int32_t tok = -1, lastpos = -1;
                        for (int base = v0; base < v1 && tok < 0; base += 32) {
                            const int i = base + lane;
                            const unsigned long long wv = i < v1 ? weight(i) : 0ull;
                            unsigned long long incl = wv;
#pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                                if (lane >= o) incl += y;
                            }
                            const unsigned hitm = __ballot_sync(
                                0xFFFFFFFFu, wv > 0 && static_cast<double>(a + incl) > t);
                            const unsigned posm = __ballot_sync(0xFFFFFFFFu, wv > 0);
                            if (posm) lastpos = base + 31 - __clz(posm);
                            if (hitm) tok = base + __ffs(hitm) - 1;
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

template <typename T>
static size_t verify_smem_bytes(int64_t slice) {
    return verify_smem_bytes_es(slice, sizeof(T));
}

bool verify_fits(int64_t V, size_t elem_bytes) {
    const int C = verify_cluster_size(V);
    return verify_smem_bytes_es(verify_slice(V, C), elem_bytes) <= 227u * 1024u;
}

template <typename T>
static cudaError_t launch_verify_sample(const vs::Params &p, int C, cudaStream_t stream) {
    const size_t smem = verify_smem_bytes<T>(p.slice);
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
    int lg = 0;
    while ((int64_t{1} << lg) < a.V + 1) ++lg;
    const int S = max(20, 52 - lg);
    p.scale = ldexpf(1.0f, S);
    p.inv_scale = ldexpf(1.0f, -S);
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
