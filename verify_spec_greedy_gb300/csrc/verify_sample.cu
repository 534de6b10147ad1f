// Speculative-sampling verification: temperature -> top-k -> top-p filtering of target and
// draft logits, the accept test U <= p/q, the residual draw at the first rejection and the
// bonus draw ("MPT (MTP, Multi-Token Prediction) 原理详解", section 三 stage 3 "rejection
// sampling" and stage 4; "The decoding loop and MTP", "Why a hand-written decoding loop" for
// the filters and "MTP speculative decoding" items 2-3 for the drawn replacement and the
// extra token).
//
// Three kernels on the caller's stream:
//  - k_verify_rr: the sampled rows.  A persistent grid of thread-block clusters, as many
//    as can be resident; cluster g takes units g, g + G, ... (a unit is one (row b,
//    position j) pair of a sampled row: the target row T[b, j] and, for j < D, the draft
//    row Q[b, j]).  CTA r of a cluster owns the contiguous vocabulary slice
//    [r*slice, (r+1)*slice) of both rows.  Large batches (and one-hot drafts) number the
//    units position-major, so that a row's earlier positions are usually decided before its
//    later ones start; a unit behind a position of its row that was already rejected skips
//    its draw, which no output reads, and a bonus unit behind one skips its filters as well
//    (a per-row flag in the workspace, agreed on by the cluster at its first exchange).
//    Data path: bulk asynchronous copies (four chunks per row, each on its own mbarrier)
//    bring a unit's two slices into shared memory, where every pass of the unit reads
//    them, so every logit is read from HBM once.  While a unit works, one thread asks L2
//    to prefetch the next unit's slices; their copies are issued as soon as this unit no
//    longer needs its buffer (after the accept test, or after the draw).
//  - the greedy rows (temperature 0) go to the streaming argmax kernel
//    (run_verify_greedy_rows), launched as a programmatic dependent so that it runs beside
//    the persistent grid.
//  - k_verify_finalize: one thread per row takes the first rejected position.
//
// Work on one unit:
//   pass 1   the slices' maxima (as the chunks land), then the softmax sums of
//            z = (x - max) * log2(e) / tau relative to them
//   E1       per-CTA maxima and sums (and the draft token's logits) meet in every CTA
//   pass 2   (top-k / top-p) a histogram over R bins per unit of z, only for elements that
//            can hold the boundary: counts (top-k) or near-exact weights (top-p: each
//            element adds its weight scaled by its bin's octave, rounded to an integer)
//   E2       reduce-scatter of the histograms to owner CTAs, then all-gather of the sums
//   plan     the bins that may hold the boundary: by exact counts (top-k) or by rigorous
//            bounds on the cumulative weight (top-p)
//            A top-k row with k <= KFAST skips its sums, pass 2, E2 and the plan: pass 1
//            also finds a lower bound on each CTA's k-th largest logit (a radix selection
//            over the threads' maxima), E1 carries the bounds, and the gather takes every
//            element at or above the cluster's bound.
//   gather   elements of those bins go to every CTA (E3); the candidates, compacted with
//            their exact weights, are ranked by counting (or sorted, when there are many)
//            for the exact thresholds.  If the boundary lies outside the binned range or too
//            many elements fall into its bins, an exact bisection over the 32-bit value
//            keys replaces this step.
//   accept   p(d), q(d) and U_acc <= p/q (ratio formed with both maxima factored out)
//   draw     only for a rejected draft or the bonus position: draw weights in fixed point
//            (2^31 per unit of probability), per-warp sums in id order, CTA sums exchanged
//            (E4), and the warp holding the target walks its run to the token.  A top-k
//            row resolved from its candidates draws in CTA 0 from them alone, with the
//            same weights in id order (no slice is read).
//
// Work that no output reads is skipped when the call requests no probabilities: a draft
// whose acceptance is already certain needs nothing but its flag.  It is seen at E1
// (in the instance built for such calls: the target mass above the draft token, summed
// in pass 1, settles that the token is kept, and U_acc lies below a lower bound of p/q),
// or after the plan (the kept masses then lie within rigorous bounds).  Such a unit skips
// the rest of its filters and releases its staged rows at once.
//
// Exchanges are point to point: a CTA writes its part into every peer's shared memory and
// then arrives (release, cluster scope) on that peer's mbarrier for the exchange; a CTA
// waits (acquire) until all C CTAs have arrived.  E1 alternates between two barriers and
// buffers by unit parity; every other exchange has one buffer, which is safe because a
// CTA can only write a peer's buffer for unit k + 1 after that peer has arrived at E1 of
// unit k + 1, i.e. after it finished unit k.  All waits are bounded and raise
// MTPSPEC_STATUS_TIMEOUT when they give up.
//
// The kernel is bound by the residency of its staged rows and by instruction issue, not by
// memory bandwidth: each phase is written for few instructions per element (no per-element branch, bins and weights leave fp32
// through exponent arithmetic, not conversions), and the latency-bound bookkeeping
// (scheduling the next unit, its L2 prefetch, the Philox words) runs in one warp while the
// others wait for E1.
//
// Weight sums are formed per thread in fp32 over a fixed set of elements, converted once
// to 64-bit fixed point and reduced as integers, so every sum is deterministic and the same
// in every CTA of a cluster.  Every decision is computed identically in every CTA from
// exchanged data, so all CTAs take the same sequence of exchanges.
#include <mutex>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace mtpspec {
namespace vs {

constexpr int NT = 1024;         // threads per CTA
constexpr int CPS = 1;           // CTAs resident per SM
constexpr int NW = NT / 32;      // warps per CTA
static_assert(NW <= 32 && NW % 2 == 0, "one warp merges the warps' partials; rows split the warps in halves");
constexpr int MAXC = 16;         // largest cluster
// Histogram bins are R per unit of z = log2 of the softmax weight w = 2^z relative to the row
// maximum: bin b holds tz = -z * R in [b, b + 1), tz an affine function of the logit, so that
// a bin's members are a value interval.
constexpr int R = 32;            // bins per octave
constexpr int ZR = 24;           // binned range: z in (-ZR, 0], weights in (2^-24, 1]
constexpr int NB = R * ZR;       // bins
// reduce-scatter inbox per row: C * RS bins, RS = ceil(NB / C) rounded up to a multiple of 4,
// at most NB + 32 for any C <= 16 (the most, 800, at C = 10)
constexpr int RSN = NB + 32;
constexpr int CAPT = RSN;        // candidate slots per row in a cluster (CAPT / C per CTA):
                                 // as many as the histograms they share storage with
constexpr int NCH = 4;           // bulk-copy chunks per row
constexpr int WVEC_SHARED = 6400;  // draw: vector weights kept in the shared state's storage
// polls of a bounded wait: an unsuccessful mbarrier poll suspends the thread for about
// 3.8 us (measured), so a wait gives up after about a second, far beyond any wait of a
// working call (microseconds, a peer's phase at most)
constexpr uint32_t WAIT_LIMIT = 1u << 18;
constexpr float FX = 2147483648.0f;  // 2^31: fixed-point scale of weights (weights <= 1)

// exchange barriers
constexpr int XB_E1 = 0;   // two, by unit parity
constexpr int XB_RS = 2;
constexpr int XB_AG = 3;
constexpr int XB_E3 = 4;
constexpr int XB_E4 = 5;   // two, by draw attempt
constexpr int XB_S = 7;    // two, by exact-search step parity
constexpr int NXB = 9;

using UnitResult = VerifyUnitRecord;

constexpr int NSMALL = NT / 2;   // candidates per row ranked by counting (both rows at once)
// Top-k rows with k <= KFAST skip the histogram: every element at or above a lower bound on
// the k-th largest logit, found in pass 1, is a candidate.
constexpr int KFAST = 128;
constexpr int PW = 8;            // plan: warps per row
constexpr int PL = PW * 32;      // plan: lanes per row
constexpr int BPL = NB / PL;     // plan: bins per lane
static_assert(NB % PL == 0 && 2 * PW <= NW, "the plan's groups tile the bins and fit the CTA");

// Per-unit parameters of a sampled row.
struct UnitParams {
    int b, j;
    float tau, pp;
    int32_t kk, d;
};
// The parameters of a unit beside its index (which gives b and j); sent as one 16-byte store.
struct __align__(16) NextParams {
    float tau, pp;
    int32_t kk, d;
};

struct __align__(16) Shared {
    unsigned long long dbar[2][NCH];   // [row][chunk] bulk-copy barriers
    unsigned long long xbar[NXB];      // exchange barriers (C arrivals each)
    float4 e1[2][MAXC];                // E1, by unit parity: (m0, s0, m1, s1) per CTA
    float2 e1d[2];                     // E1, by unit parity: the draft token's logits
    uint32_t e1k[2][MAXC];             // E1, by unit parity: each CTA's view of the row's first rejection
    // Buffers whose lifetimes within a unit do not overlap share storage.  The histograms
    // per row hold top-k counts, or top-p weights as 16-bit fixed point relative to each
    // bin's upper edge.  Peers write rsin before E2b, hist before the plan and cand after
    // the plan (once every CTA has passed E2b), so cand can take the place of hloc and rsin,
    // and the sort scratch, used after E3, the place of hist.
    union {
        struct {
            uint32_t hloc[2][RSN];     // this CTA's histograms (zero past the used bins)
            uint32_t rsin[2][RSN];     // reduce-scatter inbox [row][source CTA * RS + bin]
        } h;
        unsigned long long cand[2][CAPT];  // candidates: (value bits << 32) | token id
    } a;
    union {
        unsigned long long hist[2][RSN];  // cluster-wide histograms
        struct {
            unsigned long long skey[NT];  // sort keys; candidate weights when counting
            float sval[NT];               // sorted values; candidate values when counting
        } s;
    } b;
    uint32_t ccnt[MAXC][2];            // candidates found per CTA
    uint32_t cpre[2][MAXC];            // per row, each CTA's offset in the row's candidate list
    int32_t ncr[2];                    // per row, the candidates' count (-1: exact search)
    unsigned long long sx[2][MAXC][2];   // exact search: per step parity, per CTA
    unsigned long long dr[2][MAXC];      // draw: per attempt, each CTA's fixed-point weight
    // per-warp scratch of phases that barriers separate
    union {
        struct {
            float rf[2][NW], rs[2][NW];    // pass 1: maxima and sums
            float ra[NW];                  // pass 1: the target mass above the draft token
        } p1;
        struct {
            unsigned long long lo[NW], hi[NW];  // plan: totals of the bound scans
            uint32_t cn[NW];
        } pl;
        struct {
            float v[NW];                   // counting: reductions
            unsigned long long w[NW];
        } ct;
        struct {
            unsigned long long scan[NW];   // sort and exact search: block scans and sums
            int32_t scani[NW];
            unsigned long long ru[2][NW];
        } so;
        unsigned long long wsum[NW];       // draw: each warp's weight
    } w;
    int32_t pb1[2], pb2[2];            // plan: crossing bins found by the scan
    uint32_t pcc1[2], pcc2[2];         // plan: count bounds before b1 and through b2
    unsigned long long pma[2];         // plan: fixed-point weight of the bins before b1
    uint32_t lcnt[2];                  // candidate slot allocator of this CTA
    float xd[2];                       // the draft token's logits, if this CTA holds it
    // per-row state, identical in every CTA of the cluster
    float m[2], Z[2], invZ[2], theta[2];
    float tzb[2];     // m * c2 * R: the bin coordinate tz = -z * R = x * (-c2 * R) + tzb
    uint32_t uwd[2];  // the unit's two Philox words (accept test, draw)
    float nmc[2];     // -m * c2: z = x * c2 + nmc
    int8_t deg[2];    // a row of all -inf: a point mass on id 0
    int8_t mode[2];   // 0 no filter, 1 candidates, 2 exact bisection
    int16_t b1[2], b2[2], nbu[2];  // bins (at most NB)
    unsigned long long tgt[2];
    int32_t flags;    // bit 0: a bulk copy timed out; bit 1: an exchange timed out
    float fpick[2];
    // E1, by unit parity: the cluster's unit after the next one (-1: none) and its
    // parameters, chosen by CTA 0 two units ahead (skipping the bonus units of rows it sees
    // rejected) and sent with its E1 message, so that every CTA takes the same sequence; in
    // CTA 0 the slot of the other parity holds the unit after that, chosen during this E1
    int32_t e1su[2];
    union {
        // top-k rows with a small k: per row, the cluster's lower bound on the k-th largest logit
        float kbd[2];
        // top-p rows of a decode loop: the target's mass strictly above the draft token's
        // logit, relative to the row maximum like Z
        float above;
    };
    int32_t early;    // the unit's draft is certainly accepted before its thresholds (see below)
    NextParams e1sp[2];
    // E1, by unit parity: each CTA's target mass above the draft token (last, so that the
    // fields above keep their places)
    float e1ab[2][MAXC];
};
// The slices' shared-memory budget (the vocabulary limits stated with the entry points)
// assumes this size.
static_assert(sizeof(Shared) == 28672, "the slices' shared-memory budget assumes this size");

__device__ __forceinline__ float ex2(float z) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
    return r;
}
// a weight (<= 1) in fixed point; the float-to-32-bit conversion is a fast instruction
__device__ __forceinline__ uint32_t fix31(float w) { return __float2uint_rn(__fmul_rn(w, FX)); }
// a per-thread sum in fixed point: a slow 64-bit conversion, used once per thread
__device__ __forceinline__ unsigned long long fix_sum(float s) {
    return __float2ull_rn(__fmul_rn(s, FX));
}

// ceil(p * Z * 2^31), the fixed-point top-p target of a row whose weights (relative to the
// row maximum) sum to Z, formed in fp32 (relative error 2^-24, the same in every CTA)
__device__ __forceinline__ unsigned long long fx_target(float p, float Z) {
    return __float2ull_ru(__fmul_rn(__fmul_rn(p, Z), FX));
}
// the same for a fixed-point sum z
__device__ __forceinline__ unsigned long long fx_target_fx(float p, unsigned long long z) {
    return __float2ull_ru(__fmul_rn(p, __ull2float_rn(z)));
}
// a fixed-point weight sum as a weight
__device__ __forceinline__ float fx_to_float(unsigned long long z) {
    return __fmul_rn(__ull2float_rn(z), 1.0f / FX);
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

// The plan's barrier of row r's group (hardware barriers 1 and 2; 0 is __syncthreads).
template <int N>
__device__ __forceinline__ void group_barrier(int r) {
    if (r == 0) asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
    else asm volatile("bar.sync 2, %0;" ::"n"(N) : "memory");
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
// Wait for the phase of the given parity; false after `limit` polls.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, uint32_t parity,
                                                  uint32_t limit = WAIT_LIMIT) {
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// The same with acquire semantics at cluster scope: the peers' writes released by their
// arrivals are visible after it returns true.
__device__ __forceinline__ bool xbar_wait_bounded(unsigned long long *bar, uint32_t parity,
                                                  uint32_t limit = WAIT_LIMIT) {
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}
// Arrive on CTA `peer`'s copy of the barrier, releasing this thread's earlier writes (and,
// through a preceding __syncthreads, the whole CTA's) at cluster scope.
__device__ __forceinline__ void xarrive(unsigned long long *bar, uint32_t peer) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     peer_addr(smem_addr(bar), peer))
                 : "memory");
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
__device__ __forceinline__ void st_peer_v4(uint32_t a, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_peer_u32x4(uint32_t a, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_peer_v2(uint32_t a, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y)
                 : "memory");
}

// Every element of one row's slice in shared memory: f(x, i) for element i < nv * EPV
// (16-byte vectors v = tid, tid + NT, ...; the ragged last vector is padded with -inf).
template <typename T, typename F>
__device__ __forceinline__ void for_row(const T *s, int nv, F &&f) {
    constexpr int EPV = elems_per_16B<T>::value;
    const uint4 *vp = reinterpret_cast<const uint4 *>(s);
#pragma unroll 2
    for (int v = threadIdx.x; v < nv; v += NT) {
        float x[EPV];
        unpack(vp[v], x);
#pragma unroll
        for (int e = 0; e < EPV; ++e) f(x[e], v * EPV + e);
    }
}

// Maximum of a 16-byte vector of logits (bf16 pairs compared packed, exactly: a bf16
// maximum widens to the fp32 maximum of the widened values).
template <typename T> __device__ __forceinline__ float vec_max(const uint4 &raw);
template <> __device__ __forceinline__ float vec_max<float>(const uint4 &raw) {
    return fmaxf(fmaxf(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                 fmaxf(__uint_as_float(raw.z), __uint_as_float(raw.w)));
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <> __device__ __forceinline__ float vec_max<uint16_t>(const uint4 &raw) {
    const uint32_t m = bf16x2_max(bf16x2_max(raw.x, raw.y), bf16x2_max(raw.z, raw.w));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}
// Sum of 2^(x * c2 + nm) over a 16-byte vector of logits.
template <typename T>
__device__ __forceinline__ float vec_sum_ex2(const uint4 &raw, float c2, float nm) {
    constexpr int EPV = elems_per_16B<T>::value;
    float x[EPV];
    unpack(raw, x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) x[e] = ex2(fmaf(x[e], c2, nm));
#pragma unroll
    for (int w = 1; w < EPV; w <<= 1)
#pragma unroll
        for (int e = 0; e + w < EPV; e += 2 * w) x[e] += x[e + w];
    return x[0];
}
// The same sum, and into `above` the sum over the elements above xd: the same weights,
// and the same order for the sum itself, so that it is bit for bit vec_sum_ex2's.
template <typename T>
__device__ __forceinline__ float vec_sum_ex2_above(const uint4 &raw, float c2, float nm, float xd,
                                                   float &above) {
    constexpr int EPV = elems_per_16B<T>::value;
    float x[EPV];
    unpack(raw, x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
        const float w = ex2(fmaf(x[e], c2, nm));
        above += x[e] > xd ? w : 0.0f;
        x[e] = w;
    }
#pragma unroll
    for (int w = 1; w < EPV; w <<= 1)
#pragma unroll
        for (int e = 0; e + w < EPV; e += 2 * w) x[e] += x[e + w];
    return x[0];
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// -inf as a stored logit
template <typename T> __device__ __forceinline__ T neg_inf();
template <> __device__ __forceinline__ float neg_inf<float>() { return -INFINITY; }
template <> __device__ __forceinline__ uint16_t neg_inf<uint16_t>() { return 0xFF80u; }

// Bounds on the fixed-point weight (2^31 per unit) of bin b of a top-p histogram.  Each
// element of the bin adds q = round(w * 2^(16 + o)), o = b / R its octave, so that
// 2^15 <= q <= 2^16 up to rounding; the bin's weight is q_sum * 2^(15 - o): mid, exact but
// for the truncation of a right shift.  The margin err covers half a unit of q per element,
// the truncation, and 2^-18 of mid for the fp32 error of the weights.  An element adds at
// least 2^15 less rounding, so a bin holds at most q_sum / 32256 elements (cnt).
__device__ __forceinline__ void bin_bounds(unsigned long long qs, int b, unsigned long long &mid,
                                           unsigned long long &err, uint32_t &cnt) {
    const int sft = 15 - b / R;
    mid = sft >= 0 ? qs << sft : qs >> (-sft);
    cnt = static_cast<uint32_t>((qs >> 15) + (qs >> 21)) + 2u;
    err = (mid >> 18) + 2ull + (sft >= 1 ? static_cast<unsigned long long>(cnt) << (sft - 1)
                                         : static_cast<unsigned long long>(cnt));
}

// Top-k rows with k <= KFAST: the rank each CTA's bound is taken at (see pass 1).
__device__ __forceinline__ int kfast_nth(int k, int C) { return C > 1 ? (k + C - 2) / (C - 1) : k; }

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
    int64_t slice;  // logits per CTA (a multiple of 16)
    int32_t G;      // clusters in the persistent grid
    UnitResult *res;
    int32_t *status;
    // per row, the first position found rejected so far (0xFFFFFFFF: none), or nullptr: a
    // unit behind a rejected position of its row skips its draw, which no output reads
    uint32_t *dead;
    int32_t pmajor;  // units position-major (u = j B + b) rather than row-major (u = b (D+1) + j)
    // p_target or p_draft requested: every draft position's probabilities are an output;
    // otherwise only the positions up to a row's first rejection are read
    int32_t need_p;
};

__device__ __forceinline__ bool row_sampled(const Params &P, int64_t b) {
    const float t = P.tau[b];
    const float p = P.topp ? P.topp[b] : 1.0f;
    return t > 0.0f && p > 0.0f;  // rows with tau = 0 or bad parameters are greedy
}

// ---------------------------------------------------------------- the persistent kernel

// KT: the call passes per-row top-k values.  Without them no row has a top-k filter, and
// the top-k paths (counting histograms, the bound of small k, the draw from candidates)
// compile out of the instance that runs.  EA: a decode loop's call with draft logits and
// without top-k values (no p_target, p_draft), whose top-p drafts may be seen accepted at
// E1; the other instances compile that path out.
template <typename T, bool KT, bool EA>
__global__ void __launch_bounds__(NT, CPS) k_verify_rr(const Params P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Shared &sh = *reinterpret_cast<Shared *>(smem_raw);
    constexpr int EPV = elems_per_16B<T>::value;
    const size_t data_off = (sizeof(Shared) + 127) & ~static_cast<size_t>(127);
    const size_t row_bytes =
        ((static_cast<size_t>(P.slice) * sizeof(T)) + 127) & ~static_cast<size_t>(127);
    // without draft logits (a one-hot draft) only the target row is staged; the draft row's
    // slice then aliases it, so that reads of it stay in bounds (their values go unused)
    const bool one_hot = P.Q == nullptr;
    auto sdat = [&](int row) -> T * {
        return reinterpret_cast<T *>(smem_raw + data_off + (one_hot ? 0 : row * row_bytes));
    };

    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int g = static_cast<int>(cluster_index());
    const int D = P.D;
    const int V = static_cast<int>(P.V);
    const int U = static_cast<int>(P.B) * (D + 1);
    const int G = P.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = static_cast<int>(rank) * static_cast<int>(P.slice);
    const int n = max(0, min(V - lo, static_cast<int>(P.slice)));
    const int nvb = n / EPV;               // whole vectors (bulk-copied when aligned)
    const int nvr = (n + EPV - 1) / EPV;   // vectors with the ragged one
    const int blk = (nvb + NCH - 1) / NCH;  // whole vectors per bulk-copy chunk
    const int capc = CAPT / static_cast<int>(C);

    // ---- set-up
    if (tid == 0) {
        for (int r = 0; r < 2; ++r)
            for (int c = 0; c < NCH; ++c) mbar_init(&sh.dbar[r][c], 1);
        for (int i = 0; i < NXB; ++i) mbar_init(&sh.xbar[i], C);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh.flags = 0;
    }
    __syncthreads();
    cluster_arrive_release();  // peers may touch this CTA's shared memory after the wait below
    pdl_launch_dependents();   // the greedy-row kernel runs beside this grid

    // many units run position-major (u = j * B + b), so that a row's earlier positions are
    // usually decided before its later ones start; a few run row-major (u = b * (D + 1) + j)
    const int Bi = static_cast<int>(P.B);
    const bool pmajor = P.pmajor != 0;
    auto unit_row = [&](int u) -> int { return pmajor ? u % Bi : u / (D + 1); };
    auto load_params = [&](int u) -> UnitParams {
        UnitParams q;
        q.b = unit_row(u);
        q.j = pmajor ? u / Bi : u - q.b * (D + 1);
        q.tau = P.tau[q.b];
        q.kk = P.topk ? P.topk[q.b] : 0;
        q.pp = P.topp ? P.topp[q.b] : 1.0f;
        q.d = q.j < D ? P.d[q.b * D + q.j] : -1;
        return q;
    };
    // one whole warp (of CTA 0): the first unit after unit `from` in this cluster's sequence
    // that is sampled and has an output to give: not behind a position of its row already
    // seen rejected, when that position's outputs are not read (the bonus unit, j = D, or
    // any position when p_target and p_draft are not requested; a flag not yet set only
    // costs that unit's work), with its parameters, into slot `slot` of e1su / e1sp.  Each
    // lane loads a candidate's parameters, so 32 candidates cost one round of loads.
    auto find_next = [&](int from, int slot) {
        int found = -1;
        for (int base = from + G; from >= 0 && base < U && found < 0; base += 32 * G) {
            const int cand = base + lane * G;
            UnitParams q = {0, 0, 0.0f, 1.0f, 0, -1};
            if (cand < U) q = load_params(cand);
            const bool dead = P.dead && (q.j == D || !P.need_p) &&
                              *reinterpret_cast<volatile const uint32_t *>(P.dead + q.b) < static_cast<uint32_t>(q.j);
            const unsigned msk = __ballot_sync(0xFFFFFFFFu, cand < U && q.tau > 0.0f && q.pp > 0.0f && !dead);
            if (msk) {
                const int l = __ffs(msk) - 1;
                found = __shfl_sync(0xFFFFFFFFu, cand, l);
                if (lane == l) sh.e1sp[slot] = NextParams{q.tau, q.pp, q.kk, q.d};
            }
        }
        if (lane == 0) sh.e1su[slot] = found;
    };
    auto row_ptr = [&](int b, int j, int r) -> const T * {
        return r == 0 ? static_cast<const T *>(P.T) + (static_cast<int64_t>(b) * (D + 1) + j) * V + lo
                      : static_cast<const T *>(P.Q) + (static_cast<int64_t>(b) * D + j) * V + lo;
    };
    auto next_unit = [&](int u) -> int {
        for (u += G; u < U; u += G)
            if (row_sampled(P, unit_row(u))) return u;
        return -1;
    };
    // lane 0 of warps 0 .. 2 * NCH - 1: arm chunk barrier (warp / NCH, warp % NCH) exactly
    // once for unit (b, j), with a bulk copy of the 16-byte-aligned body of that chunk
    // one thread: ask L2 to fetch unit (b, j)'s slices ahead of their bulk copies
    auto prefetch_l2 = [&](int b, int j) {
        for (int r = 0; r < (j < D && !one_hot ? 2 : 1); ++r) {
            const T *src = row_ptr(b, j, r);
            if (nvb == 0 || (reinterpret_cast<uintptr_t>(src) & 15u) != 0) continue;
            for (int c = 0; c < NCH; ++c) {
                const int v0 = min(nvb, c * blk), v1 = min(nvb, (c + 1) * blk);
                if (v1 > v0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + v0 * EPV),
                                 "r"(static_cast<uint32_t>(v1 - v0) * 16u)
                                 : "memory");
            }
        }
    };
    auto issue = [&](int b, int j, bool after_reads) {
        if (lane != 0 || warp >= 2 * NCH) return;
        const int r = warp / NCH, c = warp % NCH;
        const int nrows = j < D && !one_hot ? 2 : 1;
        const T *src = r < nrows ? row_ptr(b, j, r) : nullptr;
        const bool bulk = r < nrows && nvb > 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
        const int v0 = min(nvb, c * blk), v1 = min(nvb, (c + 1) * blk);
        if (bulk && v1 > v0) {
            if (after_reads) fence_proxy_async_smem();
            const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
            mbar_expect_tx(&sh.dbar[r][c], bytes);
            bulk_copy_g2s(sdat(r) + v0 * EPV, src + v0 * EPV, bytes, &sh.dbar[r][c]);
        } else {
            mbar_arrive(&sh.dbar[r][c]);
        }
    };

    uint32_t ph = 0;      // current phase parity of each exchange barrier (bit i)
    uint32_t sstep = 0;   // exact-search exchanges so far
    bool xdead = false;   // an exchange wait gave up: skip the remaining waits
    auto xwait = [&](int i) {
        const uint32_t par = (ph >> i) & 1u;
        ph ^= 1u << i;
        if (xdead) return;
        if (!xbar_wait_bounded(&sh.xbar[i], par)) {
            xdead = true;
            atomicOr(&sh.flags, 2);
        }
    };

    // one whole warp: the bin of h (256 bins, scanned from the top) where the count of
    // values, starting from `above`, reaches nth; out[0] = the bin, out[1] = the count in the
    // bins above it
    auto pick_bin = [&](const uint32_t *h, uint32_t above, uint32_t nth, uint32_t *out) {
        const int top = 255 - 8 * lane;
        uint32_t s = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) s += h[top - t];
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, above + incl >= nth);
        const int hl = hit ? __ffs(hit) - 1 : 31;
        if (lane == hl) {
            uint32_t acc = above + incl - s;
            int bin = top - 7;
            for (int t = 0; t < 8; ++t) {
                const uint32_t c = h[top - t];
                if (acc + c >= nth) {
                    bin = top - t;
                    break;
                }
                acc += c;
            }
            out[0] = static_cast<uint32_t>(bin);
            out[1] = acc;
        }
    };
    // The nth largest of the threads' values t0 (row 0) and t1 (row 1), rounded down to the
    // lowest value of its 16-bit key prefix: two rounds of a 256-bin radix selection over
    // the order keys, in the zeroed histogram storage (row r: the first round's bins at
    // r * RSN, the second's at r * RSN + 256, the picks at r * RSN + 512).  nth <= NT, so
    // a bin always holds it; a bound within the bin of -inf is -inf.
    auto kth_bound = [&](float t0, float t1, int nth, int rows, float &o0, float &o1) {
        uint32_t *hs = &sh.a.h.hloc[0][0];
        const uint32_t key[2] = {order_key(t0), order_key(t1)};
        for (int r = 0; r < rows; ++r) atomicAdd(&hs[r * RSN + (key[r] >> 24)], 1u);
        __syncthreads();
        if (warp < rows) pick_bin(hs + warp * RSN, 0u, static_cast<uint32_t>(nth), hs + warp * RSN + 512);
        __syncthreads();
        for (int r = 0; r < rows; ++r)
            if ((key[r] >> 24) == hs[r * RSN + 512]) atomicAdd(&hs[r * RSN + 256 + ((key[r] >> 16) & 255u)], 1u);
        __syncthreads();
        if (warp < rows)
            pick_bin(hs + warp * RSN + 256, hs[warp * RSN + 513], static_cast<uint32_t>(nth), hs + warp * RSN + 514);
        __syncthreads();
        float o[2] = {-INFINITY, -INFINITY};
        for (int r = 0; r < rows; ++r) {
            const uint32_t edge = (hs[r * RSN + 512] << 24) | (hs[r * RSN + 514] << 16);
            o[r] = edge > order_key(-INFINITY) ? key_to_float(edge) : -INFINITY;
        }
        o0 = o[0];
        o1 = o[1];
    };
    static_assert(RSN >= 516 && KFAST <= NT, "the selection's bins and picks fit a histogram row");

    int u = -1;
    if (g < U) u = row_sampled(P, unit_row(g)) ? g : next_unit(g);
    UnitParams cnx = {0, 0, 1.0f, 1.0f, 0, -1};  // this unit's parameters
    UnitParams nxt = {0, 0, 1.0f, 1.0f, 0, -1};  // the next unit's
    int un = -1;
    if (u >= 0) {
        cnx = load_params(u);
        issue(cnx.b, cnx.j, false);
        un = next_unit(u);
        if (un >= 0) nxt = load_params(un);
    }
    // CTA 0 holds the cluster's third unit for its first E1 message
    if (rank == 0 && tid == 0) {
        const int u2 = un >= 0 ? next_unit(un) : -1;
        sh.e1su[0] = u2;
        if (u2 >= 0) {
            const UnitParams q = load_params(u2);
            sh.e1sp[0] = NextParams{q.tau, q.pp, q.kk, q.d};
        }
    }
    bool started = false;

    for (int k = 0; u >= 0; ++k) {
        const UnitParams cur = cnx;
        const uint32_t dpar = static_cast<uint32_t>(k & 1);
        const int ep = k & 1;
        const int b = cur.b, j = cur.j;
        const float tau = cur.tau, pp = cur.pp;
        const int32_t kk = cur.kk, d = cur.d;
        const int nrows = j < D && !one_hot ? 2 : 1;
        const bool k_on = KT && kk >= 1 && kk < V;
        const bool p_on = pp < 1.0f;
        const bool kfast = k_on && kk <= KFAST;
        const float c2 = __fdiv_rn(1.44269504088896340736f, tau);
        const bool dvalid = d >= 0 && d < V;
        const bool d_here = dvalid && d >= lo && d < lo + n;
        // a decode loop's top-p draft may be seen accepted at E1 (see the decision after the
        // row statistics): pass 1 then also sums the target mass above the draft token's logit
        const bool e1try = EA && !P.need_p && j < D && dvalid && !k_on && p_on;
        const float xdt =
            e1try ? widen(static_cast<const T *>(P.T)[(static_cast<int64_t>(b) * (D + 1) + j) * V + d]) : 0.0f;

        // the parts the bulk copies do not cover: a ragged tail, or a misaligned row
        for (int r = 0; r < nrows; ++r) {
            const T *src = row_ptr(b, j, r);
            const bool bulk = nvb > 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
            T *dst = sdat(r);
            for (int i = (bulk ? nvb * EPV : 0) + tid; i < nvr * EPV; i += NT)
                dst[i] = i < n ? src[i] : neg_inf<T>();
        }
        if (tid == 0) {
            sh.lcnt[0] = sh.lcnt[1] = 0;
            sh.fpick[0] = sh.fpick[1] = -INFINITY;
        }
        if (k_on || p_on)
            for (int i = tid; i < 2 * RSN; i += NT) (&sh.a.h.hloc[0][0])[i] = 0;
        __syncthreads();
        // this CTA's view of the row's first rejection, sent with E1 (only this CTA writes its
        // own slot): the load's latency hides in pass 1's wait for the unit's data
        if (tid == 0)
            sh.e1k[ep][rank] = P.dead ? *reinterpret_cast<volatile const uint32_t *>(P.dead + b) : 0xFFFFFFFFu;

        // ---- pass 1: the maxima of both rows' slices, chunk by chunk as the bulk copies land
        // (the ragged tail and misaligned rows are already in place), then the softmax sums
        // relative to this CTA's maxima.  Two plain sweeps: no per-element branch.
        const bool filt = k_on || p_on;
        const uint4 *sv0 = reinterpret_cast<const uint4 *>(sdat(0));
        const uint4 *sv1 = reinterpret_cast<const uint4 *>(sdat(1));
        float cm0, cm1, cs0, cs1, cab = 0.0f;
        {
            float mx0 = -INFINITY, mx1 = -INFINITY;
            bool timed_out = false;
            for (int c = 0; c < NCH; ++c) {
                if (!mbar_wait_bounded(&sh.dbar[0][c], dpar)) timed_out = true;
                if (!mbar_wait_bounded(&sh.dbar[1][c], dpar)) timed_out = true;
                const int v1 = min(nvb, (c + 1) * blk);
#pragma unroll 2
                for (int v = c * blk + tid; v < v1; v += NT) {
                    mx0 = fmaxf(mx0, vec_max<T>(sv0[v]));
                    if (nrows > 1) mx1 = fmaxf(mx1, vec_max<T>(sv1[v]));
                }
            }
            for (int v = nvb + tid; v < nvr; v += NT) {
                mx0 = fmaxf(mx0, vec_max<T>(sv0[v]));
                if (nrows > 1) mx1 = fmaxf(mx1, vec_max<T>(sv1[v]));
            }
            if (timed_out) atomicOr(&sh.flags, 1);
            if (d_here && tid == 0) {  // every chunk has landed for this thread
                sh.xd[0] = widen(sdat(0)[d - lo]);
                sh.xd[1] = widen(sdat(1)[d - lo]);
            }
            // top-k with a small k: the kth-largest of the threads' maxima, rounded down to its
            // 16-bit key prefix, has at least kth elements of this slice at or above it (kth =
            // ceil(k / (C - 1))); the kq-th largest of these bounds over the C CTAs (kq =
            // ceil(k / kth) <= C) then has at least k elements of the row at or above it, so it
            // lies at or below the row's k-th largest logit, and a CTA with a short slice does
            // not weaken it
            float bd0 = -INFINITY, bd1 = -INFINITY;
            if (kfast) kth_bound(mx0, mx1, kfast_nth(kk, static_cast<int>(C)), nrows, bd0, bd1);
            mx0 = warp_max(mx0);
            mx1 = warp_max(mx1);
            if (lane == 0) {
                sh.w.p1.rf[0][warp] = mx0;
                sh.w.p1.rf[1][warp] = mx1;
            }
            __syncthreads();
            // every warp reduces the warps' maxima the same way
            cm0 = warp_max(lane < NW ? sh.w.p1.rf[0][lane] : -INFINITY);
            cm1 = warp_max(lane < NW ? sh.w.p1.rf[1][lane] : -INFINITY);
            if (kfast) {
                // the top-k set is renormalised on its own: no row sum is needed, and the E1
                // message carries the bounds in its place
                cs0 = bd0;
                cs1 = bd1;
            } else {
                // z = x * c2 + nm, nm = -cm * c2 (0 for a slice of -inf alone, whose sum is 0)
                const float nm0 = cm0 > -INFINITY ? -cm0 * c2 : 0.0f;
                const float nm1 = cm1 > -INFINITY ? -cm1 * c2 : 0.0f;
                float a0 = 0.0f, a1 = 0.0f, ab = 0.0f;
                if (e1try) {
#pragma unroll 2
                    for (int v = tid; v < nvr; v += NT) {
                        a0 += vec_sum_ex2_above<T>(sv0[v], c2, nm0, xdt, ab);
                        if (nrows > 1) a1 += vec_sum_ex2<T>(sv1[v], c2, nm1);
                    }
                } else {
#pragma unroll 2
                    for (int v = tid; v < nvr; v += NT) {
                        a0 += vec_sum_ex2<T>(sv0[v], c2, nm0);
                        if (nrows > 1) a1 += vec_sum_ex2<T>(sv1[v], c2, nm1);
                    }
                }
                a0 = warp_sum_f32(a0);
                a1 = warp_sum_f32(a1);
                if (e1try) ab = warp_sum_f32(ab);
                if (lane == 0) {
                    sh.w.p1.rs[0][warp] = a0;
                    sh.w.p1.rs[1][warp] = a1;
                    if (e1try) sh.w.p1.ra[warp] = ab;
                }
                __syncthreads();
                cs0 = warp_sum_f32(lane < NW ? sh.w.p1.rs[0][lane] : 0.0f);
                cs1 = warp_sum_f32(lane < NW ? sh.w.p1.rs[1][lane] : 0.0f);
                if (e1try) cab = warp_sum_f32(lane < NW ? sh.w.p1.ra[lane] : 0.0f);
            }
        }
        if (!started) {
            cluster_wait_acquire();  // every CTA of the cluster has initialised its barriers
            started = true;
        }

        // ---- E1: warp 0 sends this CTA's maxima and sums, and the draft token's logits, to
        // every CTA
        if (warp == 0 && lane < static_cast<int>(C)) {
            const float4 part = make_float4(cm0, cs0, cm1, cs1);  // row 1: (-inf, 0) when absent
            st_peer_v4(peer_addr(smem_addr(&sh.e1[ep][rank]), lane), part);
            if (lane != static_cast<int>(rank))
                st_peer_u32(peer_addr(smem_addr(&sh.e1k[ep][rank]), lane), sh.e1k[ep][rank]);
            if (e1try) st_peer_u32(peer_addr(smem_addr(&sh.e1ab[ep][rank]), lane), __float_as_uint(cab));
            if (d_here) st_peer_v2(peer_addr(smem_addr(&sh.e1d[ep]), lane), make_float2(sh.xd[0], sh.xd[1]));
            if (rank == 0 && lane != 0) {  // the unit after the next one, and its parameters
                const NextParams q = sh.e1sp[ep];
                st_peer_u32(peer_addr(smem_addr(&sh.e1su[ep]), lane), static_cast<uint32_t>(sh.e1su[ep]));
                st_peer_v4(peer_addr(smem_addr(&sh.e1sp[ep]), lane),
                           make_float4(q.tau, q.pp, __int_as_float(q.kk), __int_as_float(q.d)));
            }
            xarrive(&sh.xbar[XB_E1 + ep], lane);
        }
        if (warp == NW - 1) {  // work whose latency the wait hides
            if (lane == 0) {
                if (un >= 0) prefetch_l2(nxt.b, nxt.j);
                uint32_t c4[4] = {static_cast<uint32_t>(b), static_cast<uint32_t>(j), 0u, 0u};
                philox(c4, static_cast<uint32_t>(P.seed), static_cast<uint32_t>(P.seed >> 32));
                sh.uwd[0] = c4[0];
                sh.uwd[1] = c4[1];
            }
            if (rank == 0) find_next(sh.e1su[ep], ep ^ 1);  // sent with the next E1
        }
        xwait(XB_E1 + ep);

        // ---- row statistics (every CTA, identical): warp 0 merges the CTAs' partials
        if (warp == 0) {
            const int r = lane >> 4, c = lane & 15;
            const bool in = r < nrows && c < static_cast<int>(C);
            float tm = -INFINITY, ts = 0.0f;
            if (in) {
                const float4 e = sh.e1[ep][c];
                tm = r == 0 ? e.x : e.z;
                ts = r == 0 ? e.y : e.w;
            }
            if (kfast) {
                // the maximum, and the kq-th largest of the CTAs' bounds: kq CTAs hold at
                // least kth elements each at or above it, kq * kth >= k
                const int kth = kfast_nth(kk, static_cast<int>(C));
                const int kq = (kk + kth - 1) / kth;
                int rk = 0;
                for (int q = 0; q < static_cast<int>(C); ++q) {
                    const float y = __shfl_sync(0xFFFFFFFFu, ts, (lane & 16) | q);
                    if (y > ts || (y == ts && q < c)) ++rk;
                }
                const unsigned hm = __ballot_sync(0xFFFFFFFFu, in && rk == kq - 1) & (r ? 0xFFFF0000u : 0x0000FFFFu);
                ts = __shfl_sync(0xFFFFFFFFu, ts, hm ? __ffs(hm) - 1 : lane);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, o));
            } else {
                if (e1try) {
                    // the target's mass above the draft token, rescaled like the sums
                    float ta = (in && r == 0) ? sh.e1ab[ep][c] : 0.0f;
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) {
                        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, tm, o);
                        const float a2 = __shfl_xor_sync(0xFFFFFFFFu, ta, o);
                        const float M = fmaxf(tm, m2);
                        ta = (ta > 0.0f ? ta * ex2(__fmul_rn(tm - M, c2)) : 0.0f) +
                             (a2 > 0.0f ? a2 * ex2(__fmul_rn(m2 - M, c2)) : 0.0f);
                        tm = M;
                    }
                    if (lane == 0) sh.above = ta;
                    tm = (r < nrows && c < static_cast<int>(C)) ? (r == 0 ? sh.e1[ep][c].x : sh.e1[ep][c].z) : -INFINITY;
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, tm, o);
                    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, ts, o);
                    ms_merge(tm, ts, m2, s2, c2);
                }
            }
            if (c == 0 && r < nrows) {
                sh.m[r] = tm;
                sh.nmc[r] = tm > -INFINITY ? -tm * c2 : 0.0f;
                sh.tzb[r] = tm * (c2 * static_cast<float>(R));
                sh.deg[r] = !(tm > -INFINITY);
                sh.mode[r] = 0;
                sh.theta[r] = -INFINITY;
                sh.Z[r] = kfast ? 1.0f : ts;
                // the fixed-point top-p target of the plan
                sh.tgt[r] = kfast ? 0ull : fx_target(pp, ts);
                if (kfast) sh.kbd[r] = ts;
                // the bins that can hold a top-p boundary: a kept token weighs at least
                // (1 - p) Z / V, since the tokens below that level weigh less than (1 - p) Z
                // together
                float zc = -static_cast<float>(ZR);
                if (!k_on && ts > 0.0f) {
                    const float lvl = __log2f((1.0f - pp) * ts / static_cast<float>(V));
                    // Z <= V keeps the level below 0; the clamps keep at least one bin for
                    // any input (NaN included)
                    zc = fminf(fmaxf(zc, lvl - 2.0f / R), -1.0f / R);
                }
                sh.nbu[r] = k_on ? NB : min(NB, static_cast<int>(-zc * R) + 1);
            }
        }
        __syncthreads();

        // A row's bonus unit is read only when every draft of the row is accepted, and (when
        // p_target and p_draft are not requested) a draft position only up to the row's first
        // rejection.  When the cluster's agreed view of the row (exchanged at E1) already holds
        // a rejection before such a unit, its filters are not computed, and its draw is
        // skipped below; its record is never read.
        uint32_t dk1 = 0xFFFFFFFFu;
        for (uint32_t c = 0; c < C; ++c) dk1 = min(dk1, sh.e1k[ep][c]);
        const bool dead_unit = (j == D || !P.need_p) && dk1 < static_cast<uint32_t>(j);
        // ---- A decode loop reads a draft position's record only for its accept flag when
        // the draft is accepted.  At E1 every CTA knows each row's sum Z and the target mass
        // strictly above the draft token's logit.  The token's group is then surely kept if
        // that mass lies below the top-p target.  A kept mass lies between its target
        // (p Z) and Z, so p/q is at least (w_t / w_q) p Z_q / Z_t, and a draft the draft row
        // drops (q = 0) is accepted anyway.  When U_acc lies below that bound (with a
        // relative slack for the sums' rounding), the acceptance is certain: the filters
        // are skipped and the staged rows released at once.  Every CTA decides from the
        // same exchanged values.
        bool early = false;  // the draft's acceptance is already certain
        if (e1try && !dead_unit) {
            if (tid == 0) {
                const float2 xdv = sh.e1d[ep];
                const float u = word_uniform(sh.uwd[0]);
                bool ok = !sh.deg[0] && sh.above < pp * sh.Z[0] * (1.0f - 1e-4f);
                if (ok) {
                    if (one_hot) {
                        ok = u <= ex2(fmaf(xdv.x, c2, sh.nmc[0])) / sh.Z[0] * (1.0f - 1e-4f);
                    } else if (sh.deg[1]) {
                        ok = false;
                    } else {
                        const float r0 = ex2(__fmul_rn((xdv.x - sh.m[0]) - (xdv.y - sh.m[1]), c2));
                        ok = u <= r0 * (pp * sh.Z[1] / sh.Z[0]) * (1.0f - 1e-4f);
                    }
                }
                sh.early = ok ? 1 : 0;
            }
            __syncthreads();
            early = sh.early != 0;
        }
        if (filt && !dead_unit && !early) {
            if (!kfast) {
                // ---- pass 2: histogram of the elements in the bins that can hold the boundary.
                // Top-k counts them; top-p adds each element's weight scaled by its bin's octave,
                // round(w * 2^(16 + o)): an exponent add, then rounding by the sum with 2^23.  Bin
                // and weight leave fp32 without conversion instructions.  One shared atomic per
                // element: its cost grows with the lanes it serves, which the bins' range keeps
                // few.
                constexpr float MAG = 8388608.0f;  // 2^23
                const float tza = -c2 * static_cast<float>(R);
                if (nrows > 1 && !sh.deg[0] && !sh.deg[1] && !k_on) {
                    // both rows in one sweep: twice the independent work per iteration
                    const float nmA = sh.nmc[0], tzbA = sh.tzb[0], fnbA = static_cast<float>(sh.nbu[0]);
                    const float nmB = sh.nmc[1], tzbB = sh.tzb[1], fnbB = static_cast<float>(sh.nbu[1]);
                    uint32_t *hA = sh.a.h.hloc[0];
                    uint32_t *hB = sh.a.h.hloc[1];
                    auto bin_w = [&](float x, float nm, float tzb, float fnb, uint32_t *hh) {
                        const float tz = fmaxf(fmaf(x, tza, tzb), 0.0f);
                        const float tb = __fadd_rz(tz, MAG);
                        const int bn = __float_as_int(tb) - 0x4B000000;
                        const float ws = __uint_as_float(__float_as_uint(ex2(fmaf(x, c2, nm))) +
                                                         (static_cast<uint32_t>((bn >> 5) + 16) << 23));
                        const uint32_t q = __float_as_uint(ws + MAG) - 0x4B000000u;
                        if (tz < fnb) atomicAdd(&hh[bn], q);
                    };
#pragma unroll 2
                    for (int v = tid; v < nvr; v += NT) {
                        float xa[EPV], xb[EPV];
                        unpack(sv0[v], xa);
                        unpack(sv1[v], xb);
#pragma unroll
                        for (int e = 0; e < EPV; ++e) {
                            bin_w(xa[e], nmA, tzbA, fnbA, hA);
                            bin_w(xb[e], nmB, tzbB, fnbB, hB);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int r = 0; r < nrows; ++r) {
                        if (sh.deg[r]) continue;
                        const float nm = sh.nmc[r], tzb = sh.tzb[r];
                        const float fnb = static_cast<float>(sh.nbu[r]);
                        uint32_t *hh = sh.a.h.hloc[r];
                        if (k_on) {
                            for_row(sdat(r), nvr, [&](float x, int) {
                                const float tz = fmaxf(fmaf(x, tza, tzb), 0.0f);
                                const float tb = __fadd_rz(tz, MAG);  // 2^23 + trunc(tz) below 2^23
                                if (tz < fnb) atomicAdd(&hh[__float_as_int(tb) - 0x4B000000], 1u);
                            });
                        } else {
                            for_row(sdat(r), nvr, [&](float x, int) {
                                // -z * R >= 0 (clamped: rounding can make it a hair negative at the
                                // maximum); bins at its integer part
                                const float tz = fmaxf(fmaf(x, tza, tzb), 0.0f);
                                const float tb = __fadd_rz(tz, MAG);
                                const int bn = __float_as_int(tb) - 0x4B000000;
                                const float ws = __uint_as_float(__float_as_uint(ex2(fmaf(x, c2, nm))) +
                                                                 (static_cast<uint32_t>((bn >> 5) + 16) << 23));
                                const uint32_t q = __float_as_uint(ws + MAG) - 0x4B000000u;
                                if (tz < fnb) atomicAdd(&hh[bn], q);
                            });
                        }
                    }
                }
                __syncthreads();
                // ---- E2a: reduce-scatter in groups of four bins, each CTA's bins to their owner
                const int nb0 = sh.nbu[0], nb1 = nrows > 1 ? sh.nbu[1] : 0;
                const int rs0 = (((nb0 + C - 1) / C) + 3) & ~3, rs1 = (((nb1 + C - 1) / C) + 3) & ~3;
                const int g0 = static_cast<int>(C) * (rs0 >> 2), g1 = static_cast<int>(C) * (rs1 >> 2);
                for (int idx = tid; idx < g0 + g1; idx += NT) {
                    const int r = idx < g0 ? 0 : 1;
                    const int q4 = r == 0 ? idx : idx - g0;  // group of 4 bins, in bin order
                    const int rsz = r == 0 ? rs0 : rs1;
                    const int owner = (q4 * 4) / rsz, kq = q4 * 4 - owner * rsz;
                    const uint4 v = *reinterpret_cast<const uint4 *>(&sh.a.h.hloc[r][q4 * 4]);
                    st_peer_u32x4(peer_addr(smem_addr(&sh.a.h.rsin[r][static_cast<int>(rank) * rsz + kq]), owner), v);
                }
                __syncthreads();
                if (tid < static_cast<int>(C)) xarrive(&sh.xbar[XB_RS], tid);
                xwait(XB_RS);
                // ---- E2b: sum the owned bins (in 64 bits: a bin of the whole row can exceed 32)
                // and broadcast them, two bins per store
                for (int idx = tid; idx < ((rs0 + rs1) >> 1); idx += NT) {
                    const int r = idx < (rs0 >> 1) ? 0 : 1;
                    const int kq = (r == 0 ? idx : idx - (rs0 >> 1)) * 2;
                    const int rsz = r == 0 ? rs0 : rs1;
                    unsigned long long c0 = 0, c1 = 0;
                    for (uint32_t c = 0; c < C; ++c) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(&sh.a.h.rsin[r][c * rsz + kq]);
                        c0 += v.x;
                        c1 += v.y;
                    }
                    // bin b goes to [b % BPL][b / BPL] (bins past NB lie past every used range)
                    const int b0 = static_cast<int>(rank) * rsz + kq;
                    const uint32_t a0 = smem_addr(&sh.b.hist[r][(b0 % BPL) * PL + b0 / BPL]);
                    const uint32_t a1 = smem_addr(&sh.b.hist[r][((b0 + 1) % BPL) * PL + (b0 + 1) / BPL]);
                    for (uint32_t c = 0; c < C; ++c) {
                        if (b0 < NB) st_peer_u64(peer_addr(a0, c), c0);
                        if (b0 + 1 < NB) st_peer_u64(peer_addr(a1, c), c1);
                    }
                }
                __syncthreads();
                if (tid < static_cast<int>(C)) xarrive(&sh.xbar[XB_AG], tid);
                xwait(XB_AG);

                // ---- plan per row: the bin range that holds the boundary, or the exact search.
                // The PW warps of group r take row r, BPL bins a lane (the gathered histogram is
                // stored transposed, bin b at [b % BPL][b / BPL], so that these loads are free of
                // bank conflicts); scans of the per-bin counts (top-k) or weights and their
                // margins (top-p) over the group's lanes find the crossing bins and the exact
                // weight of the bins before them.  The other warps go on to the barrier.
                {
                    const int r = warp / PW, j = tid - r * PL, hw = warp - r * PW;
                    if (r < nrows && !sh.deg[r]) {
                        const int nbu = sh.nbu[r];
                        const unsigned long long tgt = k_on ? 0ull : sh.tgt[r];
                        const unsigned long long *hr = sh.b.hist[r];
                        // weight, margin and element-count bound of bin bn (0 past the used bins)
                        auto bounds = [&](int bn, unsigned long long &bm, unsigned long long &be, uint32_t &bc) {
                            bm = be = 0;
                            bc = 0;
                            if (bn < nbu) {
                                const unsigned long long qs = hr[(bn % BPL) * PL + bn / BPL];
                                if (k_on) bc = static_cast<uint32_t>(qs);
                                else bin_bounds(qs, bn, bm, be, bc);
                            }
                        };
                        unsigned long long m_s = 0, e_s = 0;
                        uint32_t cn_s = 0;
#pragma unroll
                        for (int t = 0; t < BPL; ++t) {
                            unsigned long long bm, be;
                            uint32_t bc;
                            bounds(BPL * j + t, bm, be, bc);
                            m_s += bm;
                            e_s += be;
                            cn_s += bc;
                        }
                        unsigned long long m_i = m_s, e_i = e_s;
                        uint32_t cn_i = cn_s;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const unsigned long long a1 = __shfl_up_sync(0xFFFFFFFFu, m_i, o);
                            const unsigned long long a2 = __shfl_up_sync(0xFFFFFFFFu, e_i, o);
                            const uint32_t a3 = __shfl_up_sync(0xFFFFFFFFu, cn_i, o);
                            if (lane >= o) {
                                m_i += a1;
                                e_i += a2;
                                cn_i += a3;
                            }
                        }
                        if (lane == 31) {
                            sh.w.pl.lo[warp] = m_i;
                            sh.w.pl.hi[warp] = e_i;
                            sh.w.pl.cn[warp] = cn_i;
                        }
                        if (j == 0) {
                            sh.pb1[r] = nbu;
                            sh.pb2[r] = nbu;
                            sh.pcc1[r] = 0;
                            sh.pcc2[r] = 0;
                            sh.pma[r] = 0;
                        }
                        group_barrier<PL>(r);
                        // the group's earlier warps, and the row's total count
                        uint32_t cn_tot = 0;
#pragma unroll
                        for (int q = 0; q < PW; ++q) {
                            const int wi = r * PW + q;
                            if (q < hw) {
                                m_i += sh.w.pl.lo[wi];
                                e_i += sh.w.pl.hi[wi];
                                cn_i += sh.w.pl.cn[wi];
                            }
                            cn_tot += sh.w.pl.cn[wi];
                        }
                        if (k_on) {
                            // the bin holding the k-th largest value; every bin up to it is gathered
                            const uint32_t need = static_cast<uint32_t>(kk);
                            if (cn_i - cn_s < need && cn_i >= need) {
                                uint32_t acc = cn_i - cn_s;
                                for (int t = 0; t < BPL; ++t) {
                                    unsigned long long bm, be;
                                    uint32_t bc;
                                    bounds(BPL * j + t, bm, be, bc);
                                    acc += bc;
                                    if (acc >= need) {
                                        sh.pb2[r] = BPL * j + t;
                                        sh.pcc2[r] = acc;
                                        break;
                                    }
                                }
                            }
                        } else {
                            // b1: the first bin whose upper cumulative bound reaches the target
                            // (every earlier bin is kept whole); b2: the first whose lower bound
                            // reaches it (every later bin is dropped)
                            if (m_i + e_i - (m_s + e_s) < tgt && m_i + e_i >= tgt) {
                                unsigned long long am = m_i - m_s, ae = e_i - e_s;
                                uint32_t cb = cn_i - cn_s;
                                for (int t = 0; t < BPL; ++t) {
                                    unsigned long long bm, be;
                                    uint32_t bc;
                                    bounds(BPL * j + t, bm, be, bc);
                                    if (am + bm + ae + be >= tgt) {
                                        sh.pb1[r] = BPL * j + t;
                                        sh.pcc1[r] = cb;
                                        sh.pma[r] = am;
                                        break;
                                    }
                                    am += bm;
                                    ae += be;
                                    cb += bc;
                                }
                            }
                            const unsigned long long lo_i = m_i > e_i ? m_i - e_i : 0ull;
                            const unsigned long long lo_x = (m_i - m_s) > (e_i - e_s) ? (m_i - m_s) - (e_i - e_s) : 0ull;
                            if (lo_x < tgt && lo_i >= tgt) {
                                unsigned long long am = m_i - m_s, ae = e_i - e_s;
                                uint32_t cb = cn_i - cn_s;
                                for (int t = 0; t < BPL; ++t) {
                                    unsigned long long bm, be;
                                    uint32_t bc;
                                    bounds(BPL * j + t, bm, be, bc);
                                    am += bm;
                                    ae += be;
                                    cb += bc;
                                    if (am > ae && am - ae >= tgt) {
                                        sh.pb2[r] = BPL * j + t;
                                        sh.pcc2[r] = cb;
                                        break;
                                    }
                                }
                            }
                        }
                        group_barrier<PL>(r);
                        if (j == 0) {
                            int32_t b1 = 0, b2 = sh.pb2[r];
                            uint32_t ncand;
                            bool slow;
                            if (k_on) {
                                ncand = sh.pcc2[r];
                                slow = b2 >= nbu;
                                sh.pma[r] = 0;
                            } else {
                                b1 = sh.pb1[r];
                                slow = b1 >= nbu;
                                const uint32_t c2b = b2 >= nbu ? cn_tot : sh.pcc2[r];
                                if (b2 >= nbu) b2 = nbu - 1;
                                ncand = c2b - sh.pcc1[r];
                            }
                            if (ncand > static_cast<uint32_t>(NT) || ncand == 0) slow = true;
                            sh.mode[r] = slow ? 2 : 1;
                            sh.b1[r] = b1;
                            sh.b2[r] = b2;
                            sh.lcnt[r] = 0;
                        }
                    }
                    __syncthreads();
                }
            } else {
                // every element at or above the row's bound is a candidate, and none lies
                // above the candidates
                if (tid < nrows) {
                    sh.mode[tid] = sh.deg[tid] ? 0 : 1;
                    sh.pma[tid] = 0;
                }
                __syncthreads();
            }

            // ---- A decode loop reads a draft position's record only for its accept flag when
            // the draft is accepted.  After the plan every CTA holds rigorous bounds on each
            // row's kept mass: at least the top-p target (the kept groups reach it) and less
            // than the target plus the boundary bins' weight (the last kept group lies among
            // them), with a relative slack for the sums' rounding.  When the draft token's bin
            // lies before the boundary bins (kept for sure), and U_acc lies below the ratio's
            // lower bound (or the draft surely drops the token: q(d) = 0), the acceptance is
            // certain: the gather and the thresholds are skipped, and the staged rows are
            // released at once.  Every CTA decides from the same exchanged values.
            if (!P.need_p && j < D && dvalid && !k_on && p_on) {
                if (tid == 0) {
                    const float tza = -c2 * static_cast<float>(R);
                    const float2 xdv = sh.e1d[ep];
                    auto tz_of = [&](float x, int r) { return fmaxf(fmaf(x, tza, sh.tzb[r]), 0.0f); };
                    // the row's kept mass, as the thresholds would give it, lies in [lo, hi]
                    auto zb = [&](int r, float &lo, float &hi) {
                        const unsigned long long t = sh.tgt[r];
                        unsigned long long extra = 0;
                        const int nbu = sh.nbu[r];
                        for (int bn = sh.b1[r]; bn <= sh.b2[r] && bn < nbu; ++bn) {
                            unsigned long long mid, err;
                            uint32_t cnt;
                            bin_bounds(sh.b.hist[r][(bn % BPL) * PL + bn / BPL], bn, mid, err, cnt);
                            extra += mid + err + cnt;
                        }
                        lo = fx_to_float(t) * (1.0f - 1e-4f);
                        hi = fx_to_float(t + extra) * (1.0f + 1e-4f);
                    };
                    const float u = word_uniform(sh.uwd[0]);
                    bool ok = !sh.deg[0] && sh.mode[0] == 1 && tz_of(xdv.x, 0) < static_cast<float>(sh.b1[0]);
                    if (ok) {
                        float z0lo, z0hi;
                        zb(0, z0lo, z0hi);
                        if (one_hot) {
                            ok = u <= ex2(fmaf(xdv.x, c2, sh.nmc[0])) / z0hi * (1.0f - 1e-4f);
                        } else if (sh.deg[1] || sh.mode[1] != 1) {
                            ok = false;
                        } else {
                            const float tq = tz_of(xdv.y, 1);
                            if (tq >= static_cast<float>(sh.b2[1] + 1)) {
                                ok = true;  // q(d) = 0
                            } else if (tq < static_cast<float>(sh.b1[1])) {
                                float z1lo, z1hi;
                                zb(1, z1lo, z1hi);
                                const float r0 = ex2(__fmul_rn((xdv.x - sh.m[0]) - (xdv.y - sh.m[1]), c2));
                                ok = u <= r0 * (z1lo / z0hi) * (1.0f - 1e-4f);
                            } else {
                                ok = false;
                            }
                        }
                    }
                    sh.early = ok ? 1 : 0;
                }
                __syncthreads();
                early = sh.early != 0;
            }
            if (!early) {
                // ---- gather the boundary candidates into every CTA (E3)
                const bool any_fast = sh.mode[0] == 1 || (nrows > 1 && sh.mode[1] == 1);
                if (any_fast) {
                    // the candidates of row r: elements of bins [b1, b2] (bin bn = trunc(tz):
                    // bn >= b1 iff tz >= b1, bn <= b2 iff tz < b2 + 1), or, for a top-k row with a
                    // small k, every element at or above the row's bound; a vector that holds
                    // candidates claims their slots at once (the order of the slots does not
                    // matter: every later step depends on values)
                    const float tza = -c2 * static_cast<float>(R);
                    auto in_bins = [&](const float (&x)[EPV], float tzb, float fb1, float fb2) -> uint32_t {
                        uint32_t msk = 0;
#pragma unroll
                        for (int e = 0; e < EPV; ++e) {
                            const float tz = fmaxf(fmaf(x[e], tza, tzb), 0.0f);
                            msk |= (tz >= fb1 && tz < fb2) ? (1u << e) : 0u;
                        }
                        return msk;
                    };
                    auto at_least = [&](const float (&x)[EPV], float bnd) -> uint32_t {
                        uint32_t msk = 0;
#pragma unroll
                        for (int e = 0; e < EPV; ++e) msk |= x[e] >= bnd ? (1u << e) : 0u;
                        return msk;
                    };
                    auto put = [&](int r, int v, const float (&x)[EPV], uint32_t msk) {
                        if (msk) {
                            unsigned long long *cr = &sh.a.cand[r][static_cast<int>(rank) * capc];
                            uint32_t slot = atomicAdd(&sh.lcnt[r], static_cast<uint32_t>(__popc(msk)));
#pragma unroll
                            for (int e = 0; e < EPV; ++e) {
                                if (((msk >> e) & 1u) && slot < static_cast<uint32_t>(capc))
                                    cr[slot] = (static_cast<unsigned long long>(__float_as_uint(x[e])) << 32) |
                                               static_cast<uint32_t>(lo + v * EPV + e);
                                slot += (msk >> e) & 1u;
                            }
                        }
                    };
                    if (nrows > 1 && sh.mode[0] == 1 && sh.mode[1] == 1) {
                        // both rows in one sweep
                        if (kfast) {
                            const float bA = sh.kbd[0], bB = sh.kbd[1];
#pragma unroll 2
                            for (int v = tid; v < nvr; v += NT) {
                                float xa[EPV], xb[EPV];
                                unpack(sv0[v], xa);
                                unpack(sv1[v], xb);
                                put(0, v, xa, at_least(xa, bA));
                                put(1, v, xb, at_least(xb, bB));
                            }
                        } else {
                            const float tzbA = sh.tzb[0], f1A = static_cast<float>(sh.b1[0]), f2A = static_cast<float>(sh.b2[0] + 1);
                            const float tzbB = sh.tzb[1], f1B = static_cast<float>(sh.b1[1]), f2B = static_cast<float>(sh.b2[1] + 1);
#pragma unroll 2
                            for (int v = tid; v < nvr; v += NT) {
                                float xa[EPV], xb[EPV];
                                unpack(sv0[v], xa);
                                unpack(sv1[v], xb);
                                put(0, v, xa, in_bins(xa, tzbA, f1A, f2A));
                                put(1, v, xb, in_bins(xb, tzbB, f1B, f2B));
                            }
                        }
                    } else {
#pragma unroll 1
                        for (int r = 0; r < nrows; ++r) {
                            if (sh.mode[r] != 1) continue;
                            const uint4 *vp = reinterpret_cast<const uint4 *>(sdat(r));
                            if (kfast) {
                                const float bnd = sh.kbd[r];
#pragma unroll 2
                                for (int v = tid; v < nvr; v += NT) {
                                    float x[EPV];
                                    unpack(vp[v], x);
                                    put(r, v, x, at_least(x, bnd));
                                }
                            } else {
                                const float tzb = sh.tzb[r];
                                const float fb1 = static_cast<float>(sh.b1[r]), fb2 = static_cast<float>(sh.b2[r] + 1);
#pragma unroll 2
                                for (int v = tid; v < nvr; v += NT) {
                                    float x[EPV];
                                    unpack(vp[v], x);
                                    put(r, v, x, in_bins(x, tzb, fb1, fb2));
                                }
                            }
                        }
                    }
                    __syncthreads();
                    // ---- push this CTA's candidates into the other CTAs' copies of its slots
#pragma unroll 1
                    for (int r = 0; r < nrows; ++r) {
                        if (sh.mode[r] != 1) continue;
                        const int nl = min(static_cast<int>(sh.lcnt[r]), capc);
                        const int np = static_cast<int>(C) - 1;
                        for (int q = tid; q < nl * np; q += NT) {
                            const int i = q / np, c0 = q - i * np;
                            const uint32_t c = c0 >= static_cast<int>(rank) ? static_cast<uint32_t>(c0 + 1)
                                                                             : static_cast<uint32_t>(c0);
                            unsigned long long *slot = &sh.a.cand[r][static_cast<int>(rank) * capc + i];
                            st_peer_u64(peer_addr(smem_addr(slot), c), *slot);
                        }
                    }
                    __syncthreads();
                    if (tid < static_cast<int>(C)) {
                        for (int r = 0; r < 2; ++r)
                            st_peer_u32(peer_addr(smem_addr(&sh.ccnt[rank][r]), tid), sh.lcnt[r]);
                        xarrive(&sh.xbar[XB_E3], tid);
                    }
                    xwait(XB_E3);

                    // ---- exact thresholds.  Every warp, per row (lane c holding CTA c's count):
                    // the candidates' number, the CTAs' offsets in the row's list, and whether
                    // the row can be ranked by its plan group (1 to PL candidates, no CTA over its
                    // slots)
                    uint32_t ccl[2], cpl[2];
                    int ncnt[2];
                    bool grp = true;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const bool on = r < nrows && sh.mode[r] == 1;
                        const uint32_t cc = on && lane < static_cast<int>(C) ? sh.ccnt[lane][r] : 0u;
                        const bool over = __any_sync(0xFFFFFFFFu, cc > static_cast<uint32_t>(capc));
                        uint32_t incl = cc;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                            if (lane >= o) incl += y;
                        }
                        ccl[r] = cc;
                        cpl[r] = incl - cc;
                        ncnt[r] = static_cast<int>(__shfl_sync(0xFFFFFFFFu, incl, 31));
                        if (on && (over || ncnt[r] == 0 || ncnt[r] > PL)) grp = false;
                    }
                    if (grp) {
                        // ---- rank by counting in the plan's groups (PW warps a row): lane jj
                        // fetches candidate jj and its fixed-point weight; then S lanes a
                        // candidate sum the weight and number of the candidates strictly above
                        // it; the row's reductions go through its group barrier
                        const int r = warp / PW, jj = tid - r * PL;
                        if (warp < 2 * PW && r < nrows && sh.mode[r] == 1) {
                            const int nr = ncnt[r];
                            const uint32_t cpr = r == 0 ? cpl[0] : cpl[1], ccr = r == 0 ? ccl[0] : ccl[1];
                            // candidate jj's CTA: the last with candidates whose offset is <= jj
                            int c = 0;
                            for (int k = 1; k < static_cast<int>(C); ++k) {
                                const uint32_t pk = __shfl_sync(0xFFFFFFFFu, cpr, k);
                                const uint32_t ck = __shfl_sync(0xFFFFFFFFu, ccr, k);
                                if (static_cast<uint32_t>(jj) >= pk && ck > 0u) c = k;
                            }
                            const uint32_t pre_c = __shfl_sync(0xFFFFFFFFu, cpr, c);
                            float *cv = sh.b.s.sval + r * PL;
                            uint32_t *cw = reinterpret_cast<uint32_t *>(sh.b.s.skey) + r * PL;
                            if (jj < nr) {
                                const float vj = __uint_as_float(static_cast<uint32_t>(
                                    sh.a.cand[r][c * capc + jj - static_cast<int>(pre_c)] >> 32));
                                cv[jj] = vj;
                                cw[jj] = fix31(ex2(fmaf(vj, c2, sh.nmc[r])));
                            }
                            group_barrier<PL>(r);
                            int p2 = 1;
                            while (p2 < nr) p2 <<= 1;
                            const int S = min(32, PL / p2);
                            const int i = jj / S, sub = jj - i * S;
                            const bool real = i < nr;
                            const float v = real ? cv[i] : -INFINITY;
                            const uint32_t w = real ? cw[i] : 0u;
                            unsigned long long sgt = 0;
                            int cgt = 0;
                            if (real) {
#pragma unroll 4
                                for (int q = sub; q < nr; q += S) {
                                    if (cv[q] > v) {
                                        sgt += cw[q];
                                        ++cgt;
                                    }
                                }
                            }
                            for (int o = S >> 1; o > 0; o >>= 1) {
                                sgt += __shfl_xor_sync(0xFFFFFFFFu, sgt, o);
                                cgt += __shfl_xor_sync(0xFFFFFFFFu, cgt, o);
                            }
                            const bool lead = real && sub == 0;  // one lane per candidate contributes
                            const bool kept_k = lead && (!k_on || cgt < kk);
                            const unsigned long long MA = sh.pma[r];
                            unsigned long long tgt = 0;
                            if (k_on && p_on) {
                                // the top-p target within the top-k set
                                const unsigned long long ws = warp_sum_u64(kept_k ? static_cast<unsigned long long>(w) : 0ull);
                                if (lane == 0) sh.w.ct.w[warp] = ws;
                                group_barrier<PL>(r);
                                unsigned long long zk = MA;
                                for (int q = 0; q < PW; ++q) zk += sh.w.ct.w[r * PW + q];
                                tgt = fx_target_fx(pp, zk);
                                group_barrier<PL>(r);
                            } else if (p_on) {
                                tgt = sh.tgt[r];
                            }
                            const bool kept = kept_k && (!p_on || MA + sgt < tgt);
                            // the smallest kept value and the kept weight
                            float vmin = kept ? v : INFINITY;
                            unsigned long long wk = kept ? static_cast<unsigned long long>(w) : 0ull;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) {
                                vmin = fminf(vmin, __shfl_xor_sync(0xFFFFFFFFu, vmin, o));
                                wk += __shfl_xor_sync(0xFFFFFFFFu, wk, o);
                            }
                            if (lane == 0) {
                                sh.w.ct.v[warp] = vmin;
                                sh.w.ct.w[warp] = wk;
                            }
                            group_barrier<PL>(r);
                            if (jj == 0) {
                                float th = INFINITY;
                                unsigned long long zf = MA;
                                for (int q = 0; q < PW; ++q) {
                                    th = fminf(th, sh.w.ct.v[r * PW + q]);
                                    zf += sh.w.ct.w[r * PW + q];
                                }
                                sh.theta[r] = th;
                                sh.Z[r] = fx_to_float(zf);
                            }
                        }
                        __syncthreads();
                    } else {
                        // ---- exact thresholds.  Warp 0, per row: the candidates' count (-1 when some
                        // CTA overflowed its slots, or with too many or none: then the exact search)
                        // and each CTA's offset in the row's list in CTA order
                        if (warp == 0) {
        #pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const bool on = r < nrows && sh.mode[r] == 1;
                                const uint32_t cc = on && lane < static_cast<int>(C) ? sh.ccnt[lane][r] : 0u;
                                const bool over = __any_sync(0xFFFFFFFFu, cc > static_cast<uint32_t>(capc));
                                uint32_t incl = cc;
        #pragma unroll
                                for (int o = 1; o < 32; o <<= 1) {
                                    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                                    if (lane >= o) incl += y;
                                }
                                if (lane < static_cast<int>(C)) sh.cpre[r][lane] = incl - cc;
                                if (lane == 31)
                                    sh.ncr[r] = !on ? 0 : (over || incl > static_cast<uint32_t>(NT) || incl == 0) ? -1
                                                                                                            : static_cast<int>(incl);
                            }
                        }
                        __syncthreads();
                        const int ncr[2] = {sh.ncr[0], sh.ncr[1]};
                        const unsigned long long MAr[2] = {sh.mode[0] == 1 ? sh.pma[0] : 0ull,
                                                           nrows > 1 && sh.mode[1] == 1 ? sh.pma[1] : 0ull};
                        // candidate i of row r, counted over the CTAs' slots in CTA order
                        auto cand_at = [&](int r, int i) -> float {
                            int c = 0;
                            while (c + 1 < static_cast<int>(C) && i >= static_cast<int>(sh.cpre[r][c + 1])) ++c;
                            return __uint_as_float(static_cast<uint32_t>(sh.a.cand[r][c * capc + i - static_cast<int>(sh.cpre[r][c])] >> 32));
                        };
                        const bool small = ncr[0] <= NSMALL && (nrows < 2 || ncr[1] <= NSMALL);
                        if (small) {
                            // both rows' candidates into contiguous lists, with their fixed-point weights
                            for (int t = tid; t < 2 * CAPT; t += NT) {
                                const int r = t >= CAPT ? 1 : 0, slot = t - r * CAPT;
                                const int c = slot / capc, i = slot - c * capc;
                                if (ncr[r] > 0 && c < static_cast<int>(C) && i < static_cast<int>(sh.ccnt[c][r])) {
                                    const int pos = r * NSMALL + static_cast<int>(sh.cpre[r][c]) + i;
                                    const float v = __uint_as_float(static_cast<uint32_t>(sh.a.cand[r][slot] >> 32));
                                    sh.b.s.sval[pos] = v;
                                    reinterpret_cast<uint32_t *>(sh.b.s.skey)[pos] = fix31(ex2(fmaf(v, c2, sh.nmc[r])));
                                }
                            }
                            __syncthreads();
                            // ---- rank by counting, both rows at once (threads [0, NSMALL) take row
                            // 0, the rest row 1): for each candidate, the weight and number of the
                            // candidates strictly above it, each counted by S consecutive lanes over
                            // every S-th candidate; then block reductions
                            const int r = tid / NSMALL, tt = tid - r * NSMALL;
                            const int nr = r < nrows ? ncr[r] : -1;
                            int p2 = 1;
                            while (p2 < nr) p2 <<= 1;
                            const int S = min(32, NSMALL / p2);
                            const int i = tt / S, sub = tt - i * S;
                            const bool real = nr > 0 && i < nr;
                            const float *cv = sh.b.s.sval + r * NSMALL;
                            const uint32_t *cw = reinterpret_cast<const uint32_t *>(sh.b.s.skey) + r * NSMALL;
                            const float v = real ? cv[i] : -INFINITY;
                            const uint32_t w = real ? cw[i] : 0u;
                            unsigned long long sgt = 0;
                            int cgt = 0;
                            if (real) {
        #pragma unroll 4
                                for (int q = sub; q < nr; q += S) {
                                    const float vq = cv[q];
                                    if (vq > v) {
                                        sgt += cw[q];
                                        ++cgt;
                                    }
                                }
                            }
                            for (int o = S >> 1; o > 0; o >>= 1) {
                                sgt += __shfl_xor_sync(0xFFFFFFFFu, sgt, o);
                                cgt += __shfl_xor_sync(0xFFFFFFFFu, cgt, o);
                            }
                            const bool lead = real && sub == 0;  // one lane per candidate contributes
                            const bool kept_k = lead && (!k_on || cgt < kk);
                            const unsigned long long MA = MAr[r < 2 ? r : 0];
                            // reduction 1 (top-k with top-p): the weight of the top-k set
                            unsigned long long tgt = 0;
                            if (k_on && p_on) {
                                const unsigned long long ws = warp_sum_u64(kept_k ? static_cast<unsigned long long>(w) : 0ull);
                                if (lane == 0) sh.w.ct.w[warp] = ws;
                                __syncthreads();
                                unsigned long long zk = MA;
                                for (int wq = 0; wq < NW / 2; ++wq) zk += sh.w.ct.w[r * (NW / 2) + wq];
                                tgt = fx_target_fx(pp, zk);
                                __syncthreads();
                            } else if (p_on) {
                                tgt = fx_target(pp, sh.Z[r < nrows ? r : 0]);
                            }
                            const bool kept = kept_k && (!p_on || MA + sgt < tgt);
                            // reduction 2: the smallest kept value and the kept weight
                            float vmin = kept ? v : INFINITY;
                            unsigned long long wk = kept ? static_cast<unsigned long long>(w) : 0ull;
        #pragma unroll
                            for (int o = 16; o > 0; o >>= 1) {
                                vmin = fminf(vmin, __shfl_xor_sync(0xFFFFFFFFu, vmin, o));
                                wk += __shfl_xor_sync(0xFFFFFFFFu, wk, o);
                            }
                            if (lane == 0) {
                                sh.w.ct.v[warp] = vmin;
                                sh.w.ct.w[warp] = wk;
                            }
                            __syncthreads();
                            if (tt == 0 && nr > 0) {
                                float th = INFINITY;
                                unsigned long long zf = MA;
                                for (int wq = 0; wq < NW / 2; ++wq) {
                                    th = fminf(th, sh.w.ct.v[r * (NW / 2) + wq]);
                                    zf += sh.w.ct.w[r * (NW / 2) + wq];
                                }
                                sh.theta[r] = th;
                                sh.Z[r] = fx_to_float(zf);
                            }
        #pragma unroll
                            for (int rr = 0; rr < 2; ++rr)
                                if (rr < nrows && sh.mode[rr] == 1 && ncr[rr] < 0 && tid == 0) sh.mode[rr] = 2;
                            __syncthreads();
                        } else {
                            // ---- sort the candidates by value (descending) and scan, one row at a time
        #pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                if (r >= nrows || sh.mode[r] != 1) continue;
                                const int nc = ncr[r];
                                if (nc < 0) {
                                    __syncthreads();
                                    if (tid == 0) sh.mode[r] = 2;
                                    __syncthreads();
                                    continue;
                                }
                                const unsigned long long MA = MAr[r];
                                int P2 = 1;
                                while (P2 < nc) P2 <<= 1;
                                // bitonic sort of (value key, position), one key per thread; strides
                                // below 32 exchange through shuffles, wider ones through shared memory
                                unsigned long long key = 0ull;
                                if (tid < nc)
                                    key = (static_cast<unsigned long long>(order_key(cand_at(r, tid))) << 32) |
                                          static_cast<uint32_t>(tid);
                                for (int kb = 2; kb <= P2; kb <<= 1) {
                                    for (int jb = kb >> 1; jb > 0; jb >>= 1) {
                                        unsigned long long other;
                                        if (jb >= 32) {
                                            __syncthreads();
                                            sh.b.s.skey[tid] = key;
                                            __syncthreads();
                                            other = sh.b.s.skey[tid ^ jb];
                                        } else {
                                            other = __shfl_xor_sync(0xFFFFFFFFu, key, jb);
                                        }
                                        const bool lower = (tid & jb) == 0;
                                        const bool desc = (tid & kb) == 0;
                                        key = (lower == desc) ? max(key, other) : min(key, other);
                                    }
                                }
                                const bool real = tid < nc;
                                const float v = real ? key_to_float(static_cast<uint32_t>(key >> 32)) : -INFINITY;
                                const unsigned long long w =
                                    real ? static_cast<unsigned long long>(fix31(ex2(fmaf(v, c2, sh.nmc[r])))) : 0ull;
                                __syncthreads();
                                sh.b.s.sval[tid] = v;
                                // top-k: the k-th largest value (no element lies above the candidates)
                                if (k_on && tid == kk - 1) sh.fpick[r] = v;
                                __syncthreads();
                                const float thk = k_on ? sh.fpick[r] : -INFINITY;
                                const unsigned long long wk = (real && v >= thk) ? w : 0ull;
                                // weight strictly above each value: the exclusive prefix of the weights
                                // at the first position of its tie group (sorted descending)
                                const unsigned long long excl = block_excl_scan_u64(wk, sh.w.so.scan);
                                const int32_t headpos = (tid == 0 || sh.b.s.sval[tid - 1] != v) ? tid : -1;
                                const int32_t first = block_incl_max_i32(headpos, sh.w.so.scani);
                                sh.b.s.skey[tid] = excl;
                                const unsigned long long zk = MA + block_sum_u64(wk, sh.w.so.ru[r]);
                                if (tid == 0) {
                                    sh.tgt[r] = k_on ? fx_target_fx(pp, zk) : fx_target(pp, sh.Z[r]);
                                }
                                __syncthreads();
                                const unsigned long long above = MA + sh.b.s.skey[first];
                                const bool kept = real && v >= thk && (!p_on || above < sh.tgt[r]);
                                int32_t lastk = kept ? tid : -1;
        #pragma unroll
                                for (int o = 16; o > 0; o >>= 1)
                                    lastk = max(lastk, __shfl_xor_sync(0xFFFFFFFFu, lastk, o));
                                __syncthreads();
                                if (lane == 0) sh.w.so.scani[warp] = lastk;
                                __syncthreads();
                                int32_t lk = -1;
                                for (int wq = 0; wq < NW; ++wq) lk = max(lk, sh.w.so.scani[wq]);
                                const float th = sh.b.s.sval[lk < 0 ? 0 : lk];  // the smallest kept value
                                const unsigned long long zf =
                                    MA + block_sum_u64((real && v >= th) ? wk : 0ull, sh.w.so.ru[r]);
                                if (tid == 0) {
                                    sh.theta[r] = th;
                                    sh.Z[r] = fx_to_float(zf);
                                }
                                __syncthreads();
                            }
                        }
                    }
                }
                // ---- exact bisection over value keys (boundary outside the binned range, or
                // too many elements in its bins); both rows advance in lockstep
                const bool any_slow = sh.mode[0] == 2 || (nrows > 1 && sh.mode[1] == 2);
                if (any_slow) {
                    const int lim_n = n;
                    // F(t) per row: count (wt = 0) or fixed-point weight (wt = 1) of the elements
                    // with key >= max(t, floor); returns the cluster-wide sums
                    auto eval = [&](const uint32_t t[2], const uint32_t fl[2], int wt,
                                    unsigned long long out[2]) {
                        unsigned long long acc0 = 0, acc1 = 0;
#pragma unroll 1
                        for (int r = 0; r < nrows; ++r) {
                            if (sh.mode[r] != 2) continue;
                            const float nmc = sh.nmc[r];
                            const uint32_t lim = max(t[r], fl[r]);
                            float a = 0.0f;
                            uint32_t cnum = 0;
                            for_row(sdat(r), nvr, [&](float x, int li) {
                                if (li < lim_n && order_key(x) >= lim) {
                                    if (wt) a += ex2(fmaf(x, c2, nmc));
                                    else ++cnum;
                                }
                            });
                            const unsigned long long ac = wt ? fix_sum(a) : static_cast<unsigned long long>(cnum);
                            if (r == 0) acc0 = ac;
                            else acc1 = ac;
                        }
                        const unsigned long long s0 = block_sum_u64(acc0, sh.w.so.ru[0]);
                        const unsigned long long s1 = block_sum_u64(acc1, sh.w.so.ru[1]);
                        const int sp = static_cast<int>(sstep & 1u);
                        if (tid < static_cast<int>(C)) {
                            st_peer_u64(peer_addr(smem_addr(&sh.sx[sp][rank][0]), tid), s0);
                            st_peer_u64(peer_addr(smem_addr(&sh.sx[sp][rank][1]), tid), s1);
                            xarrive(&sh.xbar[XB_S + sp], tid);
                        }
                        xwait(XB_S + sp);
                        for (int r = 0; r < 2; ++r) {
                            unsigned long long sum = 0;
                            for (uint32_t c = 0; c < C; ++c) sum += sh.sx[sp][c][r];
                            out[r] = sum;
                        }
                        ++sstep;
                        __syncthreads();  // every thread has read this step's sums
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
                            need[r] = k_on ? fx_target_fx(pp, zk[r]) : fx_target(pp, sh.Z[r < nrows ? r : 0]);
                            if (need[r] == 0) need[r] = 1;
                        }
                        search(thk, 1, need, th);
                    }
                    unsigned long long zf[2];
                    eval(th, zero, 1, zf);
                    if (tid < nrows && sh.mode[tid] == 2) {
                        sh.theta[tid] = key_to_float(th[tid]);
                        sh.Z[tid] = fx_to_float(zf[tid]);
                    }
                    __syncthreads();
                }
            }
        }
        if (tid < nrows) sh.invZ[tid] = 1.0f / sh.Z[tid];
        __syncthreads();

        // ---- accept test
        const uint32_t uw1 = sh.uwd[1];  // the unit's Philox words, (b, j, 0, 0) under the seed
        const float u_acc = word_uniform(sh.uwd[0]), u_smp = word_uniform(uw1);

        // membership and probability of a token in the target (0) and draft (1) rows
        const float m0 = sh.m[0], m1 = sh.m[1], th0 = sh.theta[0], th1 = sh.theta[1];
        const float iz0 = sh.invZ[0], iz1 = sh.invZ[1], nm0 = sh.nmc[0], nm1 = sh.nmc[1];
        const bool deg0 = sh.deg[0], deg1 = sh.deg[1];
        auto prob0 = [&](float x, int64_t idx) -> float {
            if (deg0) return idx == 0 ? 1.0f : 0.0f;
            return x >= th0 ? ex2(fmaf(x, c2, nm0)) * iz0 : 0.0f;
        };
        auto prob1 = [&](float x, int64_t idx) -> float {
            if (deg1) return idx == 0 ? 1.0f : 0.0f;
            return x >= th1 ? ex2(fmaf(x, c2, nm1)) * iz1 : 0.0f;
        };

        bool accept = false;
        float pt = 0.0f, pd = 0.0f;
        if (early) {
            accept = true;  // (no output reads its probabilities)
        } else if (j < D && dvalid && one_hot) {
            // the draft is the point mass on d: q(d) = 1, held iff U_acc <= p(d)
            const float xt = sh.e1d[ep].x;
            const bool in_p = deg0 ? d == 0 : xt >= th0;
            pt = prob0(xt, d);
            pd = 1.0f;
            accept = in_p && u_acc <= pt;
        } else if (j < D && dvalid) {
            const float2 xdv = sh.e1d[ep];
            const float xt = xdv.x, xq = xdv.y;
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

        // a rejection is published for the row's later positions; a unit behind a position
        // every CTA's view agrees was rejected earlier draws nothing (no output reads it)
        if (P.dead && rank == 0 && tid == 0 && j < D && !accept) atomicMin(P.dead + b, static_cast<uint32_t>(j));
        uint32_t dkmin = 0xFFFFFFFFu;
        for (uint32_t c = 0; c < C; ++c) dkmin = min(dkmin, sh.e1k[ep][c]);
        // the slice buffer is free unless a draw reads it: bring in the next unit now
        const bool draw = ((j == D) || !accept) && !(dkmin < static_cast<uint32_t>(j));
        // A top-k row resolved from its candidates holds every kept element among them, in
        // every CTA (and so does the draft row when its residual needs q): such a draw reads
        // no slice
        const bool qpoint = one_hot || deg1;  // the draft is a point mass (q = 0 elsewhere)
        const bool local = kfast && sh.mode[0] == 1 && (j == D || qpoint || sh.mode[1] == 1);
        if ((!draw || local) && un >= 0) issue(nxt.b, nxt.j, true);

        // ---- draw (a rejected draft's residual, or the bonus).  Weights in fixed point,
        // summed as integers: the cumulative sums at every level (lane, warp, CTA, cluster)
        // are exact and agree with one another.  A distribution's weights add up to about
        // 2^31, so sums within a CTA fit 32 bits.  A degenerate target row is a point mass
        // on id 0, and so is every draw from it (its residual, when not zero, too).
        UnitResult *res = P.res + (static_cast<int64_t>(b) * (D + 1) + j);
        if (draw && deg0) {
            if (rank == 0 && tid == 0) res->token = 0;
        } else if (draw && local) {
            if (rank == 0) {
                // CTA 0 alone, from the gathered candidates: the kept target elements (value
                // >= theta0) in id order, the draft logit of each where the draft keeps that
                // id (else q = 0), then the weights the sweep below would form, summed in id
                // order as integers, so the token is the one the sweep would draw
                unsigned long long *kl = sh.b.s.skey;      // kept, as found: id << 32 | x bits
                unsigned long long *sl = &sh.a.cand[0][0];  // kept, in id order
                float *qx = sh.b.s.sval;                    // draft logit at sl[k], or -inf
                const int nslot = static_cast<int>(C) * capc;
                if (tid == 0) sh.lcnt[0] = 0;
                __syncthreads();
                for (int t = tid; t < nslot; t += NT) {
                    const int c = t / capc, i = t - c * capc;
                    if (i < static_cast<int>(min(sh.ccnt[c][0], static_cast<uint32_t>(capc)))) {
                        const unsigned long long cv = sh.a.cand[0][t];
                        const uint32_t xb = static_cast<uint32_t>(cv >> 32);
                        if (__uint_as_float(xb) >= th0)
                            kl[atomicAdd(&sh.lcnt[0], 1u)] = (static_cast<unsigned long long>(static_cast<uint32_t>(cv)) << 32) | xb;
                    }
                }
                __syncthreads();
                const int nk = static_cast<int>(sh.lcnt[0]);
                for (int k = tid; k < nk; k += NT) {  // rank by id (ids are distinct)
                    const unsigned long long me = kl[k];
                    int rk = 0;
                    for (int q = 0; q < nk; ++q) rk += (kl[q] >> 32) < (me >> 32) ? 1 : 0;
                    sl[rk] = me;
                    qx[rk] = -INFINITY;
                }
                __syncthreads();
                if (j < D && !qpoint) {
                    for (int t = tid; t < nslot; t += NT) {
                        const int c = t / capc, i = t - c * capc;
                        if (i < static_cast<int>(min(sh.ccnt[c][1], static_cast<uint32_t>(capc)))) {
                            const unsigned long long cv = sh.a.cand[1][t];
                            const float xq = __uint_as_float(static_cast<uint32_t>(cv >> 32));
                            const uint32_t id = static_cast<uint32_t>(cv);
                            if (xq >= th1) {
                                int l0 = 0, l1 = nk;  // the first kept id >= id
                                while (l0 < l1) {
                                    const int m = (l0 + l1) >> 1;
                                    if (static_cast<uint32_t>(sl[m] >> 32) < id) l0 = m + 1;
                                    else l1 = m;
                                }
                                if (l0 < nk && static_cast<uint32_t>(sl[l0] >> 32) == id) qx[l0] = xq;
                            }
                        }
                    }
                    __syncthreads();
                }
                const int pmid = one_hot ? d : 0;  // the point draft's id
                int wmode = (j == D) ? 1 : 0;      // 0: max(0, p - q), 1: p
                // (a kept set always carries weight; should rounding leave none, the lowest
                // kept id stands; the crossing element's id overwrites it below)
                if (tid == 0) res->token = nk > 0 ? static_cast<int>(sl[0] >> 32) : 0;
#pragma unroll 1
                for (int attempt = 0; attempt < 2; ++attempt) {
                    unsigned long long w = 0;
                    int myid = 0;
                    if (tid < nk) {
                        const unsigned long long e = sl[tid];
                        myid = static_cast<int>(e >> 32);
                        float pw = ex2(fmaf(__uint_as_float(static_cast<uint32_t>(e)), c2, nm0)) * iz0;
                        if (wmode == 0) {
                            if (qpoint) {
                                if (myid == pmid) pw = 0.0f;
                            } else if (qx[tid] > -INFINITY) {
                                pw = fmaxf(pw - ex2(fmaf(qx[tid], c2, nm1)) * iz1, 0.0f);
                            }
                        }
                        w = fix31(pw);
                    }
                    const unsigned long long before = block_excl_scan_u64(w, sh.w.so.scan);
                    const unsigned long long Rt = block_sum_u64(w, sh.w.so.ru[0]);
                    if (Rt > 0 || wmode == 1) {
                        // the smallest id whose cumulative weight exceeds u_smp * R (see below)
                        const unsigned long long tt =
                            (static_cast<unsigned long long>(2u * (uw1 >> 9) + 1u) * Rt) >> 24;
                        if (w > 0 && before <= tt && before + w > tt) res->token = myid;
                        break;
                    }
                    wmode = 1;  // the residual is identically zero: draw from p instead
                }
            }
        } else if (draw) {
            int wmode = (j == D) ? 1 : 0;  // 0: max(0, p - q), 1: p
            // a point-mass draft (a one-hot draft on d, or a degenerate draft row on id 0):
            // q = 0 elsewhere, and at its id the residual is p - 1 <= 0
            const float thq = qpoint ? INFINITY : th1;
            const int pm = one_hot ? d : 0;  // the point's id
            const bool pm_here = qpoint && pm >= lo && pm < lo + n;
            const int pv = pm_here ? (pm - lo) / EPV : -1, pe = pm_here ? (pm - lo) - pv * EPV : 0;
            auto weight = [&](float xt, float xq) -> uint32_t {
                if (!(xt >= th0)) return 0u;
                float p = ex2(fmaf(xt, c2, nm0)) * iz0;
                if (wmode == 0 && xq >= thq) p = fmaxf(p - ex2(fmaf(xq, c2, nm1)) * iz1, 0.0f);
                return fix31(p);
            };
            // the weight of vector v of the slice
            const uint4 *sv0 = reinterpret_cast<const uint4 *>(sdat(0));
            const uint4 *sv1 = reinterpret_cast<const uint4 *>(sdat(1));
            auto vec_weight = [&](int v) -> uint32_t {
                const uint4 rx = sv0[v];
                if (!(vec_max<T>(rx) >= th0)) return 0u;  // no target logit of the vector is kept
                float x[EPV], y[EPV];
                unpack(rx, x);
                unpack(sv1[v], y);
                uint32_t s = 0;
#pragma unroll
                for (int e = 0; e < EPV; ++e)
                    s += weight(x[e], y[e]);
                // the draft point's id carries no residual weight
                if (wmode == 0 && v == pv) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e == pe) s -= weight(x[e], y[e]);
                }
                return s;
            };
            const int nvw = (nvr + NW - 1) / NW;  // vectors per warp
            const int w0 = warp * nvw, w1 = min(nvr, w0 + nvw);
            // the vectors' weights, in the candidate and histogram storage (free by now), or
            // past the staged rows for larger slices
            const int svecs = static_cast<int>((P.slice * static_cast<int64_t>(sizeof(T)) + 15) / 16);
            uint32_t *wvec = svecs <= WVEC_SHARED
                                 ? reinterpret_cast<uint32_t *>(&sh.a)
                                 : reinterpret_cast<uint32_t *>(smem_raw + data_off + (one_hot ? 1 : 2) * row_bytes);
            static_assert(offsetof(Shared, b) == offsetof(Shared, a) + sizeof(Shared::a) &&
                              sizeof(Shared::a) + sizeof(Shared::b) >= 4 * WVEC_SHARED,
                          "the draw keeps up to WVEC_SHARED vector weights in the storage of a and b");
#pragma unroll 1
            for (int attempt = 0; attempt < 2; ++attempt) {
                // each vector's weight is kept for the walk below
                uint32_t acc = 0;
                for (int v = w0 + lane; v < w1; v += 32) {
                    const uint32_t wvv = vec_weight(v);
                    wvec[v] = wvv;
                    acc += wvv;
                }
                acc = __reduce_add_sync(0xFFFFFFFFu, acc);
                if (lane == 0) sh.w.wsum[warp] = acc;
                __syncthreads();
                if (tid < static_cast<int>(C)) {
                    unsigned long long cs = 0;
                    for (int wq = 0; wq < NW; ++wq) cs += sh.w.wsum[wq];
                    st_peer_u64(peer_addr(smem_addr(&sh.dr[attempt][rank]), tid), cs);
                    xarrive(&sh.xbar[XB_E4 + attempt], tid);
                }
                xwait(XB_E4 + attempt);
                const unsigned long long *dR = sh.dr[attempt];
                unsigned long long Rt = 0;
                for (uint32_t c = 0; c < C; ++c) Rt += dR[c];
                if (Rt > 0 || wmode == 1) {
                    // smallest id whose cumulative weight exceeds u_smp * R; a cumulative
                    // integer sum S exceeds u_smp * R exactly when S > floor(u_smp * R), and
                    // u_smp = k * 2^-24 with k odd, so floor(u_smp * R) = (k * R) >> 24 exactly
                    const unsigned long long tt =
                        (static_cast<unsigned long long>(2u * (uw1 >> 9) + 1u) * Rt) >> 24;
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
                        // the warp holding it (the last one when rounding left none crossing)
                        // and the weight before its run: every warp scans the warps' sums,
                        // lane w holding warp w's
                        const unsigned long long dw = lane < NW ? sh.w.wsum[lane] : 0ull;
                        unsigned long long iw = dw;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, iw, o);
                            if (lane >= o) iw += y;
                        }
                        iw += before;
                        const unsigned wm = __ballot_sync(0xFFFFFFFFu, lane < NW && iw > tt);
                        const int ws = wm ? __ffs(wm) - 1 : NW - 1;
                        const unsigned long long wb = __shfl_sync(0xFFFFFFFFu, iw - dw, ws);
                        if (warp == ws) {
                            // the vector that crosses the target: each lane sums a stretch of
                            // the warp's run (in id order) from the kept vector weights, a
                            // scan finds the stretch, and its lane walks it; rem = tt - (weight
                            // before this warp's run)
                            uint32_t rem = tt >= wb ? static_cast<uint32_t>(tt - wb) : 0u;
                            const int kq = (w1 - w0 + 31) / 32;
                            const int a0 = min(w1, w0 + lane * kq), a1 = min(w1, a0 + kq);
                            uint32_t sl = 0;
                            for (int v = a0; v < a1; ++v) sl += wvec[v];
                            uint32_t incl = sl;
#pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const uint32_t yv = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                                if (lane >= o) incl += yv;
                            }
                            const unsigned hitm = __ballot_sync(0xFFFFFFFFu, incl > rem);
                            const unsigned posm = __ballot_sync(0xFFFFFFFFu, sl > 0);
                            // the vector and the weight before it within the vector's stretch
                            int fv = -1;
                            uint32_t hit_rem = 0;
                            const bool hit = hitm != 0;
                            const int hl = hit ? __ffs(hitm) - 1 : (posm ? 31 - __clz(posm) : -1);
                            if (hl >= 0 && lane == hl) {
                                uint32_t cum = incl - sl;
                                for (int v = a0; v < a1; ++v) {
                                    const uint32_t wvv = wvec[v];
                                    if (hit && cum + wvv > rem) {
                                        fv = v;
                                        hit_rem = rem - cum;
                                        break;
                                    }
                                    if (wvv > 0) fv = v;  // the last positive vector
                                    cum += wvv;
                                }
                            }
                            if (hl >= 0) {
                                fv = __shfl_sync(0xFFFFFFFFu, fv, hl);
                                hit_rem = __shfl_sync(0xFFFFFFFFu, hit_rem, hl);
                            }
                            // its elements, one per lane: the first whose cumulative weight
                            // exceeds hit_rem (the last positive one when nothing crossed)
                            if (fv >= 0) {
                                uint32_t we = 0;
                                if (lane < EPV) {
                                    float x[EPV], y[EPV];
                                    unpack(sv0[fv], x);
                                    unpack(sv1[fv], y);
#pragma unroll
                                    for (int e = 0; e < EPV; ++e)
                                        if (e == lane) we = weight(x[e], y[e]);
                                    // the draft point's id carries no residual weight
                                    if (wmode == 0 && fv == pv && lane == pe) we = 0u;
                                }
                                uint32_t ce = we;
#pragma unroll
                                for (int o = 1; o < EPV; o <<= 1) {
                                    const uint32_t yv = __shfl_up_sync(0xFFFFFFFFu, ce, o);
                                    if (lane >= o) ce += yv;
                                }
                                const unsigned em = __ballot_sync(0xFFFFFFFFu, lane < EPV && we > 0 && ce > hit_rem);
                                const unsigned pm = __ballot_sync(0xFFFFFFFFu, lane < EPV && we > 0);
                                const int fe = (hit && em) ? __ffs(em) - 1 : (pm ? 31 - __clz(pm) : 0);
                                if (lane == 0) res->token = lo + fv * EPV + fe;
                            } else if (lane == 0) {
                                res->token = lo;
                            }
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
        __syncthreads();  // every thread is done with this unit's shared state
        if (draw && !local && un >= 0) issue(nxt.b, nxt.j, true);
        u = un;
        cnx = nxt;
        un = sh.e1su[ep];  // CTA 0's choice, sent with this unit's E1 (rewritten two E1s later)
        if (un >= 0) {
            const NextParams q = sh.e1sp[ep];
            const int nb = unit_row(un);
            nxt = UnitParams{nb, pmajor ? un / Bi : un - nb * (D + 1), q.tau, q.pp, q.kk, q.d};
        }
    }
    if (!started) cluster_wait_acquire();  // a cluster with no unit still completes its start
    // no CTA leaves while a peer may still write into its shared memory or arrive on its
    // barriers
    cluster_arrive_release();
    cluster_wait_acquire();
    if (tid == 0 && (sh.flags & 3) && P.status) atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
}

// Diagnostic of the bounded waits: an mbarrier of two arrivals gets one, so its phase never
// completes; both of the kernel's wait forms must give up after `limit` polls, and then
// MTPSPEC_STATUS_TIMEOUT is OR-ed into the status word, as the kernel does.
__global__ void k_wait_selftest(uint32_t limit, int32_t *status) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_arrive(&bar);
    const bool a = mbar_wait_bounded(&bar, 0, limit);
    const bool x = xbar_wait_bounded(&bar, 0, limit);
    if (!a && !x) atomicOr(status, MTPSPEC_STATUS_TIMEOUT);
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

struct VerifyGeometry {
    int C;          // CTAs per cluster
    int64_t slice;  // logits per CTA
};

static int64_t verify_slice(int64_t V, int C) {
    const int64_t s = (V + C - 1) / C;
    return (s + 15) & ~static_cast<int64_t>(15);
}

constexpr size_t kSmemLimit = 227u * 1024u;

// Shared memory of a CTA for slices of `slice` logits of `rows` rows (2: target and draft;
// 1: the target alone, for a one-hot draft), plus, past vs::WVEC_SHARED 16-byte vectors,
// a region for the draw's vector weights (they fit the shared state below that).
static size_t verify_smem_bytes(int64_t slice, size_t es, int rows) {
    const size_t vecs = (static_cast<size_t>(slice) * es + 15) / 16;
    const size_t head = (sizeof(vs::Shared) + 127) & ~static_cast<size_t>(127);
    const size_t row = ((static_cast<size_t>(slice) * es) + 127) & ~static_cast<size_t>(127);
    const size_t extra = vecs > static_cast<size_t>(vs::WVEC_SHARED) ? ((vecs * 4 + 127) & ~static_cast<size_t>(127)) : 0;
    return head + static_cast<size_t>(rows) * row + extra;
}

// Smallest cluster size whose CTAs fit their slices of the staged rows in shared memory (0:
// none up to MAXC).
static int verify_cmin(int64_t V, size_t es, int rows) {
    for (int C = 2; C <= vs::MAXC; ++C)
        if (verify_smem_bytes(verify_slice(V, C), es, rows) <= kSmemLimit) return C;
    return 0;
}

// Per-unit records, then each row's first rejected position (for skipping draws).
static size_t verify_records_bytes(int64_t B, int32_t D) {
    return static_cast<size_t>(B) * static_cast<size_t>(D + 1) * sizeof(vs::UnitResult);
}
// The chunked verifier is asked for by MTPSPEC_VERIFY_IMPL=chunks (where its limits allow).
static bool chunks_requested() {
    const char *s = getenv("MTPSPEC_VERIFY_IMPL");
    return s && strcmp(s, "chunks") == 0;
}

size_t verify_workspace_bytes(int64_t B, int32_t D, int64_t V) {
    const size_t cl = verify_records_bytes(B, D) + ((static_cast<size_t>(B) * 4 + 15) & ~static_cast<size_t>(15));
    // V that every logit type and mode stages in a cluster: the cluster kernel's records
    if (!chunks_requested() && verify_cmin(V, 4, 2) > 0) return cl;
    const size_t ch = verify_chunks_workspace_bytes(B, D, V);
    return cl > ch ? cl : ch;
}

bool verify_sample_fits(int64_t V, size_t elem_bytes, bool one_hot) {
    return verify_cmin(V, elem_bytes, one_hot ? 1 : 2) > 0 || verify_chunks_fits(V, elem_bytes);
}

bool verify_fits(int64_t V, size_t elem_bytes, bool one_hot) {
    return verify_cmin(V, elem_bytes, one_hot ? 1 : 2) > 0;
}

// Resident clusters of the persistent kernel for one configuration (cached).
template <typename T>
static int resident_clusters(int C, size_t smem) {
    constexpr int NC = 64;
    static std::mutex mu;
    static int cache_c[NC] = {0}, cache_v[NC] = {0}, dev_of[NC] = {0};
    static size_t cache_s[NC] = {0};
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
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
    if (cudaOccupancyMaxActiveClusters(&n, vs::k_verify_rr<T, true, false>, &cfg) != cudaSuccess || n < 1)
        n = 1;
    const int i = used < NC ? used++ : NC - 1;
    dev_of[i] = dev;
    cache_c[i] = C;
    cache_s[i] = smem;
    cache_v[i] = n;
    return n;
}

// Fixed cost of a unit, in logits of a CTA's slice: the exchanges and the work that does not
// scale with the slice take about as long as the passes over a slice of this length (fitted
// to timings of the 256-row serving verify over a 151,936-id vocabulary, fp32 and bf16).
constexpr int64_t kUnitFixedLogits = 5000;

// The cluster size of a launch.  Clusters are placed within GPCs, so the resident clusters
// (and the SMs they use) depend on the size; among the sizes whose slices fit, take the one
// that finishes the most units per unit time by a simple model: min(resident clusters,
// units) units in flight, each taking time in proportion to kUnitFixedLogits + slice.
// MTPSPEC_VERIFY_CLUSTER forces a size (any that fits, 2 to MAXC).
template <typename T>
static VerifyGeometry verify_geometry(int64_t V, int64_t units, int rows) {
    VerifyGeometry gm = {0, 0};
    const int Cmin = verify_cmin(V, sizeof(T), rows);
    if (Cmin == 0) return gm;
    int best = 0;
    double best_score = -1.0;
    for (int C = Cmin; C <= vs::MAXC; ++C) {
        const int64_t sl = verify_slice(V, C);
        const size_t smem = verify_smem_bytes(sl, sizeof(T), rows);
        if (smem > kSmemLimit) continue;
        const int64_t a = std::min<int64_t>(resident_clusters<T>(C, smem), units);
        const double score = static_cast<double>(a) / static_cast<double>(kUnitFixedLogits + sl);
        if (score > best_score) {
            best_score = score;
            best = C;
        }
    }
    if (const char *e = getenv("MTPSPEC_VERIFY_CLUSTER")) {
        const int c = atoi(e);
        if (c >= Cmin && c <= vs::MAXC) best = c;
    }
    gm.C = best;
    gm.slice = verify_slice(V, best);
    return gm;
}

// The kernel may take the largest shared memory and clusters up to MAXC (the occupancy
// queries of the geometry need both, on the instance with the top-k paths).
template <typename T, bool KT, bool EA>
static cudaError_t prepare_verify_rr() {
    static AttrCache a_smem, a_carve, a_cluster;
    cudaError_t e = ensure_attr(vs::k_verify_rr<T, KT, EA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemLimit), a_smem);
    if (e != cudaSuccess) return e;
    e = ensure_attr(vs::k_verify_rr<T, KT, EA>, cudaFuncAttributePreferredSharedMemoryCarveout,
                    static_cast<int>(cudaSharedmemCarveoutMaxShared), a_carve);
    if (e != cudaSuccess) return e;
    return ensure_attr(vs::k_verify_rr<T, KT, EA>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1, a_cluster);
}

template <typename T>
static cudaError_t launch_verify_rr(vs::Params p, cudaStream_t stream) {
    const int64_t units = p.B * (p.D + 1);
    // the instance: with the top-k paths when the call passes top-k values; else with the
    // E1 acceptance path for a decode loop's call with draft logits (top-p values, no
    // probabilities; a one-hot draft's units are short enough that the path costs more
    // than it saves: 267 -> 283 us on the serving workload), else without either
    const bool ea = !p.topk && p.topp && !p.need_p && p.Q;
    cudaError_t e = prepare_verify_rr<T, true, false>();
    if (e == cudaSuccess && !p.topk) e = ea ? prepare_verify_rr<T, false, true>() : prepare_verify_rr<T, false, false>();
    if (e != cudaSuccess) return e;
    const int rows = p.Q ? 2 : 1;
    const VerifyGeometry gm = verify_geometry<T>(p.V, units, rows);
    if (gm.C == 0) return cudaErrorInvalidValue;
    const int C = gm.C;
    p.slice = gm.slice;
    const size_t smem = verify_smem_bytes(p.slice, sizeof(T), rows);
    int64_t G = resident_clusters<T>(C, smem);
    if (G > units) G = units;
    p.G = static_cast<int32_t>(G);
    // Position-major order lets a cluster skip the units behind a rejection it knows of.  It
    // pays once each cluster runs many units; with a one-hot draft, whose units are short
    // beside their draws; and with more than one round of units and two drafts or more a
    // row (the later positions and the bonus units fall in the later rounds: 32 units of
    // three drafts, 74.8 -> 64.6 us).  With one draft a row and a few rounds it costs a few
    // per cent (128 units: 93.2 -> 94.8 us).
    p.pmajor = (!p.Q || units >= 8 * G || (units > G && p.D >= 2)) ? 1 : 0;
    if (const char *o = getenv("MTPSPEC_VERIFY_ORDER"))  // "row" or "position" forces the order
        p.pmajor = o[0] == 'p' ? 1 : (o[0] == 'r' ? 0 : p.pmajor);
    if (!p.pmajor) {
        p.dead = nullptr;
    } else if (p.dead) {
        e = cudaMemsetAsync(p.dead, 0xFF, static_cast<size_t>(p.B) * 4, stream);
        if (e != cudaSuccess) return e;
    }
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
    e = p.topk ? cudaLaunchKernelEx(&cfg, vs::k_verify_rr<T, true, false>, p)
        : ea   ? cudaLaunchKernelEx(&cfg, vs::k_verify_rr<T, false, true>, p)
               : cudaLaunchKernelEx(&cfg, vs::k_verify_rr<T, false, false>, p);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

static cudaError_t run_verify_sample_impl(const VerifySampleArgs &a, bool row_flags,
                                          cudaStream_t stream) {
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
    p.slice = 0;
    p.G = 1;
    p.res = static_cast<vs::UnitResult *>(a.workspace);
    p.status = a.status;
    p.pmajor = 0;
    p.need_p = (a.p_target || a.p_draft) ? 1 : 0;
    p.dead = row_flags ? reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(a.workspace) +
                                                      verify_records_bytes(a.B, a.D))
                       : nullptr;  // reset (and used) by the launch when the order is position-major
    // the sampled rows, then (beside them) the greedy rows, then the per-row finalize
    cudaError_t e = a.dtype == MTPSPEC_F32 ? launch_verify_rr<float>(p, stream)
                                           : launch_verify_rr<uint16_t>(p, stream);
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

cudaError_t run_wait_selftest_clusters(uint32_t limit, int32_t *status, cudaStream_t stream) {
    vs::k_wait_selftest<<<1, 32, 0, stream>>>(limit, status);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_verify_finalize(const VerifyUnitRecord *rec, const VerifySampleArgs &a,
                                   cudaStream_t stream) {
    vs::k_verify_finalize<<<static_cast<unsigned>((a.B + 127) / 128), 128, 0, stream>>>(
        rec, a.draft_ids, a.B, a.D, a.out_tokens, a.num_accepted, a.p_target, a.p_draft);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

// The cluster kernel wherever a cluster stages the unit's rows; beyond that (or when asked
// for) the chunked verifier, whose shared memory does not grow with V.
cudaError_t run_verify_sample(const VerifySampleArgs &a, cudaStream_t stream) {
    const size_t es = a.dtype == MTPSPEC_F32 ? 4 : 2;
    const bool one_hot = a.draft == nullptr;
    if ((chunks_requested() || !verify_fits(a.V, es, one_hot)) && verify_chunks_fits(a.V, es))
        return run_verify_chunks(a, stream);
    return run_verify_sample_impl(a, true, stream);
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
    // The array's address is looked up for the device the work runs on: the stream's
    // device (made current by the entry point before this call), or, for the legacy
    // default stream, the current device.  A stream being captured cannot be asked for its
    // device without invalidating the capture, so then the current device is taken to be
    // the stream's (the header states this rule), and its address must already be known.
    int dev = -1;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaSuccess;
    if (stream != nullptr) {
        e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return e;
    }
    if (stream != nullptr && cs == cudaStreamCaptureStatusNone) {
        e = cudaStreamGetDevice(stream, &dev);
        if (e != cudaSuccess) return e;
        int cur = -1;
        e = cudaGetDevice(&cur);
        if (e != cudaSuccess) return e;
        if (cur != dev) return cudaErrorInvalidDevice;  // the set-up needs the device current
    } else {
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
    }
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void *ptr = nullptr;
    {
        // once per device, with that device current: the device address of the array
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            if (cs != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
            e = cudaGetSymbolAddress(&ptr, g_verify_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_ptr[dev] = ptr;
        }
        ptr = g_scratch_ptr[dev];
    }
    a.workspace = ptr;
    return run_verify_sample_impl(a, false, stream);  // no row flags: every rejection draws
}

}  // namespace mtpspec
