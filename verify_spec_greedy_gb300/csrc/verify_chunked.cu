// Speculative-sampling verification over vocabulary chunks: temperature -> top-k -> top-p
// filtering of target and draft logits, the accept test U <= p/q, the residual draw at the
// first rejection and the bonus draw ("MPT (MTP, Multi-Token Prediction) 原理详解", section
// 三 stage 3 "rejection sampling" and stage 4; "The decoding loop and MTP", "Why a
// hand-written decoding loop" for the filters and "MTP speculative decoding" items 2-3 for
// the drawn replacement and the extra token).
//
// A unit is one (row b, position j): the target row T[b, j] and, for j < D, the draft row
// Q[b, j].  Each unit is cut into NC chunks of CH vocabulary ids; a work item is one chunk.
// A persistent grid of CTAs (several per SM, as many as are resident) claims items in
// order from a global counter; a CTA holds one item at a time, so a unit's chunks are held
// by running CTAs and the waits below end as long as the GPU runs at least as many of them
// as a unit has chunks (the earliest unfinished unit can always progress); otherwise the
// waits give up and the call reports MTPSPEC_STATUS_TIMEOUT.
//
// One item:
//   stage    bulk asynchronous copies bring the chunk's target and draft logits into shared
//            memory (the item one grid-width ahead is prefetched into L2 when it is claimed)
//   pass 1   per row: the chunk maximum, the sum of w = 2^((x - x_ref) c2 - o_c) (c2 =
//            log2(e) / tau, x_ref the largest of the row's first 32 logits, o_c the chunk's
//            top octave), and for top-k the k-th largest per-thread maximum, a lower bound
//            of the k-th largest logit of the row
//   W1       wait for the unit's other chunks (a counter in global memory); every CTA then
//            has the row maximum and total weight Z, and the loose cut: no logit below it
//            can be kept (top-p: w <= (1 - p) Z / V; top-k: below the largest bound)
//   pass 2   only the logits above the loose cut: a histogram of 16 bins per octave, from
//            w's bits (exponent = octave, top mantissa bits = bin), bins aligned in absolute
//            octaves across chunks; masses are w's 24-bit mantissa >> 9 per element, so the
//            plan knows each bin's mass within rigorous bounds (counts are exact for top-k)
//   W1b      wait; every CTA reads the merged histogram and plans the boundary bins: the
//            top-k bin, and the top-p window that must hold the crossing of p Z
//   gather   elements of the boundary bins go to the unit's candidate list; the exact weight
//            above them is summed; the target row's possibly-kept elements go, in id order,
//            to the unit's nucleus list (only when the unit may have to draw)
//   W2       every chunk arrives and leaves, except the last, which resolves the unit: exact
//            thresholds from the sorted candidates, kept masses, p(d), q(d), the accept
//            test, the unit record, and the draw (a rejection, or the bonus position, unless
//            an earlier position of the row is known rejected): the inverse CDF of the
//            residual max(0, p - q) in id order over the nucleus list.
// Unfiltered rows skip the histogram: each chunk sums its residual in fixed point after W1,
// and the resolving CTA re-reads only the chunk that holds the draw.  Rows whose boundary
// lies below the binned octaves, lists over capacity, chunk maxima too far apart for the
// ring of octaves, or values too large for the octave arithmetic go to an exact slow path
// run by the resolving CTA alone (radix selection over the row in global memory).  Greedy
// rows (temperature 0) take the argmax of each chunk; the last chunk to arrive merges them.
// Every decision is taken from integer or fixed-order sums over published values, so it is
// the same in every run.  All waits are bounded: a wait that gives up raises
// MTPSPEC_STATUS_TIMEOUT and an abort flag that ends the call's remaining work.
#include <math.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace mtpspec {
namespace vc {

constexpr int NT = 256;                 // threads per CTA
constexpr int NW = NT / 32;
constexpr int CPS = 3;                  // CTAs resident per SM
constexpr int RB = 16;                  // histogram bins per octave (four mantissa bits)
constexpr int ZL = 20;                  // binned octaves below a chunk's top octave: 0..ZL
constexpr int NBL = (ZL + 1) * RB;      // local bins
constexpr int NO = 48;                  // ring octaves per row
constexpr int NBR = NO * RB;            // ring bins per row
constexpr int QSH = 9;                  // histogram masses keep the 24-bit mantissa >> QSH
constexpr int CAP = 2048;               // boundary candidates per row
constexpr int NSLOT = 128;              // unit state slots at most (unit u uses slot u % nslot)
constexpr int NCMAX = 256;              // chunks per unit
constexpr int ROW_BYTES = 32768;        // staged bytes per row
constexpr int ROWB = ROW_BYTES + 128;   // a staged row's buffer (room for the alignment pad)
constexpr uint32_t POLL_LIMIT = 1u << 22;
constexpr float PMAX = 8192.0f;         // |(max - x_ref) * c2| below which octaves are exact
constexpr float FXF = 1099511627776.0f; // 2^40: fixed point of the draw weights
constexpr double FXD = 1099511627776.0;
// Masses of the plan and the resolution: 64-bit fixed point, 2^39 per unit of weight relative
// to the row's top octave (the largest weight is below 2, so every term fits 2^40).
constexpr int FSH = 39;
constexpr float FSF = 549755813888.0f;  // 2^39

static_assert(NBL <= 2 * NT, "two rounds of threads cover the local bins");
static_assert(NBL <= 11 * 32, "a warp holds a row's bins in registers, 11 per lane");
static_assert(CAP * 8 <= ROW_BYTES, "the resolver sorts its candidates in a staging buffer");

enum : int { KIND_GREEDY = 0, KIND_SAMPLE = 1, KIND_BONUS = 2 };

struct __align__(16) ChunkStat {
    float m;        // chunk maximum (greedy: the argmax value)
    int32_t otop;   // chunk top octave (greedy: the argmax id); INT32_MIN: no finite logit
    float zsum;     // sum of 2^t over the chunk, t relative to the top octave
    float kb;       // top-k: the k-th largest per-thread maximum (-inf: none); NaN: the
                    // octave arithmetic is out of range
};
// What a chunk publishes when it arrives at W2.
struct __align__(16) ChunkPub {
    unsigned long long above[2]; // weight (fixed point) above the boundary bins
    unsigned long long mid[2];   // ... between the top-p window and the top-k bin
    unsigned long long r, p;     // unfiltered units: residual and p sums (fixed point 2^40)
    uint32_t nucw[NW];           // nucleus entries of each warp's range (0xFFFFFFFF: overflow)
};
struct NucEntry {
    int32_t id;
    float xt, xq;
};

// Per-slot state cleared at the start of each call and again when a unit releases the slot.
struct SlotZ {
    uint32_t gen;        // unit u may use slot u % NSLOT once gen >= u / NSLOT
    uint32_t c1;         // arrivals after pass 1
    uint32_t c1b;        // arrivals after pass 2
    uint32_t c2;         // arrivals after the gather
    uint32_t done;       // chunks finished with the unit
    uint32_t pad0[3];
    uint32_t ncand[2];   // candidates per row
    float xd[2];         // the draft token's target and draft logits
    uint32_t pad1[4];
    unsigned long long ring_mass[2][NBR];
    unsigned long long coarse_mass[2][NO];
    uint32_t ring_cnt[2][NBR];
    uint32_t coarse_cnt[2][NO];
};
// Per-slot state written before it is read (not cleared).
struct SlotN {
    ChunkStat stat[2][NCMAX];
    ChunkPub pub[NCMAX];
    unsigned long long cand[2][CAP];
};
constexpr size_t ZSZ = (sizeof(SlotZ) + 255) & ~static_cast<size_t>(255);
constexpr size_t NSZ = (sizeof(SlotN) + 255) & ~static_cast<size_t>(255);

struct Params {
    const void *T, *Q;
    const int32_t *d;
    const float *tau;
    const int32_t *topk;
    const float *topp;
    uint64_t seed;
    int64_t B, V, CH, items;
    int32_t D, NC, seg;       // seg: nucleus entries per chunk
    int32_t nslot;            // slots of this call
    NucEntry *nuc;            // [nslot][nuc_slot] nucleus lists
    int64_t nuc_slot;         // nucleus entries per slot
    uint32_t *hdr;            // [0] next item, [1] abort, [2..7] counters
    uint32_t *rowflag;        // [B]: D + 1 - (first rejected position), 0 = none seen
    unsigned char *zone_z;    // nslot * ZSZ
    unsigned char *zone_n;    // nslot * NSZ
    VerifyUnitRecord *rec;    // [B, D + 1]
    int32_t *status;
};

// Plan of one row, computed identically by every CTA of the unit.
struct RowPlan {
    float M;             // row maximum
    float xref;
    float xcut;          // loose cut: pass 2 bins logits >= xcut
    int32_t otop;        // row top octave
    int32_t pm;          // point mass on id 0 (no finite logit)
    int32_t fallback;    // the unit needs the exact path
    unsigned long long Z; // total weight (fixed point)
    // boundary bins in row depth (octave below the top * RB + bin); -1: none
    int32_t dk;          // top-k bin
    int32_t dlo, dhi;    // top-p window
    int32_t dmax;        // deepest needed bin
    int32_t dabove;      // elements above this bin are summed exactly
    uint32_t cnt_above_k;
};

struct Misc {
    unsigned long long bar[2];
    uint32_t item;
    int32_t resolver;
    int32_t leave;
    int32_t cstar;
    float fred[NW];
    unsigned long long ured[NW][2];
    unsigned long long dred[NW][2];
    ArgMax ared[NW];
    float xref[2];
    float kb[2];
    int32_t otop[2];
    float xlo[2];
    RowPlan plan[2];
    uint32_t tk_theta;
    int32_t tk_ok;
    int32_t usep;
    uint32_t ncc;        // candidates staged in shared memory
    uint32_t cbase;      // their first slot in the unit's list
    unsigned long long pb_w[2][4][3];   // plan B: per-warp sums (lo, hi, count) of each row
    int32_t pb_dk[2], pb_dlo[2], pb_dhi[2];
    unsigned long long pb_zlo[2], pb_zhi[2];
    uint32_t pb_cab[2];
    unsigned long long tk_z;
    unsigned long long target;
};
constexpr int CCAP = 384;               // a chunk's candidates, staged in shared memory
constexpr int SCR_BYTES = NBL * 8 + NT * 4 + CCAP * 8;   // histogram, thread maxima, candidates
static_assert(NCMAX * NW * 16 <= ROW_BYTES, "the resolver's per-range draw sums fit a staging buffer");

// ---------------------------------------------------------------- small device helpers

__device__ __forceinline__ float ex2f(float z) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
    return r;
}
__device__ __forceinline__ uint32_t ld_acq(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_rel(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_ar(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}
__device__ __forceinline__ void red_add_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_add_u32(uint32_t *p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
template <typename X>
__device__ __forceinline__ X ldcg(const X *p) {
    return __ldcg(p);
}
// a chunk's statistics through L2
__device__ __forceinline__ ChunkStat ldcg(const ChunkStat *p) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(p));
    return ChunkStat{__uint_as_float(v.x), static_cast<int32_t>(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
}

// Thread 0 waits until *p >= target.  False (after raising the abort flag and the timeout
// status) if the wait gave up, or if the call was aborted elsewhere.
__device__ bool wait_geq(uint32_t *p, uint32_t target, const Params &P, uint32_t limit = POLL_LIMIT) {
    // spin first: a poll is an L2 round trip already, and a sleeping warp can wake up late
    for (uint32_t it = 0; it < limit; ++it) {
        if (ld_acq(p) >= target) return true;
        if ((it & 255u) == 255u) {
            if (ld_acq(P.hdr + 1) != 0u) return false;
            if (it > 65536u) __nanosleep(256);
        }
    }
    atomicExch(P.hdr + 1, 1u);
    if (P.status) atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
    return false;
}

// Diagnostic of the bounded wait: a counter that nothing raises (zeroed here, with the abort
// flag) must make wait_geq give up after `limit` polls, raise the abort flag and OR
// MTPSPEC_STATUS_TIMEOUT into the status word, as the kernel does.
__device__ uint32_t g_wait_selftest[4];
__global__ void k_wait_selftest(uint32_t limit, int32_t *status) {
    if (threadIdx.x != 0) return;
    g_wait_selftest[0] = 0u;  // the counter
    g_wait_selftest[1] = 0u;  // hdr[1]: the abort flag
    __threadfence();
    Params P = {};
    P.hdr = g_wait_selftest;
    P.status = status;
    const bool ok = wait_geq(&g_wait_selftest[0], 1u, P, limit);
    // a wait that did not give up, or gave up without the abort flag, leaves no timeout bit
    if (ok || ld_acq(&g_wait_selftest[1]) != 1u) atomicAnd(status, ~MTPSPEC_STATUS_TIMEOUT);
}

__device__ __forceinline__ void mbar_init1(unsigned long long *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity) {
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <typename T> __device__ __forceinline__ T ninf();
template <> __device__ __forceinline__ float ninf<float>() { return -INFINITY; }
template <> __device__ __forceinline__ uint16_t ninf<uint16_t>() { return 0xFF80u; }

template <typename T>
__device__ __forceinline__ float ld_logit(const T *p) {
    return widen(__ldg(p));
}

// Block reductions (fixed order: the same inputs give the same result in every CTA).
__device__ __forceinline__ float block_max(float v, Misc &ms) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) ms.fred[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = ms.fred[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) r = fmaxf(r, ms.fred[w]);
    return r;
}
__device__ __forceinline__ float block_sum(float v, Misc &ms) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) ms.fred[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = ms.fred[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) r += ms.fred[w];
    return r;
}
__device__ __forceinline__ void block_sum2(unsigned long long &a, unsigned long long &b,
                                           Misc &ms) {
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        ms.ured[threadIdx.x >> 5][0] = a;
        ms.ured[threadIdx.x >> 5][1] = b;
    }
    __syncthreads();
    a = b = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        a += ms.ured[w][0];
        b += ms.ured[w][1];
    }
}
// Inclusive prefix sum of one u64 per thread in thread order; *total gets the block sum.
__device__ __forceinline__ unsigned long long block_incl_scan(unsigned long long v, Misc &ms,
                                                              unsigned long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long s = v;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, s, o);
        if (lane >= o) s += y;
    }
    __syncthreads();
    if (lane == 31) ms.ured[warp][0] = s;
    __syncthreads();
    unsigned long long before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) before += ms.ured[w][0];
        tot += ms.ured[w][0];
    }
    *total = tot;
    return before + s;
}

// Depth of weight w below its chunk's top octave, in bins: 0 for w just under 2, RB per
// octave; the bits of w hold the octave (exponent) and the bin (top mantissa bits).
__device__ __forceinline__ uint32_t depth_of(uint32_t bits) { return (0x3FFFFFFFu - bits) >> 19; }
__device__ __forceinline__ uint32_t mant24(uint32_t bits) { return (bits & 0x7FFFFFu) | 0x800000u; }

// Edges of local bin d as weights relative to the chunk's top octave: [lo, hi).
__device__ __forceinline__ void bin_edges(int d, float &lo, float &hi) {
    const int oct = d / RB, sub = d % RB;
    const float sc = ldexpf(1.0f, -oct);
    lo = sc * (1.0f + (RB - 1 - sub) / float(RB));
    hi = sc * (1.0f + (RB - sub) / float(RB));
}
// Fixed-point weight of an element whose 24-bit mantissa is W and whose octave lies K below
// the row's top: W * 2^(-23 - K) * 2^FSH.
__device__ __forceinline__ unsigned long long fxw(unsigned long long W, int K) {
    return K <= FSH - 23 ? (W << (FSH - 23 - K)) : (W >> (K - (FSH - 23)));
}
// floor(u * tot) for u an odd multiple of 2^-24 in (0, 1), in integers
__device__ __forceinline__ unsigned long long scale_u24(float u, unsigned long long tot) {
    const unsigned long long k = static_cast<unsigned long long>(u * 16777216.0f);
    const unsigned long long lo = k * tot, hi = __umul64hi(k, tot);
    return (hi << 40) | (lo >> 24);
}

// ---------------------------------------------------------------- staging

// Stage elements [e0, e0 + n) of a row into buf: element i lands at byte pad + i * ES, pad =
// (address of element e0) % 16, so that the 16-byte-aligned body arrives by one bulk copy;
// the ragged head and tail are loaded by threads, and the bytes of the 16-byte vectors
// around the data are filled with -inf.  Returns pad / ES (elements).
template <typename T>
__device__ int stage_row(T *buf, const T *row, int64_t e0, int n, unsigned long long *bar) {
    constexpr int ES = sizeof(T);
    const uintptr_t ga = reinterpret_cast<uintptr_t>(row + e0);
    const int pad = static_cast<int>(ga & 15u);
    const uintptr_t a0 = (ga + 15u) & ~static_cast<uintptr_t>(15u);
    const uintptr_t a1 = (ga + static_cast<uintptr_t>(n) * ES) & ~static_cast<uintptr_t>(15u);
    const int padE = pad / ES;
    int h = n, tail0 = n;   // plain-loaded elements: [0, h) and [tail0, n)
    if (a1 > a0) {
        h = static_cast<int>((a0 - ga) / ES);
        tail0 = static_cast<int>((a1 - ga) / ES);
    }
    if (threadIdx.x == 0) {
        if (a1 > a0) {
            mbar_arrive_tx(bar, static_cast<uint32_t>(a1 - a0));
            bulk_g2s(reinterpret_cast<char *>(buf) + pad + (a0 - ga),
                     reinterpret_cast<const void *>(a0), static_cast<uint32_t>(a1 - a0), bar);
        } else {
            mbar_arrive_tx(bar, 0u);
        }
    }
    // plain elements and the -inf fill of the vectors' other bytes
    const int nvec = (pad + n * ES + 15) / 16;
    const int tot = nvec * (16 / ES);
    for (int i = threadIdx.x; i < tot; i += NT) {
        const int e = i - padE;
        if (e < 0 || e >= n) buf[i] = ninf<T>();
        else if (e < h || e >= tail0) buf[i] = row[e0 + e];
    }
    return padE;
}

// ---------------------------------------------------------------- the plan

// Plan A of row r after W1 (warp r): the row maximum, top octave, total weight, the loose cut
// for pass 2, and whether the unit must take the exact path.
__device__ void plan_a(const Params &P, const SlotN *N, int r, float xref, float c2, int32_t kk,
                       float pp, RowPlan &pl) {
    const int lane = threadIdx.x & 31;
    const bool use_k = kk >= 1 && static_cast<int64_t>(kk) < P.V;
    const bool use_p = pp < 1.0f;
    // a lane holds up to NCMAX / 32 chunks' statistics, loaded at once
    constexpr int SPL = NCMAX / 32;
    ChunkStat st[SPL];
#pragma unroll
    for (int q = 0; q < SPL; ++q) {
        const int cc = lane + 32 * q;
        st[q] = cc < P.NC ? ldcg(&N->stat[r][cc]) : ChunkStat{-INFINITY, INT32_MIN, 0.0f, -INFINITY};
    }
    float M = -INFINITY, L = -INFINITY;
    int32_t ot = INT32_MIN;
    int bad = 0;
#pragma unroll
    for (int q = 0; q < SPL; ++q) {
        M = fmaxf(M, st[q].m);
        ot = max(ot, st[q].otop);
        if (st[q].kb != st[q].kb) bad = 1;
        else L = fmaxf(L, st[q].kb);
    }
    for (int o = 16; o > 0; o >>= 1) {
        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        L = fmaxf(L, __shfl_xor_sync(0xFFFFFFFFu, L, o));
        ot = max(ot, __shfl_xor_sync(0xFFFFFFFFu, ot, o));
        bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, o);
    }
    unsigned long long z = 0;
    int alias = 0;
#pragma unroll
    for (int q = 0; q < SPL; ++q) {
        if (st[q].otop != INT32_MIN) {
            z += __float2ull_rn(ldexpf(st[q].zsum, st[q].otop - ot + FSH));
            if (ot - st[q].otop > NO - ZL - 1) alias = 1;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
        alias |= __shfl_xor_sync(0xFFFFFFFFu, alias, o);
    }
    pl.M = M;
    pl.xref = xref;
    pl.otop = ot;
    pl.pm = (ot == INT32_MIN) ? 1 : 0;
    pl.Z = z;
    pl.fallback = bad || (alias && (use_k || use_p));
    pl.dk = pl.dlo = pl.dhi = pl.dmax = pl.dabove = -1;
    pl.cnt_above_k = 0;
    float xc = -INFINITY;
    if (!pl.pm) {
        if (use_k) {
            xc = L;
        } else if (use_p) {
            // a kept logit has weight > (1 - p) Z / V: x > x_ref + (otop + log2(...)) / c2,
            // lowered by 2^-6 of an octave for the rounding of the weights
            const float lw = log2f((1.0f - pp) * __ull2float_rn(z) / static_cast<float>(P.V)) - FSH;
            xc = xref + (static_cast<float>(ot) + lw - 0.015625f) / c2;
        }
    }
    pl.xcut = xc;
}

// Plan B after W1b, by the whole CTA: each row gets 128 threads (warps 4r..4r+3), a thread
// the BPT consecutive bins t*BPT.. of the row's merged histogram (octaves 0..ZL below the
// row top, bin = octave * RB + sub).  A scan over the threads gives every bin's cumulative
// weight bounds (rigorous: each element added its mantissa >> QSH) and exact counts (top-k);
// shared atomics find the top-k bin and the window of bins that can hold the top-p crossing.
constexpr int BPT = (NBL + 127) / 128;
__device__ void plan_b_block(const SlotZ *Z, int nrows, int32_t kk, float pp, int64_t V, Misc &ms) {
    const int r = threadIdx.x >> 7, t = threadIdx.x & 127, lane = threadIdx.x & 31;
    const int wr = (threadIdx.x >> 5) & 3;
    const bool use_k = kk >= 1 && static_cast<int64_t>(kk) < V;
    const bool use_p = pp < 1.0f;
    const bool active = r < nrows && !ms.plan[r].pm && !ms.plan[r].fallback;
    RowPlan &pl = ms.plan[r < nrows ? r : 0];
    unsigned long long lo[BPT], hi[BPT];
    uint32_t cn[BPT];
    unsigned long long slo = 0, shi = 0, scn = 0;
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        const int i = t * BPT + q;
        lo[q] = hi[q] = 0ull;
        cn[q] = 0u;
        if (active && i < NBL) {
            const int K = i / RB;
            const int slot = (((pl.otop - K) % NO) + NO) % NO;
            const unsigned long long m = ldcg(&Z->ring_mass[r][slot * RB + i % RB]);
            const uint32_t c = use_k ? ldcg(&Z->ring_cnt[r][slot * RB + i % RB]) : static_cast<uint32_t>(m >> (23 - QSH));
            lo[q] = fxw(m << QSH, K);
            hi[q] = fxw((m << QSH) + static_cast<unsigned long long>(c) * ((1u << QSH) - 1u), K) +
                    (K > FSH - 23 ? static_cast<unsigned long long>(c) + 1ull : 0ull);
            cn[q] = use_k ? c : 0u;
        }
        slo += lo[q];
        shi += hi[q];
        scn += cn[q];
    }
    // exclusive prefix over the row's 128 threads: warp scans, then the warps before
    unsigned long long a = slo, bh = shi, n = scn;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long ya = __shfl_up_sync(0xFFFFFFFFu, a, o);
        const unsigned long long yb = __shfl_up_sync(0xFFFFFFFFu, bh, o);
        const unsigned long long yn = __shfl_up_sync(0xFFFFFFFFu, n, o);
        if (lane >= o) {
            a += ya;
            bh += yb;
            n += yn;
        }
    }
    if (threadIdx.x < 2) {
        ms.pb_dk[threadIdx.x] = NBL;
        ms.pb_dlo[threadIdx.x] = NBL;
        ms.pb_dhi[threadIdx.x] = -1;
    }
    if (lane == 31) {
        ms.pb_w[r][wr][0] = a;
        ms.pb_w[r][wr][1] = bh;
        ms.pb_w[r][wr][2] = n;
    }
    __syncthreads();
    unsigned long long elo = a - slo, ehi = bh - shi, ecn = n - scn;
    for (int w = 0; w < wr; ++w) {
        elo += ms.pb_w[r][w][0];
        ehi += ms.pb_w[r][w][1];
        ecn += ms.pb_w[r][w][2];
    }
    // top-k: the first bin whose cumulative count reaches kk
    if (active && use_k) {
        unsigned long long c = ecn;
#pragma unroll
        for (int q = 0; q < BPT; ++q) {
            c += cn[q];
            if (c >= static_cast<unsigned long long>(kk) && t * BPT + q < NBL) {
                atomicMin(&ms.pb_dk[r], t * BPT + q);
                break;
            }
        }
    }
    __syncthreads();
    const int dk = use_k ? ms.pb_dk[r] : NBL;
    if (active && use_k && dk < NBL && dk / BPT == t) {
        unsigned long long cl = elo, ch = ehi, cc = ecn;
        for (int q = 0; q < dk - t * BPT; ++q) {
            cl += lo[q];
            ch += hi[q];
            cc += cn[q];
        }
        ms.pb_zlo[r] = cl;
        ms.pb_zhi[r] = ch + hi[dk - t * BPT];
        ms.pb_cab[r] = static_cast<uint32_t>(cc);
    }
    __syncthreads();
    if (active && use_p && !(use_k && dk >= NBL)) {
        const unsigned long long zlo = use_k ? ms.pb_zlo[r] : pl.Z, zhi = use_k ? ms.pb_zhi[r] : pl.Z;
        // the top-p target p * Zk, widened by 2^-20 for the rounding of the product
        const unsigned long long t_lo = __float2ull_rd(pp * __ull2float_rd(zlo) * (1.0f - 9.5367431640625e-07f));
        const unsigned long long t_hi = __float2ull_ru(pp * __ull2float_ru(zhi) * (1.0f + 9.5367431640625e-07f));
        unsigned long long cl = elo, ch = ehi;
#pragma unroll
        for (int q = 0; q < BPT; ++q) {
            const int i = t * BPT + q;
            // the bin can hold the crossing: its upper bound reaches t_lo, the lower bound of
            // the weight before it stays below t_hi
            if (i < NBL && i <= dk && ch + hi[q] >= t_lo && cl < t_hi) {
                atomicMin(&ms.pb_dlo[r], i);
                atomicMax(&ms.pb_dhi[r], i);
            }
            cl += lo[q];
            ch += hi[q];
        }
    }
    __syncthreads();
    if (threadIdx.x < nrows && !ms.plan[threadIdx.x].pm && !ms.plan[threadIdx.x].fallback) {
        RowPlan &p2 = ms.plan[threadIdx.x];
        const int rr = threadIdx.x;
        if (use_k) {
            if (ms.pb_dk[rr] >= NBL) {
                p2.fallback = 1;
            } else {
                p2.dk = ms.pb_dk[rr];
                p2.dabove = p2.dk;
                p2.dmax = p2.dk;
                p2.cnt_above_k = ms.pb_cab[rr];
            }
        }
        if (use_p && !p2.fallback) {
            if (ms.pb_dlo[rr] >= NBL || ms.pb_dhi[rr] < 0) {
                p2.fallback = 1;
            } else {
                p2.dlo = ms.pb_dlo[rr];
                p2.dhi = ms.pb_dhi[rr];
                p2.dabove = p2.dlo;
                p2.dmax = use_k ? max(p2.dhi, p2.dk) : p2.dhi;
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- resolution

// Sort the first n (<= CAP) u64 keys in s in decreasing order (bitonic over the next power
// of two; the rest filled with 0, below every real key).
__device__ void sort_desc(unsigned long long *s, int n) {
    int N = 2;
    while (N < n) N <<= 1;
    for (int i = n + threadIdx.x; i < N; i += NT) s[i] = 0ull;
    __syncthreads();
    for (int k = 2; k <= N; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < N / 2; i += NT) {
                const int lo = ((i / j) * 2 * j) + (i % j);
                const int hi = lo + j;
                const bool desc = ((lo & k) == 0);
                const unsigned long long a = s[lo], b = s[hi];
                if ((a < b) == desc) {
                    s[lo] = b;
                    s[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

// Candidate entry: (order key << 32) | (octave below the row top << 24) | 24-bit mantissa.
__device__ __forceinline__ unsigned long long cand_weight(unsigned long long e) {
    const uint32_t lo = static_cast<uint32_t>(e);
    return fxw(lo & 0xFFFFFFu, static_cast<int>(lo >> 24));
}
__device__ __forceinline__ int cand_depth(unsigned long long e) {
    const uint32_t lo = static_cast<uint32_t>(e);
    return static_cast<int>(lo >> 24) * RB + (RB - 1 - static_cast<int>((lo >> 19) & 15u));
}

// Exact threshold (order key of the lowest kept logit) and kept weight of filtered row r from
// the plan, the chunks' exact sums and the candidates (sorted in s).  False: the unit needs
// the exact path.
__device__ bool resolve_row(const SlotZ *Z, const SlotN *N, int r, const RowPlan &pl, int NC,
                            int32_t kk, float pp, int64_t V, unsigned long long *s, Misc &ms,
                            uint32_t &theta, unsigned long long &zk) {
    const bool use_k = kk >= 1 && static_cast<int64_t>(kk) < V;
    const bool use_p = pp < 1.0f;
    const uint32_t nc = ldcg(&Z->ncand[r]);
    if (nc > static_cast<uint32_t>(CAP)) return false;
    const int n = static_cast<int>(nc);
    // the chunks' exact sums above the bins and in the middle band (fixed order)
    if (threadIdx.x == 0) {
        unsigned long long a = 0, m = 0;
        for (int c = 0; c < NC; ++c) {
            a += __ldcg(&N->pub[c].above[r]);
            m += __ldcg(&N->pub[c].mid[r]);
        }
        ms.dred[0][0] = a;
        ms.dred[0][1] = m;
    }
    for (int i = threadIdx.x; i < n; i += NT) s[i] = ldcg(&N->cand[r][i]);
    __syncthreads();
    const unsigned long long S_above = ms.dred[0][0], S_mid = ms.dred[0][1];
    __syncthreads();
    sort_desc(s, n);
    uint32_t theta_k = 0u;
    unsigned long long zkv = pl.Z;
    if (use_k) {
        if (threadIdx.x == 0) {
            const uint32_t need = static_cast<uint32_t>(kk) - pl.cnt_above_k;  // >= 1
            uint32_t seen = 0, th = 0u;
            for (int i = 0; i < n; ++i) {
                const unsigned long long e = s[i];
                if (cand_depth(e) != pl.dk) continue;
                const uint32_t key = static_cast<uint32_t>(e >> 32);
                if (seen < need) {
                    th = key;
                    ++seen;
                } else if (key != th) {
                    break;
                }
            }
            unsigned long long w = 0;
            for (int i = 0; i < n; ++i)
                if (static_cast<uint32_t>(s[i] >> 32) >= th) w += cand_weight(s[i]);
            ms.tk_theta = th;
            ms.tk_z = S_above + S_mid + w;
            ms.tk_ok = (seen == need) ? 1 : 0;
        }
        __syncthreads();
        const int ok = ms.tk_ok;
        theta_k = ms.tk_theta;
        zkv = ms.tk_z;
        __syncthreads();
        if (!ok) return false;
        if (!use_p) {
            theta = theta_k;
            zk = zkv;
            return true;
        }
    }
    // top-p inside the window: groups of equal logits in decreasing order; a group stays
    // when the weight strictly above it is < p * Zk.  One thread walks the sorted window
    // (it holds a few hundred entries).
    if (threadIdx.x == 0) {
        const unsigned long long target = __float2ull_rn(pp * __ull2float_rn(zkv));
        unsigned long long above = S_above, kept = 0;
        uint32_t last = 0xFFFFFFFFu;
        int i = 0;
        while (i < n) {
            const unsigned long long e = s[i];
            const uint32_t key = static_cast<uint32_t>(e >> 32);
            const int dd = cand_depth(e);
            if (dd < pl.dlo || dd > pl.dhi || key < theta_k) {
                ++i;
                continue;
            }
            // the group of this key (window entries only)
            unsigned long long g = 0;
            int j = i;
            while (j < n && static_cast<uint32_t>(s[j] >> 32) == key) {
                const int d2 = cand_depth(s[j]);
                if (d2 >= pl.dlo && d2 <= pl.dhi) g += cand_weight(s[j]);
                ++j;
            }
            if (above < target) {
                kept += g;
                last = key;
                above += g;
            } else {
                break;
            }
            i = j;
        }
        ms.tk_theta = last;
        ms.tk_z = S_above + kept;
    }
    __syncthreads();
    const uint32_t lk = ms.tk_theta;
    const unsigned long long kz = ms.tk_z;
    __syncthreads();
    if (lk == 0xFFFFFFFFu) return false;
    theta = max(lk, theta_k);
    zk = kz;
    return true;
}

// ---------------------------------------------------------------- the resolver's draw

// A nucleus entry written by another CTA, read through L2.
__device__ __forceinline__ NucEntry ld_nuc(const NucEntry *p) {
    const int32_t *w = reinterpret_cast<const int32_t *>(p);
    NucEntry e;
    e.id = __ldcg(w);
    e.xt = __int_as_float(__ldcg(w + 1));
    e.xq = __int_as_float(__ldcg(w + 2));
    return e;
}

// One unit's sampling constants, fixed by the resolution.
struct DrawCtx {
    int kind;
    int32_t dj;
    bool dvalid, one_hot;
    float c2;
    float xr[2];      // reference logits
    float ot[2];      // row top octaves
    float iz[2];      // 1 / kept weight
    uint32_t th[2];   // thresholds (order keys)
    int pm[2];        // point-mass rows
    int rows;
};

// Fixed-point residual max(0, p - q) and p of logit id with target logit xt and draft xq.
__device__ __forceinline__ void draw_weights(const DrawCtx &g, int64_t id, float xt, float xq,
                                             unsigned long long &rfx, unsigned long long &pfx) {
    float p;
    if (g.pm[0]) p = (id == 0) ? 1.0f : 0.0f;
    else p = (order_key(xt) >= g.th[0]) ? ex2f(fmaf(xt - g.xr[0], g.c2, -g.ot[0])) * g.iz[0] : 0.0f;
    float q = 0.0f;
    if (g.kind == KIND_SAMPLE && p > 0.0f) {
        if (g.one_hot) q = (g.dvalid && id == g.dj) ? 1.0f : 0.0f;
        else if (g.pm[1]) q = (id == 0) ? 1.0f : 0.0f;
        else q = (order_key(xq) >= g.th[1]) ? ex2f(fmaf(xq - g.xr[1], g.c2, -g.ot[1])) * g.iz[1] : 0.0f;
    }
    rfx = __float2ull_rn(fmaxf(p - q, 0.0f) * FXF);
    pfx = __float2ull_rn(p * FXF);
}

// The inverse CDF over the unit's nucleus list (filtered rows), kept per (chunk, warp range)
// in id order: sums per range by warps, the range that holds the target (chunks, then warp
// ranges, in order), then a block walk over its entries.  Returns the drawn id (every
// thread).  sc holds 2 * NC * NW sums.
__device__ int32_t draw_nucleus(const Params &P, const SlotN *N, const NucEntry *nucs,
                                const DrawCtx &g, float u, unsigned long long *sc, Misc &ms) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sseg = P.seg / NW;
    const int nr = P.NC * NW;
    for (int rg = warp; rg < nr; rg += NW) {
        const int c = rg / NW, w = rg % NW;
        const uint32_t cnt = min(__ldcg(&N->pub[c].nucw[w]), static_cast<uint32_t>(sseg));
        const NucEntry *base = nucs + static_cast<size_t>(c) * P.seg + static_cast<size_t>(w) * sseg;
        unsigned long long rs = 0, ps = 0;
        for (uint32_t i = lane; i < cnt; i += 32) {
            const NucEntry e = ld_nuc(base + i);
            unsigned long long rf, pf;
            draw_weights(g, e.id, e.xt, e.xq, rf, pf);
            rs += rf;
            ps += pf;
        }
        for (int o = 16; o > 0; o >>= 1) {
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, o);
            ps += __shfl_xor_sync(0xFFFFFFFFu, ps, o);
        }
        if (lane == 0) {
            sc[2 * rg] = rs;
            sc[2 * rg + 1] = ps;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long rt = 0, pt = 0;
        for (int rg = 0; rg < nr; ++rg) {
            rt += sc[2 * rg];
            pt += sc[2 * rg + 1];
        }
        const int usep = (rt == 0ull) ? 1 : 0;
        const unsigned long long tot = usep ? pt : rt;
        const unsigned long long tgt = scale_u24(u, tot);
        unsigned long long acc = 0;
        int cs = -1;
        for (int rg = 0; rg < nr && tot > 0ull; ++rg) {
            const unsigned long long v = sc[2 * rg + usep];
            if (tgt < acc + v) {
                cs = rg;
                break;
            }
            acc += v;
        }
        ms.cstar = cs;
        ms.target = tgt - acc;
        ms.usep = usep;
        ms.ured[0][1] = 0ull;
    }
    __syncthreads();
    const int cs = ms.cstar, usep = ms.usep;
    if (cs >= 0) {
        const int c = cs / NW, w = cs % NW;
        const uint32_t cnt = min(__ldcg(&N->pub[c].nucw[w]), static_cast<uint32_t>(sseg));
        const NucEntry *base = nucs + static_cast<size_t>(c) * P.seg + static_cast<size_t>(w) * sseg;
        unsigned long long want = ms.target;
        for (uint32_t b0 = 0; b0 < cnt; b0 += NT) {
            const uint32_t i = b0 + threadIdx.x;
            unsigned long long v = 0;
            NucEntry e{0, 0.0f, 0.0f};
            if (i < cnt) {
                e = ld_nuc(base + i);
                unsigned long long rf, pf;
                draw_weights(g, e.id, e.xt, e.xq, rf, pf);
                v = usep ? pf : rf;
            }
            unsigned long long tot;
            const unsigned long long inc = block_incl_scan(v, ms, &tot);
            if (want < tot) {
                if (i < cnt && want < inc && want >= inc - v) ms.ured[0][1] = static_cast<unsigned long long>(e.id);
                __syncthreads();
                break;
            }
            want -= tot;
            __syncthreads();
        }
    }
    __syncthreads();
    const int32_t tok = static_cast<int32_t>(ms.ured[0][1]);
    __syncthreads();
    return tok;
}

// The inverse CDF for an unfiltered row: the chunks' published sums pick the chunk, whose
// logits are read again from global memory and walked in id order (contiguous ranges per
// thread).  Returns the drawn id (every thread).
template <typename T>
__device__ int32_t draw_unfiltered(const Params &P, const SlotN *N, const DrawCtx &g, float u,
                                   const T *rowT, const T *rowQ, Misc &ms) {
    if (threadIdx.x == 0) {
        unsigned long long rt = 0, pt = 0;
        for (int c = 0; c < P.NC; ++c) {
            rt += __ldcg(&N->pub[c].r);
            pt += __ldcg(&N->pub[c].p);
        }
        const int usep = (rt == 0ull) ? 1 : 0;
        const unsigned long long tot = usep ? pt : rt;
        const unsigned long long tgt = scale_u24(u, tot);
        unsigned long long acc = 0;
        int cs = -1;
        for (int c = 0; c < P.NC && tot > 0ull; ++c) {
            const unsigned long long v = usep ? __ldcg(&N->pub[c].p) : __ldcg(&N->pub[c].r);
            if (tgt < acc + v) {
                cs = c;
                break;
            }
            acc += v;
        }
        ms.cstar = cs;
        ms.target = tgt - acc;
        ms.usep = usep;
        ms.ured[0][1] = 0ull;
    }
    __syncthreads();
    const int cs = ms.cstar, usep = ms.usep;
    if (cs >= 0) {
        const int64_t e0 = static_cast<int64_t>(cs) * P.CH;
        const int64_t n = min(P.CH, P.V - e0);
        const int64_t per = (n + NT - 1) / NT;
        const int64_t lo = threadIdx.x * per, hi = min(n, lo + per);
        unsigned long long s = 0;
        for (int64_t i = lo; i < hi; ++i) {
            unsigned long long rf, pf;
            draw_weights(g, e0 + i, ld_logit(rowT + e0 + i), rowQ ? ld_logit(rowQ + e0 + i) : 0.0f, rf, pf);
            s += usep ? pf : rf;
        }
        unsigned long long tot;
        const unsigned long long inc = block_incl_scan(s, ms, &tot);
        const unsigned long long want = ms.target;
        if (want >= inc - s && want < inc) {
            unsigned long long cum = inc - s;
            int64_t tok = hi - 1;
            for (int64_t i = lo; i < hi; ++i) {
                unsigned long long rf, pf;
                draw_weights(g, e0 + i, ld_logit(rowT + e0 + i), rowQ ? ld_logit(rowQ + e0 + i) : 0.0f, rf, pf);
                cum += usep ? pf : rf;
                if (cum > want) {
                    tok = i;
                    break;
                }
            }
            ms.ured[0][1] = static_cast<unsigned long long>(e0 + tok);
        }
    }
    __syncthreads();
    const int32_t tok = static_cast<int32_t>(ms.ured[0][1]);
    __syncthreads();
    return tok;
}

// ---------------------------------------------------------------- the slow exact path

// Everything about one row computed from global memory by one CTA: the maximum, the top-k
// and top-p thresholds by radix selection over the order keys, and the kept weight (fixed
// point, 2^40 per unit of the largest logit's weight).
template <typename T>
__device__ void slow_row(const T *row, int64_t V, float c2, int32_t kk, float pp,
                         unsigned long long *scr, unsigned long long *wh, Misc &ms, float &M,
                         uint32_t &theta, double &zk, int &pm) {
    float m = -INFINITY;
    for (int64_t i = threadIdx.x; i < V; i += NT) m = fmaxf(m, ld_logit(row + i));
    M = block_max(m, ms);
    pm = (M == -INFINITY) ? 1 : 0;
    theta = 0u;
    zk = 1.0;
    if (pm) return;
    const bool use_k = kk >= 1 && static_cast<int64_t>(kk) < V;
    const bool use_p = pp < 1.0f;
    auto wfx = [&](float x) -> unsigned long long {
        return __double2ull_rn(static_cast<double>(ex2f(__fmul_rn(x - M, c2))) * FXD);
    };
    uint32_t tk = 0u;
    if (use_k) {
        // the kk-th largest key, 8 bits at a time from the top
        uint32_t prefix = 0u, need = static_cast<uint32_t>(kk);
        for (int sh = 24; sh >= 0; sh -= 8) {
            uint32_t *h = reinterpret_cast<uint32_t *>(scr);
            uint32_t *hw = reinterpret_cast<uint32_t *>(wh) + (threadIdx.x >> 5) * 256;   // per warp
            for (int i = threadIdx.x; i < 256 * NW; i += NT) reinterpret_cast<uint32_t *>(wh)[i] = 0u;
            __syncthreads();
            const uint32_t hmask = sh == 24 ? 0u : (0xFFFFFFFFu << (sh + 8));
            for (int64_t i = threadIdx.x; i < V; i += NT) {
                const uint32_t key = order_key(ld_logit(row + i));
                if ((key & hmask) == prefix) atomicAdd(&hw[(key >> sh) & 255u], 1u);
            }
            __syncthreads();
            for (int i = threadIdx.x; i < 256; i += NT) {
                uint32_t t = 0u;
                for (int w = 0; w < NW; ++w) t += reinterpret_cast<uint32_t *>(wh)[w * 256 + i];
                h[i] = t;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                uint32_t acc = 0u;
                int dsel = 0;
                for (int dgt = 255; dgt >= 0; --dgt) {
                    if (acc + h[dgt] >= need) {
                        dsel = dgt;
                        break;
                    }
                    acc += h[dgt];
                }
                ms.ured[0][0] = prefix | (static_cast<uint32_t>(dsel) << sh);
                ms.ured[0][1] = need - acc;
            }
            __syncthreads();
            prefix = static_cast<uint32_t>(ms.ured[0][0]);
            need = static_cast<uint32_t>(ms.ured[0][1]);
            __syncthreads();
        }
        tk = prefix;
    }
    // kept weight of the top-k set
    unsigned long long s = 0, dummy = 0;
    for (int64_t i = threadIdx.x; i < V; i += NT) {
        const float x = ld_logit(row + i);
        if (order_key(x) >= tk) s += wfx(x);
    }
    block_sum2(s, dummy, ms);
    if (!use_p) {
        theta = tk;
        zk = static_cast<double>(s) / FXD;
        return;
    }
    const unsigned long long zkf = s;
    const unsigned long long target = __double2ull_ru(static_cast<double>(pp) * static_cast<double>(zkf));
    // the lowest key K with (weight of keys > K within the top-k set) < target
    uint32_t prefix = 0u;
    unsigned long long above = 0;
    for (int sh = 24; sh >= 0; sh -= 8) {
        unsigned long long *hw = wh + (threadIdx.x >> 5) * 256;   // per warp
        for (int i = threadIdx.x; i < 256 * NW; i += NT) wh[i] = 0ull;
        __syncthreads();
        const uint32_t hmask = sh == 24 ? 0u : (0xFFFFFFFFu << (sh + 8));
        for (int64_t i = threadIdx.x; i < V; i += NT) {
            const float x = ld_logit(row + i);
            const uint32_t key = order_key(x);
            if (key >= tk && (key & hmask) == prefix)
                atomicAdd(&hw[(key >> sh) & 255u], wfx(x));
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 256; i += NT) {
            unsigned long long t = 0ull;
            for (int w = 0; w < NW; ++w) t += wh[w * 256 + i];
            scr[i] = t;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long acc = above;
            int dsel = -1;
            unsigned long long acc_sel = above;
            for (int dgt = 255; dgt >= 0; --dgt) {
                if (scr[dgt] == 0ull) continue;
                if (acc < target) {   // the group(s) of this digit start below the target
                    dsel = dgt;
                    acc_sel = acc;
                } else {
                    break;
                }
                acc += scr[dgt];
            }
            if (dsel < 0) dsel = 255;   // unreachable: the top element always stays
            ms.ured[0][0] = prefix | (static_cast<uint32_t>(dsel) << sh);
            ms.ured[0][1] = acc_sel;
        }
        __syncthreads();
        prefix = static_cast<uint32_t>(ms.ured[0][0]);
        above = ms.ured[0][1];
        __syncthreads();
    }
    theta = max(prefix, tk);
    s = 0;
    for (int64_t i = threadIdx.x; i < V; i += NT) {
        const float x = ld_logit(row + i);
        if (order_key(x) >= theta) s += wfx(x);
    }
    block_sum2(s, dummy, ms);
    zk = static_cast<double>(s) / FXD;
}

// The whole unit on the exact path: thresholds, p(d), q(d), the accept test, and the draw.
template <typename T>
__device__ void slow_unit(const Params &P, int kind, int64_t b, int j, int32_t dj, bool dvalid,
                          float c2, int32_t kk, float pp, const T *rowT, const T *rowQ,
                          unsigned long long *scr, unsigned long long *wh, Misc &ms) {
    float Mt, Mq = 0.0f;
    uint32_t tht, thq = 0u;
    double zt, zq = 1.0;
    int pmt, pmq = 0;
    slow_row(rowT, P.V, c2, kk, pp, scr, wh, ms, Mt, tht, zt, pmt);
    if (rowQ) slow_row(rowQ, P.V, c2, kk, pp, scr, wh, ms, Mq, thq, zq, pmq);
    const int64_t ui = b * (P.D + 1) + j;
    float ua, us;
    unit_uniforms(P.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(j), ua, us);
    // weight of one logit relative to the row's largest
    auto wt = [&](float x) -> double { return pmt ? 0.0 : static_cast<double>(ex2f(__fmul_rn(x - Mt, c2))); };
    auto wq = [&](float x) -> double { return pmq ? 0.0 : static_cast<double>(ex2f(__fmul_rn(x - Mq, c2))); };
    bool draw = true;
    if (kind == KIND_SAMPLE) {
        float pt = 0.0f, pd = 0.0f;
        bool acc = false;
        if (dvalid) {
            const float xt = ld_logit(rowT + dj);
            const bool kt = pmt ? (dj == 0) : (order_key(xt) >= tht);
            const double ptd = pmt ? (dj == 0 ? 1.0 : 0.0) : (kt ? wt(xt) / zt : 0.0);
            double pdd = 1.0;
            bool kq = true;
            double xq = 0.0;
            if (rowQ) {
                xq = ld_logit(rowQ + dj);
                kq = pmq ? (dj == 0) : (order_key(static_cast<float>(xq)) >= thq);
                pdd = pmq ? (dj == 0 ? 1.0 : 0.0) : (kq ? wq(static_cast<float>(xq)) / zq : 0.0);
            }
            pt = static_cast<float>(ptd);
            pd = static_cast<float>(pdd);
            if (!kt) acc = false;
            else if (!kq) acc = true;
            else {
                double ratio;
                if (!rowQ || pmt || pmq) ratio = ptd / pdd;
                else ratio = exp2((static_cast<double>(xt) - Mt - (xq - Mq)) * c2) * (zq / zt);
                acc = static_cast<double>(ua) <= ratio;
            }
        }
        if (threadIdx.x == 0) {
            P.rec[ui].flags = acc ? 1 : 0;
            P.rec[ui].pt = pt;
            P.rec[ui].pd = pd;
            P.rec[ui].token = -1;
            if (!acc) atomicMax(P.rowflag + b, static_cast<uint32_t>(P.D + 1 - j));
            const uint32_t rf = ld_acq(P.rowflag + b);
            ms.cstar = (!acc && !(rf > static_cast<uint32_t>(P.D + 1 - j))) ? 1 : 0;
        }
    } else {
        if (threadIdx.x == 0) {
            P.rec[ui].flags = 0;
            P.rec[ui].pt = 0.0f;
            P.rec[ui].pd = 0.0f;
            P.rec[ui].token = -1;
            ms.cstar = ld_acq(P.rowflag + b) == 0u ? 1 : 0;
        }
    }
    __syncthreads();
    draw = ms.cstar != 0;   // one thread's view of the row's rejections, for every thread
    __syncthreads();
    if (!draw) return;
    // residual (or p alone) over the row in id order: contiguous ranges per thread
    const int64_t per = (P.V + NT - 1) / NT;
    const int64_t lo = threadIdx.x * per, hi = min(P.V, lo + per);
    auto weights = [&](int64_t i, unsigned long long &r, unsigned long long &p) {
        double p_i;
        if (pmt) p_i = (i == 0) ? 1.0 : 0.0;
        else {
            const float x = ld_logit(rowT + i);
            p_i = order_key(x) >= tht ? wt(x) / zt : 0.0;
        }
        double q_i = 0.0;
        if (kind == KIND_SAMPLE) {
            if (!rowQ) q_i = (dvalid && i == dj) ? 1.0 : 0.0;
            else if (pmq) q_i = (i == 0) ? 1.0 : 0.0;
            else {
                const float x = ld_logit(rowQ + i);
                q_i = order_key(x) >= thq ? wq(x) / zq : 0.0;
            }
        }
        r = __double2ull_rn(fmax(0.0, p_i - q_i) * FXD);
        p = __double2ull_rn(p_i * FXD);
    };
    unsigned long long rs = 0, ps = 0;
    for (int64_t i = lo; i < hi; ++i) {
        unsigned long long r, p;
        weights(i, r, p);
        rs += r;
        ps += p;
    }
    unsigned long long rtot = 0, ptot = 0;
    const unsigned long long rinc = block_incl_scan(rs, ms, &rtot);
    const unsigned long long pinc = block_incl_scan(ps, ms, &ptot);
    const bool use_pp = (rtot == 0ull);
    const unsigned long long tot = use_pp ? ptot : rtot;
    const unsigned long long tgt = static_cast<unsigned long long>(floor(static_cast<double>(us) * static_cast<double>(tot)));
    const unsigned long long inc = use_pp ? pinc : rinc, mine = use_pp ? ps : rs;
    const unsigned long long exc = inc - mine;
    if (tot > 0ull && tgt >= exc && tgt < inc) {
        unsigned long long c = exc;
        int64_t tok = hi - 1;
        for (int64_t i = lo; i < hi; ++i) {
            unsigned long long r, p;
            weights(i, r, p);
            c += use_pp ? p : r;
            if (c > tgt) {
                tok = i;
                break;
            }
        }
        P.rec[ui].token = static_cast<int32_t>(tok);
    }
    if (tot == 0ull && threadIdx.x == 0) P.rec[ui].token = 0;
}

// ---------------------------------------------------------------- the kernel

template <typename T>
__global__ void __launch_bounds__(NT, CPS) k_verify_chunks(const Params P) {
    constexpr int ES = sizeof(T);
    constexpr int EPV = 16 / ES;
    extern __shared__ __align__(128) unsigned char smem[];
    T *buf[2] = {reinterpret_cast<T *>(smem), reinterpret_cast<T *>(smem + ROWB)};
    unsigned char *scr = smem + 2 * ROWB;
    uint32_t *hm = reinterpret_cast<uint32_t *>(scr);                 // [NBL] masses
    uint32_t *hc = hm + NBL;                                          // [NBL] counts
    float *tmax = reinterpret_cast<float *>(hc + NBL);                // [NT] thread maxima
    unsigned long long *ccand = reinterpret_cast<unsigned long long *>(tmax + NT);   // [CCAP]
    Misc &ms = *reinterpret_cast<Misc *>(scr + SCR_BYTES);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        mbar_init1(&ms.bar[0]);
        mbar_init1(&ms.bar[1]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < 2 * NBL; i += NT) hm[i] = 0u;
    __syncthreads();
    uint32_t parity[2] = {0u, 0u};

    for (;;) {
        if (tid == 0) {
            uint32_t it = atomicAdd(P.hdr, 1u);
            if (ld_acq(P.hdr + 1) != 0u) it = 0xFFFFFFFFu;
            ms.item = it;
            // ask L2 for the chunk one grid-width ahead
            const int64_t nx = static_cast<int64_t>(it) + gridDim.x;
            if (it != 0xFFFFFFFFu && nx < P.items) {
                const int64_t un = nx / P.NC;
                const int cn = static_cast<int>(nx - un * P.NC);
                const int jn = static_cast<int>(un / P.B);
                const int64_t bn = un - static_cast<int64_t>(jn) * P.B;
                const int64_t e0 = static_cast<int64_t>(cn) * P.CH;
                const int64_t nn = min(P.CH, P.V - e0);
                const bool sampled = P.tau[bn] > 0.0f;
                const T *rows[2] = {static_cast<const T *>(P.T) + (bn * (P.D + 1) + jn) * P.V,
                                    (P.Q && jn < P.D && sampled) ? static_cast<const T *>(P.Q) + (bn * P.D + jn) * P.V : nullptr};
                for (int r = 0; r < 2; ++r) {
                    if (!rows[r]) continue;
                    const uintptr_t ga = reinterpret_cast<uintptr_t>(rows[r] + e0);
                    const uintptr_t a0 = (ga + 15u) & ~static_cast<uintptr_t>(15u);
                    const uintptr_t a1 = (ga + static_cast<uintptr_t>(nn) * ES) & ~static_cast<uintptr_t>(15u);
                    if (a1 > a0) prefetch_l2(reinterpret_cast<const void *>(a0), static_cast<uint32_t>(a1 - a0));
                }
            }
        }
        __syncthreads();
        const uint32_t item = ms.item;
        if (item == 0xFFFFFFFFu || static_cast<int64_t>(item) >= P.items) break;

        // ---- the unit
        const int64_t u = static_cast<int64_t>(item) / P.NC;
        const int c = static_cast<int>(static_cast<int64_t>(item) - u * P.NC);
        const int j = static_cast<int>(u / P.B);
        const int64_t b = u - static_cast<int64_t>(j) * P.B;
        const float tau = P.tau[b];
        const int32_t kk = P.topk ? P.topk[b] : 0;
        const float pp = P.topp ? P.topp[b] : 1.0f;
        const bool bad = !(tau >= 0.0f) || !(pp > 0.0f);
        const bool greedy = bad || tau == 0.0f;
        const int kind = greedy ? KIND_GREEDY : (j == P.D ? KIND_BONUS : KIND_SAMPLE);
        const bool use_k = kk >= 1 && static_cast<int64_t>(kk) < P.V;
        const bool use_p = pp < 1.0f;
        const bool filtered = !greedy && (use_k || use_p);
        const int32_t dj = j < P.D ? P.d[b * P.D + j] : -1;
        const bool dvalid = dj >= 0 && static_cast<int64_t>(dj) < P.V;
        const int nrows = (kind == KIND_SAMPLE && P.Q) ? 2 : 1;
        const int64_t e0 = static_cast<int64_t>(c) * P.CH;
        const int n = static_cast<int>(min(P.CH, P.V - e0));
        const T *rowp[2] = {static_cast<const T *>(P.T) + (b * (P.D + 1) + j) * P.V,
                            nrows == 2 ? static_cast<const T *>(P.Q) + (b * P.D + j) * P.V : nullptr};
        const int s_ = static_cast<int>(u % P.nslot);
        const uint32_t gen = static_cast<uint32_t>(u / P.nslot);
        NucEntry *nucs = P.nuc + static_cast<size_t>(s_) * P.nuc_slot;
        SlotZ *Z = reinterpret_cast<SlotZ *>(P.zone_z + static_cast<size_t>(s_) * ZSZ);
        SlotN *N = reinterpret_cast<SlotN *>(P.zone_n + static_cast<size_t>(s_) * NSZ);
        const float c2 = greedy ? 0.0f : __fdiv_rn(1.4426950408889634f, tau);
        const int64_t ui = b * (P.D + 1) + j;
        if (c == 0 && tid == 0 && P.status) {
            if (bad && j == 0) atomicOr(P.status, MTPSPEC_STATUS_BAD_PARAM);
            if (j < P.D && !dvalid) atomicOr(P.status, MTPSPEC_STATUS_BAD_DRAFT_ID);
        }

        // ---- stage the chunk
        if (tid == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        int padE[2] = {0, 0};
        for (int r = 0; r < nrows; ++r) padE[r] = stage_row<T>(buf[r], rowp[r], e0, n, &ms.bar[r]);
        // the reference logits: the largest of each row's first 32 ids
        if (!greedy && warp < nrows) {
            const int64_t lim = P.V < 32 ? P.V : 32;
            float x = lane < lim ? ld_logit(rowp[warp] + lane) : -INFINITY;
            for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
            if (lane == 0) ms.xref[warp] = (fabsf(x) < 3.0e38f) ? x : 0.0f;
        }
        bool ok = true;
        for (int r = 0; r < nrows; ++r) {
            ok &= mbar_wait(&ms.bar[r], parity[r]);
            parity[r] ^= 1u;
        }
        if (!ok && tid == 0 && P.status) atomicOr(P.status, MTPSPEC_STATUS_TIMEOUT);
        __syncthreads();
        const int nvec[2] = {(padE[0] * ES + n * ES + 15) / 16, (padE[1] * ES + n * ES + 15) / 16};

        // the slot: wait until the unit that used it before has released it
        if (tid == 0) ms.leave = wait_geq(&Z->gen, gen, P) ? 0 : 1;
        __syncthreads();
        bool alive = !ms.leave;

        if (kind == KIND_GREEDY) {
            // ---- greedy unit: the chunk's argmax, merged by the last chunk to arrive
            ArgMax best{-INFINITY, -1};
            const uint4 *vp = reinterpret_cast<const uint4 *>(buf[0]);
            for (int v = tid; v < nvec[0]; v += NT) {
                float x[EPV];
                unpack(vp[v], x);
#pragma unroll
                for (int k = 0; k < EPV; ++k) {
                    const int e = v * EPV + k - padE[0];
                    if (e >= 0 && e < n) best = argmax_merge(best, ArgMax{x[k], static_cast<int32_t>(e0 + e)});
                }
            }
            best = warp_argmax(best);
            __syncthreads();
            if (lane == 0) ms.ared[warp] = best;
            __syncthreads();
            if (tid == 0 && alive) {
                ArgMax t = ms.ared[0];
                for (int w = 1; w < NW; ++w) t = argmax_merge(t, ms.ared[w]);
                N->stat[0][c] = ChunkStat{t.v, t.i, 0.0f, 0.0f};
                __threadfence();
                const uint32_t old = atom_add_ar(&Z->c1, 1u);
                if (old == static_cast<uint32_t>(P.NC - 1)) {
                    ArgMax gm{-INFINITY, -1};
                    for (int cc = 0; cc < P.NC; ++cc) {
                        const ChunkStat s = ldcg(&N->stat[0][cc]);
                        gm = argmax_merge(gm, ArgMax{s.m, s.otop});
                    }
                    VerifyUnitRecord rr;
                    const bool hit = j < P.D && dvalid && dj == gm.i;
                    rr.flags = hit ? 1 : 0;
                    rr.token = gm.i;
                    rr.pt = hit ? 1.0f : 0.0f;
                    rr.pd = (j < P.D && dvalid) ? 1.0f : 0.0f;
                    P.rec[ui] = rr;
                    Z->c1 = 0u;   // release the slot
                    __threadfence();
                    st_rel(&Z->gen, gen + 1u);
                }
            }
            __syncthreads();
            continue;
        }

        // ---- pass 1 per staged row: maximum (and the top-k bound), then the weights' sum
        for (int r = 0; r < nrows; ++r) {
            const uint4 *vp = reinterpret_cast<const uint4 *>(buf[r]);
            float m = -INFINITY;
            for (int v = tid; v < nvec[r]; v += NT) {
                float x[EPV];
                unpack(vp[v], x);
#pragma unroll
                for (int k = 0; k < EPV; ++k) m = fmaxf(m, x[k]);
            }
            const float tm = m;
            m = block_max(m, ms);
            float kb = -INFINITY;
            if (use_k && kk <= NT) {
                // the kk-th largest thread maximum: a lower bound of the row's kk-th largest
                tmax[tid] = tm;
                __syncthreads();
                int gt = 0, ge = 0;
                for (int i = 0; i < NT; ++i) {
                    const float y = tmax[i];
                    gt += y > tm;
                    ge += y >= tm;
                }
                if (tid == 0) ms.kb[r] = -INFINITY;
                __syncthreads();
                if (gt < kk && kk <= ge) ms.kb[r] = tm;
                __syncthreads();
                kb = ms.kb[r];
            }
            const float xref = ms.xref[r];
            int32_t otop = INT32_MIN;
            float otf = 0.0f;
            if (m > -INFINITY) {
                const float Pv = __fmul_rn(m - xref, c2);
                if (!(fabsf(Pv) < PMAX)) kb = __int_as_float(0x7FC00000);   // NaN: exact path
                else {
                    otf = floorf(__fadd_rn(Pv, 0.0009765625f));
                    otop = static_cast<int32_t>(otf);
                }
            }
            float zs = 0.0f;
            if (otop != INT32_MIN) {
                for (int v = tid; v < nvec[r]; v += NT) {
                    float x[EPV];
                    unpack(vp[v], x);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) zs += ex2f(fmaf(x[k] - xref, c2, -otf));
                }
            }
            zs = block_sum(zs, ms);
            if (tid == 0) {
                if (alive) N->stat[r][c] = ChunkStat{m, otop, zs, kb};
                ms.otop[r] = otop;
                if (alive && dvalid && static_cast<int64_t>(dj) >= e0 && static_cast<int64_t>(dj) < e0 + n)
                    Z->xd[r] = widen(buf[r][padE[r] + (dj - e0)]);
            }
        }

        // ---- W1
        __syncthreads();
        if (tid == 0 && alive) {
            __threadfence();
            atom_add_ar(&Z->c1, 1u);
            if (!wait_geq(&Z->c1, static_cast<uint32_t>(P.NC), P)) ms.leave = 1;
        }
        __syncthreads();
        alive = !ms.leave;
        if (!alive) continue;

        // ---- plan A (warp r plans row r)
        if (warp < nrows) plan_a(P, N, warp, ms.xref[warp], c2, kk, pp, ms.plan[warp]);
        __syncthreads();
        bool fallback = false;
        for (int r = 0; r < nrows; ++r) fallback |= ms.plan[r].fallback != 0;
        // the unit may have to draw unless an earlier position of its row is known rejected
        if (tid == 0) {
            const uint32_t rf = ld_acq(P.rowflag + b);
            ms.cstar = (kind == KIND_SAMPLE) ? (rf > static_cast<uint32_t>(P.D + 1 - j)) : (rf > 0u);
        }
        __syncthreads();
        const bool want_draw = !ms.cstar && !fallback;

        if (!filtered && !fallback) {
            // ---- unfiltered: this chunk's residual and p sums for a possible draw
            unsigned long long rs = 0, ps = 0;
            if (want_draw) {
                DrawCtx g;
                g.kind = kind;
                g.dj = dj;
                g.dvalid = dvalid;
                g.one_hot = nrows == 1 && kind == KIND_SAMPLE;
                g.c2 = c2;
                g.rows = nrows;
                for (int r = 0; r < 2; ++r) {
                    const RowPlan &pl = ms.plan[r < nrows ? r : 0];
                    g.xr[r] = pl.xref;
                    g.ot[r] = static_cast<float>(pl.otop);
                    g.iz[r] = FSF / __ull2float_rn(pl.Z);
                    g.th[r] = 0u;
                    g.pm[r] = pl.pm;
                }
                const uint4 *vp = reinterpret_cast<const uint4 *>(buf[0]);
                for (int v = tid; v < nvec[0]; v += NT) {
                    float x[EPV];
                    unpack(vp[v], x);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) {
                        const int e = v * EPV + k - padE[0];
                        if (e >= 0 && e < n) {
                            const float xq = nrows == 2 ? widen(buf[1][padE[1] + e]) : 0.0f;
                            unsigned long long rf, pf;
                            draw_weights(g, e0 + e, x[k], xq, rf, pf);
                            rs += rf;
                            ps += pf;
                        }
                    }
                }
            }
            block_sum2(rs, ps, ms);
            if (tid == 0) {
                N->pub[c].r = rs;
                N->pub[c].p = ps;
            }
        }

        if (filtered && !fallback) {
            // ---- pass 2: histogram of the loose logits
            for (int r = 0; r < nrows; ++r) {
                const RowPlan &pl = ms.plan[r];
                const int32_t otop = ms.otop[r];
                if (pl.pm || otop == INT32_MIN) continue;
                const float xref = pl.xref, xcut = pl.xcut, otf = static_cast<float>(otop);
                const uint4 *vp = reinterpret_cast<const uint4 *>(buf[r]);
                const int nv = nvec[r];
                for (int v = tid; v < nv; v += 2 * NT) {
                    float x[2 * EPV];
                    unpack(vp[v], *reinterpret_cast<float(*)[EPV]>(x));
                    if (v + NT < nv) unpack(vp[v + NT], *reinterpret_cast<float(*)[EPV]>(x + EPV));
                    else {
#pragma unroll
                        for (int k = 0; k < EPV; ++k) x[EPV + k] = -INFINITY;
                    }
#pragma unroll
                    for (int k = 0; k < 2 * EPV; ++k) {
                        if (x[k] >= xcut) {
                            const uint32_t bits = __float_as_uint(ex2f(fmaf(x[k] - xref, c2, -otf)));
                            const uint32_t dep = depth_of(bits);
                            if (dep < static_cast<uint32_t>(NBL)) {
                                atomicAdd(&hm[dep], mant24(bits) >> QSH);
                                if (use_k) atomicAdd(&hc[dep], 1u);
                            }
                        }
                    }
                }
                __syncthreads();
                // publish: coarse sums per local octave, then the fine bins; clear the histogram
                if (tid <= ZL) {
                    unsigned long long msum = 0, csum = 0;
                    for (int qq = 0; qq < RB; ++qq) {
                        msum += hm[tid * RB + qq];
                        csum += hc[tid * RB + qq];
                    }
                    if (msum) {
                        const int slot = (((otop - tid) % NO) + NO) % NO;
                        red_add_u64(&Z->coarse_mass[r][slot], msum);
                        if (use_k) red_add_u32(&Z->coarse_cnt[r][slot], static_cast<uint32_t>(csum));
                    }
                }
                __syncthreads();
                for (int i = tid; i < NBL; i += NT) {
                    const uint32_t mv = hm[i];
                    if (mv) {
                        const int slot = (((otop - i / RB) % NO) + NO) % NO;
                        red_add_u64(&Z->ring_mass[r][slot * RB + i % RB], mv);
                        if (use_k) red_add_u32(&Z->ring_cnt[r][slot * RB + i % RB], hc[i]);
                        hm[i] = 0u;
                        hc[i] = 0u;
                    }
                }
                __syncthreads();
            }
            // ---- W1b
            if (tid == 0) {
                __threadfence();
                atom_add_ar(&Z->c1b, 1u);
                if (!wait_geq(&Z->c1b, static_cast<uint32_t>(P.NC), P)) ms.leave = 1;
            }
            __syncthreads();
            if (ms.leave) continue;
            // ---- plan B (the whole CTA)
            plan_b_block(Z, nrows, kk, pp, P.V, ms);
            for (int r = 0; r < nrows; ++r) fallback |= ms.plan[r].fallback != 0;
        }

        if (filtered && !fallback) {
            // ---- gather: exact sums above the boundary bins, the candidates, and the nucleus
            // list.  Warp w sweeps a contiguous range of the chunk's vectors (lanes on
            // consecutive vectors), so its nucleus entries come out in id order and go to its
            // own part of the chunk's segment.
            const int sseg = P.seg / NW;
            uint32_t nuc_w = 0;
            bool nuc_over = false;
            for (int r = 0; r < nrows; ++r) {
                const RowPlan &pl = ms.plan[r];
                const int32_t otop = ms.otop[r];
                unsigned long long above = 0, mid = 0;
                const bool want_nuc = (r == 0) && want_draw;
                if (!pl.pm && otop != INT32_MIN && pl.dmax >= (pl.otop - otop) * RB) {
                    const int sh = (pl.otop - otop) * RB;   // row depth = local depth + sh
                    if (tid == 0) {
                        float wlo, whi;
                        bin_edges(min(pl.dmax - sh, NBL - 1), wlo, whi);
                        ms.xlo[r] = pl.xref + (static_cast<float>(otop) + log2f(wlo) - 0.00390625f) / c2;
                        ms.ncc = 0u;
                    }
                    __syncthreads();
                    const float xlo = ms.xlo[r], xref = pl.xref, otf = static_cast<float>(otop);
                    const float scale = ldexpf(1.0f, otop - pl.otop + FSH);
                    float fa = 0.0f, fm = 0.0f;
                    const uint4 *vp = reinterpret_cast<const uint4 *>(buf[r]);
                    const int nv = nvec[r];
                    const int per = (nv + NW - 1) / NW;
                    const int v0 = warp * per, v1 = min(nv, v0 + per);
                    NucEntry *wseg = nucs + static_cast<size_t>(c) * P.seg + static_cast<size_t>(warp) * sseg;
                    for (int vb = v0; vb < v1; vb += 32) {
                        const int v = vb + lane;
                        float x[EPV];
                        if (v < v1) unpack(vp[v], x);
                        else {
#pragma unroll
                            for (int k = 0; k < EPV; ++k) x[k] = -INFINITY;
                        }
                        uint32_t mine = 0u;   // bit k: element k joins the nucleus list
#pragma unroll
                        for (int k = 0; k < EPV; ++k) {
                            const int e = v * EPV + k - padE[r];
                            if (x[k] >= xlo && e >= 0 && e < n) {
                                const float w = ex2f(fmaf(x[k] - xref, c2, -otf));
                                const uint32_t bits = __float_as_uint(w);
                                const int dep = static_cast<int>(depth_of(bits)) + sh;
                                if (dep < pl.dabove) {
                                    fa += w;
                                } else {
                                    const bool cand = (pl.dlo >= 0 && dep >= pl.dlo && dep <= pl.dhi) || dep == pl.dk;
                                    if (cand) {
                                        const uint32_t sl = atomicAdd(&ms.ncc, 1u);
                                        if (sl < static_cast<uint32_t>(CCAP))
                                            ccand[sl] = (static_cast<unsigned long long>(order_key(x[k])) << 32) |
                                                        (static_cast<uint32_t>(dep / RB) << 24) | mant24(bits);
                                    } else if (dep < pl.dk) {
                                        fm += w;
                                    }
                                }
                                if (want_nuc && dep <= pl.dmax) mine |= 1u << k;
                            }
                        }
                        if (want_nuc && __any_sync(0xFFFFFFFFu, mine != 0u)) {
                            // this iteration's entries in id order: a warp prefix of the counts
                            const uint32_t cnt = __popc(mine);
                            uint32_t inc = cnt;
                            for (int o = 1; o < 32; o <<= 1) {
                                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                                if (lane >= o) inc += y;
                            }
                            uint32_t pos = nuc_w + inc - cnt;
#pragma unroll
                            for (int k = 0; k < EPV; ++k) {
                                if (mine & (1u << k)) {
                                    const int e = v * EPV + k - padE[r];
                                    if (pos < static_cast<uint32_t>(sseg)) {
                                        NucEntry ne;
                                        ne.id = static_cast<int32_t>(e0 + e);
                                        ne.xt = x[k];
                                        ne.xq = nrows == 2 ? widen(buf[1][padE[1] + e]) : 0.0f;
                                        wseg[pos] = ne;
                                    }
                                    ++pos;
                                }
                            }
                            nuc_w += __shfl_sync(0xFFFFFFFFu, inc, 31);
                        }
                    }
                    above = __float2ull_rn(fa * scale);
                    mid = __float2ull_rn(fm * scale);
                    // the chunk's candidates go to the unit's list in one reservation (more
                    // than the shared list holds: reserve past the capacity, so that the
                    // resolver sees the overflow)
                    __syncthreads();
                    const uint32_t ncc = ms.ncc;
                    if (tid == 0 && ncc) ms.cbase = atomicAdd(&Z->ncand[r], ncc > static_cast<uint32_t>(CCAP) ? static_cast<uint32_t>(CAP + 1) : ncc);
                    __syncthreads();
                    if (ncc) {
                        const uint32_t base = ms.cbase;
                        for (uint32_t i = tid; i < ncc && i < static_cast<uint32_t>(CCAP); i += NT)
                            if (base + i < static_cast<uint32_t>(CAP)) N->cand[r][base + i] = ccand[i];
                    }
                }
                // fixed-order block sums
                for (int o = 16; o > 0; o >>= 1) {
                    above += __shfl_xor_sync(0xFFFFFFFFu, above, o);
                    mid += __shfl_xor_sync(0xFFFFFFFFu, mid, o);
                }
                __syncthreads();
                if (lane == 0) {
                    ms.dred[warp][0] = above;
                    ms.dred[warp][1] = mid;
                }
                __syncthreads();
                if (tid == 0) {
                    unsigned long long a2 = 0, mm = 0;
                    for (int w = 0; w < NW; ++w) {
                        a2 += ms.dred[w][0];
                        mm += ms.dred[w][1];
                    }
                    N->pub[c].above[r] = a2;
                    N->pub[c].mid[r] = mm;
                }
                if (nuc_w > static_cast<uint32_t>(sseg)) nuc_over = true;
            }
            if (lane == 0) N->pub[c].nucw[warp] = want_draw ? (nuc_over ? 0xFFFFFFFFu : nuc_w) : 0u;
        }

        // ---- W2: every chunk arrives; the last one resolves the unit
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const uint32_t old = atom_add_ar(&Z->c2, 1u);
            ms.resolver = (old == static_cast<uint32_t>(P.NC - 1)) ? 1 : 0;
        }
        __syncthreads();
        if (ms.resolver) {
            if (tid == 0) atomicAdd(P.hdr + (fallback ? 2 : 5), 1u);
            unsigned long long *sbuf = reinterpret_cast<unsigned long long *>(buf[0]);
            bool good = !fallback;
            DrawCtx g;
            g.kind = kind;
            g.dj = dj;
            g.dvalid = dvalid;
            g.one_hot = nrows == 1 && kind == KIND_SAMPLE;
            g.c2 = c2;
            g.rows = nrows;
            uint32_t th[2] = {0u, 0u};
            unsigned long long zk[2] = {1ull << FSH, 1ull << FSH};
            if (good) {
                for (int r = 0; r < nrows && good; ++r) {
                    const RowPlan pl = ms.plan[r];
                    if (pl.pm) {
                        th[r] = 0u;
                        zk[r] = 1ull << FSH;
                    } else if (!filtered) {
                        th[r] = 0u;
                        zk[r] = pl.Z;
                    } else if (!resolve_row(Z, N, r, pl, P.NC, kk, pp, P.V, sbuf, ms, th[r], zk[r])) {
                        good = false;
                    }
                }
                if (good && filtered && want_draw && kind != KIND_GREEDY) {
                    // (every thread reads the same published counts)
                    for (int cc = 0; cc < P.NC && good; ++cc)
                        for (int w = 0; w < NW; ++w)
                            if (__ldcg(&N->pub[cc].nucw[w]) == 0xFFFFFFFFu) good = false;
                }
            }
            if (!good) {
                if (tid == 0 && !fallback) atomicAdd(P.hdr + 3, 1u);
                slow_unit<T>(P, kind, b, j, dj, dvalid, c2, kk, pp, rowp[0],
                             nrows == 2 ? rowp[1] : nullptr, reinterpret_cast<unsigned long long *>(scr),
                             reinterpret_cast<unsigned long long *>(buf[1]), ms);
            } else {
                for (int r = 0; r < 2; ++r) {
                    const RowPlan &pl = ms.plan[r < nrows ? r : 0];
                    g.xr[r] = pl.xref;
                    g.ot[r] = static_cast<float>(pl.otop);
                    g.iz[r] = FSF / __ull2float_rn(zk[r < nrows ? r : 0]);
                    g.th[r] = th[r < nrows ? r : 0];
                    g.pm[r] = pl.pm;
                }
                float ua, us;
                unit_uniforms(P.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(j), ua, us);
                if (tid == 0) {
                    VerifyUnitRecord rr;
                    rr.token = -1;
                    bool draw;
                    if (kind == KIND_SAMPLE) {
                        bool acc = false;
                        float ptd = 0.0f, pdd = 0.0f;
                        if (dvalid) {
                            const RowPlan &p0 = ms.plan[0];
                            const float xt = ldcg(&Z->xd[0]);
                            const bool kt = p0.pm ? (dj == 0) : (order_key(xt) >= th[0]);
                            const float et = fmaf(xt - p0.xref, c2, -static_cast<float>(p0.otop));
                            ptd = p0.pm ? (dj == 0 ? 1.0f : 0.0f) : (kt ? ex2f(et) * g.iz[0] : 0.0f);
                            bool kq = true;
                            float eq = 0.0f;
                            pdd = 1.0f;
                            if (nrows == 2) {
                                const RowPlan &p1 = ms.plan[1];
                                const float xq = ldcg(&Z->xd[1]);
                                kq = p1.pm ? (dj == 0) : (order_key(xq) >= th[1]);
                                eq = fmaf(xq - p1.xref, c2, -static_cast<float>(p1.otop));
                                pdd = p1.pm ? (dj == 0 ? 1.0f : 0.0f) : (kq ? ex2f(eq) * g.iz[1] : 0.0f);
                            }
                            if (!kt) acc = false;
                            else if (!kq) acc = true;
                            else {
                                float ratio;
                                if (nrows == 1 || p0.pm || ms.plan[1].pm) ratio = ptd / pdd;
                                else ratio = ex2f(et - eq) * (__ull2float_rn(zk[1]) / __ull2float_rn(zk[0]));
                                acc = ua <= ratio;
                            }
                        }
                        rr.flags = acc ? 1 : 0;
                        rr.pt = ptd;
                        rr.pd = pdd;
                        if (!acc) atomicMax(P.rowflag + b, static_cast<uint32_t>(P.D + 1 - j));
                        const uint32_t rf = ld_acq(P.rowflag + b);
                        draw = !acc && !(rf > static_cast<uint32_t>(P.D + 1 - j));
                    } else {
                        rr.flags = 0;
                        rr.pt = rr.pd = 0.0f;
                        draw = ld_acq(P.rowflag + b) == 0u;
                    }
                    // a draw needs the chunks' draw data, published only when no chunk knew of
                    // an earlier rejection; a chunk that knew it, knew that no draw is needed
                    P.rec[ui] = rr;
                    ms.cstar = (draw && want_draw) ? 1 : 0;
                    if (draw) atomicAdd(P.hdr + 4, 1u);
                }
                __syncthreads();
                if (ms.cstar) {
                    int32_t tok;
                    if (g.pm[0]) tok = 0;
                    else if (filtered) tok = draw_nucleus(P, N, nucs, g, us, reinterpret_cast<unsigned long long *>(buf[0]), ms);
                    else tok = draw_unfiltered<T>(P, N, g, us, rowp[0], nrows == 2 ? rowp[1] : nullptr, ms);
                    if (tid == 0) P.rec[ui].token = tok;
                }
            }
            // every chunk has planned (all arrived at W2): clear the histograms for the
            // slot's next unit, and the staging scratch the resolution used
            if (filtered) {
                unsigned long long *rm = &Z->ring_mass[0][0];
                for (int i = tid; i < 2 * NBR; i += NT) rm[i] = 0ull;
                unsigned long long *cm = &Z->coarse_mass[0][0];
                for (int i = tid; i < 2 * NO; i += NT) cm[i] = 0ull;
                if (use_k) {
                    uint32_t *rc = &Z->ring_cnt[0][0];
                    for (int i = tid; i < 2 * NBR; i += NT) rc[i] = 0u;
                    uint32_t *ccn = &Z->coarse_cnt[0][0];
                    for (int i = tid; i < 2 * NO; i += NT) ccn[i] = 0u;
                }
            }
            for (int i = tid; i < 2 * NBL; i += NT) hm[i] = 0u;
        }

        // ---- done with the unit: the last chunk releases the slot
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const uint32_t old = atom_add_ar(&Z->done, 1u);
            if (old == static_cast<uint32_t>(P.NC - 1)) {
                Z->c1 = Z->c1b = Z->c2 = Z->done = 0u;
                Z->ncand[0] = Z->ncand[1] = 0u;
                __threadfence();
                st_rel(&Z->gen, gen + 1u);
            }
        }
        __syncthreads();
    }
}

}  // namespace vc

// ---------------------------------------------------------------- host side

// Slots of a call, and nucleus entries per slot (half the vocabulary, within limits).
static int64_t vc_nslot(int64_t B, int32_t D) {
    const int64_t units = B * (D + 1);
    return units < vc::NSLOT ? (units > 0 ? units : 1) : vc::NSLOT;
}
static int64_t vc_nuc_slot(int64_t V) {
    int64_t n = V / 3;
    if (n < 8192) n = 8192;
    if (n > 65536) n = 65536;
    return n;
}

size_t verify_chunks_workspace_bytes(int64_t B, int32_t D, int64_t V) {
    const size_t rows = (static_cast<size_t>(B) * 4 + 255) & ~static_cast<size_t>(255);
    const size_t rec = static_cast<size_t>(B) * static_cast<size_t>(D + 1) * sizeof(VerifyUnitRecord);
    const size_t ns = static_cast<size_t>(vc_nslot(B, D));
    const size_t nuc = (static_cast<size_t>(vc_nuc_slot(V)) * sizeof(vc::NucEntry) + 255) & ~static_cast<size_t>(255);
    return 256 + rows + ns * (vc::ZSZ + vc::NSZ + nuc) + rec;
}

bool verify_chunks_fits(int64_t V, size_t es) {
    // chunks per unit at most NCMAX of at most ROW_BYTES per row
    const int64_t ch = vc::ROW_BYTES / static_cast<int64_t>(es);
    return V >= 1 && (V + ch - 1) / ch <= vc::NCMAX;
}

template <typename T>
static int vc_resident_ctas(size_t smem) {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int per = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, vc::k_verify_chunks<T>, vc::NT, smem) != cudaSuccess || per < 1)
        per = 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
    const int n = per * sms;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

static AttrCache g_vc_attr[2];

template <typename T>
static cudaError_t launch_chunks(const VerifySampleArgs &a, cudaStream_t stream) {
    constexpr size_t ES = sizeof(T);
    const size_t smem = 2 * vc::ROWB + vc::SCR_BYTES + sizeof(vc::Misc);
    cudaError_t e = ensure_attr(vc::k_verify_chunks<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem), g_vc_attr[ES == 4 ? 0 : 1]);
    if (e != cudaSuccess) return e;
    const int G = vc_resident_ctas<T>(smem);
    const int64_t units = a.B * (a.D + 1);
    // chunk size: as large as a staged row allows, smaller when the call has too few units
    // to give every resident CTA a chunk (a multiple of 64 ids, at least 1024)
    int64_t ch = vc::ROW_BYTES / static_cast<int64_t>(ES);
    if (units * ((a.V + ch - 1) / ch) < G) {
        int64_t want_nc = (G + units - 1) / units;
        if (want_nc > vc::NCMAX) want_nc = vc::NCMAX;
        int64_t c2 = (a.V + want_nc - 1) / want_nc;
        c2 = ((c2 + 63) / 64) * 64;
        ch = c2 < ch ? c2 : ch;
        if (ch < 1024) ch = 1024;
    }
    const int64_t nc = (a.V + ch - 1) / ch;
    if (nc > vc::NCMAX) return cudaErrorInvalidValue;
    vc::Params P;
    P.T = a.target;
    P.Q = a.draft;
    P.d = a.draft_ids;
    P.tau = a.temperature;
    P.topk = a.top_k;
    P.topp = a.top_p;
    P.seed = a.seed;
    P.B = a.B;
    P.V = a.V;
    P.CH = ch;
    P.D = a.D;
    P.NC = static_cast<int32_t>(nc);
    const int64_t ns = vc_nslot(a.B, a.D);
    P.nslot = static_cast<int32_t>(ns);
    P.nuc_slot = vc_nuc_slot(a.V);
    P.seg = static_cast<int32_t>(P.nuc_slot / nc);
    P.items = units * nc;
    unsigned char *ws = static_cast<unsigned char *>(a.workspace);
    const size_t rows = (static_cast<size_t>(a.B) * 4 + 255) & ~static_cast<size_t>(255);
    const size_t nucb = (static_cast<size_t>(P.nuc_slot) * sizeof(vc::NucEntry) + 255) & ~static_cast<size_t>(255);
    P.hdr = reinterpret_cast<uint32_t *>(ws);
    P.rowflag = reinterpret_cast<uint32_t *>(ws + 256);
    P.zone_z = ws + 256 + rows;
    P.zone_n = P.zone_z + ns * vc::ZSZ;
    P.nuc = reinterpret_cast<vc::NucEntry *>(P.zone_n + ns * vc::NSZ);
    P.rec = reinterpret_cast<VerifyUnitRecord *>(reinterpret_cast<unsigned char *>(P.nuc) + ns * nucb);
    P.status = a.status;
    e = cudaMemsetAsync(ws, 0, 256 + rows + static_cast<size_t>(ns) * vc::ZSZ, stream);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(P.items < G ? P.items : G);
    vc::k_verify_chunks<T><<<grid, vc::NT, smem, stream>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    return launch_verify_finalize(P.rec, a, stream);
}

cudaError_t run_wait_selftest_chunks(uint32_t limit, int32_t *status, cudaStream_t stream) {
    vc::k_wait_selftest<<<1, 32, 0, stream>>>(limit, status);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_verify_chunks(const VerifySampleArgs &a, cudaStream_t stream) {
    return a.dtype == MTPSPEC_F32 ? launch_chunks<float>(a, stream) : launch_chunks<uint16_t>(a, stream);
}

}  // namespace mtpspec
