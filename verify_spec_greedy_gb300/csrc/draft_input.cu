// The MTP draft head's input stage: y = eh_proj_w @ [enorm(emb_next); hnorm(hidden)]
// ("14. MTP: speculative decoding with the built-in draft head", "The draft head":
// fc(cat(norm(e_{t+1}), norm(h_t))) with fc = Linear(2H, H, bias=False); "MPT (MTP,
// Multi-Token Prediction) 原理详解" section 二.2 steps 2-3: enorm, hnorm, concat with the
// embedding first, eh_proj).  RMSNorm: v / sqrt(mean(v^2) + eps) * w, rounded to bf16.
//
// Two paths, chosen by the token count M:
//  - M <= 4: one fused kernel.  Each CTA starts its first rows of the weight towards L2,
//    normalises the M tokens into shared memory (bf16, 2H values each), then its warps
//    stream the rows once from HBM with 16-byte loads and reduce the M dot products per
//    row.  HBM-bound on the weight.
//  - larger M: a normalisation pass writes the bf16 activations [M, 2H] to the workspace
//    (and zeroes the GEMM's counters), then the persistent tcgen05 GEMM (tcgen05_gemm.cu)
//    computes the projection on the tensor cores.  The GEMM is launched as the pass's
//    programmatic dependent: its CTAs start, and start streaming the weight, while the
//    pass runs, and read the activations once it has completed.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace mtpspec {
namespace di {

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;
constexpr int GEMV_UNROLL = 8;   // 16-byte loads in flight per lane

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&b);
}

// Sum over the block; every thread gets the result.
template <int NTH>
__device__ __forceinline__ float block_sum(float v, float *scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < NTH / 32; ++w) t += scratch[w];
    return t;
}

// out[i] = bf16(v[i] * r * w[i]) for one H-vector, r = 1/sqrt(mean(v^2) + eps).  All
// threads of the block call it.  H % 8 == 0 and 16-byte aligned vectors.
template <int NTH>
__device__ __forceinline__ void rmsnorm_row(const uint16_t *__restrict__ v,
                                            const uint16_t *__restrict__ w, int H, float eps,
                                            uint16_t *out, float *scratch) {
    const uint4 *vv = reinterpret_cast<const uint4 *>(v);
    const int nv = H / 8;
    float ss = 0.0f;
    for (int i = threadIdx.x; i < nv; i += NTH) {
        const uint4 q = vv[i];
        const uint32_t a[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float x0 = bf16_lo(a[t]), x1 = bf16_hi(a[t]);
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
        }
    }
    ss = block_sum<NTH>(ss, scratch);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
    const uint4 *ww = reinterpret_cast<const uint4 *>(w);
    uint4 *oo = reinterpret_cast<uint4 *>(out);
    for (int i = threadIdx.x; i < nv; i += NTH) {
        const uint4 q = vv[i], g = ww[i];
        const uint32_t a[4] = {q.x, q.y, q.z, q.w}, b[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint16_t lo = f32_to_bf16_bits(bf16_lo(a[t]) * r * bf16_lo(b[t]));
            const uint16_t hi = f32_to_bf16_bits(bf16_hi(a[t]) * r * bf16_hi(b[t]));
            o[t] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        oo[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Fused norm + GEMV for MT tokens: blockIdx.x owns output rows
// [blockIdx.x * rows_per_cta, ...), one warp per row at a time.
template <int MT>
__global__ void __launch_bounds__(GEMV_THREADS)
k_draft_gemv(const uint16_t *__restrict__ e, const uint16_t *__restrict__ h,
             const uint16_t *__restrict__ we, const uint16_t *__restrict__ wh,
             const uint16_t *__restrict__ W, uint16_t *__restrict__ y, int H, float eps,
             int rows_per_cta) {
    extern __shared__ __align__(16) uint16_t xs[];  // [MT][2H] normalised activations
    __shared__ float scratch[GEMV_WARPS];
    const int K = 2 * H;
    const int r0 = blockIdx.x * rows_per_cta;
    const int r1 = min(H, r0 + rows_per_cta);
    pdl_launch_dependents();  // a programmatic dependent may start its own prologue
    if (threadIdx.x == 0 && r1 > r0) {
        // the first 64 KB of this CTA's rows (contiguous) on their way to L2 during the wait
        // for the previous kernel and the norm
        const size_t slab = static_cast<size_t>(r1 - r0) * K * 2;
        const uint32_t n = static_cast<uint32_t>(slab < 65536 ? slab : 65536);  // K * 2 % 16 == 0
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W + static_cast<size_t>(r0) * K),
                     "r"(n)
                     : "memory");
    }
    // launched as a programmatic dependent: the tokens (and the output buffer) belong to
    // the previous kernel on the stream until it has completed
    pdl_wait_primary();
    for (int t = 0; t < MT; ++t) {
        rmsnorm_row<GEMV_THREADS>(e + static_cast<size_t>(t) * H, we, H, eps, xs + t * K, scratch);
        rmsnorm_row<GEMV_THREADS>(h + static_cast<size_t>(t) * H, wh, H, eps, xs + t * K + H,
                                  scratch);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nv = K / 8;  // 16-byte vectors per weight row
    for (int o = r0 + warp; o < r1; o += GEMV_WARPS) {
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + static_cast<size_t>(o) * K);
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
        for (int v0 = lane; v0 < nv; v0 += 32 * GEMV_UNROLL) {
            uint4 q[GEMV_UNROLL];
#pragma unroll
            for (int u = 0; u < GEMV_UNROLL; ++u) {
                const int vi = v0 + u * 32;
                if (vi < nv) q[u] = ld_stream_16B(wr + vi);
            }
#pragma unroll
            for (int u = 0; u < GEMV_UNROLL; ++u) {
                const int vi = v0 + u * 32;
                if (vi >= nv) continue;
                const uint32_t a[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint4 xv = reinterpret_cast<const uint4 *>(xs + t * K)[vi];
                    const uint32_t b[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc[t] = fmaf(bf16_lo(a[c]), bf16_lo(b[c]), acc[t]);
                        acc[t] = fmaf(bf16_hi(a[c]), bf16_hi(b[c]), acc[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float v = acc[t];
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, s);
            if (lane == 0) y[static_cast<size_t>(t) * H + o] = f32_to_bf16_bits(v);
        }
    }
}

// Normalisation pass of the tensor-core path for H <= 8192: one CTA per token, both halves
// at once, every value loaded once into registers (NV 16-byte vectors a thread per half).
// The sums of squares are formed in the same order as rmsnorm_row's.  CTA 0 also zeroes
// the GEMM's flag word and arrival counts (nzero words).
template <int NV>
__global__ void __launch_bounds__(256)
k_draft_norm_reg(const uint16_t *__restrict__ e, const uint16_t *__restrict__ h,
                 const uint16_t *__restrict__ we, const uint16_t *__restrict__ wh,
                 uint16_t *__restrict__ xn, int H, float eps, unsigned *__restrict__ zero,
                 int nzero) {
    __shared__ float2 scratch[8];
    pdl_launch_dependents();  // the GEMM may start its prologue and weight loads
    pdl_wait_primary();       // the tokens and the workspace belong to the previous kernel until then
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += 256) zero[i] = 0u;
    const size_t t = blockIdx.x;
    const int nv = H / 8;
    const uint4 *ev = reinterpret_cast<const uint4 *>(e + t * H);
    const uint4 *hv = reinterpret_cast<const uint4 *>(h + t * H);
    const uint4 *gw = reinterpret_cast<const uint4 *>(we);
    const uint4 *gh = reinterpret_cast<const uint4 *>(wh);
    uint4 a[NV], b[NV], ga[NV], gb[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = threadIdx.x + i * 256;
        if (k < nv) {
            a[i] = ev[k];
            b[i] = hv[k];
            ga[i] = gw[k];
            gb[i] = gh[k];
        }
    }
    float se = 0.0f, sh = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if (threadIdx.x + i * 256 >= nv) break;
        const uint32_t x[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
        const uint32_t z[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float v = bf16_lo(x[c]);
            se = fmaf(v, v, se);
            v = bf16_hi(x[c]);
            se = fmaf(v, v, se);
            v = bf16_lo(z[c]);
            sh = fmaf(v, v, sh);
            v = bf16_hi(z[c]);
            sh = fmaf(v, v, sh);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        se += __shfl_xor_sync(0xFFFFFFFFu, se, o);
        sh += __shfl_xor_sync(0xFFFFFFFFu, sh, o);
    }
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = make_float2(se, sh);
    __syncthreads();
    float te = 0.0f, th = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        te += scratch[w].x;
        th += scratch[w].y;
    }
    const float re = 1.0f / sqrtf(te / static_cast<float>(H) + eps);
    const float rh = 1.0f / sqrtf(th / static_cast<float>(H) + eps);
    uint4 *oe = reinterpret_cast<uint4 *>(xn + t * 2 * H);
    uint4 *oh = reinterpret_cast<uint4 *>(xn + t * 2 * H + H);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = threadIdx.x + i * 256;
        if (k >= nv) break;
        const uint32_t x[4] = {a[i].x, a[i].y, a[i].z, a[i].w}, gx[4] = {ga[i].x, ga[i].y, ga[i].z, ga[i].w};
        const uint32_t z[4] = {b[i].x, b[i].y, b[i].z, b[i].w}, gz[4] = {gb[i].x, gb[i].y, gb[i].z, gb[i].w};
        uint32_t u[4], v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            u[c] = static_cast<uint32_t>(f32_to_bf16_bits(bf16_lo(x[c]) * re * bf16_lo(gx[c]))) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(bf16_hi(x[c]) * re * bf16_hi(gx[c]))) << 16);
            v[c] = static_cast<uint32_t>(f32_to_bf16_bits(bf16_lo(z[c]) * rh * bf16_lo(gz[c]))) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(bf16_hi(z[c]) * rh * bf16_hi(gz[c]))) << 16);
        }
        oe[k] = make_uint4(u[0], u[1], u[2], u[3]);
        oh[k] = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

// Normalisation pass of the tensor-core path for larger H: one CTA per (token, half).  CTA 0
// also zeroes the GEMM's flag word and arrival counts (nzero words).
__global__ void __launch_bounds__(256)
k_draft_norm(const uint16_t *__restrict__ e, const uint16_t *__restrict__ h,
             const uint16_t *__restrict__ we, const uint16_t *__restrict__ wh,
             uint16_t *__restrict__ xn, int H, float eps, unsigned *__restrict__ zero, int nzero) {
    __shared__ float scratch[8];
    pdl_launch_dependents();  // the GEMM may start its prologue and weight loads
    pdl_wait_primary();       // the tokens and the workspace belong to the previous kernel until then
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += 256) zero[i] = 0u;
    const int t = blockIdx.x >> 1, half = blockIdx.x & 1;
    const uint16_t *v = (half ? h : e) + static_cast<size_t>(t) * H;
    rmsnorm_row<256>(v, half ? wh : we, H, eps, xn + static_cast<size_t>(t) * 2 * H + half * H,
                     scratch);
}

// The output layer's normalisation: one CTA per token.
__global__ void __launch_bounds__(256)
k_head_norm(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w,
            uint16_t *__restrict__ out, int H, float eps) {
    __shared__ float scratch[8];
    const size_t t = blockIdx.x;
    rmsnorm_row<256>(x + t * H, w, H, eps, out + t * H, scratch);
}

}  // namespace di

cudaError_t run_head_norm(const void *x, const void *w, void *out, int64_t M, int64_t H, float eps,
                          cudaStream_t stream) {
    di::k_head_norm<<<static_cast<unsigned>(M), 256, 0, stream>>>(
        static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(w),
        static_cast<uint16_t *>(out), static_cast<int>(H), eps);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

constexpr int kGemvMaxTokens = 4;

bool draft_input_uses_gemv(int64_t M, int64_t H) {
    (void)H;
    return M <= kGemvMaxTokens;
}

// Workspace of the tensor-core path: the GEMM's own (counters first), then the activations.
static size_t di_gemm_bytes(int64_t M, int64_t H) {
    return (gemm_workspace_bytes(M, H) + 1023) & ~static_cast<size_t>(1023);
}
size_t draft_input_workspace_bytes(int64_t M, int64_t H) {
    if (draft_input_uses_gemv(M, H)) return 0;
    const size_t xn = static_cast<size_t>(M) * static_cast<size_t>(2 * H) * 2;
    return di_gemm_bytes(M, H) + xn;
}

template <int MT>
static cudaError_t launch_gemv(const DraftInputArgs &a, cudaStream_t stream) {
    const int H = static_cast<int>(a.H);
    const size_t smem = static_cast<size_t>(MT) * 2 * H * 2;
    if (smem > 48 * 1024) {
        static AttrCache attr;
        cudaError_t e = ensure_attr(di::k_draft_gemv<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem), attr);
        if (e != cudaSuccess) return e;
    }
    // one CTA per SM, an equal share of the rows each (a warp per row at a time)
    const int rows = (H + 151) / 152;
    const int grid = (H + rows - 1) / rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(di::GEMV_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl_attr();
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, di::k_draft_gemv<MT>, static_cast<const uint16_t *>(a.e), static_cast<const uint16_t *>(a.h),
        static_cast<const uint16_t *>(a.we), static_cast<const uint16_t *>(a.wh),
        static_cast<const uint16_t *>(a.W), static_cast<uint16_t *>(a.y), H, a.eps, rows);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t run_draft_input(const DraftInputArgs &a, cudaStream_t stream) {
    if (draft_input_uses_gemv(a.M, a.H)) {
        switch (a.M) {
        case 1: return launch_gemv<1>(a, stream);
        case 2: return launch_gemv<2>(a, stream);
        case 3: return launch_gemv<3>(a, stream);
        default: return launch_gemv<4>(a, stream);
        }
    }
    void *gemm_ws = a.workspace;
    uint16_t *xn = reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(a.workspace) + di_gemm_bytes(a.M, a.H));
    const uint16_t *ve = static_cast<const uint16_t *>(a.e), *vh = static_cast<const uint16_t *>(a.h);
    const uint16_t *we = static_cast<const uint16_t *>(a.we), *wh = static_cast<const uint16_t *>(a.wh);
    const int H = static_cast<int>(a.H);
    unsigned *zero = static_cast<unsigned *>(gemm_ws);
    const int nzero = static_cast<int>(gemm_zero_bytes(a.M, a.H) / 4);
    const unsigned M = static_cast<unsigned>(a.M);
    // launched as the previous kernel's programmatic dependent (it waits before it reads)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = pdl_attr();
    cfg.numAttrs = 1;
    cudaError_t e;
    switch ((H / 8 + 255) / 256) {  // 16-byte vectors a thread per half
    case 1: e = cudaLaunchKernelEx(&cfg, di::k_draft_norm_reg<1>, ve, vh, we, wh, xn, H, a.eps, zero, nzero); break;
    case 2: e = cudaLaunchKernelEx(&cfg, di::k_draft_norm_reg<2>, ve, vh, we, wh, xn, H, a.eps, zero, nzero); break;
    case 3: e = cudaLaunchKernelEx(&cfg, di::k_draft_norm_reg<3>, ve, vh, we, wh, xn, H, a.eps, zero, nzero); break;
    case 4: e = cudaLaunchKernelEx(&cfg, di::k_draft_norm_reg<4>, ve, vh, we, wh, xn, H, a.eps, zero, nzero); break;
    default:
        cfg.gridDim = dim3(2 * M, 1, 1);
        e = cudaLaunchKernelEx(&cfg, di::k_draft_norm, ve, vh, we, wh, xn, H, a.eps, zero, nzero);
    }
    if (e != cudaSuccess) return e;
    count_launches(1);
    return run_gemm_bf16_nt(a.W, xn, a.y, a.H, a.M, 2 * a.H, gemm_ws, true, stream);
}

}  // namespace mtpspec
