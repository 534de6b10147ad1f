// Shared device helpers of libmtpspec: element loads, order-preserving keys, and the
// thread-block-cluster primitives (cluster rank, barrier, distributed shared memory).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/libmtpspec.h"

namespace mtpspec {

// ---------------------------------------------------------------- element types

// Logits are float32 or bfloat16 stored as 16-bit patterns; both widen exactly to fp32.
__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

template <typename T> struct elems_per_16B;
template <> struct elems_per_16B<float> { static constexpr int value = 4; };
template <> struct elems_per_16B<uint16_t> { static constexpr int value = 8; };

// Unpack one 16-byte vector into fp32 values.
__device__ __forceinline__ void unpack(const uint4 &v, float (&out)[4]) {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4 &v, float (&out)[8]) {
    out[0] = __uint_as_float(v.x << 16);
    out[1] = __uint_as_float(v.x & 0xFFFF0000u);
    out[2] = __uint_as_float(v.y << 16);
    out[3] = __uint_as_float(v.y & 0xFFFF0000u);
    out[4] = __uint_as_float(v.z << 16);
    out[5] = __uint_as_float(v.z & 0xFFFF0000u);
    out[6] = __uint_as_float(v.w << 16);
    out[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Streaming 16-byte load of data read exactly once (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream_16B(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Order-preserving 32-bit key of a float: a < b  <=>  key(a) < key(b), with -0 folded
// onto +0 so that equal floats have equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// (value, index) argmax candidate with the lowest-index tie rule; index < 0 means empty.
struct ArgMax {
    float v;
    int32_t i;
};
__device__ __forceinline__ ArgMax argmax_merge(ArgMax a, ArgMax b) {
    if (b.i < 0) return a;
    if (a.i < 0) return b;
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}
__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax b;
        b.v = __shfl_xor_sync(0xFFFFFFFFu, a.v, o);
        b.i = __shfl_xor_sync(0xFFFFFFFFu, a.i, o);
        a = argmax_merge(a, b);
    }
    return a;
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Full cluster barrier with release/acquire semantics on shared::cluster memory; every
// thread of every CTA in the cluster must call it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_peer_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ int32_t ld_peer_s32(uint32_t a) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_peer_u64(uint32_t a) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_peer_u32(uint32_t a, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_peer_f32(uint32_t a, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer_u64(uint32_t a, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_peer_add_u32(uint32_t a, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v)
                 : "memory");
    return old;
}

// Programmatic dependent launch: let the next kernel on the stream start its prologue,
// and wait for the previous kernel's memory to be visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// The launch attribute that makes a kernel the programmatic dependent of the previous
// kernel on the stream (it must call pdl_wait_primary before it touches that kernel's
// data or anything the earlier work may still use).
inline cudaLaunchAttribute *pdl_attr() {
    static cudaLaunchAttribute a = [] {
        cudaLaunchAttribute x = {};
        x.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        x.val.programmaticStreamSerializationAllowed = 1;
        return x;
    }();
    return &a;
}

}  // namespace mtpspec
