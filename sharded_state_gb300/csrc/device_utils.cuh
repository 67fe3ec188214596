// device_utils.cuh -- small device helpers: bf16 <-> fp32 on packed words and
// 128-bit global loads/stores with cache hints.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace ss {

// Widen the two bf16 values packed in a 32-bit word (element 2j in the low
// half, 2j+1 in the high half); exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Round two floats to bf16 (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float a) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(a));
}

// Read-only streaming 128-bit load: not kept in L1, L2 fetch in 256-byte
// granules (each element is read once per launch).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 128-bit load of data this kernel later overwrites (not .nc).
__device__ __forceinline__ float4 ld_rw_f4(const float* p) {
    float4 r;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

// Ask L2 for the line holding p ahead of its load (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Asynchronous 16-byte copy global -> shared (cp.async, L2 only, 256-byte
// L2 fetch); smem is a shared-window address, both 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t smem, const void* g) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(smem), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most K of this thread's committed groups are still in flight.
template <int K>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}

// Streaming 128-bit stores (evict-first).
__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream_u4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// 16 bytes at an address that is only 2- (or 4-) byte aligned
// ---------------------------------------------------------------------------

// Bytes [sh, sh + 16) of the 32 bytes a:b (little-endian), sh even in 2..14.
__device__ __forceinline__ uint4 realign16(uint4 a, uint4 b, int sh) {
    const int bs = (sh & 3) * 8;  // 0 or 16
    uint4 o;
    switch (sh >> 2) {
        case 0:
            o.x = __funnelshift_r(a.x, a.y, bs); o.y = __funnelshift_r(a.y, a.z, bs);
            o.z = __funnelshift_r(a.z, a.w, bs); o.w = __funnelshift_r(a.w, b.x, bs);
            break;
        case 1:
            o.x = __funnelshift_r(a.y, a.z, bs); o.y = __funnelshift_r(a.z, a.w, bs);
            o.z = __funnelshift_r(a.w, b.x, bs); o.w = __funnelshift_r(b.x, b.y, bs);
            break;
        case 2:
            o.x = __funnelshift_r(a.z, a.w, bs); o.y = __funnelshift_r(a.w, b.x, bs);
            o.z = __funnelshift_r(b.x, b.y, bs); o.w = __funnelshift_r(b.y, b.z, bs);
            break;
        default:
            o.x = __funnelshift_r(a.w, b.x, bs); o.y = __funnelshift_r(b.x, b.y, bs);
            o.z = __funnelshift_r(b.y, b.z, bs); o.w = __funnelshift_r(b.z, b.w, bs);
            break;
    }
    return o;
}

// Read-only load of the 16 bytes at p (p even).  A misaligned p is served by
// the two aligned 16-byte blocks that cover [p, p + 16): each holds at least
// one of the requested bytes, so neither can lie on a page the caller does
// not own.
__device__ __forceinline__ uint4 ld_any16(const void* p) {
    const unsigned sh = (unsigned)(reinterpret_cast<uintptr_t>(p) & 15u);
    if (sh == 0) return ld_stream_u4(p);
    const unsigned char* base = static_cast<const unsigned char*>(p) - sh;
    return realign16(ld_stream_u4(base), ld_stream_u4(base + 16), (int)sh);
}

// Store 16 bytes at p (p even): one vector store when aligned, four 32-bit
// stores when 4-byte aligned, else 2 + 4 + 4 + 4 + 2 bytes.
__device__ __forceinline__ void st_any16(void* p, uint4 v) {
    const unsigned sh = (unsigned)(reinterpret_cast<uintptr_t>(p) & 15u);
    unsigned char* c = static_cast<unsigned char*>(p);
    if (sh == 0) {
        st_stream_u4(p, v);
    } else if ((sh & 3u) == 0) {
        uint32_t* w = reinterpret_cast<uint32_t*>(c);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
        *reinterpret_cast<uint16_t*>(c) = (uint16_t)(v.x & 0xFFFFu);
        uint32_t* w = reinterpret_cast<uint32_t*>(c + 2);
        w[0] = __funnelshift_r(v.x, v.y, 16);
        w[1] = __funnelshift_r(v.y, v.z, 16);
        w[2] = __funnelshift_r(v.z, v.w, 16);
        *reinterpret_cast<uint16_t*>(c + 14) = (uint16_t)(v.w >> 16);
    }
}

}  // namespace ss
