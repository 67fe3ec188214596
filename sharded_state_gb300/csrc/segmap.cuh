// segmap.cuh -- device helpers shared by the kernels that walk the packed
// index: the packed segment map lookup (which run of which parameter a packed
// element belongs to) and 16-byte stores to a per-parameter tensor at any
// 2-byte offset, assembled across neighbouring lanes.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "device_utils.cuh"
#include "internal.h"

namespace ss {

// The plan's packed segment map on the device.
struct SegMap {
    const PmEntry* __restrict__ pm;  // data segments by packed offset
    const int* __restrict__ pm_block;  // per kMapBlock block: last entry at or before it
    int M;                             // entries (where a kernel needs them)
};

// The map entry of packed element f in block B = f / kMapBlock, given the
// block's first candidate m = pm_block[B] and e = pm[m]: unless e's segment
// holds f, a binary search over the entries that start inside the block for
// the last one that starts at or before f (m stays pm_block[B] when none
// does: f lies before the first segment).  m and e are updated.
__device__ __forceinline__ void locate(const SegMap& mp, int64_t B, int64_t f, int& m, PmEntry& e) {
    if (f >= e.packed_off && f < e.packed_off + e.len) return;
    int hi = __ldg(mp.pm_block + B + 1);
    while (m < hi) {
        const int mid = (m + hi + 1) >> 1;
        if (mp.pm[mid].packed_off <= f)
            m = mid;
        else
            hi = mid - 1;
    }
    e = mp.pm[m];
}

// The map entry of packed element f (its index in m).
__device__ __forceinline__ PmEntry lookup(const SegMap& mp, int64_t f, int& m) {
    const int64_t B = f / kMapBlock;
    m = __ldg(mp.pm_block + B);
    PmEntry e = mp.pm[m];
    locate(mp, B, f, m, e);
    return e;
}

// Store bytes [lo, hi) of the 16-byte value v to blk + lo (blk 16-byte
// aligned, lo and hi even), two bytes at a time.
__device__ __forceinline__ void st_bytes(unsigned char* blk, uint4 v, int lo, int hi) {
#pragma unroll
    for (int b = 0; b < 16; b += 2) {
        if (b >= lo && b < hi) {
            const uint32_t w = b < 4 ? v.x : b < 8 ? v.y : b < 12 ? v.z : v.w;
            *reinterpret_cast<uint16_t*>(blk + b) = (uint16_t)(w >> ((b & 2) * 8));
        }
    }
}

// The 16 bytes p at ob, sh = ob mod 16 bytes past a boundary (ob even), where
// consecutive lanes hold consecutive 16-byte pieces of one run: the aligned
// block after ob is written whole -- p's last sh bytes, then the first 16 - sh
// of nx, the next lane's piece -- when same_next (the next lane holds the
// next piece of the same run), else only p's bytes of it; unless same_prev
// (the previous lane's piece precedes p in the run and writes the block before
// whole), p's first 16 - sh bytes go into the block before.  So every byte of
// the run is written once, by one lane, and whole blocks with one store.
__device__ __forceinline__ void store_realigned(unsigned char* ob, uint4 p, uint4 nx, bool same_next,
                                                bool same_prev) {
    const int sh = (int)(reinterpret_cast<uintptr_t>(ob) & 15u);
    if (sh == 0) {
        st_stream_u4(ob, p);
        return;
    }
    unsigned char* blk = ob - sh + 16;  // the aligned block after ob
    const uint4 v = realign16(p, nx, 16 - sh);
    if (same_next)
        st_stream_u4(blk, v);
    else
        st_bytes(blk, v, 0, sh);
    if (!same_prev) st_bytes(blk - 16, realign16(p, p, 16 - sh), sh, 16);
}

}  // namespace ss
