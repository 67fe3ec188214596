// internal.h -- host-side plan object and helpers shared by the library's
// translation units (never installed; the public ABI is include/shardstate.h).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "shardstate.h"

namespace ss {

// One contiguous run of parameter elements inside the packed layout.
//   start       position in the segment table's iteration space (prefix sum
//               of lengths); a CTA finds its first segment by binary search
//               on it
//   len         elements
//   packed_off  element index in every packed buffer
//   param_off   element index inside the parameter tensor (-1 param: zero fill)
//   param       parameter index, or -1 for a pad run
struct Seg {
    int64_t start;
    int64_t len;
    int64_t packed_off;
    int64_t param_off;
    int32_t param;
    int32_t reserved;
};
static_assert(sizeof(Seg) == 40, "Seg layout");

// Work unit of the copy kernels: one CTA moves one tile of kTileBytes inside
// one segment.  Tile k of segment s covers elements [k*T, min((k+1)*T, len))
// with T = kTileBytes / elem_bytes.
constexpr int kTileBytes = 16384;
struct Tile {
    int32_t seg;
    int32_t idx;
};
static_assert(sizeof(Tile) == 8, "Tile layout");

// Block of packed elements indexed by the plan's packed segment map
// (ss_plan::pm_block); one flat CTA of 256 threads x 8 elements.
constexpr int64_t kMapBlock = 2048;

// One data segment of the packed segment map: everything a kernel needs to
// place packed elements [packed_off, packed_off + len) in their parameter.
struct PmEntry {
    int64_t packed_off;
    int64_t param_off;
    int64_t len;
    int32_t param;
    int32_t reserved;
};
static_assert(sizeof(PmEntry) == 32, "PmEntry layout");

}  // namespace ss

struct ss_plan {
    int kind = 0;
    int N = 1;
    int eb = 2;
    int n = 0;
    int G = 0;
    std::vector<int64_t> dim0, inner, numel, chunk_rows;
    std::vector<int64_t> offset;        // fsdp_plan_param_offset value
    std::vector<int> param_group;
    std::vector<int64_t> gbase, gshard;  // per group: base index, elements per rank
    std::vector<int> gfirst, gnp;        // per group: first param, param count
    int64_t shard_total = 0, total = 0, unpadded = 0;
    // data segments sorted by (param, rank); param_seg[i] = first data segment of param i
    std::vector<ss::Seg> data;
    std::vector<int> param_seg;
    // pad segments sorted by packed offset; group_zero[g] = first pad segment of group g
    std::vector<ss::Seg> zero;
    std::vector<int> group_zero;
    // tiles of the data / pad segments; seg_tile[k] = first tile of segment k (size nseg+1)
    std::vector<ss::Tile> data_tiles, zero_tiles;
    std::vector<int64_t> data_seg_tile, zero_seg_tile;
    // the data tiles with their segment's fields inline (tile index in
    // `reserved`): one load places a tile
    std::vector<ss::PmEntry> data_tiles_ext;
    // device copies
    ss::Seg* d_zero = nullptr;
    ss::Tile* d_zero_tiles = nullptr;
    ss::PmEntry* d_data_tiles_ext = nullptr;
    // The data segments in packed-offset order (pm[m], m = 0..M-1).
    // pm_block[B] is the last m whose packed offset is <= B * kMapBlock (0 if
    // none), for every block B in [0, total / kMapBlock + 1]: the segment
    // holding packed element f is among pm_block[f / kMapBlock] ..
    // pm_block[f / kMapBlock + 1].
    std::vector<ss::PmEntry> pm;
    std::vector<int> pm_block;
    ss::PmEntry* d_pm = nullptr;
    int* d_pm_block = nullptr;
    // every data segment's packed offset, parameter offset and length are
    // multiples of 16 bytes (enables the copy kernels' fast path)
    bool vec_aligned = false;
    int device = -1;
    bool has_dev = false;
};

namespace ss {

// Record a failed CUDA call for ss_last_cuda_error() and return SS_ECUDA.
int cuda_fail(cudaError_t e);

// Check the last launch; SS_OK or SS_ECUDA.  Counts the launch.
int check_launch();

// Number of SMs of the current device (cached per device).
int num_sms();

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// SS_OK if the current device is the one the plan's metadata lives on.
inline int check_device(const ss_plan* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ECUDA;
    return dev == p->device ? SS_OK : SS_EINVAL;
}

// Element range [lo, hi) of the packed buffers covered by `group` (-1 = all).
inline bool group_range(const ss_plan* p, int group, int64_t* lo, int64_t* hi) {
    if (group < 0) {
        *lo = 0;
        *hi = p->total;
        return group == -1;
    }
    if (group >= p->G) return false;
    *lo = p->gbase[group];
    *hi = p->gbase[group] + (int64_t)p->N * p->gshard[group];
    return true;
}

}  // namespace ss
