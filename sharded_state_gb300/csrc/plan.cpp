// plan.cpp -- layout planner (host) and the plan / diagnostics part of the C ABI.
//
// Layout rules ("FSDP1 vs FSDP2", section 03 and the 3+5-element table):
//   FLAT_ORIG_TRUE   param i >= 1 starts at roundup(end of param i-1, a) with
//                    a = 16 / elem_bytes; the group's flat length is rounded up
//                    to a multiple of N; c = length / N.
//   FLAT_ORIG_FALSE  offsets are prefix sums, L = sum of numels, c = ceil(L/N)
//                    (torch.chunk with every chunk padded to chunks[0]).
//   PER_PARAM_DIM0   c_i = ceil(d0_i / N) rows; param i's chunk sits at the
//                    prefix sum of c_j * inner_j inside every rank's shard;
//                    S = sum_i c_i * inner_i (FSDP2 _chunk_with_empty + group
//                    copy-in).
// Groups are laid out one after another: group g occupies
// [base_g, base_g + N * S_g) of every packed buffer, rank r's shard of it at
// base_g + r * S_g.
//
// Besides the offsets the planner emits the two segment tables the copy
// kernels use: `data` (every contiguous run of a parameter inside one rank's
// shard, ordered by parameter then rank) and `zero` (every pad run, ordered by
// packed offset), each split into 16 KiB tiles, one CTA per tile.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <new>
#include <tuple>

#include "internal.h"

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

// Largest element count any buffer may have: byte offsets must stay in int64.
constexpr int64_t kMaxElems = (int64_t)1 << 60;

int build_group(ss_plan* p, int g, int first, int count) {
    const int N = p->N;
    const int64_t a = 16 / p->eb;
    int64_t pos = 0;
    for (int i = first; i < first + count; ++i) {
        int64_t s = p->numel[i];
        if (p->kind == SS_FLAT_ORIG_TRUE) {
            if (i > first) {
                int64_t r = pos % a;
                if (r && !add_ok(pos, a - r, &pos)) return SS_EOVERFLOW;
            }
            p->offset[i] = pos;  // group-relative for now
            p->chunk_rows[i] = 0;
            if (!add_ok(pos, s, &pos)) return SS_EOVERFLOW;
        } else if (p->kind == SS_FLAT_ORIG_FALSE) {
            p->offset[i] = pos;
            p->chunk_rows[i] = 0;
            if (!add_ok(pos, s, &pos)) return SS_EOVERFLOW;
        } else {
            int64_t rows = p->dim0[i] / N + (p->dim0[i] % N ? 1 : 0);
            int64_t span;
            if (!mul_ok(rows, p->inner[i], &span)) return SS_EOVERFLOW;
            p->offset[i] = pos;
            p->chunk_rows[i] = rows;
            if (!add_ok(pos, span, &pos)) return SS_EOVERFLOW;
        }
        p->param_group[i] = g;
    }
    int64_t shard;
    if (p->kind == SS_FLAT_ORIG_TRUE) {
        int64_t r = pos % N;
        if (r && !add_ok(pos, N - r, &pos)) return SS_EOVERFLOW;
        shard = pos / N;
    } else if (p->kind == SS_FLAT_ORIG_FALSE) {
        shard = pos / N + (pos % N ? 1 : 0);
    } else {
        shard = pos;
    }
    int64_t span;
    if (!mul_ok(shard, N, &span)) return SS_EOVERFLOW;
    p->gshard[g] = shard;
    p->gfirst[g] = first;
    p->gnp[g] = count;
    return SS_OK;
}

void build_segments(ss_plan* p) {
    p->data.clear();
    p->zero.clear();
    p->param_seg.assign(p->n + 1, 0);
    p->group_zero.assign(p->G + 1, 0);
    int64_t u = 0;
    for (int i = 0; i < p->n; ++i) {
        p->param_seg[i] = (int)p->data.size();
        const int g = p->param_group[i];
        const int64_t base = p->gbase[g];
        if (p->kind != SS_PER_PARAM_DIM0) {
            if (p->numel[i] > 0) {
                ss::Seg s{u, p->numel[i], base + p->offset[i], 0, i, 0};
                p->data.push_back(s);
                u += s.len;
            }
        } else {
            const int64_t c = p->chunk_rows[i], d0 = p->dim0[i], in = p->inner[i];
            if (in == 0) continue;
            for (int r = 0; r < p->N; ++r) {
                int64_t lo = (int64_t)r * c;
                int64_t hi = std::min(lo + c, d0);
                if (lo >= hi) break;
                ss::Seg s{u, (hi - lo) * in, base + (int64_t)r * p->gshard[g] + p->offset[i],
                          lo * in, i, 0};
                p->data.push_back(s);
                u += s.len;
            }
        }
    }
    p->param_seg[p->n] = (int)p->data.size();

    // pad runs: the complement of the data runs inside each group's range
    int64_t uz = 0;
    for (int g = 0; g < p->G; ++g) {
        p->group_zero[g] = (int)p->zero.size();
        std::vector<std::pair<int64_t, int64_t>> runs;  // (packed_off, len)
        for (int k = p->param_seg[p->gfirst[g]]; k < p->param_seg[p->gfirst[g] + p->gnp[g]]; ++k)
            runs.emplace_back(p->data[k].packed_off, p->data[k].len);
        std::sort(runs.begin(), runs.end());
        int64_t cur = p->gbase[g];
        const int64_t end = p->gbase[g] + (int64_t)p->N * p->gshard[g];
        auto emit = [&](int64_t from, int64_t to) {
            if (to > from) {
                ss::Seg s{uz, to - from, from, 0, -1, 0};
                p->zero.push_back(s);
                uz += s.len;
            }
        };
        for (auto& r : runs) {
            emit(cur, r.first);
            cur = r.first + r.second;
        }
        emit(cur, end);
    }
    p->group_zero[p->G] = (int)p->zero.size();
}

// Split every segment into tiles of kTileBytes; false if a tile index would
// not fit the 32-bit fields.
bool build_tiles(const std::vector<ss::Seg>& segs, int eb, std::vector<ss::Tile>* tiles,
                 std::vector<int64_t>* seg_tile) {
    const int64_t T = ss::kTileBytes / eb;
    tiles->clear();
    seg_tile->assign(segs.size() + 1, 0);
    for (size_t k = 0; k < segs.size(); ++k) {
        (*seg_tile)[k] = (int64_t)tiles->size();
        const int64_t nt = (segs[k].len + T - 1) / T;
        if (nt > 0x7FFFFFFF || k > 0x7FFFFFFF) return false;
        for (int64_t j = 0; j < nt; ++j) tiles->push_back(ss::Tile{(int32_t)k, (int32_t)j});
    }
    (*seg_tile)[segs.size()] = (int64_t)tiles->size();
    return true;
}

// The data tiles with their segment's fields inline (the tile index in
// `reserved`), so one load places a tile.
void build_tiles_ext(ss_plan* p) {
    p->data_tiles_ext.resize(p->data_tiles.size());
    for (size_t t = 0; t < p->data_tiles.size(); ++t) {
        const ss::Tile& tl = p->data_tiles[t];
        const ss::Seg& sg = p->data[tl.seg];
        p->data_tiles_ext[t] = ss::PmEntry{sg.packed_off, sg.param_off, sg.len, sg.param, tl.idx};
    }
}

// The packed segment map: data segments by packed offset, and for every
// kMapBlock-element block the last segment starting at or before it.
void build_packed_map(ss_plan* p) {
    std::vector<int> order;
    order.reserve(p->data.size());
    for (size_t k = 0; k < p->data.size(); ++k)
        if (p->data[k].len > 0) order.push_back((int)k);
    std::sort(order.begin(), order.end(),
              [&](int a, int b) { return p->data[a].packed_off < p->data[b].packed_off; });
    p->pm.resize(order.size());
    for (size_t m = 0; m < order.size(); ++m) {
        const ss::Seg& sg = p->data[order[m]];
        p->pm[m] = ss::PmEntry{sg.packed_off, sg.param_off, sg.len, sg.param, 0};
    }
    const int64_t nb = p->total / ss::kMapBlock + 2;
    p->pm_block.assign((size_t)nb, 0);
    const int M = (int)order.size();
    int m = 0;
    for (int64_t B = 0; B < nb; ++B) {
        const int64_t pos = B * ss::kMapBlock;
        while (m + 1 < M && p->pm[m + 1].packed_off <= pos) ++m;
        p->pm_block[(size_t)B] = m;
    }
}

int upload(ss_plan* p) {
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) return ss::cuda_fail(e);
    // on the device: the pad segments and their tiles (pack's zero fill), the
    // data tiles with their segments inline (pack, all-gather) and the packed
    // segment map (the one-pass step); the plain data tables stay on the host
    const size_t nz = std::max<size_t>(p->zero.size(), 1);
    e = cudaMalloc(&p->d_zero, nz * sizeof(ss::Seg));
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SS_ENOMEM : ss::cuda_fail(e);
    if (!p->zero.empty()) {
        e = cudaMemcpy(p->d_zero, p->zero.data(), p->zero.size() * sizeof(ss::Seg),
                       cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return ss::cuda_fail(e);
    }
    const size_t ndt = std::max<size_t>(p->data_tiles.size(), 1);
    const size_t nzt = std::max<size_t>(p->zero_tiles.size(), 1);
    e = cudaMalloc(&p->d_zero_tiles, nzt * sizeof(ss::Tile));
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SS_ENOMEM : ss::cuda_fail(e);
    if (!p->zero_tiles.empty()) {
        e = cudaMemcpy(p->d_zero_tiles, p->zero_tiles.data(), p->zero_tiles.size() * sizeof(ss::Tile),
                       cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return ss::cuda_fail(e);
    }
    e = cudaMalloc(&p->d_data_tiles_ext, ndt * sizeof(ss::PmEntry));
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SS_ENOMEM : ss::cuda_fail(e);
    if (!p->data_tiles_ext.empty()) {
        e = cudaMemcpy(p->d_data_tiles_ext, p->data_tiles_ext.data(),
                       p->data_tiles_ext.size() * sizeof(ss::PmEntry), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return ss::cuda_fail(e);
    }
    e = cudaMalloc(&p->d_pm, std::max<size_t>(p->pm.size(), 1) * sizeof(ss::PmEntry));
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SS_ENOMEM : ss::cuda_fail(e);
    e = cudaMalloc(&p->d_pm_block, std::max<size_t>(p->pm_block.size(), 1) * sizeof(int));
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SS_ENOMEM : ss::cuda_fail(e);
    if (!p->pm.empty()) {
        e = cudaMemcpy(p->d_pm, p->pm.data(), p->pm.size() * sizeof(ss::PmEntry),
                       cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return ss::cuda_fail(e);
    }
    if (!p->pm_block.empty()) {
        e = cudaMemcpy(p->d_pm_block, p->pm_block.data(), p->pm_block.size() * sizeof(int),
                       cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return ss::cuda_fail(e);
    }
    p->has_dev = true;
    return SS_OK;
}

}  // namespace

namespace ss {

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return SS_ECUDA;
}

int check_launch() {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SS_OK : cuda_fail(e);
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 132;
    if (dev < 64 && cache[dev]) return cache[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 132;
    if (dev < 64) cache[dev] = v;
    return v;
}

}  // namespace ss

extern "C" {

int fsdp_plan_create(const ss_plan_desc* d, ss_plan** out) {
    if (!d || !out) return SS_EINVAL;
    *out = nullptr;
    if (d->kind != SS_FLAT_ORIG_FALSE && d->kind != SS_FLAT_ORIG_TRUE &&
        d->kind != SS_PER_PARAM_DIM0)
        return SS_EINVAL;
    if (d->world_size < 1 || d->world_size > SS_MAX_WORLD) return SS_EINVAL;
    if (d->elem_bytes != 2 && d->elem_bytes != 4) return SS_EINVAL;
    if (d->num_params < 0 || (d->num_params > 0 && !d->dim0)) return SS_EINVAL;
    if (d->flags & ~SS_PLAN_HOST_ONLY) return SS_EINVAL;
    const int n = d->num_params;
    int G = (d->num_groups <= 0 || !d->group_num_params) ? 1 : d->num_groups;
    if (d->num_groups > 0 && !d->group_num_params) return SS_EINVAL;
    if (d->group_num_params && d->num_groups > 0) {
        int64_t sum = 0;
        for (int g = 0; g < G; ++g) {
            if (d->group_num_params[g] < 0) return SS_EINVAL;
            sum += d->group_num_params[g];
        }
        if (sum != n) return SS_EINVAL;
    }

    ss_plan* p = new (std::nothrow) ss_plan();
    if (!p) return SS_ENOMEM;
    int rc = SS_OK;
    try {
        p->kind = d->kind;
        p->N = d->world_size;
        p->eb = d->elem_bytes;
        p->n = n;
        p->G = G;
        p->dim0.resize(n);
        p->inner.resize(n);
        p->numel.resize(n);
        p->chunk_rows.resize(n);
        p->offset.resize(n);
        p->param_group.resize(n);
        p->gbase.resize(G);
        p->gshard.resize(G);
        p->gfirst.resize(G);
        p->gnp.resize(G);
        for (int i = 0; i < n; ++i) {
            int64_t d0 = d->dim0[i], in = d->inner ? d->inner[i] : 1;
            if (d0 < 0 || in < 0) { rc = SS_EINVAL; break; }
            int64_t s;
            if (!mul_ok(d0, in, &s) || s > kMaxElems) { rc = SS_EOVERFLOW; break; }
            p->dim0[i] = d0;
            p->inner[i] = in;
            p->numel[i] = s;
            if (!add_ok(p->unpadded, s, &p->unpadded)) { rc = SS_EOVERFLOW; break; }
        }
        int first = 0;
        int64_t base = 0;
        for (int g = 0; rc == SS_OK && g < G; ++g) {
            int cnt = (G == 1 && !(d->num_groups > 0 && d->group_num_params)) ? n
                                                                              : d->group_num_params[g];
            rc = build_group(p, g, first, cnt);
            if (rc != SS_OK) break;
            p->gbase[g] = base;
            int64_t span = (int64_t)p->N * p->gshard[g];
            if (!add_ok(base, span, &base) || base > kMaxElems) { rc = SS_EOVERFLOW; break; }
            if (!add_ok(p->shard_total, p->gshard[g], &p->shard_total)) { rc = SS_EOVERFLOW; break; }
            first += cnt;
        }
        if (rc == SS_OK) {
            p->total = base;
            // the queried offset is absolute in the packed buffers
            for (int i = 0; i < n; ++i) p->offset[i] += p->gbase[p->param_group[i]];
            // build_segments wants group-relative offsets: undo temporarily
            std::vector<int64_t> absolute = p->offset;
            for (int i = 0; i < n; ++i) p->offset[i] -= p->gbase[p->param_group[i]];
            build_segments(p);
            p->offset = absolute;
            if (p->data.size() > (size_t)0x7FFFFFFF || p->zero.size() > (size_t)0x7FFFFFFF)
                rc = SS_EOVERFLOW;
            else if (!build_tiles(p->data, p->eb, &p->data_tiles, &p->data_seg_tile) ||
                     !build_tiles(p->zero, p->eb, &p->zero_tiles, &p->zero_seg_tile))
                rc = SS_EOVERFLOW;
            else {
                build_tiles_ext(p);
                build_packed_map(p);
            }
            const int64_t per16 = 16 / p->eb;
            p->vec_aligned = true;
            for (const ss::Seg& sg : p->data)
                p->vec_aligned &= sg.packed_off % per16 == 0 && sg.param_off % per16 == 0 &&
                                  sg.len % per16 == 0;
        }
        if (rc == SS_OK && !(d->flags & SS_PLAN_HOST_ONLY)) rc = upload(p);
    } catch (const std::bad_alloc&) {
        rc = SS_ENOMEM;
    }
    if (rc != SS_OK) {
        fsdp_plan_destroy(p);
        return rc;
    }
    *out = p;
    return SS_OK;
}

int fsdp_plan_layout(ss_layout kind, int world_size, int elem_bytes, int num_params,
                     const int64_t* dim0, const int64_t* inner, ss_plan** out) {
    ss_plan_desc d;
    std::memset(&d, 0, sizeof d);
    d.kind = kind;
    d.world_size = world_size;
    d.elem_bytes = elem_bytes;
    d.num_params = num_params;
    d.dim0 = dim0;
    d.inner = inner;
    return fsdp_plan_create(&d, out);
}

int fsdp_plan_info(const ss_plan* p, ss_plan_info* o) {
    if (!p || !o) return SS_EINVAL;
    o->shard_numel = p->shard_total;
    o->total_numel = p->total;
    o->unpadded_numel = p->unpadded;
    o->pad_numel = p->total - p->unpadded;
    o->world_size = p->N;
    o->elem_bytes = p->eb;
    o->num_params = p->n;
    o->num_groups = p->G;
    o->kind = p->kind;
    o->has_device_metadata = p->has_dev ? 1 : 0;
    return SS_OK;
}

int fsdp_plan_param_offset(const ss_plan* p, int param, int64_t* offset_out,
                           int64_t* chunk_rows_out) {
    if (!p || !offset_out || param < 0 || param >= p->n) return SS_EINVAL;
    *offset_out = p->offset[param];
    if (chunk_rows_out) *chunk_rows_out = p->chunk_rows[param];
    return SS_OK;
}

int fsdp_plan_group(const ss_plan* p, int group, int64_t* base_out, int64_t* shard_numel_out,
                    int* first_param_out, int* num_params_out) {
    if (!p || group < 0 || group >= p->G) return SS_EINVAL;
    if (base_out) *base_out = p->gbase[group];
    if (shard_numel_out) *shard_numel_out = p->gshard[group];
    if (first_param_out) *first_param_out = p->gfirst[group];
    if (num_params_out) *num_params_out = p->gnp[group];
    return SS_OK;
}

void fsdp_plan_destroy(ss_plan* p) {
    if (!p) return;
    if (p->d_zero) cudaFree(p->d_zero);
    if (p->d_zero_tiles) cudaFree(p->d_zero_tiles);
    if (p->d_data_tiles_ext) cudaFree(p->d_data_tiles_ext);
    if (p->d_pm) cudaFree(p->d_pm);
    if (p->d_pm_block) cudaFree(p->d_pm_block);
    delete p;
}

int fsdp_plan_validate(const ss_plan* p) {
    if (!p) return SS_EINVAL;
    // data segments: inside their group's range and their parameter, ordered
    // by parameter, consecutive starts
    std::vector<std::pair<int64_t, int64_t>> cover;  // (packed_off, len) of data and pads
    int64_t u = 0;
    for (size_t k = 0; k < p->data.size(); ++k) {
        const ss::Seg& s = p->data[k];
        if (s.param < 0 || s.param >= p->n || s.len <= 0 || s.start != u) return SS_EINVAL;
        if (s.param_off < 0 || s.param_off + s.len > p->numel[s.param]) return SS_EINVAL;
        const int g = p->param_group[s.param];
        const int64_t glo = p->gbase[g], ghi = glo + (int64_t)p->N * p->gshard[g];
        if (s.packed_off < glo || s.packed_off + s.len > ghi) return SS_EINVAL;
        if (k > 0 && p->data[k - 1].param > s.param) return SS_EINVAL;
        u += s.len;
        cover.emplace_back(s.packed_off, s.len);
    }
    if (u != p->unpadded) return SS_EINVAL;  // every parameter element exactly once
    int64_t uz = 0;
    for (const ss::Seg& s : p->zero) {
        if (s.param != -1 || s.len <= 0 || s.start != uz) return SS_EINVAL;
        uz += s.len;
        cover.emplace_back(s.packed_off, s.len);
    }
    // data + pads tile [0, total) with no gap and no overlap
    std::sort(cover.begin(), cover.end());
    int64_t pos = 0;
    for (auto& c : cover) {
        if (c.first != pos) return SS_EINVAL;
        pos += c.second;
    }
    if (pos != p->total) return SS_EINVAL;
    // tiles: every segment split into consecutive tiles, each inside its segment
    auto check_tiles = [&](const std::vector<ss::Seg>& segs, const std::vector<ss::Tile>& tiles,
                           const std::vector<int64_t>& seg_tile) {
        const int64_t T = ss::kTileBytes / p->eb;
        if (seg_tile.size() != segs.size() + 1 || seg_tile.back() != (int64_t)tiles.size())
            return false;
        for (size_t k = 0; k < segs.size(); ++k) {
            const int64_t nt = (segs[k].len + T - 1) / T;
            if (seg_tile[k + 1] - seg_tile[k] != nt) return false;
            for (int64_t j = 0; j < nt; ++j) {
                const ss::Tile& t = tiles[seg_tile[k] + j];
                if (t.seg != (int32_t)k || t.idx != (int32_t)j) return false;
            }
        }
        return true;
    };
    if (!check_tiles(p->data, p->data_tiles, p->data_seg_tile) ||
        !check_tiles(p->zero, p->zero_tiles, p->zero_seg_tile))
        return SS_EINVAL;
    // data tiles with their segment inline: the same tiles, same fields
    if (p->data_tiles_ext.size() != p->data_tiles.size()) return SS_EINVAL;
    for (size_t t = 0; t < p->data_tiles.size(); ++t) {
        const ss::Tile& tl = p->data_tiles[t];
        const ss::Seg& sg = p->data[tl.seg];
        const ss::PmEntry& x = p->data_tiles_ext[t];
        if (x.packed_off != sg.packed_off || x.param_off != sg.param_off || x.len != sg.len ||
            x.param != sg.param || x.reserved != tl.idx)
            return SS_EINVAL;
    }
    // packed segment map: every data segment once, by strictly increasing
    // offset; pm_block[B] is the last segment starting at or before block B
    const size_t M = p->pm.size();
    if (M != p->data.size()) return SS_EINVAL;
    {
        std::vector<std::tuple<int64_t, int64_t, int64_t, int>> segs_by_off, pm_by_off;
        for (const ss::Seg& sg : p->data)
            segs_by_off.emplace_back(sg.packed_off, sg.param_off, sg.len, sg.param);
        for (const ss::PmEntry& e : p->pm) pm_by_off.emplace_back(e.packed_off, e.param_off, e.len, e.param);
        std::sort(segs_by_off.begin(), segs_by_off.end());
        if (segs_by_off != pm_by_off) return SS_EINVAL;
    }
    for (size_t m = 0; m < M; ++m) {
        const ss::PmEntry& e = p->pm[m];
        if (e.param < 0 || e.param >= p->n || e.len <= 0) return SS_EINVAL;
        if (e.param_off < 0 || e.param_off + e.len > p->numel[e.param]) return SS_EINVAL;
        if (m > 0 && e.packed_off < p->pm[m - 1].packed_off + p->pm[m - 1].len) return SS_EINVAL;
    }
    if (p->pm_block.size() != (size_t)(p->total / ss::kMapBlock + 2)) return SS_EINVAL;
    for (size_t B = 0; B < p->pm_block.size(); ++B) {
        const int m = p->pm_block[B];
        if (M == 0) {
            if (m != 0) return SS_EINVAL;
            continue;
        }
        if (m < 0 || (size_t)m >= M) return SS_EINVAL;
        const int64_t pos = (int64_t)B * ss::kMapBlock;
        if (m > 0 && p->pm[m].packed_off > pos) return SS_EINVAL;
        if ((size_t)m + 1 < M && p->pm[m + 1].packed_off <= pos) return SS_EINVAL;
    }
    return SS_OK;
}

const char* ss_strerror(int s) {
    switch (s) {
        case SS_OK: return "ok";
        case SS_EINVAL: return "invalid argument";
        case SS_EALIGN: return "pointer misaligned";
        case SS_EOVERFLOW: return "size overflow";
        case SS_ENOMEM: return "out of memory";
        case SS_ECUDA: return "CUDA runtime error";
        case SS_ENODEVICE: return "plan has no device metadata";
        case SS_ESCRATCH: return "request exceeds the fixed scratch array";
        default: return "unknown status";
    }
}

int ss_last_cuda_error(void) { return g_last_cuda_error; }

const char* ss_version(void) { return "0.1.0"; }

uint64_t ss_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
