// ddp.cu -- DDP gradient bucketing with a bucketed mean over N virtual ranks.
//
// "Scaling data parallel", sections 3-4: a gradient is final as soon as its
// layer's backward is done, last layer first, so tensors are visited in
// reverse registration order; gradients accumulate in a bucket and, once the
// bucket holds at least bucket_cap bytes, it goes out as one all-reduce (sum,
// then divide by N).  Small buckets pay the fixed per-collective cost many
// times; a huge cap exposes the last bucket.
//
// On one GPU the N ranks' gradients are N sets of tensors in HBM, so one
// bucket's pack + all-reduce + unpack is a single pass: for each element of
// each tensor in the bucket, read N bf16 values, sum in fp32 in rank order,
// divide by N, round to bf16 and write the average (2N + 2 bytes per
// element).  One kernel launch per bucket keeps the per-collective fixed cost
// visible; inside a bucket one CTA averages one 4096-element tile, finding its
// first tensor with a warp-level search over the bucket-order prefix sums of
// the tensor sizes.  The per-tensor pointers and those prefix sums go to the
// device in a per-call table.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "device_utils.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 256;

// Sum one 8-element vector over ranks (rank order, fp32), divide by N, round.
// ANY: the inputs at k need only 2-byte alignment (read as the two aligned
// 16-byte blocks that cover them, joined in registers).
template <int NR, bool ANY = false>
__device__ __forceinline__ uint4 mean8(const void* const* in, int N, int64_t k) {
    const int n = NR > 0 ? NR : N;
    auto ld = [&](int r) {
        const uint16_t* p = static_cast<const uint16_t*>(in[r]) + k;
        return ANY ? ss::ld_any16(p) : ss::ld_stream_u4(p);
    };
    uint4 w0 = ld(0);
    float s[8] = {ss::bf16_lo(w0.x), ss::bf16_hi(w0.x), ss::bf16_lo(w0.y), ss::bf16_hi(w0.y),
                  ss::bf16_lo(w0.z), ss::bf16_hi(w0.z), ss::bf16_lo(w0.w), ss::bf16_hi(w0.w)};
    if (NR > 0) {
        uint4 w[NR > 1 ? NR - 1 : 1];
#pragma unroll
        for (int r = 1; r < NR; ++r) w[r - 1] = ld(r);
#pragma unroll
        for (int r = 1; r < NR; ++r) {
            s[0] = __fadd_rn(s[0], ss::bf16_lo(w[r - 1].x));
            s[1] = __fadd_rn(s[1], ss::bf16_hi(w[r - 1].x));
            s[2] = __fadd_rn(s[2], ss::bf16_lo(w[r - 1].y));
            s[3] = __fadd_rn(s[3], ss::bf16_hi(w[r - 1].y));
            s[4] = __fadd_rn(s[4], ss::bf16_lo(w[r - 1].z));
            s[5] = __fadd_rn(s[5], ss::bf16_hi(w[r - 1].z));
            s[6] = __fadd_rn(s[6], ss::bf16_lo(w[r - 1].w));
            s[7] = __fadd_rn(s[7], ss::bf16_hi(w[r - 1].w));
        }
    } else {
        // any N: ranks 1.. in batches of 8 loads in flight, added in rank order
        for (int r0 = 1; r0 < n; r0 += 8) {
            uint4 w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r0 + j < n) w[j] = ld(r0 + j);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r0 + j < n) {
                    s[0] = __fadd_rn(s[0], ss::bf16_lo(w[j].x));
                    s[1] = __fadd_rn(s[1], ss::bf16_hi(w[j].x));
                    s[2] = __fadd_rn(s[2], ss::bf16_lo(w[j].y));
                    s[3] = __fadd_rn(s[3], ss::bf16_hi(w[j].y));
                    s[4] = __fadd_rn(s[4], ss::bf16_lo(w[j].z));
                    s[5] = __fadd_rn(s[5], ss::bf16_hi(w[j].z));
                    s[6] = __fadd_rn(s[6], ss::bf16_lo(w[j].w));
                    s[7] = __fadd_rn(s[7], ss::bf16_hi(w[j].w));
                }
            }
        }
    }
    const float fN = (float)n;
    uint4 o;
    o.x = ss::pack_bf16x2(__fdiv_rn(s[0], fN), __fdiv_rn(s[1], fN));
    o.y = ss::pack_bf16x2(__fdiv_rn(s[2], fN), __fdiv_rn(s[3], fN));
    o.z = ss::pack_bf16x2(__fdiv_rn(s[4], fN), __fdiv_rn(s[5], fN));
    o.w = ss::pack_bf16x2(__fdiv_rn(s[6], fN), __fdiv_rn(s[7], fN));
    return o;
}

__device__ __forceinline__ uint16_t mean1(const void* const* in, int N, int64_t k) {
    float s = ss::bf16_to_f32(static_cast<const uint16_t*>(in[0])[k]);
    for (int r = 1; r < N; ++r) s = __fadd_rn(s, ss::bf16_to_f32(static_cast<const uint16_t*>(in[r])[k]));
    return ss::f32_to_bf16(__fdiv_rn(s, (float)N));
}

// Average one tensor piece [k0, k1) of the tensor whose N inputs and one
// output are ptrs[0..N] (CTA-cooperative).
// ANY false: inputs not congruent to the output go element by element (the
// host picks ANY for the buckets that hold such a tensor).
template <int NR, bool ANY>
__device__ __forceinline__ void avg_piece(const void* const* ptrs, int N, int64_t k0, int64_t k1) {
    const int tid = threadIdx.x, nt = blockDim.x;
    uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(ptrs[N]));
    // The output's stores are aligned after a scalar head.  Inputs congruent
    // to the output load as plain vectors; otherwise every input vector is
    // rebuilt from the two aligned blocks that cover it.
    const uintptr_t ref = reinterpret_cast<uintptr_t>(out + k0) & 15u;
    bool vec = true;
    for (int r = 0; r < N; ++r)
        vec &= ((reinterpret_cast<uintptr_t>(static_cast<const uint16_t*>(ptrs[r]) + k0) & 15u) == ref);
    if (!ANY && !vec) {
        for (int64_t k = k0 + tid; k < k1; k += nt) out[k] = mean1(ptrs, N, k);
        return;
    }
    int64_t head = (int64_t)(((16u - ref) & 15u) / 2);
    if (head > k1 - k0) head = k1 - k0;
    if (tid < head) out[k0 + tid] = mean1(ptrs, N, k0 + tid);
    const int64_t vb = k0 + head;
    const int64_t nvec = (k1 - vb) / 8;
    if (!ANY || vec) {
        for (int64_t q = tid; q < nvec; q += nt) {
            const int64_t k = vb + 8 * q;
            ss::st_stream_u4(out + k, mean8<NR>(ptrs, N, k));
        }
    } else {
        for (int64_t q = tid; q < nvec; q += nt) {
            const int64_t k = vb + 8 * q;
            ss::st_stream_u4(out + k, mean8<NR, ANY>(ptrs, N, k));
        }
    }
    const int64_t done = vb + 8 * nvec;
    if (tid < k1 - done) out[done + tid] = mean1(ptrs, N, done + tid);
}

// Last index o in [lo, hi) with prefix[o] <= u (prefix non-decreasing,
// prefix[lo] <= u), found by one warp with a 32-ary search: each round the 32
// lanes probe evenly spaced entries and a ballot keeps the last one <= u.
// Every lane of the warp returns the same index.
__device__ __forceinline__ int warp_find(const int64_t* __restrict__ prefix, int lo, int hi,
                                         int64_t u) {
    const int lane = threadIdx.x & 31;
    while (hi - lo > 1) {
        const int stride = (hi - lo + 31) / 32;
        const int idx = lo + lane * stride;
        const bool le = idx < hi && prefix[idx] <= u;
        const unsigned ballot = __ballot_sync(0xFFFFFFFFu, le);
        const int last = 31 - __clz(ballot);  // lane 0 probes lo, so ballot != 0
        lo += last * stride;
        hi = lo + stride < hi ? lo + stride : hi;
    }
    return lo;
}

// One bucket: tensors [o_lo, o_hi) of the bucket-ordered table; prefix[o] is
// the element offset of tensor o in bucket order.  CTA b averages bucket
// elements [b*T, (b+1)*T) (T = kTile), walking the tensors that cover them.
constexpr int64_t kTile = 4096;

template <int NR, bool ANY>
__global__ void __launch_bounds__(kThreads)
ddp_bucket_kernel(const int64_t* __restrict__ prefix, const void* const* __restrict__ ptrs, int N,
                  int o_lo, int o_hi) {
    // Buckets are independent (disjoint tensors, read-only table), so the next
    // bucket's launch may start as soon as every CTA of this one is running:
    // its CTAs then fill SMs while this bucket drains.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t u_lo = prefix[o_lo], u_hi = prefix[o_hi];
    int64_t u = u_lo + (int64_t)blockIdx.x * kTile;
    const int64_t u_end = u + kTile < u_hi ? u + kTile : u_hi;
    if (u < u_end) {
        int o = warp_find(prefix, o_lo, o_hi, u);
        while (u < u_end && o < o_hi) {
            const int64_t t_end = prefix[o + 1];
            const int64_t piece_end = t_end < u_end ? t_end : u_end;
            if (piece_end > u)
                avg_piece<NR, ANY>(ptrs + (size_t)o * (N + 1), N, u - prefix[o],
                                   piece_end - prefix[o]);
            u = piece_end > u ? piece_end : u;
            ++o;
        }
    }
    // This grid completes only after the previous bucket's has: its last CTA
    // waits for that grid once its own work is done.  Completion is thus
    // ordered along the call's buckets, and stream work after the call sees
    // every output.  The previous grid's CTAs are all resident or finished
    // by the time this grid starts (it launches once each of them has
    // triggered), so the wait ends; one waiting CTA per grid costs at most
    // one CTA slot at the tail.
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

using DdpKernel = void (*)(const int64_t*, const void* const*, int, int, int);

// Launch one bucket with programmatic stream serialisation: it may begin
// while the previous bucket's kernel on the stream is still finishing.
cudaError_t launch_bucket(DdpKernel fn, unsigned grid, cudaStream_t st, const int64_t* prefix,
                          const void* const* ptrs, int N, int o_lo, int o_hi) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1] = {};
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, prefix, ptrs, N, o_lo, o_hi);
}

template <bool ANY>
DdpKernel pick_n(int N) {
    switch (N) {
        case 1: return ddp_bucket_kernel<1, ANY>;
        case 2: return ddp_bucket_kernel<2, ANY>;
        case 3: return ddp_bucket_kernel<3, ANY>;
        case 4: return ddp_bucket_kernel<4, ANY>;
        case 5: return ddp_bucket_kernel<5, ANY>;
        case 6: return ddp_bucket_kernel<6, ANY>;
        case 7: return ddp_bucket_kernel<7, ANY>;
        case 8: return ddp_bucket_kernel<8, ANY>;
        default: return ddp_bucket_kernel<0, ANY>;
    }
}

// any: the bucket holds a tensor whose inputs are not all congruent to its
// output mod 16 bytes (they are then read through realigning loads).
DdpKernel pick(int N, bool any) { return any ? pick_n<true>(N) : pick_n<false>(N); }

// Whether tensor o of a bucket-ordered pointer table needs realigning loads.
bool needs_realign(const void* const* ptrs, int N, int o) {
    const void* const* p = ptrs + (size_t)o * (N + 1);
    const uintptr_t out = reinterpret_cast<uintptr_t>(p[N]);
    for (int r = 0; r < N; ++r)
        if ((reinterpret_cast<uintptr_t>(p[r]) ^ out) & 15u) return true;
    return false;
}

}  // namespace

namespace {

// The bucket table goes to the device with a copy from host memory that lives
// only for the call.  A stream capture would record that copy with the host
// address and replay it after the memory is gone, so both entry points refuse
// a capturing stream: SS_EINVAL, before any work is queued.
int refuse_capture(cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return ss::cuda_fail(e);
    return cs == cudaStreamCaptureStatusNone ? SS_OK : SS_EINVAL;
}

}  // namespace

extern "C" {

int ddp_bucket_assign(int num_tensors, const int64_t* numels, int elem_bytes,
                      size_t bucket_cap_bytes, int* bucket_of) {
    if (num_tensors < 0 || (num_tensors > 0 && (!numels || !bucket_of))) return SS_EINVAL;
    if (bucket_cap_bytes == 0 || (elem_bytes != 2 && elem_bytes != 4)) return SS_EINVAL;
    int bucket = 0;
    unsigned long long fill = 0;
    for (int t = num_tensors - 1; t >= 0; --t) {
        if (numels[t] < 0) return SS_EINVAL;
        bucket_of[t] = bucket;
        fill += (unsigned long long)numels[t] * (unsigned long long)elem_bytes;
        if (fill >= bucket_cap_bytes) {
            ++bucket;
            fill = 0;
        }
    }
    return fill > 0 ? bucket + 1 : bucket;
}

int ddp_bucket_pack_average(int world_size, int num_tensors, const int64_t* numels,
                            const void* const* rank_grads, size_t bucket_cap_bytes,
                            void* const* avg_out, int* num_buckets_out, ss_stream_t stream) {
    if (world_size < 1 || world_size > SS_MAX_WORLD || num_tensors < 0) return SS_EINVAL;
    if (num_tensors > 0 && (!numels || !rank_grads || !avg_out)) return SS_EINVAL;
    if (bucket_cap_bytes == 0) return SS_EINVAL;
    const int N = world_size, T = num_tensors;
    for (int t = 0; t < T; ++t) {
        if (numels[t] < 0 || numels[t] > ((int64_t)1 << 60)) return SS_EINVAL;
        if (numels[t] == 0) continue;
        if (!avg_out[t]) return SS_EINVAL;
        if (!ss::aligned(avg_out[t], 2)) return SS_EALIGN;
        for (int r = 0; r < N; ++r) {
            const void* q = rank_grads[(size_t)r * T + t];
            if (!q) return SS_EINVAL;
            if (!ss::aligned(q, 2)) return SS_EALIGN;
        }
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (int crc = refuse_capture(st)) return crc;
    std::vector<int> bucket_of((size_t)(T > 0 ? T : 1));
    const int nb = ddp_bucket_assign(T, numels, 2, bucket_cap_bytes, bucket_of.data());
    if (nb < 0) return nb;
    if (num_buckets_out) *num_buckets_out = nb;
    if (nb == 0) return SS_OK;

    // table in bucket order (reverse registration order): prefix[T+1] then ptrs[T][N+1]
    const size_t n_prefix = (size_t)T + 1;
    const size_t n_ptrs = (size_t)T * (size_t)(N + 1);
    std::vector<unsigned char> host(n_prefix * 8 + n_ptrs * 8);
    int64_t* prefix = reinterpret_cast<int64_t*>(host.data());
    const void** ptrs = reinterpret_cast<const void**>(host.data() + n_prefix * 8);
    std::vector<int> bucket_start((size_t)nb + 1, 0);
    prefix[0] = 0;
    for (int o = 0; o < T; ++o) {
        const int t = T - 1 - o;
        prefix[o + 1] = prefix[o] + numels[t];
        for (int r = 0; r < N; ++r) ptrs[(size_t)o * (N + 1) + r] = rank_grads[(size_t)r * T + t];
        ptrs[(size_t)o * (N + 1) + N] = avg_out[t];
        if (o == 0 || bucket_of[t] != bucket_of[t + 1]) bucket_start[bucket_of[t]] = o;
    }
    bucket_start[nb] = T;

    void* d_table = nullptr;
    cudaError_t e = cudaMallocAsync(&d_table, host.size(), st);
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? SS_ENOMEM : ss::cuda_fail(e);
    e = cudaMemcpyAsync(d_table, host.data(), host.size(), cudaMemcpyHostToDevice, st);
    int rc = e == cudaSuccess ? SS_OK : ss::cuda_fail(e);
    const int64_t* d_prefix = static_cast<const int64_t*>(d_table);
    const void* const* d_ptrs =
        reinterpret_cast<const void* const*>(static_cast<unsigned char*>(d_table) + n_prefix * 8);
    for (int b = 0; rc == SS_OK && b < nb; ++b) {
        const int o_lo = bucket_start[b], o_hi = bucket_start[b + 1];
        const int64_t elems = prefix[o_hi] - prefix[o_lo];
        if (elems == 0) continue;
        bool any = false;
        for (int o = o_lo; o < o_hi && !any; ++o) any = numels[T - 1 - o] > 0 && needs_realign(ptrs, N, o);
        const DdpKernel fn = pick(N, any);
        const int64_t grid = (elems + kTile - 1) / kTile;
        if (grid > 0x7FFFFFFF) {
            rc = SS_EOVERFLOW;
            break;
        }
        cudaError_t le = launch_bucket(fn, (unsigned)grid, st, d_prefix, d_ptrs, N, o_lo, o_hi);
        rc = le == cudaSuccess ? ss::check_launch() : ss::cuda_fail(le);
    }
    cudaError_t ef = cudaFreeAsync(d_table, st);
    if (rc == SS_OK && ef != cudaSuccess) rc = ss::cuda_fail(ef);
    return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// allocation-free variant: the per-call table lives in a fixed device array
// ---------------------------------------------------------------------------

// Scratch for ddp_bucket_pack_average_noalloc: prefix sums then pointers, as
// the allocating entry point lays out its table.  Shared by every call.
static __device__ __align__(256) unsigned char g_ddp_noalloc_table[SS_DDP_NOALLOC_TABLE_BYTES];

namespace {

constexpr int kMaxDevicesNoalloc = 64;

// Device address of the array, looked up with the device current and kept per
// device together with the unique id of the CUDA context it was looked up in
// (host code cannot use the symbol itself: on the host it names a stand-in,
// not device memory).  A different context on the same device -- after
// cudaDeviceReset, or a context the caller made current -- loads its own copy
// of the library's module at another address, so a changed id means a new
// lookup.
struct NoallocAddr {
    unsigned long long ctx_id;
    void* addr;
};
std::mutex g_noalloc_mutex;
NoallocAddr g_noalloc_addr[kMaxDevicesNoalloc] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context, 0 if there is none or the
// driver cannot tell (then the address is looked up again on every call).
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

int noalloc_table_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ss::cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevicesNoalloc) return SS_EINVAL;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const unsigned long long id = current_ctx_id();
    NoallocAddr& c = g_noalloc_addr[dev];
    if (id == 0 || c.ctx_id != id || !c.addr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ddp_noalloc_table);
        if (e != cudaSuccess) return ss::cuda_fail(e);
        // the lookup makes the device's context current if none was
        c.ctx_id = current_ctx_id();
        c.addr = p;
    }
    *out = c.addr;
    return SS_OK;
}

}  // namespace

extern "C" int ddp_bucket_pack_average_noalloc(int world_size, int num_tensors,
                                               const int64_t* numels,
                                               const void* const* rank_grads,
                                               size_t bucket_cap_bytes, void* const* avg_out,
                                               int* num_buckets_out, ss_stream_t stream) {
    if (world_size < 1 || world_size > SS_MAX_WORLD || num_tensors < 0) return SS_EINVAL;
    if (num_tensors > 0 && (!numels || !rank_grads || !avg_out)) return SS_EINVAL;
    if (bucket_cap_bytes == 0) return SS_EINVAL;
    const int N = world_size, T = num_tensors;
    const size_t n_prefix = (size_t)T + 1;
    const size_t n_ptrs = (size_t)T * (size_t)(N + 1);
    const size_t table_bytes = n_prefix * 8 + n_ptrs * 8;
    if (table_bytes > SS_DDP_NOALLOC_TABLE_BYTES) return SS_ESCRATCH;
    for (int t = 0; t < T; ++t) {
        if (numels[t] < 0 || numels[t] > ((int64_t)1 << 60)) return SS_EINVAL;
        if (numels[t] == 0) continue;
        if (!avg_out[t]) return SS_EINVAL;
        if (!ss::aligned(avg_out[t], 2)) return SS_EALIGN;
        for (int r = 0; r < N; ++r) {
            const void* q = rank_grads[(size_t)r * T + t];
            if (!q) return SS_EINVAL;
            if (!ss::aligned(q, 2)) return SS_EALIGN;
        }
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (int crc = refuse_capture(st)) return crc;
    void* d_table = nullptr;
    int rc = noalloc_table_address(&d_table);
    if (rc) return rc;

    std::vector<int> bucket_of((size_t)(T > 0 ? T : 1));
    const int nb = ddp_bucket_assign(T, numels, 2, bucket_cap_bytes, bucket_of.data());
    if (nb < 0) return nb;
    if (num_buckets_out) *num_buckets_out = nb;
    if (nb == 0) return SS_OK;

    // table in bucket order (reverse registration order): prefix[T+1] then ptrs[T][N+1]
    std::vector<unsigned char> host(table_bytes);
    int64_t* prefix = reinterpret_cast<int64_t*>(host.data());
    const void** ptrs = reinterpret_cast<const void**>(host.data() + n_prefix * 8);
    std::vector<int> bucket_start((size_t)nb + 1, 0);
    prefix[0] = 0;
    for (int o = 0; o < T; ++o) {
        const int t = T - 1 - o;
        prefix[o + 1] = prefix[o] + numels[t];
        for (int r = 0; r < N; ++r) ptrs[(size_t)o * (N + 1) + r] = rank_grads[(size_t)r * T + t];
        ptrs[(size_t)o * (N + 1) + N] = avg_out[t];
        if (o == 0 || bucket_of[t] != bucket_of[t + 1]) bucket_start[bucket_of[t]] = o;
    }
    bucket_start[nb] = T;

    cudaError_t e = cudaMemcpyAsync(d_table, host.data(), table_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return ss::cuda_fail(e);
    const int64_t* d_prefix = static_cast<const int64_t*>(d_table);
    const void* const* d_ptrs =
        reinterpret_cast<const void* const*>(static_cast<unsigned char*>(d_table) + n_prefix * 8);
    for (int b = 0; b < nb; ++b) {
        const int o_lo = bucket_start[b], o_hi = bucket_start[b + 1];
        const int64_t elems = prefix[o_hi] - prefix[o_lo];
        if (elems == 0) continue;
        bool any = false;
        for (int o = o_lo; o < o_hi && !any; ++o) any = numels[T - 1 - o] > 0 && needs_realign(ptrs, N, o);
        const DdpKernel fn = pick(N, any);
        const int64_t grid = (elems + kTile - 1) / kTile;
        if (grid > 0x7FFFFFFF) return SS_EOVERFLOW;
        cudaError_t le = launch_bucket(fn, (unsigned)grid, st, d_prefix, d_ptrs, N, o_lo, o_hi);
        rc = le == cudaSuccess ? ss::check_launch() : ss::cuda_fail(le);
        if (rc) return rc;
    }
    return SS_OK;
}
