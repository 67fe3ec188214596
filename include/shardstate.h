/*
 * shardstate.h -- C ABI of the GB300 (sm_103a) sharded-state step of FSDP /
 * ZeRO-3 data parallelism, with N virtual data-parallel ranks held as N
 * buffers in one GPU's HBM.
 *
 * One training step of a fully sharded data-parallel group, as the pages
 * describe it ("Scaling data parallel", sections 9.1-9.3; "FSDP1 vs FSDP2",
 * sections 03-04; "ai-infra-kb M036", section 04 layer lifecycle):
 *   1. every rank's gradient is laid out in the group's sharded layout
 *      (fsdp_pack);
 *   2. a reduce-scatter leaves rank s the mean over ranks of its 1/N shard,
 *      and each rank runs mixed-precision AdamW on its own shard of the fp32
 *      master weights and moments, writing its bf16 parameter shard
 *      (fsdp_reduce_scatter_adamw, one fused pass);
 *   3. an all-gather returns the full parameters, read back out per
 *      parameter (fsdp_all_gather_unpack).
 * DDP's bucketed gradient all-reduce sits beside it
 * (ddp_bucket_pack_average).
 *
 * Conventions for every call:
 *   - Status: 0 (SS_OK) or a negative SS_E* code; ss_strerror() names it.
 *     Argument errors are detected on the host before anything is launched.
 *     SS_ECUDA means a CUDA runtime call failed; ss_last_cuda_error() returns
 *     that cudaError_t value for the calling thread.
 *   - Device pointers are plain device addresses on the current CUDA device.
 *     A plan's metadata lives on the device that was current when it was
 *     created; launching calls made with another device current return
 *     SS_EINVAL.
 *     The caller owns all of them; the library never frees or keeps them.
 *   - Launches are asynchronous on the caller's stream (NULL = the legacy
 *     default stream).  Nothing synchronises except plan creation, which
 *     copies the plan's metadata to the device before it returns.
 *   - Pointer arrays (params, rank_grads, params_out, avg_out) are HOST
 *     arrays of device pointers; they are read during the call and may be
 *     reused as soon as it returns.
 *   - The arithmetic never traps: no device-side assert, no trap, and no
 *     kernel waits on another.
 *
 * Element types: elem_bytes 2 = bf16 (gradients, parameters, shards),
 * elem_bytes 4 = fp32.  Optimizer state is always fp32.
 */
#ifndef SHARDSTATE_H
#define SHARDSTATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* ss_stream_t;

enum {
    SS_OK = 0,
    SS_EINVAL = -1,    /* bad argument: null pointer, size, world size, dtype, index */
    SS_EALIGN = -2,    /* pointer not aligned as the call requires */
    SS_EOVERFLOW = -3, /* a size overflows int64 / the index types */
    SS_ENOMEM = -4,    /* host or device allocation failed */
    SS_ECUDA = -5,     /* a CUDA runtime call failed (ss_last_cuda_error) */
    SS_ENODEVICE = -6, /* the plan has no device metadata (created host-only) */
    SS_ESCRATCH = -7   /* the call needs more than the library's fixed scratch array */
};

/* Largest N (virtual ranks) the kernels accept. */
#define SS_MAX_WORLD 64
/* Largest number of output replicas fsdp_all_gather_unpack writes per call. */
#define SS_MAX_REPLICAS 64

/*
 * Sharded layouts ("FSDP1 vs FSDP2", section 03, and its 3+5-element table).
 *  SS_FLAT_ORIG_FALSE  FSDP1 FlatParameter, use_orig_params=False (default):
 *                      plain concatenation (length L), torch.chunk(N), every
 *                      rank padded to c = ceil(L/N).
 *  SS_FLAT_ORIG_TRUE   FSDP1 FlatParameter, use_orig_params=True: from the
 *                      2nd parameter on, zero padding so it starts on a 16-byte
 *                      boundary (at most 16/elem_bytes - 1 elements), then the
 *                      buffer padded to a multiple of N; c = padded length / N.
 *  SS_PER_PARAM_DIM0   FSDP2 per-parameter DTensor(Shard(0)): parameter i is
 *                      split on dim 0 into chunks of c_i = ceil(d0_i/N) rows
 *                      (an empty parameter gives empty chunks); rank r's shard
 *                      concatenates its (padded) chunk of every parameter of
 *                      the group, S = sum_i c_i * inner_i.
 */
typedef enum {
    SS_FLAT_ORIG_FALSE = 0,
    SS_FLAT_ORIG_TRUE = 1,
    SS_PER_PARAM_DIM0 = 2
} ss_layout;

/* Opaque plan: layout metadata on the host plus its device copy. */
typedef struct ss_plan ss_plan;

/* Plan creation flag: compute the layout on the host only (no device
 * allocation or copy).  Such a plan answers the query calls; launching calls
 * return SS_ENODEVICE. */
#define SS_PLAN_HOST_ONLY 1u

/*
 * Description of a plan.  Parameters are numbered 0..num_params-1 in
 * registration order; parameter i has shape (dim0[i], inner[i]) where inner
 * is the product of the trailing dims (inner == NULL means 1 for all;
 * a 0-d parameter is (1, 1)).  Consecutive parameters form fully_shard groups
 * ("FSDP1 vs FSDP2", section 04: sharding unit = parameter, communication
 * unit = group): group g holds group_num_params[g] parameters.  num_groups 0
 * or group_num_params NULL means one group holding every parameter.  For the
 * FLAT layouts each group is one FlatParameter.
 */
typedef struct {
    ss_layout kind;
    int world_size;                /* N, 1..SS_MAX_WORLD */
    int elem_bytes;                /* 2 (bf16) or 4 (fp32) */
    int num_params;                /* >= 0 */
    const int64_t* dim0;           /* [num_params], each >= 0 */
    const int64_t* inner;          /* [num_params] or NULL, each >= 0 */
    int num_groups;                /* 0 = one group */
    const int* group_num_params;   /* [num_groups], summing to num_params */
    unsigned flags;                /* SS_PLAN_HOST_ONLY or 0 */
} ss_plan_desc;

/*
 * Packed-buffer geometry.  Every packed buffer of a plan (each rank's
 * gradients, the optimizer state, the parameter shards) has total_numel
 * elements.  Group g occupies [base_g, base_g + N*S_g); inside it rank r's
 * shard is [base_g + r*S_g, base_g + (r+1)*S_g).  For the FLAT layouts the N
 * shards of a group side by side are exactly the padded FlatParameter.
 */
typedef struct {
    int64_t shard_numel;     /* elements per rank, summed over groups */
    int64_t total_numel;     /* N * shard_numel */
    int64_t unpadded_numel;  /* sum of parameter numels */
    int64_t pad_numel;       /* total_numel - unpadded_numel */
    int world_size;
    int elem_bytes;
    int num_params;
    int num_groups;
    int kind;                /* ss_layout */
    int has_device_metadata; /* 0 for SS_PLAN_HOST_ONLY plans */
} ss_plan_info;

/* AdamW hyper-parameters for one step (decoupled weight decay), step t >= 1. */
typedef struct {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    int64_t step;
} ss_adamw;

/* ---------------------------------------------------------------------- */
/* plans                                                                   */
/* ---------------------------------------------------------------------- */

/* Build a plan ("FSDP1 vs FSDP2", section 03: padding and chunk rules; the
 * flat metadata of numels-with-padding and shapes that split the flat view
 * back into parameters).  Unless SS_PLAN_HOST_ONLY is set, the segment tables
 * are copied to the current device before the call returns.  *out receives
 * the plan; release it with fsdp_plan_destroy.  Errors: SS_EINVAL (sizes,
 * kind, world size, dtype, group counts), SS_EOVERFLOW (a size beyond int64),
 * SS_ENOMEM, SS_ECUDA. */
int fsdp_plan_create(const ss_plan_desc* desc, ss_plan** out);

/* One-group shorthand for fsdp_plan_create (device metadata included). */
int fsdp_plan_layout(ss_layout kind, int world_size, int elem_bytes, int num_params,
                     const int64_t* dim0, const int64_t* inner, ss_plan** out);

/* Geometry of a plan. */
int fsdp_plan_info(const ss_plan* plan, ss_plan_info* out);

/* Where parameter `param` lives in every packed buffer.  FLAT layouts: the
 * element index of its first element (its rank-r elements follow from
 * index / c).  PER_PARAM_DIM0: the element index of its chunk inside rank 0's
 * shard of its group; rank r's chunk is at that index + r*S_g.  chunk_rows_out
 * (nullable) receives c_i for PER_PARAM_DIM0 and 0 for the FLAT layouts. */
int fsdp_plan_param_offset(const ss_plan* plan, int param, int64_t* offset_out,
                           int64_t* chunk_rows_out);

/* Group geometry: base index, elements per rank (S_g or c_g), first parameter
 * and parameter count.  Any output pointer may be NULL. */
int fsdp_plan_group(const ss_plan* plan, int group, int64_t* base_out, int64_t* shard_numel_out,
                    int* first_param_out, int* num_params_out);

/* Self-check of a plan's host tables: every data run lies inside its
 * parameter and its group, the runs cover each parameter element exactly once,
 * data and pad runs tile every packed buffer [0, total_numel) with no gap or
 * overlap, and the tile tables split every run exactly.  The kernels index
 * device memory only through these tables, so a plan that passes keeps every
 * access in bounds.  SS_OK or SS_EINVAL. */
int fsdp_plan_validate(const ss_plan* plan);

/* Free a plan and its device metadata (NULL is a no-op).  The caller makes
 * sure no launch that uses the plan is still pending. */
void fsdp_plan_destroy(ss_plan* plan);

/* ---------------------------------------------------------------------- */
/* step                                                                    */
/* ---------------------------------------------------------------------- */

/*
 * Pack per-parameter tensors into the plan's sharded layout, zero-filling
 * every pad element ("FSDP1 vs FSDP2", section 03: FlatParameter
 * construction; FSDP2's copy-in of a group's shards into one collective
 * buffer).  Used for parameters at initialisation and, per step, for each
 * rank's gradients (the reduce-scatter input).
 *   params  HOST array [num_params] of device pointers; params[i] is the
 *           contiguous tensor of parameter i (numel dim0*inner, the plan's
 *           dtype, aligned to its element size).  Entries of parameters
 *           outside `group` are not read.
 *   packed  device buffer of total_numel elements, 16-byte aligned.  Only the
 *           selected group's range is written.
 *   group   -1 = every group, else one group index.
 * Errors: SS_EINVAL, SS_EALIGN, SS_ENODEVICE, SS_ECUDA.
 */
int fsdp_pack(const ss_plan* plan, const void* const* params, void* packed, int group,
              ss_stream_t stream);

/*
 * Optimizer-state initialisation on every rank's shard: master = the shard
 * widened to fp32, exp_avg = exp_avg_sq = 0 ("Scaling data parallel",
 * section 1: bf16 parameters with an fp32 master copy and fp32 Adam
 * moments).  param_shards: total_numel elements of the plan dtype; master,
 * exp_avg, exp_avg_sq: total_numel floats.  All 16-byte aligned.
 */
int fsdp_init_master(const ss_plan* plan, const void* param_shards, float* master,
                     float* exp_avg, float* exp_avg_sq, int group, ss_stream_t stream);

/*
 * Reduce-scatter of N virtual ranks' gradients fused with AdamW on each
 * rank's shard ("Scaling data parallel", sections 2.1 and 9.1-9.3: the
 * reduce-scatter leaves rank s the sum over ranks of shard s, divided by N
 * for the mean; each rank updates the fp32 master weights and Adam moments
 * of its own 1/N and casts them to bf16; "FSDP1 vs FSDP2", mixed precision:
 * the reduction runs in the reduce dtype, the cast to the parameter dtype
 * happens at the all-gather boundary).
 *
 * For every element f of the selected range (all ranks' shards):
 *   g = (G_0[f] + G_1[f] + ... + G_{N-1}[f]) / N
 * summed in fp32 in rank order starting from G_0, one IEEE fp32 division;
 * then decoupled AdamW (step t = hp->step >= 1):
 *   theta *= 1 - lr*wd;  m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g*g;
 *   theta -= (lr / (1-b1^t)) * m / (sqrt(v) / sqrt(1-b2^t) + eps);
 *   param_shards[f] = round-to-nearest-even bf16(theta)   (fp32 plans: theta)
 * in fp32 arithmetic.  Pads hold zero gradients and zero state, and stay zero.
 *
 *   rank_grads        HOST array [N] of device pointers; rank_grads[r] is rank
 *                     r's packed gradient buffer (total_numel elements of the
 *                     plan dtype, as fsdp_pack writes it).
 *   master, exp_avg, exp_avg_sq   total_numel floats, updated in place.
 *                     master may be NULL: the recipe without fp32 master
 *                     weights ("FSDP1 vs FSDP2" ledger: bf16 parameters and
 *                     gradients plus 8 B of Adam moments per parameter).
 *                     theta is then the parameter shard itself, widened to
 *                     fp32, updated, and rounded back in place (2N + 20 bytes
 *                     per element instead of 2N + 26).
 *   param_shards      total_numel elements of the plan dtype, written.
 *   hp                AdamW hyper-parameters; NULL = reduce-scatter only
 *                     (state and shards untouched; reduced_grad_out required).
 *   reduced_grad_out  nullable: total_numel floats receiving g.
 *   group             -1 = every group, else one group index.
 * All device buffers 16-byte aligned and indexed by the same element index.
 * Errors: SS_EINVAL, SS_EALIGN, SS_ENODEVICE, SS_ECUDA.
 */
int fsdp_reduce_scatter_adamw(const ss_plan* plan, const void* const* rank_grads, float* master,
                              float* exp_avg, float* exp_avg_sq, void* param_shards,
                              const ss_adamw* hp, float* reduced_grad_out, int group,
                              ss_stream_t stream);

/*
 * Reduce-scatter with gradient accumulation over num_micro micro-batches per
 * optimizer step ("Scaling data parallel", section 5: accumulate gradients
 * across micro-batches and synchronise once, using their mean; section 9.2:
 * with fp32 accumulation each rank keeps an fp32 gradient for its own shard
 * and adds every reduce-scatter result into it).  With RS_j the reduce-scatter
 * of micro-batch j (as fsdp_reduce_scatter_adamw computes it):
 *   micro_step 0:                 accum = RS_0
 *   0 < micro_step < num_micro-1: accum = accum + RS_j       (fp32)
 *   micro_step = num_micro-1:     g = (accum + RS_j) / num_micro, then AdamW
 *                                 exactly as fsdp_reduce_scatter_adamw
 *                                 (reduced_grad_out, if given, receives g)
 * num_micro = 1 is fsdp_reduce_scatter_adamw.  accum: total_numel floats
 * (16-byte aligned), left holding acc_{k-1} after the last micro-batch.
 * master may be NULL (no-master recipe).  bf16 plans only.
 * Errors: SS_EINVAL, SS_EALIGN, SS_ENODEVICE, SS_ECUDA.
 */
int fsdp_reduce_scatter_accumulate(const ss_plan* plan, const void* const* rank_grads,
                                   float* accum, int micro_step, int num_micro, float* master,
                                   float* exp_avg, float* exp_avg_sq, void* param_shards,
                                   const ss_adamw* hp, float* reduced_grad_out, int group,
                                   ss_stream_t stream);

/*
 * All-gather of the N rank shards followed by unpacking into full
 * per-parameter tensors, pads dropped ("FSDP1 vs FSDP2", section 03 figure:
 * the flat metadata splits the gathered flat view back into parameters;
 * FSDP2 gathers a group's shards in one collective and copies each parameter
 * out).  The all-gather delivers the full parameters to every rank; n_out
 * replicas are written (1 = the copy one rank sees, N = every rank's).
 *   param_shards  total_numel elements (16-byte aligned), rank-major.
 *   params_out    HOST array [n_out * num_params] of device pointers; replica
 *                 j of parameter i is params_out[j*num_params + i] (numel
 *                 dim0*inner, aligned to the element size).
 *   n_out         1..SS_MAX_REPLICAS.
 *   group         -1 = every group, else one group index.
 * Errors: SS_EINVAL, SS_EALIGN, SS_ENODEVICE, SS_ECUDA.
 */
int fsdp_all_gather_unpack(const ss_plan* plan, const void* param_shards,
                           void* const* params_out, int n_out, int group, ss_stream_t stream);

/*
 * The whole sharded step in one pass over the parameters: (copy-in) +
 * reduce-scatter + AdamW + (all-gather + unpack).  Same arithmetic as
 * fsdp_reduce_scatter_adamw followed by fsdp_all_gather_unpack, with
 * bit-identical results, but the kernel knows each element's place inside its
 * parameter (the plan's runs of one parameter inside one rank's shard), so in
 * one pass it can
 *   - read rank r's gradient either from its packed buffer (rank_grads[r],
 *     as fsdp_pack writes it) or straight from rank r's per-parameter
 *     gradient tensors (rank_param_grads[r*num_params + i]), fusing away the
 *     copy-in that FSDP does before its reduce-scatter ("FSDP1 vs FSDP2",
 *     section 04: a group's gradients are concatenated into one
 *     reduce-scatter buffer);
 *   - write each new bf16 parameter value both to its shard and to the n_out
 *     per-parameter outputs (the all-gather + unpack, no second pass over the
 *     shards).
 * Pad elements are not read or written (they stay as fsdp_pack /
 * fsdp_init_master left them: zero).  bf16 plans only.
 * Per-parameter gradients and outputs need only 2-byte alignment: a run at any
 * offset still moves in 16-byte vectors, one side aligned and the other
 * realigned in registers.  With n_out = N the call is the ZeRO-1/2 step
 * ("Scaling data parallel", sections 9.1-9.2): each rank updates its own 1/N
 * and the updated parameters reach every rank.
 */
typedef struct {
    const void* const* rank_grads;        /* HOST [N] packed buffers (16-byte aligned), or NULL */
    const void* const* rank_param_grads;  /* HOST [N * num_params] per-parameter gradients, or NULL;
                                             exactly one of the two is non-NULL */
    float* master;                        /* total_numel floats, updated in place */
    float* exp_avg;
    float* exp_avg_sq;
    void* param_shards;                   /* total_numel bf16, written */
    const ss_adamw* hp;                   /* required */
    float* reduced_grad_out;              /* nullable: total_numel floats (pads not written) */
    void* const* params_out;              /* HOST [n_out * num_params] outputs, or NULL if n_out == 0 */
    int n_out;                            /* 0..SS_MAX_REPLICAS; 0 = no all-gather */
} ss_step;

/* Per launch the pointer table holds (N if rank_param_grads else 0) + n_out
 * entries per parameter within 2048 slots; more parameters are split into
 * launches over consecutive parameters.  Every form runs in one pass and
 * allocates nothing.  Errors: SS_EINVAL (including both or neither gradient
 * source, fp32 plans, (N + n_out) > 2048), SS_EALIGN, SS_ENODEVICE,
 * SS_ECUDA. */
int fsdp_sharded_step(const ss_plan* plan, const ss_step* step, int group, ss_stream_t stream);

/*
 * DDP bucketed gradient average ("Scaling data parallel", sections 3-4:
 * gradients become final last layer first, so tensors are taken in reverse
 * registration order; each joins the open bucket, and a bucket that holds at
 * least bucket_cap_bytes is full and goes out as one all-reduce, the mean
 * over ranks).  For every element of every tensor:
 *   avg_out[t][k] = bf16_rne((g_0 + g_1 + ... + g_{N-1}) / N)
 * summed in fp32 in rank order.  One kernel launch per bucket, in bucket
 * order, so the per-collective fixed cost the pages describe is visible.
 *   world_size    N, 1..SS_MAX_WORLD.
 *   numels        HOST array [num_tensors], each >= 0.
 *   rank_grads    HOST array [N * num_tensors] of device pointers; rank r's
 *                 gradient of tensor t is rank_grads[r*num_tensors + t]
 *                 (bf16, 2-byte aligned).
 *   bucket_cap_bytes  > 0.
 *   avg_out       HOST array [num_tensors] of device pointers (bf16 outputs).
 *   num_buckets_out   nullable: receives the bucket count.
 * The call stages a per-call table of pointers and sizes in device memory
 * obtained with cudaMallocAsync on `stream` and released with cudaFreeAsync
 * after the launches.  The table is copied there from host memory that lives
 * only for the call, so a stream that is being captured into a CUDA graph is
 * refused with SS_EINVAL before anything is queued.
 * Errors: SS_EINVAL, SS_EALIGN, SS_ENOMEM, SS_ECUDA.
 */
int ddp_bucket_pack_average(int world_size, int num_tensors, const int64_t* numels,
                            const void* const* rank_grads, size_t bucket_cap_bytes,
                            void* const* avg_out, int* num_buckets_out, ss_stream_t stream);

/*
 * Allocation-free variant of ddp_bucket_pack_average.  No counterpart on the
 * pages: it exists for callers that cannot call cudaMalloc or
 * cudaMallocAsync -- a host framework that owns every byte of device memory
 * through its own allocator and forbids allocations behind its back, a
 * latency-critical loop that must not risk an allocation that grows a memory
 * pool or synchronises, or a process running so close to its device-memory
 * limit that an allocation could fail in the middle of a step.
 *
 * Same arguments, arithmetic, bucket order and launches as
 * ddp_bucket_pack_average; only the per-call table of pointers and sizes
 * lives in a fixed array inside the library (a static __device__ array of
 * SS_DDP_NOALLOC_TABLE_BYTES that every GPU loading the library holds until
 * the process exits) instead of a cudaMallocAsync allocation.  The table
 * takes 8 * (num_tensors + 1) + 8 * num_tensors * (world_size + 1) bytes; a
 * call that needs more returns SS_ESCRATCH before doing anything.
 *
 * The call allocates no device memory and calls no allocating library
 * routine.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it together with
 * the id of the current CUDA context; a call under another context (after
 * cudaDeviceReset, say) looks it up again.  As for ddp_bucket_pack_average,
 * the table is copied from host memory that lives only for the call, so a
 * stream that is being captured is refused with SS_EINVAL.  Every call
 * overwrites the whole table it uses, so nothing has to be cleared between
 * calls, and calls queued one after another on one stream are ordered by it.
 * All calls share the one array, though: calls whose work can overlap on the
 * GPU (different streams without ordering between them, or several host
 * threads) race on it and must be serialised by the caller.
 */
#define SS_DDP_NOALLOC_TABLE_BYTES (256u * 1024u)
int ddp_bucket_pack_average_noalloc(int world_size, int num_tensors, const int64_t* numels,
                                    const void* const* rank_grads, size_t bucket_cap_bytes,
                                    void* const* avg_out, int* num_buckets_out,
                                    ss_stream_t stream);

/* Bucket assignment only (host, no device work): bucket_of[t] receives
 * tensor t's bucket, numbered in launch order.  Returns the bucket count, or
 * a negative SS_E* status. */
int ddp_bucket_assign(int num_tensors, const int64_t* numels, int elem_bytes,
                      size_t bucket_cap_bytes, int* bucket_of);

/* ---------------------------------------------------------------------- */
/* diagnostics                                                             */
/* ---------------------------------------------------------------------- */

/* Static description of a status code. */
const char* ss_strerror(int status);

/* cudaError_t recorded by the last SS_ECUDA returned on this thread (0 if none). */
int ss_last_cuda_error(void);

/* Library version, e.g. "0.1.0". */
const char* ss_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads), for accounting launches inside a timed region. */
uint64_t ss_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SHARDSTATE_H */
