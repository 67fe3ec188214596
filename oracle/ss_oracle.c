/*
 * ss_oracle.c -- plain, slow, obviously correct CPU oracle for the FSDP /
 * ZeRO-3 sharded-state step (layout, pack, reduce-scatter, AdamW on the
 * local shard, all-gather + unpack, DDP bucketed average).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA product path
 * never links, loads or calls it, and it shares no code, header, table or
 * helper with that path.
 *
 * Every loop below is the definition written out, element by element, in the
 * order the pages state it.  Floating point: the reduce-scatter is fixed by
 * the spec to fp32 accumulation in rank order followed by a division by N;
 * AdamW is evaluated in fp64 from the fp32 state and rounded once to the fp32
 * storage precision; bf16 outputs are round-to-nearest-even of the fp32
 * value.  Build with -ffp-contract=off so no multiply-add is fused.
 *
 * Parity is pinned for every function here (see the -m "not gpu" tests):
 * layouts against torch.chunk and a brute-force slot simulation, the printed
 * 3+5-element example, pack/unpack round trips, the reduce-scatter against an
 * exact mean and a hand-computed order-dependent sum, AdamW against
 * torch.optim.AdamW in fp64 and its t=1 closed form, bf16 rounding against
 * torch's cast, and bucket assignment against brute force.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float arithmetic evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

#define SSO_FLAT_ORIG_FALSE 0
#define SSO_FLAT_ORIG_TRUE 1
#define SSO_PER_PARAM_DIM0 2

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */

/* Number of host threads the element loops may use (1 = the definitional,
 * single-threaded oracle).  Every parallel loop is over independent output
 * elements, so the result does not depend on the thread count. */
static int g_threads = 1;

void sso_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

int sso_get_threads(void) { return g_threads; }

int sso_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32, so widening is exact. */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to the even bf16.  Written from
 * the definition: keep the upper 16 bits; the dropped lower 16 bits decide.
 * More than half an ulp rounds up, less rounds down, exactly half rounds to
 * the candidate whose last kept bit is 0.  NaNs stay NaN (quiet bit set);
 * infinities and overflow to infinity follow from the carry. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t exp_bits = (u >> 23) & 0xFFu;
    uint32_t mant = u & 0x7FFFFFu;
    if (exp_bits == 0xFFu && mant != 0) {
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t upper = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    uint32_t half = 0x8000u;
    if (dropped > half || (dropped == half && (upper & 1u))) {
        upper += 1u; /* a carry into the exponent is the correct rounding */
    }
    return (uint16_t)upper;
}

void sso_bf16_round(int64_t count, const float* in, uint16_t* out) {
#pragma omp parallel for num_threads(g_threads) schedule(static)
    for (int64_t k = 0; k < count; ++k) out[k] = f32_to_bf16_rne(in[k]);
}

void sso_bf16_widen(int64_t count, const uint16_t* in, float* out) {
    for (int64_t k = 0; k < count; ++k) out[k] = bf16_to_f32(in[k]);
}

/* ------------------------------------------------------------------------ */
/* layout planning                                                           */
/* ------------------------------------------------------------------------ */

static int64_t numel_of(const int64_t* dim0, const int64_t* inner, int i) {
    return dim0[i] * (inner ? inner[i] : 1);
}

/*
 * Layout of one fully_shard group / one FlatParameter.
 *
 * FLAT_ORIG_TRUE ("FSDP1 vs FSDP2", section 03, FlatParameter with
 *   use_orig_params=True): parameters are concatenated into one flat 1-D
 *   buffer; from the second parameter on, zero padding is inserted before a
 *   parameter until its start lies on a 16-byte boundary (a = 16/elem_bytes
 *   elements, so at most a-1 pad elements); the whole buffer is then padded
 *   to a multiple of N so every rank's chunk has the same length.
 * FLAT_ORIG_FALSE (same section, the default use_orig_params=False): plain
 *   concatenation, no alignment and no world padding; the flat buffer is split
 *   with torch.chunk(N), and each chunk is padded to chunks[0].numel(), so
 *   every rank holds ceil(L/N) elements.
 * PER_PARAM_DIM0 (same page, FSDP2 per-parameter DTensor(Shard(0))): each
 *   parameter is chunked on dim 0 into pieces of ceil(d0/N) rows, padded per
 *   parameter; an empty parameter still yields (empty) chunks.  A rank's
 *   storage is its piece of every parameter, and the group concatenates those
 *   pieces into one collective buffer ("sharding unit = parameter,
 *   communication unit = group").
 *
 * Outputs: offset[i] = FLAT: element offset of parameter i inside the padded
 * flat buffer; PER_PARAM: element offset of parameter i's chunk inside one
 * rank's shard.  chunk_rows[i] = ceil(d0_i/N) for PER_PARAM, 0 for FLAT.
 * shard_numel = elements per rank (c or S).  unpadded = sum of numels.
 * Returns 0, or -1 on bad arguments.
 */
int sso_layout(int kind, int N, int elem_bytes, int n, const int64_t* dim0, const int64_t* inner,
               int64_t* offset, int64_t* chunk_rows, int64_t* shard_numel, int64_t* unpadded) {
    if (N < 1 || n < 0 || (elem_bytes != 2 && elem_bytes != 4)) return -1;
    if (n > 0 && !dim0) return -1;
    for (int i = 0; i < n; ++i)
        if (dim0[i] < 0 || (inner && inner[i] < 0)) return -1;

    int64_t total_unpadded = 0;
    for (int i = 0; i < n; ++i) total_unpadded += numel_of(dim0, inner, i);
    if (unpadded) *unpadded = total_unpadded;

    if (kind == SSO_FLAT_ORIG_TRUE) {
        int64_t a = 16 / elem_bytes;
        int64_t pos = 0;
        for (int i = 0; i < n; ++i) {
            if (i > 0) {
                while (pos % a != 0) pos += 1; /* alignment pad before param i */
            }
            if (offset) offset[i] = pos;
            if (chunk_rows) chunk_rows[i] = 0;
            pos += numel_of(dim0, inner, i);
        }
        while (pos % N != 0) pos += 1; /* world-size pad */
        *shard_numel = pos / N;
        return 0;
    }
    if (kind == SSO_FLAT_ORIG_FALSE) {
        int64_t pos = 0;
        for (int i = 0; i < n; ++i) {
            if (offset) offset[i] = pos;
            if (chunk_rows) chunk_rows[i] = 0;
            pos += numel_of(dim0, inner, i);
        }
        /* torch.chunk(N) uses chunks of ceil(L/N); each rank pads to chunks[0] */
        *shard_numel = (pos + N - 1) / N;
        return 0;
    }
    if (kind == SSO_PER_PARAM_DIM0) {
        int64_t pos = 0;
        for (int i = 0; i < n; ++i) {
            int64_t rows = (dim0[i] + N - 1) / N;
            int64_t in = inner ? inner[i] : 1;
            if (offset) offset[i] = pos;
            if (chunk_rows) chunk_rows[i] = rows;
            pos += rows * in;
        }
        *shard_numel = pos;
        return 0;
    }
    return -1;
}

/* ------------------------------------------------------------------------ */
/* pack (per-parameter tensors -> N rank shards, rank-major)                 */
/* ------------------------------------------------------------------------ */

/*
 * Write the N rank shards of one group, rank r's shard at [r*c, (r+1)*c), with
 * every pad element zero.
 *
 * FLAT layouts: rank r's shard is elements [r*c, (r+1)*c) of the padded flat
 * buffer (torch.chunk of the flat parameter, "FSDP1 vs FSDP2" section 03 and
 * its figure: a chunk may hold the tail of one parameter, pad and the head of
 * the next), so the N shards side by side are the padded flat buffer itself.
 * PER_PARAM_DIM0: rank r holds rows [r*c_i, min((r+1)*c_i, d0_i)) of every
 * parameter i, each parameter's piece padded to c_i rows.
 */
int sso_pack(int kind, int N, int elem_bytes, int n, const int64_t* dim0, const int64_t* inner,
             const void* const* params, void* packed) {
    int64_t* off = (int64_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    int64_t* rows = (int64_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    int64_t c = 0, L = 0;
    int rc = sso_layout(kind, N, elem_bytes, n, dim0, inner, off, rows, &c, &L);
    if (rc != 0) { free(off); free(rows); return rc; }
    unsigned char* out = (unsigned char*)packed;
    const size_t e = (size_t)elem_bytes;
    memset(out, 0, (size_t)(N * c) * e);

    if (kind == SSO_FLAT_ORIG_TRUE || kind == SSO_FLAT_ORIG_FALSE) {
        for (int i = 0; i < n; ++i) {
            const unsigned char* src = (const unsigned char*)params[i];
            int64_t s = numel_of(dim0, inner, i);
            for (int64_t k = 0; k < s; ++k)
                memcpy(out + (size_t)(off[i] + k) * e, src + (size_t)k * e, e);
        }
    } else {
        for (int r = 0; r < N; ++r) {
            for (int i = 0; i < n; ++i) {
                const unsigned char* src = (const unsigned char*)params[i];
                int64_t in = inner ? inner[i] : 1;
                int64_t lo = (int64_t)r * rows[i];
                int64_t hi = lo + rows[i];
                if (hi > dim0[i]) hi = dim0[i];
                for (int64_t row = lo; row < hi; ++row) {
                    for (int64_t col = 0; col < in; ++col) {
                        int64_t dst = (int64_t)r * c + off[i] + (row - lo) * in + col;
                        memcpy(out + (size_t)dst * e, src + (size_t)(row * in + col) * e, e);
                    }
                }
            }
        }
    }
    free(off);
    free(rows);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* all-gather + unpack (N rank shards -> full per-parameter tensors)         */
/* ------------------------------------------------------------------------ */

/*
 * The all-gather hands every rank the concatenation of all N shards; the
 * parameters are then read back out of that buffer ("FSDP1 vs FSDP2": the
 * flat metadata splits the flat view back into the original shapes; FSDP2
 * copies each parameter's rows out of the group buffer).  The N shards are
 * given rank-major in one buffer, which is already the gathered buffer.
 *
 * For element k of parameter i:
 *   FLAT: flat index f = offset_i + k; owner rank f / c, local index f % c.
 *   PER_PARAM: row rho = k / inner_i; owner rank rho / c_i; local row
 *              rho % c_i inside that rank's chunk of parameter i.
 * params_out holds n_out replicas: replica j of parameter i is
 * params_out[j*n + i].
 */
int sso_all_gather_unpack(int kind, int N, int elem_bytes, int n, const int64_t* dim0,
                          const int64_t* inner, const void* shards, void* const* params_out,
                          int n_out) {
    int64_t* off = (int64_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    int64_t* rows = (int64_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    int64_t c = 0, L = 0;
    int rc = sso_layout(kind, N, elem_bytes, n, dim0, inner, off, rows, &c, &L);
    if (rc != 0 || n_out < 1) { free(off); free(rows); return rc ? rc : -1; }
    const unsigned char* gathered = (const unsigned char*)shards;
    const size_t e = (size_t)elem_bytes;
    const int flat = (kind == SSO_FLAT_ORIG_TRUE || kind == SSO_FLAT_ORIG_FALSE);

    for (int i = 0; i < n; ++i) {
        int64_t s = numel_of(dim0, inner, i);
        int64_t in = inner ? inner[i] : 1;
        int64_t ci = rows[i];
        int64_t oi = off[i];
#pragma omp parallel for num_threads(g_threads) schedule(static)
        for (int64_t k = 0; k < s; ++k) {
            int64_t src_index;
            if (flat) {
                int64_t f = oi + k;
                int64_t owner = f / c;
                int64_t local = f % c;
                src_index = owner * c + local;
            } else {
                int64_t rho = k / in;
                int64_t col = k % in;
                int64_t owner = rho / ci;
                int64_t local_row = rho % ci;
                src_index = owner * c + oi + local_row * in + col;
            }
            for (int j = 0; j < n_out; ++j) {
                unsigned char* dst = (unsigned char*)params_out[(size_t)j * (size_t)n + (size_t)i];
                memcpy(dst + (size_t)k * e, gathered + (size_t)src_index * e, e);
            }
        }
    }
    free(off);
    free(rows);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* reduce-scatter                                                            */
/* ------------------------------------------------------------------------ */

/*
 * Reduce-scatter of N equally laid out gradient buffers of N*c elements:
 * rank s receives shard s, the element-wise sum over ranks of elements
 * [s*c, (s+1)*c), divided by N to give the data-parallel mean gradient
 * ("Scaling data parallel", sections 2.1 and 9.1-9.3: all-reduce is sum then
 * divide by the DP size, reduce-scatter keeps each rank's 1/N of it).
 * The sum is taken in fp32 in rank order 0, 1, ..., N-1, starting from rank
 * 0's value, and the division is one IEEE fp32 division by N.
 * Inputs are bf16 (elem_bytes 2) or fp32 (elem_bytes 4).  out has N*c floats
 * (all ranks' shards side by side).
 */
void sso_reduce_scatter(int N, int64_t c, int elem_bytes, const void* const* rank_bufs,
                        float* out) {
    const float divisor = (float)N;
    for (int s = 0; s < N; ++s) {
#pragma omp parallel for num_threads(g_threads) schedule(static)
        for (int64_t j = 0; j < c; ++j) {
            int64_t f = (int64_t)s * c + j;
            float acc;
            if (elem_bytes == 2) {
                acc = bf16_to_f32(((const uint16_t*)rank_bufs[0])[f]);
                for (int r = 1; r < N; ++r) acc = acc + bf16_to_f32(((const uint16_t*)rank_bufs[r])[f]);
            } else {
                acc = ((const float*)rank_bufs[0])[f];
                for (int r = 1; r < N; ++r) acc = acc + ((const float*)rank_bufs[r])[f];
            }
            out[f] = acc / divisor;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* AdamW on the local shard                                                  */
/* ------------------------------------------------------------------------ */

/*
 * Mixed-precision AdamW on each rank's shard ("Scaling data parallel",
 * section 9.1: each rank updates the fp32 master copy and the Adam moments of
 * its own 1/N, then casts to bf16; "FSDP1 vs FSDP2": the optimizer updates the
 * original dtype, the cast to param_dtype happens at the all-gather boundary).
 * The pages name AdamW but do not print its formula; this is decoupled AdamW
 * (Loshchilov & Hutter), step t >= 1, m_0 = v_0 = 0:
 *   theta <- theta - lr*wd*theta
 *   m     <- b1*m + (1-b1)*g
 *   v     <- b2*v + (1-b2)*g*g
 *   mhat  =  m / (1 - b1^t),   vhat = v / (1 - b2^t)
 *   theta <- theta - lr * mhat / (sqrt(vhat) + eps)
 * evaluated in fp64 from the fp32 inputs and rounded once to fp32 storage.
 * param_out (nullable) receives the new parameter in the shard dtype: bf16
 * round-to-nearest-even of the fp32 master (elem_bytes 2) or the fp32 master
 * itself (elem_bytes 4).
 */
void sso_adamw(int64_t count, const float* grad, float* master, float* exp_avg,
               float* exp_avg_sq, void* param_out, int elem_bytes, double lr, double beta1,
               double beta2, double eps, double weight_decay, int64_t step) {
    const double bc1 = 1.0 - pow(beta1, (double)step);
    const double bc2 = 1.0 - pow(beta2, (double)step);
#pragma omp parallel for num_threads(g_threads) schedule(static)
    for (int64_t k = 0; k < count; ++k) {
        double g = (double)grad[k];
        double theta = (double)master[k];
        double m = (double)exp_avg[k];
        double v = (double)exp_avg_sq[k];
        theta = theta - lr * weight_decay * theta;
        m = beta1 * m + (1.0 - beta1) * g;
        v = beta2 * v + (1.0 - beta2) * g * g;
        double mhat = m / bc1;
        double vhat = v / bc2;
        theta = theta - lr * mhat / (sqrt(vhat) + eps);
        master[k] = (float)theta;
        exp_avg[k] = (float)m;
        exp_avg_sq[k] = (float)v;
        if (param_out) {
            if (elem_bytes == 2)
                ((uint16_t*)param_out)[k] = f32_to_bf16_rne(master[k]);
            else
                ((float*)param_out)[k] = master[k];
        }
    }
}

/* Optimizer-state initialisation for a fresh shard ("Scaling data parallel",
 * sections 1 and 9.1: bf16 parameters beside an fp32 master copy and fp32
 * Adam moments; Adam's moments start at zero): the fp32 master copy is the
 * widened parameter shard, both moments start at zero. */
void sso_init_master(int64_t count, const void* param_shards, int elem_bytes, float* master,
                     float* exp_avg, float* exp_avg_sq) {
    for (int64_t k = 0; k < count; ++k) {
        master[k] = elem_bytes == 2 ? bf16_to_f32(((const uint16_t*)param_shards)[k])
                                    : ((const float*)param_shards)[k];
        exp_avg[k] = 0.0f;
        exp_avg_sq[k] = 0.0f;
    }
}

/* The whole sharded step on one group's N*c elements: reduce-scatter of the N
 * gradient buffers, then AdamW on every rank's shard.  reduced_out (N*c
 * floats, nullable) receives the reduce-scatter result. */
void sso_reduce_scatter_adamw(int N, int64_t c, int elem_bytes, const void* const* rank_grads,
                              float* master, float* exp_avg, float* exp_avg_sq,
                              void* param_shards, float* reduced_out, double lr, double beta1,
                              double beta2, double eps, double weight_decay, int64_t step) {
    int64_t total = (int64_t)N * c;
    float* g = reduced_out ? reduced_out : (float*)malloc((size_t)(total > 0 ? total : 1) * sizeof(float));
    sso_reduce_scatter(N, c, elem_bytes, rank_grads, g);
    sso_adamw(total, g, master, exp_avg, exp_avg_sq, param_shards, elem_bytes, lr, beta1, beta2,
              eps, weight_decay, step);
    if (!reduced_out) free(g);
}

/* ------------------------------------------------------------------------ */
/* gradient accumulation over micro-batches                                  */
/* ------------------------------------------------------------------------ */

/*
 * Gradient accumulation ("Scaling data parallel", section 5 with section
 * 9.2): the k micro-batches of one optimizer step each produce a
 * reduce-scatter; with fp32 accumulation each rank keeps an fp32 buffer for
 * its own shard and adds every micro-batch's reduce-scatter result into it;
 * the optimizer uses the average over micro-batches (section 1: in practice
 * the mean, so the result does not depend on the number of steps).
 *   acc_1 = RS_1;  acc_j = acc_{j-1} + RS_j  (fp32, in micro-batch order)
 *   g = acc_k / k  (one IEEE fp32 division)
 * first != 0 starts a new accumulation (acc = RS), otherwise acc += RS.
 */
void sso_accumulate(int N, int64_t c, int elem_bytes, const void* const* rank_bufs, float* accum,
                    int first) {
    int64_t total = (int64_t)N * c;
    float* rs = (float*)malloc((size_t)(total > 0 ? total : 1) * sizeof(float));
    sso_reduce_scatter(N, c, elem_bytes, rank_bufs, rs);
    for (int64_t f = 0; f < total; ++f) accum[f] = first ? rs[f] : accum[f] + rs[f];
    free(rs);
}

void sso_accumulated_grad(int64_t count, const float* accum, int num_micro, float* grad) {
    const float k = (float)num_micro;
    for (int64_t f = 0; f < count; ++f) grad[f] = accum[f] / k;
}

/* ------------------------------------------------------------------------ */
/* DDP gradient bucketing                                                    */
/* ------------------------------------------------------------------------ */

/*
 * Bucket assignment ("Scaling data parallel", sections 3-4): gradients become
 * final last layer first, so tensors are visited in reverse registration
 * order; each is appended to the open bucket, and once the bucket holds at
 * least cap_bytes it is full, is sent as one all-reduce, and a new bucket
 * opens.  bucket_of[t] receives tensor t's bucket (buckets numbered in
 * launch order).  Returns the number of buckets.
 */
int sso_ddp_buckets(int T, const int64_t* numels, int elem_bytes, int64_t cap_bytes,
                    int* bucket_of) {
    int bucket = 0;
    int64_t fill = 0;
    for (int t = T - 1; t >= 0; --t) {
        bucket_of[t] = bucket;
        fill += numels[t] * elem_bytes;
        if (fill >= cap_bytes) {
            bucket += 1;
            fill = 0;
        }
    }
    return fill > 0 ? bucket + 1 : bucket;
}

/*
 * Gradient average of DDP: every rank ends with the mean over ranks of the
 * bf16 gradients ("Scaling data parallel", section 2.1: all-reduce sum, then
 * divide by N).  Sum in fp32 in rank order from rank 0, one fp32 division by
 * N, round to bf16.  The bucketing only groups tensors into collectives, so it
 * does not enter the values.  grads[r*T + t] is rank r's gradient of tensor t.
 */
void sso_ddp_average(int N, int T, const int64_t* numels, const uint16_t* const* grads,
                     uint16_t* const* out) {
    const float divisor = (float)N;
    for (int t = 0; t < T; ++t) {
#pragma omp parallel for num_threads(g_threads) schedule(static)
        for (int64_t k = 0; k < numels[t]; ++k) {
            float acc = bf16_to_f32(grads[t][k]);
            for (int r = 1; r < N; ++r) acc = acc + bf16_to_f32(grads[(size_t)r * (size_t)T + (size_t)t][k]);
            out[t][k] = f32_to_bf16_rne(acc / divisor);
        }
    }
}
