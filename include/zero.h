/*
 * zero.h -- C ABI of the GB300 sharded optimizer step (ZeRO-1/2/3 update).
 *
 * What the library computes.  N data-parallel ranks each hold a full padded
 * gradient buffer.  The gradients are reduce-scattered (summed over ranks in
 * rank order, divided by N): rank r receives slice r of every unit.  Each
 * rank runs AdamW on its own fp32 master/m/v slice, casts the result to bf16
 * and all-gathers it into the full parameter buffer.  An optional global
 * gradient-norm clip scales the averaged gradient first.
 *   - "ZeRO and FSDP sharding", How it works: per-unit flat buffers padded to a
 *     multiple of N, rank r owns slice r; the step is AdamW on the fp32 master
 *     slice, a cast to bf16, and one all-gather of the updated params.
 *   - "ZeRO and FSDP sharding", Code: the reduce-scatter, the division by n,
 *     AdamW::step and the all-gather; the sharded result equals unsharded
 *     AdamW on the averaged gradient bit for bit.
 *   - "ZeRO: Three Ledgers, Zero Redundancy", section 2: all-reduce =
 *     reduce-scatter + local update + all-gather; the clip norm is a
 *     decomposable sum of squares.
 *   - "ZeRO and FSDP sharding", Implementation notes: clipping needs the global
 *     norm; gradients reduced in fp32, weights gathered in bf16.
 *
 * The N ranks live on ONE GPU as N resident HBM buffers: rank q's "send
 * buffer" is its gradient buffer, the reduce-scatter is a kernel that reads
 * all N buffers at the same offset, and the all-gather is the same kernel
 * writing the rank's slice into the full buffer.
 *
 * Arithmetic: every float operation of the update is one IEEE binary32
 * operation rounded to nearest even, in the order
 *     g = (((g_0 + g_1) + g_2) + ... + g_{N-1}) / N          [* coef]
 *     m = (b1*m) + ((1-b1)*g)
 *     v = (b2*v) + (((1-b2)*g)*g)
 *     w = (w*(1-lr*wd)) - (((lr/bc1)*m) / ((sqrt(v)/bc2) + eps))
 *     bc1 = 1 - b1^t, bc2 = sqrt(1 - b2^t), b^t by binary exponentiation in
 *     binary32 (computed on the host, once per call),
 * and the bf16 output is w rounded to nearest even (a NaN stays a NaN with its
 * sign).  Results are bit-identical to that sequence; nothing is fused.
 *
 * Layout (all counts in elements).  For unit u of s_u parameters:
 *   S_u = s_u rounded up to a multiple of N, h_u = S_u / N,
 *   F_u = sum_{k<u} S_k (unit offset in the full buffer),
 *   Hoff_u = sum_{k<u} h_k (unit offset in every rank's shard buffer),
 *   P_pad = sum S_u, H = P_pad / N.
 * Rank r owns full positions [F_u + r*h_u, F_u + (r+1)*h_u) of unit u, stored
 * at [Hoff_u, Hoff_u + h_u) of its shard buffers.  Gradient and full buffers
 * have P_pad elements; master/m/v/param-shard/grad-shard buffers have H.
 * Full positions F_u + k with k >= s_u are padding: their gradient entries are
 * never read (they count as 0), and the update runs on them like on any other
 * position (pads initialised to 0 stay exactly 0).
 *
 * Conventions.
 *   - Every function returns a status (ZERO_OK = 0, negative on error) and
 *     checks all arguments on the host before anything is launched; on error
 *     nothing is launched and no memory is touched.
 *   - The caller owns all device memory and streams (PyTorch allocates them).
 *     The library owns only the opaque plan (host memory); its device tables
 *     live in a caller-provided workspace (zero_plan_attach).
 *   - Device work is asynchronous on the given stream (NULL = legacy default
 *     stream).  Calls that use the same plan's workspace must be ordered on one
 *     stream, or otherwise serialised by the caller.  Every call that updates,
 *     reduces or scatters (everything but the gathers, the norm without a
 *     plan and the reshard) hands its work out to the GPU's SMs from a counter
 *     in the workspace; two such calls on one plan running at the same time
 *     would take work from each other and leave parts undone.  The counter is
 *     back at zero when each call's kernel ends, so captured calls replay
 *     correctly from a CUDA graph.
 *   - Arrays of rank pointers ("[N]") are HOST arrays of N DEVICE pointers.
 *     Every device pointer must be 16-byte aligned (ZERO_EALIGN otherwise).
 *   - A plan is immutable after zero_plan_attach and may be shared by threads
 *     that serialise their device work.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct zero_plan zero_plan;
typedef struct CUstream_st *zero_stream_t; /* the same type as cudaStream_t */

enum {
    ZERO_OK = 0,
    ZERO_EINVAL = -1,      /* a bad argument (null, out of range, wrong dtype, size mismatch) */
    ZERO_ENOMEM = -2,      /* host allocation failed, or the workspace is too small */
    ZERO_ECUDA = -3,       /* a CUDA runtime call failed (launch, copy, device query) */
    ZERO_EALIGN = -4,      /* a device pointer is not 16-byte aligned */
    ZERO_ENONFINITE = -5,  /* zero_plan_check: a clipped step was skipped, its global norm was inf/NaN */
    ZERO_ETIMEOUT = -6,    /* zero_plan_check: a bounded wait inside a kernel expired */
    ZERO_ENOTATTACHED = -7, /* the plan has no device workspace yet (zero_plan_attach) */
    ZERO_ERANGE = -8        /* a size beyond a fixed capacity (zero_grad_sqnorm_noalloc) */
};

enum { ZERO_F32 = 0, ZERO_BF16 = 1 };

#define ZERO_MAX_RANKS 64

/* AdamW hyper-parameters of one step ("ZeRO and FSDP sharding", Code,
 * AdamW::step).  t is the 1-based step number.  max_norm > 0 turns on the
 * global-norm clip: coef = min(1, max_norm / (sqrt(S) + 1e-6)) in binary64,
 * rounded once to binary32, where S is the sum of squares of the averaged
 * gradient over all ranks and positions (pads count 0). */
typedef struct {
    float lr, b1, b2, eps, wd;
    int32_t t;
    float max_norm;
} zero_hparams;

/* ---------------------------------------------------------------- plan */

/* Build the padded layout of n_units units for n_ranks simulated ranks
 * ("ZeRO and FSDP sharding", How it works and Pitfalls: pad each flat unit
 * to a multiple of N).  Host only; needs no GPU.  unit_sizes: host array of
 * n_units non-negative counts (zero-sized units are allowed).  1 <= n_ranks
 * <= ZERO_MAX_RANKS.  On success *out owns a plan freed by zero_plan_destroy.
 * Errors: ZERO_EINVAL (bad sizes, n_ranks out of range, total beyond 2^62),
 * ZERO_ENOMEM. */
int zero_plan_create(const int64_t *unit_sizes, int32_t n_units, int32_t n_ranks, zero_plan **out);

/* zero_plan_create with an alignment option the pages leave open: every unit is
 * padded to a multiple of N * align instead of N, so every slice length h_u,
 * and with it every slice's offset in the full and the shard buffers, is a
 * multiple of align elements.  align = 8 puts every bf16 slice on a 16-byte
 * boundary (the kernels then never read a gradient row at a shifted offset);
 * the cost is at most N * align - 1 more padding positions per unit.  align = 1
 * is zero_plan_create.  1 <= align <= ZERO_MAX_ALIGN.  Every other call works
 * on an aligned plan unchanged; zero_reshard maps between plans of any
 * alignment.  Errors: as zero_plan_create. */
#define ZERO_MAX_ALIGN 4096
int zero_plan_create_aligned(const int64_t *unit_sizes, int32_t n_units, int32_t n_ranks, int32_t align,
                             zero_plan **out);

/* The plan's alignment option (1 for zero_plan_create). */
int zero_plan_align(const zero_plan *plan, int32_t *align);

/* Frees the plan (host memory only; the caller frees its workspace). NULL is a no-op. */
void zero_plan_destroy(zero_plan *plan);

/* Layout query.  Scalars and arrays are HOST memory; every pointer may be NULL.
 * p_pad, h: P_pad and H.  F, Hoff, S, h_u: arrays of n_units (unit offsets in
 * the full buffer, in the shard buffers, padded sizes, slice lengths). */
int zero_plan_query(const zero_plan *plan, int64_t *p_pad, int64_t *h, int64_t *F, int64_t *Hoff,
                    int64_t *S, int64_t *h_u);

/* Counts: units, ranks, and the number of work segments of the multi-unit
 * launch table (a segment is a contiguous run of one rank's slice). */
int zero_plan_counts(const zero_plan *plan, int32_t *n_units, int32_t *n_ranks, int64_t *n_segments);

/* The launch table, for inspection: out (HOST, 6 * n_segments int64) receives
 * per segment {full position, shard position, length, valid (non-pad) length,
 * rank, unit}.  Segments are ordered by unit, then rank, then position. */
int zero_plan_segments(const zero_plan *plan, int64_t *out);

/* The unit-local launch table, for inspection: the same slices cut so that each
 * unit has about 304 segments (two per SM of a GB300) of at least 1024 elements
 * and at most the main table's length.  Launches over one unit or a run of units
 * that keep no per-segment partial sums use it (zero_step with unit >= 0,
 * zero_step_unit, zero_step_units, zero_reduce_scatter_unit, the per-unit
 * zero_adamw_shard_step_clipped and all-gathers), so a small unit spreads over
 * every SM; results do not depend on the cut.  *n_segments (HOST) receives its
 * length; out (HOST, 6 * that many int64, may be NULL) receives the segments in
 * the layout of zero_plan_segments. */
int zero_plan_local_segments(const zero_plan *plan, int64_t *n_segments, int64_t *out);

/* Bytes of device workspace the plan needs (both work tables, per-segment
 * partial sums, scalars). Host only. */
int zero_plan_workspace_bytes(const zero_plan *plan, size_t *bytes);

/* Binds the plan to the current device: copies its work table into the
 * caller's device workspace (>= zero_plan_workspace_bytes bytes, 256-byte
 * aligned) on `stream`.  The workspace must outlive every later call with
 * this plan.  Call once, before any stream capture.  Errors: ZERO_EINVAL (NULL,
 * already attached), ZERO_ENOMEM (too small), ZERO_EALIGN, ZERO_ECUDA. */
int zero_plan_attach(zero_plan *plan, void *workspace, size_t bytes, zero_stream_t stream);

/* The host recipe for the bias corrections (t >= 1): bc1 = 1 - b1^t,
 * bc2 = sqrt(1 - b2^t), b^t by binary exponentiation in binary32.  Every
 * device call below uses exactly these values. */
int zero_bias_corrections(int32_t t, float b1, float b2, float *bc1, float *bc2);

/* ---------------------------------------------------------------- steps of the path */

/* Reduce-scatter + average ("ZeRO and FSDP sharding", Code: reduce_scatter,
 * then /= n): gshard[r][Hoff_u + j] = (sum_q grads[q][F_u + r h_u + j]) / N
 * (rank-ordered fold, fp32), times coef when coef != 1 (pass 1.0f for none).
 * grads: [N] device buffers of P_pad elements of gdtype (ZERO_BF16 or
 * ZERO_F32).  gshard: [N] device fp32 buffers of H elements (output).
 * Pads of a unit write 0. */
int zero_reduce_scatter(const zero_plan *plan, const void *const *grads, int32_t gdtype,
                        float *const *gshard, float coef, zero_stream_t stream);

/* Global squared gradient norm ("ZeRO and FSDP sharding", Implementation
 * notes; "ZeRO: Three Ledgers, Zero Redundancy", section 2): writes
 * S = sum over all positions of g^2 (g the averaged gradient, pads 0) as a
 * binary64 to *sqnorm_dev (DEVICE pointer, 8-byte aligned), asynchronously.
 * Each segment's partial sums go to the plan's workspace, then one launch adds
 * them in a fixed order: the result is the same bits on every run and every
 * GPU, within about 1e-13 relative of the exact sum. */
int zero_grad_sqnorm(const zero_plan *plan, const void *const *grads, int32_t gdtype,
                     double *sqnorm_dev, zero_stream_t stream);

/* Local AdamW on every rank's shard ("ZeRO and FSDP sharding", Code,
 * AdamW::step; How it works: AdamW on the fp32 master slice, cast to bf16
 * shard) from an already averaged fp32 gradient shard.  gshard, master, m, v:
 * [N] device fp32 buffers of H elements; master/m/v are updated in place.
 * Outputs, each optional (NULL): pshard [N] device buffers of H elements of
 * pdtype (the rank's param shard), full: a device buffer of P_pad elements of
 * pdtype (the gathered params, written directly).  No clipping is applied
 * (hp->max_norm is ignored). */
int zero_adamw_shard_step(const zero_plan *plan, const float *const *gshard, float *const *master,
                          float *const *m, float *const *v, void *const *pshard, void *full,
                          int32_t pdtype, const zero_hparams *hp, zero_stream_t stream);

/* All-gather ("ZeRO and FSDP sharding", Code: all_gather = concatenation of
 * the shards; How it works: ZeRO-3 gathers per unit): full[F_u + r h_u + j] =
 * shard[r][Hoff_u + j] for every rank r, for unit `unit`, or every unit when
 * unit == -1.  shard: [N] device buffers of H elements, full: P_pad elements,
 * both of pdtype. */
int zero_all_gather(const zero_plan *plan, const void *const *shard, void *full, int32_t pdtype,
                    int32_t unit, zero_stream_t stream);

/* zero_all_gather with pdtype = ZERO_BF16. */
int zero_all_gather_bf16(const zero_plan *plan, const uint16_t *const *shard16, uint16_t *full,
                         int32_t unit, zero_stream_t stream);

/* The fused sharded step ("ZeRO: Three Ledgers, Zero Redundancy", section 2:
 * stop the all-reduce halfway and do the update in the middle):
 * reduce-scatter + average + AdamW + cast + all-gather in ONE pass over the
 * multi-unit work table (one kernel launch), each gradient byte read once.
 *   grads   [N] device, P_pad elements of gdtype; read only.
 *   master, m, v  [N] device fp32, H elements; updated in place.
 *   full    device, P_pad elements of pdtype, or NULL (ZeRO-1/2 gather target).
 *   pshard  [N] device, H elements of pdtype, or NULL (ZeRO-3 param shards).
 *   gshard_ws [N] device fp32, H elements: required when hp->max_norm > 0
 *           (it then receives the averaged, unclipped gradient shard), else
 *           ignored (may be NULL).
 *   sqnorm_dev  DEVICE binary64 or NULL: receives S when clipping.
 *   unit    -1: all units in one launch; u >= 0: unit u only (no clipping).
 * With clipping the step is three launches (sum of squares and gradient
 * shard; fixed-order total and coefficient on the device; update), with no
 * host synchronisation.  If S is not finite the update is skipped entirely:
 * master, m, v and the outputs are left untouched, and S (inf or NaN) is still
 * written to sqnorm_dev so the caller can see it.
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ENOTATTACHED, ZERO_ECUDA. */
int zero_step(const zero_plan *plan, const void *const *grads, int32_t gdtype, float *const *master,
              float *const *m, float *const *v, void *full, void *const *pshard, int32_t pdtype,
              float *const *gshard_ws, const zero_hparams *hp, double *sqnorm_dev, int32_t unit,
              zero_stream_t stream);

/* ---------------------------------------------------------------- one unit at a time */

/* All-gather of one unit into a UNIT-SIZED destination: dst_unit (DEVICE,
 * 16-byte aligned, S_u elements of pdtype) receives the unit's gathered params,
 * element i = full position F_u + i.  This is ZeRO-3's just-in-time gather
 * ("ZeRO and FSDP sharding", How it works: per unit, all-gather the bf16
 * weights, compute, free the non-owned part; prefetching unit k+1's gather
 * while unit k computes keeps it off the critical path): two unit-sized
 * buffers instead of the whole parameter buffer. */
int zero_all_gather_unit(const zero_plan *plan, int32_t unit, const void *const *shard, void *dst_unit,
                         int32_t pdtype, zero_stream_t stream);

/* The fused step for unit `unit` only, with UNIT-LOCAL gradient buffers:
 * grads_unit[q] (DEVICE, 16-byte aligned) holds rank q's S_u padded gradient
 * positions of the unit (element i is full position F_u + i), so a caller can
 * stream gradients in unit by unit (a bucket, or a host-to-device copy) without
 * ever holding N full gradient buffers ("ZeRO: Three Ledgers, Zero Redundancy",
 * section 4: gradients streamed through buckets, never resident in full).
 * master/m/v, full and pshard are the usual full-size buffers (only the unit's
 * positions are touched).  No clipping (hp->max_norm must be <= 0: a global
 * norm needs every unit first).  Results equal zero_step's bit for bit.
 * Errors: as zero_step; ZERO_EINVAL for unit out of [0, n_units) or clipping. */
int zero_step_unit(const zero_plan *plan, int32_t unit, const void *const *grads_unit, int32_t gdtype,
                   float *const *master, float *const *m, float *const *v, void *full, void *const *pshard,
                   int32_t pdtype, const zero_hparams *hp, zero_stream_t stream);

/* zero_step_unit for the consecutive units [u0, u1) at once, from BUCKET-LOCAL
 * gradient buffers: grads_bucket[q] (DEVICE, 16-byte aligned) holds rank q's
 * padded gradient positions of those units, element i = full position F_u0 + i
 * (F_u1 - F_u0 elements).  A bucket of several units is one launch; this is
 * ZeRO-2's gradient bucket ("ZeRO: Three Ledgers, Zero Redundancy", section 4:
 * gradients streamed through buckets and reduced as they fill, so the N full
 * gradient buffers never exist).  0 <= u0 < u1 <= n_units.  No clipping.
 * Results equal zero_step's bit for bit.  Errors: as zero_step_unit. */
int zero_step_units(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads_bucket, int32_t gdtype,
                    float *const *master, float *const *m, float *const *v, void *full, void *const *pshard,
                    int32_t pdtype, const zero_hparams *hp, zero_stream_t stream);

/* zero_reduce_scatter for unit `unit` only, from unit-local gradient buffers
 * (as zero_step_unit): gshard[r][Hoff_u + j] for the unit's slices. */
int zero_reduce_scatter_unit(const zero_plan *plan, int32_t unit, const void *const *grads_unit, int32_t gdtype,
                             float *const *gshard, float coef, zero_stream_t stream);

/* The clipped step with the gradients streamed in unit by unit (the norm needs
 * every unit before any update, "ZeRO and FSDP sharding", Implementation
 * notes; a norm is a decomposable sum of squares, "ZeRO: Three Ledgers, Zero
 * Redundancy", section 2).  Three calls, in this order on one stream:
 *
 * 1. zero_clip_reduce_unit for every unit with S_u > 0 (or zero_clip_reduce_units
 *    for buckets of consecutive units), in any order, each
 *    from unit-local gradient buffers (as zero_step_unit): writes the unit's
 *    averaged fp32 gradient into gshard[r][Hoff_u + j] and the sums of squares
 *    of the unit's launch-table segments into the plan's workspace.
 * 2. zero_clip_finalize: adds every segment's partial sums in a fixed order
 *    (the same order as zero_step's) into S (*sqnorm_dev, DEVICE, 8-byte aligned,
 *    optional) and the clip coefficient min(1, max_norm / (sqrt(S) + 1e-6)),
 *    both kept on the device; S not finite skips the update of step 3 (and
 *    zero_plan_check then reports ZERO_ENONFINITE).
 * 3. zero_adamw_shard_step_clipped for all units (unit = -1) or unit by unit:
 *    zero_adamw_shard_step from gshard scaled by that coefficient.
 *
 * master/m/v, params and S equal those of a clipped zero_step bit for bit.
 * Errors: as zero_step_unit / zero_adamw_shard_step; zero_clip_finalize
 * returns ZERO_EINVAL for max_norm <= 0. */
int zero_clip_reduce_unit(const zero_plan *plan, int32_t unit, const void *const *grads_unit, int32_t gdtype,
                          float *const *gshard, zero_stream_t stream);
/* Step 1 for the consecutive units [u0, u1) at once, from a bucket-local
 * gradient buffer laid out as for zero_step_units. */
int zero_clip_reduce_units(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads_bucket,
                           int32_t gdtype, float *const *gshard, zero_stream_t stream);
int zero_clip_finalize(const zero_plan *plan, float max_norm, double *sqnorm_dev, zero_stream_t stream);
int zero_adamw_shard_step_clipped(const zero_plan *plan, const float *const *gshard, float *const *master,
                                  float *const *m, float *const *v, void *const *pshard, void *full, int32_t pdtype,
                                  const zero_hparams *hp, int32_t unit, zero_stream_t stream);

/* ---------------------------------------------------------------- checkpoint resharding */

/* Reshard a per-rank array between two layouts of the same units ("ZeRO and
 * FSDP sharding", Implementation notes: checkpoints are written sharded, each
 * rank its own shard, and resharded to a different N at load time).
 *   from, to  attached plans on the current device with identical unit sizes
 *             (any rank counts, 1..ZERO_MAX_RANKS).
 *   src       [from N] DEVICE buffers of from's H elements (aligned to the element).
 *   dst       [to N'] DEVICE buffers of to's H' elements; must not overlap src.
 *   dtype     ZERO_F32 (master, m, v, gradient shards) or ZERO_BF16 (param shards).
 * Every real position moves to its owner in the target layout bit for bit;
 * positions that are padding in the target are written as 0, source padding
 * is dropped.  One launch; errors as the other calls (ZERO_EINVAL for
 * mismatched units or devices). */
int zero_reshard(const zero_plan *from, const zero_plan *to, const void *const *src, void *const *dst,
                 int32_t dtype, zero_stream_t stream);

/* ---------------------------------------------------------------- ZeRO-Offload: the update on the host cores */

/* ZeRO-Offload ("Learn: ZeRO & FSDP", section 6, Offloading; "ZeRO and FSDP
 * sharding", Implementation notes): the optimizer state and the fp32 AdamW
 * step move to host memory and the host CPU.  The GPU reduce-scatters the
 * gradients, the averaged fp32 gradient shard goes down to the host, the host
 * cores run the update, and the updated params come back.  It trades the host
 * link's bandwidth for device memory: master, m and v (12 bytes per parameter)
 * never occupy HBM.
 *
 * An engine owns a pool of host worker threads and, from its first step on,
 * two copy streams and a few events on the plan's device.  The results are
 * those of zero_step, bit for bit: every element goes through the operations
 * listed at the top of this header, each one binary32 operation rounded to
 * nearest even (the host code is compiled without contraction and runs the
 * update in the default floating-point environment, subnormals kept).
 *   plan        the layout (it must outlive the engine; zero_offload_step
 *               needs it attached).
 *   n_threads   host threads of the update (>= 1), or 0 for every core this
 *               process may run on.
 *   batch_min   the step is pipelined over batches of consecutive units of at
 *               least this many padded elements; 0 picks 2^22.
 * Host only; needs no GPU.  Errors: ZERO_EINVAL, ZERO_ENOMEM. */
typedef struct zero_offload zero_offload;
int zero_offload_create(const zero_plan *plan, int32_t n_threads, int64_t batch_min, zero_offload **out);

/* Frees the engine (threads, copy streams, events).  NULL is a no-op. */
void zero_offload_destroy(zero_offload *eng);

/* The engine's host worker threads and pipeline batches (each batch is one
 * reduce launch and one host update per step).  Either pointer may be NULL. */
int zero_offload_info(const zero_offload *eng, int32_t *n_threads, int64_t *n_batches);

/* The update on the host cores alone, on HOST arrays (no GPU involved): for
 * every rank r and every shard position of unit `unit` (-1: all units), AdamW
 * with the averaged gradient gshard_h[r][j] on master_h/m_h/v_h[r][j].
 *   gshard_h   [N] host fp32 arrays of H elements (read only).
 *   master_h, m_h, v_h  [N] host fp32 arrays of H elements, updated in place.
 *   pshard_h   [N] host arrays of H elements of pdtype, or NULL: the param shards.
 *   full_h     a host array of P_pad elements of pdtype, or NULL: the params
 *              at their full positions (F_u + r h_u + j).
 *   sqnorm     used only when hp->max_norm > 0: the sum of squares S of the
 *              averaged gradient; the gradient is scaled by min(1, max_norm /
 *              (sqrt(S) + 1e-6)) (binary64, rounded once to binary32) first,
 *              as zero_step does; S not finite returns ZERO_ENONFINITE before
 *              anything is touched.
 * Synchronous: the engine's threads share the positions out.
 * Errors: ZERO_EINVAL, ZERO_ENONFINITE, ZERO_ENOMEM. */
int zero_offload_adamw(zero_offload *eng, const float *const *gshard_h, float *const *master_h, float *const *m_h,
                       float *const *v_h, void *const *pshard_h, void *full_h, int32_t pdtype, const zero_hparams *hp,
                       double sqnorm, int32_t unit);

/* The offloaded step, pipelined over the engine's batches of units:
 *   1. GPU (`stream`): reduce-scatter + average of the batch's units from the N
 *      device gradient buffers into gshard_dev (with clipping also the batch's
 *      sums of squares);
 *   2. GPU copy stream: the batch's slices of gshard_dev to gshard_h;
 *   3. host cores: AdamW of the batch on master_h/m_h/v_h as soon as its slices
 *      have landed, the params written to full_h;
 *   4. GPU copy stream: the batch's params from full_h to full_dev;
 * so copies down, host updates and copies up of different batches overlap.
 * With clipping (hp->max_norm > 0) the norm passes of all batches run first, S
 * is read back (the one wait for the GPU), then the updates run as above; S not
 * finite skips the update (master_h, m_h, v_h, full_h and full_dev are left
 * untouched), returns ZERO_ENONFINITE, and is also reported by a later
 * zero_plan_check, as for zero_step.
 *   grads       [N] DEVICE buffers of P_pad elements of gdtype, read only.
 *   gshard_dev  [N] DEVICE fp32 buffers of H elements: staging.
 *   gshard_h    [N] HOST fp32 arrays of H elements: staging.
 *   master_h, m_h, v_h  [N] HOST fp32 arrays of H elements: the optimizer state.
 *   full_h      a HOST array of P_pad elements of pdtype: receives the params.
 *   full_dev    a DEVICE buffer of P_pad elements of pdtype, or NULL.
 *   sqnorm_out  a HOST binary64 receiving S when clipping, or NULL.
 * Host arrays should be page-locked (cudaHostAlloc, a pinned torch tensor) so
 * that the copies run asynchronously; pageable memory gives the same results
 * with copies that block.  The call returns when the host update is done and
 * the last param copy is queued; `stream` is made to wait for every copy, so
 * work queued on it afterwards sees full_dev updated and may overwrite
 * gshard_dev.  The plan must be attached to the current device; calls with one
 * engine or one plan must not overlap.  After ZERO_ECUDA the step may be
 * partly done.  Errors: ZERO_EINVAL, ZERO_EALIGN (device pointers),
 * ZERO_ENOTATTACHED, ZERO_ECUDA, ZERO_ENONFINITE, ZERO_ENOMEM. */
int zero_offload_step(zero_offload *eng, const void *const *grads, int32_t gdtype, float *const *gshard_dev,
                      float *const *gshard_h, float *const *master_h, float *const *m_h, float *const *v_h,
                      void *full_h, void *full_dev, int32_t pdtype, const zero_hparams *hp, double *sqnorm_out,
                      zero_stream_t stream);

/* Timings of the engine's last zero_offload_step in milliseconds (waits for
 * its copies to finish): ms[0] host time inside the call; ms[1] host time spent
 * waiting for gradient slices to land (and, clipping, for S); ms[2] host time
 * spent updating; ms[3] device time from the step's start until its last param
 * copy had landed; ms[4] device time from the start until its last gradient
 * slice had landed on the host.  ZERO_EINVAL before the first step. */
int zero_offload_timings(zero_offload *eng, double *ms);

/* ---------------------------------------------------------------- without allocation */

/* No counterpart on the pages: an addition for callers that cannot allocate
 * device memory.  A gradient-norm check often has to run exactly when memory
 * is exhausted (logging the norm of a step that ran out of memory, a watchdog
 * for non-finite gradients inside a framework whose caching allocator holds
 * nearly all of the GPU); there a cudaMalloc, or a request to the framework's
 * allocator, fails or makes the allocator release and re-reserve memory.
 *
 * Computes the same quantity as zero_grad_sqnorm -- S = sum of g^2, g the
 * rank-ordered binary32 average of the N gradients, each square exact in
 * binary64, partials added in a fixed order -- over n flat positions, with no
 * plan and no workspace: every position counts, so padding entries must hold
 * 0 (as a flat-parameter layout keeps them).  It allocates nothing: the
 * per-chunk partial sums live in one array of ZERO_NOALLOC_MAX_CHUNKS binary64
 * values (256 KB) compiled into the library, which every GPU that loads the
 * library holds until the process exits.
 *   grads     [n_ranks] device pointers to n elements of gdtype each (aligned
 *             to the element size), on the current device.  With n == 0 they
 *             may be NULL.
 *   n         0 <= n <= ZERO_NOALLOC_MAX_CHUNKS * ZERO_NOALLOC_CHUNK
 *             (2^32 elements); larger n returns ZERO_ERANGE before any launch.
 *             n == 0 writes S = 0.
 *   sqnorm_dev  DEVICE binary64 receiving S (8-byte aligned), asynchronously,
 *             on the current device.
 * A gradient that is inf or NaN makes S inf or NaN (a watchdog tests S).
 * Set-up: the first call on each device, with that device current, loads the
 * library's norm kernels onto the device and looks up the array's device
 * address (cudaGetSymbolAddress); the address is cached for the life of the
 * process, so the device's context must not be reset (cudaDeviceReset) after
 * it.  Loading code takes device memory, so make that first call -- a call
 * with n = 0 is enough -- while device memory is still free, and before any
 * stream capture; later calls take no device memory at all.
 * All calls share the one array (it keeps the last call's partials, and every
 * call overwrites the ones it reads), so calls whose work overlaps on the GPU
 * -- on two streams, or from two threads -- race; order them on one stream.
 * Errors: ZERO_EINVAL (NULL, n < 0, n_ranks out of range, a pointer that is not
 * device memory of the current device), ZERO_EALIGN, ZERO_ERANGE, ZERO_ECUDA. */
#define ZERO_NOALLOC_CHUNK 131072
#define ZERO_NOALLOC_MAX_CHUNKS 32768
int zero_grad_sqnorm_noalloc(const void *const *grads, int32_t n_ranks, int32_t gdtype, int64_t n,
                             double *sqnorm_dev, zero_stream_t stream);

/* ---------------------------------------------------------------- diagnostics */

/* Reads and clears the plan's device error word, synchronising `stream`:
 * *errors = 0 when every bounded wait inside the kernels completed, non-zero
 * when one gave up (the step it belonged to stopped early and its results are
 * incomplete).  No kernel waits longer than about two seconds. */
int zero_plan_device_errors(const zero_plan *plan, zero_stream_t stream, int32_t *errors);

/* The outcome of the device work enqueued on the plan since the previous
 * check, as a status; synchronises `stream`.  Device calls return as soon as
 * their kernels are queued, so conditions found on the device are reported
 * here: ZERO_ETIMEOUT when a bounded wait expired (that work is incomplete,
 * as for zero_plan_device_errors), else ZERO_ENONFINITE when a clipped
 * zero_step found a non-finite global norm and left master, m, v and the
 * params untouched (the pages leave that case open; skipping the step is the
 * reading taken), else ZERO_OK.  Both conditions are cleared.  ZERO_EINVAL /
 * ZERO_ENOTATTACHED / ZERO_ECUDA as usual. */
int zero_plan_check(const zero_plan *plan, zero_stream_t stream);

/* Testing aid for the bounded waits (failure detection without a GPU fault):
 * arms the NEXT pipelined launch so that the copies of tile number `tile`
 * (0-based) of the launch's first segment are skipped.  That stage never fills;
 * the consumer warps waiting for it give up after about two seconds, the
 * producer's own wait for the stage runs out next, it waits (bounded) for the
 * copies it did issue, and the launch ends with incomplete results and a
 * non-zero device error word (zero_plan_device_errors).  The context stays
 * usable.  One launch only, then it disarms; -1 disarms at once. */
int zero_debug_drop_copy(int64_t tile);

/* Static text for a status code. */
const char *zero_status_string(int status);

/* The last CUDA error code this thread saw inside the library (0 if none),
 * for callers that got ZERO_ECUDA. */
int zero_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_H */
