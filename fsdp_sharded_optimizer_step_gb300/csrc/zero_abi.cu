// The C-ABI entry points of the sharded optimizer step (include/zero.h):
// argument checks on the host, the kernel parameter blocks, and the launches
// through the interface in zero_launch.h.  No device code here.
#include <cuda_runtime.h>

#include <cstdint>

#include "zero_launch.h"
#include "zero_nvtx.h"

namespace zero {

// ------------------------------------------------------------------ host helpers
static bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// A plan without elements (P_pad == 0) accepts null rank pointers: nothing is
// ever read or written through them.
static int check_rank_ptrs(const zero_plan *plan, const void *const *arr, bool required) {
    if (arr == nullptr) return required ? ZERO_EINVAL : ZERO_OK;
    for (int q = 0; q < plan->n_ranks; ++q) {
        if (arr[q] == nullptr) {
            if (plan->p_pad == 0) continue;
            return ZERO_EINVAL;
        }
        if (!aligned16(arr[q])) return ZERO_EALIGN;
    }
    return ZERO_OK;
}

static int check_ptr(const zero_plan *plan, const void *ptr, bool required) {
    if (ptr == nullptr) return (required && plan->p_pad != 0) ? ZERO_EINVAL : ZERO_OK;
    return aligned16(ptr) ? ZERO_OK : ZERO_EALIGN;
}

static int check_attached(const zero_plan *plan) {
    if (plan == nullptr) return ZERO_EINVAL;
    if (!plan->attached) return ZERO_ENOTATTACHED;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    if (dev != plan->device) return ZERO_EINVAL;
    return ZERO_OK;
}

static void fill_common(const zero_plan *plan, KParams &kp) {
    kp = KParams{};
    kp.segs = plan->d_segs;
    kp.n_ranks = plan->n_ranks;
    const int n = plan->n_ranks;
    kp.pow2 = (n & (n - 1)) == 0;
    kp.nf = static_cast<float>(n);
    kp.inv_n = kp.pow2 ? 1.0f / static_cast<float>(n) : 0.0f;  // exact for a power of two
    kp.coef = 1.0f;
    kp.partials = plan->d_partials;
    kp.err = plan->d_err;
    kp.p_pad = plan->p_pad;
    kp.h_len = plan->H;
    kp.g_origin = 0;
    kp.g_len = plan->p_pad;
    kp.drop_tile = -1;
    kp.tickets = plan->d_tickets;
}

// Segment range of one unit, or of all units.
static int seg_range(const zero_plan *plan, int32_t unit, int64_t &begin, int64_t &count) {
    if (unit < -1 || unit >= plan->n_units) return ZERO_EINVAL;
    if (unit == -1) {
        begin = 0;
        count = static_cast<int64_t>(plan->segs.size());
    } else {
        begin = plan->unit_seg_begin[unit];
        count = plan->unit_seg_begin[unit + 1] - begin;
    }
    if (count > 0x7FFFFFFF) return ZERO_EINVAL;
    return ZERO_OK;
}

// Launches over units [u0, u1) without per-segment partial sums take the
// unit-local table (each unit cut into about kLocalSegsPerUnit segments, so a
// small unit still spreads over every SM); whole-plan launches and the norm's
// passes, whose partials sit at main-table positions, take the main table.
static int use_local_table(const zero_plan *plan, int32_t u0, int32_t u1, KParams &kp, int64_t &count) {
    const int64_t begin = plan->unit_local_begin[u0];
    count = plan->unit_local_begin[u1] - begin;
    if (count > 0x7FFFFFFF) return ZERO_EINVAL;
    kp.segs = plan->d_segs_local;
    kp.seg_base = begin;
    return ZERO_OK;
}

static bool valid_dtype(int32_t d) { return d == ZERO_BF16 || d == ZERO_F32; }

int reduce_units(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads, int32_t gdtype,
                 float *const *gshard, bool want_partials, cudaStream_t st) {
    if (u0 < 0 || u1 > plan->n_units || u0 > u1) return ZERO_EINVAL;
    const int64_t begin = plan->unit_seg_begin[u0];
    const int64_t count = plan->unit_seg_begin[u1] - begin;
    if (count == 0) return ZERO_OK;
    KParams kp;
    fill_common(plan, kp);
    kp.seg_base = begin;
    kp.write_g = 1;
    kp.want_partials = want_partials ? 1 : 0;
    for (int q = 0; q < plan->n_ranks; ++q) {
        kp.grads[q] = grads[q];
        kp.gshard[q] = gshard[q];
    }
    return launch_pipe(MODE_REDUCE, gdtype, count, kp, st);
}

}  // namespace zero

using namespace zero;

// ------------------------------------------------------------------ C ABI
extern "C" int zero_plan_attach(zero_plan *plan, void *workspace, size_t bytes, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    if (plan == nullptr || workspace == nullptr || plan->attached) return ZERO_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ZERO_EALIGN;
    const WsLayout L = workspace_layout(plan);
    if (bytes < L.total) return ZERO_ENOMEM;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    char *base = static_cast<char *>(workspace);
    if (!plan->segs.empty()) {
        e = cudaMemcpyAsync(base + L.segs, plan->segs.data(), plan->segs.size() * sizeof(Seg), cudaMemcpyHostToDevice,
                            reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    }
    plan->d_segs = reinterpret_cast<Seg *>(base + L.segs);
    if (!plan->segs_local.empty()) {
        e = cudaMemcpyAsync(base + L.segs_local, plan->segs_local.data(), plan->segs_local.size() * sizeof(Seg),
                            cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    }
    plan->d_segs_local = reinterpret_cast<Seg *>(base + L.segs_local);
    plan->d_partials = reinterpret_cast<SqPartial *>(base + L.partials);
    plan->d_sqnorm = reinterpret_cast<double *>(base + L.scalars);
    plan->d_coef = reinterpret_cast<float *>(base + L.scalars + 8);
    plan->d_err = reinterpret_cast<int *>(base + L.scalars + 16);
    plan->d_tickets = reinterpret_cast<unsigned long long *>(base + L.scalars + 24);
    plan->d_skipped = reinterpret_cast<int *>(base + L.scalars + 40);
    plan->d_fin_count = reinterpret_cast<unsigned *>(base + L.scalars + 48);
    plan->d_fin_sums = reinterpret_cast<double *>(base + L.fin);
    if (!plan->unit_table.empty()) {
        e = cudaMemcpyAsync(base + L.units, plan->unit_table.data(), plan->unit_table.size() * sizeof(UnitDesc),
                            cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    }
    plan->d_units = reinterpret_cast<UnitDesc *>(base + L.units);
    e = cudaMemsetAsync(base + L.scalars, 0, 256, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    plan->device = dev;
    plan->attached = true;
    return ZERO_OK;
}

extern "C" int zero_reduce_scatter(const zero_plan *plan, const void *const *grads, int32_t gdtype,
                                   float *const *gshard, float coef, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!valid_dtype(gdtype)) return ZERO_EINVAL;
    const int n = plan->n_ranks;
    if ((rc = check_rank_ptrs(plan, grads, true)) != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    KParams kp;
    fill_common(plan, kp);
    kp.coef = coef;
    kp.write_g = 1;
    for (int q = 0; q < n; ++q) {
        kp.grads[q] = grads[q];
        kp.gshard[q] = gshard[q];
    }
    return launch_pipe(MODE_REDUCE, gdtype, static_cast<int64_t>(plan->segs.size()), kp,
                       reinterpret_cast<cudaStream_t>(stream));
}

// Pass 1 of a norm: per-segment partial sums (and optionally the gradient
// shard), then the fixed-order total (and coefficient) on the device.
static int launch_norm(const zero_plan *plan, const void *const *grads, int32_t gdtype, float *const *gshard,
                       float max_norm, double *sqnorm_out, cudaStream_t st) {
    KParams kp;
    fill_common(plan, kp);
    kp.want_partials = 1;
    kp.write_g = gshard != nullptr;
    for (int q = 0; q < plan->n_ranks; ++q) {
        kp.grads[q] = grads[q];
        if (gshard != nullptr) kp.gshard[q] = gshard[q];
    }
    const int64_t nseg = static_cast<int64_t>(plan->segs.size());
    const int rc = launch_pipe(MODE_REDUCE, gdtype, nseg, kp, st);
    if (rc != ZERO_OK) return rc;
    return launch_finalize(plan, max_norm, sqnorm_out, st);
}

extern "C" int zero_grad_sqnorm(const zero_plan *plan, const void *const *grads, int32_t gdtype, double *sqnorm_dev,
                                zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!valid_dtype(gdtype) || sqnorm_dev == nullptr) return ZERO_EINVAL;
    if ((reinterpret_cast<uintptr_t>(sqnorm_dev) & 7u) != 0) return ZERO_EALIGN;
    if ((rc = check_rank_ptrs(plan, grads, true)) != ZERO_OK) return rc;
    return launch_norm(plan, grads, gdtype, nullptr, 0.0f, sqnorm_dev, reinterpret_cast<cudaStream_t>(stream));
}

static int fill_state(const zero_plan *plan, KParams &kp, float *const *master, float *const *m, float *const *v,
                      void *const *pshard, void *full, int32_t pdtype, const zero_hparams *hp) {
    const int n = plan->n_ranks;
    int rc;
    if (!valid_dtype(pdtype) || hp == nullptr) return ZERO_EINVAL;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(master), true)) != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(m), true)) != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(v), true)) != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, pshard, false)) != ZERO_OK) return rc;
    if ((rc = check_ptr(plan, full, false)) != ZERO_OK) return rc;
    if ((rc = adam_consts(hp, &kp.c)) != ZERO_OK) return rc;
    kp.pdtype = pdtype;
    kp.full = full;
    for (int q = 0; q < n; ++q) {
        kp.master[q] = master[q];
        kp.m[q] = m[q];
        kp.v[q] = v[q];
        kp.pshard[q] = pshard != nullptr ? pshard[q] : nullptr;
    }
    return ZERO_OK;
}

extern "C" int zero_adamw_shard_step(const zero_plan *plan, const float *const *gshard, float *const *master,
                                     float *const *m, float *const *v, void *const *pshard, void *full, int32_t pdtype,
                                     const zero_hparams *hp, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    KParams kp;
    fill_common(plan, kp);
    if ((rc = fill_state(plan, kp, master, m, v, pshard, full, pdtype, hp)) != ZERO_OK) return rc;
    for (int q = 0; q < plan->n_ranks; ++q) kp.gshard[q] = const_cast<float *>(gshard[q]);
    return launch_pipe(MODE_SHARD, ZERO_F32, static_cast<int64_t>(plan->segs.size()), kp,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_all_gather(const zero_plan *plan, const void *const *shard, void *full, int32_t pdtype, int32_t unit,
                               zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!valid_dtype(pdtype)) return ZERO_EINVAL;
    if ((rc = check_rank_ptrs(plan, shard, true)) != ZERO_OK) return rc;
    if ((rc = check_ptr(plan, full, true)) != ZERO_OK) return rc;
    int64_t begin = 0, count = 0;
    if ((rc = seg_range(plan, unit, begin, count)) != ZERO_OK) return rc;
    KParams kp;
    fill_common(plan, kp);
    kp.seg_base = begin;
    if (unit >= 0 && (rc = use_local_table(plan, unit, unit + 1, kp, count)) != ZERO_OK) return rc;
    kp.pdtype = pdtype;
    kp.full = full;
    for (int q = 0; q < plan->n_ranks; ++q) kp.pshard[q] = const_cast<void *>(shard[q]);
    if (count == 0) return ZERO_OK;
    return launch_gather(count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_all_gather_unit(const zero_plan *plan, int32_t unit, const void *const *shard, void *dst_unit,
                                    int32_t pdtype, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!valid_dtype(pdtype) || unit < 0 || unit >= plan->n_units) return ZERO_EINVAL;
    int64_t begin = 0, count = 0;
    if ((rc = seg_range(plan, unit, begin, count)) != ZERO_OK) return rc;
    if (count == 0) return ZERO_OK;
    if ((rc = check_rank_ptrs(plan, shard, true)) != ZERO_OK) return rc;
    if (dst_unit == nullptr) return ZERO_EINVAL;
    if (!aligned16(dst_unit)) return ZERO_EALIGN;
    KParams kp;
    fill_common(plan, kp);
    if ((rc = use_local_table(plan, unit, unit + 1, kp, count)) != ZERO_OK) return rc;
    kp.pdtype = pdtype;
    kp.full = dst_unit;
    kp.g_origin = plan->F[unit];
    for (int q = 0; q < plan->n_ranks; ++q) kp.pshard[q] = const_cast<void *>(shard[q]);
    return launch_gather(count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_all_gather_bf16(const zero_plan *plan, const uint16_t *const *shard16, uint16_t *full, int32_t unit,
                                    zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    return zero_all_gather(plan, reinterpret_cast<const void *const *>(shard16), full, ZERO_BF16, unit, stream);
}

extern "C" int zero_step(const zero_plan *plan, const void *const *grads, int32_t gdtype, float *const *master,
                         float *const *m, float *const *v, void *full, void *const *pshard, int32_t pdtype,
                         float *const *gshard_ws, const zero_hparams *hp, double *sqnorm_dev, int32_t unit,
                         zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!valid_dtype(gdtype) || hp == nullptr) return ZERO_EINVAL;
    const int n = plan->n_ranks;
    if ((rc = check_rank_ptrs(plan, grads, true)) != ZERO_OK) return rc;
    const bool clip = hp->max_norm > 0.0f;
    if (clip) {
        if (unit != -1) return ZERO_EINVAL;  // the global norm needs every unit
        if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard_ws), true)) != ZERO_OK) return rc;
        if (sqnorm_dev != nullptr && (reinterpret_cast<uintptr_t>(sqnorm_dev) & 7u) != 0) return ZERO_EALIGN;
    }
    int64_t begin = 0, count = 0;
    if ((rc = seg_range(plan, unit, begin, count)) != ZERO_OK) return rc;
    KParams kp;
    fill_common(plan, kp);
    if ((rc = fill_state(plan, kp, master, m, v, pshard, full, pdtype, hp)) != ZERO_OK) return rc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!clip) {
        for (int q = 0; q < n; ++q) kp.grads[q] = grads[q];
        kp.seg_base = begin;
        if (unit >= 0 && (rc = use_local_table(plan, unit, unit + 1, kp, count)) != ZERO_OK) return rc;
        return launch_pipe(MODE_FUSED, gdtype, count, kp, st);
    }
    // clipped: norm pass (writes the averaged gradient shard), device
    // coefficient, then the update from the shard scaled by that coefficient
    if ((rc = launch_norm(plan, grads, gdtype, gshard_ws, hp->max_norm, sqnorm_dev, st)) != ZERO_OK) return rc;
    for (int q = 0; q < n; ++q) kp.gshard[q] = gshard_ws[q];
    kp.use_coef_dev = 1;
    kp.coef_dev = plan->d_coef;
    return launch_pipe(MODE_SHARD, ZERO_F32, count, kp, st);
}

// Bucket-local variants: grads_b[q] holds only the padded gradient positions
// of units [u0, u1), element i = full position F_u0 + i (one unit: u1 = u0 + 1).
static int units_common(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads_b, int32_t gdtype,
                        bool local, int64_t &count, KParams &kp) {
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!valid_dtype(gdtype) || u0 < 0 || u1 <= u0 || u1 > plan->n_units) return ZERO_EINVAL;
    const int64_t begin = plan->unit_seg_begin[u0];
    count = plan->unit_seg_begin[u1] - begin;
    if (count > 0x7FFFFFFF) return ZERO_EINVAL;
    const int64_t f_end = u1 < plan->n_units ? plan->F[u1] : plan->p_pad;
    fill_common(plan, kp);
    kp.g_origin = plan->F[u0];
    kp.g_len = f_end - plan->F[u0];
    kp.seg_base = begin;
    if (local && (rc = use_local_table(plan, u0, u1, kp, count)) != ZERO_OK) return rc;
    if (kp.g_len == 0) return ZERO_OK;
    if (grads_b == nullptr) return ZERO_EINVAL;
    for (int q = 0; q < plan->n_ranks; ++q) {
        if (grads_b[q] == nullptr) return ZERO_EINVAL;
        if (!aligned16(grads_b[q])) return ZERO_EALIGN;
        kp.grads[q] = grads_b[q];
    }
    return ZERO_OK;
}

static int unit_common(const zero_plan *plan, int32_t unit, const void *const *grads_unit, int32_t gdtype,
                       bool local, int64_t &count, KParams &kp) {
    if (plan == nullptr) return ZERO_EINVAL;
    if (unit < 0 || unit >= plan->n_units) return ZERO_EINVAL;
    return units_common(plan, unit, unit + 1, grads_unit, gdtype, local, count, kp);
}

extern "C" int zero_step_unit(const zero_plan *plan, int32_t unit, const void *const *grads_unit, int32_t gdtype,
                              float *const *master, float *const *m, float *const *v, void *full, void *const *pshard,
                              int32_t pdtype, const zero_hparams *hp, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    if (hp == nullptr || hp->max_norm > 0.0f) return ZERO_EINVAL;  // a global clip needs every unit
    int64_t count = 0;
    KParams kp;
    int rc = unit_common(plan, unit, grads_unit, gdtype, true, count, kp);
    if (rc != ZERO_OK || count == 0) return rc;
    if ((rc = fill_state(plan, kp, master, m, v, pshard, full, pdtype, hp)) != ZERO_OK) return rc;
    return launch_pipe(MODE_FUSED, gdtype, count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_step_units(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads_bucket,
                               int32_t gdtype, float *const *master, float *const *m, float *const *v, void *full,
                               void *const *pshard, int32_t pdtype, const zero_hparams *hp, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    if (hp == nullptr || hp->max_norm > 0.0f) return ZERO_EINVAL;  // a global clip needs every unit
    int64_t count = 0;
    KParams kp;
    int rc = units_common(plan, u0, u1, grads_bucket, gdtype, true, count, kp);
    if (rc != ZERO_OK || count == 0) return rc;
    if ((rc = fill_state(plan, kp, master, m, v, pshard, full, pdtype, hp)) != ZERO_OK) return rc;
    return launch_pipe(MODE_FUSED, gdtype, count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_clip_reduce_units(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads_bucket,
                                      int32_t gdtype, float *const *gshard, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int64_t count = 0;
    KParams kp;
    int rc = units_common(plan, u0, u1, grads_bucket, gdtype, false, count, kp);
    if (rc != ZERO_OK || count == 0) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    kp.write_g = 1;
    kp.want_partials = 1;
    for (int q = 0; q < plan->n_ranks; ++q) kp.gshard[q] = gshard[q];
    return launch_pipe(MODE_REDUCE, gdtype, count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_reduce_scatter_unit(const zero_plan *plan, int32_t unit, const void *const *grads_unit,
                                        int32_t gdtype, float *const *gshard, float coef, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int64_t count = 0;
    KParams kp;
    int rc = unit_common(plan, unit, grads_unit, gdtype, true, count, kp);
    if (rc != ZERO_OK || count == 0) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    kp.coef = coef;
    kp.write_g = 1;
    for (int q = 0; q < plan->n_ranks; ++q) kp.gshard[q] = gshard[q];
    return launch_pipe(MODE_REDUCE, gdtype, count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_clip_reduce_unit(const zero_plan *plan, int32_t unit, const void *const *grads_unit,
                                     int32_t gdtype, float *const *gshard, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int64_t count = 0;
    KParams kp;
    int rc = unit_common(plan, unit, grads_unit, gdtype, false, count, kp);
    if (rc != ZERO_OK || count == 0) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    kp.write_g = 1;
    kp.want_partials = 1;  // this unit's segments' sums of squares, at their table positions
    for (int q = 0; q < plan->n_ranks; ++q) kp.gshard[q] = gshard[q];
    return launch_pipe(MODE_REDUCE, gdtype, count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_clip_finalize(const zero_plan *plan, float max_norm, double *sqnorm_dev, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (!(max_norm > 0.0f)) return ZERO_EINVAL;
    if (sqnorm_dev != nullptr && (reinterpret_cast<uintptr_t>(sqnorm_dev) & 7u) != 0) return ZERO_EALIGN;
    return launch_finalize(plan, max_norm, sqnorm_dev, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_adamw_shard_step_clipped(const zero_plan *plan, const float *const *gshard, float *const *master,
                                             float *const *m, float *const *v, void *const *pshard, void *full,
                                             int32_t pdtype, const zero_hparams *hp, int32_t unit,
                                             zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    int64_t begin = 0, count = 0;
    if ((rc = seg_range(plan, unit, begin, count)) != ZERO_OK) return rc;
    KParams kp;
    fill_common(plan, kp);
    if ((rc = fill_state(plan, kp, master, m, v, pshard, full, pdtype, hp)) != ZERO_OK) return rc;
    for (int q = 0; q < plan->n_ranks; ++q) kp.gshard[q] = const_cast<float *>(gshard[q]);
    kp.seg_base = begin;
    if (unit >= 0 && (rc = use_local_table(plan, unit, unit + 1, kp, count)) != ZERO_OK) return rc;
    kp.use_coef_dev = 1;  // the coefficient zero_clip_finalize left on the device (NaN: skip)
    kp.coef_dev = plan->d_coef;
    return launch_pipe(MODE_SHARD, ZERO_F32, count, kp, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int zero_debug_drop_copy(int64_t tile) {
    if (tile < -1) return ZERO_EINVAL;
    arm_drop_tile(tile);
    return ZERO_OK;
}

extern "C" int zero_plan_check(const zero_plan *plan, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t err = 0, skipped = 0;
    cudaError_t e = cudaMemcpyAsync(&err, plan->d_err, sizeof(err), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&skipped, plan->d_skipped, sizeof(skipped), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->d_err, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->d_skipped, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    if (err != 0) return ZERO_ETIMEOUT;
    if (skipped != 0) return ZERO_ENONFINITE;
    return ZERO_OK;
}

extern "C" int zero_plan_device_errors(const zero_plan *plan, zero_stream_t stream, int32_t *errors) {
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if (errors == nullptr) return ZERO_EINVAL;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, plan->d_err, sizeof(host), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->d_err, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    *errors = host;
    return ZERO_OK;
}
