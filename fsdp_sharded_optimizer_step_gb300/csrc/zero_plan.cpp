// Host side of the library: the padded layout, the multi-unit launch table,
// the bias corrections and the AdamW constants.  No CUDA here, so all of it
// runs (and is tested) without a GPU.  Built with -ffp-contract=off: the
// binary32 constants below must not be fused into multiply-adds.
#include <cmath>
#include <cstring>
#include <new>

#include "zero_internal.h"

namespace zero {

static thread_local int g_last_cuda_error = 0;
void set_last_cuda_error(int code) { g_last_cuda_error = code; }

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout workspace_layout(const zero_plan *plan) {
    WsLayout L{};
    const size_t nseg = plan->segs.size();
    L.segs = 0;
    L.partials = round_up(nseg * sizeof(Seg), 256);
    L.scalars = L.partials + round_up(nseg * zero::kPartialSlots * sizeof(zero::SqPartial), 256);
    L.units = L.scalars + 256;
    L.fin = L.units + round_up(plan->unit_table.size() * sizeof(UnitDesc), 256);
    L.segs_local = L.fin + round_up(zero::kFinBlocks * sizeof(double), 256);
    L.total = L.segs_local + round_up(plan->segs_local.size() * sizeof(Seg), 256);
    return L;
}

// b^t by binary exponentiation in binary32: walk the bits of t from the low
// end, multiplying the result by the running square where a bit is set.
static float pow_by_squaring(float b, int32_t t) {
    float result = 1.0f;
    float square = b;
    for (uint32_t bitsleft = static_cast<uint32_t>(t); bitsleft != 0u; bitsleft >>= 1) {
        if (bitsleft & 1u) result = result * square;
        if (bitsleft > 1u) square = square * square;
    }
    return result;
}

int adam_consts(const zero_hparams *hp, AdamConsts *out) {
    if (hp == nullptr || out == nullptr || hp->t < 1) return ZERO_EINVAL;
    float bc1 = 0.f, bc2 = 0.f;
    zero_bias_corrections(hp->t, hp->b1, hp->b2, &bc1, &bc2);
    out->b1 = hp->b1;
    out->b2 = hp->b2;
    out->omb1 = 1.0f - hp->b1;
    out->omb2 = 1.0f - hp->b2;
    const float lr_wd = hp->lr * hp->wd;
    out->decay = 1.0f - lr_wd;
    out->lr_bc1 = hp->lr / bc1;
    out->bc2 = bc2;
    out->eps = hp->eps;
    return ZERO_OK;
}

// Cuts unit u's N slices into segments of at most seg_len elements, appended to
// table.  The first segment of a slice ends where the shard position reaches a
// multiple of 8, so every later segment starts 32-byte aligned.
static void cut_unit(const zero_plan *p, int32_t u, int64_t seg_len, std::vector<Seg> &table) {
    const int64_t hu = p->h[u];
    for (int32_t r = 0; r < p->n_ranks; ++r) {
        int64_t j = 0;
        while (j < hu) {
            const int64_t s_off = p->Hoff[u] + j;
            int64_t len = seg_len;
            if (j == 0) len -= (s_off & 7);
            if (len > hu - j) len = hu - j;
            Seg sg;
            sg.g_off = p->F[u] + static_cast<int64_t>(r) * hu + j;
            sg.s_off = s_off;
            sg.len = static_cast<int32_t>(len);
            const int64_t unit_pos = static_cast<int64_t>(r) * hu + j;  // position inside the unit
            int64_t valid = p->sizes[u] - unit_pos;
            if (valid < 0) valid = 0;
            if (valid > len) valid = len;
            sg.valid = static_cast<int32_t>(valid);
            sg.rank = r;
            sg.unit = u;
            table.push_back(sg);
            j += len;
        }
    }
}

// Segment length of unit u in the unit-local table: about kLocalSegsPerUnit
// segments, a multiple of 8, between kLocalSegMin and the main table's length.
static int64_t local_seg_len(int64_t S, int64_t seg_max) {
    int64_t len = (S + kLocalSegsPerUnit - 1) / kLocalSegsPerUnit;
    len = (len + 7) / 8 * 8;
    if (len < kLocalSegMin) len = kLocalSegMin;
    return len < seg_max ? len : seg_max;
}

}  // namespace zero

using zero::Seg;

extern "C" int zero_bias_corrections(int32_t t, float b1, float b2, float *bc1, float *bc2) {
    if (t < 1 || bc1 == nullptr || bc2 == nullptr) return ZERO_EINVAL;
    *bc1 = 1.0f - zero::pow_by_squaring(b1, t);
    *bc2 = std::sqrt(1.0f - zero::pow_by_squaring(b2, t));
    return ZERO_OK;
}

extern "C" int zero_plan_create(const int64_t *unit_sizes, int32_t n_units, int32_t n_ranks, zero_plan **out) {
    return zero_plan_create_aligned(unit_sizes, n_units, n_ranks, 1, out);
}

extern "C" int zero_plan_create_aligned(const int64_t *unit_sizes, int32_t n_units, int32_t n_ranks, int32_t align,
                                        zero_plan **out) {
    if (out == nullptr) return ZERO_EINVAL;
    *out = nullptr;
    if (n_units < 0 || (n_units > 0 && unit_sizes == nullptr)) return ZERO_EINVAL;
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS) return ZERO_EINVAL;
    if (align < 1 || align > ZERO_MAX_ALIGN) return ZERO_EINVAL;
    zero_plan *p = new (std::nothrow) zero_plan();
    if (p == nullptr) return ZERO_ENOMEM;
    try {
        p->n_units = n_units;
        p->n_ranks = n_ranks;
        p->align = align;
        p->sizes.assign(unit_sizes, unit_sizes + n_units);
        p->S.resize(n_units);
        p->h.resize(n_units);
        p->F.resize(n_units);
        p->Hoff.resize(n_units);
        p->unit_seg_begin.resize(static_cast<size_t>(n_units) + 1);
        const int64_t limit = int64_t(1) << 62;
        int64_t full = 0, shard = 0;
        // Padded layout: each unit rounded up to a multiple of N (of N*align with
        // the alignment option), rank r owning the r-th of N equal slices ("ZeRO
        // and FSDP sharding", How it works).
        const int64_t quantum = static_cast<int64_t>(n_ranks) * align;
        for (int32_t u = 0; u < n_units; ++u) {
            const int64_t s = unit_sizes[u];
            if (s < 0 || s > limit - full - quantum) { delete p; return ZERO_EINVAL; }
            const int64_t padded = (s + quantum - 1) / quantum * quantum;
            p->S[u] = padded;
            p->h[u] = padded / n_ranks;
            p->F[u] = full;
            p->Hoff[u] = shard;
            full += padded;
            shard += padded / n_ranks;
        }
        p->p_pad = full;
        p->H = shard;
        // Launch tables: the main one, slices cut into segments of at most
        // seg_max_for(N) elements, and the unit-local one.
        const int64_t seg_max = zero::seg_max_for(n_ranks);
        p->unit_local_begin.resize(static_cast<size_t>(n_units) + 1);
        for (int32_t u = 0; u < n_units; ++u) {
            p->unit_seg_begin[u] = static_cast<int64_t>(p->segs.size());
            zero::cut_unit(p, u, seg_max, p->segs);
            p->unit_local_begin[u] = static_cast<int64_t>(p->segs_local.size());
            zero::cut_unit(p, u, zero::local_seg_len(p->S[u], seg_max), p->segs_local);
        }
        p->unit_seg_begin[n_units] = static_cast<int64_t>(p->segs.size());
        p->unit_local_begin[n_units] = static_cast<int64_t>(p->segs_local.size());
        p->unit_table.resize(n_units);
        for (int32_t u = 0; u < n_units; ++u)
            p->unit_table[u] = zero::UnitDesc{p->F[u], p->S[u], p->h[u], p->Hoff[u], p->sizes[u], p->unit_seg_begin[u]};
    } catch (const std::bad_alloc &) {
        delete p;
        return ZERO_ENOMEM;
    }
    *out = p;
    return ZERO_OK;
}

extern "C" void zero_plan_destroy(zero_plan *plan) { delete plan; }

extern "C" int zero_plan_query(const zero_plan *plan, int64_t *p_pad, int64_t *h, int64_t *F, int64_t *Hoff,
                               int64_t *S, int64_t *h_u) {
    if (plan == nullptr) return ZERO_EINVAL;
    const size_t n = static_cast<size_t>(plan->n_units);
    if (p_pad) *p_pad = plan->p_pad;
    if (h) *h = plan->H;
    if (F && n) std::memcpy(F, plan->F.data(), n * sizeof(int64_t));
    if (Hoff && n) std::memcpy(Hoff, plan->Hoff.data(), n * sizeof(int64_t));
    if (S && n) std::memcpy(S, plan->S.data(), n * sizeof(int64_t));
    if (h_u && n) std::memcpy(h_u, plan->h.data(), n * sizeof(int64_t));
    return ZERO_OK;
}

extern "C" int zero_plan_align(const zero_plan *plan, int32_t *align) {
    if (plan == nullptr || align == nullptr) return ZERO_EINVAL;
    *align = plan->align;
    return ZERO_OK;
}

extern "C" int zero_plan_counts(const zero_plan *plan, int32_t *n_units, int32_t *n_ranks, int64_t *n_segments) {
    if (plan == nullptr) return ZERO_EINVAL;
    if (n_units) *n_units = plan->n_units;
    if (n_ranks) *n_ranks = plan->n_ranks;
    if (n_segments) *n_segments = static_cast<int64_t>(plan->segs.size());
    return ZERO_OK;
}

extern "C" int zero_plan_segments(const zero_plan *plan, int64_t *out) {
    if (plan == nullptr || out == nullptr) return ZERO_EINVAL;
    for (size_t i = 0; i < plan->segs.size(); ++i) {
        const Seg &sg = plan->segs[i];
        int64_t *o = out + 6 * i;
        o[0] = sg.g_off;
        o[1] = sg.s_off;
        o[2] = sg.len;
        o[3] = sg.valid;
        o[4] = sg.rank;
        o[5] = sg.unit;
    }
    return ZERO_OK;
}

extern "C" int zero_plan_local_segments(const zero_plan *plan, int64_t *n_segments, int64_t *out) {
    if (plan == nullptr || n_segments == nullptr) return ZERO_EINVAL;
    *n_segments = static_cast<int64_t>(plan->segs_local.size());
    if (out == nullptr) return ZERO_OK;
    for (size_t i = 0; i < plan->segs_local.size(); ++i) {
        const Seg &sg = plan->segs_local[i];
        int64_t *o = out + 6 * i;
        o[0] = sg.g_off;
        o[1] = sg.s_off;
        o[2] = sg.len;
        o[3] = sg.valid;
        o[4] = sg.rank;
        o[5] = sg.unit;
    }
    return ZERO_OK;
}

extern "C" int zero_plan_workspace_bytes(const zero_plan *plan, size_t *bytes) {
    if (plan == nullptr || bytes == nullptr) return ZERO_EINVAL;
    *bytes = zero::workspace_layout(plan).total;
    return ZERO_OK;
}

extern "C" const char *zero_status_string(int status) {
    switch (status) {
        case ZERO_OK: return "ok";
        case ZERO_EINVAL: return "invalid argument";
        case ZERO_ENOMEM: return "out of memory (host) or workspace too small";
        case ZERO_ECUDA: return "CUDA runtime error";
        case ZERO_EALIGN: return "device pointer not 16-byte aligned";
        case ZERO_ENONFINITE: return "a clipped step was skipped: the global gradient norm was not finite";
        case ZERO_ETIMEOUT: return "a bounded wait inside a kernel expired: that work is incomplete";
        case ZERO_ENOTATTACHED: return "plan has no device workspace (call zero_plan_attach)";
        case ZERO_ERANGE: return "size beyond the fixed capacity of the allocation-free entry point";
        default: return "unknown status";
    }
}

extern "C" int zero_last_cuda_error(void) { return zero::g_last_cuda_error; }
