// Internal types shared by the host plan (zero_plan.cpp) and the kernels
// (zero_kernels.cu).  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/zero.h"

namespace zero {

// One work segment: a contiguous run of one rank's slice of one unit.  The
// multi-unit launch table lists every segment of every (unit, rank) slice,
// ordered by unit, then rank, then position; a kernel launch maps one CTA to
// one segment, so thousands of small units cost one launch, not thousands.
struct Seg {
    int64_t g_off;  // full-buffer position of the segment's first element: F_u + r*h_u + j0
    int64_t s_off;  // shard-buffer position of the same element: Hoff_u + j0
    int32_t len;    // elements in the segment (1..seg_max_for(N))
    int32_t valid;  // elements before the unit's padding starts (0..len)
    int32_t rank;
    int32_t unit;
};
static_assert(sizeof(Seg) == 32, "Seg must stay 32 bytes");

// Longest segment: 8192 elements for up to 8 ranks, 32256 for more (measured:
// at N = 8 the shorter segments shorten the tail of every launch, which per-unit
// and per-bucket launches pay each time; at N = 16 the longer segment fits the
// pipeline better, and 32256 is 21 whole tiles of its 1536 elements, so a full
// segment ends with no part-filled stage).  ZERO_SEG_MAX fixes one length for
// all N (for measurements).  Segments after the first one of a slice start at a
// shard position that is a multiple of 8, so 32-byte vector access needs no
// peeling.
constexpr int32_t kSegMaxSmallN = 8192, kSegMaxLargeN = 32256;

// The unit-local launch table: the same slices cut so that each unit has about
// kLocalSegsPerUnit segments (two per SM of a GB300) of at least kLocalSegMin
// elements, at most the main table's length.  Launches over one unit or a run
// of units without per-segment partial sums use it, so a small unit spreads
// over every SM instead of one SM per slice; the element-wise results do not
// depend on how the slices are cut.
constexpr int64_t kLocalSegsPerUnit = 304, kLocalSegMin = 1024;
inline int32_t seg_max_for(int32_t n_ranks) {
#ifdef ZERO_SEG_MAX
    (void)n_ranks;
    static_assert(ZERO_SEG_MAX >= 64 && ZERO_SEG_MAX % 8 == 0 && ZERO_SEG_MAX <= kSegMaxLargeN,
                  "segments hold whole 8-element groups");
    return ZERO_SEG_MAX;
#else
    return n_ranks <= 8 ? kSegMaxSmallN : kSegMaxLargeN;
#endif
}

// Per segment, the clip's sum of squares is kept as kPartialSlots partials
// (one per consumer warp of the pipelined kernel; unused slots hold 0), added
// later in a fixed order.  A partial is a binary32 pair (hi + lo, the warp's
// squares added in pair arithmetic) plus a binary64 part for values outside the
// pair's range; the binary64 work happens only when the partials are added up.
struct SqPartial {
    float hi, lo;
    double wide;
};
static_assert(sizeof(SqPartial) == 16, "SqPartial must stay 16 bytes");
constexpr int kPartialSlots = 16;

// Per-unit description, mirrored into the plan's device workspace.
struct UnitDesc {
    int64_t F;      // offset of the unit in the full buffer
    int64_t S;      // padded size (multiple of N)
    int64_t h;      // slice length S / N
    int64_t Hoff;   // offset of the unit's slice in every shard buffer
    int64_t size;   // true size s_u (positions >= size are padding)
    int64_t seg_begin;  // first launch-table segment of the unit
};
static_assert(sizeof(UnitDesc) == 48, "UnitDesc must stay 48 bytes");

// The binary32 constants of one AdamW step, computed once on the host
// (compiled without FMA contraction) from zero_hparams.
struct AdamConsts {
    float b1, b2;
    float omb1, omb2;  // 1 - b1, 1 - b2
    float decay;       // 1 - lr*wd
    float lr_bc1;      // lr / bc1
    float bc2, eps;
};

}  // namespace zero

struct zero_plan {
    int32_t n_units = 0, n_ranks = 0;
    int32_t align = 1;  // every slice length is a multiple of align (zero_plan_create_aligned)
    std::vector<int64_t> sizes, S, h, F, Hoff;
    int64_t p_pad = 0, H = 0;
    std::vector<zero::Seg> segs;           // host copy of the launch table
    std::vector<int64_t> unit_seg_begin;   // [n_units + 1]: segments of unit u
    std::vector<zero::Seg> segs_local;     // host copy of the unit-local launch table
    std::vector<int64_t> unit_local_begin;  // [n_units + 1]: its segments of unit u
    std::vector<zero::UnitDesc> unit_table;  // host copy of the device unit table
    // device side, set by zero_plan_attach
    bool attached = false;
    int device = -1;
    zero::Seg *d_segs = nullptr;
    zero::Seg *d_segs_local = nullptr;
    zero::SqPartial *d_partials = nullptr;  // kPartialSlots partial sums of squares per segment
    double *d_sqnorm = nullptr;     // S of the last clipped step
    float *d_coef = nullptr;        // clip coefficient of the last clipped step
    int *d_err = nullptr;           // device error word: non-zero after a bounded wait expired
    unsigned long long *d_tickets = nullptr;  // [2]: segment tickets and finished CTAs of a pipelined launch
    int *d_skipped = nullptr;       // non-zero after a clipped step found a non-finite norm (zero_plan_check)
    unsigned *d_fin_count = nullptr;  // blocks of the total's first pass done (0 between launches)
    double *d_fin_sums = nullptr;   // kFinBlocks per-block sums of the total's first pass
    zero::UnitDesc *d_units = nullptr;  // device unit table
};

namespace zero {
// Blocks of the fixed-order total of the partials (its first pass).
constexpr int kFinBlocks = 128;

// Workspace layout (byte offsets from the workspace base).
struct WsLayout {
    size_t segs, partials, scalars, units, fin, segs_local, total;
};
WsLayout workspace_layout(const zero_plan *plan);
int adam_consts(const zero_hparams *hp, AdamConsts *out);
void set_last_cuda_error(int code);
}  // namespace zero
