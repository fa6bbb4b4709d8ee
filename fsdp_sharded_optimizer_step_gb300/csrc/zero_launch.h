// Launch interface between the C-ABI layer (zero_abi.cu: argument checks,
// parameter blocks) and the sm_103a kernels (zero_kernels.cu).  Not part of
// the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "zero_internal.h"

namespace zero {

// MODE_FUSED:  N gradient rows + master/m/v -> master/m/v + params (one pass)
// MODE_REDUCE: N gradient rows -> fp32 gradient shard and/or per-segment
//              binary64 sums of squares of the averaged gradient
// MODE_SHARD:  fp32 gradient shard (x device clip coefficient) + master/m/v
//              -> master/m/v + params
enum { MODE_FUSED = 0, MODE_REDUCE = 1, MODE_SHARD = 2 };

// Kernel parameter block, passed by value to every launch.
struct KParams {
    const Seg *segs;
    int64_t seg_base;       // first segment of this launch
    int32_t n_ranks;
    int32_t pdtype;
    int32_t pow2;           // N is a power of two: g = acc * inv_n is bit-identical to acc / N
    float inv_n, nf;
    AdamConsts c;
    float coef;             // host clip coefficient (reduce-scatter); 1 = none
    int32_t write_g, want_partials, use_coef_dev;
    SqPartial *partials;    // kPartialSlots per segment, indexed by absolute segment number
    int *err;               // device error word (a bounded wait expired)
    int32_t tile, stages;   // pipeline geometry of k_pipe
    int64_t p_pad, h_len;   // element counts of full-length and shard buffers
    int64_t g_origin;       // full position of element 0 of each gradient row (0, or F_u for unit-local rows)
    int64_t g_len;          // elements in each gradient row (P_pad, or S_u for unit-local rows)
    int64_t drop_tile;      // testing aid: the copies of this tile of segment 0 are skipped (-1: none)
    unsigned long long *tickets;  // k_pipe's schedule: [0] next segment ticket, [1] CTAs done (0, 0 between launches)
    const float *coef_dev;  // device clip coefficient (NaN: skip the step)
    void *full;
    const void *grads[ZERO_MAX_RANKS];
    float *master[ZERO_MAX_RANKS];
    float *m[ZERO_MAX_RANKS];
    float *v[ZERO_MAX_RANKS];
    void *pshard[ZERO_MAX_RANKS];
    float *gshard[ZERO_MAX_RANKS];
};

// Status of the last launch (ZERO_ECUDA with the CUDA error recorded).
int launch_status();

// One pipelined launch in `mode` over segments [kp.seg_base, kp.seg_base + nseg)
// (fills the pipeline geometry into kp).
int launch_pipe(int mode, int gd, int64_t nseg, KParams &kp, cudaStream_t st);

// Fixed-order total of all of the plan's per-segment partials into its S
// (and *sqnorm_out, a device binary64, when not null); with max_norm > 0 also
// the clip coefficient (NaN and the skipped flag set when S is not finite).
int launch_finalize(const zero_plan *plan, float max_norm, double *sqnorm_out, cudaStream_t st);

// Gather of `count` segments from kp.seg_base: rank shards (kp.pshard) into kp.full.
int launch_gather(int64_t count, const KParams &kp, cudaStream_t st);

// Testing aid: the next pipelined launch skips the copies of tile `tile` of its first segment.
void arm_drop_tile(int64_t tile);

// Reduce-scatter + average of units [u0, u1) from full-length gradient rows into
// the fp32 gradient shard, one launch; with want_partials also the units'
// per-segment sums of squares (at their table positions in the workspace).
// The plan must be attached to the current device (checked by the caller).
int reduce_units(const zero_plan *plan, int32_t u0, int32_t u1, const void *const *grads, int32_t gdtype,
                 float *const *gshard, bool want_partials, cudaStream_t st);

}  // namespace zero
