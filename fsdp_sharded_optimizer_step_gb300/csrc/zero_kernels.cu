// Kernels of the sharded optimizer step for sm_103a, and the C-ABI entry
// points that launch them.
//
// The path is element-wise and HBM-bound (no contraction, so no tensor
// cores): per padded element the fused step reads N gradients plus master/m/v
// and writes master/m/v plus the gathered param.  The kernels therefore aim
// at bytes in flight: one CTA per launch-table segment, 256 threads, each
// thread moving 8 consecutive elements per iteration with 16/32-byte vector
// accesses (all N gradient rows loaded before the first add), streaming cache
// hints on data touched once.
//
// Exactness: every float operation uses an explicit _rn intrinsic in the
// order the header documents ("ZeRO and FSDP sharding", Code, AdamW::step),
// and the file is compiled with --fmad=false: nothing is contracted.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "zero_internal.h"

namespace zero {

constexpr int kThreads = 256;
#ifndef ZERO_PIPE_CONSUMER_WARPS
#define ZERO_PIPE_CONSUMER_WARPS 16
#endif
constexpr int kConsumerWarps = ZERO_PIPE_CONSUMER_WARPS;
constexpr int kPipeThreads = (kConsumerWarps + 1) * 32;

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
    double *partials;       // per segment, indexed by absolute segment number
    int *err;               // device error word (a bounded wait expired)
    int32_t tile, stages;   // pipeline geometry of k_fused_pipe
    int64_t p_pad, h_len;   // element counts of full-length and shard buffers (diagnostic bounds checks)
    const float *coef_dev;  // device clip coefficient (NaN: skip the step)
    void *full;
    const void *grads[ZERO_MAX_RANKS];
    float *master[ZERO_MAX_RANKS];
    float *m[ZERO_MAX_RANKS];
    float *v[ZERO_MAX_RANKS];
    void *pshard[ZERO_MAX_RANKS];
    float *gshard[ZERO_MAX_RANKS];
};

// Diagnostic build (-DZERO_SELFCHECK): every shared/global access of the
// pipeline is checked against its buffer and alignment first; a failed check
// records its code in *err and the access is skipped.
#ifdef ZERO_SELFCHECK
__device__ __forceinline__ bool guard_ok(bool ok, int code, int *err) {
    if (!ok) atomicCAS(err, 0, code);
    return ok;
}
#define ZERO_GUARD(cond, code) guard_ok((cond), (code), p.err)
#else
#define ZERO_GUARD(cond, code) true
#endif

__device__ __forceinline__ bool aligned_to(const void *ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0;
}

// ------------------------------------------------------------------ element math
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// binary32 -> bfloat16, round to nearest even: add 0x7FFF plus the lowest kept
// bit, then drop the low half (the carry moves into the exponent correctly,
// overflow gives inf).  A NaN keeps its sign and top payload, quiet bit set.
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (u >> 16) | 0x0040u;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return u >> 16;
}

__device__ __forceinline__ float average(float acc, const KParams &p) {
    return p.pow2 ? __fmul_rn(acc, p.inv_n) : __fdiv_rn(acc, p.nf);
}

// One AdamW element in the page's operation order; every op rounded alone.
__device__ __forceinline__ void adamw(float g, float &w, float &m, float &v, const AdamConsts &c) {
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(__fmul_rn(c.omb2, g), g));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), c.bc2), c.eps);
    w = __fsub_rn(__fmul_rn(w, c.decay), __fdiv_rn(__fmul_rn(c.lr_bc1, m), den));
}

template <int GD>
__device__ __forceinline__ float load_grad1(const void *base, int64_t i) {
    if (GD == ZERO_BF16) return bf16_bits_to_f32(__ldcs(static_cast<const unsigned short *>(base) + i));
    return __ldcs(static_cast<const float *>(base) + i);
}

// 8 consecutive gradient values of one rank.  vec: the position is 16-byte
// aligned for bf16 / 32-byte for fp32 (host and segment layout guarantee it).
template <int GD>
struct Grad8 {
    uint4 raw[GD == ZERO_BF16 ? 1 : 2];
};

template <int GD>
__device__ __forceinline__ void load_grad8(const void *base, int64_t i, bool vec, Grad8<GD> &out) {
    if constexpr (GD == ZERO_BF16) {
        const unsigned short *b = static_cast<const unsigned short *>(base) + i;
        if (vec) {
            out.raw[0] = __ldcs(reinterpret_cast<const uint4 *>(b));
        } else {
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = __ldcs(b + e);
            out.raw[0] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
    } else {
        const float *f = static_cast<const float *>(base) + i;
        if (vec) {
            const float4 a = __ldcs(reinterpret_cast<const float4 *>(f));
            const float4 b = __ldcs(reinterpret_cast<const float4 *>(f) + 1);
            out.raw[0] = make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z), __float_as_uint(a.w));
            out.raw[1] = make_uint4(__float_as_uint(b.x), __float_as_uint(b.y), __float_as_uint(b.z), __float_as_uint(b.w));
        } else {
            uint32_t x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __float_as_uint(__ldcs(f + e));
            out.raw[0] = make_uint4(x[0], x[1], x[2], x[3]);
            out.raw[1] = make_uint4(x[4], x[5], x[6], x[7]);
        }
    }
}

template <int GD>
__device__ __forceinline__ void unpack8(const Grad8<GD> &g, float (&x)[8]) {
    if constexpr (GD == ZERO_BF16) {
        const uint4 r = g.raw[0];
        x[0] = __uint_as_float(r.x << 16); x[1] = __uint_as_float(r.x & 0xFFFF0000u);
        x[2] = __uint_as_float(r.y << 16); x[3] = __uint_as_float(r.y & 0xFFFF0000u);
        x[4] = __uint_as_float(r.z << 16); x[5] = __uint_as_float(r.z & 0xFFFF0000u);
        x[6] = __uint_as_float(r.w << 16); x[7] = __uint_as_float(r.w & 0xFFFF0000u);
    } else {
        x[0] = __uint_as_float(g.raw[0].x); x[1] = __uint_as_float(g.raw[0].y);
        x[2] = __uint_as_float(g.raw[0].z); x[3] = __uint_as_float(g.raw[0].w);
        x[4] = __uint_as_float(g.raw[1].x); x[5] = __uint_as_float(g.raw[1].y);
        x[6] = __uint_as_float(g.raw[1].z); x[7] = __uint_as_float(g.raw[1].w);
    }
}

// Reduce-scatter of 8 elements: the rank-ordered fold over all N rows.  With
// a compile-time N every row is loaded before the first add, so N+ loads are
// in flight per thread.
template <int GD, int NR>
__device__ __forceinline__ void fold8(const KParams &p, int64_t gpos, bool vec, float (&acc)[8]) {
    if constexpr (NR > 0) {
        Grad8<GD> rows[NR > 0 ? NR : 1];
#pragma unroll
        for (int q = 0; q < NR; ++q) load_grad8<GD>(p.grads[q], gpos, vec, rows[q]);
        unpack8<GD>(rows[0], acc);
#pragma unroll
        for (int q = 1; q < NR; ++q) {
            float x[8];
            unpack8<GD>(rows[q], x);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
        }
    } else {
        Grad8<GD> row;
        load_grad8<GD>(p.grads[0], gpos, vec, row);
        unpack8<GD>(row, acc);
        for (int q = 1; q < p.n_ranks; ++q) {
            load_grad8<GD>(p.grads[q], gpos, vec, row);
            float x[8];
            unpack8<GD>(row, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
        }
    }
}

template <int GD, int NR>
__device__ __forceinline__ float fold1(const KParams &p, int64_t gpos) {
    float acc = load_grad1<GD>(p.grads[0], gpos);
    const int n = NR > 0 ? NR : p.n_ranks;
#pragma unroll
    for (int q = 1; q < n; ++q) acc = __fadd_rn(acc, load_grad1<GD>(p.grads[q], gpos));
    return acc;
}

__device__ __forceinline__ void load8(const float *src, float (&x)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(src));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(src) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void store8(float *dst, const float (&x)[8]) {
    __stcs(reinterpret_cast<float4 *>(dst), make_float4(x[0], x[1], x[2], x[3]));
    __stcs(reinterpret_cast<float4 *>(dst) + 1, make_float4(x[4], x[5], x[6], x[7]));
}

// Writes 8 params (bf16 or fp32) at dst + i; vec: 16-byte (bf16) / 32-byte (fp32) aligned.
__device__ __forceinline__ void store_param8(void *base, int64_t i, int32_t pdtype, bool vec, const float (&w)[8]) {
    if (pdtype == ZERO_BF16) {
        unsigned short *d = static_cast<unsigned short *>(base) + i;
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = f32_to_bf16_rne(w[e]);
        if (vec) {
            __stcs(reinterpret_cast<uint4 *>(d), make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16),
                                                            h[4] | (h[5] << 16), h[6] | (h[7] << 16)));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) d[e] = static_cast<unsigned short>(h[e]);
        }
    } else {
        float *d = static_cast<float *>(base) + i;
        if (vec) {
            store8(d, w);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) d[e] = w[e];
        }
    }
}

__device__ __forceinline__ void store_param1(void *base, int64_t i, int32_t pdtype, float w) {
    if (pdtype == ZERO_BF16) static_cast<unsigned short *>(base)[i] = static_cast<unsigned short>(f32_to_bf16_rne(w));
    else static_cast<float *>(base)[i] = w;
}

// Elements [k0, k0 + 8*ngroups) of a segment go through 8-wide groups; the
// head (before the shard position reaches a multiple of 8) and the tail go
// one element at a time.
struct SegSplit {
    int k0, ngroups, tail0;
    bool gvec;  // full/gradient positions are aligned like the shard positions
};

__device__ __forceinline__ SegSplit split_segment(const Seg &sg) {
    SegSplit s;
    s.k0 = static_cast<int>((8 - (sg.s_off & 7)) & 7);
    if (s.k0 > sg.len) s.k0 = sg.len;
    s.ngroups = (sg.len - s.k0) >> 3;
    s.tail0 = s.k0 + 8 * s.ngroups;
    s.gvec = ((sg.g_off + s.k0) & 7) == 0;
    return s;
}

// ------------------------------------------------------------------ fused step
// reduce-scatter + average + AdamW + cast + all-gather, one pass.

// Direct (register) path for one segment, spread over nthr threads: the
// 8-wide groups of [k0, tail0) when `body` is set, and always the head and
// tail elements.
template <int GD, int NR>
__device__ __forceinline__ void fused_direct(const KParams &p, const Seg &sg, const SegSplit &sp, int tid, int nthr,
                                             bool body) {
    const int r = sg.rank;
    float *__restrict__ W = p.master[r] + sg.s_off;
    float *__restrict__ M = p.m[r] + sg.s_off;
    float *__restrict__ V = p.v[r] + sg.s_off;
    void *full = p.full;
    void *ps = p.pshard[r];
    if (body) {
        for (int i = tid; i < sp.ngroups; i += nthr) {
            const int k = sp.k0 + 8 * i;
            if (!ZERO_GUARD(k + 8 <= sg.len && sg.s_off + k + 8 <= p.h_len && sg.g_off + k + 8 <= p.p_pad &&
                                aligned_to(W + k, 16),
                            30))
                continue;
            float acc[8], w[8], m[8], v[8];
            fold8<GD, NR>(p, sg.g_off + k, sp.gvec, acc);
            load8(W + k, w);
            load8(M + k, m);
            load8(V + k, v);
            if (k + 8 > sg.valid) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (k + e >= sg.valid) acc[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) adamw(average(acc[e], p), w[e], m[e], v[e], p.c);
            store8(W + k, w);
            store8(M + k, m);
            store8(V + k, v);
            if (full != nullptr) store_param8(full, sg.g_off + k, p.pdtype, sp.gvec, w);
            if (ps != nullptr) store_param8(ps, sg.s_off + k, p.pdtype, true, w);
        }
    }
    // head and tail, one element per thread
    const int nedge = sp.k0 + (sg.len - sp.tail0);
    for (int t = tid; t < nedge; t += nthr) {
        const int k = t < sp.k0 ? t : sp.tail0 + (t - sp.k0);
        if (!ZERO_GUARD(k >= 0 && k < sg.len && sg.s_off + k < p.h_len && sg.g_off + k < p.p_pad, 31)) continue;
        float acc = fold1<GD, NR>(p, sg.g_off + k);
        if (k >= sg.valid) acc = 0.0f;
        float w = W[k], m = M[k], v = V[k];
        adamw(average(acc, p), w, m, v, p.c);
        W[k] = w;
        M[k] = m;
        V[k] = v;
        if (full != nullptr) store_param1(full, sg.g_off + k, p.pdtype, w);
        if (ps != nullptr) store_param1(ps, sg.s_off + k, p.pdtype, w);
    }
}

// ------------------------------------------------------------------ fused step, bulk-copy pipeline
// Persistent, warp-specialised: CTA b takes segments b, b + gridDim.x, ...
// One producer thread streams each aligned segment body, tile by tile, into a
// ring of `stages` shared-memory buffers with 1-D bulk copies (cp.async.bulk,
// completion counted in bytes on a per-stage mbarrier): the N gradient rows
// and master/m/v of `tile` elements.  The consumer warps wait for a stage,
// compute from shared memory, store master/m/v and the params straight to
// global memory, and release the stage.  Copies stay in flight while the
// consumers compute, which the register-only kernel cannot do.  Heads, tails
// and segments whose gradient positions are not aligned like their shard
// positions take the direct path in the consumer warps.
//
// Every wait is bounded (kWaitLimitNs of %globaltimer): on expiry the waiting
// thread records the failure in *p.err, stops issuing work, and the producer
// waits (again bounded) for the copies it already issued before the CTA exits.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the phase of `bar` with the given parity has completed, for at
// most kWaitLimitNs; false on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
#ifdef ZERO_PIPE_EVICT_FIRST
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
#else
    (void)policy;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst_smem)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
#endif
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol = 0;
#ifdef ZERO_PIPE_EVICT_FIRST
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#endif
    return pol;
}

// Stage layout: N gradient rows of `tile` elements, then master, m, v.
struct StageLayout {
    uint32_t grad_row_bytes, state_off, bytes;
};

__device__ __forceinline__ StageLayout stage_layout(int n_ranks, int gbytes, int tile) {
    StageLayout L;
    L.grad_row_bytes = static_cast<uint32_t>(tile * gbytes);
    L.state_off = L.grad_row_bytes * n_ranks;
    L.bytes = L.state_off + 3u * static_cast<uint32_t>(tile) * 4u;
    return L;
}

template <int GD, int NR>
__global__ void __launch_bounds__(kPipeThreads, 1) k_fused_pipe(const KParams p, int64_t nseg) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int GB = GD == ZERO_BF16 ? 2 : 4;
    const int n = NR > 0 ? NR : p.n_ranks;
    const int tile = p.tile, stages = p.stages;
    const StageLayout L = stage_layout(n, GB, tile);
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(stages) * L.bytes);
    uint64_t *empty_bar = full_bar + stages;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumerWarps);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer
        if (lane != 0) return;
        const uint64_t pol = evict_first_policy();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;  // per stage: copies issued at least once, parity of the last
        bool ok = true;
        for (int64_t si = blockIdx.x; si < nseg && ok; si += gridDim.x) {
            const Seg sg = p.segs[p.seg_base + si];
            const SegSplit sp = split_segment(sg);
            if (!sp.gvec) continue;
            const int r = sg.rank;
            for (int k = sp.k0; k < sp.tail0; k += tile) {
                const int len = min(tile, sp.tail0 - k);
                if (!mbar_wait(&empty_bar[stage], phase ^ 1u) || *reinterpret_cast<volatile int *>(&abort_flag)) {
                    ok = false;
                    break;
                }
                unsigned char *buf = smem + static_cast<size_t>(stage) * L.bytes;
                const uint32_t gbytes = static_cast<uint32_t>(len * GB), sbytes = static_cast<uint32_t>(len * 4);
                if (!ZERO_GUARD(len > 0 && len <= tile && (gbytes & 15u) == 0 && sg.g_off + k + len <= p.p_pad &&
                                    sg.s_off + k + len <= p.h_len && r >= 0 && r < n && stage >= 0 && stage < stages,
                                10)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full_bar[stage], gbytes * n + 3u * sbytes);
                for (int q = 0; q < n; ++q) {
                    const unsigned char *src = static_cast<const unsigned char *>(p.grads[q]) + (sg.g_off + k) * GB;
                    if (ZERO_GUARD(aligned_to(src, 16) && aligned_to(buf + q * L.grad_row_bytes, 16), 11))
                        bulk_load(buf + q * L.grad_row_bytes, src, gbytes, &full_bar[stage], pol);
                }
                unsigned char *st = buf + L.state_off;
                if (ZERO_GUARD(aligned_to(p.master[r] + sg.s_off + k, 16) && aligned_to(p.m[r] + sg.s_off + k, 16) &&
                                   aligned_to(p.v[r] + sg.s_off + k, 16) && aligned_to(st, 16) &&
                                   L.state_off + 3u * static_cast<uint32_t>(tile) * 4u <= L.bytes,
                               12)) {
                    bulk_load(st, p.master[r] + sg.s_off + k, sbytes, &full_bar[stage], pol);
                    bulk_load(st + tile * 4, p.m[r] + sg.s_off + k, sbytes, &full_bar[stage], pol);
                    bulk_load(st + 2 * tile * 4, p.v[r] + sg.s_off + k, sbytes, &full_bar[stage], pol);
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            atomicExch(p.err, 1);
            abort_flag = 1;
            // drain: wait (bounded) for the last copies issued into each stage
            for (int s = 0; s < stages; ++s)
                if (issued_mask & (1u << s)) mbar_wait(&full_bar[s], (issued_parity >> s) & 1u);
        }
        return;
    }

    // ---------------- consumers: every consumer warp takes every tile, so each
    // stage's mbarrier phases are always waited on in order by the same warps
    // (a stage shared between consumer sets that alternate would let a waiter
    // for phase k pass while the barrier is still in phase k-1: the parity of
    // phase k then reads as already complete).
    const int ct = threadIdx.x;  // 0 .. kConsumerWarps*32 - 1
    constexpr int CT = kConsumerWarps * 32;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t si = blockIdx.x; si < nseg; si += gridDim.x) {
        const Seg sg = p.segs[p.seg_base + si];
        const SegSplit sp = split_segment(sg);
        fused_direct<GD, NR>(p, sg, sp, ct, CT, !sp.gvec);
        if (!sp.gvec) continue;
        const int r = sg.rank;
        float *__restrict__ Wg = p.master[r] + sg.s_off;
        float *__restrict__ Mg = p.m[r] + sg.s_off;
        float *__restrict__ Vg = p.v[r] + sg.s_off;
        void *full = p.full;
        void *ps = p.pshard[r];
        for (int k = sp.k0; k < sp.tail0; k += tile) {
            const int len = min(tile, sp.tail0 - k);
            if (!mbar_wait(&full_bar[stage], phase) || *reinterpret_cast<volatile int *>(&abort_flag)) {
                if (lane == 0) atomicExch(p.err, 2);
                abort_flag = 1;
                return;
            }
            const unsigned char *buf = smem + static_cast<size_t>(stage) * L.bytes;
            const float *Ws = reinterpret_cast<const float *>(buf + L.state_off);
            const float *Ms = Ws + tile;
            const float *Vs = Ms + tile;
            for (int e = 4 * ct; e < len; e += 4 * CT) {
                if (!ZERO_GUARD(e + 4 <= tile && sg.s_off + k + e + 4 <= p.h_len && sg.g_off + k + e + 4 <= p.p_pad &&
                                    aligned_to(Wg + k + e, 16) && aligned_to(Ws + e, 16) &&
                                    (full == nullptr || aligned_to(static_cast<unsigned char *>(full) + (sg.g_off + k + e) * (p.pdtype == ZERO_BF16 ? 2 : 4), p.pdtype == ZERO_BF16 ? 8 : 16)),
                                20))
                    continue;
                float acc[4];
                if constexpr (GD == ZERO_BF16) {
                    const uint2 x0 = *reinterpret_cast<const uint2 *>(buf + e * 2);
                    acc[0] = __uint_as_float(x0.x << 16); acc[1] = __uint_as_float(x0.x & 0xFFFF0000u);
                    acc[2] = __uint_as_float(x0.y << 16); acc[3] = __uint_as_float(x0.y & 0xFFFF0000u);
#pragma unroll
                    for (int q = 1; q < (NR > 0 ? NR : ZERO_MAX_RANKS); ++q) {
                        if (NR == 0 && q >= n) break;
                        const uint2 x = *reinterpret_cast<const uint2 *>(buf + q * L.grad_row_bytes + e * 2);
                        acc[0] = __fadd_rn(acc[0], __uint_as_float(x.x << 16));
                        acc[1] = __fadd_rn(acc[1], __uint_as_float(x.x & 0xFFFF0000u));
                        acc[2] = __fadd_rn(acc[2], __uint_as_float(x.y << 16));
                        acc[3] = __fadd_rn(acc[3], __uint_as_float(x.y & 0xFFFF0000u));
                    }
                } else {
                    const float4 x0 = *reinterpret_cast<const float4 *>(buf + e * 4);
                    acc[0] = x0.x; acc[1] = x0.y; acc[2] = x0.z; acc[3] = x0.w;
#pragma unroll
                    for (int q = 1; q < (NR > 0 ? NR : ZERO_MAX_RANKS); ++q) {
                        if (NR == 0 && q >= n) break;
                        const float4 x = *reinterpret_cast<const float4 *>(buf + q * L.grad_row_bytes + e * 4);
                        acc[0] = __fadd_rn(acc[0], x.x);
                        acc[1] = __fadd_rn(acc[1], x.y);
                        acc[2] = __fadd_rn(acc[2], x.z);
                        acc[3] = __fadd_rn(acc[3], x.w);
                    }
                }
                const float4 w4 = *reinterpret_cast<const float4 *>(Ws + e);
                const float4 m4 = *reinterpret_cast<const float4 *>(Ms + e);
                const float4 v4 = *reinterpret_cast<const float4 *>(Vs + e);
                float w[4] = {w4.x, w4.y, w4.z, w4.w}, m[4] = {m4.x, m4.y, m4.z, m4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
                const int kk = k + e;
                if (kk + 4 > sg.valid) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (kk + i >= sg.valid) acc[i] = 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) adamw(average(acc[i], p), w[i], m[i], v[i], p.c);
                __stcs(reinterpret_cast<float4 *>(Wg + kk), make_float4(w[0], w[1], w[2], w[3]));
                __stcs(reinterpret_cast<float4 *>(Mg + kk), make_float4(m[0], m[1], m[2], m[3]));
                __stcs(reinterpret_cast<float4 *>(Vg + kk), make_float4(v[0], v[1], v[2], v[3]));
                if (p.pdtype == ZERO_BF16) {
                    const uint2 h = make_uint2(f32_to_bf16_rne(w[0]) | (f32_to_bf16_rne(w[1]) << 16),
                                               f32_to_bf16_rne(w[2]) | (f32_to_bf16_rne(w[3]) << 16));
                    if (full != nullptr) __stcs(reinterpret_cast<uint2 *>(static_cast<unsigned short *>(full) + sg.g_off + kk), h);
                    if (ps != nullptr) __stcs(reinterpret_cast<uint2 *>(static_cast<unsigned short *>(ps) + sg.s_off + kk), h);
                } else {
                    const float4 f = make_float4(w[0], w[1], w[2], w[3]);
                    if (full != nullptr) __stcs(reinterpret_cast<float4 *>(static_cast<float *>(full) + sg.g_off + kk), f);
                    if (ps != nullptr) __stcs(reinterpret_cast<float4 *>(static_cast<float *>(ps) + sg.s_off + kk), f);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// ------------------------------------------------------------------ reduce-scatter / sum of squares
// Writes the averaged (optionally coef-scaled) gradient shard and/or the
// segment's binary64 sum of squares of the averaged gradient (each square is
// exact in binary64; the block adds them in a fixed order).
__device__ __forceinline__ double block_sum(double x, double *smem) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xFFFFFFFFu, x, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) smem[warp] = x;
    __syncthreads();
    double s = 0.0;
    if (warp == 0) {
        s = lane < (blockDim.x >> 5) ? smem[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_down_sync(0xFFFFFFFFu, s, o));
    }
    return s;  // valid in thread 0
}

template <int GD, int NR>
__global__ void __launch_bounds__(kThreads, 2) k_reduce(const KParams p) {
    __shared__ double smem[kThreads / 32];
    const Seg sg = p.segs[p.seg_base + blockIdx.x];
    const SegSplit sp = split_segment(sg);
    float *__restrict__ G = p.write_g ? p.gshard[sg.rank] + sg.s_off : nullptr;
    const bool scale = p.coef != 1.0f;
    double sq = 0.0;
    for (int i = threadIdx.x; i < sp.ngroups; i += kThreads) {
        const int k = sp.k0 + 8 * i;
        float acc[8];
        fold8<GD, NR>(p, sg.g_off + k, sp.gvec, acc);
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            g[e] = (k + e >= sg.valid) ? 0.0f : average(acc[e], p);
            if (scale) g[e] = __fmul_rn(g[e], p.coef);
            const double d = static_cast<double>(g[e]);
            sq = __dadd_rn(sq, __dmul_rn(d, d));
        }
        if (G != nullptr) store8(G + k, g);
    }
    const int nedge = sp.k0 + (sg.len - sp.tail0);
    for (int t = threadIdx.x; t < nedge; t += kThreads) {
        const int k = t < sp.k0 ? t : sp.tail0 + (t - sp.k0);
        float g = (k >= sg.valid) ? 0.0f : average(fold1<GD, NR>(p, sg.g_off + k), p);
        if (scale) g = __fmul_rn(g, p.coef);
        const double d = static_cast<double>(g);
        sq = __dadd_rn(sq, __dmul_rn(d, d));
        if (G != nullptr) G[k] = g;
    }
    if (p.want_partials) {
        const double s = block_sum(sq, smem);
        if (threadIdx.x == 0) p.partials[p.seg_base + blockIdx.x] = s;
    }
}

// One CTA adds the per-segment partials in a fixed order (thread t takes
// segments t, t+1024, ... in sequence, then a fixed tree), writes S and, when
// max_norm > 0, the clip coefficient min(1, max_norm / (sqrt(S) + 1e-6))
// rounded once to binary32 (NaN when S is not finite: the update then skips).
constexpr int kFinThreads = 1024;
__global__ void __launch_bounds__(kFinThreads) k_finalize(const double *partials, int64_t nseg, float max_norm,
                                                          double *sqnorm_ws, double *sqnorm_out, float *coef_out) {
    __shared__ double smem[kFinThreads / 32];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < nseg; i += kFinThreads) s = __dadd_rn(s, partials[i]);
    const double S = block_sum(s, smem);
    if (threadIdx.x == 0) {
        *sqnorm_ws = S;
        if (sqnorm_out != nullptr) *sqnorm_out = S;
        if (max_norm > 0.0f) {
            float coef;
            if (!isfinite(S)) {
                coef = __int_as_float(0x7FC00000);
            } else {
                double c = __ddiv_rn(static_cast<double>(max_norm), __dadd_rn(__dsqrt_rn(S), 1e-6));
                if (c > 1.0) c = 1.0;
                coef = __double2float_rn(c);
            }
            *coef_out = coef;
        }
    }
}

// ------------------------------------------------------------------ AdamW from a gradient shard
__global__ void __launch_bounds__(kThreads, 2) k_adamw_shard(const KParams p) {
    float coef = 1.0f;
    if (p.use_coef_dev) {
        coef = *p.coef_dev;
        if (coef != coef) return;  // non-finite global norm: the step is skipped
    }
    const Seg sg = p.segs[p.seg_base + blockIdx.x];
    const SegSplit sp = split_segment(sg);
    const int r = sg.rank;
    const float *__restrict__ G = p.gshard[r] + sg.s_off;
    float *__restrict__ W = p.master[r] + sg.s_off;
    float *__restrict__ M = p.m[r] + sg.s_off;
    float *__restrict__ V = p.v[r] + sg.s_off;
    void *full = p.full;
    void *ps = p.pshard[r];
    const bool scale = p.use_coef_dev != 0;
    for (int i = threadIdx.x; i < sp.ngroups; i += kThreads) {
        const int k = sp.k0 + 8 * i;
        float g[8], w[8], m[8], v[8];
        load8(G + k, g);
        load8(W + k, w);
        load8(M + k, m);
        load8(V + k, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float ge = scale ? __fmul_rn(g[e], coef) : g[e];
            adamw(ge, w[e], m[e], v[e], p.c);
        }
        store8(W + k, w);
        store8(M + k, m);
        store8(V + k, v);
        if (full != nullptr) store_param8(full, sg.g_off + k, p.pdtype, sp.gvec, w);
        if (ps != nullptr) store_param8(ps, sg.s_off + k, p.pdtype, true, w);
    }
    const int nedge = sp.k0 + (sg.len - sp.tail0);
    for (int t = threadIdx.x; t < nedge; t += kThreads) {
        const int k = t < sp.k0 ? t : sp.tail0 + (t - sp.k0);
        const float ge = scale ? __fmul_rn(G[k], coef) : G[k];
        float w = W[k], m = M[k], v = V[k];
        adamw(ge, w, m, v, p.c);
        W[k] = w;
        M[k] = m;
        V[k] = v;
        if (full != nullptr) store_param1(full, sg.g_off + k, p.pdtype, w);
        if (ps != nullptr) store_param1(ps, sg.s_off + k, p.pdtype, w);
    }
}

// ------------------------------------------------------------------ all-gather
// full[F_u + r h_u + j] = shard[r][Hoff_u + j]: a copy per segment, 16-byte
// vectors where the full position is aligned like the shard position.
__global__ void __launch_bounds__(kThreads) k_gather(const KParams p) {
    const Seg sg = p.segs[p.seg_base + blockIdx.x];
    const SegSplit sp = split_segment(sg);
    const int esz = p.pdtype == ZERO_BF16 ? 2 : 4;
    const char *src = static_cast<const char *>(p.pshard[sg.rank]) + sg.s_off * esz;
    char *dst = static_cast<char *>(p.full) + sg.g_off * esz;
    for (int i = threadIdx.x; i < sp.ngroups; i += kThreads) {
        const int k = sp.k0 + 8 * i;
        if (esz == 2) {
            const uint4 x = __ldcs(reinterpret_cast<const uint4 *>(src + k * 2));
            if (sp.gvec) {
                __stcs(reinterpret_cast<uint4 *>(dst + k * 2), x);
            } else {
                unsigned short *d = reinterpret_cast<unsigned short *>(dst) + k;
                const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    d[2 * e] = static_cast<unsigned short>(w4[e] & 0xFFFFu);
                    d[2 * e + 1] = static_cast<unsigned short>(w4[e] >> 16);
                }
            }
        } else {
            float x[8];
            load8(reinterpret_cast<const float *>(src) + k, x);
            float *d = reinterpret_cast<float *>(dst) + k;
            if (sp.gvec) {
                store8(d, x);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) d[e] = x[e];
            }
        }
    }
    const int nedge = sp.k0 + (sg.len - sp.tail0);
    for (int t = threadIdx.x; t < nedge; t += kThreads) {
        const int k = t < sp.k0 ? t : sp.tail0 + (t - sp.k0);
        if (esz == 2) reinterpret_cast<unsigned short *>(dst)[k] = reinterpret_cast<const unsigned short *>(src)[k];
        else reinterpret_cast<float *>(dst)[k] = reinterpret_cast<const float *>(src)[k];
    }
}

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
}

static int launch_status() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    return ZERO_OK;
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

#define ZERO_KERNEL_DISPATCH(kernel)                                                                 \
    static void launch_##kernel(int gd, int nr, dim3 grid, cudaStream_t st, const KParams &kp) {     \
        if (gd == ZERO_BF16) {                                                                       \
            switch (nr) {                                                                            \
                case 1: kernel<ZERO_BF16, 1><<<grid, kThreads, 0, st>>>(kp); break;                  \
                case 2: kernel<ZERO_BF16, 2><<<grid, kThreads, 0, st>>>(kp); break;                  \
                case 4: kernel<ZERO_BF16, 4><<<grid, kThreads, 0, st>>>(kp); break;                  \
                case 8: kernel<ZERO_BF16, 8><<<grid, kThreads, 0, st>>>(kp); break;                  \
                case 16: kernel<ZERO_BF16, 16><<<grid, kThreads, 0, st>>>(kp); break;                \
                default: kernel<ZERO_BF16, 0><<<grid, kThreads, 0, st>>>(kp); break;                 \
            }                                                                                        \
        } else {                                                                                     \
            switch (nr) {                                                                            \
                case 1: kernel<ZERO_F32, 1><<<grid, kThreads, 0, st>>>(kp); break;                   \
                case 2: kernel<ZERO_F32, 2><<<grid, kThreads, 0, st>>>(kp); break;                   \
                case 4: kernel<ZERO_F32, 4><<<grid, kThreads, 0, st>>>(kp); break;                   \
                case 8: kernel<ZERO_F32, 8><<<grid, kThreads, 0, st>>>(kp); break;                   \
                case 16: kernel<ZERO_F32, 16><<<grid, kThreads, 0, st>>>(kp); break;                 \
                default: kernel<ZERO_F32, 0><<<grid, kThreads, 0, st>>>(kp); break;                  \
            }                                                                                        \
        }                                                                                            \
    }

ZERO_KERNEL_DISPATCH(k_reduce)

static bool valid_dtype(int32_t d) { return d == ZERO_BF16 || d == ZERO_F32; }

// ------------------------------------------------------------------ pipeline geometry and launch
#ifndef ZERO_PIPE_SMEM_BUDGET
#define ZERO_PIPE_SMEM_BUDGET (200 * 1024)
#endif
#ifndef ZERO_PIPE_STAGE_TARGET
#define ZERO_PIPE_STAGE_TARGET (64 * 1024)
#endif
constexpr int kMaxStages = 16;

struct PipeGeometry {
    int tile, stages;
    size_t smem;
};

// Tile: a multiple of the consumers' pass width (4 elements per consumer
// thread) close to ZERO_PIPE_STAGE_TARGET bytes per stage (N gradient rows +
// master/m/v), halved while two stages would not fit the shared-memory
// budget; then as many stages as fit the budget.
static PipeGeometry pipe_geometry(int n_ranks, int gdtype) {
    const int gb = gdtype == ZERO_BF16 ? 2 : 4;
    const size_t per_elem = static_cast<size_t>(n_ranks) * gb + 12;
    const size_t quantum = 4 * kConsumerWarps * 32;
    size_t mult = ZERO_PIPE_STAGE_TARGET / (quantum * per_elem);
    size_t tile = quantum * (mult > 0 ? mult : 1);
    while (tile > 64 && 2 * tile * per_elem > ZERO_PIPE_SMEM_BUDGET) tile >>= 1;
    const size_t stage_bytes = tile * per_elem;
    int stages = static_cast<int>(ZERO_PIPE_SMEM_BUDGET / stage_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    PipeGeometry g;
    g.tile = static_cast<int>(tile);
    g.stages = stages;
    g.smem = stage_bytes * stages + 2 * sizeof(uint64_t) * stages;
    return g;
}

static int sm_count_current_device(int *out) {
    static int cached[ZERO_MAX_RANKS] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && dev < ZERO_MAX_RANKS && cached[dev] > 0) { *out = cached[dev]; return ZERO_OK; }
    int n = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    if (dev < ZERO_MAX_RANKS) cached[dev] = n;
    *out = n;
    return ZERO_OK;
}

template <int GD, int NR>
static int launch_pipe_one(int64_t nseg, const KParams &kp, const PipeGeometry &g, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_fused_pipe<GD, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(g.smem));
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    int sms = 0;
    const int rc = sm_count_current_device(&sms);
    if (rc != ZERO_OK) return rc;
    const int64_t grid = nseg < sms ? nseg : sms;
    k_fused_pipe<GD, NR><<<static_cast<unsigned>(grid), kPipeThreads, g.smem, st>>>(kp, nseg);
    return launch_status();
}

static int launch_pipe(int gd, int nr, int64_t nseg, KParams &kp, cudaStream_t st) {
    const PipeGeometry g = pipe_geometry(kp.n_ranks, gd);
    kp.tile = g.tile;
    kp.stages = g.stages;
#define ZERO_PIPE_CASE(GDV, NRV) return launch_pipe_one<GDV, NRV>(nseg, kp, g, st)
    if (gd == ZERO_BF16) {
        switch (nr) {
            case 1: ZERO_PIPE_CASE(ZERO_BF16, 1);
            case 2: ZERO_PIPE_CASE(ZERO_BF16, 2);
            case 4: ZERO_PIPE_CASE(ZERO_BF16, 4);
            case 8: ZERO_PIPE_CASE(ZERO_BF16, 8);
            case 16: ZERO_PIPE_CASE(ZERO_BF16, 16);
            default: ZERO_PIPE_CASE(ZERO_BF16, 0);
        }
    }
    switch (nr) {
        case 1: ZERO_PIPE_CASE(ZERO_F32, 1);
        case 2: ZERO_PIPE_CASE(ZERO_F32, 2);
        case 4: ZERO_PIPE_CASE(ZERO_F32, 4);
        case 8: ZERO_PIPE_CASE(ZERO_F32, 8);
        case 16: ZERO_PIPE_CASE(ZERO_F32, 16);
        default: ZERO_PIPE_CASE(ZERO_F32, 0);
    }
#undef ZERO_PIPE_CASE
}

}  // namespace zero

using namespace zero;

// ------------------------------------------------------------------ C ABI
extern "C" int zero_plan_attach(zero_plan *plan, void *workspace, size_t bytes, zero_stream_t stream) {
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
    plan->d_partials = reinterpret_cast<double *>(base + L.partials);
    plan->d_sqnorm = reinterpret_cast<double *>(base + L.scalars);
    plan->d_coef = reinterpret_cast<float *>(base + L.scalars + 8);
    plan->d_err = reinterpret_cast<int *>(base + L.scalars + 16);
    e = cudaMemsetAsync(base + L.scalars, 0, 256, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    plan->device = dev;
    plan->attached = true;
    return ZERO_OK;
}

extern "C" int zero_reduce_scatter(const zero_plan *plan, const void *const *grads, int32_t gdtype,
                                   float *const *gshard, float coef, zero_stream_t stream) {
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
    const int64_t nseg = static_cast<int64_t>(plan->segs.size());
    if (nseg == 0) return ZERO_OK;
    launch_k_reduce(gdtype, n, dim3(static_cast<unsigned>(nseg)), reinterpret_cast<cudaStream_t>(stream), kp);
    return launch_status();
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
    if (nseg > 0) {
        launch_k_reduce(gdtype, plan->n_ranks, dim3(static_cast<unsigned>(nseg)), st, kp);
        const int rc = launch_status();
        if (rc != ZERO_OK) return rc;
    }
    k_finalize<<<1, kFinThreads, 0, st>>>(plan->d_partials, nseg, max_norm, plan->d_sqnorm, sqnorm_out, plan->d_coef);
    return launch_status();
}

extern "C" int zero_grad_sqnorm(const zero_plan *plan, const void *const *grads, int32_t gdtype, double *sqnorm_dev,
                                zero_stream_t stream) {
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
    int rc = check_attached(plan);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_rank_ptrs(plan, reinterpret_cast<const void *const *>(gshard), true)) != ZERO_OK) return rc;
    KParams kp;
    fill_common(plan, kp);
    if ((rc = fill_state(plan, kp, master, m, v, pshard, full, pdtype, hp)) != ZERO_OK) return rc;
    for (int q = 0; q < plan->n_ranks; ++q) kp.gshard[q] = const_cast<float *>(gshard[q]);
    const int64_t nseg = static_cast<int64_t>(plan->segs.size());
    if (nseg == 0) return ZERO_OK;
    k_adamw_shard<<<static_cast<unsigned>(nseg), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(kp);
    return launch_status();
}

extern "C" int zero_all_gather(const zero_plan *plan, const void *const *shard, void *full, int32_t pdtype, int32_t unit,
                               zero_stream_t stream) {
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
    kp.pdtype = pdtype;
    kp.full = full;
    for (int q = 0; q < plan->n_ranks; ++q) kp.pshard[q] = const_cast<void *>(shard[q]);
    if (count == 0) return ZERO_OK;
    k_gather<<<static_cast<unsigned>(count), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(kp);
    return launch_status();
}

extern "C" int zero_all_gather_bf16(const zero_plan *plan, const uint16_t *const *shard16, uint16_t *full, int32_t unit,
                                    zero_stream_t stream) {
    return zero_all_gather(plan, reinterpret_cast<const void *const *>(shard16), full, ZERO_BF16, unit, stream);
}

extern "C" int zero_step(const zero_plan *plan, const void *const *grads, int32_t gdtype, float *const *master,
                         float *const *m, float *const *v, void *full, void *const *pshard, int32_t pdtype,
                         float *const *gshard_ws, const zero_hparams *hp, double *sqnorm_dev, int32_t unit,
                         zero_stream_t stream) {
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
        if (count == 0) return ZERO_OK;
        return launch_pipe(gdtype, n, count, kp, st);
    }
    // clipped: norm pass (writes the averaged gradient shard), device
    // coefficient, then the update from the shard scaled by that coefficient
    if ((rc = launch_norm(plan, grads, gdtype, gshard_ws, hp->max_norm, sqnorm_dev, st)) != ZERO_OK) return rc;
    for (int q = 0; q < n; ++q) kp.gshard[q] = gshard_ws[q];
    kp.use_coef_dev = 1;
    kp.coef_dev = plan->d_coef;
    if (count == 0) return ZERO_OK;
    k_adamw_shard<<<static_cast<unsigned>(count), kThreads, 0, st>>>(kp);
    return launch_status();
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
