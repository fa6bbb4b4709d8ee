// The sm_103a kernels of the sharded optimizer step and their launch
// functions (the interface in zero_launch.h; the C ABI is in zero_abi.cu).
//
// The path is element-wise and HBM-bound (no contraction, so no tensor
// cores): per padded element the fused step reads N gradients plus master/m/v
// and writes master/m/v plus the gathered param.  k_pipe is a persistent,
// warp-specialised kernel: per CTA one producer thread streams segment tiles
// into a shared-memory ring with bulk copies while 12 or 16 consumer warps
// compute from the ring, and segments are handed out dynamically from a ticket
// counter.  k_finalize adds the clip's per-segment partial sums in a fixed
// order; k_gather is the per-unit all-gather.
//
// Exactness: every float operation uses an explicit _rn intrinsic in the
// order the header documents ("ZeRO and FSDP sharding", Code, AdamW::step),
// and the file is compiled with --fmad=false: nothing is contracted.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "zero_launch.h"

namespace zero {

constexpr int kThreads = 256;
constexpr int kSegRing = 8;  // segment numbers the producer may take ahead of its consumers

// Consumer warps of k_pipe for NR gradient rows (0: any count): 16, or 12 for
// 16 rows, where a stage holds a 1536-element tile (two stages fit the shared
// memory budget) and 12 warps take it in exactly one pass of 4 elements per
// thread.  ZERO_PIPE_CONSUMER_WARPS overrides the choice (for measurements).
template <int NR>
__host__ __device__ constexpr int consumer_warps() {
#ifdef ZERO_PIPE_CONSUMER_WARPS
    return ZERO_PIPE_CONSUMER_WARPS;
#else
    return NR >= 16 ? 12 : 16;
#endif
}
static_assert(consumer_warps<16>() <= kPartialSlots && consumer_warps<8>() <= kPartialSlots,
              "one partial slot per consumer warp");

// k_pipe in FUSED and SHARD mode has one more warp, the edge warp: it updates
// each segment's head and tail elements (before the shard position reaches a
// multiple of 8, after the last 8-group) with direct loads while the consumer
// warps stream the body, so the latency of those loads no longer holds up the
// ring.  REDUCE mode keeps them in the consumer warps, whose partial sums of
// squares they belong to.
template <int MODE>
__host__ __device__ constexpr int edge_warps() {
    return MODE == MODE_REDUCE ? 0 : 1;
}
template <int MODE, int NR>
__host__ __device__ constexpr int pipe_threads() {
    return (consumer_warps<NR>() + 1 + edge_warps<MODE>()) * 32;
}

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
    bool gvec;  // gradient positions (relative to the rows' origin) are aligned like the shard positions
    bool fvec;  // full-buffer positions are aligned like the shard positions
};

// g_origin: the full position held by element 0 of each gradient row (0 for
// full-length rows, F_u for unit-local rows).
__device__ __forceinline__ SegSplit split_segment(const Seg &sg, int64_t g_origin) {
    SegSplit s;
    s.k0 = static_cast<int>((8 - (sg.s_off & 7)) & 7);
    if (s.k0 > sg.len) s.k0 = sg.len;
    s.ngroups = (sg.len - s.k0) >> 3;
    s.tail0 = s.k0 + 8 * s.ngroups;
    s.gvec = ((sg.g_off - g_origin + s.k0) & 7) == 0;
    s.fvec = ((sg.g_off + s.k0) & 7) == 0;
    return s;
}

// ------------------------------------------------------------------ the update modes (MODE_* in zero_launch.h)

// Per-thread sum of squares without binary64 arithmetic per element (the
// binary64 rate of this GPU is a small fraction of its binary32 rate): each
// square is split exactly into a binary32 pair (hi = fl(g*g), lo = fma(g, g,
// -hi), an error-free product), the pairs are added with TwoSum into a
// binary32 (hi, lo) accumulator that is renormalised after every add, and
// the warps' accumulators are added across the warp in the same pair
// arithmetic at the end of a segment; the pair goes to binary64 only when the
// partials are added up (k_finalize).  The pair is error-free only while every
// bit of g*g is representable: |g| >= 2^-51 keeps the lowest bit of g*g at or
// above 2^-148 (the error term is never a rounded subnormal), and |g| <= 2^56
// keeps the squares one warp adds in a segment (at most 32 x 86) below 2^125.
// Values outside that range (and inf/NaN) go to a binary64 accumulator
// directly.  Relative error per segment and warp is below ~1e-13.
struct SqAcc {
    float hi, lo;
    double wide;
};

__device__ __forceinline__ void sq_reset(SqAcc &a) {
    a.hi = 0.0f;
    a.lo = 0.0f;
    a.wide = 0.0;
}

// The binary64 path of the rare values, kept out of line: inlined, the compiler
// predicates it and issues its binary64 instructions for every element (the
// binary64 pipe was 44% busy in the norm pass), as a call it runs only when taken.
__device__ __noinline__ double add_square_wide(double acc, float g) {
    const double d = static_cast<double>(g);
    return __dadd_rn(acc, __dmul_rn(d, d));
}

__device__ __forceinline__ void add_square(SqAcc &a, float g) {
    const float mag = fabsf(g);
    if (!(mag <= 0x1p56f) || (mag < 0x1p-51f && mag != 0.0f)) {
        a.wide = add_square_wide(a.wide, g);
        return;
    }
    const float ph = __fmul_rn(g, g);
    const float pl = __fmaf_rn(g, g, -ph);  // exact: g*g - ph
    const float t = __fadd_rn(a.hi, ph);    // TwoSum(a.hi, ph) = t + e exactly
    const float bp = __fsub_rn(t, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(t, bp)), __fsub_rn(ph, bp));
    const float l = __fadd_rn(a.lo, __fadd_rn(e, pl));
    a.hi = __fadd_rn(t, l);                 // FastTwoSum renormalisation
    a.lo = __fsub_rn(l, __fsub_rn(a.hi, t));
}

// (hi, lo) += (bhi, blo) in binary32 pair arithmetic: TwoSum of the high parts,
// the low parts and the error added, then renormalised (FastTwoSum).
__device__ __forceinline__ void pair_add(float &hi, float &lo, float bhi, float blo) {
    const float s = __fadd_rn(hi, bhi);
    const float bp = __fsub_rn(s, hi);
    const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(bhi, bp));
    const float t = __fadd_rn(__fadd_rn(lo, blo), e);
    hi = __fadd_rn(s, t);
    lo = __fsub_rn(t, __fsub_rn(hi, s));
}

// The binary64 parts added across the warp (lane 0 holds the sum), out of line
// for the same reason as add_square_wide.
__device__ __noinline__ double warp_wide(double w) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = __dadd_rn(w, __shfl_down_sync(0xFFFFFFFFu, w, o));
    return w;
}

// A warp's accumulators added across the warp (a fixed shuffle tree; lane 0
// holds the result): the pair in binary32 pair arithmetic, the binary64 part only
// when some lane has one (values outside the pair's range are rare).
__device__ __forceinline__ SqPartial warp_sq(const SqAcc &a) {
    SqPartial r{a.hi, a.lo, a.wide};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ohi = __shfl_down_sync(0xFFFFFFFFu, r.hi, o);
        const float olo = __shfl_down_sync(0xFFFFFFFFu, r.lo, o);
        pair_add(r.hi, r.lo, ohi, olo);
    }
    if (__any_sync(0xFFFFFFFFu, __double_as_longlong(r.wide) != 0)) r.wide = warp_wide(r.wide);
    return r;
}

// Direct (register) path for one segment, spread over nthr threads: the
// 8-wide groups of [k0, tail0) when `body` is set, and always the head and
// tail elements.  `coef` scales the gradient when `scale` is set (REDUCE:
// the host coefficient; SHARD: the device clip coefficient).
template <int MODE, int GD, int NR>
__device__ __forceinline__ void direct_segment(const KParams &p, const Seg &sg, const SegSplit &sp, int tid, int nthr,
                                               bool body, bool edges, bool scale, float coef, SqAcc &sq) {
    const int r = sg.rank;
    float *__restrict__ W = p.master[r] + sg.s_off;
    float *__restrict__ M = p.m[r] + sg.s_off;
    float *__restrict__ V = p.v[r] + sg.s_off;
    float *__restrict__ G = p.gshard[r] != nullptr ? p.gshard[r] + sg.s_off : nullptr;
    void *full = p.full;
    void *ps = p.pshard[r];
    if (body) {
        for (int i = tid; i < sp.ngroups; i += nthr) {
            const int k = sp.k0 + 8 * i;
            if (!ZERO_GUARD(k + 8 <= sg.len && sg.s_off + k + 8 <= p.h_len && sg.g_off + k + 8 <= p.p_pad &&
                                sg.g_off - p.g_origin + k + 8 <= p.g_len && aligned_to(W + k, 16),
                            30))
                continue;
            float g[8];
            if constexpr (MODE == MODE_SHARD) {
                load8(G + k, g);
            } else {
                float acc[8];
                fold8<GD, NR>(p, sg.g_off - p.g_origin + k, sp.gvec, acc);
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = (k + e >= sg.valid) ? 0.0f : average(acc[e], p);
            }
            if (scale) {
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = __fmul_rn(g[e], coef);
            }
            if constexpr (MODE == MODE_REDUCE) {
#pragma unroll
                for (int e = 0; e < 8; ++e) add_square(sq, g[e]);
                if (G != nullptr && p.write_g) store8(G + k, g);
            } else {
                float w[8], m[8], v[8];
                load8(W + k, w);
                load8(M + k, m);
                load8(V + k, v);
#pragma unroll
                for (int e = 0; e < 8; ++e) adamw(g[e], w[e], m[e], v[e], p.c);
                store8(W + k, w);
                store8(M + k, m);
                store8(V + k, v);
                if (full != nullptr) store_param8(full, sg.g_off + k, p.pdtype, sp.fvec, w);
                if (ps != nullptr) store_param8(ps, sg.s_off + k, p.pdtype, true, w);
            }
        }
    }
    const int nedge = edges ? sp.k0 + (sg.len - sp.tail0) : 0;
    for (int t = tid; t < nedge; t += nthr) {
        const int k = t < sp.k0 ? t : sp.tail0 + (t - sp.k0);
        if (!ZERO_GUARD(k >= 0 && k < sg.len && sg.s_off + k < p.h_len && sg.g_off + k < p.p_pad &&
                            sg.g_off - p.g_origin + k < p.g_len,
                        31))
            continue;
        float g;
        if constexpr (MODE == MODE_SHARD) {
            g = G[k];
        } else {
            g = (k >= sg.valid) ? 0.0f : average(fold1<GD, NR>(p, sg.g_off - p.g_origin + k), p);
        }
        if (scale) g = __fmul_rn(g, coef);
        if constexpr (MODE == MODE_REDUCE) {
            add_square(sq, g);
            if (G != nullptr && p.write_g) G[k] = g;
        } else {
            float w = W[k], m = M[k], v = V[k];
            adamw(g, w, m, v, p.c);
            W[k] = w;
            M[k] = m;
            V[k] = v;
            if (full != nullptr) store_param1(full, sg.g_off + k, p.pdtype, w);
            if (ps != nullptr) store_param1(ps, sg.s_off + k, p.pdtype, w);
        }
    }
}

// ------------------------------------------------------------------ bulk-copy pipeline
// Persistent, warp-specialised, dynamically scheduled: each CTA's producer
// thread takes the next segment of the launch table from the plan's ticket
// counter when it is ready for more work, and hands the segment number to its
// consumer warps through a small shared-memory ring.  Segments are handed out
// in table order, so the CTAs always work on neighbouring parts of the
// buffers, and every CTA finishes within about one segment of the others
// however unequal the segments are.
// The producer streams each segment body, tile by tile, into a ring of
// `stages` shared-memory buffers with 1-D bulk copies (cp.async.bulk,
// completion counted in bytes on a per-stage mbarrier).  The consumer warps
// wait for a stage, compute from shared memory, store straight to global
// memory and release the stage; copies stay in flight while they compute.
// Gradient rows whose positions are not 16-byte aligned are copied as the
// aligned superset of the tile and read at an element offset (`shift`), so
// misaligned slices stream like aligned ones.  Heads and tails (before the
// shard position reaches a multiple of 8, after the last 8-group), and the
// rare segment whose superset would pass the last whole 16 bytes of a row,
// take the direct path in the consumer warps.
//
// Every wait is bounded (kWaitLimitNs of %globaltimer): on expiry the waiting
// thread records the failure in *p.err and stops waiting; the producer then
// waits (again bounded) for the copies it already issued before it exits.
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

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst_smem)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Stage layout: gradient rows (room for a shift of up to 7 elements, 16-byte
// rounded), then master, m, v rows of `tile` fp32.  Shared by host and device.
struct StageLayout {
    uint32_t grad_rows, grad_row_bytes, state_off, bytes;
};

__host__ __device__ __forceinline__ StageLayout stage_layout(int mode, int n_ranks, int gbytes, int tile) {
    StageLayout L;
    if (mode == MODE_SHARD) {
        L.grad_rows = 1;
        L.grad_row_bytes = static_cast<uint32_t>(tile) * 4u;
    } else {
        L.grad_rows = static_cast<uint32_t>(n_ranks);
        L.grad_row_bytes = (static_cast<uint32_t>(tile + 8) * static_cast<uint32_t>(gbytes) + 15u) & ~15u;
    }
    L.state_off = L.grad_rows * L.grad_row_bytes;
    L.bytes = L.state_off + (mode == MODE_REDUCE ? 0u : 3u * static_cast<uint32_t>(tile) * 4u);
    return L;
}

// 4 consecutive gradient values from a shared-memory row at element offset
// `off` (a multiple of 4 plus the row's shift).
template <int GD, bool ALIGNED>
__device__ __forceinline__ void smem_load4(const unsigned char *row, int off, float (&x)[4]) {
    if constexpr (GD == ZERO_BF16) {
        const unsigned char *b = row + off * 2;
        uint32_t lo, hi;
        if (ALIGNED || (off & 3) == 0) {
            const uint2 u = *reinterpret_cast<const uint2 *>(b);
            lo = u.x;
            hi = u.y;
        } else if ((off & 1) == 0) {
            lo = *reinterpret_cast<const uint32_t *>(b);
            hi = *reinterpret_cast<const uint32_t *>(b + 4);
        } else {
            const unsigned short *h = reinterpret_cast<const unsigned short *>(b);
            lo = static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
            hi = static_cast<uint32_t>(h[2]) | (static_cast<uint32_t>(h[3]) << 16);
        }
        x[0] = __uint_as_float(lo << 16);
        x[1] = __uint_as_float(lo & 0xFFFF0000u);
        x[2] = __uint_as_float(hi << 16);
        x[3] = __uint_as_float(hi & 0xFFFF0000u);
    } else {
        const float *f = reinterpret_cast<const float *>(row) + off;
        if (ALIGNED || (off & 3) == 0) {
            const float4 u = *reinterpret_cast<const float4 *>(f);
            x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
        } else {
            x[0] = f[0]; x[1] = f[1]; x[2] = f[2]; x[3] = f[3];
        }
    }
}

// 4 params at element position i of a full-length buffer (ALIGNED: i is a
// multiple of 4; otherwise any alignment).
template <bool ALIGNED>
__device__ __forceinline__ void store_param4(void *base, int64_t i, int32_t pdtype, const float (&w)[4]) {
    if (pdtype == ZERO_BF16) {
        unsigned short *d = static_cast<unsigned short *>(base) + i;
        const uint32_t h0 = f32_to_bf16_rne(w[0]), h1 = f32_to_bf16_rne(w[1]);
        const uint32_t h2 = f32_to_bf16_rne(w[2]), h3 = f32_to_bf16_rne(w[3]);
        if (ALIGNED || (i & 3) == 0) {
            __stcs(reinterpret_cast<uint2 *>(d), make_uint2(h0 | (h1 << 16), h2 | (h3 << 16)));
        } else if ((i & 1) == 0) {
            reinterpret_cast<uint32_t *>(d)[0] = h0 | (h1 << 16);
            reinterpret_cast<uint32_t *>(d)[1] = h2 | (h3 << 16);
        } else {
            d[0] = static_cast<unsigned short>(h0);
            d[1] = static_cast<unsigned short>(h1);
            d[2] = static_cast<unsigned short>(h2);
            d[3] = static_cast<unsigned short>(h3);
        }
    } else {
        float *d = static_cast<float *>(base) + i;
        if (ALIGNED || (i & 3) == 0) {
            __stcs(reinterpret_cast<float4 *>(d), make_float4(w[0], w[1], w[2], w[3]));
        } else {
            d[0] = w[0]; d[1] = w[1]; d[2] = w[2]; d[3] = w[3];
        }
    }
}

// Consumer work on one tile in shared memory: elements [k, k + len) of the
// segment, 4 per thread per pass.  ALIGNED: the gradient rows have no shift,
// so every shared-memory read and parameter store is a full vector.
template <int MODE, int GD, int NR, bool ALIGNED>
__device__ __forceinline__ void consume_tile(const KParams &p, const Seg &sg, const unsigned char *buf,
                                             const StageLayout &L, int tile, int k, int len, int shift, int ct,
                                             bool scale, float coef, SqAcc &sq, float *__restrict__ Wg,
                                             float *__restrict__ Mg, float *__restrict__ Vg, float *__restrict__ Gg,
                                             void *full, void *ps, int n) {
    constexpr int CT = consumer_warps<NR>() * 32;
    const float *Ws = reinterpret_cast<const float *>(buf + L.state_off);
    const float *Ms = Ws + tile;
    const float *Vs = Ms + tile;
    for (int e = 4 * ct; e < len; e += 4 * CT) {
        const int kk = k + e;
        if (!ZERO_GUARD(e + 4 <= tile && sg.s_off + kk + 4 <= p.h_len && sg.g_off + kk + 4 <= p.p_pad &&
                            aligned_to(Wg + kk, 16) && (!ALIGNED || ((sg.g_off + kk) & 3) == 0),
                        20))
            continue;
        float g[4];
        if constexpr (MODE == MODE_SHARD) {
            const float4 u = *reinterpret_cast<const float4 *>(buf + e * 4);
            g[0] = u.x; g[1] = u.y; g[2] = u.z; g[3] = u.w;
        } else {
            float acc[4];
            smem_load4<GD, ALIGNED>(buf, shift + e, acc);
#pragma unroll
            for (int q = 1; q < (NR > 0 ? NR : ZERO_MAX_RANKS); ++q) {
                if (NR == 0 && q >= n) break;
                float x[4];
                smem_load4<GD, ALIGNED>(buf + q * L.grad_row_bytes, shift + e, x);
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = __fadd_rn(acc[i], x[i]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) g[i] = (kk + i >= sg.valid) ? 0.0f : average(acc[i], p);
        }
        if (scale) {
#pragma unroll
            for (int i = 0; i < 4; ++i) g[i] = __fmul_rn(g[i], coef);
        }
        if constexpr (MODE == MODE_REDUCE) {
#pragma unroll
            for (int i = 0; i < 4; ++i) add_square(sq, g[i]);
            if (Gg != nullptr && p.write_g)
                __stcs(reinterpret_cast<float4 *>(Gg + kk), make_float4(g[0], g[1], g[2], g[3]));
        } else {
            const float4 w4 = *reinterpret_cast<const float4 *>(Ws + e);
            const float4 m4 = *reinterpret_cast<const float4 *>(Ms + e);
            const float4 v4 = *reinterpret_cast<const float4 *>(Vs + e);
            float w[4] = {w4.x, w4.y, w4.z, w4.w}, m[4] = {m4.x, m4.y, m4.z, m4.w}, v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) adamw(g[i], w[i], m[i], v[i], p.c);
            __stcs(reinterpret_cast<float4 *>(Wg + kk), make_float4(w[0], w[1], w[2], w[3]));
            __stcs(reinterpret_cast<float4 *>(Mg + kk), make_float4(m[0], m[1], m[2], m[3]));
            __stcs(reinterpret_cast<float4 *>(Vg + kk), make_float4(v[0], v[1], v[2], v[3]));
            if (full != nullptr) store_param4<ALIGNED>(full, sg.g_off + kk, p.pdtype, w);
            if (ps != nullptr) store_param4<true>(ps, sg.s_off + kk, p.pdtype, w);
        }
    }
}

// Whether the segment body streams through the pipeline (both the producer
// and the consumers evaluate this identically).
template <int MODE, int GB>
__device__ __forceinline__ bool pipe_eligible(const KParams &p, const Seg &sg, const SegSplit &sp) {
    if (sp.ngroups == 0) return false;
    if (MODE == MODE_SHARD) return true;
    const int64_t end_bytes = ((sg.g_off - p.g_origin + sp.tail0) * GB + 15) & ~static_cast<int64_t>(15);
    const int64_t limit = (p.g_len * GB) & ~static_cast<int64_t>(15);
    return end_bytes <= limit;
}

// A segment descriptor handed through shared memory (volatile: the ring's
// mbarriers order these accesses, the compiler must not move them).
__device__ __forceinline__ void put_seg(Seg *dst, const Seg &sg) {
    volatile int64_t *d = reinterpret_cast<volatile int64_t *>(dst);
    const int64_t *s = reinterpret_cast<const int64_t *>(&sg);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = s[i];
}

__device__ __forceinline__ Seg get_seg(const Seg *src) {
    Seg sg;
    const volatile int64_t *s = reinterpret_cast<const volatile int64_t *>(src);
    int64_t *d = reinterpret_cast<int64_t *>(&sg);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = s[i];
    return sg;
}

template <int MODE, int GD, int NR>
__global__ void __launch_bounds__(pipe_threads<MODE, NR>(), 1) k_pipe(const KParams p, int64_t nseg) {
    constexpr int CW = consumer_warps<NR>();
    constexpr int EW = edge_warps<MODE>();
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int GB = GD == ZERO_BF16 ? 2 : 4;  // bytes per gradient element
    constexpr int SHIFT_MASK = 16 / GB - 1;      // elements per 16 bytes, minus one
    const int n = NR > 0 ? NR : p.n_ranks;
    const int tile = p.tile, stages = p.stages;
    const StageLayout L = stage_layout(MODE, n, GB, tile);
    // clip coefficient of a SHARD update (NaN: the global norm was not finite, skip the step)
    float coef = p.coef;
    bool scale = MODE == MODE_REDUCE && p.coef != 1.0f;
    if (MODE == MODE_SHARD && p.use_coef_dev) {
        coef = *p.coef_dev;
        if (coef != coef) return;
        scale = true;
    }
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(stages) * L.bytes);
    uint64_t *empty_bar = full_bar + stages;
    __shared__ int abort_flag;
    // segment ring: the producer publishes each segment number it took (-1: no more) in
    // seg_ring[slot], its descriptor in seg_data[slot], and arrives on seg_full[slot]; every
    // consumer warp (and the edge warp) arrives on seg_empty[slot] once it has read them
    __shared__ int64_t seg_ring[kSegRing];
    __shared__ Seg seg_data[kSegRing];
    __shared__ __align__(8) uint64_t seg_full[kSegRing], seg_empty[kSegRing];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CW);
        }
        for (int s = 0; s < kSegRing; ++s) {
            mbar_init(&seg_full[s], 1);
            mbar_init(&seg_empty[s], CW + EW);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == CW) {
        // ---------------- producer
        if (lane != 0) return;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;  // per stage: copies issued at least once, parity of the last
        bool ok = true;
        int rs = 0;
        uint32_t rphase = 0;
        // the next ticket is taken as soon as a segment is published, so the atomic's latency
        // overlaps the copies of the segment at hand
        unsigned long long next_ticket = atomicAdd(&p.tickets[0], 1ull);
        for (;;) {
            const unsigned long long t = next_ticket;
            const int64_t si = ok && t < static_cast<unsigned long long>(nseg) ? static_cast<int64_t>(t) : -1;
            Seg sg{};
            if (si >= 0) sg = p.segs[p.seg_base + si];
            if (!mbar_wait(&seg_empty[rs], rphase ^ 1u)) {  // the consumers stopped taking segments
                ok = false;
                break;
            }
            put_seg(&seg_data[rs], sg);
            *reinterpret_cast<volatile int64_t *>(&seg_ring[rs]) = si;
            mbar_arrive(&seg_full[rs]);  // release: the number is visible to the warps that see the phase
            if (++rs == kSegRing) {
                rs = 0;
                rphase ^= 1u;
            }
            if (si < 0) break;
            next_ticket = atomicAdd(&p.tickets[0], 1ull);
            int64_t tile_no = 0;  // position of the tile in its segment
            const SegSplit sp = split_segment(sg, p.g_origin);
            if (!pipe_eligible<MODE, GB>(p, sg, sp)) continue;
            const int r = sg.rank;
            const int shift = MODE == MODE_SHARD ? 0 : static_cast<int>((sg.g_off - p.g_origin + sp.k0) & SHIFT_MASK);
            for (int k = sp.k0; k < sp.tail0; k += tile) {
                const int len = min(tile, sp.tail0 - k);
                if (!mbar_wait(&empty_bar[stage], phase ^ 1u) || *reinterpret_cast<volatile int *>(&abort_flag)) {
                    ok = false;
                    break;
                }
                unsigned char *buf = smem + static_cast<size_t>(stage) * L.bytes;
                const uint32_t gbytes = MODE == MODE_SHARD
                                            ? static_cast<uint32_t>(len) * 4u
                                            : (static_cast<uint32_t>(len + shift) * GB + 15u) & ~15u;
                const uint32_t sbytes = static_cast<uint32_t>(len) * 4u;
                if (!ZERO_GUARD(len > 0 && len <= tile && gbytes <= L.grad_row_bytes && sg.g_off + k + len <= p.p_pad &&
                                    sg.g_off - p.g_origin + k + len <= p.g_len &&
                                    sg.s_off + k + len <= p.h_len && r >= 0 && r < p.n_ranks,
                                10)) {
                    ok = false;
                    break;
                }
                if (si == 0 && tile_no++ == p.drop_tile) {
                    // testing aid: this stage never fills, so its consumers' bounded waits run out
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                mbar_arrive_expect_tx(&full_bar[stage], gbytes * L.grad_rows + (MODE == MODE_REDUCE ? 0u : 3u * sbytes));
                if constexpr (MODE == MODE_SHARD) {
                    bulk_load(buf, p.gshard[r] + sg.s_off + k, gbytes, &full_bar[stage]);
                } else {
                    for (int q = 0; q < n; ++q) {
                        const unsigned char *src =
                            static_cast<const unsigned char *>(p.grads[q]) + (sg.g_off - p.g_origin + k - shift) * GB;
                        if (ZERO_GUARD(aligned_to(src, 16), 11))
                            bulk_load(buf + q * L.grad_row_bytes, src, gbytes, &full_bar[stage]);
                    }
                }
                if constexpr (MODE != MODE_REDUCE) {
                    unsigned char *st = buf + L.state_off;
                    if (ZERO_GUARD(aligned_to(p.master[r] + sg.s_off + k, 16), 12)) {
                        bulk_load(st, p.master[r] + sg.s_off + k, sbytes, &full_bar[stage]);
                        bulk_load(st + tile * 4, p.m[r] + sg.s_off + k, sbytes, &full_bar[stage]);
                        bulk_load(st + 2 * tile * 4, p.v[r] + sg.s_off + k, sbytes, &full_bar[stage]);
                    }
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
        // every producer has taken its last ticket before it counts itself done, so the last
        // one can re-arm the counter for the next launch (which a CUDA graph may replay as is)
        if (atomicAdd(&p.tickets[1], 1ull) == static_cast<unsigned long long>(gridDim.x) - 1ull) {
            atomicExch(&p.tickets[0], 0ull);
            atomicExch(&p.tickets[1], 0ull);
        }
        return;
    }

    if (EW > 0 && warp == CW + 1) {
        // ---------------- edge warp: the heads and tails of the segments, in ring order
        int rs = 0;
        uint32_t rphase = 0;
        SqAcc sq;  // no sums of squares in these modes
        sq_reset(sq);
        for (;;) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&seg_full[rs], rphase))) {  // no segment number in time
                if (lane == 0) atomicExch(p.err, 3);
                abort_flag = 1;
                break;
            }
            const int64_t si = *reinterpret_cast<volatile int64_t *>(&seg_ring[rs]);
            const Seg sg = get_seg(&seg_data[rs]);
            const int slot = rs;
            if (++rs == kSegRing) {
                rs = 0;
                rphase ^= 1u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&seg_empty[slot]);
            if (si < 0) break;
            const SegSplit sp = split_segment(sg, p.g_origin);
            direct_segment<MODE, GD, NR>(p, sg, sp, lane, 32, false, true, scale, coef, sq);
        }
        return;
    }

    // ---------------- consumers: every consumer warp takes every tile, so each
    // stage's mbarrier phases are always waited on in order by the same warps
    // (a stage shared between consumer sets that alternate would let a waiter
    // for phase k pass while the barrier is still in phase k-1: the parity of
    // phase k then reads as already complete).
    const int ct = threadIdx.x;  // 0 .. CW*32 - 1
    constexpr int CT = CW * 32;
    int stage = 0;
    uint32_t phase = 0;
    bool dead = false;  // a stage wait gave up: stop consuming tiles, keep taking part in the rings
    int rs = 0;
    uint32_t rphase = 0;
    for (;;) {
        // wait results are made warp-uniform: the lanes of a warp must take the same path
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&seg_full[rs], rphase))) {  // no segment number in time: give up
            if (lane == 0) atomicExch(p.err, 3);
            abort_flag = 1;
            break;
        }
        const int64_t si = *reinterpret_cast<volatile int64_t *>(&seg_ring[rs]);
        const Seg sg = get_seg(&seg_data[rs]);
        const int slot = rs;
        if (++rs == kSegRing) {
            rs = 0;
            rphase ^= 1u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&seg_empty[slot]);
        if (si < 0) break;
        const SegSplit sp = split_segment(sg, p.g_origin);
        const bool piped = pipe_eligible<MODE, GB>(p, sg, sp);
        SqAcc sq;
        sq_reset(sq);
        if (!piped || EW == 0) direct_segment<MODE, GD, NR>(p, sg, sp, ct, CT, !piped, EW == 0, scale, coef, sq);
        if (piped && !dead) {
            const int r = sg.rank;
            const int shift = MODE == MODE_SHARD ? 0 : static_cast<int>((sg.g_off - p.g_origin + sp.k0) & SHIFT_MASK);
            float *__restrict__ Wg = p.master[r] + sg.s_off;
            float *__restrict__ Mg = p.m[r] + sg.s_off;
            float *__restrict__ Vg = p.v[r] + sg.s_off;
            float *__restrict__ Gg = p.gshard[r] != nullptr ? p.gshard[r] + sg.s_off : nullptr;
            void *full = p.full;
            void *ps = p.pshard[r];
            for (int k = sp.k0; k < sp.tail0 && !dead; k += tile) {
                const int len = min(tile, sp.tail0 - k);
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full_bar[stage], phase) &&
                                                 !*reinterpret_cast<volatile int *>(&abort_flag))) {
                    if (lane == 0) atomicExch(p.err, 2);
                    abort_flag = 1;
                    dead = true;
                    break;
                }
                const unsigned char *buf = smem + static_cast<size_t>(stage) * L.bytes;
                // vector path: no gradient-row shift and 4-aligned full positions (the latter is
                // not implied in SHARD mode, which has no gradient rows)
                if (shift == 0 && ((sg.g_off + sp.k0) & 3) == 0)
                    consume_tile<MODE, GD, NR, true>(p, sg, buf, L, tile, k, len, 0, ct, scale, coef, sq, Wg, Mg, Vg, Gg,
                                                     full, ps, n);
                else
                    consume_tile<MODE, GD, NR, false>(p, sg, buf, L, tile, k, len, shift, ct, scale, coef, sq, Wg, Mg,
                                                      Vg, Gg, full, ps, n);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[stage]);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if constexpr (MODE == MODE_REDUCE) {
            if (p.want_partials) {
                // this warp's share of the segment's sum of squares, in the warp's own slot: no
                // warp waits for another; the slots past the consumer warps are written as 0
                const SqPartial x = warp_sq(sq);
                if (lane == 0) {
                    SqPartial *dst = p.partials + (p.seg_base + si) * kPartialSlots;
                    dst[warp] = x;
                    if (warp < kPartialSlots - CW) dst[CW + warp] = SqPartial{0.0f, 0.0f, 0.0};
                }
            }
        }
    }
}

// ------------------------------------------------------------------ fixed-order total of the sum of squares
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

// The fixed-order total of the segments' partials (kPartialSlots each, each
// widened to binary64 as (hi + lo) + wide), in one
// launch of kFinBlocks-or-fewer CTAs.  CTA b adds the contiguous block b of the
// partials (thread t takes partials t, t + kFinThreads, ... of the block in
// sequence, then a fixed tree) and stores its sum; the CTA that finishes last
// (a counter, no waiting) adds the block sums in block order with the same
// tree, writes S and, when max_norm > 0, the clip coefficient
// min(1, max_norm / (sqrt(S) + 1e-6)) rounded once to binary32 (NaN when S is
// not finite: the update then skips), and resets the counter for the next
// launch.  The blocks depend only on the number of partials, so S is the same
// bits on every run and every GPU.
constexpr int kFinThreads = 512;
__global__ void __launch_bounds__(kFinThreads) k_finalize(const SqPartial *partials, int64_t n, int64_t block,
                                                          float max_norm, double *block_sums, unsigned *done,
                                                          double *sqnorm_ws, double *sqnorm_out, float *coef_out,
                                                          int *skipped) {
    __shared__ double smem[kFinThreads / 32];
    __shared__ bool last;
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * block;
    const int64_t b1 = b0 + block < n ? b0 + block : n;
    double s = 0.0;
    for (int64_t i = b0 + threadIdx.x; i < b1; i += kFinThreads) {
        const SqPartial q = partials[i];
        s = __dadd_rn(s, __dadd_rn(__dadd_rn(static_cast<double>(q.hi), static_cast<double>(q.lo)), q.wide));
    }
    s = block_sum(s, smem);
    if (threadIdx.x == 0) {
        block_sums[blockIdx.x] = s;
        __threadfence();  // the sum is visible before the count says so
        last = atomicAdd(done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const double x = threadIdx.x < gridDim.x ? *reinterpret_cast<volatile double *>(&block_sums[threadIdx.x]) : 0.0;
    __syncthreads();  // smem is reused by the second tree
    const double S = block_sum(x, smem);
    if (threadIdx.x == 0) {
        *done = 0u;
        *sqnorm_ws = S;
        if (sqnorm_out != nullptr) *sqnorm_out = S;
        if (max_norm > 0.0f) {
            float coef;
            if (!isfinite(S)) {
                coef = __int_as_float(0x7FC00000);
                *skipped = 1;
            } else {
                double c = __ddiv_rn(static_cast<double>(max_norm), __dadd_rn(__dsqrt_rn(S), 1e-6));
                if (c > 1.0) c = 1.0;
                coef = __double2float_rn(c);
            }
            *coef_out = coef;
        }
    }
}

// ------------------------------------------------------------------ all-gather
// full[F_u + r h_u + j] = shard[r][Hoff_u + j]: a copy per segment in 16-byte
// vectors, whether or not the full position is aligned like the shard one.
// Bytes [sb, sb + 16) of the 32-byte concatenation a:b (sb even, 0..14).
__device__ __forceinline__ uint4 shift_pair(const uint4 &a, const uint4 &b, int sb) {
    const uint32_t r = static_cast<uint32_t>(sb & 3) * 8u;  // 0 or 16 bits
    uint32_t w0, w1, w2, w3, w4;
    switch (sb >> 2) {
        case 0: w0 = a.x; w1 = a.y; w2 = a.z; w3 = a.w; w4 = b.x; break;
        case 1: w0 = a.y; w1 = a.z; w2 = a.w; w3 = b.x; w4 = b.y; break;
        case 2: w0 = a.z; w1 = a.w; w2 = b.x; w3 = b.y; w4 = b.z; break;
        default: w0 = a.w; w1 = b.x; w2 = b.y; w3 = b.z; w4 = b.w; break;
    }
    return make_uint4(__funnelshift_r(w0, w1, r), __funnelshift_r(w1, w2, r), __funnelshift_r(w2, w3, r),
                      __funnelshift_r(w3, w4, r));
}

__global__ void __launch_bounds__(kThreads) k_gather(const KParams p) {
    const Seg sg = p.segs[p.seg_base + blockIdx.x];
    const SegSplit sp = split_segment(sg, p.g_origin);
    const int esz = p.pdtype == ZERO_BF16 ? 2 : 4;
    const char *src = static_cast<const char *>(p.pshard[sg.rank]) + sg.s_off * esz;
    // destination element 0 is full position g_origin (0, or F_u for a unit-sized destination);
    // sp.gvec is the alignment relative to that origin
    char *dst = static_cast<char *>(p.full) + (sg.g_off - p.g_origin) * esz;
    int head, tail0;  // elements [0, head) and [tail0, len) are copied one by one below
    if (sp.gvec) {
        // aligned like the shard: whole 16-byte vectors, four in flight per thread
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src + sp.k0 * esz);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst + sp.k0 * esz);
        const int nv = sp.ngroups * (esz / 2);  // a group is 8 elements: 1 vector (bf16) or 2 (fp32)
        int v = threadIdx.x;
        for (; v + 3 * kThreads < nv; v += 4 * kThreads) {
            const uint4 x0 = __ldcs(s4 + v), x1 = __ldcs(s4 + v + kThreads);
            const uint4 x2 = __ldcs(s4 + v + 2 * kThreads), x3 = __ldcs(s4 + v + 3 * kThreads);
            __stcs(d4 + v, x0);
            __stcs(d4 + v + kThreads, x1);
            __stcs(d4 + v + 2 * kThreads, x2);
            __stcs(d4 + v + 3 * kThreads, x3);
        }
        for (; v < nv; v += kThreads) __stcs(d4 + v, __ldcs(s4 + v));
        head = sp.k0;
        tail0 = sp.tail0;
    } else {
        // the destination is aligned differently from the shard: every aligned 16-byte
        // destination vector is assembled from the two aligned source vectors it overlaps
        // (both hold bytes of the segment, so no read leaves the aligned blocks it covers)
        const int lenb = sg.len * esz;
        const int e0b = static_cast<int>((16u - (reinterpret_cast<uintptr_t>(dst) & 15u)) & 15u);
        const int nv = lenb > e0b ? (lenb - e0b) >> 4 : 0;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(src) + static_cast<uintptr_t>(e0b);
        const int sb = static_cast<int>(sa & 15u);
        const uint4 *s4 = reinterpret_cast<const uint4 *>(sa - static_cast<uintptr_t>(sb));
        uint4 *d4 = reinterpret_cast<uint4 *>(dst + e0b);
        int v = threadIdx.x;
        for (; v + kThreads < nv; v += 2 * kThreads) {
            const uint4 a0 = __ldcs(s4 + v), b0 = sb ? __ldcs(s4 + v + 1) : a0;
            const uint4 a1 = __ldcs(s4 + v + kThreads), b1 = sb ? __ldcs(s4 + v + kThreads + 1) : a1;
            __stcs(d4 + v, shift_pair(a0, b0, sb));
            __stcs(d4 + v + kThreads, shift_pair(a1, b1, sb));
        }
        for (; v < nv; v += kThreads) {
            const uint4 a = __ldcs(s4 + v), b = sb ? __ldcs(s4 + v + 1) : a;
            __stcs(d4 + v, shift_pair(a, b, sb));
        }
        head = nv > 0 ? e0b / esz : sg.len;
        tail0 = nv > 0 ? (e0b + 16 * nv) / esz : sg.len;
    }
    const int nedge = head + (sg.len - tail0);
    for (int t = threadIdx.x; t < nedge; t += kThreads) {
        const int k = t < head ? t : tail0 + (t - head);
        if (esz == 2) reinterpret_cast<unsigned short *>(dst)[k] = reinterpret_cast<const unsigned short *>(src)[k];
        else reinterpret_cast<float *>(dst)[k] = reinterpret_cast<const float *>(src)[k];
    }
}

// ------------------------------------------------------------------ launch status
int launch_status() {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    return ZERO_OK;
}

// ------------------------------------------------------------------ pipeline geometry and launch
#ifndef ZERO_PIPE_SMEM_BUDGET
#define ZERO_PIPE_SMEM_BUDGET (200 * 1024)
#endif
#ifndef ZERO_PIPE_MIN_STAGES
#define ZERO_PIPE_MIN_STAGES 2
#endif
#ifndef ZERO_PIPE_TILE_STEP
#define ZERO_PIPE_TILE_STEP 0  // 0: halve the tile while the stages do not fit; else shrink it by this many elements
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
// thread) close to ZERO_PIPE_STAGE_TARGET bytes per stage, reduced while
// ZERO_PIPE_MIN_STAGES stages would not fit the shared-memory budget; then as
// many stages as fit.  (A tile below the pass width leaves some consumer
// threads without work in a pass; the loop allows any multiple of 8.)
static PipeGeometry pipe_geometry(int mode, int n_ranks, int gdtype, int cw) {
    const int gb = gdtype == ZERO_BF16 ? 2 : 4;
    const size_t per_elem = mode == MODE_SHARD ? 16 : static_cast<size_t>(n_ranks) * gb + (mode == MODE_FUSED ? 12 : 0);
    const size_t quantum = 4 * static_cast<size_t>(cw) * 32;
    const size_t mult = ZERO_PIPE_STAGE_TARGET / (quantum * per_elem);
    int tile = static_cast<int>(quantum * (mult > 0 ? mult : 1));
    while (tile > 64 && static_cast<size_t>(ZERO_PIPE_MIN_STAGES) * stage_layout(mode, n_ranks, gb, tile).bytes >
                            ZERO_PIPE_SMEM_BUDGET)
        tile = (ZERO_PIPE_TILE_STEP > 0 && tile > 2 * ZERO_PIPE_TILE_STEP) ? tile - ZERO_PIPE_TILE_STEP : tile >> 1;
    const size_t stage_bytes = stage_layout(mode, n_ranks, gb, tile).bytes;
    int stages = static_cast<int>(ZERO_PIPE_SMEM_BUDGET / stage_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    PipeGeometry g;
    g.tile = tile;
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

template <int MODE, int GD, int NR>
static int launch_pipe_one(int64_t nseg, KParams &kp, cudaStream_t st) {
    constexpr int CW = consumer_warps<NR>();
    const PipeGeometry g = pipe_geometry(MODE, kp.n_ranks, GD, CW);
    kp.tile = g.tile;
    kp.stages = g.stages;
    cudaError_t e = cudaFuncSetAttribute(k_pipe<MODE, GD, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(g.smem));
    if (e != cudaSuccess) { set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    int sms = 0;
    const int rc = sm_count_current_device(&sms);
    if (rc != ZERO_OK) return rc;
    const int64_t grid = nseg < sms ? nseg : sms;
    k_pipe<MODE, GD, NR><<<static_cast<unsigned>(grid), pipe_threads<MODE, NR>(), g.smem, st>>>(kp, nseg);
    return launch_status();
}

template <int MODE>
static int launch_pipe_mode(int gd, int nr, int64_t nseg, KParams &kp, cudaStream_t st) {
    if (gd == ZERO_BF16) {
        switch (nr) {
            case 1: return launch_pipe_one<MODE, ZERO_BF16, 1>(nseg, kp, st);
            case 2: return launch_pipe_one<MODE, ZERO_BF16, 2>(nseg, kp, st);
            case 4: return launch_pipe_one<MODE, ZERO_BF16, 4>(nseg, kp, st);
            case 8: return launch_pipe_one<MODE, ZERO_BF16, 8>(nseg, kp, st);
            case 16: return launch_pipe_one<MODE, ZERO_BF16, 16>(nseg, kp, st);
            default: return launch_pipe_one<MODE, ZERO_BF16, 0>(nseg, kp, st);
        }
    }
    switch (nr) {
        case 1: return launch_pipe_one<MODE, ZERO_F32, 1>(nseg, kp, st);
        case 2: return launch_pipe_one<MODE, ZERO_F32, 2>(nseg, kp, st);
        case 4: return launch_pipe_one<MODE, ZERO_F32, 4>(nseg, kp, st);
        case 8: return launch_pipe_one<MODE, ZERO_F32, 8>(nseg, kp, st);
        case 16: return launch_pipe_one<MODE, ZERO_F32, 16>(nseg, kp, st);
        default: return launch_pipe_one<MODE, ZERO_F32, 0>(nseg, kp, st);
    }
}

static std::atomic<int64_t> g_drop_tile{-1};

// One launch of the pipeline in `mode` over segments [kp.seg_base, kp.seg_base + nseg).
int launch_pipe(int mode, int gd, int64_t nseg, KParams &kp, cudaStream_t st) {
    if (nseg <= 0) return ZERO_OK;
    kp.drop_tile = g_drop_tile.exchange(-1);
    switch (mode) {
        case MODE_FUSED: return launch_pipe_mode<MODE_FUSED>(gd, kp.n_ranks, nseg, kp, st);
        case MODE_REDUCE: return launch_pipe_mode<MODE_REDUCE>(gd, kp.n_ranks, nseg, kp, st);
        default: return launch_pipe_one<MODE_SHARD, ZERO_F32, 1>(nseg, kp, st);  // no gradient rows: one instance
    }
}

void arm_drop_tile(int64_t tile) { g_drop_tile.store(tile); }

int launch_finalize(const zero_plan *plan, float max_norm, double *sqnorm_out, cudaStream_t st) {
    const int64_t n = static_cast<int64_t>(plan->segs.size()) * kPartialSlots;
    // blocks of a whole number of passes, at most kFinBlocks of them (at least one, for S = 0)
    int64_t block = (n + kFinBlocks - 1) / kFinBlocks;
    block = block > 0 ? (block + kFinThreads - 1) / kFinThreads * kFinThreads : kFinThreads;
    const int64_t blocks = n > 0 ? (n + block - 1) / block : 1;
    k_finalize<<<static_cast<unsigned>(blocks), kFinThreads, 0, st>>>(
        plan->d_partials, n, block, max_norm, plan->d_fin_sums, plan->d_fin_count, plan->d_sqnorm, sqnorm_out,
        plan->d_coef, plan->d_skipped);
    return launch_status();
}

int launch_gather(int64_t count, const KParams &kp, cudaStream_t st) {
    if (count <= 0) return ZERO_OK;
    k_gather<<<static_cast<unsigned>(count), kThreads, 0, st>>>(kp);
    return launch_status();
}

}  // namespace zero
