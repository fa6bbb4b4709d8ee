/*
 * zero_oracle.c -- CPU oracle for the ZeRO-1/2/3 sharded optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file states, in plain single-threaded C,
 * what the sharded update computes.  It is loaded only by the test suite, by
 * the package's smoke check and by the benchmark's CPU-baseline leg.  It
 * shares no code, header, table or constant with the CUDA library, and the
 * product never loads it.
 *
 * Arithmetic contract: every floating-point expression below is a sequence of
 * single IEEE-754 binary32 operations, round to nearest even.  The file must
 * be compiled with -ffp-contract=off and without -ffast-math (oracle/build.py
 * does this), so that no multiply-add is fused.
 *
 * Sources (page title, section):
 *   [P1] "ZeRO and FSDP sharding" -- How it works; Code (the ZeRO-2-on-threads
 *        toy: Comm::reduce_scatter, Comm::all_gather, AdamW::step, the
 *        unsharded check); Implementation notes; Pitfalls.
 *   [P3] "ZeRO: Three Ledgers, Zero Redundancy" -- section 1 (the update is
 *        element-wise), section 2 (all-reduce = reduce-scatter + local update
 *        + all-gather; the norm is a decomposable sum of squares).
 *   [P4] "Learn: ZeRO & FSDP" -- section 3 (fp32 master weights, bf16 working
 *        copy), section 5 (FlatParameter: flatten, concatenate, chunk).
 *
 * Pins (what each function is checked against, besides itself) are listed in
 * tests/test_oracle_pins.py; every function here has at least one.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENONFINITE (-5)

typedef struct {
    float lr, b1, b2, eps, wd;
    int32_t t;        /* 1-based step number */
    float max_norm;   /* <= 0: no clipping */
} orc_hparams;

/* ------------------------------------------------------------------------ */
/* Layout.  [P1] How it works: flatten each unit's parameters into one buffer
 * padded to a multiple of N; rank r owns slice r.  [P1] Pitfalls: the flat
 * numel must be divisible by N.  [P4] section 5: FlatParameter flattens,
 * concatenates and chunks a unit's tensors.
 *
 * For unit u of s_u parameters:  S_u = s_u rounded up to a multiple of N,
 * h_u = S_u / N (slice length), F_u = sum_{k<u} S_k (offset of the unit in the
 * full flat buffer), Hoff_u = sum_{k<u} h_k (offset of the unit's slice inside
 * every rank's shard buffer).  totals[0] = P_pad = sum S_u, totals[1] = H =
 * P_pad / N.  Rank r owns full positions [F_u + r h_u, F_u + (r+1) h_u).
 *
 * Every layout function takes `align` (>= 1): the padding quantum is N*align
 * instead of N, so every slice length h_u is a multiple of align.  The pages
 * fix no alignment; align = 1 is their layout, larger values are an option
 * (slices that start on whole vectors). */
static int64_t orc_pad_to(int64_t s, int64_t quantum)
{
    int64_t rem = s % quantum;
    return rem == 0 ? s : s + (quantum - rem);
}

int orc_plan(const int64_t *sizes, int32_t n_units, int32_t n_ranks, int32_t align,
             int64_t *S, int64_t *h, int64_t *F, int64_t *Hoff, int64_t *totals)
{
    if (n_units < 0 || n_ranks < 1 || align < 1) return ORC_EINVAL;
    int64_t f = 0, hh = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        if (sizes[u] < 0) return ORC_EINVAL;
        int64_t padded = orc_pad_to(sizes[u], (int64_t)n_ranks * align);
        S[u] = padded;
        h[u] = padded / n_ranks;
        F[u] = f;
        Hoff[u] = hh;
        f += padded;
        hh += padded / n_ranks;
    }
    totals[0] = f;
    totals[1] = hh;
    return ORC_OK;
}

/* map[r*H + p] = full-buffer position held at position p of rank r's shard
 * buffer (the shard buffer concatenates the rank's slices in unit order). */
int orc_shard_map(const int64_t *sizes, int32_t n_units, int32_t n_ranks, int32_t align, int64_t *map)
{
    if (n_units < 0 || n_ranks < 1 || align < 1) return ORC_EINVAL;
    const int64_t q = (int64_t)n_ranks * align;
    int64_t H = 0;
    for (int32_t u = 0; u < n_units; ++u) H += orc_pad_to(sizes[u], q) / n_ranks;
    int64_t f = 0, hh = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        int64_t Su = orc_pad_to(sizes[u], q);
        int64_t hu = Su / n_ranks;
        for (int32_t r = 0; r < n_ranks; ++r)
            for (int64_t j = 0; j < hu; ++j)
                map[(int64_t)r * H + hh + j] = f + (int64_t)r * hu + j;
        f += Su;
        hh += hu;
    }
    return ORC_OK;
}

/* Reshard (checkpoint resharding: "ZeRO and FSDP sharding", Implementation
 * notes).  dst (n_to rank buffers) receives, for every target rank r and
 * position j of unit u's slice, the unit position k = r*h'_u + j taken from
 * the rank that owns k in the source layout; target padding is 0.  Elements
 * are esize raw bytes. */
int orc_reshard(const int64_t *sizes, int32_t n_units, int32_t n_from, int32_t align_from, int32_t n_to,
                int32_t align_to, int32_t esize, const void *const *src, void *const *dst)
{
    if (n_units < 0 || n_from < 1 || n_to < 1 || align_from < 1 || align_to < 1 || (esize != 2 && esize != 4))
        return ORC_EINVAL;
    int64_t hh_from = 0, hh_to = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        int64_t s = sizes[u];
        int64_t S_from = orc_pad_to(s, (int64_t)n_from * align_from);
        int64_t S_to = orc_pad_to(s, (int64_t)n_to * align_to);
        int64_t h_from = S_from / n_from, h_to = S_to / n_to;
        for (int32_t r = 0; r < n_to; ++r)
            for (int64_t j = 0; j < h_to; ++j) {
                int64_t k = (int64_t)r * h_to + j;
                unsigned char *d = (unsigned char *)dst[r] + (hh_to + j) * esize;
                if (k < s) {
                    int64_t rs = k / h_from, js = k % h_from;
                    memcpy(d, (const unsigned char *)src[rs] + (hh_from + js) * esize, (size_t)esize);
                } else {
                    memset(d, 0, (size_t)esize);
                }
            }
        hh_from += h_from;
        hh_to += h_to;
    }
    return ORC_OK;
}

/* pad[i] = 1 where full position i is padding (position >= s_u inside unit u). */
int orc_pad_mask(const int64_t *sizes, int32_t n_units, int32_t n_ranks, int32_t align, uint8_t *pad)
{
    if (n_units < 0 || n_ranks < 1 || align < 1) return ORC_EINVAL;
    int64_t f = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        int64_t Su = orc_pad_to(sizes[u], (int64_t)n_ranks * align);
        for (int64_t k = 0; k < Su; ++k) pad[f + k] = (uint8_t)(k >= sizes[u]);
        f += Su;
    }
    return ORC_OK;
}

/* For n full-buffer positions: the owning rank, the position inside that
 * rank's shard buffer, and whether the position is padding.  (Searches the
 * units in order; the same layout as orc_plan.) */
int orc_locate(const int64_t *sizes, int32_t n_units, int32_t n_ranks, int32_t align, int64_t n, const int64_t *pos,
               int32_t *rank, int64_t *shard_pos, uint8_t *is_pad)
{
    if (n_units < 0 || n_ranks < 1 || align < 1 || n < 0) return ORC_EINVAL;
    /* the layout of every unit once: F (full offset), S (padded size), h (slice), Hoff */
    int64_t *t = (int64_t *)malloc(sizeof(int64_t) * 4 * (size_t)(n_units > 0 ? n_units : 1));
    if (t == NULL) return ORC_EINVAL;
    int64_t f = 0, hh = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        int64_t Su = orc_pad_to(sizes[u], (int64_t)n_ranks * align);
        t[4 * u] = f;
        t[4 * u + 1] = Su;
        t[4 * u + 2] = Su / n_ranks;
        t[4 * u + 3] = hh;
        f += Su;
        hh += Su / n_ranks;
    }
    int rc = ORC_OK;
    for (int64_t i = 0; i < n && rc == ORC_OK; ++i) {
        /* the last unit whose offset F is <= pos (a unit of size 0 owns no position) */
        int32_t lo = 0, hi = n_units - 1, u = -1;
        while (lo <= hi) {
            int32_t mid = lo + (hi - lo) / 2;
            if (t[4 * mid] <= pos[i]) { u = mid; lo = mid + 1; } else { hi = mid - 1; }
        }
        while (u >= 0 && t[4 * u + 1] == 0) --u;
        if (u < 0 || pos[i] < t[4 * u] || pos[i] >= t[4 * u] + t[4 * u + 1]) { rc = ORC_EINVAL; break; }
        int64_t k = pos[i] - t[4 * u];
        rank[i] = (int32_t)(k / t[4 * u + 2]);
        shard_pos[i] = t[4 * u + 3] + k % t[4 * u + 2];
        is_pad[i] = (uint8_t)(k >= sizes[u]);
    }
    free(t);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* bfloat16.  [P1] How it works: "cast to bf16 shard"; [P4] section 3: the
 * bf16 working copy is a rounded view of the fp32 master.  Reading: round to
 * nearest, ties to even, on the 16 low bits that are dropped.  A NaN stays a
 * NaN: its quiet bit is set and its sign kept. */
uint16_t orc_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xFFFFu;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)(hi | 0x0040u);
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u; /* may carry into the exponent: correct, overflow gives inf */
    return (uint16_t)hi;
}

void orc_bf16_rne_array(int64_t n, const float *x, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(x[i]);
}

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

/* ------------------------------------------------------------------------ */
/* Bias corrections.  [P1] Code, AdamW::step: bc1 = 1 - b1^t,
 * bc2 = sqrt(1 - b2^t), with t incremented before use (t is 1-based here).
 * Reading: b^t is binary exponentiation in binary32 (square and multiply over
 * the bits of t, low bit first), the usual integer-power routine. */
static float orc_powi(float b, int32_t t)
{
    float r = 1.0f;
    float a = b;
    uint32_t e = (uint32_t)t;
    while (e != 0u) {
        if (e & 1u) r = r * a;
        e >>= 1;
        if (e != 0u) a = a * a;
    }
    return r;
}

int orc_bias_corrections(int32_t t, float b1, float b2, float *bc1, float *bc2)
{
    if (t < 1) return ORC_EINVAL;
    *bc1 = 1.0f - orc_powi(b1, t);
    *bc2 = sqrtf(1.0f - orc_powi(b2, t));
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Reduce-scatter + average for one full-buffer position i.
 * [P1] Code, Comm::reduce_scatter: sum over ranks (rank order), rank r keeps
 * slice r; then every element is divided by n.  [P1] unsharded check: the
 * same sum over ranks then / n.  The fold starts from rank 0's value (the
 * same as starting from -0.0).  Padding positions contribute 0. */
static float orc_load_grad(const void *g, int32_t dtype, int64_t i)
{
    if (dtype == ORC_F32) return ((const float *)g)[i];
    return orc_bf16_to_f32(((const uint16_t *)g)[i]);
}

static float orc_avg_grad(int32_t n_ranks, const void *const *grads, int32_t gdtype,
                          const uint8_t *pad, int64_t i)
{
    if (pad != NULL && pad[i]) return 0.0f;
    float acc = orc_load_grad(grads[0], gdtype, i);
    for (int32_t q = 1; q < n_ranks; ++q) acc = acc + orc_load_grad(grads[q], gdtype, i);
    return acc / (float)n_ranks;
}

/* The averaged gradient itself at n positions (the reduce-scatter's output). */
int orc_avg_grad_array(int64_t n, int32_t n_ranks, const void *const *grads, int32_t gdtype,
                       const uint8_t *pad, float *out)
{
    if (n < 0 || n_ranks < 1 || (gdtype != ORC_F32 && gdtype != ORC_BF16)) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) out[i] = orc_avg_grad(n_ranks, grads, gdtype, pad, i);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Global gradient norm.  [P1] Implementation notes: clipping needs the global
 * norm, the squared norms of the local shards summed and then all-reduced.
 * [P3] section 2: a norm is a sum of squares, a decomposable reduction.
 * Reading: the norm is that of the averaged gradient; S = sum of g_i^2 is
 * computed EXACTLY (every fp32 square is an integer times a power of two, kept
 * in a 768-bit fixed-point accumulator) and rounded once to binary64, so S
 * does not depend on any summation order. */
#define ORC_ACC_LIMBS 12
typedef struct {
    uint64_t limb[ORC_ACC_LIMBS]; /* value = sum limb[k] 2^(64k) * 2^-298 */
    uint32_t nan_seen;
    uint32_t inf_seen;
} orc_sqacc;

int32_t orc_sqacc_bytes(void) { return (int32_t)sizeof(orc_sqacc); }

void orc_sqacc_add_square(orc_sqacc *a, float g)
{
    uint32_t u;
    memcpy(&u, &g, sizeof u);
    uint32_t e = (u >> 23) & 0xFFu;
    uint32_t f = u & 0x7FFFFFu;
    if (e == 0xFFu) {
        if (f != 0u) a->nan_seen = 1u; else a->inf_seen = 1u;
        return;
    }
    uint64_t M;
    int32_t E; /* |g| = M * 2^E exactly */
    if (e == 0u) { M = f; E = -149; } else { M = (uint64_t)(f | 0x800000u); E = (int32_t)e - 150; }
    if (M == 0u) return;
    uint64_t sq = M * M;              /* < 2^48: exact */
    int32_t s = 2 * E + 298;          /* g^2 = sq * 2^(s - 298), s in [0, 506] */
    int32_t k = s / 64, off = s % 64;
    unsigned __int128 x = (unsigned __int128)sq << off; /* < 2^111 */
    uint64_t lo = (uint64_t)x, hi = (uint64_t)(x >> 64);
    uint64_t old = a->limb[k];
    a->limb[k] = old + lo;
    uint64_t carry = a->limb[k] < old ? 1u : 0u;
    int32_t j = k + 1;
    unsigned __int128 t = (unsigned __int128)a->limb[j] + hi + carry;
    a->limb[j] = (uint64_t)t;
    carry = (uint64_t)(t >> 64);
    while (carry != 0u && ++j < ORC_ACC_LIMBS) {
        a->limb[j] += 1u;
        carry = a->limb[j] == 0u ? 1u : 0u;
    }
}

/* dst += src, exactly (limb-wise addition with carry), so that partial sums of
 * squares taken over disjoint sets of positions combine into the same exact
 * value as one pass over all of them. */
void orc_sqacc_merge(orc_sqacc *dst, const orc_sqacc *src)
{
    uint64_t carry = 0u;
    for (int k = 0; k < ORC_ACC_LIMBS; ++k) {
        unsigned __int128 t = (unsigned __int128)dst->limb[k] + src->limb[k] + carry;
        dst->limb[k] = (uint64_t)t;
        carry = (uint64_t)(t >> 64);
    }
    dst->nan_seen |= src->nan_seen;
    dst->inf_seen |= src->inf_seen;
}

static int orc_bitlen128(unsigned __int128 x)
{
    int n = 0;
    while (x != 0) { x >>= 1; ++n; }
    return n;
}

double orc_sqacc_result(const orc_sqacc *a)
{
    if (a->nan_seen) return NAN;
    if (a->inf_seen) return INFINITY;
    int top = -1;
    for (int k = ORC_ACC_LIMBS - 1; k >= 0; --k)
        if (a->limb[k] != 0u) { top = k; break; }
    if (top < 0) return 0.0;
    /* window = the two highest limbs; sticky = any bit below them */
    int base = top >= 1 ? top - 1 : 0;
    unsigned __int128 w = top >= 1 ? (((unsigned __int128)a->limb[top] << 64) | a->limb[top - 1])
                                   : (unsigned __int128)a->limb[0];
    int sticky = 0;
    for (int k = 0; k < base; ++k) if (a->limb[k] != 0u) sticky = 1;
    int L = orc_bitlen128(w);
    int shift = L > 53 ? L - 53 : 0;
    unsigned __int128 q = w >> shift;
    if (shift > 0) {
        unsigned __int128 rem = w & ((((unsigned __int128)1) << shift) - 1);
        unsigned __int128 half = ((unsigned __int128)1) << (shift - 1);
        if (rem > half || (rem == half && (sticky || (q & 1)))) q += 1;
    }
    /* q <= 2^53 is exact in binary64; scaling by a power of two is exact here */
    return ldexp((double)(uint64_t)q, shift + 64 * base - 298);
}

/* Adds the squares of the averaged gradient at n positions to the accumulator. */
int orc_sqnorm_accumulate(orc_sqacc *a, int64_t n, int32_t n_ranks, const void *const *grads,
                          int32_t gdtype, const uint8_t *pad)
{
    if (n < 0 || n_ranks < 1 || (gdtype != ORC_F32 && gdtype != ORC_BF16)) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) orc_sqacc_add_square(a, orc_avg_grad(n_ranks, grads, gdtype, pad, i));
    return ORC_OK;
}

/* Clip coefficient from the squared norm S.  Reading (the pages name the
 * operation, not its formula): norm = sqrt(S), coef = min(1, max_norm /
 * (norm + 1e-6)), all in binary64, rounded once to binary32.  A non-finite S
 * returns NaN, which means "skip the step". */
float orc_clip_coef(double S, float max_norm)
{
    if (!isfinite(S)) return NAN;
    double c = (double)max_norm / (sqrt(S) + 1e-6);
    if (c > 1.0) c = 1.0;
    return (float)c;
}

/* ------------------------------------------------------------------------ */
/* Unsharded AdamW on the rank-ordered averaged gradient.
 * [P1] Code, AdamW::step (b1, b2, eps, wd, decoupled weight decay, bias
 * corrections) and the unsharded check that the sharded run must equal bit
 * for bit.  [P3] section 1: the update is element-wise, so any partition of
 * the elements gives the same result.  Operation order, each one rounded:
 *   m = (b1*m) + ((1-b1)*g)
 *   v = (b2*v) + (((1-b2)*g)*g)
 *   w = (w*(1 - lr*wd)) - (((lr/bc1)*m) / ((sqrt(v)/bc2) + eps))
 * If clip != 0, g is first multiplied by coef (binary32).  The output is the
 * bf16 rounding of w (pdtype BF16) or w itself (pdtype F32); out may be NULL.
 * n positions; grads[q] points at rank q's values for those same positions. */
int orc_adamw(int64_t n, int32_t n_ranks, const void *const *grads, int32_t gdtype,
              const uint8_t *pad, float *w, float *m, float *v, void *out, int32_t pdtype,
              const orc_hparams *hp, int32_t clip, float coef)
{
    if (n < 0 || n_ranks < 1 || (gdtype != ORC_F32 && gdtype != ORC_BF16) ||
        (pdtype != ORC_F32 && pdtype != ORC_BF16) || hp == NULL)
        return ORC_EINVAL;
    float bc1, bc2;
    if (orc_bias_corrections(hp->t, hp->b1, hp->b2, &bc1, &bc2) != ORC_OK) return ORC_EINVAL;
    const float one_minus_b1 = 1.0f - hp->b1;
    const float one_minus_b2 = 1.0f - hp->b2;
    const float decay = 1.0f - hp->lr * hp->wd;
    const float lr_over_bc1 = hp->lr / bc1;
    for (int64_t i = 0; i < n; ++i) {
        float g = orc_avg_grad(n_ranks, grads, gdtype, pad, i);
        if (clip) g = g * coef;
        float mi = hp->b1 * m[i] + one_minus_b1 * g;
        float vi = hp->b2 * v[i] + one_minus_b2 * g * g;
        float wi = w[i] * decay - lr_over_bc1 * mi / (sqrtf(vi) / bc2 + hp->eps);
        m[i] = mi;
        v[i] = vi;
        w[i] = wi;
        if (out != NULL) {
            if (pdtype == ORC_F32) ((float *)out)[i] = wi;
            else ((uint16_t *)out)[i] = orc_bf16_rne(wi);
        }
    }
    return ORC_OK;
}

/* One whole step over n positions: with clipping on (max_norm > 0), S over
 * these positions, coef, and a skipped step (state untouched, ORC_ENONFINITE)
 * when S is not finite; then the update.  *sqnorm (nullable) receives S. */
int orc_step(int64_t n, int32_t n_ranks, const void *const *grads, int32_t gdtype,
             const uint8_t *pad, float *w, float *m, float *v, void *out, int32_t pdtype,
             const orc_hparams *hp, double *sqnorm)
{
    if (hp == NULL) return ORC_EINVAL;
    int clip = hp->max_norm > 0.0f;
    float coef = 1.0f;
    if (clip) {
        orc_sqacc acc;
        memset(&acc, 0, sizeof acc);
        int rc = orc_sqnorm_accumulate(&acc, n, n_ranks, grads, gdtype, pad);
        if (rc != ORC_OK) return rc;
        double S = orc_sqacc_result(&acc);
        if (sqnorm != NULL) *sqnorm = S;
        coef = orc_clip_coef(S, hp->max_norm);
        if (isnan(coef)) return ORC_ENONFINITE;
    }
    return orc_adamw(n, n_ranks, grads, gdtype, pad, w, m, v, out, pdtype, hp, clip, coef);
}

/* ------------------------------------------------------------------------ */
/* The pages' toy, both ways.  [P1] Code: N ranks hold the full weights w, each
 * with its own target; the local loss is 1/2 |w - target|^2 so the local
 * gradient is w - target.  Each step the ranks reduce-scatter the gradient,
 * divide by n, run AdamW on their fp32 master slice, and all-gather the
 * updated slices.  The claim: every rank ends with exactly the weights of
 * unsharded AdamW on the averaged gradient.  P is padded to a multiple of N
 * (the page leaves this to "real code"); padding positions carry gradient 0. */
typedef struct {
    int32_t N;
    int64_t P, Ppad, h;
    int32_t steps;
    const float *targets; /* [N][P] */
    const float *w0;      /* [P] */
    const orc_hparams *hp;
    float *w_out;         /* [N][P] */
    pthread_barrier_t barrier;
    float **slots;        /* the shared exchange slots, one per rank */
} orc_toy_ctx;

typedef struct { orc_toy_ctx *ctx; int32_t rank; int rc; } orc_toy_arg;

static void orc_toy_exchange(orc_toy_ctx *c, int32_t rank, float *buf)
{
    c->slots[rank] = buf;                 /* publish */
    pthread_barrier_wait(&c->barrier);    /* everyone has published */
}

static void *orc_toy_rank(void *p)
{
    orc_toy_arg *arg = (orc_toy_arg *)p;
    orc_toy_ctx *c = arg->ctx;
    const int32_t r = arg->rank, N = c->N;
    const int64_t h = c->h;
    float *w = calloc((size_t)c->Ppad, sizeof(float));
    float *g = calloc((size_t)c->Ppad, sizeof(float));
    float *master = calloc((size_t)h, sizeof(float));
    float *m = calloc((size_t)h, sizeof(float));
    float *v = calloc((size_t)h, sizeof(float));
    float *gs = calloc((size_t)h, sizeof(float));
    if (!w || !g || !master || !m || !v || !gs) { arg->rc = ORC_EINVAL; }
    /* every rank must reach every barrier, so an allocation failure is only
       reported at the end */
    if (arg->rc == ORC_OK) {
        memcpy(w, c->w0, (size_t)c->P * sizeof(float));
        for (int64_t j = 0; j < h; ++j) master[j] = w[(int64_t)r * h + j];
    }
    orc_hparams hp = *c->hp;
    const float *tr = c->targets + (int64_t)r * c->P;
    for (int32_t step = 0; step < c->steps; ++step) {
        if (arg->rc == ORC_OK)
            for (int64_t i = 0; i < c->Ppad; ++i) g[i] = i < c->P ? w[i] - tr[i] : 0.0f;
        /* reduce-scatter: rank r sums slice r over all ranks, in rank order */
        orc_toy_exchange(c, r, g);
        if (arg->rc == ORC_OK)
            for (int64_t j = 0; j < h; ++j) {
                float acc = c->slots[0][(int64_t)r * h + j];
                for (int32_t q = 1; q < N; ++q) acc = acc + c->slots[q][(int64_t)r * h + j];
                gs[j] = acc / (float)N;
            }
        pthread_barrier_wait(&c->barrier); /* nobody overwrites before all have read */
        /* local AdamW on the master slice; the step counter is 1-based */
        hp.t = step + 1;
        if (arg->rc == ORC_OK) {
            const void *gsp[1] = {gs};
            orc_adamw(h, 1, gsp, ORC_F32, NULL, master, m, v, NULL, ORC_F32, &hp, 0, 1.0f);
        }
        /* all-gather of the updated slices (fp32 in the toy) */
        orc_toy_exchange(c, r, master);
        if (arg->rc == ORC_OK)
            for (int32_t q = 0; q < N; ++q)
                memcpy(w + (int64_t)q * h, c->slots[q], (size_t)h * sizeof(float));
        pthread_barrier_wait(&c->barrier);
    }
    if (arg->rc == ORC_OK) memcpy(c->w_out + (int64_t)r * c->P, w, (size_t)c->P * sizeof(float));
    free(w); free(g); free(master); free(m); free(v); free(gs);
    return NULL;
}

/* Sharded: N threads, barrier-synchronised exchange.  w_out[r][:] = rank r's
 * final full weights. */
int orc_toy_zero2_threads(int32_t N, int64_t P, int32_t steps, const float *targets,
                          const float *w0, const orc_hparams *hp, float *w_out)
{
    if (N < 1 || N > 1024 || P < 0 || steps < 0 || hp == NULL) return ORC_EINVAL;
    orc_toy_ctx c;
    c.N = N; c.P = P; c.steps = steps; c.targets = targets; c.w0 = w0; c.hp = hp; c.w_out = w_out;
    c.Ppad = (P % N == 0) ? P : P + (N - P % N);
    c.h = c.Ppad / N;
    c.slots = calloc((size_t)N, sizeof(float *));
    pthread_t *th = calloc((size_t)N, sizeof(pthread_t));
    orc_toy_arg *args = calloc((size_t)N, sizeof(orc_toy_arg));
    if (!c.slots || !th || !args) { free(c.slots); free(th); free(args); return ORC_EINVAL; }
    pthread_barrier_init(&c.barrier, NULL, (unsigned)N);
    int rc = ORC_OK;
    int32_t started = 0;
    for (int32_t r = 0; r < N; ++r) {
        args[r].ctx = &c; args[r].rank = r; args[r].rc = ORC_OK;
        if (pthread_create(&th[r], NULL, orc_toy_rank, &args[r]) != 0) { rc = ORC_EINVAL; break; }
        ++started;
    }
    /* a rank that failed to start would leave the others at the barrier */
    if (started != N) abort();
    for (int32_t r = 0; r < N; ++r) {
        pthread_join(th[r], NULL);
        if (args[r].rc != ORC_OK) rc = args[r].rc;
    }
    pthread_barrier_destroy(&c.barrier);
    free(c.slots); free(th); free(args);
    return rc;
}

/* Unsharded: one AdamW over all P weights on the averaged gradient
 * sum_r (w - target_r) / n, summed in rank order. */
int orc_toy_unsharded(int32_t N, int64_t P, int32_t steps, const float *targets,
                      const float *w0, const orc_hparams *hp, float *w_out)
{
    if (N < 1 || P < 0 || steps < 0 || hp == NULL) return ORC_EINVAL;
    float *m = calloc((size_t)(P > 0 ? P : 1), sizeof(float));
    float *v = calloc((size_t)(P > 0 ? P : 1), sizeof(float));
    float *g = calloc((size_t)(P > 0 ? P : 1), sizeof(float));
    if (!m || !v || !g) { free(m); free(v); free(g); return ORC_EINVAL; }
    memcpy(w_out, w0, (size_t)P * sizeof(float));
    orc_hparams hp1 = *hp;
    for (int32_t step = 0; step < steps; ++step) {
        for (int64_t i = 0; i < P; ++i) {
            float acc = w_out[i] - targets[i];
            for (int32_t q = 1; q < N; ++q) acc = acc + (w_out[i] - targets[(int64_t)q * P + i]);
            g[i] = acc / (float)N;
        }
        hp1.t = step + 1;
        const void *gp[1] = {g};
        orc_adamw(P, 1, gp, ORC_F32, NULL, w_out, m, v, NULL, ORC_F32, &hp1, 0, 1.0f);
    }
    free(m); free(v); free(g);
    return ORC_OK;
}
