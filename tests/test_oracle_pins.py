"""Pins of the CPU oracle to what the pages and the mathematics fix (no GPU).

Each test names the passage it pins (page title, section) and what a plausible
mistake in the oracle would do to it.
"""
import json
import math
import os
from concurrent.futures import ThreadPoolExecutor
from fractions import Fraction

import numpy as np
import pytest
import torch

import fp_exact as X
from fsdp_sharded_optimizer_step_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOY_HP = dict(lr=0.01, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)


def hp(orc, **kw):
    d = dict(TOY_HP)
    d.update(kw)
    return orc.hparams(**d)


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ----------------------------------------------------------------------------
# "ZeRO and FSDP sharding", Code: ZeRO-2 on threads must equal unsharded AdamW
# on the averaged gradient, bit for bit (N=4, P=1000, 50 steps).  Catches any
# error in the reduce-scatter slice indexing, the rank order or the gather.
def test_toy_sharded_threads_equal_unsharded_bit_for_bit(orc):
    t = W.toy_targets(4, 1000).numpy()
    w0 = np.zeros(1000, np.float32)
    res = orc.toy_zero2_threads(t, w0, 50, hp(orc))
    ref = orc.toy_unsharded(t, w0, 50, hp(orc))
    for r in range(4):
        assert np.array_equal(bits(res[r]), bits(ref)), f"rank {r}"
    assert np.all(ref > 0.3)  # the weights really moved


@pytest.mark.parametrize("N", range(1, 9))
def test_sharded_equals_unsharded_brute_force_with_padding(orc, N):
    """P not a multiple of N exercises the padding ("ZeRO and FSDP sharding", Pitfalls)."""
    rng = np.random.default_rng(100 + N)
    for P in [1, 2, 3, 5, 7, 11, 13, 17, 31, 37, 64]:
        t = rng.normal(0.0, 3.0, size=(N, P)).astype(np.float32)
        w0 = rng.normal(0.0, 1.0, P).astype(np.float32)
        res = orc.toy_zero2_threads(t, w0, 4, hp(orc))
        ref = orc.toy_unsharded(t, w0, 4, hp(orc))
        for r in range(N):
            assert np.array_equal(bits(res[r]), bits(ref)), (N, P, r)


# ----------------------------------------------------------------------------
# "ZeRO and FSDP sharding", Code, AdamW::step.  Closed form of step 1 with
# m0 = v0 = 0: m1 = (1-b1) g, v1 = (1-b2) g^2, so the bias-corrected ratio is
# g/(|g| + eps) and w1 = w0 (1 - lr wd) - lr g/(|g| + eps).  Catches a missing
# or wrong bias correction, a coupled (L2) weight decay, a sign error.
def test_first_step_closed_form(orc):
    rng = np.random.default_rng(7)
    n = 4000
    w0 = rng.normal(0, 1, n).astype(np.float32)
    mag = np.exp(rng.uniform(np.log(1e-6), np.log(1e3), n))
    g = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    # two ranks holding the same value: the average is exactly g
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    orc.adamw([g, g], orc.F32, w, m, v, hp(orc, t=1))
    lr, wd, eps = float(np.float32(0.01)), float(np.float32(0.1)), float(np.float32(1e-8))
    gd = g.astype(np.float64)
    expect = w0.astype(np.float64) * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    tol = 2e-6 * (np.abs(w0) + lr)
    assert np.all(np.abs(w - expect) <= tol), np.max(np.abs(w - expect) / tol)


def test_toy_first_step_moves_every_weight_by_lr(orc):
    """Toy: w0 = 0 and g = -mean_r target < 0 for every i, so w1 = +lr (to rounding)."""
    t = W.toy_targets(4, 1000).numpy()
    w1 = orc.toy_unsharded(t, np.zeros(1000, np.float32), 1, hp(orc))
    assert np.all(np.abs(w1 - 0.01) <= 1e-8), np.max(np.abs(w1 - 0.01))


# Constant gradient for T steps: m_t = (1 - b1^t) g and v_t = (1 - b2^t) g^2
# exactly in real arithmetic, so every bias-corrected step is lr g/(|g|+eps):
#   w_T = c^T w0 - lr s sum_{k<T} c^k,   c = 1 - lr wd,   s = g/(|g|+eps).
# Catches a bias correction applied with the wrong power, without the square
# root, or not at all, at every t (b1 != b2 keeps the two corrections apart).
def test_constant_gradient_closed_form_over_steps(orc):
    rng = np.random.default_rng(11)
    n, T = 2000, 60
    w0 = rng.normal(0, 1, n).astype(np.float32)
    g = (np.exp(rng.uniform(np.log(1e-4), np.log(10.0), n)) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, T + 1):
        orc.adamw([g], orc.F32, w, m, v, hp(orc, t=t))
    lr, wd, eps = float(np.float32(0.01)), float(np.float32(0.1)), float(np.float32(1e-8))
    c = 1 - lr * wd
    s = g.astype(np.float64) / (np.abs(g.astype(np.float64)) + eps)
    expect = c ** T * w0.astype(np.float64) - lr * s * sum(c ** k for k in range(T))
    assert np.max(np.abs(w - expect)) <= 2e-5, np.max(np.abs(w - expect))


# "ZeRO and FSDP sharding", Code: local loss 1/2 |w - target|^2, so the
# averaged gradient is w - mean target and the optimum is the mean target.
# Over the toy's 50 steps every |w_i - mean_i| shrinks monotonically (all
# means are >= 1.5, since the four residues 7i + 13r mod 11 are distinct, and a
# step is at most about 1.17 lr), and w_50 stays below 50 x 1.17 lr.  Catches
# a gradient-sign or target-indexing error.
def test_toy_converges_toward_mean_target(orc):
    N, P = 4, 1000
    t = W.toy_targets(N, P).numpy()
    tbar = t.astype(np.float64).mean(axis=0)
    assert tbar.min() >= 1.5
    w, m, v = np.zeros(P, np.float32), np.zeros(P, np.float32), np.zeros(P, np.float32)
    dist = np.abs(w - tbar)
    for step in range(1, 51):
        grads = [w - t[r] for r in range(N)]  # each rank's local gradient of the toy loss
        orc.adamw(grads, orc.F32, w, m, v, hp(orc, t=step), pdtype=orc.F32)
        d = np.abs(w - tbar)
        assert np.all(d < dist), step
        dist = d
    assert np.all(w > 0.3) and np.all(w < 50 * 1.17 * 0.01)
    assert np.array_equal(bits(w), bits(orc.toy_unsharded(t, np.zeros(P, np.float32), 50, hp(orc))))


# ----------------------------------------------------------------------------
# "ZeRO and FSDP sharding", Code, Comm::reduce_scatter: the sum runs over the
# ranks in rank order.  With b1 = 0, m after one step equals the averaged
# gradient exactly, which exposes the fold.
def _avg_grad_via_m(orc, grads, gdtype=None):
    gdtype = orc.F32 if gdtype is None else gdtype
    n = np.asarray(grads[0]).size
    w, m, v = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    orc.adamw(grads, gdtype, w, m, v, hp(orc, b1=0.0, t=1))
    return m


def test_reduce_is_a_left_fold_in_rank_order(orc):
    big = np.float32(2.0 ** 24)
    one = np.float32(1.0)
    # [1, 2^24, -2^24]: ((1 + 2^24) + -2^24) = 0 (the tie rounds to even); any
    # other bracketing gives 1/3
    g = [np.array([one]), np.array([big]), np.array([-big])]
    assert _avg_grad_via_m(orc, g)[0] == 0.0
    # [2^24, 1, 1, -2^24]: left fold 0, pairwise 0.25, reversed 0.5
    g = [np.array([big]), np.array([one]), np.array([one]), np.array([-big])]
    assert _avg_grad_via_m(orc, g)[0] == 0.0


def test_reduce_and_average_are_correctly_rounded(orc):
    rng = np.random.default_rng(5)
    for N in (1, 2, 3, 5, 7, 8, 16):
        vals = (rng.normal(0, 1, (N, 300)) * np.exp(rng.uniform(-20, 20, (N, 300)))).astype(np.float32)
        m = _avg_grad_via_m(orc, list(vals))
        for i in range(300):
            acc = vals[0, i]
            for q in range(1, N):
                acc = X.add(acc, vals[q, i])
            expect = X.div(acc, np.float32(N))
            assert bits(m[i]) == bits(expect), (N, i)


def test_average_divides_by_n_not_multiplies_by_reciprocal(orc):
    """"ZeRO and FSDP sharding", Code: x /= n.  For N = 3 a division and a
    multiplication by fp32(1/3) differ on some inputs; the oracle must divide."""
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, 20000).astype(np.float32)
    recip = np.float32(1.0) / np.float32(3.0)
    differ = x[(x / np.float32(3.0)) != (x * recip)]
    assert differ.size > 10
    z = np.zeros_like(differ)
    m = _avg_grad_via_m(orc, [differ, z, z])
    expect = np.array([X.div(a, np.float32(3.0)) for a in differ], np.float32)
    assert np.array_equal(bits(m), bits(expect))
    assert not np.array_equal(bits(m), bits(differ * recip))


def test_padding_positions_contribute_zero(orc):
    rng = np.random.default_rng(9)
    g = [rng.normal(0, 1, 50).astype(np.float32) for _ in range(3)]
    pad = (np.arange(50) >= 40).astype(np.uint8)
    n = 50
    w, m, v = np.ones(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    orc.adamw(g, orc.F32, w, m, v, hp(orc, b1=0.0), pad=pad)
    assert np.all(m[40:] == 0.0) and np.all(v[40:] == 0.0)
    decay = X.sub(np.float32(1), X.mul(np.float32(0.01), np.float32(0.1)))
    assert np.all(bits(w[40:]) == bits(decay))  # 1 * decay - 0/(0 + eps)


# ----------------------------------------------------------------------------
# Arithmetic contract: each operation of the update is one correctly rounded
# binary32 operation, in the order the page's AdamW::step writes them.  The
# expected values come from exact rational arithmetic (fp_exact), not from any
# floating-point unit; a fused multiply-add or an approximate sqrt/divide in
# the oracle fails this.
def test_update_is_sequence_of_correctly_rounded_ops(orc):
    rng = np.random.default_rng(21)
    n = 400
    w0 = rng.normal(0, 1, n).astype(np.float32)
    m0 = (rng.normal(0, 1e-2, n)).astype(np.float32)
    v0 = np.abs(rng.normal(0, 1e-4, n)).astype(np.float32)
    g = (rng.normal(0, 1, n) * np.exp(rng.uniform(-8, 3, n))).astype(np.float32)
    for t in (1, 2, 7, 1000):
        w, m, v = w0.copy(), m0.copy(), v0.copy()
        out = orc.adamw([g], orc.F32, w, m, v, hp(orc, t=t), pdtype=orc.BF16)
        b1, b2 = np.float32(0.9), np.float32(0.95)
        lr, eps, wd = np.float32(0.01), np.float32(1e-8), np.float32(0.1)
        bc1, bc2 = orc.bias_corrections(t)
        omb1, omb2 = X.sub(np.float32(1), b1), X.sub(np.float32(1), b2)
        decay = X.sub(np.float32(1), X.mul(lr, wd))
        lr_bc1 = X.div(lr, bc1)
        for i in range(n):
            mi = X.add(X.mul(b1, m0[i]), X.mul(omb1, g[i]))
            vi = X.add(X.mul(b2, v0[i]), X.mul(X.mul(omb2, g[i]), g[i]))
            den = X.add(X.div(X.sqrt(vi), bc2), eps)
            wi = X.sub(X.mul(w0[i], decay), X.div(X.mul(lr_bc1, mi), den))
            assert bits(m[i]) == bits(mi) and bits(v[i]) == bits(vi) and bits(w[i]) == bits(wi), (t, i)
            assert out[i] == X.rn_bf16_bits(wi), (t, i)


def test_bias_corrections(orc):
    """"ZeRO and FSDP sharding", Code: bc1 = 1 - b1^t, bc2 = sqrt(1 - b2^t)."""
    b1, b2 = np.float32(0.9), np.float32(0.95)
    bc1, bc2 = orc.bias_corrections(1)
    assert bits(bc1) == bits(X.sub(np.float32(1), b1))
    assert bits(bc2) == bits(X.sqrt(X.sub(np.float32(1), b2)))
    for t in list(range(1, 200)) + [500, 1000, 5000, 100000]:
        bc1, bc2 = orc.bias_corrections(t)
        e1 = 1 - float(b1) ** t
        e2 = math.sqrt(1 - float(b2) ** t)
        assert abs(bc1 - e1) <= 2e-6 and abs(bc2 - e2) <= 2e-6, t
    with pytest.raises(RuntimeError):
        orc.bias_corrections(0)


# ----------------------------------------------------------------------------
# bf16 cast ("ZeRO and FSDP sharding", How it works: cast to bf16 shard).
# Reading: round to nearest even.  Pinned to torch's float->bfloat16
# conversion (a library routine with that rounding) on every high half and a
# set of low halves that includes every tie, and to exact rounding.
def test_bf16_matches_library_conversion(orc):
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    rng = np.random.default_rng(1)
    lows = np.concatenate([np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32),
                           rng.integers(0, 1 << 16, 26).astype(np.uint32)])
    b = (hi[:, None] | lows[None, :]).ravel()
    x = b.view(np.float32)
    ours = orc.bf16_rne_array(x)
    nan = np.isnan(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours[~nan], ref[~nan])
    o = ours[nan]
    assert np.all((o & 0x7F80) == 0x7F80) and np.all((o & 0x7F) | 0x40 != 0) and np.all(o & 0x40)
    assert np.array_equal(o & 0x8000, (b[nan] >> 16).astype(np.uint16) & 0x8000)


def test_bf16_exhaustive_against_library_conversion(orc):
    """Every one of the 2^32 binary32 bit patterns: the oracle's cast equals
    torch's float->bfloat16 conversion on all non-NaN inputs; NaN inputs (two
    known ranges of bit patterns) give a quiet NaN of the same sign."""
    ch = 1 << 24
    base = np.arange(ch, dtype=np.uint32)
    nan_ranges = [(0x7F800001, 0x80000000), (0xFF800001, 1 << 32)]

    def check(c):
        lo = c * ch
        b = base + np.uint32(lo)
        x = b.view(np.float32)
        ours = orc.bf16_rne_array(x)
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ne = ours != ref
        for a, e in nan_ranges:
            s, t = max(a, lo) - lo, min(e, lo + ch) - lo
            if s < t:
                ne[s:t] = False
                o = ours[s:t]
                assert np.all((o & 0x7F80) == 0x7F80) and np.all(o & 0x40)
                assert np.array_equal(o >> 15, (b[s:t] >> 31).astype(np.uint16))
        return int(np.count_nonzero(ne))

    with ThreadPoolExecutor(os.cpu_count() or 1) as ex:  # the oracle's C call releases the GIL
        assert sum(ex.map(check, range((1 << 32) // ch))) == 0


def test_bf16_matches_exact_rounding(orc):
    rng = np.random.default_rng(2)
    b = rng.integers(0, 1 << 32, 3000, dtype=np.uint64).astype(np.uint32)
    b[:500] = (b[:500] & 0xFFFF0000) | 0x8000  # exact ties
    x = b.view(np.float32)
    x = x[np.isfinite(x)]
    ours = orc.bf16_rne_array(x)
    for xi, oi in zip(x, ours):
        assert int(oi) == X.rn_bf16_bits(xi), hex(X.f32_bits(xi))


# ----------------------------------------------------------------------------
# Global gradient norm ("ZeRO and FSDP sharding", Implementation notes; "ZeRO:
# Three Ledgers, Zero Redundancy", section 2: a sum of squares).  The oracle's
# S is the exact sum rounded once; pinned to exact rational summation and to
# math.fsum (a correctly rounded library sum).
def test_sqnorm_is_exact_sum_of_squares(orc):
    rng = np.random.default_rng(4)
    for trial in range(20):
        n = int(rng.integers(1, 300))
        x = (rng.normal(0, 1, n) * np.exp(rng.uniform(-90, 60, n))).astype(np.float32)
        S = orc.sqnorm([x], orc.F32)
        exact = sum(Fraction(float(a)) ** 2 for a in x)
        assert S == X.rn64(exact), trial
    x = (rng.normal(0, 1, 200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    assert orc.sqnorm([x], orc.F32) == math.fsum(float(a) ** 2 for a in x.astype(np.float64))


def test_sqnorm_partial_accumulators_merge_exactly(orc):
    """Squares taken over disjoint chunks and merged give the one-pass S, which is
    the exact rational sum rounded once (the accumulator is free of any order)."""
    rng = np.random.default_rng(11)
    x = (rng.normal(0, 1, 3000) * np.exp(rng.uniform(-60, 60, 3000))).astype(np.float32)
    x[:40] = np.float32(3.0e38)  # carries across limbs
    whole = orc.sqnorm([x], orc.F32)
    assert whole == X.rn64(sum(Fraction(float(a)) ** 2 for a in x))
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, x.size), 7, replace=False))
        acc = orc.SqAcc()
        for part in np.split(x, cuts):
            a = orc.SqAcc()
            a.add_avg_grad([part], orc.F32)
            acc.merge(a)
        assert acc.result() == whole, trial
    # a carry out of a full limb: 2^21 squares of 1.0 fill half of one 64-bit limb, two halves overflow it
    ones = np.ones(1 << 21, np.float32)
    a, b = orc.SqAcc(), orc.SqAcc()
    a.add_avg_grad([ones], orc.F32)
    b.add_avg_grad([ones], orc.F32)
    a.merge(b)
    assert a.result() == float(1 << 22)
    a, b = orc.SqAcc(), orc.SqAcc()
    a.add_avg_grad([x[:10]], orc.F32)
    b.add_avg_grad([np.array([np.inf], np.float32)], orc.F32)
    a.merge(b)
    assert math.isinf(a.result())
    b.add_avg_grad([np.array([np.nan], np.float32)], orc.F32)
    a.merge(b)
    assert math.isnan(a.result())


def test_sqnorm_of_averaged_gradient_with_pads(orc):
    rng = np.random.default_rng(6)
    g = [rng.normal(0, 1, 64).astype(np.float32) for _ in range(4)]
    pad = (np.arange(64) % 9 == 0).astype(np.uint8)
    avg = _avg_grad_via_m(orc, g)  # pinned above
    avg[pad == 1] = 0.0
    assert orc.sqnorm(g, orc.F32, pad) == math.fsum(float(a) ** 2 for a in avg.astype(np.float64))


def test_sqnorm_non_finite(orc):
    assert math.isinf(orc.sqnorm([np.array([1.0, np.inf], np.float32)], orc.F32))
    assert math.isnan(orc.sqnorm([np.array([1.0, np.nan, np.inf], np.float32)], orc.F32))
    assert orc.sqnorm([np.zeros(5, np.float32)], orc.F32) == 0.0


def test_clip_rescales_global_norm_to_max_norm(orc):
    """Clipping by the global norm leaves a gradient of norm max_norm (up to the
    1e-6 guard), and leaves a gradient already inside the ball untouched."""
    rng = np.random.default_rng(8)
    x = rng.normal(0, 1, 5000).astype(np.float32)
    S = orc.sqnorm([x], orc.F32)
    for max_norm in (0.5, 1.0, 3.0):
        c = orc.clip_coef(S, max_norm)
        assert 0 < c < 1
        S2 = orc.sqnorm([x * c], orc.F32)
        assert abs(math.sqrt(S2) - max_norm) <= 1e-5 * max_norm
    assert orc.clip_coef(S, 10 * math.sqrt(S)) == 1.0
    assert orc.clip_coef(0.0, 1.0) == 1.0
    assert math.isnan(orc.clip_coef(math.inf, 1.0)) and math.isnan(orc.clip_coef(math.nan, 1.0))


def test_clip_coef_matches_library_clip(orc):
    """The clip formula is a reading (the pages name the operation, not its
    formula): the library routine torch.nn.utils.clip_grad_norm_ (fp64 grads,
    so its norm is accurate to a few binary64 ulps) gives the same coefficient
    after rounding to binary32, including the 1e-6 guard at norm == max_norm."""
    rng = np.random.default_rng(13)
    cases = [(np.array([3.0, 4.0], np.float32), 5.0), (np.array([3.0, 4.0], np.float32), 1.0)]
    for _ in range(30):
        x = (rng.normal(0, 1, int(rng.integers(1, 500))) * np.exp(rng.uniform(-5, 5))).astype(np.float32)
        cases.append((x, float(np.float32(rng.uniform(0.1, 3.0)))))
    for x, max_norm in cases:
        S = orc.sqnorm([x], orc.F32)
        c = orc.clip_coef(S, max_norm)
        p = torch.nn.Parameter(torch.zeros(x.size, dtype=torch.float64))
        p.grad = torch.from_numpy(x.astype(np.float64))
        torch.nn.utils.clip_grad_norm_([p], max_norm)
        k = int(np.argmax(np.abs(x)))
        c_lib = np.float32(p.grad[k].item() / float(x[k]))
        assert c == c_lib, (max_norm, c, c_lib)
    # at norm == max_norm the guard keeps the coefficient strictly below 1
    assert orc.clip_coef(25.0, 5.0) < 1.0


def test_step_with_clip_scales_gradient_by_coef(orc):
    rng = np.random.default_rng(10)
    g = (rng.normal(0, 1, 3000) * 10).astype(np.float32)
    n = g.size
    w, m, v = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    rc, _, S = orc.step([g], orc.F32, w, m, v, hp(orc, b1=0.0, max_norm=1.0))
    assert rc == orc.OK
    assert S == math.fsum(float(a) ** 2 for a in g.astype(np.float64))
    c = orc.clip_coef(S, 1.0)
    assert np.array_equal(bits(m), bits(np.array([X.mul(a, c) for a in g], np.float32)))


def test_step_skipped_when_norm_not_finite(orc):
    g = np.array([1.0, np.inf, 2.0], np.float32)
    w, m, v = np.ones(3, np.float32), np.full(3, 0.5, np.float32), np.full(3, 0.25, np.float32)
    rc, _, S = orc.step([g], orc.F32, w, m, v, hp(orc, max_norm=1.0))
    assert rc == orc.ENONFINITE and math.isinf(S)
    assert np.all(w == 1.0) and np.all(m == 0.5) and np.all(v == 0.25)


def test_clip_off_equals_no_clip_when_inside_ball(orc):
    rng = np.random.default_rng(12)
    g = [(rng.normal(0, 1e-3, 700)).astype(np.float32) for _ in range(2)]
    outs = []
    for max_norm in (0.0, 100.0):
        w, m, v = np.ones(700, np.float32), np.zeros(700, np.float32), np.zeros(700, np.float32)
        rc, out, _ = orc.step(g, orc.F32, w, m, v, hp(orc, max_norm=max_norm))
        assert rc == orc.OK
        outs.append((bits(w).copy(), bits(m).copy(), out.copy()))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


# ----------------------------------------------------------------------------
# Layout ("ZeRO and FSDP sharding", How it works and Pitfalls; "Learn: ZeRO &
# FSDP", section 5).  Brute force over unit lists and N: every unit padded to
# the next multiple of N, slices tile each unit once, the shard map is a
# permutation, pads are the trailing S_u - s_u positions of each unit.  The
# alignment option (align > 1, not on the pages) pads to the next multiple of
# N*align instead, so every slice length is a multiple of align.
@pytest.mark.parametrize("align", [1, 2, 8])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 13, 16])
def test_plan_brute_force(orc, N, align):
    rng = np.random.default_rng(N * 10 + align)
    q = N * align
    for trial in range(30):
        U = int(rng.integers(1, 12))
        sizes = rng.integers(0, 60, U)
        sizes[rng.random(U) < 0.2] = 0
        p = orc.Plan(sizes, N, align)
        for u in range(U):
            s = int(sizes[u])
            assert p.S[u] % q == 0 and s <= p.S[u] < s + q
            assert p.S[u] == min(k for k in range(s, s + q) if k % q == 0)
            assert p.h[u] * N == p.S[u] and p.h[u] % align == 0
            assert p.F[u] == sum(p.S[:u]) and p.Hoff[u] == sum(p.h[:u])
        assert p.P_pad == sum(p.S) and p.H * N == p.P_pad
        mp = p.shard_map()
        assert np.array_equal(np.sort(mp.ravel()), np.arange(p.P_pad))
        for u in range(U):
            for r in range(N):
                sl = mp[r, p.Hoff[u]:p.Hoff[u] + p.h[u]]
                assert np.array_equal(sl, p.F[u] + r * p.h[u] + np.arange(p.h[u]))
        pad = p.pad_mask()
        assert pad.sum() == p.P_pad - sizes.sum()
        for u in range(U):
            seg = pad[p.F[u]:p.F[u] + p.S[u]]
            assert np.array_equal(seg, (np.arange(p.S[u]) >= sizes[u]).astype(np.uint8))
        # locate is the inverse of the shard map, with the pad flag of the position
        if p.P_pad:
            allpos = np.arange(p.P_pad, dtype=np.int64)
            rank, spos, isp = p.locate(allpos[::-1].copy())
            assert np.array_equal(mp[rank, spos], allpos[::-1])
            assert np.array_equal(isp, pad[::-1])
        with pytest.raises(RuntimeError):
            p.locate(np.array([p.P_pad], np.int64))


def test_plan_named_workloads(orc):
    p = orc.Plan(W.toy_units(), 4)
    assert list(p.S) == [1000] and list(p.h) == [250] and p.P_pad == 1000
    p = orc.Plan(W.gpt2l_units(), 8)
    assert p.P_pad == 774_030_080 and p.H == 96_753_760 and np.all(p.S == W.gpt2l_units())
    p = orc.Plan(W.gpt_1p3b_units(), 8)
    assert p.P_pad == 1_311_524_864 and p.H == 163_940_608
    p = orc.Plan(W.llm_4b_units(), 8)
    assert p.P_pad == 3_999_989_760
    sizes = W.finewrap_units()
    p = orc.Plan(sizes, 16)
    assert np.all(p.S % 16 == 0) and np.mean(p.S != sizes) > 0.9


def test_plan_rejects_bad_input(orc):
    with pytest.raises(RuntimeError):
        orc.Plan([5, -1], 2)
    with pytest.raises(RuntimeError):
        orc.Plan([5], 0)
    with pytest.raises(RuntimeError):
        orc.Plan([5], 2, 0)


# ----------------------------------------------------------------------------
# Memory and communication ledger: every worked value the pages print.
def test_ledger_worked_examples():
    from oracle import ledger
    d = json.load(open(os.path.join(GOLDEN, "ledger_examples.json")))
    for e in d["memory"]:
        got = ledger.model_state_bytes(e["psi"], e["n"], e["stage"]) / e["unit"]
        assert abs(got - e["value"]) <= e["tol"] + 1e-12, (e["cite"], got)
    for e in d["differences"]:
        got = (ledger.model_state_bytes(e["psi"], e["n"], e["from_stage"]) -
               ledger.model_state_bytes(e["psi"], e["n"], e["to_stage"])) / e["unit"]
        assert abs(got - e["value"]) <= e["tol"], (e["cite"], got)
    for e in d["inconsistent"]:
        got = ledger.model_state_bytes(e["psi"], e["n"], e["stage"]) / e["unit"]
        assert abs(got - e["formula_value"]) < 1e-9 and abs(got - e["printed"]) > 0.3
    for e in d["min_ranks"]:
        assert ledger.min_ranks_to_fit(e["psi"], e["hbm"], e["stage"]) == e["value"], e["cite"]
    for e in d["comm"]:
        assert ledger.comm_elements(1.0, e["stage"]) == e["value_psi"], e["cite"]
    e = d["toy_floats_per_rank"]
    assert 3 * (e["p"] // e["n"]) == e["per_rank"] and 3 * e["p"] == e["unsharded"]


def test_toy_optimizer_floats_per_rank(orc):
    """"ZeRO and FSDP sharding", Code: each rank keeps 3p/n = 750 optimizer floats, not 3p = 3000."""
    p = orc.Plan(W.toy_units(), 4)
    assert 3 * p.H == 750 and 3 * p.P_pad == 3000


# ----------------------------------------------------------------------------
# Checkpoint resharding ("ZeRO and FSDP sharding", Implementation notes: a
# sharded checkpoint is resharded to a different N at load time).  Pinned to
# the composition of the two (already pinned) layout maps through the unit
# positions, and to round trips.
def _reshard_by_maps(orc, sizes, n_from, n_to, src, a_from=1, a_to=1):
    pf, pt = orc.Plan(sizes, n_from, a_from), orc.Plan(sizes, n_to, a_to)
    full_from = np.zeros(pf.P_pad, src.dtype)
    full_from[pf.shard_map().ravel()] = src.ravel()
    full_to = np.zeros(pt.P_pad, src.dtype)
    for u, s in enumerate(sizes):
        full_to[pt.F[u]:pt.F[u] + s] = full_from[pf.F[u]:pf.F[u] + s]  # real positions keep their unit position
    return full_to[pt.shard_map()]


@pytest.mark.parametrize("n_from,n_to", [(1, 4), (4, 1), (8, 16), (16, 8), (3, 5), (7, 2), (4, 4)])
def test_reshard_is_the_composition_of_the_layouts(orc, n_from, n_to):
    rng = np.random.default_rng(n_from * 31 + n_to)
    sizes = [int(x) for x in rng.integers(0, 90, 9)] + [1, 257]
    src = rng.normal(0, 1, (n_from, orc.Plan(sizes, n_from).H)).astype(np.float32)
    got = orc.reshard(sizes, n_from, n_to, src)
    assert np.array_equal(got.view(np.uint32), _reshard_by_maps(orc, sizes, n_from, n_to, src).view(np.uint32))
    bits = rng.integers(0, 1 << 16, src.shape, dtype=np.int64).astype(np.uint16)
    assert np.array_equal(orc.reshard(sizes, n_from, n_to, bits), _reshard_by_maps(orc, sizes, n_from, n_to, bits))


@pytest.mark.parametrize("n_from,a_from,n_to,a_to", [(8, 1, 16, 8), (16, 8, 8, 1), (4, 8, 3, 1), (5, 2, 5, 1)])
def test_reshard_between_aligned_layouts(orc, n_from, a_from, n_to, a_to):
    rng = np.random.default_rng(n_from * 7 + a_from * 3 + n_to)
    sizes = [int(x) for x in rng.integers(0, 300, 9)] + [1, 257]
    src = rng.normal(0, 1, (n_from, orc.Plan(sizes, n_from, a_from).H)).astype(np.float32)
    got = orc.reshard(sizes, n_from, n_to, src, align_from=a_from, align_to=a_to)
    want = _reshard_by_maps(orc, sizes, n_from, n_to, src, a_from, a_to)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_reshard_round_trip_and_identity(orc):
    rng = np.random.default_rng(3)
    sizes = [int(x) for x in rng.integers(1, 200, 12)]
    p8 = orc.Plan(sizes, 8)
    src = rng.normal(0, 1, (8, p8.H)).astype(np.float32)
    pad = p8.pad_mask()[p8.shard_map()].astype(bool)
    src[pad] = 0.0  # padding holds 0, as the update keeps it
    for n2 in (1, 3, 5, 16):
        back = orc.reshard(sizes, n2, 8, orc.reshard(sizes, 8, n2, src))
        assert np.array_equal(back.view(np.uint32), src.view(np.uint32)), n2
    assert np.array_equal(orc.reshard(sizes, 8, 8, src).view(np.uint32), src.view(np.uint32))
