"""ZeRO-Offload's host update (zero_offload_adamw) against the CPU oracle, on
the host alone (no GPU): bit for bit on master, m, v and the params.

The host update is product code (csrc/zero_offload.cpp) that shares nothing
with the oracle.  Its input is the averaged gradient shard; here that shard is
the oracle's own rank-ordered average of N seeded gradient rows, mapped to the
shard layout with the oracle's map, and the expected state is the oracle's
unsharded step over the same rows.  Edge values (subnormals, values near
overflow, inf and NaN gradients) go through a single fp32 gradient row, whose
average is the row itself.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import binding as B
from fsdp_sharded_optimizer_step_gb300 import workloads as W
from oracle import oracle as O

HP = dict(lr=0.01, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)


@pytest.fixture(scope="module", autouse=True)
def built():
    from fsdp_sharded_optimizer_step_gb300 import build
    build.build()
    Z.lib()


def _bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _nan(b):
    if b.dtype == np.uint16:
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x7FFFFF) != 0)


def _assert_same(got, want, what):
    g, w = _bits(got), _bits(want)
    bad = (g != w) & ~(_nan(g) & _nan(w))  # any two NaNs count as equal
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} differ, first at {np.flatnonzero(bad.ravel())[0]}"


class HostCase:
    """State in the shard layout on the host, and its unsharded copy for the oracle."""

    def __init__(self, sizes, N, pdtype=W.BF16, seed=0, n_threads=0, batch_min=0, wide=False):
        self.plan = Z.ZeroPlan(sizes, N)  # host-only plan: the host update needs no device
        self.o = O.Plan(sizes, N)
        self.N, self.pdtype = N, pdtype
        P, H = self.plan.P_pad, self.plan.H
        self.map = self.o.shard_map()
        self.pad = self.o.pad_mask()
        rng = np.random.default_rng(seed)
        if wide:  # one fp32 gradient row spanning the whole range, state likewise
            self.rows = [W.wide_range_f32(P, seed + 1)]
            self.gd = O.F32
            w = W.wide_range_f32(P, seed + 2)
            m = W.wide_range_f32(P, seed + 3)
            v = W.wide_range_f32(P, seed + 4, nonneg=True)
        else:
            g = W.make_grads(N, P, W.BF16, sigma=1e-2, seed=seed + 1, outlier_frac=1e-3, outlier_scale=100.0)
            self.rows = [r for r in g.view(torch.int16).numpy().view(np.uint16)]
            self.gd = O.BF16
            w = (rng.standard_normal(P) * 0.02).astype(np.float32)
            m = (rng.standard_normal(P) * 1e-3).astype(np.float32)
            v = (rng.random(P) * 1e-6).astype(np.float32)
        pad = None if wide else self.pad
        avg = O.avg_grad(self.rows, self.gd, pad)
        self.w_o, self.m_o, self.v_o = w.copy(), m.copy(), v.copy()
        mp = self.map
        self.gshard = torch.from_numpy(np.ascontiguousarray(avg[mp]))
        self.master = torch.from_numpy(np.ascontiguousarray(w[mp]))
        self.m = torch.from_numpy(np.ascontiguousarray(m[mp]))
        self.v = torch.from_numpy(np.ascontiguousarray(v[mp]))
        tdt = torch.bfloat16 if pdtype == W.BF16 else torch.float32
        self.full = torch.zeros(P, dtype=tdt)
        self.pshard = torch.zeros(N, H, dtype=tdt)
        self.eng = B.OffloadEngine(self.plan, n_threads=n_threads, batch_min=batch_min)
        self.opad = pad

    def host_step(self, t, max_norm=0.0, sqnorm=0.0, unit=-1, pshard=True):
        hp = Z.AdamW(t=t, max_norm=max_norm, **HP)
        return Z.zero_offload_adamw(self.eng, self.gshard, self.master, self.m, self.v, hp, full_h=self.full,
                                    pshard_h=self.pshard if pshard else None, sqnorm=sqnorm, unit=unit)

    def oracle_step(self, t, coef=None):
        ohp = O.hparams(t=t, **HP)
        pd = O.BF16 if self.pdtype == W.BF16 else O.F32
        return O.adamw(self.rows, self.gd, self.w_o, self.m_o, self.v_o, ohp, pdtype=pd, pad=self.opad,
                       clip=coef is not None, coef=1.0 if coef is None else coef)

    def assert_equal(self, out_o):
        mp = self.map
        for name, got, want in (("master", self.master, self.w_o), ("m", self.m, self.m_o), ("v", self.v, self.v_o)):
            _assert_same(got.numpy(), want[mp], name)
        full = self.full.view(torch.int16).numpy().view(np.uint16) if self.pdtype == W.BF16 else self.full.numpy()
        _assert_same(full, out_o, "full")
        ps = (self.pshard.view(torch.int16).numpy().view(np.uint16) if self.pdtype == W.BF16
              else self.pshard.numpy())
        _assert_same(ps, out_o[mp], "pshard")


CASES = [
    ([1000], 4, W.F32, 1),
    ([5, 0, 13, 1, 64, 257, 4099], 4, W.BF16, 3),
    ([70001, 3, 65537, 12345], 8, W.BF16, 0),
    ([99991, 7, 40000], 3, W.F32, 2),
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 131071], 16, W.BF16, 5),
    ([300, 17, 9000], 64, W.BF16, 8),
    ([], 4, W.BF16, 2),
]


@pytest.mark.parametrize("sizes,N,pd,threads", CASES)
def test_host_update_bit_exact(sizes, N, pd, threads):
    c = HostCase(sizes, N, pd, seed=N + len(sizes), n_threads=threads)
    for t in (1, 2, 3):
        assert c.host_step(t) == B.ZERO_OK
        c.assert_equal(c.oracle_step(t))


def test_host_update_per_unit_equals_all_units():
    sizes = W.finewrap_units(n_units=60, lo_log2=0, hi_log2=17, seed=3)
    c = HostCase(sizes, 16, W.BF16, seed=4, n_threads=4)
    for u in range(len(sizes)):
        assert c.host_step(1, unit=u) == B.ZERO_OK
    c.assert_equal(c.oracle_step(1))


@pytest.mark.parametrize("max_norm", [1e-3, 1.0, 1e6])
def test_host_update_clipped(max_norm):
    """The clip coefficient comes from S inside the library (binary64, rounded once):
    the oracle's S in, the oracle's clipped step out."""
    c = HostCase([70001, 3, 65537, 12345], 8, W.BF16, seed=11, n_threads=5)
    S = O.sqnorm(c.rows, c.gd, c.pad)
    coef = O.clip_coef(S, max_norm)
    assert (coef < 1.0) == (max_norm < 1e3)
    for t in (1, 2):
        assert c.host_step(t, max_norm=max_norm, sqnorm=S) == B.ZERO_OK
        c.assert_equal(c.oracle_step(t, coef=coef))


def test_host_update_non_finite_norm_skips():
    c = HostCase([4096, 77], 4, W.BF16, seed=12)
    before = [x.clone() for x in (c.master, c.m, c.v, c.full, c.pshard)]
    for S in (float("inf"), float("nan")):
        assert c.host_step(1, max_norm=1.0, sqnorm=S) == B.ZERO_ENONFINITE
    for x, y in zip(before, (c.master, c.m, c.v, c.full, c.pshard)):
        assert torch.equal(x.view(torch.uint8) if x.dtype != torch.float32 else x.view(torch.int32),
                           y.view(torch.uint8) if y.dtype != torch.float32 else y.view(torch.int32))


@pytest.mark.parametrize("pd", [W.BF16, W.F32])
def test_host_update_edge_values(pd):
    """Gradients, weights and moments across the whole binary32 range (a third
    subnormal, a third with any exponent, inf and NaN gradients included)."""
    c = HostCase([30011, 5, 20000], 4, pd, seed=13, n_threads=3, wide=True)
    g = c.rows[0]
    g[[3, 100, 2000]] = [np.inf, -np.inf, np.nan]
    c.gshard.copy_(torch.from_numpy(np.ascontiguousarray(g[c.map])))
    for t in (1, 2):
        assert c.host_step(t) == B.ZERO_OK
        c.assert_equal(c.oracle_step(t))


def test_host_update_thread_counts_agree():
    sizes = W.finewrap_units(n_units=40, lo_log2=4, hi_log2=18, seed=6)
    outs = []
    for threads in (1, 2, 7):
        c = HostCase(sizes, 8, W.BF16, seed=7, n_threads=threads)
        assert c.host_step(1) == B.ZERO_OK
        outs.append((c.master.clone(), c.full.clone()))
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b.view(torch.int16), outs[0][1].view(torch.int16))


def test_host_update_rejects_bad_arguments():
    c = HostCase([1000, 24], 4, W.BF16, seed=14)
    hp = Z.AdamW(t=0, **HP)
    with pytest.raises(B.ZeroError):
        Z.zero_offload_adamw(c.eng, c.gshard, c.master, c.m, c.v, hp, full_h=c.full)
    hp = Z.AdamW(t=1, **HP)
    with pytest.raises(B.ZeroError):
        Z.zero_offload_adamw(c.eng, c.gshard, c.master, c.m, c.v, hp, full_h=c.full, unit=2)
    with pytest.raises(ValueError):
        Z.zero_offload_adamw(c.eng, c.gshard[:, :10], c.master, c.m, c.v, hp, full_h=c.full)
    L = Z.lib()
    assert L.zero_offload_create(None, 0, 0, None) == B.ZERO_EINVAL


def test_engine_reports_threads_and_batches():
    """Batches are consecutive units of at least batch_min padded elements, a zero-sized unit
    joining the batch before it; the engine reports them and its thread count."""
    plan = Z.ZeroPlan([100, 0, 300, 50, 0, 0, 700, 10], 2)  # padded sizes 100, 0, 300, 50, 0, 0, 700, 10
    # batch_min 1: {100, 0} {300} {50, 0, 0} {700} {10}; 150: {100, 0, 300} {50, 0, 0, 700} {10};
    # 400: the same three; 10^6: everything in one
    for batch_min, want in ((1, 5), (150, 3), (400, 3), (10 ** 6, 1)):
        eng = B.OffloadEngine(plan, n_threads=3, batch_min=batch_min)
        assert Z.zero_offload_info(eng) == (3, want), batch_min
    assert Z.zero_offload_info(B.OffloadEngine(Z.ZeroPlan([], 4)))[1] == 0
