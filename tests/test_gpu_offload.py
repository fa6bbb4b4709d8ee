"""ZeRO-Offload end to end on the GPU machine: the GPU reduce-scatters, the
averaged gradient shard goes down to pinned host memory, the host cores run
AdamW on the host-resident master/m/v, and the params come back to the device
(zero_offload_step).  Every step is compared with the CPU oracle bit for bit:
the host state, the params on the device and their host copy; with clipping
also S (relative 1e-12 of the oracle's exact sum) and the coefficient.
"""
import math

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import binding as B
from fsdp_sharded_optimizer_step_gb300 import workloads as W
from oracle import oracle as O
from parity import SampledCase, SmallCase, f32bits, host_bits, hp_for, mismatch, oracle_grad_rows

pytestmark = pytest.mark.gpu

S_RTOL = 1e-12


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_optimizer_step_gb300 import build
    build.build()
    Z.lib()


def _pinned_like(x):
    h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    h.copy_(x)
    return h


class Offloaded:
    """A small case whose optimizer state lives in pinned host memory."""

    def __init__(self, c: SmallCase, n_threads=0, batch_min=0):
        self.c = c
        self.master_h, self.m_h, self.v_h = (_pinned_like(x) for x in (c.master, c.m, c.v))
        self.gshard_h = torch.zeros(c.N, c.plan.H, dtype=torch.float32, pin_memory=True)
        self.full_h = torch.zeros(c.plan.P_pad, dtype=c.full.dtype, pin_memory=True)
        self.eng = B.OffloadEngine(c.plan, n_threads=n_threads, batch_min=batch_min)

    def step(self, t, max_norm=0.0, stream=None):
        hp, _ = hp_for(t, max_norm)
        rc, S = Z.zero_offload_step(self.eng, self.c.grads, self.c.gshard, self.gshard_h, self.master_h, self.m_h,
                                    self.v_h, self.full_h, hp, full_dev=self.c.full, stream=stream)
        torch.cuda.synchronize()
        return rc, S

    def assert_equal_oracle(self):
        c = self.c
        for dev_t, host_t in ((c.master, self.master_h), (c.m, self.m_h), (c.v, self.v_h)):
            dev_t.copy_(host_t)  # the host state, checked through the harness's shard map
        c.assert_state_equal()
        c.assert_full_equal()
        want = c.out_o if c.pdtype == W.BF16 else f32bits(c.out_o)
        assert not mismatch(host_bits(self.full_h), want).any()


OFFLOAD_CASES = [
    # (sizes, N, gdtype, pdtype, threads, batch_min)
    ([1000], 4, W.F32, W.F32, 2, 0),
    ([5, 0, 13, 1, 64, 257, 4099], 4, W.BF16, W.BF16, 3, 64),
    ([70001, 3, 65537, 12345], 8, W.BF16, W.BF16, 0, 0),
    ([70001, 3, 65537, 12345], 8, W.F32, W.BF16, 4, 50000),
    ([99991, 7, 40000], 3, W.BF16, W.F32, 5, 1),
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 131071], 16, W.BF16, W.BF16, 8, 1000),
    ([300, 17, 9000], 64, W.BF16, W.BF16, 2, 0),
]


@pytest.mark.parametrize("sizes,N,gd,pd,threads,batch_min", OFFLOAD_CASES)
def test_offload_step_bit_exact(sizes, N, gd, pd, threads, batch_min):
    c = SmallCase(sizes, N, gd, pd, seed=N * 3 + len(sizes))
    off = Offloaded(c, threads, batch_min)
    for t in (1, 2, 3):
        rc, _ = off.step(t)
        assert rc == B.ZERO_OK
        assert c.oracle_step(t) == O.OK
        off.assert_equal_oracle()


def test_offload_step_finewrap_shaped_on_a_side_stream():
    """Many small units at N=16 in small batches, on a stream that is not the current one."""
    sizes = W.finewrap_units(n_units=300, lo_log2=0, hi_log2=15, seed=4)
    c = SmallCase(sizes, 16, W.BF16, W.BF16, seed=17)
    off = Offloaded(c, n_threads=6, batch_min=20000)
    side = torch.cuda.Stream()
    for t in (1, 2):
        rc, _ = off.step(t, stream=side)
        assert rc == B.ZERO_OK
        assert c.oracle_step(t) == O.OK
        off.assert_equal_oracle()
    tm = Z.zero_offload_timings(off.eng)
    assert all(v >= 0 for v in tm.values())
    assert tm["device_to_params_ms"] >= tm["device_to_grads_ms"] > 0


@pytest.mark.parametrize("max_norm", [1e-3, 1e6])
def test_offload_clipped_step(max_norm):
    sizes = [70001, 3, 65537, 12345, 9]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=19, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0)
    off = Offloaded(c, n_threads=4, batch_min=30000)
    for t in (1, 2):
        rc, S = off.step(t, max_norm=max_norm)
        assert rc == B.ZERO_OK
        assert c.oracle_step(t, max_norm=max_norm) == O.OK
        assert abs(S - c.S_o) <= S_RTOL * c.S_o
        assert O.clip_coef(S, max_norm) == O.clip_coef(c.S_o, max_norm)
        off.assert_equal_oracle()
    assert Z.zero_plan_check(c.plan) == B.ZERO_OK
    # a non-finite norm: nothing is updated, the status says so (and zero_plan_check after it)
    c.grads[5, 11] = float("inf")
    before = [x.clone() for x in (off.master_h, off.m_h, off.v_h, off.full_h, c.full)]
    rc, S = off.step(3, max_norm=max_norm)
    assert rc == B.ZERO_ENONFINITE and math.isinf(S)
    for x, y in zip(before, (off.master_h, off.m_h, off.v_h, off.full_h, c.full)):
        assert np.array_equal(host_bits(x), host_bits(y))
    assert Z.zero_plan_check(c.plan) == B.ZERO_ENONFINITE
    c.g_o = oracle_grad_rows(c.grads)
    assert c.oracle_step(3, max_norm=max_norm) == O.ENONFINITE


@pytest.mark.slow
def test_gpt2l_offload_full_size_sampled():
    """The bench's offload workload (GPT-2-Large shapes, N=8, state in 9.3 GB of
    pinned host memory): one step, 300k sampled positions, every slice boundary and
    one whole block unit against the oracle."""
    c = SampledCase("gpt2l", n_random=300000, extra_units=(5,))
    N, H, P = c.N, c.plan.H, c.plan.P_pad
    master_h, m_h, v_h = (_pinned_like(x) for x in (c.master, c.m, c.v))
    del c.master, c.m, c.v
    torch.cuda.empty_cache()
    gshard_dev = Z.rank_buffers(N, H, torch.float32, c.device)
    gshard_h = torch.empty(N, H, dtype=torch.float32, pin_memory=True)
    full_h = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
    eng = B.OffloadEngine(c.plan)
    hp, _ = hp_for(1)
    rc, _ = Z.zero_offload_step(eng, c.grads, gshard_dev, gshard_h, master_h, m_h, v_h, full_h, hp, full_dev=c.full)
    torch.cuda.synchronize()
    assert rc == B.ZERO_OK
    out = c.oracle_step(1)
    ridx = torch.from_numpy(c.rank.astype(np.int64))
    sidx = torch.from_numpy(c.spos)
    for name, host_t, ora in (("master", master_h, c.w_s), ("m", m_h, c.m_s), ("v", v_h, c.v_s)):
        got = host_bits(host_t[ridx, sidx])
        assert not mismatch(got, f32bits(ora)).any(), name
    assert not mismatch(host_bits(c.full[c.pos_t]), out).any()
    assert not mismatch(host_bits(full_h[torch.from_numpy(c.pos)]), out).any()
