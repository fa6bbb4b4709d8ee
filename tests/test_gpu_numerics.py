"""GPU numerics at the edges of binary32: every bf16 cast input, subnormals and
values near overflow, and the sum of squares of tiny gradients.

The CUDA path runs through the C ABI and is compared with the CPU oracle:
floating point bit for bit (any two NaNs count as equal: IEEE 754 leaves the
payload of a NaN produced by arithmetic to the platform), the clip's binary64
sum of squares within a relative 1e-12 of the oracle's exact sum.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import workloads as W
from oracle import oracle as O
from parity import SmallCase, host_bits, mismatch

pytestmark = pytest.mark.gpu

S_RTOL = 1e-12


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_optimizer_step_gb300 import build
    build.build()
    Z.lib()


@pytest.fixture(autouse=True)
def release_memory():
    yield
    import gc
    gc.collect()
    torch.cuda.empty_cache()


def test_bf16_cast_every_bit_pattern_through_the_step():
    """"ZeRO and FSDP sharding", How it works: the updated fp32 shard is cast to
    bf16.  All 2^32 binary32 patterns are the master weights of an identity
    step (lr = 0, zero gradients and moments, so w*1 - 0/(0/bc2 + eps) = w
    exactly), and the step's bf16 output is compared with the oracle's cast of
    the same pattern; the master weights must come back unchanged."""
    dev = torch.device("cuda")
    ch = 1 << 28
    plan = Z.ZeroPlan([ch], 1, dev)
    grads = Z.rank_buffers(1, ch, torch.bfloat16, dev, zero=True)
    master, m, v = (Z.rank_buffers(1, ch, torch.float32, dev, zero=True) for _ in range(3))
    full = torch.empty(ch, dtype=torch.bfloat16, device=dev)
    hp = Z.AdamW(lr=0.0, wd=0.0, t=1)
    base = np.arange(ch, dtype=np.uint32)
    sub = 1 << 24
    with ThreadPoolExecutor(os.cpu_count() or 1) as ex:
        for c in range((1 << 32) // ch):
            b = base + np.uint32(c * ch)
            x = b.view(np.float32)
            master[0].copy_(torch.from_numpy(x))
            Z.zero_step(plan, grads, master, m, v, hp, full=full)
            want = np.concatenate(list(ex.map(lambda k: O.bf16_rne_array(x[k * sub:(k + 1) * sub]),
                                              range(ch // sub))))
            bad = np.flatnonzero(mismatch(host_bits(full), want))
            assert bad.size == 0, f"cast: {bad.size} differ, first input {int(b[bad[0]]):#010x}"
            bad = np.flatnonzero(mismatch(host_bits(master[0]), b))
            assert bad.size == 0, f"identity step moved {int(b[bad[0]]):#010x}"


WIDE = [
    # (sizes, N, gdtype, pdtype)
    ([70001, 3, 65537], 8, W.F32, W.BF16),
    ([99991, 7, 4000], 3, W.F32, W.F32),
    ([70001, 12345], 8, W.BF16, W.BF16),
    ([5000, 33, 40000], 5, W.BF16, W.F32),
]


@pytest.mark.parametrize("sizes,N,gd,pd", WIDE)
def test_subnormal_and_extreme_values_bit_exact(sizes, N, gd, pd):
    """Gradients, master weights and moments drawn over the whole finite
    binary32 range (a third subnormal, a third with any exponent): the GPU must
    neither flush subnormals nor contract operations, and overflow must give
    the same inf/NaN as the oracle."""
    seed = sum(sizes) + N
    c = SmallCase(sizes, N, gd, pd, seed=seed)
    P, H = c.plan.P_pad, c.plan.H
    c.grads.copy_(torch.from_numpy(W.wide_range_f32((N, P), seed)))
    c.master.copy_(torch.from_numpy(W.wide_range_f32((N, H), seed + 1, sigma=0.02)))
    c.m.copy_(torch.from_numpy(W.wide_range_f32((N, H), seed + 2)))
    c.v.copy_(torch.from_numpy(W.wide_range_f32((N, H), seed + 3, nonneg=True, sigma=1e-6)))
    c.reload()
    for t in (1, 2, 3):
        c.gpu_step(t)
        assert c.oracle_step(t) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()


@pytest.mark.parametrize("lo,hi", [(-62, -45), (-149, -126), (-55, -50), (40, 70), (-80, 100)])
def test_clipped_step_with_tiny_gradients(lo, hi):
    """Gradients whose squares are far below 1 (down to subnormal gradients), or
    far above it (|g| past 2^56, where the binary32 pair accumulation hands over
    to binary64), or both in one buffer: the sum of squares stays within 1e-12 of
    the exact sum, the clip coefficient and the whole update are bit-exact.
    max_norm is half the norm, so the coefficient is about one half."""
    sizes = [70001, 3, 65537, 12345]
    N = 8
    c = SmallCase(sizes, N, W.F32, W.BF16, seed=lo * 7 + hi)
    rng = np.random.default_rng(-lo if lo < 0 else 1000 + lo)
    mag = np.exp2(rng.uniform(lo, hi, (N, c.plan.P_pad)))
    g = (mag * rng.choice([-1.0, 1.0], mag.shape)).astype(np.float32)
    c.grads.copy_(torch.from_numpy(g))
    c.reload()
    S_exact = O.sqnorm(c.g_o, O.F32, c.pad)
    norm = float(np.sqrt(S_exact))
    max_norm = 0.5 * (norm + 1e-6)  # coefficient about one half
    for t in (1, 2):
        c.gpu_step(t, max_norm=max_norm)
        assert c.oracle_step(t, max_norm=max_norm) == O.OK
        S_gpu = c.sq.item()
        assert abs(S_gpu - c.S_o) <= S_RTOL * c.S_o, (S_gpu, c.S_o)
        assert O.clip_coef(S_gpu, max_norm) == O.clip_coef(c.S_o, max_norm)
        assert O.clip_coef(c.S_o, max_norm) < 1.0
        c.assert_state_equal()
        c.assert_full_equal()
