"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Floating point is bit-exact (the method's arithmetic is fixed operation by
operation; nothing is fused), integers exact.  The one quantity that is not
bit-exact by construction is the binary64 sum of squares for the clip: the GPU
adds per-segment partials in its own fixed order, so S is checked to a relative
1e-12 of the oracle's exact sum, and the clip coefficient derived from it must
then match bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import workloads as W
from oracle import oracle as O
from parity import SampledCase, SmallCase, aligned_copy, f32bits, host_bits, hp_for, oracle_grad_rows

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


# ------------------------------------------------------------------ the pages' toy
def test_toy_zero2_bit_exact_every_step():
    """"ZeRO and FSDP sharding", Code: N=4, P=1000, w0=0, fp32 grads w - target_r,
    50 steps, fp32 gather; every step equals unsharded AdamW bit for bit."""
    dev = torch.device("cuda")
    N, P, steps = 4, 1000, 50
    plan = Z.ZeroPlan(W.toy_units(), N, dev)
    targets = W.toy_targets(N, P, device=dev)
    full = torch.zeros(P, dtype=torch.float32, device=dev)  # the gathered weights every rank sees
    master, m, v = (Z.rank_buffers(N, plan.H, torch.float32, dev, zero=True) for _ in range(3))
    grads = Z.rank_buffers(N, P, torch.float32, dev)
    t_np = targets.cpu().numpy()
    w_o = np.zeros(P, np.float32)
    m_o = np.zeros(P, np.float32)
    v_o = np.zeros(P, np.float32)
    for t in range(1, steps + 1):
        torch.sub(full.unsqueeze(0), targets, out=grads)  # each rank's local gradient of 1/2|w - target|^2
        hp, ohp = hp_for(t)
        Z.zero_step(plan, grads, master, m, v, hp, full=full)
        g_o = [w_o - t_np[r] for r in range(N)]
        O.adamw(g_o, O.F32, w_o, m_o, v_o, ohp, pdtype=O.F32)
        assert np.array_equal(host_bits(full), f32bits(w_o)), f"step {t}"
    ref = O.toy_unsharded(t_np, np.zeros(P, np.float32), steps, O.hparams())
    assert np.array_equal(host_bits(full), f32bits(ref))
    assert np.array_equal(host_bits(master).ravel(), f32bits(ref))


@pytest.mark.slow
def test_toy_3000_steps_bit_exact():
    """The pages' toy run for 3000 steps (well past the bias corrections' transient and
    into Adam's oscillation band around the mean target): the GPU state equals the
    oracle's after every 100th step, and at the end."""
    dev = torch.device("cuda")
    N, P = 4, 1000
    plan = Z.ZeroPlan(W.toy_units(), N, dev)
    targets = W.toy_targets(N, P, device=dev)
    full = torch.zeros(P, dtype=torch.float32, device=dev)
    master, m, v = (Z.rank_buffers(N, plan.H, torch.float32, dev, zero=True) for _ in range(3))
    grads = Z.rank_buffers(N, P, torch.float32, dev)
    t_np = targets.cpu().numpy()
    w_o, m_o, v_o = (np.zeros(P, np.float32) for _ in range(3))
    for t in range(1, 3001):
        torch.sub(full.unsqueeze(0), targets, out=grads)
        hp, ohp = hp_for(t)
        Z.zero_step(plan, grads, master, m, v, hp, full=full)
        O.adamw([w_o - t_np[r] for r in range(N)], O.F32, w_o, m_o, v_o, ohp, pdtype=O.F32)
        if t % 100 == 0:
            assert np.array_equal(host_bits(full), f32bits(w_o)), f"step {t}"
    assert np.array_equal(host_bits(master).ravel(), f32bits(w_o))
    assert np.array_equal(host_bits(m).ravel(), f32bits(m_o)) and np.array_equal(host_bits(v).ravel(), f32bits(v_o))


def test_random_layouts_and_hyperparameters():
    """A seeded fuzz over unit lists, rank counts, gradient and param dtypes, the alignment
    option and the AdamW constants (b1, b2, eps, lr, weight decay including 0, step numbers
    up to 10^6, clipping on and off): every case bit-exact against the oracle."""
    rng = np.random.default_rng(2026)
    for case in range(24):
        U = int(rng.integers(1, 9))
        sizes = [int(x) for x in rng.integers(0, 40000, U)]
        N = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 24]))
        gd, pd = (W.BF16 if rng.random() < 0.7 else W.F32), (W.BF16 if rng.random() < 0.7 else W.F32)
        align = int(rng.choice([1, 1, 2, 8]))
        c = SmallCase(sizes, N, gd, pd, seed=case, align=align, grad_sigma=float(10 ** rng.uniform(-5, 0)))
        over = dict(lr=float(10 ** rng.uniform(-5, -1)), b1=float(rng.choice([0.0, 0.5, 0.9, 0.99])),
                    b2=float(rng.choice([0.9, 0.95, 0.999, 0.9999])), eps=float(10 ** rng.uniform(-12, -4)),
                    wd=float(rng.choice([0.0, 0.01, 0.1, 0.5])))
        t0 = int(rng.choice([1, 2, 10, 1000, 10 ** 6]))
        for k in range(2):
            max_norm = float(10 ** rng.uniform(-3, 1)) if rng.random() < 0.4 else 0.0
            c.gpu_step(t0 + k, max_norm=max_norm, **over)
            assert c.oracle_step(t0 + k, max_norm=max_norm, **over) == O.OK, case
            if max_norm > 0:
                assert abs(c.sq.item() - c.S_o) <= S_RTOL * c.S_o, case
            c.assert_state_equal()
            c.assert_full_equal()
            c.assert_pshard_equal()


# ------------------------------------------------------------------ small configs, every element
SMALL = [
    # (sizes, N, gdtype, pdtype)
    ([1000], 4, W.F32, W.F32),
    ([5, 0, 13, 1, 64, 257, 4099], 4, W.BF16, W.BF16),
    ([70001, 3, 65537, 12345], 8, W.BF16, W.BF16),
    ([70001, 3, 65537, 12345], 8, W.F32, W.BF16),
    ([99991, 7, 40000], 3, W.BF16, W.F32),
    ([33, 100003, 2, 77777], 5, W.F32, W.F32),
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 131071], 16, W.BF16, W.BF16),
    ([131072 * 3 + 5], 2, W.BF16, W.BF16),
    ([4097, 1], 1, W.BF16, W.BF16),
    ([300, 17, 9000], 64, W.BF16, W.BF16),
    ([1000, 2000], 12, W.BF16, W.BF16),
]


@pytest.mark.parametrize("sizes,N,gd,pd", SMALL)
def test_fused_step_bit_exact(sizes, N, gd, pd):
    c = SmallCase(sizes, N, gd, pd, seed=len(sizes) * 31 + N)
    for t in (1, 2, 3):
        c.gpu_step(t)
        assert c.oracle_step(t) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()


def test_finewrap_shaped_small_bit_exact():
    """Many small units at N=16 (log-uniform sizes): most slices have gradient
    positions misaligned relative to their shard positions."""
    sizes = W.finewrap_units(n_units=400, lo_log2=0, hi_log2=13, seed=4)
    c = SmallCase(sizes, 16, W.BF16, W.BF16, seed=4)
    segs = Z.zero_plan_segments(c.plan.handle)
    assert sum(1 for s in segs if (s[0] - s[1]) % 8) > len(segs) // 2
    for t in (1, 2):
        c.gpu_step(t)
        assert c.oracle_step(t) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()


@pytest.mark.parametrize("align,gd", [(8, W.BF16), (4, W.F32), (2, W.BF16)])
def test_aligned_plan_steps_bit_exact(align, gd):
    """Plans with the alignment option (every unit padded to a multiple of N*align):
    fine-wrap-shaped units at N=16, where an unaligned plan puts most slices at
    shifted offsets; here no segment is shifted, and the fused and the clipped
    steps equal the oracle's on the same aligned layout."""
    sizes = W.finewrap_units(n_units=300, lo_log2=0, hi_log2=14, seed=5)
    c = SmallCase(sizes, 16, gd, W.BF16, seed=align, align=align, grad_sigma=1e-2, outlier_frac=1e-3,
                  outlier_scale=100.0)
    segs = Z.zero_plan_segments(c.plan.handle)
    assert all((g - s_) % align == 0 for (g, s_, _, _, _, _) in segs)
    for t, max_norm in ((1, 0.0), (2, 1e-3), (3, 0.0)):
        c.gpu_step(t, max_norm=max_norm)
        assert c.oracle_step(t, max_norm=max_norm) == O.OK
        if max_norm > 0:
            assert abs(c.sq.item() - c.S_o) <= S_RTOL * c.S_o
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()


@pytest.mark.parametrize("n_from,a_from,n_to,a_to", [(16, 1, 16, 8), (16, 8, 8, 1), (8, 8, 3, 2)])
def test_reshard_between_alignments_bit_exact(n_from, a_from, n_to, a_to):
    sizes = W.finewrap_units(n_units=30, lo_log2=0, hi_log2=15, seed=n_from + a_from) + [1, 70001]
    dev = torch.device("cuda", torch.cuda.current_device())
    pf, pt = Z.ZeroPlan(sizes, n_from, dev, align=a_from), Z.ZeroPlan(sizes, n_to, dev, align=a_to)
    g = torch.Generator().manual_seed(n_from * 3 + a_to)
    src_h = torch.randn(n_from, pf.H, generator=g)
    src = aligned_copy(src_h, dev)
    dst = Z.rank_buffers(n_to, pt.H, torch.float32, dev)
    dst.fill_(7.0)
    Z.zero_reshard(pf, pt, src, dst)
    want = O.reshard(sizes, n_from, n_to, host_bits(src_h), align_from=a_from, align_to=a_to)
    assert np.array_equal(host_bits(dst), want)


def test_empty_and_degenerate_plans():
    for sizes, N in (([], 4), ([0, 0], 3), ([1], 64), ([0, 1, 0], 2)):
        c = SmallCase(sizes, N, W.BF16, W.BF16)
        c.gpu_step(1)
        assert c.oracle_step(1) == O.OK
        if c.plan.P_pad:
            c.assert_state_equal()
            c.assert_full_equal()
        torch.cuda.synchronize()


def test_pads_stay_zero():
    sizes = [13, 1, 250]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, state="zero")
    pad = torch.from_numpy(c.pad.astype(bool))
    mp = torch.from_numpy(c.map)
    padpos = pad[mp].to(c.device)  # [N, H] mask of padding shard positions
    c.master[padpos] = 0.0
    c.reload()
    for t in (1, 2, 3, 4):
        c.gpu_step(t)
        assert c.oracle_step(t) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()
    assert torch.all(c.master[padpos] == 0) and torch.all(c.m[padpos] == 0) and torch.all(c.v[padpos] == 0)
    assert torch.all(c.full[torch.from_numpy(c.pad.astype(bool)).to(c.device)].float() == 0)


def test_per_unit_launches_equal_one_multi_unit_launch():
    sizes = [5000, 3, 70000, 1, 40961]
    a = SmallCase(sizes, 8, W.BF16, W.BF16, seed=3)
    b = SmallCase(sizes, 8, W.BF16, W.BF16, seed=3)
    a.gpu_step(1)
    for u in range(len(sizes)):
        b.gpu_step(1, unit=u)
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.full, b.full), (a.pshard, b.pshard)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))
    assert b.oracle_step(1) == O.OK  # the per-unit side against the oracle too
    b.assert_state_equal()
    b.assert_full_equal()
    b.assert_pshard_equal()


def test_unit_steps_marshalled_once_bit_exact():
    """UnitSteps (arguments marshalled once, one direct zero_step call per unit, in any
    order) against the oracle over three steps, with param shards and the full buffer;
    a clipped step is refused."""
    sizes = W.finewrap_units(n_units=40, lo_log2=0, hi_log2=16, seed=9) + [0, 70001]
    c = SmallCase(sizes, 16, W.BF16, W.BF16, seed=41)
    us = Z.UnitSteps(c.plan, c.grads, c.master, c.m, c.v, full=c.full, pshard=c.pshard)
    order = list(range(len(sizes)))[::-1]
    for t in (1, 2, 3):
        hp, _ = hp_for(t)
        us.step(hp, units=order if t == 2 else None)
        assert c.oracle_step(t) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()
    with pytest.raises(ValueError):
        us.step(hp_for(4, 1.0)[0])


def test_per_unit_steps_replay_from_a_cuda_graph():
    """The per-unit launches of one step captured in a CUDA graph (the library
    makes no synchronising or allocating call on that path) and replayed: the
    result equals the oracle's step bit for bit; a second replay repeats the
    captured step (the step counter is a launch argument)."""
    sizes = [5000, 3, 70000, 1, 40961]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=33)
    c.gpu_step(1, unit=0)  # first launch of each kernel outside the capture
    c.reload()
    hp, _ = hp_for(2)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
        for u in range(len(sizes)):
            Z.zero_step(c.plan, c.grads, c.master, c.m, c.v, hp, full=c.full, pshard=c.pshard, unit=u)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert c.oracle_step(2) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()


def host_bits_t(x):
    return torch.from_numpy(host_bits(x).astype(np.int64))


# ------------------------------------------------------------------ unit-local gradient buffers
def _unit_rows(c, u):
    F, S = c.plan.F[u], c.plan.S[u]
    rows = Z.rank_buffers(c.N, S, c.grads.dtype, c.device)
    rows.copy_(c.grads[:, F:F + S])
    return rows


@pytest.mark.parametrize("N,gd", [(16, W.BF16), (3, W.F32), (8, W.BF16)])
def test_unit_local_step_equals_full_step(N, gd):
    """zero_step_unit over every unit, each from a buffer holding only that unit's
    gradients (unit offsets F_u of any alignment), equals one zero_step bit for bit."""
    sizes = W.finewrap_units(n_units=40, lo_log2=0, hi_log2=16, seed=9)
    a = SmallCase(sizes, N, gd, W.BF16, seed=N)
    b = SmallCase(sizes, N, gd, W.BF16, seed=N)
    a.gpu_step(1)
    hp, _ = hp_for(1)
    for u in range(len(sizes)):
        Z.zero_step_unit(b.plan, u, _unit_rows(b, u), b.master, b.m, b.v, hp, full=b.full, pshard=b.pshard)
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.full, b.full), (a.pshard, b.pshard)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))
    assert b.oracle_step(1) == O.OK
    b.assert_state_equal()
    b.assert_full_equal()
    b.assert_pshard_equal()


def test_unit_local_reduce_scatter_equals_full():
    """zero_reduce_scatter_unit over every unit from unit-local buffers: the oracle's
    averaged gradient times the coefficient (one binary32 multiply) at every shard
    position, and the same bits as the all-units zero_reduce_scatter."""
    sizes = W.finewrap_units(n_units=40, lo_log2=0, hi_log2=16, seed=10)
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=10)
    coef = np.float32(0.3711)
    for u in range(len(sizes)):
        Z.zero_reduce_scatter_unit(c.plan, u, _unit_rows(c, u), c.gshard, coef=float(coef))
    want = (O.avg_grad(c.g_o, O.BF16, c.pad) * coef).astype(np.float32)
    assert np.array_equal(host_bits(c.gshard), f32bits(want)[c.map])
    ref = host_bits(c.gshard).copy()
    c.gshard.zero_()
    Z.zero_reduce_scatter(c.plan, c.grads, c.gshard, coef=float(coef))
    assert np.array_equal(host_bits(c.gshard), ref)


def test_host_streamed_step_equals_device_step():
    """Gradients in pinned host memory, streamed unit by unit with overlapped copies:
    the same bits as the device-resident step, and the params come back to the host."""
    from fsdp_sharded_optimizer_step_gb300.streaming import HostStreamedStep
    sizes = [70001, 3, 65537, 12345, 0, 9, 1 << 20]
    a = SmallCase(sizes, 8, W.BF16, W.BF16, seed=21)
    b = SmallCase(sizes, 8, W.BF16, W.BF16, seed=21)
    host_grads = torch.empty(8, b.plan.P_pad, dtype=torch.bfloat16, pin_memory=True)
    host_grads.copy_(b.grads.cpu())
    host_full = torch.zeros(b.plan.P_pad, dtype=torch.bfloat16, pin_memory=True)
    streamer = HostStreamedStep(b.plan, torch.bfloat16)
    for t in (1, 2):
        a.gpu_step(t, pshard=False)
        hp, _ = hp_for(t)
        streamer.step(host_grads, b.master, b.m, b.v, hp, b.full, host_full=host_full)
        torch.cuda.synchronize()
        assert b.oracle_step(t) == O.OK  # the streamed side against the oracle, every step
        b.assert_state_equal()
        b.assert_full_equal()
        assert np.array_equal(host_bits(host_full), b.out_o)
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.full, b.full)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))
    assert np.array_equal(host_bits(host_full), host_bits(a.full))


@pytest.mark.parametrize("max_norm", [1e-3, 1e6])
def test_host_streamed_clipped_step_equals_device_clipped_step(max_norm):
    """The clipped step with the gradients streamed in from pinned host memory
    (per-unit norm passes, device total, per-unit shard updates with the params
    copied back) gives the bits of the clipped zero_step, S included, and the
    oracle's step; a coefficient below 1 and one that is exactly 1."""
    from fsdp_sharded_optimizer_step_gb300 import binding as B
    from fsdp_sharded_optimizer_step_gb300.streaming import HostStreamedStep
    sizes = [70001, 3, 65537, 12345, 0, 9, 1 << 20]
    a = SmallCase(sizes, 8, W.BF16, W.BF16, seed=23, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0)
    b = SmallCase(sizes, 8, W.BF16, W.BF16, seed=23, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0)
    host_grads = torch.empty(8, b.plan.P_pad, dtype=torch.bfloat16, pin_memory=True)
    host_grads.copy_(b.grads.cpu())
    host_full = torch.zeros(b.plan.P_pad, dtype=torch.bfloat16, pin_memory=True)
    streamer = HostStreamedStep(b.plan, torch.bfloat16)
    for t in (1, 2):
        a.gpu_step(t, max_norm=max_norm, pshard=False)
        hp, _ = hp_for(t, max_norm)
        streamer.step_clipped(host_grads, b.gshard, b.master, b.m, b.v, hp, b.full, host_full=host_full,
                              sqnorm_out=b.sq)
        torch.cuda.synchronize()
        assert b.sq.item() == a.sq.item()  # same segments, same fixed order
        assert b.oracle_step(t, max_norm=max_norm) == O.OK
        b.assert_state_equal()
        b.assert_full_equal()
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.full, b.full), (a.gshard, b.gshard)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))
    assert np.array_equal(host_bits(host_full), host_bits(a.full))
    assert Z.zero_plan_check(b.plan) == B.ZERO_OK
    # a non-finite norm: the streamed step leaves the state alone and says so
    host_grads[3, 17] = float("inf")
    before = [x.clone() for x in (b.master, b.m, b.v, b.full)]
    hp, _ = hp_for(3, max_norm)
    streamer.step_clipped(host_grads, b.gshard, b.master, b.m, b.v, hp, b.full, sqnorm_out=b.sq)
    assert Z.zero_plan_check(b.plan) == B.ZERO_ENONFINITE
    assert math.isinf(b.sq.item())
    for x, y in zip(before, (b.master, b.m, b.v, b.full)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))


# ------------------------------------------------------------------ unfused parts
def test_parts_compose_to_the_fused_step():
    """reduce-scatter -> AdamW on the shard -> all-gather == the fused step, bit for bit;
    each part also against the oracle."""
    sizes = [70001, 3, 65537, 12345, 0, 9]
    fused = SmallCase(sizes, 8, W.BF16, W.BF16, seed=9)
    parts = SmallCase(sizes, 8, W.BF16, W.BF16, seed=9)
    fused.gpu_step(1)
    hp, _ = hp_for(1)
    Z.zero_reduce_scatter(parts.plan, parts.grads, parts.gshard)
    avg = O.avg_grad(parts.g_o, O.BF16, parts.pad)
    assert np.array_equal(host_bits(parts.gshard), f32bits(avg)[parts.map])
    Z.zero_adamw_shard_step(parts.plan, parts.gshard, parts.master, parts.m, parts.v, hp, pshard=parts.pshard)
    Z.zero_all_gather_bf16(parts.plan, parts.pshard, parts.full)
    for x, y in ((fused.master, parts.master), (fused.m, parts.m), (fused.v, parts.v), (fused.full, parts.full),
                 (fused.pshard, parts.pshard)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))
    assert parts.oracle_step(1) == O.OK
    parts.assert_state_equal()
    parts.assert_pshard_equal()
    parts.assert_full_equal()


def test_reduce_scatter_with_coefficient():
    sizes = [1000, 77, 33333]
    c = SmallCase(sizes, 4, W.F32, W.BF16, seed=2)
    coef = np.float32(0.3711)
    Z.zero_reduce_scatter(c.plan, c.grads, c.gshard, coef=float(coef))
    avg = O.avg_grad(c.g_o, O.F32, c.pad)
    want = (avg * coef).astype(np.float32)  # one binary32 multiply per element
    assert np.array_equal(host_bits(c.gshard), f32bits(want)[c.map])


def test_all_gather_per_unit_and_fp32():
    sizes = [1001, 5, 20000, 3]
    for pd in (W.BF16, W.F32):
        c = SmallCase(sizes, 4, W.BF16, pd, seed=5)
        g = torch.Generator().manual_seed(1)
        src = aligned_copy(torch.randn(4, c.plan.H, generator=g).to(c.pshard.dtype), c.device)
        ref = src.cpu().numpy() if pd == W.F32 else None
        full = torch.zeros_like(c.full)
        for u in range(len(sizes)):
            Z.zero_all_gather(c.plan, src, full, unit=u)
        want = np.zeros(c.plan.P_pad, dtype=np.uint32 if pd == W.F32 else np.uint16)
        want[c.map.ravel()] = host_bits(src).ravel()
        assert np.array_equal(host_bits(full), want)
        if ref is not None:
            assert np.array_equal(full.cpu().numpy()[c.map], ref)


@pytest.mark.parametrize("N,pd", [(16, W.BF16), (16, W.F32), (3, W.BF16), (5, W.F32)])
def test_all_gather_misaligned_slices_integer_exact(N, pd):
    """Fine-wrap-shaped units: most slices land in the full buffer at positions
    aligned differently from their shard positions (the shifted-vector path).
    The gather of all units, per-unit gathers, and per-unit gathers into
    unit-sized buffers all place every shard element at its full position."""
    sizes = W.finewrap_units(n_units=200, lo_log2=0, hi_log2=15, seed=7)
    c = SmallCase(sizes, N, W.BF16, pd, seed=N)
    segs = Z.zero_plan_segments(c.plan.handle)
    assert sum(1 for sg in segs if (sg[0] - sg[1]) % 8) > len(segs) // 2
    g = torch.Generator().manual_seed(N)
    src = aligned_copy(torch.randn(N, c.plan.H, generator=g).to(c.pshard.dtype), c.device)
    want = np.zeros(c.plan.P_pad, dtype=np.uint32 if pd == W.F32 else np.uint16)
    want[c.map.ravel()] = host_bits(src).ravel()
    full = torch.zeros_like(c.full)
    Z.zero_all_gather(c.plan, src, full)
    assert np.array_equal(host_bits(full), want)
    full.zero_()
    for u in range(len(sizes)):
        Z.zero_all_gather(c.plan, src, full, unit=u)
    assert np.array_equal(host_bits(full), want)
    for u in range(len(sizes)):
        F, S = c.plan.F[u], c.plan.S[u]
        if S == 0:
            continue
        buf = torch.zeros(S + 8, dtype=c.full.dtype, device=c.device)
        Z.zero_all_gather_unit(c.plan, u, src, buf[:S])
        assert np.array_equal(host_bits(buf[:S]), want[F:F + S]), u
        assert not host_bits(buf[S:]).any()  # nothing written past the unit


def test_grad_sqnorm_close_to_exact_and_deterministic():
    sizes = [70001, 3, 65537, 12345, 9]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=11, outlier_frac=1e-3, outlier_scale=100.0)
    out = torch.zeros(1, dtype=torch.float64, device=c.device)
    Z.zero_grad_sqnorm(c.plan, c.grads, out)
    S1 = out.item()
    Z.zero_grad_sqnorm(c.plan, c.grads, out)
    assert out.item() == S1  # fixed reduction order: same bits every run
    S_o = O.sqnorm(c.g_o, O.BF16, c.pad)
    assert abs(S1 - S_o) <= S_RTOL * S_o


# ------------------------------------------------------------------ clipping
@pytest.mark.parametrize("max_norm", [1e-4, 1.0, 1e6])
def test_clipped_step_bit_exact(max_norm):
    sizes = [70001, 3, 65537, 12345, 9]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=12, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0)
    for t in (1, 2):
        c.gpu_step(t, max_norm=max_norm)
        assert c.oracle_step(t, max_norm=max_norm) == O.OK
        S_gpu = c.sq.item()
        assert abs(S_gpu - c.S_o) <= S_RTOL * c.S_o
        assert O.clip_coef(S_gpu, max_norm) == O.clip_coef(c.S_o, max_norm)
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()
        avg = O.avg_grad(c.g_o, O.BF16, c.pad)
        assert np.array_equal(host_bits(c.gshard), f32bits(avg)[c.map])  # the unclipped averaged shard


def test_clipped_step_skipped_when_norm_not_finite():
    sizes = [1000, 3000]
    c = SmallCase(sizes, 4, W.BF16, W.BF16, seed=13)
    c.grads[2, 17] = float("inf")
    before = [x.clone() for x in (c.master, c.m, c.v, c.full, c.pshard)]
    c.gpu_step(1, max_norm=1.0)
    assert math.isinf(c.sq.item())
    for x, y in zip(before, (c.master, c.m, c.v, c.full, c.pshard)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))
    from fsdp_sharded_optimizer_step_gb300 import binding as B
    assert Z.zero_plan_check(c.plan) == B.ZERO_ENONFINITE  # reported on the host, then cleared
    assert Z.zero_plan_check(c.plan) == B.ZERO_OK
    c.g_o = oracle_grad_rows(c.grads)
    assert c.oracle_step(1, max_norm=1.0) == O.ENONFINITE


def test_nan_and_inf_without_clip_follow_ieee():
    sizes = [4096]
    c = SmallCase(sizes, 4, W.F32, W.BF16, seed=14)
    c.grads[1, 5] = float("nan")
    c.grads[0, 9] = float("inf")
    c.grads[3, 9] = float("-inf")
    c.grads[2, 11] = float("inf")
    c.g_o = oracle_grad_rows(c.grads)
    c.gpu_step(1)
    assert c.oracle_step(1) == O.OK
    c.assert_state_equal()
    c.assert_full_equal()


def test_runs_on_a_side_stream():
    c = SmallCase([70001, 5], 8, W.BF16, W.BF16, seed=15)
    s = torch.cuda.Stream()
    hp, _ = hp_for(1)
    with torch.cuda.stream(s):
        Z.zero_step(c.plan, c.grads, c.master, c.m, c.v, hp, full=c.full, stream=s)
    s.synchronize()
    assert c.oracle_step(1) == O.OK
    c.assert_full_equal()


# ------------------------------------------------------------------ full-size workloads (sampled)
@pytest.mark.slow
def test_gpt2l_zero1_full_size_sampled():
    c = SampledCase("gpt2l", n_random=300000, extra_units=(37,))
    for t in (1, 2):
        c.gpu_step(t)
        out = c.oracle_step(t)
        c.assert_sample_equal(out)


@pytest.mark.slow
def test_1p3b_zero2_clip_full_size():
    c = SampledCase("1p3b_clip", n_random=200000)
    S = c.oracle_sqnorm()
    coef = O.clip_coef(S, 1.0)
    assert coef < 1.0  # the outliers make the norm exceed 1: clipping is active
    for t in (1, 2):
        c.gpu_step(t)
        S_gpu = c.sq.item()
        assert abs(S_gpu - S) <= S_RTOL * S
        assert O.clip_coef(S_gpu, 1.0) == coef
        out = c.oracle_step(t, coef=coef)
        c.assert_sample_equal(out)


@pytest.mark.slow
def test_finewrap_full_size_sampled():
    c = SampledCase("finewrap", n_random=200000, extra_units=(0, 1, 2, 4095))
    c.gpu_step(1)
    c.assert_sample_equal(c.oracle_step(1))


@pytest.mark.slow
def test_finewrap600_one_launch_then_per_unit_full_size_sampled():
    """The fine-wrap law at the stated ~600M total (4096 units in [2^10, 2^20), N=16):
    step 1 as the one multi-unit launch, step 2 as one launch per unit, each against the
    oracle on 200k random positions, every slice boundary and four whole units."""
    c = SampledCase("finewrap600", n_random=200000, extra_units=(0, 1, 2048, 4095))
    c.gpu_step(1)
    c.assert_sample_equal(c.oracle_step(1))
    hp, _ = hp_for(2)
    for u in range(c.plan.n_units):
        Z.zero_step(c.plan, c.grads, c.master, c.m, c.v, hp, full=c.full, unit=u)
    c.assert_sample_equal(c.oracle_step(2))
    assert Z.zero_plan_check(c.plan) == 0


@pytest.mark.slow
def test_4b_zero3_full_size_sampled():
    """4B ZeRO-3 (128 GB resident): 300k random positions, every slice boundary, and
    every element of four whole 113M-parameter block units (first, second, a middle
    one and the last block before the embedding)."""
    c = SampledCase("4b_z3", n_random=300000, extra_units=(0, 1, 16, 31))
    c.gpu_step(1)
    c.assert_sample_equal(c.oracle_step(1))


def _index_width_positions(o):
    """Full positions on either side of 2^31 and 2^32, the last one, and for every rank the
    full positions whose shard positions sit on either side of 2^31."""
    P, N = o.P_pad, o.N
    pos = [p for b in (2 ** 31, 2 ** 32) for p in (b - 2, b - 1, b, b + 1) if 0 <= p < P] + [P - 1]
    hoff = np.concatenate([[0], np.cumsum(o.h)])
    for s in (2 ** 31 - 2, 2 ** 31 - 1, 2 ** 31, 2 ** 31 + 1):
        u = int(np.searchsorted(hoff, s, side="right")) - 1
        if u < len(o.sizes) and s < hoff[u + 1]:
            pos += [int(o.F[u]) + r * int(o.h[u]) + int(s - hoff[u]) for r in range(N)]
    return pos


@pytest.mark.slow
def test_beyond_2p32_positions_clipped_then_zero3():
    """Index width: 4,311,744,532 padded positions at N=2, two units longer than 2^31,
    so full positions pass 2^32 and shard positions (8.6 GB into each fp32 rank buffer)
    pass 2^31.  Step 1 is the clipped step (S over every position within the norm
    bound of the oracle's exact sum, the coefficient bit-exact), step 2 the unclipped
    step with bf16 param shards and per-unit gathers (ZeRO-3); both against the oracle
    on 200k random positions, every slice boundary and the positions either side of
    2^31 and 2^32 in both index spaces."""
    o = O.Plan(W.CONFIGS["beyond_2p32"]["units"](), 2)
    extra = _index_width_positions(o)
    assert max(extra) >= 2 ** 32 and len(extra) >= 9 + 4 * 2
    c = SampledCase("beyond_2p32", n_random=200000, stage=3, extra_pos=extra)
    assert c.plan.P_pad > 2 ** 32 and c.plan.H > 2 ** 31
    S = c.oracle_sqnorm()
    coef = O.clip_coef(S, 1.0)
    assert coef < 1.0
    hp, _ = hp_for(1, 1.0)
    Z.zero_step(c.plan, c.grads, c.master, c.m, c.v, hp, full=c.full, pshard=c.pshard, gshard_ws=c.gshard,
                sqnorm_out=c.sq)
    S_gpu = c.sq.item()
    assert abs(S_gpu - S) <= S_RTOL * S
    assert O.clip_coef(S_gpu, 1.0) == coef
    c.assert_sample_equal(c.oracle_step(1, coef=coef))
    assert Z.zero_plan_check(c.plan) == 0
    c.full.zero_()
    c.clip = False
    hp, _ = hp_for(2)
    Z.zero_step(c.plan, c.grads, c.master, c.m, c.v, hp, full=None, pshard=c.pshard)
    for u in range(c.plan.n_units):  # ZeRO-3: the param shards gathered unit by unit
        Z.zero_all_gather_bf16(c.plan, c.pshard, c.full, unit=u)
    c.assert_sample_equal(c.oracle_step(2))
    assert Z.zero_plan_check(c.plan) == 0


# ------------------------------------------------------------------ checkpoint resharding
@pytest.mark.parametrize("n_from,n_to", [(8, 16), (16, 8), (8, 3), (3, 8), (5, 5)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_reshard_bit_exact(n_from, n_to, dtype):
    sizes = W.finewrap_units(n_units=30, lo_log2=0, hi_log2=15, seed=n_from + n_to) + [1, 3, 70001]
    dev = torch.device("cuda", torch.cuda.current_device())
    pf, pt = Z.ZeroPlan(sizes, n_from, dev), Z.ZeroPlan(sizes, n_to, dev)
    g = torch.Generator().manual_seed(n_from * 7 + n_to)
    src_h = torch.randn(n_from, pf.H, generator=g).to(dtype)
    src = aligned_copy(src_h, dev)
    dst = Z.rank_buffers(n_to, pt.H, dtype, dev)
    dst.fill_(7.0)  # every position must be written, padding included
    Z.zero_reshard(pf, pt, src, dst)
    want = O.reshard(sizes, n_from, n_to, host_bits(src_h))
    assert np.array_equal(host_bits(dst), want)


def test_sharded_checkpoint_reshard_then_continue(tmp_path):
    """Save the state of an N=8 run rank by rank, load it into N=4 (resharded on the
    GPU), continue with N=4 gradients: bit-exact against the oracle, which keeps
    the state unsharded and only ever changes how it is sliced."""
    from fsdp_sharded_optimizer_step_gb300 import checkpoint
    sizes = [70001, 3, 65537, 12345, 9, 1 << 16]
    c8 = SmallCase(sizes, 8, W.BF16, W.BF16, seed=31)
    c8.gpu_step(1)
    assert c8.oracle_step(1) == O.OK
    checkpoint.save(str(tmp_path), c8.plan, {"master": c8.master, "m": c8.m, "v": c8.v}, step=1)
    c4 = SmallCase(sizes, 4, W.BF16, W.BF16, seed=32)
    state, step = checkpoint.load(str(tmp_path), c4.plan)
    assert step == 1
    for name, gpu8 in (("master", c8.master), ("m", c8.m), ("v", c8.v)):
        want = O.reshard(sizes, 8, 4, host_bits(gpu8))
        assert np.array_equal(host_bits(state[name]), want), name
        getattr(c4, name).copy_(state[name])
    # the oracle continues from the same unsharded state (its padding for N=4 holds 0)
    for arr, src in ((c4.w_o, c4.master), (c4.m_o, c4.m), (c4.v_o, c4.v)):
        arr[c4.map.ravel()] = src.cpu().numpy().ravel()
    c4.gpu_step(2)
    assert c4.oracle_step(2) == O.OK
    c4.assert_state_equal()
    c4.assert_full_equal()


def test_checkpoint_between_alignments(tmp_path):
    """Save from an aligned N=16 plan, load into an unaligned N=8 plan: the reshard at
    load time maps between the two layouts exactly as the oracle does."""
    from fsdp_sharded_optimizer_step_gb300 import checkpoint
    sizes = W.finewrap_units(n_units=25, lo_log2=4, hi_log2=16, seed=8)
    dev = torch.device("cuda", torch.cuda.current_device())
    pa, pb = Z.ZeroPlan(sizes, 16, dev, align=8), Z.ZeroPlan(sizes, 8, dev)
    g = torch.Generator().manual_seed(88)
    arrays = {"master": aligned_copy(torch.randn(16, pa.H, generator=g), dev)}
    checkpoint.save(str(tmp_path), pa, arrays, step=2)
    state, step = checkpoint.load(str(tmp_path), pb)
    assert step == 2
    want = O.reshard(sizes, 16, 8, host_bits(arrays["master"]), align_from=8, align_to=1)
    assert np.array_equal(host_bits(state["master"]), want)


def test_checkpoint_load_on_a_side_stream(tmp_path):
    """load() given a stream that is not the current one: seven arrays (fp32 and bf16)
    resharded 8 -> 3 on that stream, back to back, each equal to the oracle's remap
    (one array's staging buffers are not reused by the next array's copies while its
    reshard still reads them)."""
    from fsdp_sharded_optimizer_step_gb300 import checkpoint
    sizes = W.finewrap_units(n_units=30, lo_log2=8, hi_log2=20, seed=5) + [1 << 20]
    dev = torch.device("cuda", torch.cuda.current_device())
    p8, p3 = Z.ZeroPlan(sizes, 8, dev), Z.ZeroPlan(sizes, 3, dev)
    g = torch.Generator().manual_seed(77)
    arrays = {f"a{k}": aligned_copy(torch.randn(8, p8.H, generator=g), dev) for k in range(6)}
    arrays["p16"] = aligned_copy(torch.randn(8, p8.H, generator=g).to(torch.bfloat16), dev)
    checkpoint.save(str(tmp_path), p8, arrays, step=5)
    side = torch.cuda.Stream()
    state, step = checkpoint.load(str(tmp_path), p3, stream=side)
    assert step == 5 and list(state) == list(arrays)
    for name, a in arrays.items():
        assert np.array_equal(host_bits(state[name]), O.reshard(sizes, 8, 3, host_bits(a))), name


# ------------------------------------------------------------------ ZeRO-3 gather with prefetch, ZeRO-2 buckets
def test_zero3_unit_gather_with_prefetch_gives_every_unit_its_params():
    from fsdp_sharded_optimizer_step_gb300.zero3 import UnitGatherer
    sizes = [70001, 3, 65537, 12345, 9, 1 << 16, 777]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=41)
    c.gpu_step(1)  # fills the param shards (and the full buffer)
    assert c.oracle_step(1) == O.OK
    c.assert_pshard_equal()  # the gatherer's input, checked against the oracle
    full = c.out_o  # every unit's params in the oracle's full layout
    seen = {}
    gatherer = UnitGatherer(c.plan, c.pshard)
    for prefetch in (True, False):
        def compute(u, params_u):
            seen[(prefetch, u)] = params_u.clone()
        gatherer.run(compute, order=reversed(range(len(sizes))), prefetch=prefetch)
        torch.cuda.synchronize()
        for u in range(len(sizes)):
            F, S = c.plan.F[u], c.plan.S[u]
            assert np.array_equal(host_bits(seen[(prefetch, u)]), full[F:F + S]), (prefetch, u)


def test_zero2_bucketed_reduce_scatter_then_shard_update_equals_fused_step():
    """Gradients produced unit by unit (reverse order, like a backward pass) into one
    reused bucket, reduce-scattered at once, then the shard update: the same bits
    as the fused step that reads N full gradient buffers."""
    from fsdp_sharded_optimizer_step_gb300.zero3 import BucketedReduceScatter
    sizes = W.finewrap_units(n_units=25, lo_log2=2, hi_log2=16, seed=12)
    a = SmallCase(sizes, 8, W.BF16, W.BF16, seed=13)
    b = SmallCase(sizes, 8, W.BF16, W.BF16, seed=13)
    a.gpu_step(1, pshard=False)
    buckets = BucketedReduceScatter(b.plan)
    assert buckets.bucket_bytes < b.grads.numel() * 2  # never the N full gradient buffers

    def fill(u, view):  # stands in for the backward of unit u
        view.copy_(b.grads[:, b.plan.F[u]:b.plan.F[u] + b.plan.S[u]])

    for u in reversed(range(len(sizes))):
        buckets.reduce(u, fill, b.gshard)
    avg = O.avg_grad(b.g_o, O.BF16, b.pad)
    assert np.array_equal(host_bits(b.gshard), f32bits(avg)[b.map])
    hp, _ = hp_for(1)
    Z.zero_adamw_shard_step(b.plan, b.gshard, b.master, b.m, b.v, hp, full=b.full)
    assert b.oracle_step(1) == O.OK
    b.assert_state_equal()
    b.assert_full_equal()
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.full, b.full)):
        assert torch.equal(host_bits_t(x), host_bits_t(y))


@pytest.mark.parametrize("bucket_elems,max_norm", [(1, 0.0), (150000, 0.0), (None, 0.0), (150000, 1e-3), (1, 1e6)])
def test_zero2_bucketed_step_bit_exact(bucket_elems, max_norm):
    """The ZeRO-2 step through one reusable gradient bucket, filled in backward order:
    one unit per bucket, several units per bucket, everything in one bucket; with
    clipping the buckets' norm passes, then the coefficient and the shard update.
    Every step equals the oracle's, S included."""
    from fsdp_sharded_optimizer_step_gb300.zero3 import BucketedStep
    sizes = W.finewrap_units(n_units=25, lo_log2=2, hi_log2=16, seed=12) + [70001, 0, 3]
    c = SmallCase(sizes, 8, W.BF16, W.BF16, seed=14, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0)
    bs = BucketedStep(c.plan, bucket_elems=bucket_elems)
    assert bs.bucket_bytes < c.grads.shape[0] * c.grads.stride(0) * 2 or bucket_elems is None
    if bucket_elems == 1:
        assert len(bs.buckets) == sum(1 for s in c.plan.S if s)
    seen = []

    def fill(u0, u1, view):  # stands in for the backward of units [u0, u1)
        seen.append((u0, u1))
        F0 = c.plan.F[u0]
        view.copy_(c.grads[:, F0:F0 + view.shape[1]])

    for t in (1, 2):
        hp, _ = hp_for(t, max_norm)
        bs.step(fill, c.master, c.m, c.v, hp, full=c.full, pshard=c.pshard, gshard=c.gshard, sqnorm_out=c.sq)
        torch.cuda.synchronize()
        assert c.oracle_step(t, max_norm=max_norm) == O.OK
        if max_norm > 0:
            assert abs(c.sq.item() - c.S_o) <= S_RTOL * c.S_o
            assert O.clip_coef(c.sq.item(), max_norm) == O.clip_coef(c.S_o, max_norm)
        c.assert_state_equal()
        c.assert_full_equal()
        c.assert_pshard_equal()
    covered = sorted(u for u0, u1 in seen[:len(bs.buckets)] for u in range(u0, u1))
    assert covered == [u for u in range(len(sizes)) if c.plan.S[u] or u in covered]


@pytest.mark.slow
def test_gpt2l_zero2_bucketed_full_size_sampled():
    """The bucketed ZeRO-2 step as the bench times it (GPT-2L, N=8, the default buckets,
    filled in backward order from the full gradient rows): 300k sampled positions,
    every slice boundary and one whole block unit against the oracle, two steps."""
    from fsdp_sharded_optimizer_step_gb300.zero3 import BucketedStep
    c = SampledCase("gpt2l", n_random=300000, extra_units=(20,))
    bs = BucketedStep(c.plan)
    assert len(bs.buckets) == 7 and bs.bucket_bytes < c.grads.shape[0] * c.grads.stride(0) * 2

    def fill(u0, u1, view):
        F0 = c.plan.F[u0]
        view.copy_(c.grads[:, F0:F0 + view.shape[1]])

    for t in (1, 2):
        hp, _ = hp_for(t)
        bs.step(fill, c.master, c.m, c.v, hp, full=c.full)
        torch.cuda.synchronize()
        c.assert_sample_equal(c.oracle_step(t))


# ------------------------------------------------------------------ failure detection without a GPU fault
def test_bounded_wait_runs_out_and_is_reported():
    """A pipeline stage that never fills (one tile's copies dropped in the first segment by the
    testing aid): the waiting warps give up after about two seconds instead of
    hanging, the launch ends, the device error word reports it, and the context
    still runs a correct step afterwards."""
    import time
    from fsdp_sharded_optimizer_step_gb300 import binding as B
    c = SmallCase([70001, 3000], 8, W.BF16, W.BF16, seed=51)
    assert B.zero_plan_device_errors(c.plan) == 0
    B.zero_debug_drop_copy(3)
    t0 = time.time()
    c.gpu_step(1)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert B.zero_plan_device_errors(c.plan) != 0
    assert 1.5 < elapsed < 30.0
    assert B.zero_plan_device_errors(c.plan) == 0  # read-and-clear
    B.zero_debug_drop_copy(3)  # the same, reported as a status
    c.gpu_step(2)
    assert Z.zero_plan_check(c.plan) == B.ZERO_ETIMEOUT
    assert Z.zero_plan_check(c.plan) == B.ZERO_OK
    # the aborted launches left the same plan usable: its segment schedule starts clean, and a
    # step from whatever state they left is exact again (the fused step and the clipped one)
    for t, max_norm in ((3, 0.0), (4, 1e-3)):
        c.reload()
        c.gpu_step(t, max_norm=max_norm)
        assert c.oracle_step(t, max_norm=max_norm) == O.OK
        c.assert_state_equal()
        c.assert_full_equal()
        assert Z.zero_plan_check(c.plan) == B.ZERO_OK
    d = SmallCase([70001, 3000], 8, W.BF16, W.BF16, seed=52)
    d.gpu_step(1)
    assert d.oracle_step(1) == O.OK
    d.assert_state_equal()
    d.assert_full_equal()
    assert B.zero_plan_device_errors(d.plan) == 0
