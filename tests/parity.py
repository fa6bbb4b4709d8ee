"""Harness for comparing the CUDA path with the CPU oracle on the same seeded inputs.

Small cases compare every element bit for bit: the oracle runs unsharded over
the full padded buffer, and the GPU's per-rank shard buffers are mapped to full
positions with the oracle's own layout (shard_map / locate).  Full-size cases
compare a seeded sample of positions the oracle can follow one by one (the
update is element-wise, so each sampled position depends only on its own
gradients, state and the global clip coefficient).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import workloads as W
from oracle import oracle as O

TOY_HP = dict(lr=0.01, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)

TDT = {W.BF16: torch.bfloat16, W.F32: torch.float32}
ODT = {W.BF16: O.BF16, W.F32: O.F32}


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a tensor on the host: uint16 for bf16, uint32 for fp32."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    raise TypeError(t.dtype)


def oracle_grad_rows(t: torch.Tensor):
    """[N, L] gradient tensor -> list of numpy rows in the oracle's format (bf16 bits or fp32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return [r for r in t.view(torch.int16).numpy().view(np.uint16)]
    return [r for r in t.numpy()]


def f32bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _isnan_bits(b):
    if b.dtype == np.uint16:
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x7FFFFF) != 0)


def mismatch(got, want):
    """Positions where two bit arrays differ, counting any two NaNs as equal
    (IEEE 754 leaves NaN payloads and the default NaN to the platform)."""
    got = np.asarray(got)
    want = np.asarray(want)
    bad = got != want
    if bad.any():
        bad &= ~(_isnan_bits(got) & _isnan_bits(want))
    return bad


def aligned_copy(src: torch.Tensor, device, guards=None):
    """Copy a [N, L] tensor into rank buffers whose rows are 16-byte aligned
    (guarded ones when a guard list is given)."""
    if guards is None:
        out = Z.rank_buffers(src.shape[0], src.shape[1], src.dtype, device)
    else:
        out = guarded_buffers(guards, src.shape[1], src.dtype, device, rows=src.shape[0])
    out.copy_(src)
    return out


# Guard bands: every device buffer of a small case sits inside a larger allocation
# whose other bytes hold a canary pattern; a kernel that writes outside the
# elements it was given (before a row, past its end, into the row padding)
# changes a canary, which check_guards finds after the step.
CANARY = 0xA5
GUARD_BYTES = 64


def guarded_buffers(guards: list, length, dtype, device, rows=None, zero=False):
    """A [rows, length] view (or a 1-D view of `length` when rows is None) whose rows
    start 16-byte aligned, inside an allocation with GUARD_BYTES of canary before
    and after every row; (allocation, canary mask) is appended to `guards`."""
    esz = torch.empty((), dtype=dtype).element_size()
    g = GUARD_BYTES // esz
    per16 = 16 // esz
    stride = max((length + per16 - 1) // per16 * per16, 1)
    n = 1 if rows is None else rows
    backing = torch.empty(n, g + stride + g, dtype=dtype, device=device)
    backing.view(torch.uint8).fill_(CANARY)
    mask = torch.ones(n, (g + stride + g) * esz, dtype=torch.bool, device=device)
    mask[:, g * esz:(g + length) * esz] = False
    guards.append((backing, mask))
    view = backing[:, g:g + length]
    if zero:
        view.zero_()
    return view[0] if rows is None else view


def check_guards(guards: list):
    """Every canary byte of every guarded allocation is intact."""
    for k, (backing, mask) in enumerate(guards):
        u8 = backing.view(torch.uint8)
        bad = int((u8[mask] != CANARY).sum().item())
        assert bad == 0, f"guarded buffer {k}: {bad} canary bytes overwritten"


def hp_for(t, max_norm=0.0, **over):
    d = dict(TOY_HP)
    d.update(over)
    return Z.AdamW(t=t, max_norm=max_norm, **d), O.hparams(t=t, max_norm=max_norm, **d)


class SmallCase:
    """A config small enough that the oracle follows every element."""

    def __init__(self, sizes, N, gdtype=W.BF16, pdtype=W.BF16, seed=0, device="cuda", grad_sigma=1e-3,
                 state="random", outlier_frac=0.0, outlier_scale=1.0, align=1):
        self.sizes, self.N, self.gdtype, self.pdtype = list(sizes), N, gdtype, pdtype
        self.device = torch.device(device)
        self.plan = Z.ZeroPlan(self.sizes, N, self.device, align=align)
        self.o = O.Plan(self.sizes, N, align)
        assert self.plan.P_pad == self.o.P_pad and self.plan.H == self.o.H
        P, H = self.plan.P_pad, self.plan.H
        self.guards = []  # every device buffer below sits between canary bands
        self.grads = aligned_copy(W.make_grads(N, P, gdtype, sigma=grad_sigma, device="cpu", seed=seed + 1,
                                               outlier_frac=outlier_frac, outlier_scale=outlier_scale), self.device,
                                  self.guards)
        master, m, v = W.make_state(N, H, device="cpu", seed=seed + 1000)
        if state == "random":  # non-zero moments exercise every term of the update
            g = torch.Generator().manual_seed(seed + 7)
            m = torch.randn(N, H, generator=g) * 1e-3
            v = torch.rand(N, H, generator=g) * 1e-6
        self.master, self.m, self.v = (aligned_copy(x, self.device, self.guards) for x in (master, m, v))
        self.full = guarded_buffers(self.guards, P, TDT[pdtype], self.device, zero=True)
        self.pshard = guarded_buffers(self.guards, H, TDT[pdtype], self.device, rows=N, zero=True)
        self.gshard = guarded_buffers(self.guards, H, torch.float32, self.device, rows=N, zero=True)
        self.sq = torch.zeros(1, dtype=torch.float64, device=self.device)
        # oracle state in the full (unsharded) layout
        self.map = self.o.shard_map()  # [N, H] -> full position
        self.pad = self.o.pad_mask()
        self.w_o = np.zeros(P, np.float32)
        self.m_o = np.zeros(P, np.float32)
        self.v_o = np.zeros(P, np.float32)
        for name, src in (("w_o", self.master), ("m_o", self.m), ("v_o", self.v)):
            arr = getattr(self, name)
            arr[self.map.ravel()] = src.cpu().numpy().ravel()
        self.g_o = oracle_grad_rows(self.grads)
        self.out_o = None
        self.S_o = None

    def reload(self):
        """Re-read the oracle's copies after a test overwrote the GPU inputs."""
        for name, src in (("w_o", self.master), ("m_o", self.m), ("v_o", self.v)):
            getattr(self, name)[self.map.ravel()] = src.cpu().numpy().ravel()
        self.g_o = oracle_grad_rows(self.grads)

    # -------------------------------------------------------------- runs
    def gpu_step(self, t, max_norm=0.0, full=True, pshard=True, unit=-1, **over):
        hp, _ = hp_for(t, max_norm, **over)
        Z.zero_step(self.plan, self.grads, self.master, self.m, self.v, hp,
                    full=self.full if full else None, pshard=self.pshard if pshard else None,
                    gshard_ws=self.gshard if max_norm > 0 else None, sqnorm_out=self.sq if max_norm > 0 else None,
                    unit=unit)
        self.check_guards()

    def check_guards(self):
        check_guards(self.guards)

    def oracle_step(self, t, max_norm=0.0, **over):
        _, ohp = hp_for(t, max_norm, **over)
        rc, out, S = O.step(self.g_o, ODT[self.gdtype], self.w_o, self.m_o, self.v_o, ohp, pdtype=ODT[self.pdtype],
                            pad=self.pad)
        if rc == O.OK:
            self.out_o = out
        self.S_o = S
        return rc

    # -------------------------------------------------------------- comparisons
    def assert_state_equal(self):
        self.check_guards()
        mp = self.map
        for name, gpu, ora in (("master", self.master, self.w_o), ("m", self.m, self.m_o), ("v", self.v, self.v_o)):
            got = host_bits(gpu)
            want = f32bits(ora)[mp]
            bad = np.argwhere(mismatch(got, want))
            assert bad.size == 0, f"{name}: {bad.shape[0]} of {got.size} differ, first at rank/pos {bad[0]}"

    def assert_full_equal(self):
        self.check_guards()
        got = host_bits(self.full)
        want = self.out_o if self.pdtype == W.BF16 else f32bits(self.out_o)
        bad = np.flatnonzero(mismatch(got, want))
        assert bad.size == 0, f"full: {bad.size} of {got.size} differ, first at {bad[0]}"

    def assert_pshard_equal(self):
        got = host_bits(self.pshard)
        want = (self.out_o if self.pdtype == W.BF16 else f32bits(self.out_o))[self.map]
        bad = np.argwhere(mismatch(got, want))
        assert bad.size == 0, f"pshard: {bad.shape[0]} differ, first at {bad[0]}"


def segment_edges(plan) -> np.ndarray:
    """The first and last full position of every segment of the library's two launch
    tables (where a CTA's work, a head, a tail or a tile begins or ends)."""
    out = []
    for segs in (Z.zero_plan_segments(plan.handle), Z.zero_plan_local_segments(plan.handle)):
        if segs:
            a = np.array(segs, dtype=np.int64)
            out += [a[:, 0], a[:, 0] + a[:, 2] - 1]
    return np.unique(np.concatenate(out)) if out else np.zeros(0, np.int64)


def sample_positions(plan_o: "O.Plan", n_random, seed, extra_units=(), extra_pos=()):
    """Seeded random full positions plus every unit's first/last element, every
    slice boundary and ragged tail, the given extra positions, and all positions
    of the units in extra_units."""
    rng = np.random.default_rng(seed)
    P = plan_o.P_pad
    pos = [rng.integers(0, P, n_random), np.asarray(extra_pos, np.int64)]
    N = plan_o.N
    for u in range(len(plan_o.sizes)):
        F, S, h = int(plan_o.F[u]), int(plan_o.S[u]), int(plan_o.h[u])
        if S == 0:
            continue
        b = [F, F + S - 1, F + int(plan_o.sizes[u]) - 1 if plan_o.sizes[u] > 0 else F]
        for r in range(N):
            b += [F + r * h, F + r * h + h - 1, min(F + r * h + 7, F + S - 1)]
        pos.append(np.array(b, np.int64))
    pos = np.unique(np.concatenate(pos))
    pos = pos[(pos >= 0) & (pos < P)]
    # whole units: contiguous ranges, added without a global sort (hundreds of millions of positions)
    ranges = [(int(plan_o.F[u]), int(plan_o.F[u] + plan_o.S[u])) for u in sorted(set(extra_units))]
    if not ranges:
        return pos
    inside = np.zeros(pos.size, bool)
    for a, b in ranges:
        inside |= (pos >= a) & (pos < b)
    return np.concatenate([pos[~inside]] + [np.arange(a, b, dtype=np.int64) for a, b in ranges])


class SampledCase:
    """A full-size config: GPU runs everything, the oracle follows a sample."""

    def __init__(self, name, n_random=200000, seed=0, device="cuda", extra_units=(), stage=None, extra_pos=()):
        cfg = W.CONFIGS[name]
        self.cfg = cfg
        self.sizes = cfg["units"]()
        self.N = N = cfg["N"]
        self.gdtype, self.pdtype = cfg["gdtype"], cfg["pdtype"]
        self.device = torch.device(device)
        self.plan = Z.ZeroPlan(self.sizes, N, self.device)
        self.o = O.Plan(self.sizes, N)
        P, H = self.plan.P_pad, self.plan.H
        self.grads = W.make_grads(N, P, self.gdtype, sigma=cfg.get("grad_sigma", 1e-3), device=self.device, seed=1,
                                  outlier_frac=cfg.get("outlier_frac", 0.0),
                                  outlier_scale=cfg.get("outlier_scale", 1.0),
                                  out=Z.rank_buffers(N, P, TDT[self.gdtype], self.device))
        self.master, self.m, self.v = W.make_state(
            N, H, sigma=cfg.get("master_sigma", 0.02), device=self.device,
            out=tuple(Z.rank_buffers(N, H, torch.float32, self.device) for _ in range(3)))
        self.stage = cfg["stage"] if stage is None else stage
        self.full = torch.zeros(P, dtype=TDT[self.pdtype], device=self.device)
        self.pshard = Z.rank_buffers(N, H, TDT[self.pdtype], self.device, zero=True) if self.stage == 3 else None
        self.clip = cfg.get("max_norm", 0.0) > 0
        self.gshard = Z.rank_buffers(N, H, torch.float32, self.device) if self.clip else None
        self.sq = torch.zeros(1, dtype=torch.float64, device=self.device)
        # the sample
        extra_pos = np.concatenate([np.asarray(extra_pos, np.int64), segment_edges(self.plan)])
        self.pos = sample_positions(self.o, n_random, seed, extra_units, extra_pos)
        self.rank, self.spos, self.padflag = self.o.locate(self.pos)
        pos_t = torch.from_numpy(self.pos).to(self.device)
        self.g_s = oracle_grad_rows(self.grads.index_select(1, pos_t))
        self.ridx = torch.from_numpy(self.rank.astype(np.int64)).to(self.device)
        self.sidx = torch.from_numpy(self.spos).to(self.device)
        self.w_s = self.master[self.ridx, self.sidx].cpu().numpy().copy()
        self.m_s = self.m[self.ridx, self.sidx].cpu().numpy().copy()
        self.v_s = self.v[self.ridx, self.sidx].cpu().numpy().copy()
        self.pos_t = pos_t
        self.S_o = None

    def oracle_sqnorm(self, chunk=1 << 25, threads=8):
        """Exact S over every position, streamed through host memory in chunks on a
        few host threads, each with its own exact accumulator; exact sums merge
        exactly, so the split does not change the result."""
        pad = self.o.pad_mask()
        P = self.plan.P_pad

        def part(a):
            acc = O.SqAcc()
            b = min(P, a + chunk)
            acc.add_avg_grad(oracle_grad_rows(self.grads[:, a:b]), ODT[self.gdtype], pad[a:b])
            return acc

        total = O.SqAcc()
        with ThreadPoolExecutor(max(1, min(threads, os.cpu_count() or 1))) as ex:
            for acc in ex.map(part, range(0, P, chunk)):
                total.merge(acc)
        self.S_o = total.result()
        return self.S_o

    def gpu_step(self, t):
        hp, _ = hp_for(t, self.cfg.get("max_norm", 0.0))
        if self.stage == 3:
            Z.zero_step(self.plan, self.grads, self.master, self.m, self.v, hp, full=None, pshard=self.pshard)
            for u in range(self.plan.n_units):  # ZeRO-3: gather unit by unit
                Z.zero_all_gather_bf16(self.plan, self.pshard, self.full, unit=u)
        else:
            Z.zero_step(self.plan, self.grads, self.master, self.m, self.v, hp, full=self.full,
                        gshard_ws=self.gshard, sqnorm_out=self.sq if self.clip else None)

    def oracle_step(self, t, coef=1.0):
        _, ohp = hp_for(t, 0.0)
        return O.adamw(self.g_s, ODT[self.gdtype], self.w_s, self.m_s, self.v_s, ohp, pdtype=ODT[self.pdtype],
                       pad=self.padflag, clip=self.clip, coef=coef)

    def assert_sample_equal(self, out_o):
        for name, gpu, ora in (("master", self.master, self.w_s), ("m", self.m, self.m_s), ("v", self.v, self.v_s)):
            got = host_bits(gpu[self.ridx, self.sidx])
            bad = np.flatnonzero(mismatch(got, f32bits(ora)))
            assert bad.size == 0, f"{name}: {bad.size} of {got.size} sampled differ, first at {self.pos[bad[0]]}"
        got = host_bits(self.full[self.pos_t])
        want = out_o if self.pdtype == W.BF16 else f32bits(out_o)
        bad = np.flatnonzero(mismatch(got, want))
        assert bad.size == 0, f"full: {bad.size} sampled differ, first at {self.pos[bad[0]]}"
        if self.pshard is not None:
            got = host_bits(self.pshard[self.ridx, self.sidx])
            bad = np.flatnonzero(mismatch(got, want))
            assert bad.size == 0, f"pshard: {bad.size} sampled differ"
