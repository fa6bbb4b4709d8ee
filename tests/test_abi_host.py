"""Host-side tests of the C ABI (no GPU): the library loads and exports every
declared symbol; the plan's layout and launch table are integer-exact against
the oracle; the host bias corrections match the oracle bit for bit; argument
errors are reported before anything touches a device."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import binding as B
from fsdp_sharded_optimizer_step_gb300 import build as zbuild
from fsdp_sharded_optimizer_step_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero.h")


@pytest.fixture(scope="module")
def zlib():
    zbuild.build()
    return Z.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(zlib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(zlib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", zbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (zero_[a-z0-9_]+)", out))
    assert set(names) <= exported
    # the binding wraps every declared function under the same name
    for n in names:
        assert n in B.SYMBOLS or n in ("zero_plan_segments",), n
        assert hasattr(B, n) or n in ("zero_status_string", "zero_last_cuda_error"), n


def _units_cases():
    rng = np.random.default_rng(0)
    cases = [([1000], 4), ([0], 3), ([], 5), ([1], 16), ([1, 2, 3], 64), ([7, 0, 13, 1, 64], 8)]
    for _ in range(40):
        U = int(rng.integers(1, 20))
        sizes = rng.integers(0, 200000, U)
        sizes[rng.random(U) < 0.15] = int(rng.integers(0, 20))
        cases.append((sizes.tolist(), int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 31, 64]))))
    return cases


@pytest.mark.parametrize("sizes,N", _units_cases())
def test_plan_layout_matches_oracle(zlib, orc, sizes, N):
    p = Z.ZeroPlan(sizes, N)
    o = orc.Plan(sizes, N)
    assert p.P_pad == o.P_pad and p.H == o.H
    assert p.F == o.F.tolist() and p.Hoff == o.Hoff.tolist() and p.S == o.S.tolist() and p.h == o.h.tolist()


@pytest.mark.parametrize("align", [2, 8, 64])
@pytest.mark.parametrize("sizes,N", _units_cases()[::4])
def test_aligned_plan_layout_matches_oracle(zlib, orc, sizes, N, align):
    p = Z.ZeroPlan(sizes, N, align=align)
    o = orc.Plan(sizes, N, align)
    assert Z.zero_plan_align(p.handle) == align
    assert p.P_pad == o.P_pad and p.H == o.H
    assert p.F == o.F.tolist() and p.Hoff == o.Hoff.tolist() and p.S == o.S.tolist() and p.h == o.h.tolist()
    # every slice starts on a multiple of align in the full and the shard buffers, so every
    # segment's full and shard positions are aligned alike (no shifted gradient rows)
    for (g, s, ln, valid, r, u) in Z.zero_plan_segments(p.handle):
        assert (g - s) % align == 0 and (p.F[u] + r * p.h[u]) % align == 0


@pytest.mark.parametrize("table", ["main", "local"])
@pytest.mark.parametrize("align", [1, 8])
@pytest.mark.parametrize("sizes,N", _units_cases()[:20])
def test_launch_table_covers_every_slice_once(zlib, orc, sizes, N, align, table):
    """Both launch tables: the main one (whole-plan launches, norm passes) and the
    unit-local one (one unit or a run of units, cut into about 304 segments each)."""
    p = Z.ZeroPlan(sizes, N, align=align)
    segs = Z.zero_plan_segments(p.handle) if table == "main" else Z.zero_plan_local_segments(p.handle)
    o = orc.Plan(sizes, N, align)
    if table == "local":
        seg_max = 8192 if N <= 8 else 32256
        for u in range(len(sizes)):
            n_u = sum(1 for sg in segs if sg[5] == u)
            if o.S[u] >= 304 * 1024 and o.S[u] <= 304 * seg_max:
                # about 304 per unit: each slice's first segment may be cut short by the alignment
                assert 304 - N <= n_u <= 304 + 2 * N, (u, n_u)
    if o.P_pad == 0:
        assert segs == []
        return
    covered = np.zeros(o.P_pad, np.int32)
    mp = o.shard_map()
    pad = o.pad_mask()
    for (g, s, ln, valid, r, u) in segs:
        assert 1 <= ln <= 32256 and 0 <= valid <= ln
        covered[g:g + ln] += 1
        # the segment's full positions are exactly rank r's shard positions s..s+ln
        assert np.array_equal(mp[r, s:s + ln], np.arange(g, g + ln))
        # pads are exactly the tail after `valid`
        assert np.array_equal(pad[g:g + ln], (np.arange(ln) >= valid).astype(np.uint8))
        assert o.F[u] <= g and g + ln <= o.F[u] + o.S[u]
    assert np.all(covered == 1)
    # after the first segment of a slice, shard positions start 8-aligned
    for i in range(1, len(segs)):
        g0, s0, l0, _, r0, u0 = segs[i - 1]
        g1, s1, l1, _, r1, u1 = segs[i]
        if (r0, u0) == (r1, u1):
            assert s1 == s0 + l0 and s1 % 8 == 0


@pytest.mark.parametrize("N", [3, 8, 16])
def test_local_table_spreads_small_units(zlib, N):
    """The unit-local table cuts a unit of 2^20 elements into about 304 segments
    (the main table: 128 at N = 8, 48 at N = 16), leaves large units as the main
    table cuts them, and never goes below 1024 elements a segment except at the
    end of a slice."""
    sizes = [1000, 1 << 20, 64328960]
    p = Z.ZeroPlan(sizes, N)
    local, main = Z.zero_plan_local_segments(p.handle), Z.zero_plan_segments(p.handle)
    per_unit = lambda segs, u: [sg for sg in segs if sg[5] == u]
    assert 304 <= len(per_unit(local, 1)) <= 304 + 2 * N > len(per_unit(main, 1))
    assert per_unit(local, 2) == per_unit(main, 2)
    assert per_unit(local, 0) == per_unit(main, 0)  # a slice shorter than 1024 is one segment either way
    h = p.h[1]
    for (g, s, ln, valid, r, u) in per_unit(local, 1):
        at_slice_end = g + ln == p.F[1] + (r + 1) * h
        first = g == p.F[1] + r * h
        assert ln >= 1024 - 7 or at_slice_end or first


def test_named_workloads_layout(zlib, orc):
    for fn, N in [(W.gpt2l_units, 8), (W.gpt_1p3b_units, 8), (W.llm_4b_units, 8), (W.finewrap_units, 16),
                  (W.CONFIGS["finewrap600"]["units"], 16)]:
        sizes = fn()
        p = Z.ZeroPlan(sizes, N)
        o = orc.Plan(sizes, N)
        assert p.P_pad == o.P_pad and p.F == o.F.tolist() and p.Hoff == o.Hoff.tolist()
        assert p.workspace is None
        assert Z.zero_plan_workspace_bytes(p.handle) >= 40 * p.n_segments


def test_index_width_workload_layout(zlib, orc):
    """The index-width workload's plan passes 2^32 full positions and 2^31 shard
    positions, and its launch table still covers every position once, each segment
    at the same offset into its slice in both index spaces."""
    sizes = W.CONFIGS["beyond_2p32"]["units"]()
    p = Z.ZeroPlan(sizes, 2)
    o = orc.Plan(sizes, 2)
    assert p.P_pad == o.P_pad > 2 ** 32 and p.H == o.H > 2 ** 31
    assert p.F == o.F.tolist() and p.Hoff == o.Hoff.tolist() and p.h == o.h.tolist()
    seg = np.array(Z.zero_plan_segments(p.handle), dtype=np.int64)
    g, s, ln, valid, r, u = seg.T
    F, Hoff, h = (np.array(x, np.int64) for x in (p.F, p.Hoff, p.h))
    assert ln.sum() == p.P_pad and (g + ln).max() == p.P_pad
    assert np.array_equal(g - F[u] - r * h[u], s - Hoff[u])
    order = np.argsort(g, kind="stable")
    assert np.array_equal(g[order][1:], (g + ln)[order][:-1])  # contiguous, no overlap
    assert (s + ln).max() == p.H


def test_bias_corrections_match_oracle_bitwise(zlib, orc):
    for b1, b2 in [(0.9, 0.95), (0.9, 0.999), (0.8, 0.99), (0.5, 0.5)]:
        for t in list(range(1, 3000)) + [10000, 123457, 2 ** 31 - 1]:
            z = np.float32(Z.zero_bias_corrections(t, b1, b2))
            o = orc.bias_corrections(t, b1, b2)
            assert np.array_equal(np.array(z, np.float32).view(np.uint32), np.array(o, np.float32).view(np.uint32)), t


def test_argument_errors_are_reported_on_the_host(zlib):
    h = C.c_void_p()
    sizes = (C.c_int64 * 2)(5, 7)
    L = zlib
    assert L.zero_plan_create(sizes, 2, 0, C.byref(h)) == B.ZERO_EINVAL
    assert L.zero_plan_create(sizes, 2, 65, C.byref(h)) == B.ZERO_EINVAL
    bad = (C.c_int64 * 2)(5, -1)
    assert L.zero_plan_create(bad, 2, 2, C.byref(h)) == B.ZERO_EINVAL
    assert L.zero_plan_create(None, 2, 2, C.byref(h)) == B.ZERO_EINVAL
    assert L.zero_plan_create(sizes, 2, 2, None) == B.ZERO_EINVAL
    huge = (C.c_int64 * 2)(2 ** 62, 2 ** 62)
    assert L.zero_plan_create(huge, 2, 2, C.byref(h)) == B.ZERO_EINVAL
    assert L.zero_plan_create_aligned(sizes, 2, 2, 0, C.byref(h)) == B.ZERO_EINVAL
    assert L.zero_plan_create_aligned(sizes, 2, 2, 4097, C.byref(h)) == B.ZERO_EINVAL
    assert L.zero_plan_align(None, C.byref(C.c_int32())) == B.ZERO_EINVAL
    assert L.zero_plan_create(sizes, 2, 2, C.byref(h)) == B.ZERO_OK
    # device calls on a plan without a workspace fail before any CUDA call
    ptrs = (C.c_void_p * 2)(16, 32)
    hp = B.AdamW().c()
    assert L.zero_step(h, ptrs, B.ZERO_BF16, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, None, C.byref(hp), None, -1,
                       None) == B.ZERO_ENOTATTACHED
    assert L.zero_reduce_scatter(h, ptrs, B.ZERO_BF16, ptrs, C.c_float(1.0), None) == B.ZERO_ENOTATTACHED
    assert L.zero_all_gather(h, ptrs, C.c_void_p(64), B.ZERO_BF16, -1, None) == B.ZERO_ENOTATTACHED
    assert L.zero_grad_sqnorm(h, ptrs, B.ZERO_BF16, C.c_void_p(64), None) == B.ZERO_ENOTATTACHED
    assert L.zero_step_unit(h, 0, ptrs, B.ZERO_BF16, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(hp),
                            None) == B.ZERO_ENOTATTACHED
    assert L.zero_reduce_scatter_unit(h, 1, ptrs, B.ZERO_BF16, ptrs, C.c_float(1.0), None) == B.ZERO_ENOTATTACHED
    clip = B.AdamW(max_norm=1.0).c()
    assert L.zero_step_unit(h, 0, ptrs, B.ZERO_BF16, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(clip),
                            None) == B.ZERO_EINVAL
    assert L.zero_plan_attach(h, None, 1 << 20, None) == B.ZERO_EINVAL
    assert L.zero_plan_attach(h, C.c_void_p(1 << 12 | 8), 1 << 20, None) == B.ZERO_EALIGN
    assert L.zero_plan_attach(h, C.c_void_p(1 << 12), 8, None) == B.ZERO_ENOMEM
    assert L.zero_bias_corrections(0, C.c_float(0.9), C.c_float(0.95), C.byref(C.c_float()), C.byref(C.c_float())) \
        == B.ZERO_EINVAL
    assert L.zero_plan_query(None, None, None, None, None, None, None) == B.ZERO_EINVAL
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8, -99):
        assert len(L.zero_status_string(s)) > 0
    for s in (-5, -6):  # the statuses zero_plan_check reports have their own text
        assert L.zero_status_string(s) != L.zero_status_string(-99)
    assert L.zero_plan_check(h, None) == B.ZERO_ENOTATTACHED
    assert L.zero_clip_reduce_unit(h, 0, ptrs, B.ZERO_BF16, ptrs, None) == B.ZERO_ENOTATTACHED
    assert L.zero_clip_finalize(h, C.c_float(1.0), None, None) == B.ZERO_ENOTATTACHED
    assert L.zero_adamw_shard_step_clipped(h, ptrs, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(hp), -1,
                                           None) == B.ZERO_ENOTATTACHED
    assert L.zero_clip_finalize(None, C.c_float(1.0), None, None) == B.ZERO_EINVAL
    assert L.zero_plan_check(None, None) == B.ZERO_EINVAL
    # bucket-local calls
    assert L.zero_step_units(h, 0, 2, ptrs, B.ZERO_BF16, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(hp),
                             None) == B.ZERO_ENOTATTACHED
    assert L.zero_step_units(h, 0, 2, ptrs, B.ZERO_BF16, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(clip),
                             None) == B.ZERO_EINVAL  # no clipping from a bucket
    assert L.zero_clip_reduce_units(h, 0, 2, ptrs, B.ZERO_BF16, ptrs, None) == B.ZERO_ENOTATTACHED
    assert L.zero_clip_reduce_units(None, 0, 2, ptrs, B.ZERO_BF16, ptrs, None) == B.ZERO_EINVAL
    # the offload engine: creation and the host update need no device, the step needs an attached plan
    eng = C.c_void_p()
    assert L.zero_offload_create(None, 0, 0, C.byref(eng)) == B.ZERO_EINVAL
    assert L.zero_offload_create(h, -1, 0, C.byref(eng)) == B.ZERO_EINVAL
    assert L.zero_offload_create(h, 2, -5, C.byref(eng)) == B.ZERO_EINVAL
    assert L.zero_offload_create(h, 2, 0, C.byref(eng)) == B.ZERO_OK
    threads, batches = C.c_int32(), C.c_int64()
    assert L.zero_offload_info(eng, C.byref(threads), C.byref(batches)) == B.ZERO_OK
    assert (threads.value, batches.value) == (2, 1)
    assert L.zero_offload_step(eng, ptrs, B.ZERO_BF16, ptrs, ptrs, ptrs, ptrs, ptrs, C.c_void_p(64), None,
                               B.ZERO_BF16, C.byref(hp), None, None) == B.ZERO_ENOTATTACHED
    assert L.zero_offload_adamw(eng, ptrs, ptrs, ptrs, ptrs, None, None, 7, C.byref(hp), C.c_double(0.0),
                                -1) == B.ZERO_EINVAL  # dtype
    assert L.zero_offload_adamw(eng, ptrs, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(hp), C.c_double(0.0),
                                2) == B.ZERO_EINVAL  # unit out of range
    assert L.zero_offload_adamw(eng, None, ptrs, ptrs, ptrs, None, None, B.ZERO_BF16, C.byref(hp), C.c_double(0.0),
                                -1) == B.ZERO_EINVAL  # missing gradient shard
    assert L.zero_offload_timings(eng, (C.c_double * 5)()) == B.ZERO_EINVAL  # no step has run
    L.zero_offload_destroy(eng)
    L.zero_offload_destroy(None)
    L.zero_plan_destroy(h)
    L.zero_plan_destroy(None)


def test_binding_refuses_wrong_tensors_on_the_host(zlib):
    import torch
    p = Z.ZeroPlan([10, 3], 2)  # host-only plan: device is None
    with pytest.raises(ValueError):
        Z.zero_reduce_scatter(p, torch.zeros(2, p.P_pad, dtype=torch.bfloat16),
                              torch.zeros(2, p.H, dtype=torch.float32))


def test_unit_steps_checks_its_tensors_once_on_the_host(zlib):
    """UnitSteps validates and marshals its tensors at construction (a wrong shape,
    dtype or device raises there, before any launch)."""
    import torch
    p = Z.ZeroPlan([10, 3], 2)  # host-only plan: no device, so CPU tensors are refused too
    g = torch.zeros(2, p.P_pad, dtype=torch.bfloat16)
    st = [torch.zeros(2, p.H) for _ in range(3)]
    with pytest.raises(ValueError):
        Z.UnitSteps(p, g, *st)
    with pytest.raises(ValueError):
        Z.UnitSteps(p, g[:, :-1], *st)


def test_rank_pointers_of_a_2d_tensor_match_its_rows():
    """The binding takes the N rank pointers of a [N, L] tensor from its row stride;
    they must be the pointers of its rows (padded rows, views, empty buffers)."""
    import torch

    class Plan:
        n_ranks = 4
        device = torch.device("cpu")

    for x in (torch.zeros(4, 1000, dtype=torch.bfloat16), torch.zeros(4, 1008, dtype=torch.float32)[:, :1000],
              torch.zeros(5, 1000, dtype=torch.bfloat16)[1:], torch.zeros(4, 0, dtype=torch.bfloat16)):
        L = x.shape[1]
        fast, dt = B._rows(Plan, x, L, "x", B._G)
        rows, dt2 = B._rows(Plan, list(x.unbind(0)), L, "x", B._G)
        assert dt == dt2 and [fast[i] for i in range(4)] == [rows[i] for i in range(4)]
    with pytest.raises(ValueError):
        B._rows(Plan, torch.zeros(4, 10, dtype=torch.bfloat16)[:, ::2], 5, "x", B._G)  # rows not contiguous
    with pytest.raises(ValueError):
        B._rows(Plan, torch.zeros(3, 10, dtype=torch.bfloat16), 10, "x", B._G)  # wrong rank count
    with pytest.raises(ValueError):
        B._rows(Plan, torch.zeros(4, 10, dtype=torch.float16), 10, "x", B._G)  # dtype


def test_committed_profiles_describe_the_current_kernel_source():
    """Every ncu summary under profiles/ records the hash of the kernel source it was
    captured from; the bench reports its DRAM traffic only while the hash matches, so a
    kernel change must come with recaptured summaries."""
    import glob
    import sys
    sys.path.insert(0, ROOT)
    import bench
    want = {"kernel": bench.kernel_source_hash(), "reshard": bench.reshard_source_hash()}
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert files
    for path in files:
        text = open(path).read()
        m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
        assert m, path
        kind = "reshard" if os.path.basename(path).startswith("k_reshard") else "kernel"
        assert m.group(1) == want[kind], f"{os.path.basename(path)} was captured from another kernel source"
        assert re.search(r"dram_bytes_per_launch:\s*[0-9]+", text), path
