"""zero_grad_sqnorm_noalloc: the gradient norm for callers that cannot allocate.

A norm check often has to run when device memory is exhausted (reporting the
norm of a step that ran out of memory, or a watchdog for non-finite gradients
inside a framework whose caching allocator holds nearly all of the GPU).  The
allocation-free entry point keeps its partial sums in an array compiled into
the library instead of a workspace.  These tests call it through the C ABI
and compare each result with the oracle's exact sum of squares (and with the
plan-based zero_grad_sqnorm) within the relative 1e-12 the parity tests use:
two calls in a row, the second smaller than the first, so partials left by the
first call must not leak into the second; more chunks than the final pass's
1024 threads; n = 0; inf and NaN gradients; argument errors; and a call made
after the device's memory has been used up.  This file is collected last, so a
run that stops at the first failure has already run every other test.
"""
import ctypes as C
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import binding as B
from fsdp_sharded_optimizer_step_gb300 import workloads as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu

S_RTOL = 1e-12
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zlib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_optimizer_step_gb300 import build
    build.build()
    return Z.lib()


def _oracle_rows(t: torch.Tensor):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return [r for r in t.view(torch.int16).numpy().view(np.uint16)], O.BF16
    return [r for r in t.numpy()], O.F32


def _noalloc(zlib, grads, n, dev):
    """One call through the C ABI; returns (status, S)."""
    N = grads.shape[0]
    out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    ptrs = (C.c_void_p * N)(*[grads[r].data_ptr() for r in range(N)])
    gd = B.ZERO_BF16 if grads.dtype == torch.bfloat16 else B.ZERO_F32
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = zlib.zero_grad_sqnorm_noalloc(ptrs, N, gd, int(n), C.c_void_p(out.data_ptr()), stream)
    torch.cuda.synchronize(dev)
    return rc, out.item()


def _seeded_grads(N, n, dtype, seed, dev):
    grads = Z.rank_buffers(N, n, dtype, dev)
    grads.copy_(W.make_grads(N, n, W.BF16 if dtype == torch.bfloat16 else W.F32, sigma=1e-2, seed=seed,
                             outlier_frac=1e-3, outlier_scale=100.0))
    return grads


def _three_ways(zlib, sizes, N, dtype, seed):
    """The oracle's exact S, the plan-based GPU norm and the allocation-free one on the
    same gradients; the unit sizes are multiples of N, so the flat buffers have no
    padding and all three sum over the same positions."""
    dev = torch.device("cuda", torch.cuda.current_device())
    assert all(s % N == 0 for s in sizes)
    plan = Z.ZeroPlan(sizes, N, dev)
    grads = _seeded_grads(N, plan.P_pad, dtype, seed, dev)
    ref = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    Z.zero_grad_sqnorm(plan, grads, ref)
    rc, got = _noalloc(zlib, grads, plan.P_pad, dev)
    assert rc == B.ZERO_OK, zlib.zero_status_string(rc)
    rows, gd = _oracle_rows(grads)
    return O.sqnorm(rows, gd), ref.item(), got


def test_noalloc_sqnorm_matches_oracle_on_two_calls_in_a_row(zlib):
    # first call: 8 ranks of bf16 gradients, 4,048,576 positions (31 chunks)
    s_o, a_ref, a = _three_ways(zlib, [3_000_000, 1_048_576], 8, torch.bfloat16, seed=21)
    assert s_o > 0 and abs(a - s_o) <= S_RTOL * s_o and abs(a_ref - s_o) <= S_RTOL * s_o
    # second call, right after: 3 ranks of fp32 (division by 3), 337,035 positions (3 chunks)
    s_o, b_ref, b = _three_ways(zlib, [300_000, 37_035], 3, torch.float32, seed=22)
    assert s_o > 0 and abs(b - s_o) <= S_RTOL * s_o and abs(b_ref - s_o) <= S_RTOL * s_o


def test_noalloc_sqnorm_more_chunks_than_final_threads(zlib):
    """1025 chunks (131,072 positions each, the last one partial): the final pass's
    1024 threads each add more than one partial."""
    dev = torch.device("cuda", torch.cuda.current_device())
    n = 1024 * 131072 + 12346
    grads = _seeded_grads(2, n, torch.bfloat16, 23, dev)
    rc, got = _noalloc(zlib, grads, n, dev)
    assert rc == B.ZERO_OK
    rows, gd = _oracle_rows(grads)
    s_o = O.sqnorm(rows, gd)
    assert abs(got - s_o) <= S_RTOL * s_o


def test_noalloc_sqnorm_empty_and_non_finite(zlib):
    dev = torch.device("cuda", torch.cuda.current_device())
    out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    null_ptrs = (C.c_void_p * 2)()
    rc = zlib.zero_grad_sqnorm_noalloc(null_ptrs, 2, B.ZERO_BF16, 0, C.c_void_p(out.data_ptr()), None)
    torch.cuda.synchronize(dev)
    assert rc == B.ZERO_OK and out.item() == 0.0 and not math.copysign(1.0, out.item()) < 0
    for bad, check in ((float("inf"), math.isinf), (float("nan"), math.isnan)):
        grads = _seeded_grads(3, 5000, torch.float32, 24, dev)
        grads[1, 17] = bad
        rc, got = _noalloc(zlib, grads, 5000, dev)
        assert rc == B.ZERO_OK
        rows, gd = _oracle_rows(grads)
        s_o = O.sqnorm(rows, gd)
        assert check(got) and check(s_o), (bad, got, s_o)
    # +inf and -inf in one position: their sum is NaN
    grads = _seeded_grads(3, 5000, torch.float32, 25, dev)
    grads[0, 9], grads[2, 9] = float("inf"), float("-inf")
    rc, got = _noalloc(zlib, grads, 5000, dev)
    assert rc == B.ZERO_OK and math.isnan(got)


def test_noalloc_sqnorm_rejects_bad_arguments(zlib):
    """Checked on the host: nothing is launched or touched."""
    fn = zlib.zero_grad_sqnorm_noalloc
    dev = torch.device("cuda", torch.cuda.current_device())
    out = torch.zeros(1, dtype=torch.float64, device=dev)
    g = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    ptrs = (C.c_void_p * 1)(g.data_ptr())
    too_many = 131072 * 32768 + 1
    assert fn(ptrs, 1, B.ZERO_BF16, too_many, C.c_void_p(out.data_ptr()), None) == B.ZERO_ERANGE
    assert fn(ptrs, 0, B.ZERO_BF16, 16, C.c_void_p(out.data_ptr()), None) == B.ZERO_EINVAL
    assert fn(ptrs, 1, B.ZERO_BF16, -1, C.c_void_p(out.data_ptr()), None) == B.ZERO_EINVAL
    odd = (C.c_void_p * 1)(g.data_ptr() + 1)  # bf16 gradients one byte off
    assert fn(odd, 1, B.ZERO_BF16, 16, C.c_void_p(out.data_ptr()), None) == B.ZERO_EALIGN
    assert fn(ptrs, 1, B.ZERO_BF16, 16, C.c_void_p(out.data_ptr() + 4), None) == B.ZERO_EALIGN
    host = torch.zeros(64, dtype=torch.bfloat16)  # not device memory
    hptrs = (C.c_void_p * 1)(host.data_ptr())
    assert fn(hptrs, 1, B.ZERO_BF16, 16, C.c_void_p(out.data_ptr()), None) == B.ZERO_EINVAL
    host_out = torch.zeros(1, dtype=torch.float64)
    assert fn(ptrs, 1, B.ZERO_BF16, 16, C.c_void_p(host_out.data_ptr()), None) == B.ZERO_EINVAL


_AFTER_OOM = r"""
import ctypes as C, json, sys
sys.path.insert(0, sys.argv[1])
import torch
import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import binding as B
from fsdp_sharded_optimizer_step_gb300 import workloads as W
L = Z.lib()
dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
N, n = 4, 3 * 131072 + 77
grads = Z.rank_buffers(N, n, torch.bfloat16, dev)
grads.copy_(W.make_grads(N, n, W.BF16, sigma=1e-2, seed=26))
out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
st = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
ptrs = (C.c_void_p * N)(*[grads[r].data_ptr() for r in range(N)])
# the set-up call, while memory is free: n = 0 loads the kernels and finds the array
warm = L.zero_grad_sqnorm_noalloc((C.c_void_p * N)(), N, B.ZERO_BF16, 0, C.c_void_p(out.data_ptr()), st)
torch.cuda.synchronize(dev)
# use up the device's memory with plain allocations (never touched)
blocks, chunk = [], 1 << 32
while chunk >= (1 << 21):
    try:
        blocks.append(torch.empty(chunk, dtype=torch.uint8, device=dev))
    except RuntimeError:
        chunk //= 2
exhausted = False
try:
    torch.empty(64 << 20, dtype=torch.uint8, device=dev)
except RuntimeError:
    exhausted = True
free_bytes = torch.cuda.mem_get_info(dev)[0]
results = []
for _ in range(2):
    out.fill_(-1.0)
    rc = L.zero_grad_sqnorm_noalloc(ptrs, N, B.ZERO_BF16, n, C.c_void_p(out.data_ptr()), st)
    torch.cuda.synchronize(dev)
    results.append((rc, out.item()))
held = sum(b.numel() for b in blocks)
del blocks
print(json.dumps({"warm": warm, "exhausted": exhausted, "free_bytes": free_bytes, "held_bytes": held,
                  "results": results}))
"""


def test_noalloc_sqnorm_after_device_memory_is_used_up(zlib):
    """In a fresh process: the set-up call (n = 0) while memory is free, then every
    free byte of the device taken by plain allocations until one more 64 MiB
    request fails, then two calls: both succeed with the oracle's sum."""
    proc = subprocess.run([sys.executable, "-c", _AFTER_OOM, ROOT], capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    res = json.loads(proc.stdout.strip().splitlines()[-1])
    assert res["warm"] == B.ZERO_OK
    assert res["exhausted"], res
    N, n = 4, 3 * 131072 + 77
    rows, gd = _oracle_rows(W.make_grads(N, n, W.BF16, sigma=1e-2, seed=26))
    s_o = O.sqnorm(rows, gd)
    for rc, got in res["results"]:
        assert rc == B.ZERO_OK
        assert abs(got - s_o) <= S_RTOL * s_o
