"""zero_grad_sqnorm_noalloc: the gradient norm for callers that cannot allocate.

A norm check often has to run when device memory is exhausted (reporting the
norm of a step that ran out of memory, or a watchdog for non-finite gradients
inside a framework whose caching allocator holds nearly all of the GPU).  The
allocation-free entry point keeps its partial sums in an array compiled into
the library instead of a workspace.  These tests call it through the C ABI
twice in a row -- the second call smaller than the first, so partials left by
the first call must not leak into the second -- and compare each result with
the plan-based zero_grad_sqnorm within the relative 1e-12 the parity tests use.
This file is collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes as C

import pytest
import torch

import fsdp_sharded_optimizer_step_gb300 as Z
from fsdp_sharded_optimizer_step_gb300 import binding as B
from fsdp_sharded_optimizer_step_gb300 import workloads as W

pytestmark = pytest.mark.gpu

S_RTOL = 1e-12


@pytest.fixture(scope="module")
def zlib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_optimizer_step_gb300 import build
    build.build()
    return Z.lib()


def _plan_sqnorm_and_noalloc(zlib, sizes, N, dtype, seed):
    """Both entry points on the same gradients; the unit sizes are multiples of N,
    so the flat buffers have no padding and both sum over the same positions."""
    dev = torch.device("cuda", torch.cuda.current_device())
    assert all(s % N == 0 for s in sizes)
    plan = Z.ZeroPlan(sizes, N, dev)
    grads = Z.rank_buffers(N, plan.P_pad, dtype, dev)
    grads.copy_(W.make_grads(N, plan.P_pad, W.BF16 if dtype == torch.bfloat16 else W.F32, sigma=1e-2, seed=seed,
                             outlier_frac=1e-3, outlier_scale=100.0))
    ref = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    Z.zero_grad_sqnorm(plan, grads, ref)
    out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    ptrs = (C.c_void_p * N)(*[grads[r].data_ptr() for r in range(N)])
    gd = B.ZERO_BF16 if dtype == torch.bfloat16 else B.ZERO_F32
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = zlib.zero_grad_sqnorm_noalloc(ptrs, N, gd, plan.P_pad, C.c_void_p(out.data_ptr()), stream)
    assert rc == B.ZERO_OK, zlib.zero_status_string(rc)
    torch.cuda.synchronize(dev)
    return ref.item(), out.item()


def test_noalloc_sqnorm_matches_plan_sqnorm_on_two_calls_in_a_row(zlib):
    # first call: 8 ranks of bf16 gradients, 4,048,576 positions (31 chunks)
    a_ref, a = _plan_sqnorm_and_noalloc(zlib, [3_000_000, 1_048_576], 8, torch.bfloat16, seed=21)
    assert a_ref > 0 and abs(a - a_ref) <= S_RTOL * a_ref
    # second call, right after: 3 ranks of fp32 (division by 3), 337,035 positions (3 chunks)
    b_ref, b = _plan_sqnorm_and_noalloc(zlib, [300_000, 37_035], 3, torch.float32, seed=22)
    assert b_ref > 0 and abs(b - b_ref) <= S_RTOL * b_ref


def test_noalloc_sqnorm_rejects_sizes_beyond_its_capacity(zlib):
    cap = B.lib().zero_grad_sqnorm_noalloc  # checked on the host: nothing is launched or touched
    dev = torch.device("cuda", torch.cuda.current_device())
    out = torch.zeros(1, dtype=torch.float64, device=dev)
    g = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    ptrs = (C.c_void_p * 1)(g.data_ptr())
    too_many = 131072 * 32768 + 1
    assert cap(ptrs, 1, B.ZERO_BF16, too_many, C.c_void_p(out.data_ptr()), None) == B.ZERO_ERANGE
    assert cap(ptrs, 0, B.ZERO_BF16, 16, C.c_void_p(out.data_ptr()), None) == B.ZERO_EINVAL
