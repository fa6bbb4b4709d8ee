"""Every entry point of the library on a spread of small cases, each result
checked against the CPU oracle, with canary bands around every device buffer
and the plan's device error word read after every call.

Run as a child process by tests/test_gpu_selfcheck.py, once with the normal
build and once with the diagnostic build (-DZERO_SELFCHECK: every shared- and
global-memory access of the pipelined kernel is bounds- and alignment-checked
first, and a failed check records a code in the error word instead of making
the access).  It prints one JSON line: the error words, and a hash of every
output buffer, which must be the same for both builds.

    python tests/selfcheck_cases.py        (ZERO_LIB=<path> selects the build)
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import fsdp_sharded_optimizer_step_gb300 as Z  # noqa: E402
from fsdp_sharded_optimizer_step_gb300 import binding as B  # noqa: E402
from fsdp_sharded_optimizer_step_gb300 import workloads as W  # noqa: E402
from oracle import oracle as O  # noqa: E402
from parity import ODT, SmallCase, check_guards, f32bits, guarded_buffers, host_bits, hp_for  # noqa: E402

S_RTOL = 1e-12
MAX_NORM = 0.5

# (unit sizes, N, gradient dtype): N from 1 to 64, fp32 and bf16 gradients, ragged
# unit lists, units spanning several segments, fine-wrap-shaped lists whose slices
# sit at misaligned full positions
CASES = [
    ([1000], 4, W.F32),
    ([5, 0, 13, 1, 64, 257, 4099], 4, W.BF16),
    ([70001, 3, 65537, 12345], 8, W.BF16),
    ([70001, 3, 65537, 12345], 8, W.F32),
    ([99991, 7, 40000], 3, W.BF16),
    ([33, 100003, 2, 77777], 5, W.F32),
    ([1, 2, 3, 4, 5, 6, 7, 8, 9, 131071], 16, W.BF16),
    ([131072 * 3 + 5], 2, W.BF16),
    ([4097, 1], 1, W.BF16),
    ([300, 17, 9000], 64, W.BF16),
    (W.finewrap_units(n_units=300, lo_log2=0, hi_log2=16, seed=4), 16, W.BF16),
    (W.finewrap_units(n_units=200, lo_log2=4, hi_log2=18, seed=9), 8, W.F32),
]


def _unit_rows(c, u):
    F, S = c.plan.F[u], c.plan.S[u]
    rows = guarded_buffers(c.guards, S, c.grads.dtype, c.device, rows=c.N)
    rows.copy_(c.grads[:, F:F + S])
    return rows


def _check_oracle_step(c, t, max_norm=0.0):
    assert c.oracle_step(t, max_norm=max_norm) == O.OK
    c.assert_state_equal()
    c.assert_full_equal()
    c.assert_pshard_equal()


def _check_norm(S_gpu, S_o):
    assert abs(S_gpu - S_o) <= S_RTOL * S_o, (S_gpu, S_o)
    assert O.clip_coef(S_gpu, MAX_NORM) == O.clip_coef(S_o, MAX_NORM)


def run_case(ci, sizes, N, gd, digest):
    c = SmallCase(sizes, N, gd, W.BF16, seed=ci + 1, grad_sigma=1e-2, outlier_frac=1e-3, outlier_scale=100.0)
    plan, U = c.plan, len(sizes)
    errors = []

    def after(what):
        torch.cuda.synchronize()
        errors.append((what, B.zero_plan_device_errors(plan)))
        c.check_guards()

    # fused step, all units in one launch
    c.gpu_step(1)
    after("fused")
    _check_oracle_step(c, 1)
    # clipped step (norm pass, device total, shard update)
    c.gpu_step(2, max_norm=MAX_NORM)
    after("clipped")
    _check_oracle_step(c, 2, MAX_NORM)
    _check_norm(c.sq.item(), c.S_o)
    # one launch per unit
    for u in range(U):
        c.gpu_step(3, unit=u)
    after("per-unit")
    _check_oracle_step(c, 3)
    # unit-local gradient buffers
    hp, _ = hp_for(4)
    for u in range(U):
        if plan.S[u]:
            Z.zero_step_unit(plan, u, _unit_rows(c, u), c.master, c.m, c.v, hp, full=c.full, pshard=c.pshard)
    after("unit-local step")
    _check_oracle_step(c, 4)
    # the unfused parts: reduce-scatter, shard update, all-gather
    Z.zero_reduce_scatter(plan, c.grads, c.gshard)
    after("reduce-scatter")
    avg = O.avg_grad(c.g_o, ODT[c.gdtype], c.pad)
    assert np.array_equal(host_bits(c.gshard), f32bits(avg)[c.map])
    hp, _ = hp_for(5)
    Z.zero_adamw_shard_step(plan, c.gshard, c.master, c.m, c.v, hp, pshard=c.pshard)
    c.full.zero_()
    Z.zero_all_gather_bf16(plan, c.pshard, c.full)
    after("shard update + gather")
    _check_oracle_step(c, 5)
    # the streamed clipped step: per-unit norm passes, device total, per-unit update
    for u in range(U):
        if plan.S[u]:
            Z.zero_clip_reduce_unit(plan, u, _unit_rows(c, u), c.gshard)
    Z.zero_clip_finalize(plan, MAX_NORM, c.sq)
    hp, _ = hp_for(6, MAX_NORM)
    for u in range(U):
        if plan.S[u]:
            Z.zero_adamw_shard_step_clipped(plan, c.gshard, c.master, c.m, c.v, hp, full=c.full, pshard=c.pshard,
                                            unit=u)
    after("streamed clipped step")
    _check_oracle_step(c, 6, MAX_NORM)
    _check_norm(c.sq.item(), c.S_o)
    # the plan's norm, and the unit-local reduce-scatter with a coefficient
    Z.zero_grad_sqnorm(plan, c.grads, c.sq)
    after("norm")
    _check_norm(c.sq.item(), O.sqnorm(c.g_o, ODT[c.gdtype], c.pad))
    coef = np.float32(0.3711)
    for u in range(U):
        if plan.S[u]:
            Z.zero_reduce_scatter_unit(plan, u, _unit_rows(c, u), c.gshard, coef=float(coef))
    after("unit-local reduce-scatter")
    assert np.array_equal(host_bits(c.gshard), f32bits((avg * coef).astype(np.float32))[c.map])
    # ZeRO-3 gathers into unit-sized buffers
    for u in range(U):
        F, S = plan.F[u], plan.S[u]
        if S:
            dst = guarded_buffers(c.guards, S, torch.bfloat16, c.device, zero=True)
            Z.zero_all_gather_unit(plan, u, c.pshard, dst)
            after(f"unit gather {u}")
            assert np.array_equal(host_bits(dst), c.out_o[F:F + S])
    # checkpoint reshard to another rank count
    N2 = 3 if N != 3 else 8
    p2 = Z.ZeroPlan(sizes, N2, c.device)
    dst = guarded_buffers(c.guards, p2.H, torch.float32, c.device, rows=N2)
    Z.zero_reshard(plan, p2, c.master, dst)
    torch.cuda.synchronize()
    check_guards(c.guards)
    assert np.array_equal(host_bits(dst), O.reshard(sizes, N, N2, host_bits(c.master)))
    for x in (c.master, c.m, c.v, c.full, c.pshard, c.gshard, dst):
        digest.update(host_bits(x).tobytes())
    digest.update(c.sq.cpu().numpy().tobytes())
    return errors


def main():
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 2
    Z.lib()
    digest = hashlib.sha256()
    errors = {}
    for ci, (sizes, N, gd) in enumerate(CASES):
        errors[ci] = run_case(ci, sizes, N, gd, digest)
    bad = {ci: [e for e in errs if e[1] != 0] for ci, errs in errors.items()}
    bad = {ci: errs for ci, errs in bad.items() if errs}
    print(json.dumps({"lib": os.environ.get("ZERO_LIB") or B._build.LIB, "cases": len(CASES),
                      "nonzero_error_words": bad, "hash": digest.hexdigest()[:16]}), flush=True)
    return 0 if not bad else 1


if __name__ == "__main__":
    sys.exit(main())
