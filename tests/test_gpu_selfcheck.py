"""The diagnostic build on the GPU: a stand-in for a memory checker.

The library is built a second time with -DZERO_SELFCHECK: every shared- and
global-memory access of the pipelined kernel is checked against its buffer's
bounds and alignment before it is made, and a failed check records a code in
the plan's device error word and skips the access instead of faulting.  Both
builds run every entry point over twelve small cases (tests/selfcheck_cases.py,
one child process per build), each result checked against the CPU oracle, with
canary bands around every device buffer.  The error word must stay 0 after
every call, and both builds must produce the same bits.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(env_lib):
    env = dict(os.environ)
    env.pop("ZERO_LIB", None)
    if env_lib:
        env["ZERO_LIB"] = env_lib
    proc = subprocess.run([sys.executable, os.path.join(HERE, "selfcheck_cases.py")], env=env, capture_output=True,
                          text=True, timeout=1200)
    assert proc.returncode == 0, (proc.stdout[-2000:], proc.stderr[-4000:])
    return json.loads(proc.stdout.strip().splitlines()[-1])


def test_selfcheck_build_runs_every_entry_point_clean():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_optimizer_step_gb300 import build
    normal_lib = build.build()
    checked_lib = build.build_variant("selfcheck", ["ZERO_SELFCHECK"])
    normal = _run(None)
    checked = _run(checked_lib)
    assert normal["lib"] == normal_lib and checked["lib"] == checked_lib
    assert normal["cases"] == checked["cases"] == 12
    assert normal["nonzero_error_words"] == {} and checked["nonzero_error_words"] == {}
    assert normal["hash"] == checked["hash"]
