"""The bench's multi-process plumbing on CPU (gloo, world size 2): the
max-over-ranks timing reduction and barrier, a rank that dies before the
barrier (the survivor fails after the process-group timeout instead of
hanging), and the reference arm under torchrun (rank 0 alone runs and prints
one JSON line, the other rank exits 0)."""
import json
import os
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + rank * 5.5, world, torch.device("cpu"))
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.5, 1: 15.5}


def _dying_worker(rank, world, port, q):
    """Rank 1 leaves before the barrier (between steps: it has no work in flight);
    rank 0 must get an error from its barrier within the timeout, not hang."""
    import argparse
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_setup(argparse.Namespace(impl="reference", dist_timeout=3.0))
    def report(msg):
        q.put((rank, msg))
        q.close()
        q.join_thread()  # flushed before the process ends without cleanup
        os._exit(0)

    if rank == 1:
        report("left")
    t0 = time.time()
    try:
        bench.barrier(world)
        report("no error")
    except Exception as e:  # the collective failed: the missing rank was detected
        report(f"error after {time.time() - t0:.1f} s: {type(e).__name__}")


def test_a_rank_that_dies_is_detected_not_waited_for():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29800 + os.getpid() % 1000
    procs = [ctx.Process(target=_dying_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res[1] == "left"
    assert res[0].startswith("error after"), res[0]
    assert float(res[0].split()[2]) < 60.0


def _check_reference_line(line, world):
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["n_gpus"] == world and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("gpt2l")


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--ref-sample", "65536"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_under_torchrun_world_2():
    port = 30500 + os.getpid() % 1000
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-sample", "65536"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 only
    _check_reference_line(lines[0], 2)


def test_all_cores_oracle_step_is_bit_identical_to_the_oracle_step():
    """The bench's all-cores CPU row runs the oracle's functions on one chunk of
    positions per thread (clip: exact partial sums of squares merged); w, m, v, the
    output and S must equal one single-threaded oracle step bit for bit."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from oracle import build as obuild
    from oracle import oracle as O
    obuild.build()
    rng = np.random.default_rng(3)
    n, N = 100_003, 8
    for gd, max_norm in ((O.BF16, 0.0), (O.BF16, 1e-3), (O.F32, 0.5), (O.F32, 0.0)):
        g = (rng.normal(0, 1e-2, (N, n))).astype(np.float32)
        rows = [(r.view(np.uint32) >> 16).astype(np.uint16) for r in g] if gd == O.BF16 else list(g)
        w0 = rng.normal(0, 0.02, n).astype(np.float32)
        m0 = (rng.normal(0, 1e-3, n)).astype(np.float32)
        v0 = (rng.random(n) * 1e-6).astype(np.float32)
        hp = O.hparams(t=3, max_norm=max_norm)
        w1, m1, v1 = w0.copy(), m0.copy(), v0.copy()
        rc1, out1, S1 = O.step(rows, gd, w1, m1, v1, hp, pdtype=O.BF16)
        w2, m2, v2 = w0.copy(), m0.copy(), v0.copy()
        with ThreadPoolExecutor(7) as ex:
            rc2, out2, S2 = bench.oracle_step_all_cores(ex, 7, rows, gd, w2, m2, v2, hp, O.BF16, max_norm)
        assert rc1 == rc2 == O.OK
        for a, b in ((w1, w2), (m1, m2), (v1, v2)):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(out1, out2)
        if max_norm > 0:
            assert S1 == S2
    # a non-finite norm: the step is skipped on both sides
    rows = [np.full(10, np.inf, np.float32)] + [np.zeros(10, np.float32)] * 3
    w = np.zeros(10, np.float32)
    with ThreadPoolExecutor(3) as ex:
        rc, out, S = bench.oracle_step_all_cores(ex, 3, rows, O.F32, w, w.copy(), w.copy(),
                                                 O.hparams(t=1, max_norm=1.0), O.BF16, 1.0)
    assert rc == O.ENONFINITE and S == float("inf")
