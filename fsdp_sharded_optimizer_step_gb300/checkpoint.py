"""Sharded checkpoint of the per-rank optimizer state, resharded at load time.

"ZeRO and FSDP sharding", Implementation notes: write the checkpoint sharded
(each rank writes its own shard; gathering the whole state onto one rank is
slow and can run out of memory) and reshard to a different N when loading.

On disk, a directory holds layout.json (unit sizes, rank count, alignment,
step, and the name/dtype of every array) and one file per rank, rankNNNNN.bin, with that
rank's shard of every array concatenated in layout order.  Loading into a plan
with another rank count reads the old shards into device buffers and remaps
them with zero_reshard (one launch per array); the same rank count and
alignment is a plain copy.  Host IO only here: the remap runs in the CUDA library.
"""
import json
import os

import numpy as np
import torch

from . import binding as B

_DT = {"f32": (torch.float32, np.float32), "bf16": (torch.bfloat16, np.uint16)}


def _kind(t: torch.Tensor) -> str:
    if t.dtype == torch.float32:
        return "f32"
    if t.dtype == torch.bfloat16:
        return "bf16"
    raise ValueError(f"unsupported dtype {t.dtype}")


def _host_bytes(row: torch.Tensor) -> bytes:
    row = row.detach().cpu().contiguous()
    if row.dtype == torch.bfloat16:
        row = row.view(torch.int16)
    return row.numpy().tobytes()


def save(path, plan, arrays: dict, step: int):
    """arrays: name -> [N, H] tensors (rank rows); every rank writes its own file."""
    os.makedirs(path, exist_ok=True)
    names = list(arrays)
    for name in names:
        a = arrays[name]
        if len(a) != plan.n_ranks or any(r.numel() != plan.H for r in a):
            raise ValueError(f"{name}: need {plan.n_ranks} rank rows of {plan.H} elements")
    layout = {"unit_sizes": plan.unit_sizes, "n_ranks": plan.n_ranks, "align": plan.align, "H": plan.H,
              "step": int(step),
              "arrays": [{"name": n, "dtype": _kind(arrays[n][0])} for n in names]}
    for r in range(plan.n_ranks):
        tmp = os.path.join(path, f"rank{r:05d}.bin.tmp")
        with open(tmp, "wb") as f:
            for n in names:
                f.write(_host_bytes(arrays[n][r]))
        os.replace(tmp, os.path.join(path, f"rank{r:05d}.bin"))
    with open(os.path.join(path, "layout.json.tmp"), "w") as f:
        json.dump(layout, f)
    os.replace(os.path.join(path, "layout.json.tmp"), os.path.join(path, "layout.json"))


def load(path, plan, stream=None):
    """Returns ({name: [N', H'] device tensors in plan's layout}, step).

    stream: the CUDA stream the copies and the reshard run on (default: the
    current stream).  The whole load runs with that stream current, so the
    staging buffers are allocated, filled, read and released on the one stream
    that uses them (the caching allocator cannot hand a buffer the reshard is
    still reading to the next array's copies)."""
    with open(os.path.join(path, "layout.json")) as f:
        layout = json.load(f)
    if [int(s) for s in layout["unit_sizes"]] != plan.unit_sizes:
        raise ValueError("checkpoint units differ from the plan's")
    dev = plan.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev), torch.cuda.stream(stream):
        out = _load_arrays(path, layout, plan, dev, stream)
    stream.synchronize()
    return out, int(layout["step"])


def _load_arrays(path, layout, plan, dev, stream):
    n_old, H_old, a_old = int(layout["n_ranks"]), int(layout["H"]), int(layout.get("align", 1))
    same = n_old == plan.n_ranks and a_old == plan.align
    old = None if same else B.ZeroPlan(layout["unit_sizes"], n_old, dev, stream=stream, align=a_old)
    out = {}
    offset = 0  # bytes into every rank file
    for spec in layout["arrays"]:
        tdt, ndt = _DT[spec["dtype"]]
        src = B.rank_buffers(n_old, H_old, tdt, dev)
        for r in range(n_old):
            host = np.fromfile(os.path.join(path, f"rank{r:05d}.bin"), dtype=ndt, count=H_old, offset=offset)
            t = torch.from_numpy(host)
            if tdt == torch.bfloat16:
                t = t.view(torch.bfloat16)
            src[r].copy_(t)
        if old is None:
            out[spec["name"]] = src
        else:
            dst = B.rank_buffers(plan.n_ranks, plan.H, tdt, dev)
            B.zero_reshard(old, plan, src, dst, stream=stream)
            out[spec["name"]] = dst
        offset += H_old * np.dtype(ndt).itemsize
    return out
