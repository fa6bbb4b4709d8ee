"""ZeRO-3 just-in-time parameter gather with prefetch, and ZeRO-2 bucketed
gradient reduce-scatter -- the two steps either side of the update.

"ZeRO and FSDP sharding", How it works: per unit, all-gather the bf16 weights,
compute, free the non-owned part; prefetching unit k+1's all-gather while unit
k computes keeps it off the critical path, and the peak extra memory is about
two units of full weights (Complexity and constants).  "ZeRO: Three Ledgers,
Zero Redundancy", section 4: gradients streamed through buckets never exist in
full, which is why stage 1 and stage 2 measure the same.

Orchestration only (streams, events, unit-sized buffers); the gathers,
reduce-scatters and updates run in the CUDA library (zero_all_gather_unit,
zero_reduce_scatter_unit, zero_step_units, zero_clip_reduce_units).
"""
import ctypes

import torch

from . import binding as B


class UnitGatherer:
    """Gathers one unit at a time from the rank param shards into one of
    `n_buffers` unit-sized buffers; with prefetch, unit k+1 is gathered on a side
    stream while the caller's compute runs on unit k.

    A gather of one GPT-2-Large block moves ~79 MB (~11 us of HBM time), less than
    a checked call through the binding costs on the host, so the arguments are
    checked and marshalled once here (shard pointers, buffer pointers, dtype) and
    each gather is one direct call of zero_all_gather_unit."""

    def __init__(self, plan, pshard, dtype=torch.bfloat16, n_buffers=2):
        self.plan, self.pshard = plan, pshard
        dev = plan.device
        max_s = max(list(plan.S) + [1])
        per16 = 16 // torch.empty((), dtype=dtype).element_size()
        stride = (max_s + per16 - 1) // per16 * per16
        self.buffers = [torch.empty(stride, dtype=dtype, device=dev) for _ in range(n_buffers)]
        self.side = torch.cuda.Stream(dev)
        self.ready = [torch.cuda.Event() for _ in range(n_buffers)]
        self.free = [torch.cuda.Event() for _ in range(n_buffers)]
        self._shards, self._pdtype = B._rows(plan, pshard, plan.H, "pshard", (dtype,))
        self._dst = [ctypes.c_void_p(buf.data_ptr()) for buf in self.buffers]
        self._fn = B.lib().zero_all_gather_unit

    def _gather(self, u, b, stream):
        st = ctypes.c_void_p(stream.cuda_stream)
        rc = self._fn(self.plan.handle, u, self._shards, self._dst[b], self._pdtype, st)
        if rc != B.ZERO_OK:
            raise B.ZeroError(rc, "zero_all_gather_unit")

    def run(self, compute, order=None, prefetch=True, stream=None):
        """compute(u, params_u) is called for every unit in `order`, on `stream`
        (default: the current stream), with params_u the unit's gathered params."""
        main = stream if stream is not None else torch.cuda.current_stream(self.plan.device)
        order = list(range(self.plan.n_units)) if order is None else list(order)
        order = [u for u in order if self.plan.S[u] > 0]
        nb = len(self.buffers)
        start = torch.cuda.Event()
        start.record(main)
        self.side.wait_event(start)
        for b in range(nb):
            self.free[b].record(main)

        def issue(i):
            b = i % nb
            if prefetch:
                self.side.wait_event(self.free[b])
                self._gather(order[i], b, self.side)
                self.ready[b].record(self.side)
            else:
                self._gather(order[i], b, main)

        if order:
            issue(0)
        for i, u in enumerate(order):
            b = i % nb
            if prefetch:
                main.wait_event(self.ready[b])
                if i + 1 < len(order):
                    issue(i + 1)
            compute(u, self.buffers[b][:self.plan.S[u]])
            self.free[b].record(main)
            if not prefetch and i + 1 < len(order):
                issue(i + 1)
        end = torch.cuda.Event()
        end.record(self.side)
        main.wait_event(end)


class BucketedReduceScatter:
    """ZeRO-2 gradient flow through one reusable bucket: fill(u, bucket) writes
    unit u's N rank gradients (the backward of that unit), and the bucket is
    reduce-scattered into the fp32 gradient shard right away."""

    def __init__(self, plan, grad_dtype=torch.bfloat16):
        self.plan = plan
        self.bucket = B.rank_buffers(plan.n_ranks, max(list(plan.S) + [1]), grad_dtype, plan.device)

    @property
    def bucket_bytes(self):
        return self.bucket.shape[0] * self.bucket.stride(0) * self.bucket.element_size()

    def reduce(self, unit, fill, gshard, coef=1.0, stream=None):
        S = self.plan.S[unit]
        if S == 0:
            return
        view = self.bucket[:, :S]
        fill(unit, view)
        B.zero_reduce_scatter_unit(self.plan, unit, view, gshard, coef=coef, stream=stream)


def backward_buckets(plan, bucket_elems):
    """Buckets of consecutive units in backward order (last unit first): each holds
    units [u0, u1) whose padded sizes add up to at most bucket_elems (a larger unit
    forms a bucket of its own); units without elements join their neighbours."""
    out, u = [], plan.n_units
    while u > 0:
        u1, total = u, 0
        while u > 0 and (total == 0 or total + plan.S[u - 1] <= bucket_elems):
            total += plan.S[u - 1]
            u -= 1
        if total > 0:
            out.append((u, u1))
    return out


class BucketedStep:
    """The ZeRO-2 step with the gradients streamed through one reusable bucket.

    The backward produces the gradients bucket by bucket, last units first
    (fill(u0, u1, view) writes the N rank gradients of units [u0, u1) into
    `view`, on the step's stream); each bucket is consumed as soon as it is full:
    without clipping by the fused update of its units (zero_step_units: reduce-
    scatter, AdamW, cast and gather in one launch, no gradient shard in memory);
    with clipping by its norm pass (zero_clip_reduce_units: averaged fp32
    gradient shard plus sums of squares), and once every bucket is in, the
    global coefficient and the shard update.  Same bits as zero_step.  Memory:
    one bucket of N x bucket_elems gradients instead of N full gradient buffers.
    bucket_elems: padded elements per bucket (default: the largest unit, at least 2^27)."""

    def __init__(self, plan, grad_dtype=torch.bfloat16, bucket_elems=None):
        self.plan = plan
        if bucket_elems is None:
            bucket_elems = max(max(list(plan.S) + [1]), 1 << 27)
        self.buckets = backward_buckets(plan, bucket_elems)
        longest = max([(plan.F[u1] if u1 < plan.n_units else plan.P_pad) - plan.F[u0] for u0, u1 in self.buckets] + [1])
        self.bucket = B.rank_buffers(plan.n_ranks, longest, grad_dtype, plan.device)

    @property
    def bucket_bytes(self):
        return self.bucket.shape[0] * self.bucket.stride(0) * self.bucket.element_size()

    def view(self, u0, u1):
        end = self.plan.F[u1] if u1 < self.plan.n_units else self.plan.P_pad
        return self.bucket[:, :end - self.plan.F[u0]]

    def step(self, fill, master, m, v, hp, full=None, pshard=None, gshard=None, sqnorm_out=None, stream=None):
        clip = hp.max_norm > 0
        if clip and gshard is None:
            raise ValueError("a clipped step needs the fp32 gradient shard (gshard)")
        for u0, u1 in self.buckets:
            view = self.view(u0, u1)
            fill(u0, u1, view)
            if clip:
                B.zero_clip_reduce_units(self.plan, u0, u1, view, gshard, stream=stream)
            else:
                B.zero_step_units(self.plan, u0, u1, view, master, m, v, hp, full=full, pshard=pshard, stream=stream)
        if clip:
            B.zero_clip_finalize(self.plan, hp.max_norm, sqnorm_out, stream=stream)
            B.zero_adamw_shard_step_clipped(self.plan, gshard, master, m, v, hp, pshard=pshard, full=full,
                                            stream=stream)
