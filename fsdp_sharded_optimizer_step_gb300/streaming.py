"""The sharded step with the gradients in pinned host memory, streamed unit by unit.

Orchestration only (host-to-device and device-to-host copies on their own
streams, ordered by events); every step of the update runs in the CUDA library.
While unit u is processed on the compute stream, the N rank slices of unit
u+1 are copied into the next staging buffer, and the gathered params of
finished units are copied back, so a step costs about the time of its host
transfers instead of transfers plus update.  step: zero_step_unit per unit.
step_clipped: the clipped step, whose global norm needs every unit before any
update: zero_clip_reduce_unit per unit as the gradients arrive (averaged
gradient shard + sums of squares), zero_clip_finalize, then
zero_adamw_shard_step_clipped per unit while finished units' params go back.
Staging: n_buffers x N x max(S_u) gradient elements on the device.
"""
import torch

from . import binding as B


class HostStreamedStep:
    def __init__(self, plan, grad_dtype, n_buffers=2):
        self.plan = plan
        self.dev = plan.device
        self.N = plan.n_ranks
        max_s = max([s for s in plan.S] + [1])
        self.staging = [B.rank_buffers(self.N, max_s, grad_dtype, self.dev) for _ in range(n_buffers)]
        self.copy_in = torch.cuda.Stream(self.dev)
        self.copy_out = torch.cuda.Stream(self.dev)
        self.free = [torch.cuda.Event() for _ in range(n_buffers)]    # staging buffer b may be overwritten
        self.landed = [torch.cuda.Event() for _ in range(n_buffers)]  # staging buffer b holds its unit

    def _begin(self, compute):
        start = torch.cuda.Event()
        start.record(compute)
        self.copy_in.wait_event(start)
        self.copy_out.wait_event(start)
        for ev in self.free:
            ev.record(compute)

    def _streamed_units(self, host_grads, compute, work):
        """Copies every unit's rank slices in (double-buffered) and calls work(u, rows) on the
        compute stream once they have landed."""
        plan, N, nb = self.plan, self.N, len(self.staging)
        for u in range(plan.n_units):
            F, S = plan.F[u], plan.S[u]
            if S == 0:
                continue
            b = u % nb
            buf = self.staging[b][:, :S]
            with torch.cuda.stream(self.copy_in):
                self.copy_in.wait_event(self.free[b])
                for q in range(N):
                    buf[q].copy_(host_grads[q][F:F + S], non_blocking=True)
                self.landed[b].record(self.copy_in)
            compute.wait_event(self.landed[b])
            work(u, buf)
            self.free[b].record(compute)

    def _copy_back(self, u, full, host_full, compute):
        if host_full is None:
            return
        F, S = self.plan.F[u], self.plan.S[u]
        done = torch.cuda.Event()
        done.record(compute)
        self.copy_out.wait_event(done)
        with torch.cuda.stream(self.copy_out):
            host_full[F:F + S].copy_(full[F:F + S], non_blocking=True)

    def _end(self, compute):
        end = torch.cuda.Event()
        end.record(self.copy_out)
        compute.wait_event(end)

    def step(self, host_grads, master, m, v, hp, full, host_full=None, stream=None):
        """host_grads: [N, P_pad] pinned host tensor (or N rows); full: device params (P_pad);
        host_full: optional pinned host tensor receiving the gathered params."""
        compute = stream if stream is not None else torch.cuda.current_stream(self.dev)
        self._begin(compute)

        def update(u, rows):
            B.zero_step_unit(self.plan, u, rows, master, m, v, hp, full=full, stream=compute)
            self._copy_back(u, full, host_full, compute)

        self._streamed_units(host_grads, compute, update)
        self._end(compute)

    def step_clipped(self, host_grads, gshard, master, m, v, hp, full, host_full=None, sqnorm_out=None,
                     stream=None):
        """The clipped step (hp.max_norm > 0); gshard: the [N, H] fp32 gradient shard workspace;
        sqnorm_out: optional float64 device tensor receiving S.  Equal to a clipped zero_step."""
        compute = stream if stream is not None else torch.cuda.current_stream(self.dev)
        self._begin(compute)
        self._streamed_units(host_grads, compute,
                             lambda u, rows: B.zero_clip_reduce_unit(self.plan, u, rows, gshard, stream=compute))
        B.zero_clip_finalize(self.plan, hp.max_norm, sqnorm_out, stream=compute)
        for u in range(self.plan.n_units):
            if self.plan.S[u] == 0:
                continue
            B.zero_adamw_shard_step_clipped(self.plan, gshard, master, m, v, hp, full=full, unit=u, stream=compute)
            self._copy_back(u, full, host_full, compute)
        self._end(compute)
