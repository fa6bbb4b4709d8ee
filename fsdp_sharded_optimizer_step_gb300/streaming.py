"""The sharded step with the gradients in pinned host memory, streamed unit by unit.

Orchestration only (host-to-device and device-to-host copies on their own
streams, ordered by events); every step of the update runs in the CUDA library
through zero_step_unit.  While the update of unit u runs on the compute
stream, the N rank slices of unit u+1 are copied into the next staging buffer,
and the gathered params of finished units are copied back, so a step costs
about the time of its host transfers instead of transfers plus update.
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

    def step(self, host_grads, master, m, v, hp, full, host_full=None, stream=None):
        """host_grads: [N, P_pad] pinned host tensor (or N rows); full: device params (P_pad);
        host_full: optional pinned host tensor receiving the gathered params."""
        plan, N = self.plan, self.N
        compute = stream if stream is not None else torch.cuda.current_stream(self.dev)
        start = torch.cuda.Event()
        start.record(compute)
        self.copy_in.wait_event(start)
        self.copy_out.wait_event(start)
        nb = len(self.staging)
        for b in range(nb):
            self.free[b].record(compute)
        done = torch.cuda.Event()
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
            B.zero_step_unit(plan, u, buf, master, m, v, hp, full=full, stream=compute)
            self.free[b].record(compute)
            if host_full is not None:
                done.record(compute)
                self.copy_out.wait_event(done)
                with torch.cuda.stream(self.copy_out):
                    host_full[F:F + S].copy_(full[F:F + S], non_blocking=True)
                done = torch.cuda.Event()
        end = torch.cuda.Event()
        end.record(self.copy_out)
        compute.wait_event(end)
