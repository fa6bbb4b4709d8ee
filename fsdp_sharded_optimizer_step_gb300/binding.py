"""Thin ctypes binding over the C ABI (include/zero.h), with the same names.

Argument marshalling only: tensors become device pointers, rank lists become
host pointer arrays, streams become cudaStream_t handles; every step of the
path runs in the CUDA library.  The binding checks what ctypes cannot (device,
dtype, contiguity, length of every tensor) so that a wrong tensor is refused on
the host instead of reaching a kernel.  There is no fallback: if the library
is not built this module raises.
"""
import ctypes as C
import os
from dataclasses import dataclass

import torch

from . import build as _build

ZERO_OK, ZERO_EINVAL, ZERO_ENOMEM, ZERO_ECUDA, ZERO_EALIGN, ZERO_ENOTATTACHED, ZERO_ERANGE = 0, -1, -2, -3, -4, -7, -8
ZERO_ENONFINITE, ZERO_ETIMEOUT = -5, -6
ZERO_F32, ZERO_BF16 = 0, 1
ZERO_MAX_RANKS = 64

_DTYPES = {torch.float32: ZERO_F32, torch.bfloat16: ZERO_BF16}


class ZeroError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = lib().zero_status_string(status).decode()
        extra = ""
        if status == ZERO_ECUDA:
            extra = f" (cudaError {lib().zero_last_cuda_error()})"
        super().__init__(f"{what}: {msg}{extra} [{status}]")


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("b1", C.c_float), ("b2", C.c_float), ("eps", C.c_float),
                ("wd", C.c_float), ("t", C.c_int32), ("max_norm", C.c_float)]


@dataclass
class AdamW:
    """zero_hparams: AdamW constants, 1-based step t, max_norm > 0 to clip."""
    lr: float = 0.01
    b1: float = 0.9
    b2: float = 0.95
    eps: float = 1e-8
    wd: float = 0.1
    t: int = 1
    max_norm: float = 0.0

    def c(self) -> Hparams:
        return Hparams(self.lr, self.b1, self.b2, self.eps, self.wd, int(self.t), self.max_norm)


_LIB = None
SYMBOLS = {}


def lib():
    """Loads the CUDA library (fails loudly when it is not built).  ZERO_LIB in the
    environment names another build of the same library (build.build_variant)."""
    global _LIB
    if _LIB is None:
        path = os.environ.get("ZERO_LIB") or _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: build it with "
                               "fsdp_sharded_optimizer_step_gb300.build.build() (or __graft_entry__.build())")
        L = C.CDLL(path)
        p, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
        pp = C.POINTER(C.c_void_p)
        sig = {
            "zero_plan_create": (C.c_int, [p, i32, i32, C.POINTER(C.c_void_p)]),
            "zero_plan_create_aligned": (C.c_int, [p, i32, i32, i32, C.POINTER(C.c_void_p)]),
            "zero_plan_align": (C.c_int, [p, p]),
            "zero_plan_destroy": (None, [p]),
            "zero_plan_query": (C.c_int, [p, p, p, p, p, p, p]),
            "zero_plan_counts": (C.c_int, [p, p, p, p]),
            "zero_plan_segments": (C.c_int, [p, p]),
            "zero_plan_local_segments": (C.c_int, [p, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
            "zero_plan_workspace_bytes": (C.c_int, [p, C.POINTER(C.c_size_t)]),
            "zero_plan_attach": (C.c_int, [p, p, C.c_size_t, p]),
            "zero_bias_corrections": (C.c_int, [i32, f32, f32, p, p]),
            "zero_reduce_scatter": (C.c_int, [p, pp, i32, pp, f32, p]),
            "zero_grad_sqnorm": (C.c_int, [p, pp, i32, p, p]),
            "zero_adamw_shard_step": (C.c_int, [p, pp, pp, pp, pp, pp, p, i32, p, p]),
            "zero_all_gather": (C.c_int, [p, pp, p, i32, i32, p]),
            "zero_all_gather_bf16": (C.c_int, [p, pp, p, i32, p]),
            "zero_step": (C.c_int, [p, pp, i32, pp, pp, pp, p, pp, i32, pp, p, p, i32, p]),
            "zero_grad_sqnorm_noalloc": (C.c_int, [pp, i32, i32, i64, p, p]),
            "zero_step_unit": (C.c_int, [p, i32, pp, i32, pp, pp, pp, p, pp, i32, p, p]),
            "zero_step_units": (C.c_int, [p, i32, i32, pp, i32, pp, pp, pp, p, pp, i32, p, p]),
            "zero_clip_reduce_units": (C.c_int, [p, i32, i32, pp, i32, pp, p]),
            "zero_reshard": (C.c_int, [p, p, pp, pp, i32, p]),
            "zero_all_gather_unit": (C.c_int, [p, i32, pp, p, i32, p]),
            "zero_reduce_scatter_unit": (C.c_int, [p, i32, pp, i32, pp, f32, p]),
            "zero_clip_reduce_unit": (C.c_int, [p, i32, pp, i32, pp, p]),
            "zero_clip_finalize": (C.c_int, [p, f32, p, p]),
            "zero_adamw_shard_step_clipped": (C.c_int, [p, pp, pp, pp, pp, pp, p, i32, p, i32, p]),
            "zero_offload_create": (C.c_int, [p, i32, i64, C.POINTER(C.c_void_p)]),
            "zero_offload_destroy": (None, [p]),
            "zero_offload_adamw": (C.c_int, [p, pp, pp, pp, pp, pp, p, i32, p, C.c_double, i32]),
            "zero_offload_step": (C.c_int, [p, pp, i32, pp, pp, pp, pp, pp, p, p, i32, p, p, p]),
            "zero_offload_timings": (C.c_int, [p, p]),
            "zero_offload_info": (C.c_int, [p, p, p]),
            "zero_plan_device_errors": (C.c_int, [p, p, p]),
            "zero_plan_check": (C.c_int, [p, p]),
            "zero_debug_drop_copy": (C.c_int, [i64]),
            "zero_status_string": (C.c_char_p, [C.c_int]),
            "zero_last_cuda_error": (C.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
            SYMBOLS[name] = fn
        _LIB = L
    return _LIB


def _check(status, what):
    if status != ZERO_OK:
        raise ZeroError(status, what)


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


# ------------------------------------------------------------------ plan
def zero_plan_create(unit_sizes, n_ranks):
    sizes = (C.c_int64 * len(unit_sizes))(*[int(s) for s in unit_sizes])
    h = C.c_void_p()
    _check(lib().zero_plan_create(sizes, len(unit_sizes), int(n_ranks), C.byref(h)), "zero_plan_create")
    return h


def zero_plan_create_aligned(unit_sizes, n_ranks, align):
    sizes = (C.c_int64 * len(unit_sizes))(*[int(s) for s in unit_sizes])
    h = C.c_void_p()
    _check(lib().zero_plan_create_aligned(sizes, len(unit_sizes), int(n_ranks), int(align), C.byref(h)),
           "zero_plan_create_aligned")
    return h


def zero_plan_align(handle):
    a = C.c_int32()
    _check(lib().zero_plan_align(handle, C.byref(a)), "zero_plan_align")
    return a.value


def zero_plan_destroy(handle):
    lib().zero_plan_destroy(handle)


def zero_plan_counts(handle):
    u, n, s = C.c_int32(), C.c_int32(), C.c_int64()
    _check(lib().zero_plan_counts(handle, C.byref(u), C.byref(n), C.byref(s)), "zero_plan_counts")
    return u.value, n.value, s.value


def zero_plan_query(handle):
    """Layout as python ints / lists: P_pad, H, F, Hoff, S, h."""
    U, _, _ = zero_plan_counts(handle)
    P, H = C.c_int64(), C.c_int64()
    arrs = [(C.c_int64 * max(U, 1))() for _ in range(4)]
    _check(lib().zero_plan_query(handle, C.byref(P), C.byref(H), *arrs), "zero_plan_query")
    F, Hoff, S, h = ([int(a[i]) for i in range(U)] for a in arrs)
    return dict(P_pad=P.value, H=H.value, F=F, Hoff=Hoff, S=S, h=h)


def zero_plan_segments(handle):
    """Launch table as a list of (full_pos, shard_pos, len, valid, rank, unit)."""
    _, _, nseg = zero_plan_counts(handle)
    out = (C.c_int64 * max(6 * nseg, 1))()
    _check(lib().zero_plan_segments(handle, out), "zero_plan_segments")
    return [tuple(out[6 * i:6 * i + 6]) for i in range(nseg)]


def zero_plan_local_segments(handle):
    """Unit-local launch table, in the layout of zero_plan_segments."""
    n = C.c_int64()
    _check(lib().zero_plan_local_segments(handle, C.byref(n), None), "zero_plan_local_segments")
    out = (C.c_int64 * max(6 * n.value, 1))()
    _check(lib().zero_plan_local_segments(handle, C.byref(n), out), "zero_plan_local_segments")
    return [tuple(out[6 * i:6 * i + 6]) for i in range(n.value)]


def zero_plan_workspace_bytes(handle):
    b = C.c_size_t()
    _check(lib().zero_plan_workspace_bytes(handle, C.byref(b)), "zero_plan_workspace_bytes")
    return b.value


def zero_plan_attach(handle, workspace: torch.Tensor, stream=None):
    _check(lib().zero_plan_attach(handle, C.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                                  _stream(stream, workspace.device)), "zero_plan_attach")


def zero_plan_device_errors(plan, stream=None):
    """Reads and clears the plan's device error word (0: every bounded wait completed)."""
    e = C.c_int32()
    _check(lib().zero_plan_device_errors(plan.handle, _stream(stream, plan.device), C.byref(e)),
           "zero_plan_device_errors")
    return e.value


def zero_plan_check(plan, stream=None):
    """Status of the device work queued on the plan since the last check (synchronises the stream):
    ZERO_OK, ZERO_ETIMEOUT (a bounded wait expired) or ZERO_ENONFINITE (a clipped step was skipped
    because its global norm was not finite).  Clears both conditions; argument errors raise."""
    rc = lib().zero_plan_check(plan.handle, _stream(stream, plan.device))
    if rc in (ZERO_OK, ZERO_ETIMEOUT, ZERO_ENONFINITE):
        return rc
    _check(rc, "zero_plan_check")


def zero_debug_drop_copy(tile):
    """Testing aid: the next pipelined launch drops the copies of one tile of its first segment (see include/zero.h)."""
    _check(lib().zero_debug_drop_copy(int(tile)), "zero_debug_drop_copy")


def zero_bias_corrections(t, b1=0.9, b2=0.95):
    bc1, bc2 = C.c_float(), C.c_float()
    _check(lib().zero_bias_corrections(int(t), b1, b2, C.byref(bc1), C.byref(bc2)), "zero_bias_corrections")
    return bc1.value, bc2.value


class ZeroPlan:
    """Owns a plan and its device workspace (a torch uint8 tensor on `device`).

    device=None builds the host-side plan only (layout queries work without a
    GPU; device calls then fail with ZERO_ENOTATTACHED).  align > 1 pads every
    unit to a multiple of n_ranks * align (zero_plan_create_aligned)."""

    def __init__(self, unit_sizes, n_ranks, device=None, stream=None, align=1):
        self.unit_sizes = [int(s) for s in unit_sizes]
        self.n_ranks = int(n_ranks)
        self.align = int(align)
        self.handle = (zero_plan_create(self.unit_sizes, self.n_ranks) if self.align == 1
                       else zero_plan_create_aligned(self.unit_sizes, self.n_ranks, self.align))
        q = zero_plan_query(self.handle)
        self.P_pad, self.H = q["P_pad"], q["H"]
        self.F, self.Hoff, self.S, self.h = q["F"], q["Hoff"], q["S"], q["h"]
        self.n_units, _, self.n_segments = zero_plan_counts(self.handle)
        self.device = None
        self.workspace = None
        if device is not None:
            device = torch.device(device)
            if device.type == "cuda" and device.index is None:
                device = torch.device("cuda", torch.cuda.current_device())
            self.device = device
            nbytes = zero_plan_workspace_bytes(self.handle)
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            zero_plan_attach(self.handle, self.workspace, stream)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _LIB is not None:
            zero_plan_destroy(h)
            self.handle = None


# ------------------------------------------------------------------ allocation helper
def rank_buffers(n_ranks, length, dtype, device, zero=False):
    """[n_ranks, length] view whose rows start 16-byte aligned (the row stride
    is padded to a multiple of 16 bytes), as the C ABI requires of every rank
    buffer."""
    per16 = 16 // torch.empty((), dtype=dtype).element_size()
    stride = (length + per16 - 1) // per16 * per16
    alloc = torch.zeros if zero else torch.empty
    return alloc(n_ranks, max(stride, 1), dtype=dtype, device=device)[:, :length]


# ------------------------------------------------------------------ tensor marshalling
def _rows(plan, x, length, what, dtypes):
    """A [N, length] tensor or a list of N 1-D tensors -> host array of N device pointers, dtype code."""
    if isinstance(x, torch.Tensor) and x.dim() == 2:
        # rows of one 2-D tensor: pointers from its row stride, no per-row tensor objects
        if x.shape[0] != plan.n_ranks:
            raise ValueError(f"{what}: expected {plan.n_ranks} rank buffers, got {x.shape[0]}")
        if x.device != plan.device:
            raise ValueError(f"{what}: tensor on {x.device}, plan on {plan.device}")
        if x.dtype not in dtypes:
            raise ValueError(f"{what}: dtype {x.dtype} not allowed")
        if x.shape[1] != length or (length > 1 and x.stride(1) != 1):
            raise ValueError(f"{what}: each rank buffer must be contiguous 1-D of {length} elements")
        if length == 0:  # nothing to address: null pointers, as for empty rows below
            return (C.c_void_p * plan.n_ranks)(), _DTYPES[x.dtype]
        base, step = x.data_ptr(), x.stride(0) * x.element_size()
        return (C.c_void_p * plan.n_ranks)(*[base + r * step for r in range(plan.n_ranks)]), _DTYPES[x.dtype]
    rows = list(x.unbind(0)) if isinstance(x, torch.Tensor) else list(x)
    if len(rows) != plan.n_ranks:
        raise ValueError(f"{what}: expected {plan.n_ranks} rank buffers, got {len(rows)}")
    dt = rows[0].dtype
    for r in rows:
        if r.device != plan.device:
            raise ValueError(f"{what}: tensor on {r.device}, plan on {plan.device}")
        if r.dtype != dt or dt not in dtypes:
            raise ValueError(f"{what}: dtype {r.dtype} not allowed")
        if r.dim() != 1 or not r.is_contiguous() or r.numel() != length:
            raise ValueError(f"{what}: each rank buffer must be contiguous 1-D of {length} elements")
    arr = (C.c_void_p * len(rows))(*[r.data_ptr() for r in rows])
    return arr, _DTYPES[dt]


def _one(plan, x, length, what, dtypes):
    if x.device != plan.device or x.dtype not in dtypes or not x.is_contiguous() or x.numel() != length:
        raise ValueError(f"{what}: need a contiguous {length}-element tensor of {dtypes} on {plan.device}")
    return C.c_void_p(x.data_ptr()), _DTYPES[x.dtype]


_G = (torch.bfloat16, torch.float32)
_F = (torch.float32,)


def zero_reduce_scatter(plan, grads, gshard, coef=1.0, stream=None):
    g, gd = _rows(plan, grads, plan.P_pad, "grads", _G)
    gs, _ = _rows(plan, gshard, plan.H, "gshard", _F)
    _check(lib().zero_reduce_scatter(plan.handle, g, gd, gs, float(coef), _stream(stream, plan.device)),
           "zero_reduce_scatter")


def zero_grad_sqnorm(plan, grads, sqnorm_out, stream=None):
    g, gd = _rows(plan, grads, plan.P_pad, "grads", _G)
    if sqnorm_out.device != plan.device or sqnorm_out.dtype != torch.float64 or sqnorm_out.numel() < 1:
        raise ValueError("sqnorm_out: need a float64 tensor on the plan's device")
    _check(lib().zero_grad_sqnorm(plan.handle, g, gd, C.c_void_p(sqnorm_out.data_ptr()), _stream(stream, plan.device)),
           "zero_grad_sqnorm")


def _outputs(plan, full, pshard):
    pdt = None
    fp = None
    if full is not None:
        fp, pdt = _one(plan, full, plan.P_pad, "full", _G)
    ps = None
    if pshard is not None:
        ps, d = _rows(plan, pshard, plan.H, "pshard", _G)
        if pdt is not None and d != pdt:
            raise ValueError("full and pshard must have the same dtype")
        pdt = d
    return fp, ps, (ZERO_BF16 if pdt is None else pdt)


def zero_adamw_shard_step(plan, gshard, master, m, v, hp: AdamW, pshard=None, full=None, stream=None):
    gs, _ = _rows(plan, gshard, plan.H, "gshard", _F)
    W, _ = _rows(plan, master, plan.H, "master", _F)
    M, _ = _rows(plan, m, plan.H, "m", _F)
    V, _ = _rows(plan, v, plan.H, "v", _F)
    fp, ps, pdt = _outputs(plan, full, pshard)
    c = hp.c()
    _check(lib().zero_adamw_shard_step(plan.handle, gs, W, M, V, ps, fp, pdt, C.byref(c), _stream(stream, plan.device)),
           "zero_adamw_shard_step")


def zero_all_gather(plan, shards, full, unit=-1, stream=None):
    s, sd = _rows(plan, shards, plan.H, "shards", _G)
    fp, fd = _one(plan, full, plan.P_pad, "full", _G)
    if sd != fd:
        raise ValueError("shards and full must have the same dtype")
    _check(lib().zero_all_gather(plan.handle, s, fp, fd, int(unit), _stream(stream, plan.device)), "zero_all_gather")


def zero_all_gather_bf16(plan, shards, full, unit=-1, stream=None):
    s, sd = _rows(plan, shards, plan.H, "shards", (torch.bfloat16,))
    fp, _ = _one(plan, full, plan.P_pad, "full", (torch.bfloat16,))
    _check(lib().zero_all_gather_bf16(plan.handle, s, fp, int(unit), _stream(stream, plan.device)),
           "zero_all_gather_bf16")


def zero_step(plan, grads, master, m, v, hp: AdamW, full=None, pshard=None, gshard_ws=None, sqnorm_out=None,
              unit=-1, stream=None):
    """The fused sharded step (see include/zero.h)."""
    g, gd = _rows(plan, grads, plan.P_pad, "grads", _G)
    W, _ = _rows(plan, master, plan.H, "master", _F)
    M, _ = _rows(plan, m, plan.H, "m", _F)
    V, _ = _rows(plan, v, plan.H, "v", _F)
    fp, ps, pdt = _outputs(plan, full, pshard)
    gs = None
    if gshard_ws is not None:
        gs, _ = _rows(plan, gshard_ws, plan.H, "gshard_ws", _F)
    sq = None
    if sqnorm_out is not None:
        if sqnorm_out.device != plan.device or sqnorm_out.dtype != torch.float64:
            raise ValueError("sqnorm_out: need a float64 tensor on the plan's device")
        sq = C.c_void_p(sqnorm_out.data_ptr())
    c = hp.c()
    _check(lib().zero_step(plan.handle, g, gd, W, M, V, fp, ps, pdt, gs, C.byref(c), sq, int(unit),
                           _stream(stream, plan.device)), "zero_step")


class UnitSteps:
    """The unclipped fused step as one zero_step launch per unit, with the tensors
    checked and marshalled once: a per-unit loop from Python then costs one direct
    C call per unit instead of a full binding call (rank-pointer arrays, dtype and
    shape checks) each time.  The tensors must stay alive and in place while the
    object is used."""

    def __init__(self, plan, grads, master, m, v, full=None, pshard=None):
        self.plan = plan
        self._g, self._gd = _rows(plan, grads, plan.P_pad, "grads", _G)
        self._w, _ = _rows(plan, master, plan.H, "master", _F)
        self._m, _ = _rows(plan, m, plan.H, "m", _F)
        self._v, _ = _rows(plan, v, plan.H, "v", _F)
        self._fp, self._ps, self._pdt = _outputs(plan, full, pshard)
        self._keep = (grads, master, m, v, full, pshard)
        self._fn = lib().zero_step

    def step(self, hp: AdamW, units=None, stream=None):
        """Updates `units` (default: every unit, in order), one launch each."""
        if hp.max_norm > 0:
            raise ValueError("a clipped step needs every unit at once: use zero_step")
        c = hp.c()
        st = _stream(stream, self.plan.device)
        h, fn = self.plan.handle, self._fn
        for u in (range(self.plan.n_units) if units is None else units):
            rc = fn(h, self._g, self._gd, self._w, self._m, self._v, self._fp, self._ps, self._pdt, None, C.byref(c),
                    None, u, st)
            if rc != ZERO_OK:
                raise ZeroError(rc, "zero_step")


def zero_grad_sqnorm_noalloc(grads, sqnorm_out, stream=None):
    """Sum of squares of the averaged gradient over flat rank buffers, with no
    device allocation (see include/zero.h); padding entries must hold 0."""
    rows = list(grads.unbind(0)) if isinstance(grads, torch.Tensor) else list(grads)
    n = rows[0].numel()
    dev = rows[0].device
    for r in rows:
        if r.device != dev or r.dtype != rows[0].dtype or r.dim() != 1 or not r.is_contiguous() or r.numel() != n:
            raise ValueError("grads: rank buffers must be contiguous 1-D tensors of one dtype, length and device")
    if rows[0].dtype not in _DTYPES:
        raise ValueError(f"grads: dtype {rows[0].dtype} not allowed")
    if sqnorm_out.device != dev or sqnorm_out.dtype != torch.float64:
        raise ValueError("sqnorm_out: need a float64 tensor on the gradients' device")
    if dev.type != "cuda":
        raise ValueError("grads: need CUDA tensors")
    arr = (C.c_void_p * len(rows))(*[r.data_ptr() for r in rows])
    with torch.cuda.device(dev):  # the library works on the current device
        _check(lib().zero_grad_sqnorm_noalloc(arr, len(rows), _DTYPES[rows[0].dtype], n,
                                              C.c_void_p(sqnorm_out.data_ptr()), _stream(stream, dev)),
               "zero_grad_sqnorm_noalloc")


def zero_step_unit(plan, unit, grads_unit, master, m, v, hp: AdamW, full=None, pshard=None, stream=None):
    """The fused step for one unit from unit-local gradient buffers (rank q's S_u positions of the unit)."""
    g, gd = _rows(plan, grads_unit, plan.S[unit], "grads_unit", _G)
    W, _ = _rows(plan, master, plan.H, "master", _F)
    M, _ = _rows(plan, m, plan.H, "m", _F)
    V, _ = _rows(plan, v, plan.H, "v", _F)
    fp, ps, pdt = _outputs(plan, full, pshard)
    c = hp.c()
    _check(lib().zero_step_unit(plan.handle, int(unit), g, gd, W, M, V, fp, ps, pdt, C.byref(c),
                                _stream(stream, plan.device)), "zero_step_unit")


def _bucket_len(plan, u0, u1):
    if not (0 <= u0 < u1 <= plan.n_units):
        raise ValueError(f"unit range [{u0}, {u1}) outside [0, {plan.n_units})")
    return (plan.F[u1] if u1 < plan.n_units else plan.P_pad) - plan.F[u0]


def zero_step_units(plan, u0, u1, grads_bucket, master, m, v, hp: AdamW, full=None, pshard=None, stream=None):
    """The fused step for units [u0, u1) from bucket-local gradient buffers (rank q's padded
    positions F_u0 .. F_u1 - 1), one launch."""
    g, gd = _rows(plan, grads_bucket, _bucket_len(plan, u0, u1), "grads_bucket", _G)
    W, _ = _rows(plan, master, plan.H, "master", _F)
    M, _ = _rows(plan, m, plan.H, "m", _F)
    V, _ = _rows(plan, v, plan.H, "v", _F)
    fp, ps, pdt = _outputs(plan, full, pshard)
    c = hp.c()
    _check(lib().zero_step_units(plan.handle, int(u0), int(u1), g, gd, W, M, V, fp, ps, pdt, C.byref(c),
                                 _stream(stream, plan.device)), "zero_step_units")


def zero_clip_reduce_units(plan, u0, u1, grads_bucket, gshard, stream=None):
    """Clipped step, pass 1 for units [u0, u1) from a bucket-local gradient buffer."""
    g, gd = _rows(plan, grads_bucket, _bucket_len(plan, u0, u1), "grads_bucket", _G)
    gs, _ = _rows(plan, gshard, plan.H, "gshard", _F)
    _check(lib().zero_clip_reduce_units(plan.handle, int(u0), int(u1), g, gd, gs, _stream(stream, plan.device)),
           "zero_clip_reduce_units")


def zero_reduce_scatter_unit(plan, unit, grads_unit, gshard, coef=1.0, stream=None):
    """zero_reduce_scatter for one unit from unit-local gradient buffers."""
    g, gd = _rows(plan, grads_unit, plan.S[unit], "grads_unit", _G)
    gs, _ = _rows(plan, gshard, plan.H, "gshard", _F)
    _check(lib().zero_reduce_scatter_unit(plan.handle, int(unit), g, gd, gs, float(coef), _stream(stream, plan.device)),
           "zero_reduce_scatter_unit")


def zero_clip_reduce_unit(plan, unit, grads_unit, gshard, stream=None):
    """Clipped step, pass 1 for one unit (see include/zero.h): averaged gradient shard + sums of squares."""
    g, gd = _rows(plan, grads_unit, plan.S[unit], "grads_unit", _G)
    gs, _ = _rows(plan, gshard, plan.H, "gshard", _F)
    _check(lib().zero_clip_reduce_unit(plan.handle, int(unit), g, gd, gs, _stream(stream, plan.device)),
           "zero_clip_reduce_unit")


def zero_clip_finalize(plan, max_norm, sqnorm_out=None, stream=None):
    """Clipped step, pass 2: S over every unit and the clip coefficient, on the device."""
    sq = None
    if sqnorm_out is not None:
        if sqnorm_out.device != plan.device or sqnorm_out.dtype != torch.float64 or sqnorm_out.numel() < 1:
            raise ValueError("sqnorm_out: need a float64 tensor on the plan's device")
        sq = C.c_void_p(sqnorm_out.data_ptr())
    _check(lib().zero_clip_finalize(plan.handle, float(max_norm), sq, _stream(stream, plan.device)),
           "zero_clip_finalize")


def zero_adamw_shard_step_clipped(plan, gshard, master, m, v, hp: AdamW, pshard=None, full=None, unit=-1,
                                  stream=None):
    """Clipped step, pass 3: the shard update scaled by the device coefficient (all units or one)."""
    gs, _ = _rows(plan, gshard, plan.H, "gshard", _F)
    W, _ = _rows(plan, master, plan.H, "master", _F)
    M, _ = _rows(plan, m, plan.H, "m", _F)
    V, _ = _rows(plan, v, plan.H, "v", _F)
    fp, ps, pdt = _outputs(plan, full, pshard)
    c = hp.c()
    _check(lib().zero_adamw_shard_step_clipped(plan.handle, gs, W, M, V, ps, fp, pdt, C.byref(c), int(unit),
                                               _stream(stream, plan.device)), "zero_adamw_shard_step_clipped")


def zero_reshard(plan_from, plan_to, src, dst, stream=None):
    """Remap per-rank shards from plan_from's layout ([N, H]) to plan_to's ([N', H'])."""
    s, sd = _rows(plan_from, src, plan_from.H, "src", _G)
    d, dd = _rows(plan_to, dst, plan_to.H, "dst", _G)
    if sd != dd:
        raise ValueError("src and dst must have the same dtype")
    _check(lib().zero_reshard(plan_from.handle, plan_to.handle, s, d, sd, _stream(stream, plan_to.device)),
           "zero_reshard")


def zero_all_gather_unit(plan, unit, shards, dst_unit, stream=None):
    """Gather one unit's params from the rank shards into a unit-sized buffer (S_u elements)."""
    s, sd = _rows(plan, shards, plan.H, "shards", _G)
    dp, dd = _one(plan, dst_unit, plan.S[unit], "dst_unit", _G)
    if sd != dd:
        raise ValueError("shards and dst_unit must have the same dtype")
    _check(lib().zero_all_gather_unit(plan.handle, int(unit), s, dp, sd, _stream(stream, plan.device)),
           "zero_all_gather_unit")


# ------------------------------------------------------------------ ZeRO-Offload (host-resident state)
def _host_rows(plan, x, length, what, dtypes):
    """A [N, length] HOST tensor (or N 1-D host tensors) -> host array of N host pointers, dtype code."""
    rows = list(x.unbind(0)) if isinstance(x, torch.Tensor) and x.dim() == 2 else list(x)
    if len(rows) != plan.n_ranks:
        raise ValueError(f"{what}: expected {plan.n_ranks} rank arrays, got {len(rows)}")
    dt = rows[0].dtype
    for r in rows:
        if r.device.type != "cpu":
            raise ValueError(f"{what}: host (CPU) tensors expected, got {r.device}")
        if r.dtype != dt or dt not in dtypes:
            raise ValueError(f"{what}: dtype {r.dtype} not allowed")
        if r.dim() != 1 or not r.is_contiguous() or r.numel() != length:
            raise ValueError(f"{what}: each rank array must be contiguous 1-D of {length} elements")
    return (C.c_void_p * len(rows))(*[r.data_ptr() if r.numel() else 0 for r in rows]), _DTYPES[dt]


def _host_one(x, length, what, dtypes):
    if x.device.type != "cpu" or x.dtype not in dtypes or not x.is_contiguous() or x.numel() != length:
        raise ValueError(f"{what}: need a contiguous {length}-element host tensor of {dtypes}")
    return C.c_void_p(x.data_ptr()), _DTYPES[x.dtype]


def zero_offload_create(plan, n_threads=0, batch_min=0):
    h = C.c_void_p()
    _check(lib().zero_offload_create(plan.handle, int(n_threads), int(batch_min), C.byref(h)), "zero_offload_create")
    return h


def zero_offload_destroy(handle):
    lib().zero_offload_destroy(handle)


def zero_offload_adamw(eng, gshard_h, master_h, m_h, v_h, hp: AdamW, full_h=None, pshard_h=None, sqnorm=0.0, unit=-1):
    """The host-core update alone on host tensors (see include/zero.h); returns the status
    (ZERO_OK, or ZERO_ENONFINITE when clipping with a non-finite S); other errors raise."""
    plan = eng.plan
    gs, _ = _host_rows(plan, gshard_h, plan.H, "gshard_h", _F)
    W, _ = _host_rows(plan, master_h, plan.H, "master_h", _F)
    M, _ = _host_rows(plan, m_h, plan.H, "m_h", _F)
    V, _ = _host_rows(plan, v_h, plan.H, "v_h", _F)
    pdt = None
    fp = None
    if full_h is not None:
        fp, pdt = _host_one(full_h, plan.P_pad, "full_h", _G)
    ps = None
    if pshard_h is not None:
        ps, d = _host_rows(plan, pshard_h, plan.H, "pshard_h", _G)
        if pdt is not None and d != pdt:
            raise ValueError("full_h and pshard_h must have the same dtype")
        pdt = d
    c = hp.c()
    rc = lib().zero_offload_adamw(eng.handle, gs, W, M, V, ps, fp, ZERO_BF16 if pdt is None else pdt, C.byref(c),
                                  float(sqnorm), int(unit))
    if rc not in (ZERO_OK, ZERO_ENONFINITE):
        _check(rc, "zero_offload_adamw")
    return rc


def zero_offload_step(eng, grads, gshard_dev, gshard_h, master_h, m_h, v_h, full_h, hp: AdamW, full_dev=None,
                      stream=None):
    """The offloaded step (see include/zero.h).  grads, gshard_dev: device [N, P_pad] / [N, H];
    gshard_h, master_h, m_h, v_h: host [N, H] (pinned for overlap); full_h: host [P_pad];
    full_dev: device [P_pad] or None.  Returns (status, S): status ZERO_OK or ZERO_ENONFINITE
    (clipped step skipped), S the global sum of squares when clipping (else None)."""
    plan = eng.plan
    g, gd = _rows(plan, grads, plan.P_pad, "grads", _G)
    gsd, _ = _rows(plan, gshard_dev, plan.H, "gshard_dev", _F)
    gsh, _ = _host_rows(plan, gshard_h, plan.H, "gshard_h", _F)
    W, _ = _host_rows(plan, master_h, plan.H, "master_h", _F)
    M, _ = _host_rows(plan, m_h, plan.H, "m_h", _F)
    V, _ = _host_rows(plan, v_h, plan.H, "v_h", _F)
    fh, pdt = _host_one(full_h, plan.P_pad, "full_h", _G)
    fd = None
    if full_dev is not None:
        fd, d = _one(plan, full_dev, plan.P_pad, "full_dev", _G)
        if d != pdt:
            raise ValueError("full_h and full_dev must have the same dtype")
    c = hp.c()
    S = C.c_double(float("nan"))
    with torch.cuda.device(plan.device):
        rc = lib().zero_offload_step(eng.handle, g, gd, gsd, gsh, W, M, V, fh, fd, pdt, C.byref(c), C.byref(S),
                                     _stream(stream, plan.device))
    if rc not in (ZERO_OK, ZERO_ENONFINITE):
        _check(rc, "zero_offload_step")
    return rc, (S.value if hp.max_norm > 0 else None)


def zero_offload_info(eng):
    """(host worker threads, pipeline batches) of an engine."""
    t, b = C.c_int32(), C.c_int64()
    _check(lib().zero_offload_info(eng.handle, C.byref(t), C.byref(b)), "zero_offload_info")
    return t.value, b.value


def zero_offload_timings(eng):
    """Last step's timings (ms): call, waiting for gradient slices, host update, device time to
    the last param copy, device time to the last gradient slice (see include/zero.h)."""
    ms = (C.c_double * 5)()
    _check(lib().zero_offload_timings(eng.handle, ms), "zero_offload_timings")
    return dict(call_ms=ms[0], wait_ms=ms[1], update_ms=ms[2], device_to_params_ms=ms[3],
                device_to_grads_ms=ms[4])


class OffloadEngine:
    """Owns a zero_offload engine for a plan (host worker threads; copy streams on first step)."""

    def __init__(self, plan, n_threads=0, batch_min=0):
        self.plan = plan  # the engine keeps a pointer to the plan: hold it as long
        self.handle = zero_offload_create(plan, n_threads, batch_min)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _LIB is not None:
            zero_offload_destroy(h)
            self.handle = None
