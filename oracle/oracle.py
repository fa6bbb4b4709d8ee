"""ctypes wrapper over the C oracle (oracle/zero_oracle.c).

TEST INFRASTRUCTURE ONLY.  Arrays are numpy; bf16 values travel as uint16 bit
patterns.  Nothing here does arithmetic of the method: every value comes from
the C oracle.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
OK, EINVAL, ENONFINITE = 0, -1, -5


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("b1", C.c_float), ("b2", C.c_float), ("eps", C.c_float),
                ("wd", C.c_float), ("t", C.c_int32), ("max_norm", C.c_float)]


def hparams(lr=0.01, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, t=1, max_norm=0.0) -> Hparams:
    """AdamW constants of the pages' toy ("ZeRO and FSDP sharding", Code) as defaults."""
    return Hparams(lr, b1, b2, eps, wd, t, max_norm)


_lib = None


def lib():
    global _lib
    if _lib is None:
        # ZERO_ORACLE_LIB lets the mutation test load a deliberately broken copy
        _lib = C.CDLL(os.environ.get("ZERO_ORACLE_LIB") or _build.build())
        p, i32, i64, f32, f64 = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_double
        sig = {
            "orc_plan": (C.c_int, [p, i32, i32, i32, p, p, p, p, p]),
            "orc_shard_map": (C.c_int, [p, i32, i32, i32, p]),
            "orc_pad_mask": (C.c_int, [p, i32, i32, i32, p]),
            "orc_locate": (C.c_int, [p, i32, i32, i32, i64, p, p, p, p]),
            "orc_reshard": (C.c_int, [p, i32, i32, i32, i32, i32, i32, p, p]),
            "orc_avg_grad_array": (C.c_int, [i64, i32, p, i32, p, p]),
            "orc_bf16_rne": (C.c_uint16, [f32]),
            "orc_bf16_rne_array": (None, [i64, p, p]),
            "orc_bf16_to_f32": (f32, [C.c_uint16]),
            "orc_bias_corrections": (C.c_int, [i32, f32, f32, p, p]),
            "orc_sqacc_bytes": (i32, []),
            "orc_sqacc_add_square": (None, [p, f32]),
            "orc_sqacc_result": (f64, [p]),
            "orc_sqacc_merge": (None, [p, p]),
            "orc_sqnorm_accumulate": (C.c_int, [p, i64, i32, p, i32, p]),
            "orc_clip_coef": (f32, [f64, f32]),
            "orc_adamw": (C.c_int, [i64, i32, p, i32, p, p, p, p, p, i32, p, i32, f32]),
            "orc_step": (C.c_int, [i64, i32, p, i32, p, p, p, p, p, i32, p, p]),
            "orc_toy_zero2_threads": (C.c_int, [i32, i64, i32, p, p, p, p]),
            "orc_toy_unsharded": (C.c_int, [i32, i64, i32, p, p, p, p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(rc, what):
    if rc != OK:
        raise RuntimeError(f"oracle {what} returned {rc}")


# ---------------------------------------------------------------- layout
class Plan:
    """Integer layout of the padded flat buffers (S, h, F, Hoff, P_pad, H); align > 1
    pads every unit to a multiple of N*align (slice lengths multiples of align)."""

    def __init__(self, sizes, n_ranks, align=1):
        self.sizes = np.ascontiguousarray(sizes, dtype=np.int64)
        self.N = int(n_ranks)
        self.align = int(align)
        U = len(self.sizes)
        self.S = np.zeros(U, np.int64)
        self.h = np.zeros(U, np.int64)
        self.F = np.zeros(U, np.int64)
        self.Hoff = np.zeros(U, np.int64)
        tot = np.zeros(2, np.int64)
        _check(lib().orc_plan(_ptr(self.sizes), U, self.N, self.align, _ptr(self.S), _ptr(self.h), _ptr(self.F),
                              _ptr(self.Hoff), _ptr(tot)), "plan")
        self.P_pad, self.H = int(tot[0]), int(tot[1])

    def shard_map(self):
        """map[r, p] = full-buffer position stored at position p of rank r's shard."""
        out = np.zeros(self.N * self.H, np.int64)
        _check(lib().orc_shard_map(_ptr(self.sizes), len(self.sizes), self.N, self.align, _ptr(out)), "shard_map")
        return out.reshape(self.N, self.H)

    def locate(self, pos):
        """(rank, shard position, is_pad) of each full-buffer position in `pos`."""
        pos = np.ascontiguousarray(pos, np.int64)
        rank = np.zeros(pos.size, np.int32)
        spos = np.zeros(pos.size, np.int64)
        pad = np.zeros(pos.size, np.uint8)
        _check(lib().orc_locate(_ptr(self.sizes), len(self.sizes), self.N, self.align, pos.size, _ptr(pos), _ptr(rank),
                                _ptr(spos),
                                _ptr(pad)), "locate")
        return rank, spos, pad

    def pad_mask(self):
        out = np.zeros(self.P_pad, np.uint8)
        _check(lib().orc_pad_mask(_ptr(self.sizes), len(self.sizes), self.N, self.align, _ptr(out)), "pad_mask")
        return out


def reshard(sizes, n_from, n_to, src, align_from=1, align_to=1):
    """src: [n_from, H_from] array (float32 or uint16 bits) -> [n_to, H_to] in the target layout."""
    sizes = np.ascontiguousarray(sizes, np.int64)
    src = np.ascontiguousarray(src)
    H_to = Plan(sizes, n_to, align_to).H
    dst = np.zeros((n_to, H_to), src.dtype)
    sp = (C.c_void_p * n_from)(*[src[r].ctypes.data for r in range(n_from)])
    dp = (C.c_void_p * n_to)(*[dst[r].ctypes.data for r in range(n_to)])
    _check(lib().orc_reshard(_ptr(sizes), len(sizes), n_from, align_from, n_to, align_to, src.dtype.itemsize, sp, dp),
           "reshard")
    return dst


# ---------------------------------------------------------------- scalars
def bf16_rne(x: float) -> int:
    return int(lib().orc_bf16_rne(float(x)))


def bf16_rne_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32).ravel()
    out = np.empty(x.size, np.uint16)
    lib().orc_bf16_rne_array(x.size, _ptr(x), _ptr(out))
    return out


def bias_corrections(t, b1=0.9, b2=0.95):
    bc1, bc2 = C.c_float(), C.c_float()
    _check(lib().orc_bias_corrections(t, b1, b2, C.byref(bc1), C.byref(bc2)), "bias_corrections")
    return np.float32(bc1.value), np.float32(bc2.value)


def clip_coef(S: float, max_norm: float) -> np.float32:
    return np.float32(lib().orc_clip_coef(float(S), float(max_norm)))


# ---------------------------------------------------------------- norm
class SqAcc:
    """Exact accumulator of squares (streamed over chunks of positions)."""

    def __init__(self):
        self.buf = (C.c_uint8 * lib().orc_sqacc_bytes())()

    def add_square(self, g: float):
        lib().orc_sqacc_add_square(self.buf, float(g))

    def add_avg_grad(self, grads, gdtype, pad=None):
        grads = [np.ascontiguousarray(g) for g in grads]
        n = grads[0].size
        arr = (C.c_void_p * len(grads))(*[g.ctypes.data for g in grads])
        _check(lib().orc_sqnorm_accumulate(self.buf, n, len(grads), arr, gdtype, _ptr(pad)), "sqnorm")

    def merge(self, other: "SqAcc"):
        """Adds another accumulator's exact sum into this one."""
        lib().orc_sqacc_merge(self.buf, other.buf)

    def result(self) -> float:
        return lib().orc_sqacc_result(self.buf)


def sqnorm(grads, gdtype, pad=None) -> float:
    a = SqAcc()
    a.add_avg_grad(grads, gdtype, pad)
    return a.result()


# ---------------------------------------------------------------- update
def avg_grad(grads, gdtype, pad=None):
    """The rank-ordered averaged gradient at every given position."""
    grads, arr = _grad_ptrs(grads, gdtype)
    out = np.zeros(grads[0].size, np.float32)
    _check(lib().orc_avg_grad_array(out.size, len(grads), arr, gdtype, _ptr(pad), _ptr(out)), "avg_grad")
    return out


def _grad_ptrs(grads, gdtype):
    want = np.float32 if gdtype == F32 else np.uint16
    grads = [np.ascontiguousarray(g, dtype=want) for g in grads]
    return grads, (C.c_void_p * len(grads))(*[g.ctypes.data for g in grads])


def adamw(grads, gdtype, w, m, v, hp, pdtype=BF16, pad=None, clip=False, coef=1.0):
    """In place on w, m, v (float32 arrays of n); returns the cast output."""
    grads, arr = _grad_ptrs(grads, gdtype)
    n = w.size
    out = np.zeros(n, np.float32 if pdtype == F32 else np.uint16)
    _check(lib().orc_adamw(n, len(grads), arr, gdtype, _ptr(pad), _ptr(w), _ptr(m), _ptr(v), _ptr(out),
                           pdtype, C.byref(hp), int(bool(clip)), float(coef)), "adamw")
    return out


def step(grads, gdtype, w, m, v, hp, pdtype=BF16, pad=None):
    """Whole step (norm, clip, update) over the given positions; returns (rc, out, S)."""
    grads, arr = _grad_ptrs(grads, gdtype)
    n = w.size
    out = np.zeros(n, np.float32 if pdtype == F32 else np.uint16)
    S = C.c_double(float("nan"))
    rc = lib().orc_step(n, len(grads), arr, gdtype, _ptr(pad), _ptr(w), _ptr(m), _ptr(v), _ptr(out), pdtype,
                        C.byref(hp), C.byref(S))
    return rc, out, S.value


# ---------------------------------------------------------------- the pages' toy
def toy_zero2_threads(targets, w0, steps, hp):
    N, P = targets.shape
    out = np.zeros((N, P), np.float32)
    t = np.ascontiguousarray(targets, np.float32)
    w0 = np.ascontiguousarray(w0, np.float32)
    _check(lib().orc_toy_zero2_threads(N, P, steps, _ptr(t), _ptr(w0), C.byref(hp), _ptr(out)), "toy threads")
    return out


def toy_unsharded(targets, w0, steps, hp):
    N, P = targets.shape
    out = np.zeros(P, np.float32)
    t = np.ascontiguousarray(targets, np.float32)
    w0 = np.ascontiguousarray(w0, np.float32)
    _check(lib().orc_toy_unsharded(N, P, steps, _ptr(t), _ptr(w0), C.byref(hp), _ptr(out)), "toy unsharded")
    return out
