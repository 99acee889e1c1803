"""CPU oracle for the data-parallel ZeRO-2 gradient step.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product library never does.  It
wraps ``oracle.c`` (plain single-threaded C, binary32 round-to-nearest, no
FMA contraction) through ctypes over numpy arrays.  See ``oracle.c`` for the
sources each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK = 0
EINVAL = -1
EZERO_TOKENS = -2
BF16 = 0
F32 = 1

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, a second or two)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    subprocess.run([cc, *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        # ORACLE_LIB points the tests at a deliberately broken copy (mutation
        # testing of the pins); normally the library is built next to oracle.c
        path = os.environ.get("ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f32, f64, u16 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_uint16)
        L.oracle_bf16_to_f32.argtypes = [u16]
        L.oracle_bf16_to_f32.restype = f32
        L.oracle_f32_to_bf16.argtypes = [f32]
        L.oracle_f32_to_bf16.restype = u16
        L.oracle_f32_to_bf16_array.argtypes = [P, P, i64]
        L.oracle_bf16_to_f32_array.argtypes = [P, P, i64]
        L.oracle_plan_buckets.argtypes = [P, i32, i64, i32, P, P, P, P, P, P]
        L.oracle_plan_buckets.restype = ctypes.c_int
        L.oracle_pack.argtypes = [i32, P, P, P, i64, P]
        L.oracle_unpack.argtypes = [i32, P, P, P, P]
        L.oracle_accumulate.argtypes = [i64, P, P, i32]
        L.oracle_export_state.argtypes = [i32, P, P, P, P]
        L.oracle_clip_coef.argtypes = [P, i64, f64, P, P]
        L.oracle_scale_range.argtypes = [P, i64, f32]
        L.oracle_import_state.argtypes = [i32, P, P, P, i64, P]
        L.oracle_grad_scale.argtypes = [P, i32, P]
        L.oracle_grad_scale.restype = ctypes.c_int
        L.oracle_reduce_range.argtypes = [i32, P, i32, P, f32, i64, i64, P]
        L.oracle_allreduce.argtypes = [i32, i64, P, i32, P, f32, P]
        L.oracle_adam_range.argtypes = [P, P, P, P, i64, i64, f64, f64, f64, f64, f64, i64]
        L.oracle_adam_range.restype = ctypes.c_int
        L.oracle_step.argtypes = [i32, P, P, i32, P, i32, P, P, i32, f64, f64, f64, f64,
                                  f64, i64, P, P, P, P, i32, P, P]
        L.oracle_step.restype = ctypes.c_int
        L.oracle_allgather.argtypes = [i64, P, P, i32]
        L.oracle_model_state_bytes.argtypes = [i32, f64, i32]
        L.oracle_model_state_bytes.restype = f64
        _lib = L
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: oracle status {status}")
        self.status = status


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _ptr_array(arrs: Sequence[np.ndarray]):
    arr = (ctypes.c_void_p * max(1, len(arrs)))()
    for i, a in enumerate(arrs):
        arr[i] = a.ctypes.data
    return arr


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# --------------------------------------------------------------------------
# bf16 helpers (bf16 values travel as uint16 bit patterns)
# --------------------------------------------------------------------------

def f32_to_bf16(x) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(x), _ptr(y), x.size)
    return y


def bf16_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    y = np.empty(h.shape, dtype=np.float32)
    lib().oracle_bf16_to_f32_array(_ptr(h), _ptr(y), h.size)
    return y


# --------------------------------------------------------------------------
# plan
# --------------------------------------------------------------------------

class Plan:
    """Result of the oracle's bucket planner (see oracle.c)."""

    def __init__(self, numels, cap_bytes: int, R: int):
        numels = _c(numels, np.int64)
        n = numels.size
        self.numels = numels
        self.R = R
        self.cap_bytes = cap_bytes
        self.param_bucket = np.empty(max(n, 1), dtype=np.int32)
        self.param_offset = np.empty(max(n, 1), dtype=np.int64)
        bo = np.empty(max(n, 1), dtype=np.int64)
        bp = np.empty(max(n, 1), dtype=np.int64)
        nb = ctypes.c_int32(0)
        tot = ctypes.c_int64(0)
        st = lib().oracle_plan_buckets(_ptr(numels), n, cap_bytes, R, _ptr(self.param_bucket),
                                       _ptr(self.param_offset), _ptr(bo), _ptr(bp),
                                       ctypes.byref(nb), ctypes.byref(tot))
        if st != OK:
            raise OracleError(st, "oracle_plan_buckets")
        self.param_bucket = self.param_bucket[:n]
        self.param_offset = self.param_offset[:n]
        self.n_buckets = nb.value
        self.bucket_offset = bo[: nb.value].copy()
        self.bucket_padded = bp[: nb.value].copy()
        self.total_padded = tot.value

    @property
    def shard_numel(self) -> np.ndarray:
        return self.bucket_padded // self.R


def plan_buckets(numels, cap_bytes: int, R: int) -> Plan:
    return Plan(numels, cap_bytes, R)


def pack(plan: Plan, grads: Sequence[np.ndarray]) -> np.ndarray:
    gs = [_c(g, np.uint16).reshape(-1) for g in grads]
    flat = np.empty(plan.total_padded, dtype=np.uint16)
    lib().oracle_pack(len(gs), _ptr(plan.numels), _ptr(plan.param_offset), _ptr_array(gs),
                      plan.total_padded, _ptr(flat))
    return flat


def unpack(plan: Plan, flat: np.ndarray) -> list:
    flat = _c(flat, np.uint16)
    outs = [np.empty(int(n), dtype=np.uint16) for n in plan.numels]
    lib().oracle_unpack(len(outs), _ptr(plan.numels), _ptr(plan.param_offset), _ptr(flat),
                        _ptr_array(outs))
    return outs


def export_state(plan: Plan, flat: np.ndarray) -> np.ndarray:
    """Canonical (registration-order, unpadded) copy of one fp32 flat array."""
    flat = _c(flat, np.float32)
    canon = np.empty(int(plan.numels.sum()), dtype=np.float32)
    lib().oracle_export_state(plan.numels.size, _ptr(plan.numels), _ptr(plan.param_offset),
                              _ptr(flat), _ptr(canon))
    return canon


def import_state(plan: Plan, canon: np.ndarray) -> np.ndarray:
    """Flat fp32 array of the plan's layout from a canonical one (padding 0)."""
    canon = _c(canon, np.float32)
    flat = np.empty(plan.total_padded, dtype=np.float32)
    lib().oracle_import_state(plan.numels.size, _ptr(plan.numels), _ptr(plan.param_offset),
                              _ptr(canon), plan.total_padded, _ptr(flat))
    return flat


def accumulate(g_bf16: np.ndarray, acc: np.ndarray, first: bool) -> np.ndarray:
    """In place on acc (float32); returns acc."""
    g = _c(g_bf16, np.uint16)
    assert acc.dtype == np.float32 and acc.flags.c_contiguous and acc.size == g.size
    lib().oracle_accumulate(g.size, _ptr(g), _ptr(acc), 1 if first else 0)
    return acc


def grad_scale(tokens) -> float:
    t = _c(tokens, np.int64)
    out = ctypes.c_float(0.0)
    st = lib().oracle_grad_scale(_ptr(t), t.size, ctypes.byref(out))
    if st != OK:
        raise OracleError(st, "oracle_grad_scale")
    return np.float32(out.value)


def _dtype_code(arrs) -> int:
    if arrs[0].dtype == np.uint16:
        return BF16
    if arrs[0].dtype == np.float32:
        return F32
    raise TypeError("gradients must be uint16 (bf16 bits) or float32")


def reduce(grads: Sequence[np.ndarray], scale: float, last=None, lo: int = 0,
           hi: Optional[int] = None) -> np.ndarray:
    """Rank-ordered fp32 reduce of elements [lo, hi), times scale."""
    gs = [np.ascontiguousarray(g).reshape(-1) for g in grads]
    n = gs[0].size
    hi = n if hi is None else hi
    ls = None if last is None else [_c(x, np.uint16).reshape(-1) for x in last]
    out = np.zeros(n, dtype=np.float32)
    lib().oracle_reduce_range(len(gs), _ptr_array(gs), _dtype_code(gs),
                              None if ls is None else _ptr_array(ls), float(scale), lo, hi,
                              _ptr(out))
    return out[lo:hi].copy() if (lo, hi) != (0, n) else out


def allreduce(grads: Sequence[np.ndarray], scale: float, last=None) -> list:
    gs = [np.ascontiguousarray(g).reshape(-1) for g in grads]
    n = gs[0].size
    ls = None if last is None else [_c(x, np.uint16).reshape(-1) for x in last]
    outs = [np.empty(n, dtype=np.float32) for _ in gs]
    lib().oracle_allreduce(len(gs), n, _ptr_array(gs), _dtype_code(gs),
                           None if ls is None else _ptr_array(ls), float(scale),
                           _ptr_array(outs))
    return outs


def clip_coef(g: np.ndarray, max_norm: float):
    """(global L2 norm in binary64, binary32 clip coefficient)."""
    g = _c(g, np.float32)
    norm = ctypes.c_double(0.0)
    coef = ctypes.c_float(0.0)
    lib().oracle_clip_coef(_ptr(g), g.size, float(max_norm), ctypes.byref(norm), ctypes.byref(coef))
    return norm.value, np.float32(coef.value)


def scale(g: np.ndarray, coef) -> np.ndarray:
    """A copy of g multiplied by coef in binary32."""
    out = np.array(g, dtype=np.float32, copy=True)
    lib().oracle_scale_range(_ptr(out), out.size, float(coef))
    return out


def adam(g, master, m, v, *, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, t=1):
    """In place on master/m/v (float32 arrays); g is float32."""
    g = _c(g, np.float32)
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == g.size
    st = lib().oracle_adam_range(_ptr(g), _ptr(master), _ptr(m), _ptr(v), 0, g.size,
                                 lr, beta1, beta2, eps, wd, t)
    if st != OK:
        raise OracleError(st, "oracle_adam_range")


def step(bucket_offset, bucket_padded, grads, tokens, master, m, v, *, last=None,
         n_views: int = 1, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, t=1,
         want_reduced: bool = False):
    """Whole step, in place on master/m/v.  Returns (views, reduced, sqnorm)."""
    bo = _c(bucket_offset, np.int64)
    bp = _c(bucket_padded, np.int64)
    gs = [np.ascontiguousarray(g).reshape(-1) for g in grads]
    total = int(gs[0].size)
    ls = None if last is None else [_c(x, np.uint16).reshape(-1) for x in last]
    tk = _c(tokens, np.int64)
    views = [np.empty(total, dtype=np.uint16) for _ in range(n_views)]
    reduced = np.empty(total, dtype=np.float32) if want_reduced else None
    sq = np.empty(max(1, bo.size), dtype=np.float64)
    st = lib().oracle_step(bo.size, _ptr(bo), _ptr(bp), len(gs), _ptr_array(gs),
                           _dtype_code(gs), None if ls is None else _ptr_array(ls), _ptr(tk),
                           tk.size, lr, beta1, beta2, eps, wd, t, _ptr(master), _ptr(m), _ptr(v),
                           _ptr_array(views), n_views, _ptr(reduced), _ptr(sq))
    if st != OK:
        raise OracleError(st, "oracle_step")
    return views, reduced, sq[: bo.size]


def allgather(master: np.ndarray, n_views: int = 1) -> list:
    master = _c(master, np.float32)
    views = [np.empty(master.size, dtype=np.uint16) for _ in range(n_views)]
    lib().oracle_allgather(master.size, _ptr(master), _ptr_array(views), n_views)
    return views


def model_state_bytes(stage: int, psi: float, N: int) -> float:
    return lib().oracle_model_state_bytes(stage, float(psi), N)
