"""GB300 data-parallel ZeRO-2 gradient step -- Python binding of libdpg.so.

Thin ctypes marshalling over the C ABI in include/dpg.h: every function has
the C name, takes torch tensors (or raw integer device pointers) and the
current CUDA stream, and calls the library; all arithmetic of the step runs
in the library's sm_103a kernels.  PyTorch only supplies device memory and
streams.  If libdpg.so has not been built, importing works but every call
raises ``DpgLibraryMissing``: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence, Union

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# DPG_LIBRARY=debug loads the index-checking build (libdpg_debug.so) instead
LIB_PATH = os.path.join(_PKG, "libdpg_debug.so" if os.environ.get("DPG_LIBRARY") == "debug"
                        else "libdpg.so")

DPG_OK = 0
DPG_ERR_INVALID_ARG = -1
DPG_ERR_ZERO_TOKENS = -2
DPG_ERR_MISALIGNED = -3
DPG_ERR_CUDA = -4
DPG_ERR_DEVICE_TIMEOUT = -5
DPG_ERR_OOM = -6
DPG_BF16 = 0
DPG_F32 = 1
DPG_MAX_REPLICAS = 64
DPG_MAX_VIEWS = 64

# symbols declared in include/dpg.h
EXPORTED = (
    "dpg_last_error", "dpg_status_string", "dpg_abi_version", "dpg_plan_buckets",
    "dpg_plan_destroy", "dpg_plan_info", "dpg_plan_bucket", "dpg_plan_param",
    "dpg_plan_export", "dpg_plan_upload", "dpg_pack", "dpg_unpack", "dpg_accumulate",
    "dpg_reduce_scatter_adam", "dpg_allgather_params", "dpg_step", "dpg_launch_count",
    "dpg_time_next_fused_launch", "dpg_step_noalloc", "dpg_export_state", "dpg_import_state",
    "dpg_step_clipped", "dpg_step_staged", "dpg_check_device_status", "dpg_set_staged_fault",
    "dpg_allreduce_grads", "dpg_adam_from_reduced", "dpg_gather_params_bf16",
    "dpg_accumulate_pair", "dpg_step_fold2", "dpg_set_fused_max_ctas",
    "dpg_set_programmatic_launch", "dpg_reduce_scatter_adam_when_ready", "dpg_step_deferred",
    "dpg_plan_shards", "dpg_debug_checks", "dpg_debug_set_limit",
)
DPG_MAX_STATE_ARRAYS = 8
DPG_NOALLOC_SCRATCH_BYTES = 8 << 20


class DpgLibraryMissing(ImportError):
    pass


class DpgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)} ({status}): {message}")
        self.status = status


class dpg_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("step", ctypes.c_int64)]


@dataclass
class HParams:
    """Adam hyper-parameters; ``step`` is t of this update (first update: 1)."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    step: int = 1

    def c(self) -> dpg_hparams:
        return dpg_hparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                           int(self.step))


_lib = None


def lib() -> ctypes.CDLL:
    """Load libdpg.so (built in-tree by zero_optimizer_step_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise DpgLibraryMissing(
                f"{LIB_PATH} is missing: build it with `python -m zero_optimizer_step_gb300.build`"
                + (" --debug" if LIB_PATH.endswith("_debug.so") else ""))
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        c_int = ctypes.c_int
        L.dpg_last_error.restype = ctypes.c_char_p
        L.dpg_status_string.restype = ctypes.c_char_p
        L.dpg_status_string.argtypes = [c_int]
        L.dpg_abi_version.restype = c_int
        L.dpg_plan_buckets.argtypes = [P, i32, i64, i32, ctypes.POINTER(P)]
        L.dpg_plan_destroy.argtypes = [P]
        L.dpg_plan_destroy.restype = None
        L.dpg_plan_info.argtypes = [P, P, P, P, P]
        L.dpg_plan_bucket.argtypes = [P, i32, P, P, P]
        L.dpg_plan_param.argtypes = [P, i32, P, P, P]
        L.dpg_plan_export.argtypes = [P, P, P, P, P]
        L.dpg_plan_upload.argtypes = [P]
        L.dpg_pack.argtypes = [P, P, P, P]
        L.dpg_unpack.argtypes = [P, P, P, P]
        L.dpg_accumulate.argtypes = [P, P, P, i32, P]
        L.dpg_accumulate_pair.argtypes = [P, P, P, P, i32, P]
        L.dpg_set_fused_max_ctas.argtypes = [i32]
        L.dpg_set_programmatic_launch.argtypes = [i32]
        L.dpg_step_deferred.argtypes = [P, P, i32, P, i32, P, P, P, P, P, i32, P, P, P]
        L.dpg_reduce_scatter_adam_when_ready.argtypes = [P, P, i32, P, P, i32, P, P, P, P, P, i32,
                                                         P, P, P, i32, i32, P, P]
        L.dpg_step_fold2.argtypes = [P, P, P, P, P, i32, P, P, P, P, P, i32, P, P, P]
        L.dpg_reduce_scatter_adam.argtypes = [P, P, i32, P, P, i32, P, P, P, P, P, i32, P, P, P,
                                              i32, i32, P]
        L.dpg_allgather_params.argtypes = [P, P, P, i32, i32, i32, P]
        L.dpg_step.argtypes = [P, P, i32, P, P, i32, P, P, P, P, P, i32, P, P, P]
        L.dpg_step_noalloc.argtypes = [P, P, i32, P, P, i32, P, P, P, P, P, i32, P, P, P]
        L.dpg_launch_count.restype = i64
        L.dpg_step_clipped.argtypes = [P, P, i32, P, P, i32, P, ctypes.c_double, P, P, P, P, i32,
                                       P, P, P, P, P]
        L.dpg_step_staged.argtypes = [P, P, i32, P, i32, P, P, P, P, P, i32, P, P, P]
        L.dpg_allreduce_grads.argtypes = [P, P, i32, P, P, i32, P, P, P, i32, i32, P]
        L.dpg_gather_params_bf16.argtypes = [P, P, P, i32, i32, i32, P]
        L.dpg_adam_from_reduced.argtypes = [P, P, P, P, P, P, P, i32, P, P, i32, i32, P]
        L.dpg_check_device_status.argtypes = [P, P]
        L.dpg_set_staged_fault.argtypes = [i64, i64]
        L.dpg_export_state.argtypes = [P, P, P, i32, P]
        L.dpg_import_state.argtypes = [P, P, P, i32, P]
        L.dpg_time_next_fused_launch.argtypes = [P, P]
        L.dpg_plan_shards.argtypes = [P, ctypes.POINTER(P)]
        L.dpg_debug_checks.argtypes = [P, P, P]
        L.dpg_debug_set_limit.argtypes = [i64]
        L.dpg_time_next_fused_launch.restype = c_int
        for name in ("dpg_plan_buckets", "dpg_plan_info", "dpg_plan_bucket", "dpg_plan_param",
                     "dpg_plan_export", "dpg_plan_upload", "dpg_pack", "dpg_unpack",
                     "dpg_accumulate", "dpg_reduce_scatter_adam", "dpg_allgather_params",
                     "dpg_step", "dpg_step_noalloc", "dpg_export_state", "dpg_import_state",
                     "dpg_step_clipped", "dpg_step_staged", "dpg_check_device_status",
                     "dpg_set_staged_fault", "dpg_allreduce_grads", "dpg_adam_from_reduced",
                     "dpg_gather_params_bf16", "dpg_accumulate_pair", "dpg_step_fold2",
                     "dpg_set_fused_max_ctas", "dpg_set_programmatic_launch",
                     "dpg_reduce_scatter_adam_when_ready", "dpg_step_deferred",
                     "dpg_plan_shards", "dpg_debug_checks", "dpg_debug_set_limit"):
            getattr(L, name).restype = c_int
        _lib = L
    return _lib


def _status_name(status: int) -> str:
    try:
        return lib().dpg_status_string(status).decode()
    except Exception:
        return "DPG_ERR"


def _check(status: int):
    if status != DPG_OK:
        raise DpgError(status, lib().dpg_last_error().decode())


# --------------------------------------------------------------------------
# argument marshalling
# --------------------------------------------------------------------------
Ptr = Union[int, "torch.Tensor", None]  # noqa: F821


def _ptr(x: Ptr) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptrs(xs: Sequence[Ptr]):
    arr = (ctypes.c_void_p * max(1, len(xs)))()
    for k, x in enumerate(xs):
        arr[k] = _ptr(x)
    return arr


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _tokens(valid_tokens):
    t = np.ascontiguousarray(np.asarray(valid_tokens, dtype=np.int64).reshape(-1))
    return t, t.size


def _need(t, dtype_name: str, numel: int, what: str):
    """Tensors must be CUDA, contiguous, of the right dtype and large enough."""
    if t is None or isinstance(t, int):
        return
    import torch
    want = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype_name]
    if t.dtype != want:
        raise TypeError(f"{what}: expected {want}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{what}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: tensor must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{what}: needs >= {numel} elements, has {t.numel()}")


def _need_in(t, dtype_name: str, numel: int, what: str):
    """Gradient inputs may also be page-locked host tensors: under unified
    addressing the kernels read them over the host link at the same address."""
    if t is not None and not isinstance(t, int) and not t.is_cuda and t.is_pinned():
        import torch
        want = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype_name]
        if t.dtype != want:
            raise TypeError(f"{what}: expected {want}, got {t.dtype}")
        if not t.is_contiguous() or t.numel() < numel:
            raise ValueError(f"{what}: needs a contiguous tensor of >= {numel} elements")
        return
    _need(t, dtype_name, numel, what)


# --------------------------------------------------------------------------
# plan
# --------------------------------------------------------------------------
class Plan:
    """Owning handle of a dpg_plan_t plus numpy copies of its maps."""

    def __init__(self, handle: int, numels=None):
        self._h = ctypes.c_void_p(handle)
        self.numels = None if numels is None else np.asarray(numels, np.int64).copy()
        L = lib()
        n_params, n_buckets, R = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        total = ctypes.c_int64()
        _check(L.dpg_plan_info(self._h, ctypes.byref(n_params), ctypes.byref(n_buckets),
                               ctypes.byref(total), ctypes.byref(R)))
        self.n_params, self.n_buckets = n_params.value, n_buckets.value
        self.total_padded, self.R = total.value, R.value
        self.param_bucket = np.zeros(max(1, self.n_params), np.int32)
        self.param_offset = np.zeros(max(1, self.n_params), np.int64)
        self.bucket_offset = np.zeros(max(1, self.n_buckets), np.int64)
        self.bucket_padded = np.zeros(max(1, self.n_buckets), np.int64)
        _check(L.dpg_plan_export(self._h, self.param_bucket.ctypes.data,
                                 self.param_offset.ctypes.data, self.bucket_offset.ctypes.data,
                                 self.bucket_padded.ctypes.data))
        self.param_bucket = self.param_bucket[: self.n_params]
        self.param_offset = self.param_offset[: self.n_params]
        self.bucket_offset = self.bucket_offset[: self.n_buckets]
        self.bucket_padded = self.bucket_padded[: self.n_buckets]

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise ValueError("plan has been destroyed")
        return self._h

    @property
    def shard_numel(self) -> np.ndarray:
        return self.bucket_padded // self.R

    @property
    def canon_total(self) -> int:
        """Elements of the canonical (registration-order, unpadded) layout."""
        return int(self.numels.sum())

    def destroy(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.dpg_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def dpg_plan_buckets(numels: Sequence[int], cap_bytes: int, R: int) -> Plan:
    n = np.ascontiguousarray(np.asarray(numels, dtype=np.int64).reshape(-1))
    out = ctypes.c_void_p()
    _check(lib().dpg_plan_buckets(n.ctypes.data if n.size else None, n.size, int(cap_bytes),
                                  int(R), ctypes.byref(out)))
    return Plan(out.value, n)


def dpg_plan_shards(plan: Plan) -> Plan:
    """Shard plan of the ZeRO-2 split across plan.R ranks: one bucket per
    bucket of `plan`, holding that bucket's shard (see include/dpg.h)."""
    out = ctypes.c_void_p()
    _check(lib().dpg_plan_shards(plan.handle, ctypes.byref(out)))
    return Plan(out.value, plan.shard_numel[::-1])


def dpg_plan_upload(plan: Plan):
    _check(lib().dpg_plan_upload(plan.handle))


def dpg_plan_bucket(plan: Plan, b: int):
    o, pd, sh = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().dpg_plan_bucket(plan.handle, b, ctypes.byref(o), ctypes.byref(pd), ctypes.byref(sh)))
    return o.value, pd.value, sh.value


def dpg_plan_param(plan: Plan, p: int):
    b, o, n = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().dpg_plan_param(plan.handle, p, ctypes.byref(b), ctypes.byref(o), ctypes.byref(n)))
    return b.value, o.value, n.value


# --------------------------------------------------------------------------
# device calls
# --------------------------------------------------------------------------
def dpg_pack(plan: Plan, param_grads: Sequence[Ptr], flat_bf16: Ptr, stream=None):
    if len(param_grads) != plan.n_params:
        raise ValueError(f"need {plan.n_params} gradients, got {len(param_grads)}")
    _need(flat_bf16, "bf16", plan.total_padded, "flat_bf16")
    for k, g in enumerate(param_grads):
        _need(g, "bf16", 0, f"param_grads[{k}]")
    _check(lib().dpg_pack(plan.handle, _ptrs(param_grads), _ptr(flat_bf16), _stream(stream)))


def dpg_unpack(plan: Plan, flat_bf16: Ptr, param_grads: Sequence[Ptr], stream=None):
    if len(param_grads) != plan.n_params:
        raise ValueError(f"need {plan.n_params} gradients, got {len(param_grads)}")
    _need(flat_bf16, "bf16", plan.total_padded, "flat_bf16")
    for k, g in enumerate(param_grads):
        _need(g, "bf16", 0, f"param_grads[{k}]")
    _check(lib().dpg_unpack(plan.handle, _ptr(flat_bf16), _ptrs(param_grads), _stream(stream)))


def dpg_export_state(plan: Plan, flat: Sequence[Ptr], canon: Sequence[Ptr], stream=None):
    """canon[k] <- flat[k] for the fp32 state arrays (see include/dpg.h)."""
    if len(flat) != len(canon):
        raise ValueError("flat and canon need the same number of arrays")
    for k, (f, c) in enumerate(zip(flat, canon)):
        _need(f, "f32", plan.total_padded, f"flat[{k}]")
        _need(c, "f32", plan.canon_total, f"canon[{k}]")
    _check(lib().dpg_export_state(plan.handle, _ptrs(flat), _ptrs(canon), len(flat),
                                  _stream(stream)))


def dpg_import_state(plan: Plan, canon: Sequence[Ptr], flat: Sequence[Ptr], stream=None):
    """flat[k] <- canon[k] (padding zeroed) for the fp32 state arrays."""
    if len(flat) != len(canon):
        raise ValueError("flat and canon need the same number of arrays")
    for k, (f, c) in enumerate(zip(flat, canon)):
        _need(f, "f32", plan.total_padded, f"flat[{k}]")
        _need(c, "f32", plan.canon_total, f"canon[{k}]")
    _check(lib().dpg_import_state(plan.handle, _ptrs(canon), _ptrs(flat), len(flat),
                                  _stream(stream)))


def dpg_accumulate(plan: Plan, flat_bf16: Ptr, acc_f32: Ptr, first: bool, stream=None):
    _need_in(flat_bf16, "bf16", plan.total_padded, "flat_bf16")
    _need(acc_f32, "f32", plan.total_padded, "acc_f32")
    _check(lib().dpg_accumulate(plan.handle, _ptr(flat_bf16), _ptr(acc_f32), 1 if first else 0,
                                _stream(stream)))


def dpg_accumulate_pair(plan: Plan, micro_a_bf16: Ptr, micro_b_bf16: Ptr, acc_f32: Ptr,
                        first: bool, stream=None):
    """acc <- (acc + a) + b (or a + b when first): two microbatches in one pass."""
    _need_in(micro_a_bf16, "bf16", plan.total_padded, "micro_a_bf16")
    _need_in(micro_b_bf16, "bf16", plan.total_padded, "micro_b_bf16")
    _need(acc_f32, "f32", plan.total_padded, "acc_f32")
    _check(lib().dpg_accumulate_pair(plan.handle, _ptr(micro_a_bf16), _ptr(micro_b_bf16),
                                     _ptr(acc_f32), 1 if first else 0, _stream(stream)))


def dpg_step_fold2(plan: Plan, acc_f32: Sequence[Ptr], micro_a: Sequence[Ptr],
                   micro_b: Sequence[Ptr], valid_tokens, hp: HParams, master: Ptr, exp_avg: Ptr,
                   exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (), *, bucket_sqnorm: Ptr = None,
                   bucket_nonfinite: Ptr = None, stream=None):
    """Whole step with the last two bf16 microbatches folded into the reduction."""
    for name, xs in (("acc_f32", acc_f32), ("micro_a", micro_a), ("micro_b", micro_b)):
        if len(xs) != plan.R:
            raise ValueError(f"{name}: need R={plan.R} buffers, got {len(xs)}")
    N = plan.total_padded
    for k in range(plan.R):
        _need_in(acc_f32[k], "f32", N, f"acc_f32[{k}]")
        _need_in(micro_a[k], "bf16", N, f"micro_a[{k}]")
        _need_in(micro_b[k], "bf16", N, f"micro_b[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_step_fold2(
        plan.handle, _ptrs(acc_f32), _ptrs(micro_a), _ptrs(micro_b), tok.ctypes.data, n_tok,
        ctypes.byref(hpc), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptrs(param_views),
        len(param_views), _ptr(bucket_sqnorm), _ptr(bucket_nonfinite), _stream(stream)))


def _grad_dtype(grads) -> int:
    import torch
    g0 = grads[0]
    if isinstance(g0, int):
        raise TypeError("pass grads_dtype explicitly with raw pointers")
    return DPG_BF16 if g0.dtype == torch.bfloat16 else DPG_F32


def dpg_reduce_scatter_adam(plan: Plan, grads: Sequence[Ptr], valid_tokens, hp: HParams,
                            master: Ptr, exp_avg: Ptr, exp_avg_sq: Ptr,
                            param_views: Sequence[Ptr] = (), *, last_micro: Sequence[Ptr] = None,
                            bucket_sqnorm: Ptr = None, bucket_nonfinite: Ptr = None,
                            reduced_grad: Ptr = None, b0: int = 0, b1: Optional[int] = None,
                            grads_dtype: Optional[int] = None, stream=None):
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    gd = _grad_dtype(grads) if grads_dtype is None else grads_dtype
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need_in(g, "bf16" if gd == DPG_BF16 else "f32", N, f"grads[{k}]")
    for k, g in enumerate(last_micro or ()):
        _need_in(g, "bf16", N, f"last_micro[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq),
                    ("reduced_grad", reduced_grad)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_reduce_scatter_adam(
        plan.handle, _ptrs(grads), gd, None if last_micro is None else _ptrs(last_micro),
        tok.ctypes.data, n_tok, ctypes.byref(hpc), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
        _ptrs(param_views), len(param_views), _ptr(bucket_sqnorm), _ptr(bucket_nonfinite),
        _ptr(reduced_grad), b0, plan.n_buckets if b1 is None else b1, _stream(stream)))


def dpg_step_deferred(plan: Plan, micro: Sequence[Sequence[Ptr]], valid_tokens, hp: HParams,
                      master: Ptr, exp_avg: Ptr, exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (),
                      *, bucket_sqnorm: Ptr = None, bucket_nonfinite: Ptr = None, stream=None):
    """Step of a K-microbatch cycle from every replica's K bf16 microbatch
    buffers (micro[r][k]), summed inside the fused pass in microbatch order:
    the bits of K-1 dpg_accumulate passes plus dpg_step."""
    if len(micro) != plan.R:
        raise ValueError(f"need R={plan.R} replicas of microbatch buffers, got {len(micro)}")
    K = len(micro[0]) if micro else 0
    if any(len(mr) != K for mr in micro):
        raise ValueError("every replica needs the same number of microbatches")
    N = plan.total_padded
    flat = [t for mr in micro for t in mr]
    for k, t in enumerate(flat):
        _need_in(t, "bf16", N, f"micro[{k // max(1, K)}][{k % max(1, K)}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_step_deferred(
        plan.handle, _ptrs(flat), K, tok.ctypes.data, n_tok, ctypes.byref(hpc), _ptr(master),
        _ptr(exp_avg), _ptr(exp_avg_sq), _ptrs(param_views), len(param_views),
        _ptr(bucket_sqnorm), _ptr(bucket_nonfinite), _stream(stream)))


def _event_handle(e) -> Optional[int]:
    if e is None or isinstance(e, int):
        return e
    return e.cuda_event          # torch.cuda.Event: its cudaEvent_t, once recorded


def dpg_reduce_scatter_adam_when_ready(plan: Plan, grads: Sequence[Ptr], valid_tokens,
                                       hp: HParams, master: Ptr, exp_avg: Ptr, exp_avg_sq: Ptr,
                                       param_views: Sequence[Ptr] = (), *, ready_events,
                                       last_micro: Sequence[Ptr] = None,
                                       bucket_sqnorm: Ptr = None, bucket_nonfinite: Ptr = None,
                                       reduced_grad: Ptr = None, b0: int = 0,
                                       b1: Optional[int] = None,
                                       grads_dtype: Optional[int] = None, stream=None):
    """dpg_reduce_scatter_adam over [b0, b1), bucket b launched on `stream` only
    after ready_events[b - b0] (recorded by the producer of its gradients)."""
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    b1 = plan.n_buckets if b1 is None else b1
    if len(ready_events) != max(0, b1 - b0):
        raise ValueError(f"need {max(0, b1 - b0)} ready events, got {len(ready_events)}")
    gd = _grad_dtype(grads) if grads_dtype is None else grads_dtype
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need_in(g, "bf16" if gd == DPG_BF16 else "f32", N, f"grads[{k}]")
    for k, g in enumerate(last_micro or ()):
        _need_in(g, "bf16", N, f"last_micro[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq),
                    ("reduced_grad", reduced_grad)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    evs = (ctypes.c_void_p * max(1, len(ready_events)))(*[_event_handle(e) for e in ready_events])
    _check(lib().dpg_reduce_scatter_adam_when_ready(
        plan.handle, _ptrs(grads), gd, None if last_micro is None else _ptrs(last_micro),
        tok.ctypes.data, n_tok, ctypes.byref(hpc), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
        _ptrs(param_views), len(param_views), _ptr(bucket_sqnorm), _ptr(bucket_nonfinite),
        _ptr(reduced_grad), b0, b1, evs, _stream(stream)))


def dpg_step(plan: Plan, grads: Sequence[Ptr], valid_tokens, hp: HParams, master: Ptr,
             exp_avg: Ptr, exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (), *,
             last_micro: Sequence[Ptr] = None, bucket_sqnorm: Ptr = None,
             bucket_nonfinite: Ptr = None, grads_dtype: Optional[int] = None, stream=None):
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    gd = _grad_dtype(grads) if grads_dtype is None else grads_dtype
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need_in(g, "bf16" if gd == DPG_BF16 else "f32", N, f"grads[{k}]")
    for k, g in enumerate(last_micro or ()):
        _need_in(g, "bf16", N, f"last_micro[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_step(
        plan.handle, _ptrs(grads), gd, None if last_micro is None else _ptrs(last_micro),
        tok.ctypes.data, n_tok, ctypes.byref(hpc), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
        _ptrs(param_views), len(param_views), _ptr(bucket_sqnorm), _ptr(bucket_nonfinite),
        _stream(stream)))


def dpg_step_clipped(plan: Plan, grads: Sequence[Ptr], valid_tokens, hp: HParams, max_norm: float,
                     master: Ptr, exp_avg: Ptr, exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (),
                     *, last_micro: Sequence[Ptr] = None, bucket_sqnorm: Ptr = None,
                     bucket_nonfinite: Ptr = None, reduced_grad: Ptr = None, clip_out: Ptr = None,
                     grads_dtype: Optional[int] = None, stream=None):
    """dpg_step with global gradient-norm clipping (see include/dpg.h)."""
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    gd = _grad_dtype(grads) if grads_dtype is None else grads_dtype
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need_in(g, "bf16" if gd == DPG_BF16 else "f32", N, f"grads[{k}]")
    for k, g in enumerate(last_micro or ()):
        _need_in(g, "bf16", N, f"last_micro[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq),
                    ("reduced_grad", reduced_grad)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    _need(clip_out, "f32", 2, "clip_out")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_step_clipped(
        plan.handle, _ptrs(grads), gd, None if last_micro is None else _ptrs(last_micro),
        tok.ctypes.data, n_tok, ctypes.byref(hpc), float(max_norm), _ptr(master), _ptr(exp_avg),
        _ptr(exp_avg_sq), _ptrs(param_views), len(param_views), _ptr(bucket_sqnorm),
        _ptr(bucket_nonfinite), _ptr(reduced_grad), _ptr(clip_out), _stream(stream)))


def dpg_step_staged(plan: Plan, grads: Sequence[Ptr], valid_tokens, hp: HParams, master: Ptr,
                    exp_avg: Ptr, exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (), *,
                    bucket_sqnorm: Ptr = None, bucket_nonfinite: Ptr = None, stream=None):
    """dpg_step through the bulk-copy staged pass (bf16 gradients, R in 1/2/4/8)."""
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need(g, "bf16", N, f"grads[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_step_staged(
        plan.handle, _ptrs(grads), DPG_BF16, tok.ctypes.data, n_tok, ctypes.byref(hpc),
        _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptrs(param_views), len(param_views),
        _ptr(bucket_sqnorm), _ptr(bucket_nonfinite), _stream(stream)))


def dpg_check_device_status(plan: Plan, stream=None):
    """Synchronise the stream; raise DpgError if the last staged step timed out."""
    _check(lib().dpg_check_device_status(plan.handle, _stream(stream)))


def dpg_set_staged_fault(skip_unit: int = -1, timeout_ns: int = 0):
    """Test-only: the next staged launch skips fetching one half-tile."""
    _check(lib().dpg_set_staged_fault(int(skip_unit), int(timeout_ns)))


def dpg_allreduce_grads(plan: Plan, grads: Sequence[Ptr], valid_tokens, reduced_grad: Ptr, *,
                        last_micro: Sequence[Ptr] = None, bucket_sqnorm: Ptr = None,
                        bucket_nonfinite: Ptr = None, b0: int = 0, b1: Optional[int] = None,
                        grads_dtype: Optional[int] = None, stream=None):
    """DDP all-reduce: reduced_grad = rank-ordered sum x fp32(1/G), every element."""
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    gd = _grad_dtype(grads) if grads_dtype is None else grads_dtype
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need_in(g, "bf16" if gd == DPG_BF16 else "f32", N, f"grads[{k}]")
    for k, g in enumerate(last_micro or ()):
        _need_in(g, "bf16", N, f"last_micro[{k}]")
    _need(reduced_grad, "f32", N, "reduced_grad")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    _check(lib().dpg_allreduce_grads(
        plan.handle, _ptrs(grads), gd, None if last_micro is None else _ptrs(last_micro),
        tok.ctypes.data, n_tok, _ptr(reduced_grad), _ptr(bucket_sqnorm), _ptr(bucket_nonfinite),
        b0, plan.n_buckets if b1 is None else b1, _stream(stream)))


def dpg_adam_from_reduced(plan: Plan, reduced_grad: Ptr, hp: HParams, master: Ptr, exp_avg: Ptr,
                          exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (), *,
                          bucket_sqnorm: Ptr = None, bucket_nonfinite: Ptr = None, b0: int = 0,
                          b1: Optional[int] = None, stream=None):
    """One DDP replica's Adam step on its full state from the all-reduced gradient."""
    N = plan.total_padded
    for name, t in (("reduced_grad", reduced_grad), ("master", master), ("exp_avg", exp_avg),
                    ("exp_avg_sq", exp_avg_sq)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    hpc = hp.c()
    _check(lib().dpg_adam_from_reduced(
        plan.handle, _ptr(reduced_grad), ctypes.byref(hpc), _ptr(master), _ptr(exp_avg),
        _ptr(exp_avg_sq), _ptrs(param_views), len(param_views), _ptr(bucket_sqnorm),
        _ptr(bucket_nonfinite), b0, plan.n_buckets if b1 is None else b1, _stream(stream)))


def dpg_step_noalloc(plan: Plan, grads: Sequence[Ptr], valid_tokens, hp: HParams, master: Ptr,
                     exp_avg: Ptr, exp_avg_sq: Ptr, param_views: Sequence[Ptr] = (), *,
                     last_micro: Sequence[Ptr] = None, bucket_sqnorm: Ptr = None,
                     bucket_nonfinite: Ptr = None, grads_dtype: Optional[int] = None,
                     stream=None):
    """dpg_step for callers that must not have the library allocate device
    memory: tables and norm partials live in the library's static device array
    (DPG_NOALLOC_SCRATCH_BYTES); larger plans are rejected.  Calls that overlap
    on the GPU share that array and race."""
    if len(grads) != plan.R:
        raise ValueError(f"need R={plan.R} gradient buffers, got {len(grads)}")
    gd = _grad_dtype(grads) if grads_dtype is None else grads_dtype
    N = plan.total_padded
    for k, g in enumerate(grads):
        _need(g, "bf16" if gd == DPG_BF16 else "f32", N, f"grads[{k}]")
    for k, g in enumerate(last_micro or ()):
        _need(g, "bf16", N, f"last_micro[{k}]")
    for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq)):
        _need(t, "f32", N, name)
    for k, t in enumerate(param_views):
        _need(t, "bf16", N, f"param_views[{k}]")
    _need(bucket_sqnorm, "f32", plan.n_buckets, "bucket_sqnorm")
    tok, n_tok = _tokens(valid_tokens)
    hpc = hp.c()
    _check(lib().dpg_step_noalloc(
        plan.handle, _ptrs(grads), gd, None if last_micro is None else _ptrs(last_micro),
        tok.ctypes.data, n_tok, ctypes.byref(hpc), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
        _ptrs(param_views), len(param_views), _ptr(bucket_sqnorm), _ptr(bucket_nonfinite),
        _stream(stream)))


def dpg_allgather_params(plan: Plan, master: Ptr, param_views: Sequence[Ptr], *, b0: int = 0,
                         b1: Optional[int] = None, stream=None):
    _need(master, "f32", plan.total_padded, "master")
    for k, t in enumerate(param_views):
        _need(t, "bf16", plan.total_padded, f"param_views[{k}]")
    _check(lib().dpg_allgather_params(plan.handle, _ptr(master), _ptrs(param_views),
                                      len(param_views), b0,
                                      plan.n_buckets if b1 is None else b1, _stream(stream)))


def dpg_gather_params_bf16(plan: Plan, param_bf16: Ptr, param_views: Sequence[Ptr], *, b0: int = 0,
                           b1: Optional[int] = None, stream=None):
    """ZeRO-3 all-gather of the bf16 parameter shards into full replica views."""
    _need(param_bf16, "bf16", plan.total_padded, "param_bf16")
    for k, t in enumerate(param_views):
        _need(t, "bf16", plan.total_padded, f"param_views[{k}]")
    _check(lib().dpg_gather_params_bf16(plan.handle, _ptr(param_bf16), _ptrs(param_views),
                                        len(param_views), b0, plan.n_buckets if b1 is None else b1,
                                        _stream(stream)))


def dpg_set_fused_max_ctas(max_ctas: int = 0):
    """Cap the CTAs of later fused passes from this thread: > 0 selects the
    persistent grid-stride kernels on at most max_ctas CTAs, 0 restores the
    default chunked launch (one small CTA per 1024-element chunk)."""
    _check(lib().dpg_set_fused_max_ctas(int(max_ctas)))


def dpg_set_programmatic_launch(on: bool = True):
    """Programmatic dependent launch for later launches from this thread
    (default on): same stream order and results, shorter gaps between
    back-to-back kernels."""
    _check(lib().dpg_set_programmatic_launch(1 if on else 0))


def dpg_debug_checks(plan: Plan):
    """(built, first_failure): whether the loaded library checks indices, and
    the first failed check recorded for `plan` since the last call (0: none)."""
    built, first = ctypes.c_int32(), ctypes.c_int64()
    _check(lib().dpg_debug_checks(plan.handle, ctypes.byref(built), ctypes.byref(first)))
    return bool(built.value), int(first.value)


def dpg_debug_set_limit(limit: int = -1):
    _check(lib().dpg_debug_set_limit(int(limit)))


def dpg_launch_count() -> int:
    return int(lib().dpg_launch_count())


def dpg_time_next_fused_launch(start_event, stop_event):
    """Events are torch.cuda.Event objects already recorded once (so that
    their CUDA handles exist), or raw cudaEvent_t integers, or None."""
    h = lambda e: None if e is None else (e if isinstance(e, int) else e.cuda_event)
    _check(lib().dpg_time_next_fused_launch(h(start_event), h(stop_event)))


def dpg_abi_version() -> int:
    return int(lib().dpg_abi_version())
