"""ctypes binding of liblapl_attn.so: the C ABI of include/lapl_attn.h, same names.

Argument marshalling only.  Every step of the attention runs in the CUDA kernels of the
library; there is no fallback.  If the shared library is missing or fails to load, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblapl_attn.so")

LAPL_OK = 0
LAPL_ERR_INVALID_ARG = 1
LAPL_ERR_UNSUPPORTED = 2
LAPL_ERR_WORKSPACE = 3
LAPL_ERR_ALIGNMENT = 4
LAPL_ERR_CUDA = 5
LAPL_ERR_DEVICE_TIMEOUT = 6
LAPL_ERR_NOT_IMPLEMENTED = 7

LAPL_F32 = 0
LAPL_BF16 = 1
LAPL_KERNEL_LAPLACIAN = 0
LAPL_KERNEL_GAUSSIAN = 1
LAPL_SOLVER_NEWTON_SCHULZ = 0
LAPL_SOLVER_CG = 1


class lapl_attn_config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("heads", ctypes.c_int),
        ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("num_landmarks", ctypes.c_int),
        ("lam", ctypes.c_float), ("eps", ctypes.c_float), ("delta", ctypes.c_float),
        ("ns_steps", ctypes.c_int), ("whiten", ctypes.c_int),
        ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
        ("kernel", ctypes.c_int), ("solver", ctypes.c_int),
    ]


_FP = ctypes.POINTER(ctypes.c_float)


class lapl_attn_debug(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("d_ql", "d_ll", "d_lk", "landmarks", "w", "x", "a", "mu", "rstd", "bv", "m")]


class lapl_attn_plan_info(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in
                ("cdist_tma", "cdist_ctas", "cdist_threads", "ns_cluster", "ns_tensor_core",
                 "ns_exclusive", "bv_splits", "bv_tensor_core", "out_tensor_core")]


class LaplAttnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" + (f" ({detail})" if detail else ""))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()'); there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    H = ctypes.c_void_p
    sigs = {
        "lapl_attn_version": ([], ctypes.c_int),
        "lapl_attn_status_string": ([st], ctypes.c_char_p),
        "lapl_attn_last_error": ([H], ctypes.c_char_p),
        "lapl_attn_create": ([ctypes.POINTER(lapl_attn_config), ctypes.POINTER(H)], st),
        "lapl_attn_workspace_size": ([H, ctypes.POINTER(sz)], st),
        "lapl_attn_forward": ([H, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "lapl_attn_forward_train": ([H, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "lapl_attn_forward_debug": ([H, vp, vp, vp, vp, vp, vp, sz, vp,
                                     ctypes.POINTER(lapl_attn_debug)], st),
        "lapl_attn_host_staging_size": ([H, ctypes.POINTER(sz)], st),
        "lapl_attn_forward_host": ([H, vp, vp, vp, vp, vp, vp, sz, vp], st),
        "lapl_attn_set_timing": ([H, ctypes.c_int], st),
        "lapl_attn_stage_times": ([H, ctypes.POINTER(ctypes.c_float)], st),
        "lapl_attn_stage_marks": ([H, ctypes.POINTER(ctypes.c_float)], st),
        "lapl_attn_kernels_per_forward": ([H], ctypes.c_int),
        "lapl_attn_forward_noalloc": ([H, vp, vp, vp, vp, vp, vp], st),
        "lapl_attn_device_errors": ([H, vp, ctypes.POINTER(ctypes.c_uint)], st),
        "lapl_attn_set_fault_injection": ([H, ctypes.c_ulonglong, ctypes.c_int], st),
        "lapl_attn_plan_info_get": ([H, ctypes.POINTER(lapl_attn_plan_info)], st),
        "lapl_attn_backward_workspace_size": ([H, ctypes.POINTER(sz)], st),
        "lapl_attn_backward": ([H, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp], st),
        "lapl_attn_backward_kernels": ([H], ctypes.c_int),
        "lapl_attn_destroy": ([H], st),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


LIB = _load()
EXPORTED = ["lapl_attn_version", "lapl_attn_status_string", "lapl_attn_last_error",
            "lapl_attn_create", "lapl_attn_workspace_size", "lapl_attn_forward",
            "lapl_attn_forward_train",
            "lapl_attn_forward_debug", "lapl_attn_host_staging_size", "lapl_attn_forward_host",
            "lapl_attn_set_timing", "lapl_attn_stage_times", "lapl_attn_stage_marks",
            "lapl_attn_kernels_per_forward",
            "lapl_attn_forward_noalloc", "lapl_attn_device_errors",
            "lapl_attn_set_fault_injection", "lapl_attn_plan_info_get",
            "lapl_attn_backward_workspace_size", "lapl_attn_backward",
            "lapl_attn_backward_kernels", "lapl_attn_destroy"]


def status_string(status: int) -> str:
    return LIB.lapl_attn_status_string(int(status)).decode()


def _check(status: int, where: str, handle=None):
    if status != LAPL_OK:
        detail = ""
        if handle is not None:
            detail = LIB.lapl_attn_last_error(handle).decode()
        raise LaplAttnError(status, where, detail)


# ---- same-name wrappers of the C entry points --------------------------------------------
def lapl_attn_version() -> int:
    return LIB.lapl_attn_version()


def lapl_attn_status_string(status: int) -> str:
    return status_string(status)


def lapl_attn_last_error(handle) -> str:
    return LIB.lapl_attn_last_error(handle).decode()


def lapl_attn_create(cfg: lapl_attn_config):
    h = ctypes.c_void_p()
    _check(LIB.lapl_attn_create(ctypes.byref(cfg), ctypes.byref(h)), "lapl_attn_create")
    return h


def lapl_attn_workspace_size(handle) -> int:
    n = ctypes.c_size_t()
    _check(LIB.lapl_attn_workspace_size(handle, ctypes.byref(n)), "lapl_attn_workspace_size")
    return n.value


def lapl_attn_host_staging_size(handle) -> int:
    n = ctypes.c_size_t()
    _check(LIB.lapl_attn_host_staging_size(handle, ctypes.byref(n)),
           "lapl_attn_host_staging_size")
    return n.value


def lapl_attn_forward(handle, q, k, v, bias, out, workspace, workspace_bytes, stream) -> None:
    _check(LIB.lapl_attn_forward(handle, q, k, v, bias, out, workspace, workspace_bytes, stream),
           "lapl_attn_forward", handle)


def lapl_attn_forward_train(handle, q, k, v, bias, out, workspace, workspace_bytes,
                            stream) -> None:
    _check(LIB.lapl_attn_forward_train(handle, q, k, v, bias, out, workspace, workspace_bytes,
                                       stream), "lapl_attn_forward_train", handle)


def lapl_attn_forward_debug(handle, q, k, v, bias, out, workspace, workspace_bytes, stream,
                            dbg: lapl_attn_debug) -> None:
    _check(LIB.lapl_attn_forward_debug(handle, q, k, v, bias, out, workspace, workspace_bytes,
                                       stream, ctypes.byref(dbg)),
           "lapl_attn_forward_debug", handle)


def lapl_attn_forward_host(handle, q, k, v, bias, out, staging, staging_bytes, stream) -> None:
    _check(LIB.lapl_attn_forward_host(handle, q, k, v, bias, out, staging, staging_bytes, stream),
           "lapl_attn_forward_host", handle)


def lapl_attn_forward_noalloc(handle, q, k, v, bias, out, stream) -> None:
    """Forward without a workspace argument (the library's static device scratch is used)."""
    _check(LIB.lapl_attn_forward_noalloc(handle, q, k, v, bias, out, stream),
           "lapl_attn_forward_noalloc", handle)


STAGES = ("pool", "newton_schulz", "cdist", "bv", "finish", "output")


def lapl_attn_set_timing(handle, enable: bool) -> None:
    _check(LIB.lapl_attn_set_timing(handle, int(bool(enable))), "lapl_attn_set_timing", handle)


def lapl_attn_stage_times(handle) -> dict:
    ms = (ctypes.c_float * len(STAGES))()
    _check(LIB.lapl_attn_stage_times(handle, ms), "lapl_attn_stage_times", handle)
    return dict(zip(STAGES, [float(x) for x in ms]))


MARKS = ("start", "pool_done", "ns_start", "ns_done", "cdist_start", "cdist_done", "bv_done",
         "mix_done", "output_done")


def lapl_attn_stage_marks(handle) -> dict:
    ms = (ctypes.c_float * len(MARKS))()
    _check(LIB.lapl_attn_stage_marks(handle, ms), "lapl_attn_stage_marks", handle)
    return dict(zip(MARKS, [float(x) for x in ms]))


def lapl_attn_kernels_per_forward(handle) -> int:
    return LIB.lapl_attn_kernels_per_forward(handle)


def lapl_attn_backward_workspace_size(handle) -> int:
    n = ctypes.c_size_t()
    _check(LIB.lapl_attn_backward_workspace_size(handle, ctypes.byref(n)),
           "lapl_attn_backward_workspace_size", handle)
    return n.value


def lapl_attn_backward(handle, q, k, v, bias, dout, dq, dk, dv, dbias, fwd_workspace,
                       fwd_workspace_bytes, bwd_workspace, bwd_workspace_bytes, stream) -> None:
    _check(LIB.lapl_attn_backward(handle, q, k, v, bias, dout, dq, dk, dv, dbias, fwd_workspace,
                                  fwd_workspace_bytes, bwd_workspace, bwd_workspace_bytes,
                                  stream), "lapl_attn_backward", handle)


def lapl_attn_backward_kernels(handle) -> int:
    return LIB.lapl_attn_backward_kernels(handle)


def lapl_attn_device_errors(handle, stream) -> int:
    """Read and clear the device error word (synchronises `stream`); raises on a set flag."""
    flags = ctypes.c_uint(0)
    _check(LIB.lapl_attn_device_errors(handle, stream, ctypes.byref(flags)),
           "lapl_attn_device_errors", handle)
    return flags.value


def lapl_attn_set_fault_injection(handle, wait_ns: int, skip_last_copy: int) -> None:
    _check(LIB.lapl_attn_set_fault_injection(handle, int(wait_ns), int(skip_last_copy)),
           "lapl_attn_set_fault_injection", handle)


def lapl_attn_plan_info_get(handle) -> dict:
    info = lapl_attn_plan_info()
    _check(LIB.lapl_attn_plan_info_get(handle, ctypes.byref(info)), "lapl_attn_plan_info_get",
           handle)
    return {name: int(getattr(info, name)) for name, _ in lapl_attn_plan_info._fields_}


def lapl_attn_destroy(handle) -> None:
    _check(LIB.lapl_attn_destroy(handle), "lapl_attn_destroy")
