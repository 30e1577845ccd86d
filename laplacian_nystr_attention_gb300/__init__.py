"""GB300 (sm_103a) Laplacian-kernel Nystrom attention, forward pass.

Per (batch, head): landmarks L = 2-D average pooling of K; A = exp(-cdist_L1(Q, L)/lambda),
whitened column-wise; W = exp(-cdist_L1(L, L)/lambda) + eps I inverted by T Newton-Schulz
steps; B = exp(-cdist_L1(L, K)/lambda); O = A^ (X (B V)).  ("LaplacianFormer: Rethinking
Linear Attention with Laplacian Kernel", explainer pages.)

The compute lives in liblapl_attn.so (hand-written CUDA kernels, C ABI in
include/lapl_attn.h).  ``_lib`` binds that ABI with the same names; ``LaplacianNystromAttention``
below is a convenience layer that uses PyTorch only to allocate device memory and to pick the
current CUDA stream.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (LAPL_BF16, LAPL_F32, LAPL_KERNEL_GAUSSIAN, LAPL_KERNEL_LAPLACIAN,
                   LAPL_SOLVER_CG, LAPL_SOLVER_NEWTON_SCHULZ, LaplAttnError, lapl_attn_config, lapl_attn_create,
                   lapl_attn_debug, lapl_attn_destroy, lapl_attn_device_errors,
                   lapl_attn_forward, lapl_attn_set_fault_injection,
                   lapl_attn_forward_debug, lapl_attn_forward_host, lapl_attn_host_staging_size,
                   lapl_attn_kernels_per_forward, lapl_attn_last_error,
                   lapl_attn_set_timing, lapl_attn_stage_marks, lapl_attn_stage_times,
                   lapl_attn_status_string,
                   lapl_attn_plan_info_get, lapl_attn_version, lapl_attn_workspace_size,
                   lapl_attn_backward, lapl_attn_backward_kernels, lapl_attn_forward_train,
                   lapl_attn_backward_workspace_size)

__all__ = [
    "LaplacianNystromAttention", "LaplAttnError", "lapl_attn_config", "lapl_attn_debug",
    "lapl_attn_create", "lapl_attn_destroy", "lapl_attn_forward", "lapl_attn_forward_debug",
    "lapl_attn_forward_host", "lapl_attn_host_staging_size", "lapl_attn_last_error",
    "lapl_attn_status_string", "lapl_attn_version", "lapl_attn_workspace_size", "LAPL_F32",
    "LAPL_BF16", "lapl_attn_set_timing", "lapl_attn_stage_times", "lapl_attn_stage_marks",
    "lapl_attn_kernels_per_forward", "lapl_attn_device_errors", "lapl_attn_set_fault_injection",
    "lapl_attn_plan_info_get",
    "make_config", "lapl_attn_backward", "lapl_attn_backward_kernels", "lapl_attn_forward_train",
    "lapl_attn_backward_workspace_size", "LAPL_KERNEL_LAPLACIAN", "LAPL_KERNEL_GAUSSIAN", "LAPL_SOLVER_NEWTON_SCHULZ",
    "LAPL_SOLVER_CG",
]

_DTYPES = {"f32": LAPL_F32, "bf16": LAPL_BF16}
_KERNELS = {"laplacian": LAPL_KERNEL_LAPLACIAN, "gaussian": LAPL_KERNEL_GAUSSIAN}
_SOLVERS = {"newton_schulz": LAPL_SOLVER_NEWTON_SCHULZ, "cg": LAPL_SOLVER_CG}


def make_config(batch, heads, grid_h, grid_w, head_dim, num_landmarks, lam=4.0, eps=1e-3,
                delta=1e-5, ns_steps=20, whiten=1, in_dtype="f32", out_dtype="f32",
                kernel="laplacian", solver="newton_schulz", **_ignored) -> lapl_attn_config:
    """kernel: "laplacian" (exp(-L1 / lam), the method) or "gaussian" (exp(-squared l2 / lam)),
    or the lapl_kernel integer.  solver: "newton_schulz" (X by ns_steps Newton-Schulz steps,
    M = X (B V)) or "cg" (ns_steps conjugate-gradient iterations on W M = B V), or the
    lapl_solver integer."""
    return lapl_attn_config(int(batch), int(heads), int(grid_h), int(grid_w), int(head_dim),
                            int(num_landmarks), float(lam), float(eps), float(delta),
                            int(ns_steps), int(whiten), _DTYPES.get(in_dtype, in_dtype),
                            _DTYPES.get(out_dtype, out_dtype), _KERNELS.get(kernel, kernel),
                            _SOLVERS.get(solver, solver))


class LaplacianNystromAttention:
    """One plan plus its device workspace (allocated with torch on the current device)."""

    def __init__(self, cfg: lapl_attn_config):
        import torch
        self.cfg = cfg
        self.handle = lapl_attn_create(cfg)
        self.workspace_bytes = lapl_attn_workspace_size(self.handle)
        self.workspace = torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8,
                                     device="cuda")

    @classmethod
    def from_dict(cls, d: dict, **kw):
        c = dict(d)
        c.update(kw)
        if "dtype" in c and "in_dtype" not in c:
            c["in_dtype"] = c["dtype"]
        return cls(make_config(**c))

    def _torch_dtype(self, code):
        import torch
        return torch.bfloat16 if code == LAPL_BF16 else torch.float32

    def _check_io(self, t, dtype_code, name):
        import torch
        c = self.cfg
        shape = (c.batch, c.heads, c.grid_h * c.grid_w, c.head_dim)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name}: expected shape {shape}, got {tuple(t.shape)}")
        if t.dtype != self._torch_dtype(dtype_code):
            raise ValueError(f"{name}: expected {self._torch_dtype(dtype_code)}, got {t.dtype}")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: must be a contiguous CUDA tensor")
        return t

    def forward(self, q, k, v, bias=None, out=None, stream=None, debug: dict | None = None,
                keep_for_backward: bool = False):
        """O = attention(q, k, v) on ``stream`` (default: torch's current stream).

        debug: optional dict name -> fp32 CUDA tensor for the lapl_attn_debug fields.
        keep_for_backward: run lapl_attn_forward_train, which keeps the Newton-Schulz iterates
        that backward() needs.
        """
        import torch
        c = self.cfg
        for name, t in (("q", q), ("k", k), ("v", v)):
            self._check_io(t, c.in_dtype, name)
        if out is None:
            out = torch.empty((c.batch, c.heads, c.grid_h * c.grid_w, c.head_dim),
                              dtype=self._torch_dtype(c.out_dtype), device=q.device)
        self._check_io(out, c.out_dtype, "out")
        if bias is not None:
            if tuple(bias.shape) != (c.heads, c.num_landmarks) or bias.dtype != torch.float32:
                raise ValueError("bias must be a float32 [H, m] tensor")
            bias = bias.contiguous()
        st = stream if stream is not None else torch.cuda.current_stream()
        args = (self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                bias.data_ptr() if bias is not None else None, out.data_ptr(),
                self.workspace.data_ptr(), self.workspace_bytes, st.cuda_stream)
        if debug:
            dbg = lapl_attn_debug(**{kname: t.data_ptr() for kname, t in debug.items()})
            lapl_attn_forward_debug(*args, dbg)
        elif keep_for_backward:
            lapl_attn_forward_train(*args)
        else:
            lapl_attn_forward(*args)
        self._kept = bool(keep_for_backward) and not debug
        return out

    __call__ = forward

    def backward(self, q, k, v, dout, bias=None, grads=None, stream=None):
        """(dq, dk, dv, dbias) for a loss with dLoss/dO = dout, after
        forward(q, k, v, bias, keep_for_backward=True) on this object (whose workspace holds
        what that forward kept; run nothing else on it in between).  dout: fp32 [B,H,N,d].  grads: optional dict with preallocated fp32 "dq",
        "dk", "dv" ([B,H,N,d]) and "dbias" ([H,m]) tensors.  The backward workspace is
        allocated on first use."""
        import torch
        c = self.cfg
        if not getattr(self, "_kept", False):
            raise RuntimeError("backward() needs a preceding forward(..., keep_for_backward=True)")
        for name, t in (("q", q), ("k", k), ("v", v)):
            self._check_io(t, c.in_dtype, name)
        self._check_io(dout, LAPL_F32, "dout")
        shape = (c.batch, c.heads, c.grid_h * c.grid_w, c.head_dim)
        g = dict(grads or {})
        for name in ("dq", "dk", "dv"):
            if name not in g:
                g[name] = torch.empty(shape, dtype=torch.float32, device=q.device)
            self._check_io(g[name], LAPL_F32, name)
        if "dbias" not in g:
            g["dbias"] = torch.empty((c.heads, c.num_landmarks), dtype=torch.float32,
                                     device=q.device)
        if bias is not None:
            bias = bias.contiguous()
        if getattr(self, "bwd_workspace", None) is None:
            self.bwd_workspace_bytes = lapl_attn_backward_workspace_size(self.handle)
            self.bwd_workspace = torch.empty(max(self.bwd_workspace_bytes, 256),
                                             dtype=torch.uint8, device=q.device)
        st = stream if stream is not None else torch.cuda.current_stream()
        lapl_attn_backward(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           bias.data_ptr() if bias is not None else None, dout.data_ptr(),
                           g["dq"].data_ptr(), g["dk"].data_ptr(), g["dv"].data_ptr(),
                           g["dbias"].data_ptr(), self.workspace.data_ptr(),
                           self.workspace_bytes, self.bwd_workspace.data_ptr(),
                           self.bwd_workspace_bytes, st.cuda_stream)
        return g["dq"], g["dk"], g["dv"], g["dbias"]

    def close(self):
        if getattr(self, "handle", None) is not None:
            lapl_attn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
