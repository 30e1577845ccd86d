"""Helpers shared by the GPU parity tests: run the CUDA path (through the C ABI) and the CPU
oracle on the same seeded inputs and compare.

Error metric for O (floating point): per (b, h) slice, max|O - O_ref| / max|O_ref|, reported
as the maximum over slices.  O has zero column means after whitening, so many entries are
near zero and an elementwise relative error would be ill-posed.
"""
from __future__ import annotations

import ctypes

import numpy as np

# Tolerances on O (normwise per slice, see module docstring).
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def slice_rel_err(out: np.ndarray, ref: np.ndarray) -> float:
    """max over (b,h) of max|out-ref| / max|ref|."""
    if out.size == 0:
        return 0.0
    o = out.reshape(-1, out.shape[-2] * out.shape[-1]).astype(np.float64)
    r = ref.reshape(-1, ref.shape[-2] * ref.shape[-1]).astype(np.float64)
    num = np.abs(o - r).max(axis=1)
    den = np.abs(r).max(axis=1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def rel_to_max(out: np.ndarray, ref: np.ndarray) -> float:
    ref = ref.astype(np.float64)
    den = np.abs(ref).max()
    return float(np.abs(out.astype(np.float64) - ref).max() / (den if den > 0 else 1.0))


def elem_rel(out: np.ndarray, ref: np.ndarray, floor_frac: float = 1e-6) -> float:
    """max |out-ref| / max(|ref|, floor_frac * max|ref|)."""
    ref = ref.astype(np.float64)
    floor = floor_frac * max(np.abs(ref).max(), 1e-300)
    return float((np.abs(out.astype(np.float64) - ref) / np.maximum(np.abs(ref), floor)).max())


def to_device(arr: np.ndarray, dtype: str):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)          # exact: the values are bf16-representable
    return t.cuda()


def run_gpu(w, q, k, v, bias=None, debug=False, out_dtype="f32", info=None, **cfg_over):
    """Run the CUDA path via the C ABI.  Returns (out float64 ndarray, dict of intermediates).

    info: optional dict that receives the plan's launch choices (lapl_attn_plan_info fields)
    and "device_errors" (the device error word after the forward, then cleared)."""
    import torch
    import laplacian_nystr_attention_gb300 as lna
    cfg = w.config()
    cfg.update(cfg_over)
    cfg["in_dtype"] = cfg.pop("dtype", w.dtype)
    cfg["out_dtype"] = out_dtype
    att = lna.LaplacianNystromAttention(lna.make_config(**cfg))
    B, H, N, d, m = w.batch, w.heads, w.n, w.head_dim, cfg["num_landmarks"]
    dq, dk, dv = (to_device(x, cfg["in_dtype"]) for x in (q, k, v))
    db = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    dbg = None
    if debug:
        shapes = dict(d_ql=(B, H, N, m), d_ll=(B, H, m, m), d_lk=(B, H, m, N),
                      landmarks=(B, H, m, d), w=(B, H, m, m), x=(B, H, m, m), a=(B, H, N, m),
                      mu=(B, H, m), rstd=(B, H, m), bv=(B, H, m, d), m=(B, H, m, d))
        dbg = {kname: torch.full(s, float("nan"), dtype=torch.float32, device="cuda")
               for kname, s in shapes.items()}
    out = att.forward(dq, dk, dv, bias=db, debug=dbg)
    torch.cuda.synchronize()
    if info is not None:
        info.update(lna.lapl_attn_plan_info_get(att.handle))
        flags = ctypes.c_uint(0)
        lna._lib.LIB.lapl_attn_device_errors(att.handle, torch.cuda.current_stream().cuda_stream,
                                            ctypes.byref(flags))
        info["device_errors"] = flags.value
    res = out.float().cpu().numpy().astype(np.float64)
    inter = {kname: t.cpu().numpy().astype(np.float64) for kname, t in (dbg or {}).items()}
    att.close()
    return res, inter


def host_threads() -> int:
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_each_slice(cfg: dict, q, k, v, bias=None, slices=None):
    """The oracle's output for each (b, h) slice, computed one slice per host thread (the
    oracle's C call releases the GIL).  Each slice is its own 1 x 1 problem: every step of the
    method is per (batch, head), so this is the same arithmetic as the full call.

    Returns {s: [N, d] float64} for s = b * H + h over ``slices`` (default: all)."""
    import concurrent.futures as cf

    import oracle
    B, H = int(cfg["batch"]), int(cfg["heads"])
    one = dict(cfg, batch=1, heads=1)
    todo = range(B * H) if slices is None else slices

    def run(s):
        b, h = divmod(s, H)
        bb = None if bias is None else np.asarray(bias)[h:h + 1]
        out, _ = oracle.forward(one, q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                v[b:b + 1, h:h + 1], bias=bb)
        return s, out[0, 0]

    oracle.build()
    with cf.ThreadPoolExecutor(max_workers=host_threads()) as ex:
        return dict(ex.map(run, todo))


def worst_slice(out: np.ndarray, refs: dict) -> tuple:
    """(largest per-slice normwise error, its slice) of ``out`` [B,H,N,d] against
    ``oracle_each_slice`` results."""
    H = out.shape[1]
    worst = (0.0, -1)
    for s, r in refs.items():
        b, h = divmod(s, H)
        e = slice_rel_err(out[b, h][None, None], r[None, None])
        worst = max(worst, (e, s))
    return worst
