"""GPU parity: the CUDA path (called through the C ABI) against the fp64 CPU oracle on the
same seeded inputs.

Bars: distance matrices and landmarks bit-exact on small-integer inputs; O within a normwise
relative error of 1e-4 per (b,h) slice for fp32 inputs and 2e-2 for bf16 inputs (the oracle
receives the bf16-rounded values, so both sides compute the same function).
"""
import ctypes

import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_bias, make_inputs
from parity_utils import (TOL_BF16, TOL_F32, elem_rel, oracle_each_slice, rel_to_max, run_gpu,
                          slice_rel_err, to_device, worst_slice)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    import oracle
    oracle.build()


def oracle_run(w, q, k, v, bias=None, slices=None, inter=False, **over):
    import oracle
    cfg = w.config()
    cfg.update(over)
    return oracle.forward(cfg, q, k, v, bias=bias, intermediates=inter, slices=slices)


def tol_of(w):
    return TOL_BF16 if w.dtype == "bf16" else TOL_F32


# ---- every intermediate on the tiny workload ------------------------------------------------
def test_tiny_intermediates():
    w = WORKLOADS["tiny_f32"]
    q, k, v = make_inputs(w)
    out, g = run_gpu(w, q, k, v, debug=True)
    ref, o = oracle_run(w, q, k, v, inter=True)
    assert rel_to_max(g["landmarks"], o["landmarks"]) < 1e-6
    assert elem_rel(g["d_ql"], o["d_ql"]) < 1e-5
    assert elem_rel(g["d_lk"], o["d_lk"]) < 1e-5
    assert rel_to_max(g["d_ll"], o["d_ll"]) < 1e-5
    assert elem_rel(g["a"], o["a"]) < 1e-5
    assert rel_to_max(g["w"], o["w"]) < 1e-6
    assert np.array_equal(np.diag(g["w"][0, 0]), np.full(16, np.float32(1) + np.float32(1e-3)))
    assert rel_to_max(g["x"], o["x"]) < 1e-4
    assert elem_rel(g["mu"], o["mu"]) < 1e-5
    rstd_ref = 1.0 / np.sqrt(o["var"] + w.config()["delta"])
    assert elem_rel(g["rstd"], rstd_ref) < 1e-4
    assert rel_to_max(g["bv"], o["bv"]) < 1e-5
    assert rel_to_max(g["m"], o["m_mat"]) < 1e-4
    assert slice_rel_err(out, ref) < TOL_F32


def test_integer_inputs_distances_bit_exact():
    w = WORKLOADS["tiny_int"]
    q, k, v = make_inputs(w)
    out, g = run_gpu(w, q, k, v, debug=True)
    ref, o = oracle_run(w, q, k, v, inter=True)
    for name in ("landmarks", "d_ql", "d_ll", "d_lk"):
        assert np.array_equal(g[name], o[name]), name
    assert slice_rel_err(out, ref) < TOL_F32


@pytest.mark.parametrize("name", ["stage1_f32", "stage23_bf16", "hires_bf16"])
def test_integer_variant_of_each_shape_bit_exact(name):
    """Same shapes and launch configuration as the workload, integer-valued Q and K."""
    w = WORKLOADS[name].replace(dist="integer", batch=1)
    q, k, v = make_inputs(w)
    _, g = run_gpu(w, q, k, v, debug=True)
    _, o = oracle_run(w, q, k, v, inter=True, slices=(0, 1))
    for nm in ("landmarks", "d_ql", "d_ll", "d_lk"):
        assert np.array_equal(g[nm][0, 0], o[nm][0, 0]), nm


# ---- the five workloads, end to end --------------------------------------------------------
FULL = ["tiny_f32", "stage1_f32", "stage23_bf16"]
# Large launches: the full-size forward on the GPU, then the oracle on every (b, h) slice, one
# slice per host thread.  Covers the high-resolution shape and the whole sequence-length
# sweep (fp32 and bf16, N = 1024 ... 65536).
EVERY_SLICE = ["hires_bf16"] + [f"sweep_{dt}_{n}" for dt in ("f32", "bf16")
                                for n in (1024, 4096, 16384, 65536)]


@pytest.mark.parametrize("name", FULL)
def test_workload_full(name):
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    out, _ = run_gpu(w, q, k, v)
    ref, _ = oracle_run(w, q, k, v)
    err = slice_rel_err(out, ref)
    assert err < tol_of(w), err


@pytest.mark.parametrize("name", EVERY_SLICE)
def test_workload_every_slice(name):
    """Full-size launch; the oracle computes every (b, h) slice."""
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    out, _ = run_gpu(w, q, k, v)
    assert np.isfinite(out).all()
    refs = oracle_each_slice(w.config(), q, k, v)
    assert len(refs) == w.batch * w.heads
    err, s = worst_slice(out, refs)
    assert err < tol_of(w), (s, err)


@pytest.mark.parametrize("name", ["hires_bf16", "sweep_f32_65536"])
def test_single_head_long_sequence(name):
    """B * H = 1 with 128 or 512 token chunks: the B V kernel's split count reaches its cap of
    64 CTAs per head (the M kernel stages every split's partial in shared memory)."""
    w = WORKLOADS[name].replace(batch=1, heads=1)
    q, k, v = make_inputs(w)
    info = {}
    out, _ = run_gpu(w, q, k, v, info=info)
    ref, _ = oracle_run(w, q, k, v)
    assert info["bv_splits"] == 64
    assert slice_rel_err(out, ref) < tol_of(w)


# ---- edge cases ----------------------------------------------------------------------------
TINY = WORKLOADS["tiny_f32"]

EDGE = {
    "ragged_14x14_m49": dict(grid_h=14, grid_w=14, num_landmarks=49),
    "nonsquare_20x12_m16": dict(grid_h=20, grid_w=12, num_landmarks=16),
    "m1": dict(num_landmarks=1),
    "m4": dict(num_landmarks=4),
    "m64_pool2": dict(num_landmarks=64),
    "single_token": dict(grid_h=1, grid_w=1, num_landmarks=1),
    "d8": dict(head_dim=8),
    "d16": dict(head_dim=16),
    "d24": dict(head_dim=24),
    "d128": dict(head_dim=128),
    "T0": dict(ns_steps=0),
    "T1": dict(ns_steps=1),
    "T3": dict(ns_steps=3),
    "whiten_off": dict(whiten=0),
    "lambda_large": dict(lam=1e6, eps=1.0, whiten=0),
    "batch_heads": dict(batch=3, heads=5),
    "n_equals_tile": dict(grid_h=8, grid_w=16, num_landmarks=4),
    "n_tile_plus_1": dict(grid_h=3, grid_w=43, num_landmarks=1),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_case(case):
    w = TINY.replace(**EDGE[case])
    q, k, v = make_inputs(w)
    out, _ = run_gpu(w, q, k, v)
    ref, _ = oracle_run(w, q, k, v)
    err = slice_rel_err(out, ref)
    assert err < TOL_F32, err


def test_unconverged_iteration_heavy_tailed():
    """T = 4 on a kappa ~ 65 landmark matrix: X is far from W^-1, the iterate itself is compared."""
    w = WORKLOADS["stage1_f32"].replace(batch=1, heads=2, ns_steps=4)
    q, k, v = make_inputs(w)
    out, g = run_gpu(w, q, k, v, debug=True)
    ref, o = oracle_run(w, q, k, v, inter=True)
    assert o["ns_resid"][0, 0, -1] > 0.5
    assert rel_to_max(g["x"], o["x"]) < 1e-5
    assert slice_rel_err(out, ref) < TOL_F32


def test_bias_and_bf16_output():
    w = TINY.replace(heads=3, batch=2)
    q, k, v = make_inputs(w)
    bias = make_bias(w)
    ref, _ = oracle_run(w, q, k, v, bias=bias)
    out, _ = run_gpu(w, q, k, v, bias=bias)
    assert slice_rel_err(out, ref) < TOL_F32
    out16, _ = run_gpu(w, q, k, v, bias=bias, out_dtype="bf16")
    assert slice_rel_err(out16, ref) < 2 ** -8


def test_constant_keys_closed_form_regime():
    w = TINY.replace(eps=1.0, ns_steps=30)
    q, k, v = make_inputs(w)
    k = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    out, _ = run_gpu(w, q, k, v)
    ref, _ = oracle_run(w, q, k, v)
    assert slice_rel_err(out, ref) < TOL_F32


def test_empty_batch():
    import torch
    import laplacian_nystr_attention_gb300 as lna
    w = TINY.replace(batch=0)
    att = lna.LaplacianNystromAttention(lna.make_config(**w.config()))
    z = torch.zeros((0, 1, 256, 32), device="cuda")
    out = att.forward(z, z, z)
    assert out.shape == (0, 1, 256, 32)
    att.close()


# ---- determinism, errors, host entry point ------------------------------------------------
def test_deterministic():
    w = WORKLOADS["stage1_f32"]
    q, k, v = make_inputs(w)
    a, _ = run_gpu(w, q, k, v)
    b, _ = run_gpu(w, q, k, v)
    assert np.array_equal(a, b)


def test_error_paths():
    import torch
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    w = TINY
    att = lna.LaplacianNystromAttention(lna.make_config(**w.config()))
    q = torch.randn(1, 1, 256, 32, device="cuda")
    out = torch.empty_like(q)
    h = att.handle
    st = torch.cuda.current_stream().cuda_stream
    ws = att.workspace
    L = _lib.LIB
    assert L.lapl_attn_forward(h, q.data_ptr(), q.data_ptr(), q.data_ptr(), None, out.data_ptr(),
                               ws.data_ptr(), att.workspace_bytes - 1, st) == _lib.LAPL_ERR_WORKSPACE
    assert L.lapl_attn_forward(h, q.data_ptr() + 4, q.data_ptr(), q.data_ptr(), None,
                               out.data_ptr(), ws.data_ptr(), att.workspace_bytes,
                               st) == _lib.LAPL_ERR_ALIGNMENT
    assert L.lapl_attn_forward(h, None, q.data_ptr(), q.data_ptr(), None, out.data_ptr(),
                               ws.data_ptr(), att.workspace_bytes, st) == _lib.LAPL_ERR_INVALID_ARG
    # the handle still works after rejected calls
    assert L.lapl_attn_forward(h, q.data_ptr(), q.data_ptr(), q.data_ptr(), None, out.data_ptr(),
                               ws.data_ptr(), att.workspace_bytes, st) == _lib.LAPL_OK
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    att.close()


HOST_CASES = {
    "stage1_batch2": ("stage1_f32", dict(batch=2), False),
    "stage1_full": ("stage1_f32", dict(), False),
    "stage23_batch3_bias": ("stage23_bf16", dict(batch=3), True),
    "tiny_batch1": ("tiny_f32", dict(), False),
    "sweep_bf16_4096_batch2": ("sweep_bf16_4096", dict(batch=2, heads=4), True),
}


@pytest.mark.parametrize("split", ["1", "0"])
@pytest.mark.parametrize("case", sorted(HOST_CASES))
def test_forward_host_matches_device_path(case, split, monkeypatch):
    """lapl_attn_forward_host (two half-batch forwards for a batch of two or more, or one with
    LAPL_ATTN_HOST_SPLIT=0) gives O bit for bit equal to lapl_attn_forward."""
    import torch
    import laplacian_nystr_attention_gb300 as lna
    name, over, with_bias = HOST_CASES[case]
    w = WORKLOADS[name].replace(**over)
    q, k, v = make_inputs(w)
    bias = make_bias(w) if with_bias else None
    dev, _ = run_gpu(w, q, k, v, bias=bias)
    monkeypatch.setenv("LAPL_ATTN_HOST_SPLIT", split)
    cfg = lna.make_config(**{**w.config(), "in_dtype": w.dtype})
    h = lna.lapl_attn_create(cfg)
    try:
        nbytes = lna.lapl_attn_host_staging_size(h)
        staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)) for x in (q, k, v))
        if w.dtype == "bf16":
            tq, tk, tv = (t.to(torch.bfloat16) for t in (tq, tk, tv))
        hq, hk, hv = (t.pin_memory() for t in (tq, tk, tv))
        hb = torch.from_numpy(np.ascontiguousarray(bias, dtype=np.float32)).pin_memory() \
            if with_bias else None
        hout = torch.full(q.shape, float("nan"), dtype=torch.float32).pin_memory()
        st = torch.cuda.current_stream()
        lna.lapl_attn_forward_host(h, hq.data_ptr(), hk.data_ptr(), hv.data_ptr(),
                                   hb.data_ptr() if hb is not None else None, hout.data_ptr(),
                                   staging.data_ptr(), nbytes, st.cuda_stream)
        st.synchronize()
        assert np.array_equal(hout.numpy().astype(np.float64), dev)
        assert lna.lapl_attn_device_errors(h, st.cuda_stream) == 0
    finally:
        lna.lapl_attn_destroy(h)
