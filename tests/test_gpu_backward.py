"""GPU parity of the backward pass (lapl_attn_backward) against the fp64 oracle's backward.

Comparison, per (b, h) slice and gradient (dQ, dK, dV; dbias per head): with scale = max |ref|
over the slice, every entry must satisfy |gpu - ref| <= tol * scale + amb, where amb is the
oracle's tie bound -- for the Laplacian kernel, how far the entry can move when a sign
decision sgn(x - y) with |x - y| <= 2^-15 (|x| + |y|) goes the other way (the GPU pools the
landmarks in float32, so such decisions are not unique); zero for the Gaussian kernel and for
dV and dbias.  On integer inputs the landmarks are exact dyadic values on both sides, every
sign decision (sgn(0) = 0 included) is the same, and amb is not used.
tol = 1e-4 (fp32 inputs) / 2e-2 (bf16 inputs; the oracle receives the bf16-rounded values).
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_bias, make_inputs
from parity_utils import TOL_BF16, TOL_F32, to_device

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


def tol_of(w):
    return TOL_BF16 if w.dtype == "bf16" else TOL_F32


def make_dout(w, seed=21):
    return np.random.default_rng(seed).standard_normal(
        (w.batch, w.heads, w.n, w.head_dim)).astype(np.float32)


def gpu_backward(w, q, k, v, G, bias=None, **over):
    import torch
    import laplacian_nystr_attention_gb300 as lna
    cfg = w.config()
    cfg.update(over)
    cfg["in_dtype"] = cfg.pop("dtype", w.dtype)
    att = lna.LaplacianNystromAttention(lna.make_config(**cfg))
    dq_, dk_, dv_ = (to_device(x, cfg["in_dtype"]) for x in (q, k, v))
    db = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    dG = torch.from_numpy(np.ascontiguousarray(G, np.float32)).cuda()
    att.forward(dq_, dk_, dv_, bias=db, keep_for_backward=True)
    gq, gk, gv, gb = att.backward(dq_, dk_, dv_, dG, bias=db)
    torch.cuda.synchronize()
    res = tuple(t.cpu().numpy().astype(np.float64) for t in (gq, gk, gv, gb))
    att.close()
    return res


def oracle_backward(w, q, k, v, G, bias=None, slices=None, **over):
    import oracle
    cfg = w.config()
    cfg.update(over)
    return oracle.backward(cfg, q, k, v, G, bias=bias, slices=slices)


def check(name, gpu, ref, amb, tol, slices):
    for s in slices:
        b, h = s
        g, r = gpu[b, h], ref[b, h]
        a = amb[b, h] if amb is not None else 0.0
        scale = max(np.abs(r).max(), 1e-30)
        excess = np.abs(g - r) - (tol * scale + a)
        assert excess.max() <= 0, (name, s, float(np.abs(g - r).max() / scale))


def compare(w, got, ref, tol, slices, use_amb=True):
    dq, dk, dv, db = got
    rq, rk, rv, rb, aq, ak = ref
    check("dq", dq, rq, aq if use_amb else None, tol, slices)
    check("dk", dk, rk, ak if use_amb else None, tol, slices)
    check("dv", dv, rv, None, tol, slices)
    scale = max(np.abs(rb).max(), 1e-30)
    assert np.abs(db - rb).max() <= tol * scale


def all_slices(w):
    return [(b, h) for b in range(w.batch) for h in range(w.heads)]


TINY = WORKLOADS["tiny_f32"]


@pytest.mark.parametrize("kernel", [0, 1])
def test_tiny(kernel):
    w = TINY.replace(heads=2)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    bias = make_bias(w)
    got = gpu_backward(w, q, k, v, G, bias=bias, kernel=kernel)
    ref = oracle_backward(w, q, k, v, G, bias=bias, kernel=kernel)
    compare(w, got, ref, TOL_F32, all_slices(w))


def test_integer_inputs_same_sign_decisions():
    w = WORKLOADS["tiny_int"].replace(heads=2)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    got = gpu_backward(w, q, k, v, G)
    ref = oracle_backward(w, q, k, v, G)
    assert ref[4].any()                           # ties are present, and must agree
    compare(w, got, ref, TOL_F32, all_slices(w), use_amb=False)


@pytest.mark.parametrize("name", ["stage1_f32", "stage23_bf16"])
def test_integer_variant_of_shape(name):
    w = WORKLOADS[name].replace(dist="integer", batch=1, heads=1)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    got = gpu_backward(w, q, k, v, G)
    ref = oracle_backward(w, q, k, v, G)
    compare(w, got, ref, tol_of(w), all_slices(w), use_amb=False)


@pytest.mark.parametrize("name,batch", [("stage1_f32", 1), ("stage23_bf16", 1)])
def test_workload(name, batch):
    w = WORKLOADS[name].replace(batch=batch)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    got = gpu_backward(w, q, k, v, G)
    ref = oracle_backward(w, q, k, v, G)
    compare(w, got, ref, tol_of(w), all_slices(w))


def test_high_resolution_first_slice():
    w = WORKLOADS["hires_bf16"].replace(batch=1, heads=2)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    got = gpu_backward(w, q, k, v, G)
    ref = oracle_backward(w, q, k, v, G, slices=(0, 1))
    dq, dk, dv, _ = got
    compare(w, (dq, dk, dv, ref[3]), ref, tol_of(w), [(0, 0)])


EDGE = {
    "no_whiten": dict(whiten=0),
    "m1": dict(num_landmarks=1),
    "m64": dict(num_landmarks=64),
    "ragged_14x14_m49": dict(grid_h=14, grid_w=14, num_landmarks=49),
    "nonsquare_20x12_m16": dict(grid_h=20, grid_w=12, num_landmarks=16),
    "d8": dict(head_dim=8),
    "d24": dict(head_dim=24),
    "d128": dict(head_dim=128),
    "T0": dict(ns_steps=0),
    "T3": dict(ns_steps=3),
    "batch_heads": dict(batch=3, heads=2),
    "gaussian_no_whiten": dict(kernel=1, whiten=0),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_case(case):
    over = dict(EDGE[case])
    kern = over.pop("kernel", 0)
    w = TINY.replace(**over)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    bias = make_bias(w)
    got = gpu_backward(w, q, k, v, G, bias=bias, kernel=kern)
    ref = oracle_backward(w, q, k, v, G, bias=bias, kernel=kern)
    compare(w, got, ref, TOL_F32, all_slices(w))


def test_deterministic():
    w = WORKLOADS["stage1_f32"].replace(batch=1)
    q, k, v = make_inputs(w)
    G = make_dout(w)
    a = gpu_backward(w, q, k, v, G)
    b = gpu_backward(w, q, k, v, G)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_unsupported_with_cg_and_errors():
    import torch
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    att = lna.LaplacianNystromAttention(lna.make_config(**TINY.config(), solver="cg"))
    with pytest.raises(_lib.LaplAttnError) as e:
        lna.lapl_attn_backward_workspace_size(att.handle)
    assert e.value.status == _lib.LAPL_ERR_UNSUPPORTED
    att.close()
    att = lna.LaplacianNystromAttention(lna.make_config(**TINY.config()))
    nbytes = lna.lapl_attn_backward_workspace_size(att.handle)
    assert lna.lapl_attn_backward_kernels(att.handle) == 8     # dA^, mid, NS, query, key, dL
                                                               # partials, dL, pooling
    x = torch.zeros((1, 1, 256, 32), device="cuda")
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    L = _lib.LIB
    p = x.data_ptr()
    assert L.lapl_attn_backward(att.handle, p, p, p, None, p, p, p, p, None,
                                att.workspace.data_ptr(), att.workspace_bytes, ws.data_ptr(),
                                nbytes - 1, st) == _lib.LAPL_ERR_WORKSPACE
    assert L.lapl_attn_backward(att.handle, p + 4, p, p, None, p, p, p, p, None,
                                att.workspace.data_ptr(), att.workspace_bytes, ws.data_ptr(),
                                nbytes, st) == _lib.LAPL_ERR_ALIGNMENT
    att.close()


def test_training_forward_same_output_and_backward_needs_it():
    import torch
    import laplacian_nystr_attention_gb300 as lna
    w = WORKLOADS["stage1_f32"].replace(batch=1)
    q, k, v = (to_device(x, "f32") for x in make_inputs(w))
    att = lna.LaplacianNystromAttention(lna.make_config(**w.config()))
    a = att.forward(q, k, v).clone()
    with pytest.raises(RuntimeError):
        att.backward(q, k, v, torch.zeros_like(q))
    b = att.forward(q, k, v, keep_for_backward=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    att.close()
