"""GPU parity of the Gaussian-kernel variant (kernel = 1: k(x, y) = exp(-|x - y|_2^2 / lambda)
in A, B and W, every other step unchanged) against the fp64 CPU oracle.

The LaplacianFormer pages set the Laplacian kernel against the Gaussian one that softmax-free
attention uses (English explainer page, 1 "Theoretical Mismatch"); this variant is that
baseline run through the same Nystrom pipeline.  Bars as for the Laplacian kernel: distance
matrices bit-exact on small-integer inputs (every partial sum of squares of the dyadic
differences is a float32 integer multiple of the grid's unit, below 2^24 units, so the
summation order cannot matter), O within 1e-4 (fp32) / 2e-2 (bf16) normwise per (b, h) slice.
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_bias, make_inputs
from parity_utils import (TOL_BF16, TOL_F32, elem_rel, oracle_each_slice, rel_to_max, run_gpu,
                          slice_rel_err, worst_slice)

pytestmark = pytest.mark.gpu

GAUSS = 1


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
    cfg["kernel"] = GAUSS
    return oracle.forward(cfg, q, k, v, bias=bias, intermediates=inter, slices=slices)


def gpu_run(w, q, k, v, **kw):
    return run_gpu(w, q, k, v, kernel=GAUSS, **kw)


def tol_of(w):
    return TOL_BF16 if w.dtype == "bf16" else TOL_F32


def expected_feed(w) -> int:
    """plan_info cdist_tma: 3 where the tensor-core distance kernel is instantiated (d = 32 or
    64), else 0 (the CUDA-core kernel)."""
    return 3 if w.head_dim in (32, 64) else 0


def expansion_bound(x, lm):
    """Bound on |D_gpu - D| for D = |x - l|^2 evaluated as |x|^2 + |l|^2 - 2 x.l in fp32 with
    the cross term from TF32 high/low pieces: each of the three sums of at most d <= 64 terms
    rounds within (d + 4) 2^-24 of its sum of magnitudes, the dropped low x low product and the
    TF32 truncation of the low pieces add under 2^-20 of sum |x_c l_c|, and the fp32 landmarks
    differ from the exact ones by 2^-24 relative; 2^-17 covers all of it.  x [N, d], lm [m, d]
    (fp64); returns [N, m]."""
    ax, al = np.abs(x), np.abs(lm)
    nx = (x * x).sum(-1)
    nl = (lm * lm).sum(-1)
    return 2.0 ** -17 * (nx[:, None] + nl[None, :] + 2.0 * ax @ al.T)


def test_tiny_intermediates():
    w = WORKLOADS["tiny_f32"]
    q, k, v = make_inputs(w)
    info = {}
    out, g = gpu_run(w, q, k, v, debug=True, info=info)
    ref, o = oracle_run(w, q, k, v, inter=True)
    assert info["cdist_tma"] == expected_feed(w) and info["device_errors"] == 0
    assert rel_to_max(g["landmarks"], o["landmarks"]) < 1e-6
    # squared distances: same values as sum_c (x_c - y_c)^2 in fp64, to fp32 rounding
    qd = q[0, 0].astype(np.float64)
    lm = o["landmarks"][0, 0]
    brute = ((qd[:, None, :] - lm[None, :, :]) ** 2).sum(-1)
    assert elem_rel(o["d_ql"][0, 0], brute) < 1e-12
    assert elem_rel(g["d_ql"], o["d_ql"]) < 1e-5
    assert elem_rel(g["d_lk"], o["d_lk"]) < 1e-5
    assert rel_to_max(g["d_ll"], o["d_ll"]) < 1e-5
    assert elem_rel(g["a"], o["a"]) < 1e-5
    assert rel_to_max(g["w"], o["w"]) < 1e-6
    assert np.array_equal(g["w"][0, 0], g["w"][0, 0].T)
    assert np.array_equal(np.diag(g["w"][0, 0]), np.full(16, np.float32(1) + np.float32(1e-3)))
    assert rel_to_max(g["x"], o["x"]) < 1e-4
    assert elem_rel(g["mu"], o["mu"]) < 1e-5
    assert rel_to_max(g["bv"], o["bv"]) < 1e-5
    assert rel_to_max(g["m"], o["m_mat"]) < 1e-4
    assert slice_rel_err(out, ref) < TOL_F32


def test_differs_from_laplacian():
    """The kernel field reaches every distance: the Gaussian run's distances are the squared
    l2 ones, not the L1 ones of the default kernel."""
    w = WORKLOADS["tiny_int"]
    q, k, v = make_inputs(w)
    _, g = gpu_run(w, q, k, v, debug=True)
    _, l1 = run_gpu(w, q, k, v, debug=True)
    lm = g["landmarks"][0, 0]
    assert np.array_equal(lm, l1["landmarks"][0, 0])
    diff = q[0, 0].astype(np.float64)[:, None, :] - lm[None, :, :]
    assert np.array_equal(g["d_ql"][0, 0], (diff ** 2).sum(-1))
    assert np.array_equal(l1["d_ql"][0, 0], np.abs(diff).sum(-1))


@pytest.mark.parametrize("name", ["tiny_int", "stage1_f32", "stage23_bf16"])
def test_integer_inputs_distances_bit_exact(name):
    """Integer Q, K on {-3..3}: landmarks are multiples of 1/16 (tiny, stage 2/3) or 1/64
    (stage 1), and every partial sum of squared differences stays an exact float32."""
    w = WORKLOADS[name].replace(dist="integer", batch=1)
    q, k, v = make_inputs(w)
    out, g = gpu_run(w, q, k, v, debug=True)
    ref, o = oracle_run(w, q, k, v, inter=True, slices=(0, 1))
    for nm in ("landmarks", "d_ql", "d_ll", "d_lk"):
        assert np.array_equal(g[nm][0, 0], o[nm][0, 0]), nm
    assert slice_rel_err(out[0, 0][None, None], ref[0, 0][None, None]) < tol_of(w)


@pytest.mark.parametrize("name", ["tiny_f32", "stage1_f32", "stage23_bf16"])
def test_workload_full(name):
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    info = {}
    out, _ = gpu_run(w, q, k, v, info=info)
    ref, _ = oracle_run(w, q, k, v)
    assert info["cdist_tma"] == expected_feed(w) and info["device_errors"] == 0
    err = slice_rel_err(out, ref)
    assert err < tol_of(w), err


@pytest.mark.parametrize("name", ["hires_bf16", "sweep_f32_16384", "sweep_bf16_65536"])
def test_workload_every_slice(name):
    """Full-size launch; the oracle computes every (b, h) slice, one per host thread."""
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    out, _ = gpu_run(w, q, k, v)
    assert np.isfinite(out).all()
    cfg = w.config()
    cfg["kernel"] = GAUSS
    refs = oracle_each_slice(cfg, q, k, v)
    assert len(refs) == w.batch * w.heads
    err, s = worst_slice(out, refs)
    assert err < tol_of(w), (s, err)


TINY = WORKLOADS["tiny_f32"]
EDGE = {
    "ragged_14x14_m49": dict(grid_h=14, grid_w=14, num_landmarks=49),
    "m1": dict(num_landmarks=1),
    "m64_pool2": dict(num_landmarks=64),
    "single_token": dict(grid_h=1, grid_w=1, num_landmarks=1),
    "d8": dict(head_dim=8),
    "d24": dict(head_dim=24),
    "d128": dict(head_dim=128),
    "T0": dict(ns_steps=0),
    "whiten_off": dict(whiten=0),
    "lambda_64": dict(lam=64.0),
    "batch_heads": dict(batch=3, heads=5),
    "n_tile_plus_1": dict(grid_h=3, grid_w=43, num_landmarks=1),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_case(case):
    w = TINY.replace(**EDGE[case])
    q, k, v = make_inputs(w)
    out, _ = gpu_run(w, q, k, v)
    ref, _ = oracle_run(w, q, k, v)
    err = slice_rel_err(out, ref)
    assert err < TOL_F32, err


@pytest.mark.parametrize("ns", ["ffma", "tc"])
def test_both_solvers(ns, monkeypatch):
    """The CUDA-core and tensor-core Newton-Schulz kernels both take the Gaussian W."""
    monkeypatch.setenv("LAPL_ATTN_NS_KERNEL", ns)
    w = WORKLOADS["stage1_f32"].replace(batch=1)
    q, k, v = make_inputs(w)
    info = {}
    out, g = gpu_run(w, q, k, v, debug=True, info=info)
    ref, o = oracle_run(w, q, k, v, inter=True)
    assert info["ns_tensor_core"] == (1 if ns == "tc" else 0)
    assert rel_to_max(g["w"], o["w"]) < 1e-6
    assert slice_rel_err(out, ref) < TOL_F32


ILL = {
    # head dim 8: the landmarks sit close together in squared-l2 terms, W is nearly rank
    # deficient (kappa 1.8e3 .. 2.9e4) and 20 steps leave the slow modes unconverged
    "m16_d8": dict(head_dim=8),
    "m49_d8": dict(grid_h=14, grid_w=14, num_landmarks=49, head_dim=8),
    "m64_d8": dict(grid_h=16, grid_w=16, num_landmarks=64, head_dim=8),
    "m49_d8_28x28": dict(grid_h=28, grid_w=28, num_landmarks=49, head_dim=8),
}


@pytest.mark.parametrize("ns", ["ffma", "pair", "tc"])
@pytest.mark.parametrize("case", sorted(ILL))
def test_ill_conditioned_unconverged(case, ns, monkeypatch):
    """Every solver keeps X exactly symmetric by averaging V = 2X - X P with its transpose;
    on these matrices that holds O to the fp32 bar, where keeping one triangle of V does not.
    The pair request falls back to one CTA for m <= 32."""
    monkeypatch.setenv("LAPL_ATTN_NS_KERNEL", ns)
    w = TINY.replace(**ILL[case])
    q, k, v = make_inputs(w)
    out, g = gpu_run(w, q, k, v, debug=True)
    ref, o = oracle_run(w, q, k, v, inter=True)
    assert o["ns_resid"][0, 0, -1] > 0.5           # the iterate itself is compared
    x = g["x"][0, 0]
    assert np.array_equal(x, x.T)
    assert rel_to_max(g["x"], o["x"]) < 1e-4
    err = slice_rel_err(out, ref)
    assert err < TOL_F32, err


def test_bias_deterministic():
    w = TINY.replace(heads=3, batch=2)
    q, k, v = make_inputs(w)
    bias = make_bias(w)
    a, _ = gpu_run(w, q, k, v, bias=bias)
    b, _ = gpu_run(w, q, k, v, bias=bias)
    assert np.array_equal(a, b)
    ref, _ = oracle_run(w, q, k, v, bias=bias)
    assert slice_rel_err(a, ref) < TOL_F32


# Shapes for the tensor-core distance kernel against the direct sum: ragged chunks, one head,
# fewer rows than a chunk, every padding of m to 16 columns, both input types and head dims.
TC_CASES = {
    "f32_d32_m49_ragged": dict(batch=2, heads=2, grid_h=14, grid_w=14, num_landmarks=49),
    "f32_d64_m16_15heads": dict(batch=3, heads=5, grid_h=20, grid_w=12, head_dim=64,
                                num_landmarks=16),
    "bf16_d64_m49": dict(batch=2, heads=2, grid_h=28, grid_w=28, head_dim=64, num_landmarks=49,
                         dtype="bf16"),
    "bf16_d32_m16": dict(dtype="bf16"),
    "f32_d32_m1_129": dict(grid_h=3, grid_w=43, num_landmarks=1),
    "f32_d32_m64": dict(grid_h=16, grid_w=16, num_landmarks=64),
    "f32_d64_m36": dict(batch=2, heads=3, grid_h=12, grid_w=24, head_dim=64, num_landmarks=36),
    "f32_d32_m4_64_tokens": dict(grid_h=8, grid_w=8, num_landmarks=4),
    "f32_d32_m9": dict(grid_h=12, grid_w=12, num_landmarks=9),
    "f32_d32_m25": dict(grid_h=20, grid_w=20, num_landmarks=25),
}


def _dyadic_window(w) -> bool:
    s = int(round(w.num_landmarks ** 0.5))
    win = (w.grid_h // s) * (w.grid_w // s)
    return win & (win - 1) == 0


@pytest.mark.parametrize("case", sorted(TC_CASES))
def test_tensor_core_distances(case, monkeypatch):
    """The tensor-core kernel (|x|^2 + |l|^2 - 2 x.l) against the oracle and against the
    CUDA-core kernel's direct sum: bit for bit on integer inputs with dyadic landmarks (every
    term exact), within the expansion's rounding bound on float inputs; O within the bars."""
    w = TINY.replace(**TC_CASES[case])
    for dist in ("integer", "gaussian"):
        wd = w.replace(dist=dist)
        q, k, v = make_inputs(wd, seed=5)
        ref, o = oracle_run(wd, q, k, v, inter=True)
        runs = {}
        for feed in ("auto", "cp.async"):
            if feed == "auto":
                monkeypatch.delenv("LAPL_ATTN_CDIST_FEED", raising=False)
            else:
                monkeypatch.setenv("LAPL_ATTN_CDIST_FEED", feed)
            info = {}
            runs[feed] = gpu_run(wd, q, k, v, debug=True, info=info)
            assert info["device_errors"] == 0
            assert info["cdist_tma"] == (expected_feed(wd) if feed == "auto" else 0)
        (out, g), (out_d, g_d) = runs["auto"], runs["cp.async"]
        if dist == "integer" and _dyadic_window(wd):
            for name in ("d_ql", "d_lk", "a"):
                assert np.array_equal(g[name], g_d[name]), name
            assert np.array_equal(g["d_ql"], o["d_ql"])
            assert np.array_equal(g["d_lk"], o["d_lk"])
        else:
            for b in range(wd.batch):
                for h in range(wd.heads):
                    lm = o["landmarks"][b, h]
                    bq = expansion_bound(q[b, h].astype(np.float64), lm)
                    bk = expansion_bound(k[b, h].astype(np.float64), lm)
                    assert (np.abs(g["d_ql"][b, h] - o["d_ql"][b, h]) <= bq).all(), (b, h)
                    assert (np.abs(g["d_lk"][b, h].T - o["d_lk"][b, h].T) <= bk).all(), (b, h)
        # O against the oracle, and against the direct sum's O to the same bar: on integer
        # inputs at d = 64 the kernel values reach the fp32 normal limit, where the
        # exponential flushes to zero and a last-bit difference of D decides which entries do.
        assert slice_rel_err(out, ref) < tol_of(wd)
        assert slice_rel_err(out, out_d) < tol_of(wd)


def test_tensor_core_timeout_reported():
    """Fault injection reaches the tensor-core distance kernel: its converters never publish
    each CTA's last chunk, the MMA and epilogue waits run out, the distance kernel's bit is
    reported, and a normal forward afterwards matches the oracle."""
    import ctypes
    import torch
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    from parity_utils import to_device
    w = WORKLOADS["stage1_f32"].replace(batch=2)
    q, k, v = make_inputs(w)
    dq, dk, dv = (to_device(x, w.dtype) for x in (q, k, v))
    cfg = {**w.config(), "in_dtype": w.dtype, "kernel": GAUSS}
    h = lna.lapl_attn_create(lna.make_config(**cfg))
    try:
        assert lna.lapl_attn_plan_info_get(h)["cdist_tma"] == 3
        nbytes = lna.lapl_attn_workspace_size(h)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = torch.empty(dq.shape, dtype=torch.float32, device="cuda")
        st = torch.cuda.current_stream().cuda_stream
        args = (h, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, out.data_ptr(),
                ws.data_ptr(), nbytes, st)
        lna.lapl_attn_device_errors(h, st)
        lna.lapl_attn_set_fault_injection(h, 50_000, 1)
        lna.lapl_attn_forward(*args)
        flags = ctypes.c_uint(0)
        assert _lib.LIB.lapl_attn_device_errors(h, st, ctypes.byref(flags)) == \
            _lib.LAPL_ERR_DEVICE_TIMEOUT
        assert flags.value == 1
        lna.lapl_attn_set_fault_injection(h, 0, 0)
        out.fill_(float("nan"))
        lna.lapl_attn_forward(*args)
        assert lna.lapl_attn_device_errors(h, st) == 0
        ref, _ = oracle_run(w, q, k, v)
        assert slice_rel_err(out.cpu().numpy().astype(np.float64), ref) < TOL_F32
    finally:
        lna.lapl_attn_destroy(h)
