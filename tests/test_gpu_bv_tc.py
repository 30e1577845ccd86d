"""B V on the tensor cores (bv_tc.cu) against the oracle.

The kernel runs by default for d = 64 and, for smaller head dims, for sequences of at least
4096 tokens (covered end to end by the every-slice workload tests); LAPL_ATTN_BV=tc forces it
here on short, ragged and edge shapes.
B V itself is compared with the oracle's intermediate: the TF32 high/low split leaves out only
the product of the two low parts (2^-20 relative), so the bar is 1e-5 of the largest entry.
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_bias, make_inputs
from parity_utils import TOL_BF16, TOL_F32, rel_to_max, run_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny_f32"]

CASES = {
    "tiny_f32": dict(),
    "tiny_bf16": dict(dtype="bf16"),
    "ragged_14x14_m49": dict(grid_h=14, grid_w=14, num_landmarks=49),
    "m1": dict(num_landmarks=1),
    "m64": dict(num_landmarks=64),
    "d16": dict(head_dim=16),
    "d64_bf16_2x3": dict(batch=2, heads=3, head_dim=64, dtype="bf16"),
    "d64_f32": dict(head_dim=64),
    "no_whiten": dict(whiten=0),
    "stage1_shape": dict(batch=8, heads=2, grid_h=56, grid_w=56, num_landmarks=49,
                         dist="student_t"),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    import oracle
    oracle.build()


@pytest.mark.parametrize("case", sorted(CASES))
def test_bv_tensor_core_matches_oracle(case, monkeypatch):
    import oracle
    monkeypatch.setenv("LAPL_ATTN_BV", "tc")
    w = TINY.replace(**CASES[case])
    q, k, v = make_inputs(w, seed=5)
    info = {}
    out, g = run_gpu(w, q, k, v, debug=True, info=info)
    assert info["bv_tensor_core"] == 1
    assert info["device_errors"] == 0
    ref, o = oracle.forward(w.config(), q, k, v, intermediates=True)
    assert rel_to_max(g["bv"], o["bv"]) < 1e-5
    if w.whiten:
        assert np.allclose(g["mu"], o["mu"], rtol=1e-5, atol=0)
    tol = TOL_BF16 if w.dtype == "bf16" else TOL_F32
    assert slice_rel_err(out, ref) < tol


def test_bv_tensor_core_with_bias_and_cg(monkeypatch):
    import oracle
    monkeypatch.setenv("LAPL_ATTN_BV", "tc")
    w = TINY.replace(batch=2, heads=2, num_landmarks=16)
    q, k, v = make_inputs(w, seed=9)
    bias = make_bias(w)
    for solver in (0, 1):
        info = {}
        out, _ = run_gpu(w, q, k, v, bias=bias, info=info, solver=solver)
        assert info["bv_tensor_core"] == 1 and info["device_errors"] == 0
        cfg = w.config()
        cfg["solver"] = solver
        ref, _ = oracle.forward(cfg, q, k, v, bias=bias)
        assert slice_rel_err(out, ref) < TOL_F32, solver


def test_bv_choice(monkeypatch):
    """Automatic: tensor cores for d = 64, for smaller d from 4096 tokens; never for N not a
    multiple of 4 or d not a multiple of 16; LAPL_ATTN_BV=cuda turns it off."""
    import laplacian_nystr_attention_gb300 as lna

    def choice(w):
        h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": w.dtype}))
        try:
            return lna.lapl_attn_plan_info_get(h)["bv_tensor_core"]
        finally:
            lna.lapl_attn_destroy(h)

    monkeypatch.delenv("LAPL_ATTN_BV", raising=False)
    assert choice(WORKLOADS["hires_bf16"]) == 1
    assert choice(WORKLOADS["sweep_f32_4096"]) == 1
    assert choice(WORKLOADS["stage1_f32"]) == 0                               # d = 32
    assert choice(WORKLOADS["stage23_bf16"]) == 1                             # d = 64
    monkeypatch.setenv("LAPL_ATTN_BV", "tc")
    assert choice(TINY) == 1
    assert choice(TINY.replace(grid_h=3, grid_w=43, num_landmarks=1)) == 0    # N = 129
    assert choice(TINY.replace(head_dim=24)) == 0
    monkeypatch.setenv("LAPL_ATTN_BV", "cuda")
    assert choice(WORKLOADS["hires_bf16"]) == 0


@pytest.mark.parametrize("debug", [False, True])
def test_statistics_beside_bv_same_output(debug, monkeypatch):
    """The column statistics on a stream of their own beside the tensor-core B V (forced on a
    shape whose distance chain runs on the launching stream) give the same output and the same
    statistics bit for bit as the statistics launched before B V, and match the oracle."""
    import oracle
    w = WORKLOADS["stage23_bf16"].replace(batch=12)        # 48 heads: the distance chain leads
    q, k, v = make_inputs(w)
    runs = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("LAPL_ATTN_STATS_BESIDE", mode)
        info = {}
        runs[mode] = run_gpu(w, q, k, v, debug=debug, info=info)
        assert info["bv_tensor_core"] == 1 and info["ns_exclusive"] == 0
        assert info["device_errors"] == 0
    (a, ga), (b, gb) = runs["1"], runs["0"]
    assert np.array_equal(a, b)
    if debug:
        assert np.array_equal(ga["mu"], gb["mu"]) and np.array_equal(ga["rstd"], gb["rstd"])
    ref, _ = oracle.forward(w.config(), q, k, v)
    assert slice_rel_err(a, ref) < TOL_BF16
