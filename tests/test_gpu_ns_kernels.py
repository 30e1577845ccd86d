"""The three Newton-Schulz kernels against the oracle and against each other.

  ffma  one CTA per head, products on the CUDA cores (the default);
  pair  a cluster of two CTAs per head that split every product and exchange halves through
        distributed shared memory (m > 32);
  tc    one CTA per head, products on the tensor cores (tcgen05, TF32 operands split into an
        exact high/low pair, fp32 accumulation in tensor memory).

ffma and pair accumulate every element over the same k quarters in the same order, so their X
agree bit for bit.  tc sums the same products in another order and at slightly lower
precision per product (about 2^-22 relative), so its X agrees to rounding; all three match the
oracle's X within 1e-4 (relative to max |X|) and O within the parity tolerances.  The kernel is
chosen with LAPL_ATTN_NS_KERNEL at plan creation.
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs
from parity_utils import TOL_BF16, TOL_F32, rel_to_max, run_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny_f32"]

CASES = {
    "m36_d32": dict(grid_h=12, grid_w=12, num_landmarks=36),
    "m49_d32_3heads": dict(heads=3, grid_h=14, grid_w=14, num_landmarks=49),
    "m64_d64": dict(batch=2, grid_h=16, grid_w=16, head_dim=64, num_landmarks=64),
    "m49_d128": dict(grid_h=14, grid_w=14, head_dim=128, num_landmarks=49),
    "m49_T0": dict(grid_h=14, grid_w=14, num_landmarks=49, ns_steps=0),
    "m49_T1": dict(grid_h=14, grid_w=14, num_landmarks=49, ns_steps=1),
    "m64_bf16_T24": dict(grid_h=16, grid_w=16, head_dim=64, num_landmarks=64, ns_steps=24,
                         dtype="bf16"),
}
# Shapes with m <= 32 (one warp tile): ffma and tc only.
SMALL = {
    "m1": dict(num_landmarks=1),
    "m4": dict(num_landmarks=4),
    "m9_d24": dict(grid_h=12, grid_w=12, num_landmarks=9, head_dim=24),
    "m16": dict(num_landmarks=16),
    "m25": dict(grid_h=20, grid_w=20, num_landmarks=25),
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


def _run_kernels(case_over, kernels, monkeypatch):
    import oracle
    w = TINY.replace(dist="student_t", **case_over)
    q, k, v = make_inputs(w, seed=5)
    ref, o = oracle.forward(w.config(), q, k, v, intermediates=True)
    res = {}
    for kern in kernels:
        monkeypatch.setenv("LAPL_ATTN_NS_KERNEL", kern)
        info = {}
        out, g = run_gpu(w, q, k, v, debug=True, info=info)
        assert info["device_errors"] == 0, kern
        assert info["ns_cluster"] == (2 if kern == "pair" else 1), kern
        assert info["ns_tensor_core"] == int(kern == "tc"), kern
        assert rel_to_max(g["x"], o["x"]) < 1e-4, kern
        assert rel_to_max(g["w"], o["w"]) < 1e-6, kern
        tol = TOL_BF16 if w.dtype == "bf16" else TOL_F32
        assert slice_rel_err(out, ref) < tol, kern
        res[kern] = (out, g)
    return res


@pytest.mark.parametrize("case", sorted(CASES))
def test_three_kernels(case, monkeypatch):
    res = _run_kernels(CASES[case], ("ffma", "pair", "tc"), monkeypatch)
    gf, gp, gt = res["ffma"][1], res["pair"][1], res["tc"][1]
    for name in ("x", "w", "d_ll"):
        assert np.array_equal(gf[name], gp[name]), name
    assert np.array_equal(gf["w"], gt["w"])
    assert rel_to_max(gt["x"], gf["x"]) < 1e-4
    # X from every kernel is exactly symmetric
    for g in (gf, gp, gt):
        x = g["x"][0, 0]
        assert np.array_equal(x, x.T)


@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_m(case, monkeypatch):
    res = _run_kernels(SMALL[case], ("ffma", "tc"), monkeypatch)
    assert rel_to_max(res["tc"][1]["x"], res["ffma"][1]["x"]) < 1e-4


def test_pair_request_ignored_for_small_m(monkeypatch):
    monkeypatch.setenv("LAPL_ATTN_NS_KERNEL", "pair")
    w = TINY.replace(num_landmarks=16)
    q, k, v = make_inputs(w)
    info = {}
    run_gpu(w, q, k, v, info=info)
    assert info["ns_cluster"] == 1 and info["ns_tensor_core"] == 0
