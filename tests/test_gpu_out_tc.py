"""O = A^ M on the tensor cores (out_tc.cu) against the oracle and the CUDA-core kernel.

The kernel is the default wherever its shapes allow (d a multiple of 16 and at most 64, N a
multiple of 4) for d = 64, and for smaller d from N = 4096; LAPL_ATTN_OUT=tc / =cuda force
either.  It whitens A on the way into the
operand and splits operands into TF32 high/low pairs (three cross products, about 2^-21
relative), so O agrees with the CUDA-core kernel to rounding and with the oracle within the
usual bars.
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_bias, make_inputs
from parity_utils import TOL_BF16, TOL_F32, run_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny_f32"]

CASES = {
    "tiny_f32": dict(),
    "tiny_bf16_in": dict(dtype="bf16"),
    "ragged_14x14_m49": dict(grid_h=14, grid_w=14, num_landmarks=49),
    "m1": dict(num_landmarks=1),
    "m4": dict(num_landmarks=4),
    "m64": dict(num_landmarks=64),
    "d16": dict(head_dim=16),
    "d64_2x3": dict(batch=2, heads=3, head_dim=64),
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
def test_out_tensor_core_matches_oracle_and_cuda_cores(case, monkeypatch):
    import oracle
    w = TINY.replace(**CASES[case])
    q, k, v = make_inputs(w, seed=4)
    outs = {}
    for mode in ("tc", "cuda"):
        monkeypatch.setenv("LAPL_ATTN_OUT", mode)
        info = {}
        outs[mode], _ = run_gpu(w, q, k, v, info=info)
        assert info["out_tensor_core"] == (1 if mode == "tc" else 0)
        assert info["device_errors"] == 0
    ref, _ = oracle.forward(w.config(), q, k, v)
    tol = TOL_BF16 if w.dtype == "bf16" else TOL_F32
    assert slice_rel_err(outs["tc"], ref) < tol
    assert slice_rel_err(outs["tc"], outs["cuda"]) < 1e-5


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_out_tensor_core_bias_and_output_dtype(out_dtype, monkeypatch):
    import oracle
    monkeypatch.setenv("LAPL_ATTN_OUT", "tc")
    w = TINY.replace(batch=2, heads=2)
    q, k, v = make_inputs(w, seed=6)
    bias = make_bias(w)
    info = {}
    out, _ = run_gpu(w, q, k, v, bias=bias, out_dtype=out_dtype, info=info)
    assert info["out_tensor_core"] == 1
    ref, _ = oracle.forward(w.config(), q, k, v, bias=bias)
    assert slice_rel_err(out, ref) < (TOL_BF16 if out_dtype == "bf16" else TOL_F32)


def test_out_choice(monkeypatch):
    import laplacian_nystr_attention_gb300 as lna

    def choice(w):
        h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": w.dtype}))
        try:
            return lna.lapl_attn_plan_info_get(h)["out_tensor_core"]
        finally:
            lna.lapl_attn_destroy(h)

    monkeypatch.delenv("LAPL_ATTN_OUT", raising=False)
    assert choice(WORKLOADS["stage1_f32"]) == 0                               # d 32, N < 4096
    assert choice(WORKLOADS["stage23_bf16"]) == 1                             # d = 64
    assert choice(WORKLOADS["hires_bf16"]) == 1
    assert choice(WORKLOADS["sweep_f32_4096"]) == 1
    monkeypatch.setenv("LAPL_ATTN_OUT", "tc")
    assert choice(TINY) == 1
    assert choice(TINY.replace(head_dim=128)) == 0                            # 4d > 256
    assert choice(TINY.replace(grid_h=3, grid_w=43, num_landmarks=1)) == 0    # N = 129
    assert choice(TINY.replace(head_dim=24)) == 0
    monkeypatch.setenv("LAPL_ATTN_OUT", "cuda")
    assert choice(WORKLOADS["stage1_f32"]) == 0
