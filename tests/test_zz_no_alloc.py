"""The workspace-free entry point, lapl_attn_forward_noalloc, against lapl_attn_forward.

lapl_attn_forward_noalloc exists for callers that cannot allocate device memory themselves (an
application that owns every allocation, a plugin that must not call cudaMalloc): it keeps the
workspace in a fixed 32 MiB array inside the library.  Both entry points run the same kernels
on the same plan, and the library is deterministic, so the outputs must agree bit for bit.
This file is named so that pytest collects it last; it must pass on its own in a fresh process
and after the other tests.
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs
from parity_utils import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()


def _forward_both(w, seeds, solver="newton_schulz", poison_seed=None):
    """For each seed: output of lapl_attn_forward and of lapl_attn_forward_noalloc (same handle,
    the no-allocation calls back to back).  With poison_seed, one no-allocation call on other
    inputs (and a bias) runs first, so the shared array starts out full of another problem's
    values."""
    import torch
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    cfg = lna.make_config(**{**w.config(), "in_dtype": w.dtype, "solver": solver})
    h = lna.lapl_attn_create(cfg)
    ws_bytes = lna.lapl_attn_workspace_size(h)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    if poison_seed is not None:
        q, k, v = (to_device(3.0 * x, "f32" if w.dtype == "f32" else "bf16")
                   for x in make_inputs(w, seed=poison_seed))
        bias = torch.full((w.heads, w.num_landmarks), 0.5, dtype=torch.float32, device="cuda")
        junk = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        assert _lib.LIB.lapl_attn_forward_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                  bias.data_ptr(), junk.data_ptr(),
                                                  st) == _lib.LAPL_OK
    inputs = [tuple(to_device(x, w.dtype) for x in make_inputs(w, seed=s)) for s in seeds]
    ref, got = [], []
    for q, k, v in inputs:
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        assert lna.lapl_attn_forward(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None,
                                     out.data_ptr(), ws.data_ptr(), ws_bytes, st) is None
        ref.append(out)
    for q, k, v in inputs:            # two no-allocation calls in a row
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        status = _lib.LIB.lapl_attn_forward_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                    None, out.data_ptr(), st)
        assert status == _lib.LAPL_OK, _lib.lapl_attn_last_error(h)
        got.append(out)
    torch.cuda.synchronize()
    lna.lapl_attn_destroy(h)
    return ([r.cpu().numpy() for r in ref], [g.cpu().numpy() for g in got])


CASES = {
    "stage1_f32": (WORKLOADS["stage1_f32"], "newton_schulz"),
    "tiny_bf16": (WORKLOADS["tiny_f32"].replace(dtype="bf16"), "newton_schulz"),
    "stage1_f32_cg": (WORKLOADS["stage1_f32"], "cg"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_forward_on_two_calls(case):
    w, solver = CASES[case]
    ref, got = _forward_both(w, seeds=[0, 7], solver=solver, poison_seed=11)
    assert not np.array_equal(ref[0], ref[1])     # the two calls really differ
    for r, g in zip(ref, got):
        assert np.isfinite(g).all()
        assert np.array_equal(g, r)


@pytest.mark.parametrize("name", ["stage23_bf16", "sweep_f32_65536"])
def test_noalloc_rejects_workspace_beyond_capacity(name):
    """Stage 2/3 (A^T and B^T alone are 2 x 19.7 MB) and the long sequences do not fit."""
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    w = WORKLOADS[name]
    h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": w.dtype}))
    assert lna.lapl_attn_workspace_size(h) > 32 << 20
    status = _lib.LIB.lapl_attn_forward_noalloc(h, None, None, None, None, None, None)
    assert status == _lib.LAPL_ERR_WORKSPACE
    assert "static scratch" in _lib.lapl_attn_last_error(h)
    lna.lapl_attn_destroy(h)
