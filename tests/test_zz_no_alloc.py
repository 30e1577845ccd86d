"""The workspace-free entry point, lapl_attn_forward_noalloc, against lapl_attn_forward.

lapl_attn_forward_noalloc exists for callers that cannot allocate device memory themselves (an
application that owns every allocation, a plugin that must not call cudaMalloc): it keeps the
workspace in a fixed 32 MiB array inside the library.  This file is named so that pytest
collects it last; it must pass on its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs
from parity_utils import TOL_F32, slice_rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()


def _forward_both(w, seeds):
    """For each seed: output of lapl_attn_forward and of lapl_attn_forward_noalloc (same handle,
    the no-allocation calls back to back)."""
    import torch
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    cfg = lna.make_config(**{**w.config(), "in_dtype": w.dtype})
    h = lna.lapl_attn_create(cfg)
    ws_bytes = lna.lapl_attn_workspace_size(h)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    inputs = [tuple(to_device(x, w.dtype) for x in make_inputs(w, seed=s)) for s in seeds]
    ref, got = [], []
    for q, k, v in inputs:
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        lna.lapl_attn_forward(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None,
                              out.data_ptr(), ws.data_ptr(), ws_bytes, st)
        ref.append(out)
    for q, k, v in inputs:            # two no-allocation calls in a row
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        status = _lib.LIB.lapl_attn_forward_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                    None, out.data_ptr(), st)
        assert status == _lib.LAPL_OK, _lib.lapl_attn_last_error(h)
        got.append(out)
    torch.cuda.synchronize()
    lna.lapl_attn_destroy(h)
    return ([r.cpu().numpy().astype(np.float64) for r in ref],
            [g.cpu().numpy().astype(np.float64) for g in got])


def test_noalloc_matches_forward_on_two_calls():
    w = WORKLOADS["stage1_f32"]
    ref, got = _forward_both(w, seeds=[0, 7])
    assert not np.array_equal(ref[0], ref[1])     # the two calls really differ
    for r, g in zip(ref, got):
        assert np.isfinite(g).all()
        assert slice_rel_err(g, r) < TOL_F32


def test_noalloc_rejects_workspace_beyond_capacity():
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    w = WORKLOADS["sweep_f32_65536"]            # A^T alone is 128 MiB
    h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": "f32"}))
    assert lna.lapl_attn_workspace_size(h) > 32 << 20
    status = _lib.LIB.lapl_attn_forward_noalloc(h, None, None, None, None, None, None)
    assert status == _lib.LAPL_ERR_WORKSPACE
    assert "static scratch" in _lib.lapl_attn_last_error(h)
    lna.lapl_attn_destroy(h)
