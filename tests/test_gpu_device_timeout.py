"""The device-side failure report, driven without faulting the GPU.

The distance kernel's barrier waits are bounded; lapl_attn_set_fault_injection shortens the
bound and makes the kernel's producer skip the copy of each CTA's last chunk, so the waits on
that chunk (and only those) run out.  Nothing is in flight when they do.  The forward must then
end, report LAPL_ERR_DEVICE_TIMEOUT with the distance kernel's bit through
lapl_attn_device_errors, and leave the context usable: a normal forward afterwards matches the
oracle.  The same holds for the tensor-core output and B V kernels (modes 2 and 3: their
copying thread or warp skips each CTA's last tile; reported as the output chain's bit).
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
    import oracle
    oracle.build()


@pytest.mark.parametrize("name", ["stage1_f32", "tiny_f32"])
def test_distance_wait_runs_out_then_recovers(name):
    import torch
    import oracle
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    dq, dk, dv = (to_device(x, w.dtype) for x in (q, k, v))
    h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": w.dtype}))
    try:
        assert lna.lapl_attn_plan_info_get(h)["cdist_tma"] == 2
        nbytes = lna.lapl_attn_workspace_size(h)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = torch.empty(dq.shape, dtype=torch.float32, device="cuda")
        st = torch.cuda.current_stream().cuda_stream
        args = (h, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, out.data_ptr(),
                ws.data_ptr(), nbytes, st)
        lna.lapl_attn_device_errors(h, st)                 # start from a clear word

        lna.lapl_attn_set_fault_injection(h, 50_000, 1)    # 50 us bound, last copies skipped
        lna.lapl_attn_forward(*args)
        flags = ctypes.c_uint(0)
        status = _lib.LIB.lapl_attn_device_errors(h, st, ctypes.byref(flags))
        assert status == _lib.LAPL_ERR_DEVICE_TIMEOUT
        assert flags.value == 1                            # the distance kernel's bit only
        assert "distance kernel" in _lib.lapl_attn_last_error(h)
        assert _lib.LIB.lapl_attn_device_errors(h, st, ctypes.byref(flags)) == _lib.LAPL_OK
        assert flags.value == 0                            # read-and-clear

        lna.lapl_attn_set_fault_injection(h, 0, 0)         # back to normal operation
        out.fill_(float("nan"))
        lna.lapl_attn_forward(*args)
        assert lna.lapl_attn_device_errors(h, st) == 0
        got = out.cpu().numpy().astype(np.float64)
        ref, _ = oracle.forward(w.config(), q, k, v)
        assert slice_rel_err(got, ref) < TOL_F32
    finally:
        lna.lapl_attn_destroy(h)


def test_fault_injection_rejects_bad_switch():
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    w = WORKLOADS["tiny_f32"]
    h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": "f32"}))
    try:
        assert _lib.LIB.lapl_attn_set_fault_injection(h, 0, 4) == _lib.LAPL_ERR_INVALID_ARG
        assert _lib.LIB.lapl_attn_set_fault_injection(h, 0, -1) == _lib.LAPL_ERR_INVALID_ARG
        assert _lib.LIB.lapl_attn_set_fault_injection(None, 0, 0) == _lib.LAPL_ERR_INVALID_ARG
        for mode in (0, 1, 2, 3):
            assert _lib.LIB.lapl_attn_set_fault_injection(h, 0, mode) == _lib.LAPL_OK
    finally:
        lna.lapl_attn_destroy(h)


@pytest.mark.parametrize("mode,kernel", [(2, "out_tensor_core"), (3, "bv_tensor_core")])
def test_chain_wait_runs_out_then_recovers(mode, kernel):
    """d = 64: both tensor-core chain kernels run by default; the chosen one never copies each
    CTA's last tile, its waits on that tile give up after 50 us, the forward ends and reports
    the output chain's bit alone, and the next normal forward matches the oracle."""
    import torch
    import oracle
    import laplacian_nystr_attention_gb300 as lna
    from laplacian_nystr_attention_gb300 import _lib
    w = WORKLOADS["tiny_f32"].replace(head_dim=64, heads=2)
    q, k, v = make_inputs(w)
    dq, dk, dv = (to_device(x, w.dtype) for x in (q, k, v))
    h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": w.dtype}))
    try:
        assert lna.lapl_attn_plan_info_get(h)[kernel] == 1
        nbytes = lna.lapl_attn_workspace_size(h)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = torch.empty(dq.shape, dtype=torch.float32, device="cuda")
        st = torch.cuda.current_stream().cuda_stream
        args = (h, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, out.data_ptr(),
                ws.data_ptr(), nbytes, st)
        lna.lapl_attn_device_errors(h, st)                 # start from a clear word

        lna.lapl_attn_set_fault_injection(h, 50_000, mode)
        lna.lapl_attn_forward(*args)
        flags = ctypes.c_uint(0)
        status = _lib.LIB.lapl_attn_device_errors(h, st, ctypes.byref(flags))
        assert status == _lib.LAPL_ERR_DEVICE_TIMEOUT
        assert flags.value == 4                            # the output chain's bit only
        assert "output chain" in _lib.lapl_attn_last_error(h)

        lna.lapl_attn_set_fault_injection(h, 0, 0)
        out.fill_(float("nan"))
        lna.lapl_attn_forward(*args)
        assert lna.lapl_attn_device_errors(h, st) == 0
        got = out.cpu().numpy().astype(np.float64)
        ref, _ = oracle.forward(w.config(), q, k, v)
        assert slice_rel_err(got, ref) < TOL_F32
    finally:
        lna.lapl_attn_destroy(h)
