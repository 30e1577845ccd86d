"""Host-side checks of the parity harness itself (no GPU)."""
import numpy as np

import oracle
from lapl_workloads import WORKLOADS, make_bias, make_inputs
from parity_utils import oracle_each_slice, slice_rel_err, worst_slice


def test_each_slice_equals_the_full_oracle_call():
    """The per-slice oracle (one 1 x 1 problem per thread) gives, bit for bit, the slices of
    one full call: every step of the method is per (batch, head)."""
    w = WORKLOADS["tiny_f32"].replace(batch=2, heads=3, grid_h=8, grid_w=8, num_landmarks=4)
    q, k, v = make_inputs(w)
    bias = make_bias(w)
    full, _ = oracle.forward(w.config(), q, k, v, bias=bias)
    refs = oracle_each_slice(w.config(), q, k, v, bias=bias)
    assert sorted(refs) == list(range(6))
    for s, r in refs.items():
        b, h = divmod(s, 3)
        assert np.array_equal(r, full[b, h]), s
    assert worst_slice(full, refs) == (0.0, 5)


def test_worst_slice_finds_the_planted_error():
    w = WORKLOADS["tiny_f32"].replace(batch=2, heads=2, grid_h=8, grid_w=8, num_landmarks=4)
    q, k, v = make_inputs(w)
    full, _ = oracle.forward(w.config(), q, k, v)
    refs = oracle_each_slice(w.config(), q, k, v, slices=[1, 2])
    bad = full.copy()
    bad[1, 0, 3, 5] += 1e-2 * np.abs(full[1, 0]).max()
    err, s = worst_slice(bad, refs)
    assert s == 2 and abs(err - 1e-2) < 1e-9
    assert err == slice_rel_err(bad[1, 0][None, None], full[1, 0][None, None])
