"""The three variants of the fused distance + exp kernel against the oracle and each other.

  "tma"       token chunks brought into shared memory by the Tensor Memory Accelerator (a
              producer warp and mbarriers; fp32 with d = 32 or 64, bf16 with d = 64);
  "cp.async"  chunks copied by the whole CTA (every shape);
  "l1"        TMA-fed with a helper warp, and half of each warp's landmarks computed through
              |q - l| = q + l - 2 min(q, l) on the ALU pipe (fp32 with d = 32 or 64, bf16
              with d = 64; for s = 8 one CTA per SM with two row groups of warps).
LAPL_ATTN_CDIST_FEED at plan creation forces one.  "tma" and "cp.async" add |x_c - l_c| over
the channels in the same order, so their distances agree bit for bit; "l1" rounds differently
on float inputs (agreement to 1e-6 relative).  On small-integer inputs pooled over a
power-of-two window the landmarks are dyadic and every partial sum of every form is exact in
fp32, so all three equal the oracle exactly; other windows round the landmark and are compared
within 1e-5.  The partitions may differ (the kernels have different occupancy), so the
whitening statistics, and O, agree to rounding.  Every case ends with the device error word
clear (no bounded wait gave up).
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs
from parity_utils import TOL_BF16, TOL_F32, elem_rel, run_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

TINY = WORKLOADS["tiny_f32"]

# name -> (workload overrides, expect TMA when allowed)
CASES = {
    # ragged: N = 196 is not a multiple of the 128-token chunk; 4 heads
    "f32_d32_m49_ragged": (dict(batch=2, heads=2, grid_h=14, grid_w=14, num_landmarks=49), True),
    # d = 64 (two TMA boxes per row), 15 heads, N = 240
    "f32_d64_m16_15heads": (dict(batch=3, heads=5, grid_h=20, grid_w=12, head_dim=64,
                                  num_landmarks=16), True),
    "bf16_d64_m49": (dict(batch=2, heads=2, grid_h=28, grid_w=28, head_dim=64,
                          num_landmarks=49, dtype="bf16"), True),
    # one head: the switch from query to key tokens keeps the same landmarks
    "f32_d32_m1_one_head_129": (dict(grid_h=3, grid_w=43, num_landmarks=1), True),
    # exactly one chunk of rows in the whole tensor
    "f32_d32_m4_128_rows": (dict(grid_h=8, grid_w=16, num_landmarks=4), True),
    "f32_d32_m64": (dict(grid_h=16, grid_w=16, num_landmarks=64), True),
    "bf16_d64_m64": (dict(batch=2, grid_h=16, grid_w=16, head_dim=64, num_landmarks=64,
                          dtype="bf16"), True),
    "f32_d64_m36": (dict(batch=2, heads=3, grid_h=12, grid_w=24, head_dim=64,
                         num_landmarks=36), True),
    # fewer rows than one chunk: always cp.async
    "f32_d32_m4_below_chunk": (dict(grid_h=8, grid_w=8, num_landmarks=4), False),
    # head dims without a TMA instantiation
    "f32_d16_m16": (dict(head_dim=16), False),
    "bf16_d32_m16": (dict(dtype="bf16"), False),
}


FEEDS = ("tma", "cp.async", "l1")


def _expected_variant(w, feed) -> int:
    """plan_info cdist_tma for a forced feed: 2 (l1), 1 (tma) or 0 (cp.async); a feed that has
    no instantiation for the shape falls back to the automatic choice."""
    s = int(round(w.num_landmarks ** 0.5))
    rows_ok = w.batch * w.heads * w.n >= 128
    has_l1 = rows_ok and ((w.dtype == "f32" and w.head_dim in (32, 64)) or
                          (w.dtype == "bf16" and w.head_dim == 64))
    has_tma = rows_ok and ((w.dtype == "f32" and w.head_dim in (32, 64)) or
                           (w.dtype == "bf16" and w.head_dim == 64))
    if feed == "l1" and has_l1:
        return 2
    if feed == "tma" and has_tma:
        return 1
    if feed == "cp.async":
        return 0
    if has_l1:
        return 2
    return int(has_tma and w.dtype == "f32" and w.head_dim == 32 and s <= 7)


def _dyadic_window(w) -> bool:
    s = int(round(w.num_landmarks ** 0.5))
    win = (w.grid_h // s) * (w.grid_w // s)
    return win & (win - 1) == 0


def _oracle(w, q, k, v):
    import oracle
    return oracle.forward(w.config(), q, k, v, intermediates=True)


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
def test_all_feeds_match_oracle_and_each_other(case, monkeypatch):
    over, _ = CASES[case]
    w = TINY.replace(dist="integer", **over)
    q, k, v = make_inputs(w, seed=3)
    ref, o = _oracle(w, q, k, v)
    runs = {}
    for feed in FEEDS:
        monkeypatch.setenv("LAPL_ATTN_CDIST_FEED", feed)
        info = {}
        out, g = run_gpu(w, q, k, v, debug=True, info=info)
        assert info["device_errors"] == 0, feed
        assert info["cdist_tma"] == _expected_variant(w, feed), feed
        for name in ("d_ql", "d_lk", "d_ll", "landmarks"):
            if _dyadic_window(w):
                assert np.array_equal(g[name], o[name]), (feed, name)
            else:
                assert elem_rel(g[name], o[name]) < 1e-5, (feed, name)
        tol = TOL_BF16 if w.dtype == "bf16" else TOL_F32
        assert slice_rel_err(out, ref) < tol, feed
        runs[feed] = (out, g)
    if _dyadic_window(w):
        for feed in ("cp.async", "l1"):
            for name in ("d_ql", "d_lk", "a"):
                assert np.array_equal(runs["tma"][1][name], runs[feed][1][name]), (feed, name)
    for feed in ("cp.async", "l1"):
        assert slice_rel_err(runs["tma"][0], runs[feed][0]) < 1e-5, feed


SHAPES = {name: WORKLOADS[name] for name in ("stage1_f32", "stage23_bf16", "hires_bf16")}
SHAPES["stage23_as_f32"] = WORKLOADS["stage23_bf16"].replace(dtype="f32")   # d = 64, m = 49


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_workload_shape_feeds_agree(name, monkeypatch):
    """Full launch configuration of the workload, float inputs: the distances of the tma and
    cp.async feeds are identical bit for bit, those of the l1 kernel (where it exists) agree to
    1e-6 relative; O agrees to rounding."""
    w = SHAPES[name]
    q, k, v = make_inputs(w, seed=11)
    outs = {}
    for feed in FEEDS:
        monkeypatch.setenv("LAPL_ATTN_CDIST_FEED", feed)
        info = {}
        outs[feed] = run_gpu(w, q, k, v, debug=True, info=info)
        assert info["cdist_tma"] == _expected_variant(w, feed), feed
        assert info["device_errors"] == 0
    (o1, g1), (o2, g2), (o3, g3) = outs["tma"], outs["cp.async"], outs["l1"]
    if w.dtype == "bf16" or w.head_dim == 32:      # the plain TMA kernel exists
        assert np.array_equal(g1["d_ql"], g2["d_ql"])
        assert np.array_equal(g1["d_lk"], g2["d_lk"])
    for name in ("d_ql", "d_lk"):
        assert elem_rel(g3[name], g2[name]) < 1e-6, name
    # A = exp(-D / lambda): a relative change e of D moves A by about e * D / lambda relative
    # (D / lambda reaches 20 here), plus the exponential's few ulp.
    assert elem_rel(g3["a"], g2["a"], floor_frac=1e-3) < 5e-5
    assert slice_rel_err(o1, o2) < 1e-5
    assert slice_rel_err(o3, o2) < 1e-5


@pytest.mark.parametrize("over,expect", [
    (dict(grid_h=56, grid_w=56, num_landmarks=49), 2),                      # fp32, d = 32
    (dict(grid_h=56, grid_w=56, num_landmarks=64), 2),                      # s = 8: two groups
    (dict(grid_h=28, grid_w=28, head_dim=64, num_landmarks=49), 2),         # fp32, d = 64
    (dict(grid_h=28, grid_w=28, head_dim=64, num_landmarks=49, dtype="bf16"), 2),
])
def test_automatic_feed_choice(over, expect, monkeypatch):
    import laplacian_nystr_attention_gb300 as lna
    monkeypatch.delenv("LAPL_ATTN_CDIST_FEED", raising=False)
    w = TINY.replace(**over)
    h = lna.lapl_attn_create(lna.make_config(**{**w.config(), "in_dtype": w.dtype}))
    try:
        assert lna.lapl_attn_plan_info_get(h)["cdist_tma"] == expect
    finally:
        lna.lapl_attn_destroy(h)


@pytest.mark.parametrize("over", [
    dict(batch=2, heads=2, grid_h=14, grid_w=14, num_landmarks=49),              # s = 7, d = 32
    dict(batch=2, grid_h=16, grid_w=16, head_dim=64, num_landmarks=64),          # s = 8, d = 64
    dict(grid_h=24, grid_w=40, num_landmarks=64),                                # s = 8, ragged
    dict(batch=2, grid_h=16, grid_w=16, head_dim=64, num_landmarks=64, dtype="bf16"),
    dict(batch=3, grid_h=14, grid_w=21, head_dim=64, num_landmarks=49, dtype="bf16"),
])
def test_split_pipe_row_groups_agree(over, monkeypatch):
    """The split-pipe kernel with one row group per CTA (two CTAs per SM) and with two (one CTA
    of twice the warps per SM; the default for s = 8): every (token, landmark) distance is the
    same arithmetic in the same order, so A, B, D and O agree bit for bit; O meets the oracle."""
    w = TINY.replace(**over)
    s = int(round(w.num_landmarks ** 0.5))
    q, k, v = make_inputs(w, seed=7)
    runs = {}
    monkeypatch.setenv("LAPL_ATTN_CDIST_FEED", "l1")
    for g in (1, 2):
        monkeypatch.setenv("LAPL_ATTN_CDIST_GROUPS", str(g))
        info = {}
        runs[g] = run_gpu(w, q, k, v, debug=True, info=info)
        assert info["cdist_tma"] == 2 and info["device_errors"] == 0
        assert info["cdist_threads"] == 32 * (g * s + 1)
    for name in ("d_ql", "d_lk", "a"):
        assert np.array_equal(runs[1][1][name], runs[2][1][name]), name
    assert np.array_equal(runs[1][0], runs[2][0])
    ref, _ = _oracle(w, q, k, v)
    assert slice_rel_err(runs[2][0], ref) < (TOL_BF16 if w.dtype == "bf16" else TOL_F32)
