"""The TF32 high/low split of the tensor-core Newton-Schulz kernel, restated on the host.

The kernel rounds an fp32 value to TF32 by adding 2^12 to its bit pattern and clearing the low
13 bits (round to nearest, ties away from zero, in sign-magnitude).  These checks pin that
rule against its definition: the result has at most 11 significant bits, it is the nearest
such value, ties go away from zero, and hi + lo with lo = x - hi reproduces x exactly.
"""
import numpy as np


def tf32_rna(x: np.ndarray) -> np.ndarray:
    b = x.astype(np.float32).view(np.uint32)
    return ((b + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def test_nearest_and_ties_away():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    hi = tf32_rna(x)
    assert np.all(hi.view(np.uint32) & np.uint32(0x1FFF) == 0)
    # nearest: the two TF32 neighbours of x bracket it and hi is the closer one
    down = (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    up = (down.view(np.uint32) + np.uint32(0x2000)).view(np.float32)
    dd = np.abs(x.astype(np.float64) - down)
    du = np.abs(up.astype(np.float64) - x)
    want = np.where(du < dd, up, np.where(dd < du, down, up))     # tie -> away from zero
    assert np.array_equal(hi, want)


def test_exact_split():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(100000).astype(np.float32)
    hi = tf32_rna(x)
    lo = (x - hi).astype(np.float32)
    assert np.array_equal((hi.astype(np.float64) + lo.astype(np.float64)).astype(np.float32), x)
    # |lo| <= half a TF32 ulp of hi, so lo itself needs at most 13 significant bits
    assert np.all(np.abs(lo) <= np.abs(hi) * 2.0 ** -11 + 1e-45)


def test_binade_carry_and_zero():
    x = np.array([0.0, -0.0, 1.9999999, -1.9999999, 2.0 ** -126], dtype=np.float32)
    hi = tf32_rna(x)
    assert hi[0] == 0.0 and hi[1] == 0.0
    assert hi[2] == 2.0 and hi[3] == -2.0
    assert hi[4] == np.float32(2.0 ** -126)
