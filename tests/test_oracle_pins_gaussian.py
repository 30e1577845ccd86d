"""Pins of the oracle's Gaussian-kernel variant (kernel = 1), the kernel the pages compare the
Laplacian one against: k(x,y) = exp(-||x-y||_2^2 / lambda), similarity decaying with the
squared l2 distance (English explainer page, 1 "Theoretical Mismatch").

What fixes the expected values, without retyping the oracle:
  * rotation invariance: an orthogonal change of basis of the channels, applied to Q and K,
    leaves every squared l2 distance unchanged (pooling is linear, so it commutes) -- an l1
    distance would change;
  * degree-2 homogeneity: scaling Q and K by 2 multiplies every distance by exactly 4 (by 2
    for l1);
  * Gaussian Gram matrices of distinct points are positive definite, with unit diagonal;
  * with one landmark per token (m = N), no whitening and eps = 0 the pipeline is exact
    Gaussian kernel attention, checked against brute force;
  * the Laplacian variant is unchanged by the new field (kernel = 0 is the default).
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs

TINY = WORKLOADS["tiny_f32"]


def run(oracle_mod, cfg, q, k, v, inter=True):
    return oracle_mod.forward(cfg, q, k, v, intermediates=inter)


def gcfg(w, **kw):
    c = w.config()
    c.update(kernel=1)
    c.update(kw)
    return c


def test_rotation_invariance(oracle_mod):
    w = TINY.replace(heads=2)
    q, k, v = make_inputs(w, seed=4)
    rng = np.random.default_rng(9)
    rot, _ = np.linalg.qr(rng.standard_normal((w.head_dim, w.head_dim)))
    _, o1 = run(oracle_mod, gcfg(w), q, k, v)
    _, o2 = run(oracle_mod, gcfg(w), q @ rot, k @ rot, v)
    for name in ("d_ql", "d_lk", "d_ll"):
        assert np.allclose(o1[name], o2[name], rtol=1e-11, atol=1e-11), name
    # the Laplacian distances do change under the same rotation
    _, l1 = run(oracle_mod, w.config(), q, k, v)
    _, l2 = run(oracle_mod, w.config(), q @ rot, k @ rot, v)
    assert not np.allclose(l1["d_ql"], l2["d_ql"], rtol=1e-3)


def test_degree_two_homogeneity(oracle_mod):
    q, k, v = make_inputs(TINY, seed=5)
    _, o1 = run(oracle_mod, gcfg(TINY), q, k, v)
    _, o2 = run(oracle_mod, gcfg(TINY), 2.0 * q, 2.0 * k, v)
    for name in ("d_ql", "d_lk", "d_ll"):
        assert np.array_equal(4.0 * o1[name], o2[name]), name
    _, l1 = run(oracle_mod, TINY.config(), q, k, v)
    _, l2 = run(oracle_mod, TINY.config(), 2.0 * q, 2.0 * k, v)
    assert np.array_equal(2.0 * l1["d_ql"], l2["d_ql"])


def test_gram_positive_definite_unit_diagonal(oracle_mod):
    w = TINY.replace(num_landmarks=16)
    q, k, v = make_inputs(w, seed=6)
    cfg = gcfg(w, eps=0.0)
    _, o = run(oracle_mod, cfg, q, k, v)
    W = o["w"][0, 0]
    assert np.array_equal(np.diag(W), np.ones(16))
    assert np.allclose(W, W.T, rtol=0, atol=0)
    np.linalg.cholesky(W)                          # raises unless positive definite
    assert np.linalg.eigvalsh(W).min() > 0


def test_distance_small_integers_exact(oracle_mod):
    w = TINY.replace(dist="integer")
    q, k, v = make_inputs(w)
    _, o = run(oracle_mod, gcfg(w), q, k, v)
    L = o["landmarks"][0, 0]
    Q = q[0, 0].astype(np.float64)
    brute = ((Q[:, None, :] - L[None, :, :]) ** 2).sum(-1)      # dyadic: exact in fp64
    assert np.array_equal(o["d_ql"][0, 0], brute)


@pytest.mark.parametrize("grid", [(4, 4), (3, 3)])
def test_m_equals_n_is_exact_gaussian_attention(oracle_mod, grid):
    gh, gw = grid
    n = gh * gw
    w = TINY.replace(grid_h=gh, grid_w=gw, num_landmarks=n, head_dim=8, ns_steps=40)
    q, k, v = make_inputs(w, seed=7)
    cfg = gcfg(w, eps=0.0, whiten=0, lam=8.0)
    out, _ = run(oracle_mod, cfg, q, k, v, inter=False)
    Q, K, V = (x[0, 0].astype(np.float64) for x in (q, k, v))
    kernel = np.exp(-((Q[:, None, :] - K[None, :, :]) ** 2).sum(-1) / 8.0)
    assert np.allclose(out[0, 0], kernel @ V, rtol=1e-8, atol=1e-10)


def test_laplacian_default_unchanged(oracle_mod):
    q, k, v = make_inputs(TINY, seed=8)
    a, _ = run(oracle_mod, TINY.config(), q, k, v, inter=False)
    b, _ = run(oracle_mod, {**TINY.config(), "kernel": 0}, q, k, v, inter=False)
    assert np.array_equal(a, b)


def test_rejects_unknown_kernel(oracle_mod):
    q, k, v = make_inputs(TINY)
    with pytest.raises(oracle_mod.OracleError):
        run(oracle_mod, gcfg(TINY, kernel=2), q, k, v)
