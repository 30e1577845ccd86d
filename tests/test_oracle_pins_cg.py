"""Pins of the oracle's conjugate-gradient solver (solver = 1): M = T CG iterations on
W M = B V, column by column from zero, in place of M = X (B V) with the Newton-Schulz X.  The
pages compare the two solvers (German explainer page, 4; English page, 4 "Solver
Robustness") without describing the CG variant; the reading is the classical method.

What fixes the expected values, without retyping the oracle:
  * Krylov optimality: after t iterations, y_t minimises the W-norm of the error over the
    Krylov space span{b, W b, ..., W^(t-1) b}; the minimiser is computed here by a projected
    solve on an orthonormal Krylov basis (numpy QR + LAPACK solve), a different algorithm;
  * finite termination: t = m iterations solve W y = b (LAPACK solve);
  * the error's W-norm never increases from one iteration to the next;
  * closed forms: T = 0 gives M = 0 (so O = 0), T = 1 gives y = (b.b / b.Wb) b, and m = 1
    gives y = b / w after one iteration;
  * the reported residual is that of the returned M, ||B V - W M||_F / ||B V||_F;
  * a zero right-hand side stays zero (no 0/0), and the Newton-Schulz default is unchanged.
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs

TINY = WORKLOADS["tiny_f32"]


def cgcfg(w, **kw):
    c = w.config()
    c.update(solver=1)
    c.update(kw)
    return c


def krylov_minimiser(W, b, t):
    """argmin over y in K_t(W, b) of (y - W^-1 b)^T W (y - W^-1 b)."""
    if t == 0:
        return np.zeros_like(b)
    cols = [b]
    for _ in range(t - 1):
        cols.append(W @ cols[-1])
    Q, _ = np.linalg.qr(np.stack(cols, axis=1))
    c = np.linalg.solve(Q.T @ W @ Q, Q.T @ b)
    return Q @ c


@pytest.mark.parametrize("t", [1, 2, 3, 4, 6])
def test_krylov_optimality(oracle_mod, t):
    w = TINY.replace(ns_steps=t)            # m = 16, kappa(W) ~ 4
    q, k, v = make_inputs(w, seed=11)
    _, o = oracle_mod.forward(cgcfg(w), q, k, v, intermediates=True)
    W, BV, M = o["w"][0, 0], o["bv"][0, 0], o["m_mat"][0, 0]
    for j in range(0, w.head_dim, 5):
        ref = krylov_minimiser(W, BV[:, j], t)
        assert np.allclose(M[:, j], ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max()), (t, j)


def test_terminates_after_m_iterations(oracle_mod):
    w = TINY.replace(num_landmarks=4, ns_steps=4)
    q, k, v = make_inputs(w, seed=12)
    _, o = oracle_mod.forward(cgcfg(w), q, k, v, intermediates=True)
    W, BV, M = o["w"][0, 0], o["bv"][0, 0], o["m_mat"][0, 0]
    assert np.allclose(M, np.linalg.solve(W, BV), rtol=1e-10, atol=1e-13)
    assert o["ns_resid"][0, 0, -1] < 1e-12


def test_error_energy_norm_non_increasing(oracle_mod):
    w = TINY.replace(grid_h=14, grid_w=14, num_landmarks=49)
    q, k, v = make_inputs(w, seed=13)
    errs = []
    for t in range(0, 12):
        _, o = oracle_mod.forward(cgcfg(w, ns_steps=t), q, k, v, intermediates=True)
        W, BV, M = o["w"][0, 0], o["bv"][0, 0], o["m_mat"][0, 0]
        E = M - np.linalg.solve(W, BV)
        errs.append(np.einsum("ij,ik,kj->j", E, W, E))     # per column e^T W e
    errs = np.array(errs)
    assert (np.diff(errs, axis=0) <= 1e-12 * errs[0]).all()
    assert (errs[-1] < 0.5 * errs[0]).all()


def test_zero_and_one_iteration_closed_forms(oracle_mod):
    q, k, v = make_inputs(TINY, seed=14)
    out0, o0 = oracle_mod.forward(cgcfg(TINY, ns_steps=0), q, k, v, intermediates=True)
    assert not o0["m_mat"].any() and not out0.any()
    _, o1 = oracle_mod.forward(cgcfg(TINY, ns_steps=1), q, k, v, intermediates=True)
    W, BV = o1["w"][0, 0], o1["bv"][0, 0]
    step = (BV * BV).sum(0) / (BV * (W @ BV)).sum(0)
    assert np.allclose(o1["m_mat"][0, 0], BV * step, rtol=1e-12)


def test_single_landmark_exact(oracle_mod):
    w = TINY.replace(num_landmarks=1, ns_steps=3)
    q, k, v = make_inputs(w, seed=15)
    _, o = oracle_mod.forward(cgcfg(w), q, k, v, intermediates=True)
    assert np.allclose(o["m_mat"][0, 0], o["bv"][0, 0] / o["w"][0, 0, 0, 0], rtol=1e-14)


def test_reported_residual_is_that_of_m(oracle_mod):
    w = TINY.replace(grid_h=14, grid_w=14, num_landmarks=49, ns_steps=7)
    q, k, v = make_inputs(w, seed=16)
    _, o = oracle_mod.forward(cgcfg(w), q, k, v, intermediates=True)
    W, BV, M = o["w"][0, 0], o["bv"][0, 0], o["m_mat"][0, 0]
    true = np.linalg.norm(BV - W @ M) / np.linalg.norm(BV)
    assert o["ns_resid"][0, 0, 0] == 1.0
    assert abs(o["ns_resid"][0, 0, -1] - true) <= 1e-9 * true + 1e-14


def test_zero_right_hand_side(oracle_mod):
    q, k, v = make_inputs(TINY, seed=17)
    v = v.copy()
    v[..., 3] = 0.0                          # B V column 3 is exactly zero
    out, o = oracle_mod.forward(cgcfg(TINY), q, k, v, intermediates=True)
    assert np.isfinite(out).all() and np.isfinite(o["m_mat"]).all()
    assert not o["m_mat"][0, 0, :, 3].any()


def test_output_uses_the_solution(oracle_mod):
    """O = A_hat M with the CG M; X is not formed."""
    w = TINY.replace(heads=2)
    q, k, v = make_inputs(w, seed=18)
    out, o = oracle_mod.forward(cgcfg(w), q, k, v, intermediates=True)
    assert not o["x"].any()
    for h in range(2):
        assert np.allclose(out[0, h], o["a_hat"][0, h] @ o["m_mat"][0, h], rtol=1e-12,
                           atol=1e-14)


def test_matches_newton_schulz_when_both_converge(oracle_mod):
    w = TINY.replace(ns_steps=40)
    q, k, v = make_inputs(w, seed=19)
    ns, _ = oracle_mod.forward(w.config(), q, k, v)
    cg, _ = oracle_mod.forward(cgcfg(w), q, k, v)
    assert np.allclose(cg, ns, rtol=1e-9, atol=1e-12 * np.abs(ns).max())


def test_default_solver_unchanged_and_bad_solver_rejected(oracle_mod):
    q, k, v = make_inputs(TINY, seed=20)
    a, _ = oracle_mod.forward(TINY.config(), q, k, v)
    b, _ = oracle_mod.forward({**TINY.config(), "solver": 0}, q, k, v)
    assert np.array_equal(a, b)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.forward({**TINY.config(), "solver": 2}, q, k, v)
