"""Pins of the oracle's backward pass (oracle.backward): the gradients of a loss with
dLoss/dO = G through the whole forward, derived by hand step by step in the C source.

What fixes the expected values, without retyping the derivation:
  * central finite differences of the oracle's forward (itself pinned elsewhere) on random
    entries of Q, K, V and the bias, for both kernels, whitening on and off, converged and
    unconverged Newton-Schulz iterates, T = 0, one landmark, and non-dyadic windows;
  * exact identities of the method:
      - translation invariance: shifting Q and K by one vector leaves every distance, hence O,
        unchanged, so sum_i dQ_i + sum_n dK_n = 0 channel by channel (both kernels);
      - rotation invariance of the Gaussian kernel: Q^T dQ + K^T dK is symmetric;
      - O is linear in V, so <dV, V> = <G, O> (Euler's identity);
      - the loss is linear in G, so the gradients are too;
  * the tie bound: zero for the Gaussian kernel, non-zero on integer inputs, where sign
    decisions sit exactly at 0 (finite differences skip the entries it marks).
"""
import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs

BASE = WORKLOADS["tiny_f32"].replace(grid_h=8, grid_w=8, num_landmarks=4, head_dim=4,
                                     ns_steps=6, lam=2.0)

CASES = {
    "laplacian": dict(),
    "laplacian_no_whiten": dict(whiten=0),
    "gaussian": dict(kernel=1),
    "gaussian_no_whiten": dict(kernel=1, whiten=0),
    "unconverged_T2": dict(ns_steps=2),
    "T0": dict(ns_steps=0),
    "one_landmark": dict(num_landmarks=1),
    "m9_windows_4x4": dict(grid_h=12, grid_w=12, num_landmarks=9),
    "m16_d8_two_heads": dict(num_landmarks=16, head_dim=8, heads=2),
    "large_eps": dict(eps=0.5),
}


def cfg_of(case):
    over = dict(CASES[case])
    kern = over.pop("kernel", 0)
    w = BASE.replace(**over)
    c = w.config()
    c["kernel"] = kern
    return w, c


def loss(oracle_mod, cfg, q, k, v, bias, G):
    out, _ = oracle_mod.forward(cfg, q, k, v, bias=bias)
    return float((out * G).sum())


@pytest.mark.parametrize("case", sorted(CASES))
def test_finite_differences(oracle_mod, case):
    w, cfg = cfg_of(case)
    q, k, v = (x.astype(np.float64) for x in make_inputs(w, seed=3))
    rng = np.random.default_rng(7)
    G = rng.standard_normal(q.shape)
    bias = 0.1 * rng.standard_normal((w.heads, w.num_landmarks))
    dq, dk, dv, db, aq, ak = oracle_mod.backward(cfg, q, k, v, G, bias=bias)
    h = 1e-6
    grads = {"q": dq, "k": dk, "v": dv}
    ties = {"q": aq, "k": ak, "v": np.zeros_like(aq)}
    for name in ("q", "k", "v"):
        arrs = {"q": q, "k": k, "v": v}
        for _ in range(10):
            idx = tuple(int(rng.integers(0, s)) for s in q.shape)
            while ties[name][idx] > 0:               # entries next to a kink: no derivative
                idx = tuple(int(rng.integers(0, s)) for s in q.shape)
            plus = {n: a.copy() for n, a in arrs.items()}
            minus = {n: a.copy() for n, a in arrs.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            fd = (loss(oracle_mod, cfg, plus["q"], plus["k"], plus["v"], bias, G) -
                  loss(oracle_mod, cfg, minus["q"], minus["k"], minus["v"], bias, G)) / (2 * h)
            scale = np.abs(grads[name]).max()
            assert abs(fd - grads[name][idx]) <= 1e-7 * scale + 1e-12, (name, idx)
    for j in range(w.num_landmarks):
        b1, b2 = bias.copy(), bias.copy()
        b1[0, j] += h
        b2[0, j] -= h
        fd = (loss(oracle_mod, cfg, q, k, v, b1, G) - loss(oracle_mod, cfg, q, k, v, b2, G)) / (2 * h)
        assert abs(fd - db[0, j]) <= 1e-7 * max(np.abs(db).max(), 1e-30) + 1e-12
    if not cfg["whiten"]:
        assert not db.any()


@pytest.mark.parametrize("kernel", [0, 1])
def test_translation_invariance(oracle_mod, kernel):
    w = BASE.replace(heads=2, num_landmarks=16, head_dim=8)
    q, k, v = make_inputs(w, seed=4)
    G = np.random.default_rng(8).standard_normal(q.shape)
    dq, dk, _, _, _, _ = oracle_mod.backward({**w.config(), "kernel": kernel}, q, k, v, G)
    total = dq.sum(axis=2) + dk.sum(axis=2)              # [B, H, d]
    assert np.abs(total).max() <= 1e-10 * np.abs(dq).max()


def test_gaussian_rotation_invariance(oracle_mod):
    w = BASE.replace(num_landmarks=16, head_dim=8)
    q, k, v = (x.astype(np.float64) for x in make_inputs(w, seed=5))
    G = np.random.default_rng(9).standard_normal(q.shape)
    dq, dk, _, _, _, _ = oracle_mod.backward({**w.config(), "kernel": 1}, q, k, v, G)
    S = q[0, 0].T @ dq[0, 0] + k[0, 0].T @ dk[0, 0]
    assert np.abs(S - S.T).max() <= 1e-10 * np.abs(S).max()
    # the Laplacian kernel has no such symmetry
    dq1, dk1, _, _, _, _ = oracle_mod.backward(w.config(), q, k, v, G)
    S1 = q[0, 0].T @ dq1[0, 0] + k[0, 0].T @ dk1[0, 0]
    assert np.abs(S1 - S1.T).max() > 1e-3 * np.abs(S1).max()


@pytest.mark.parametrize("kernel", [0, 1])
def test_value_euler_identity_and_linearity(oracle_mod, kernel):
    w = BASE.replace(heads=2)
    cfg = {**w.config(), "kernel": kernel}
    q, k, v = (x.astype(np.float64) for x in make_inputs(w, seed=6))
    rng = np.random.default_rng(10)
    G1, G2 = rng.standard_normal(q.shape), rng.standard_normal(q.shape)
    bias = 0.1 * rng.standard_normal((w.heads, w.num_landmarks))
    out, _ = oracle_mod.forward(cfg, q, k, v, bias=bias)
    g1 = oracle_mod.backward(cfg, q, k, v, G1, bias=bias)
    g2 = oracle_mod.backward(cfg, q, k, v, G2, bias=bias)
    g12 = oracle_mod.backward(cfg, q, k, v, 2.0 * G1 - G2, bias=bias)
    for a, b, c in zip(g1[:4], g2[:4], g12[:4]):
        assert np.allclose(c, 2.0 * a - b, rtol=1e-10, atol=1e-12 * np.abs(a).max())
    for s in range(w.heads):
        assert np.isclose((g1[2][0, s] * v[0, s]).sum(), (G1[0, s] * out[0, s]).sum(),
                          rtol=1e-10)


def test_tie_bound(oracle_mod):
    w = BASE.replace(dist="integer", num_landmarks=16, head_dim=8)
    q, k, v = make_inputs(w)
    G = np.random.default_rng(11).standard_normal(q.shape)
    _, _, _, _, aq, ak = oracle_mod.backward(w.config(), q, k, v, G)
    assert aq.any() and ak.any()                 # integer Q, K: sign decisions at exactly 0
    _, _, _, _, gq, gk = oracle_mod.backward({**w.config(), "kernel": 1}, q, k, v, G)
    assert not gq.any() and not gk.any()


def test_conjugate_gradient_backward_rejected(oracle_mod):
    q, k, v = make_inputs(BASE)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.backward({**BASE.config(), "solver": 1}, q, k, v, np.zeros(q.shape))
