"""Pins of the fp64 CPU oracle to facts that do not come from the oracle itself.

Each test states what fixes the expected value: a closed form, an algebraic identity of the
method, a textbook routine (Gauss-Jordan elimination), a library routine (LAPACK through
numpy), or brute force on tiny inputs.  Together they are chosen so that a plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a wrong window)
fails at least one of them.

Method source: "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel",
explainer pages (English 2.A-2.C, Korean 2.2-2.3, Chinese 2.2).
"""
import math

import numpy as np
import pytest

from lapl_workloads import WORKLOADS, make_inputs, make_bias


def cfg_of(w, **kw):
    c = w.config()
    c.update(kw)
    return c


def run(oracle_mod, cfg, q, k, v, bias=None, inter=True):
    return oracle_mod.forward(cfg, q, k, v, bias=bias, intermediates=inter)


def gauss_jordan_inverse(a):
    """Textbook Gauss-Jordan elimination with partial pivoting (independent of the oracle)."""
    n = a.shape[0]
    aug = np.concatenate([a.astype(np.float64), np.eye(n)], axis=1)
    for col in range(n):
        piv = col + int(np.argmax(np.abs(aug[col:, col])))
        aug[[col, piv]] = aug[[piv, col]]
        aug[col] /= aug[col, col]
        for r in range(n):
            if r != col:
                aug[r] -= aug[r, col] * aug[col]
    return aug[:, n:]


def brute_pool(K, gh, gw, s):
    """Average pooling by reshape: [N,d] -> [s*s,d], windows row-major."""
    d = K.shape[-1]
    ph, pw = gh // s, gw // s
    g = K.reshape(s, ph, s, pw, d)
    return g.mean(axis=(1, 3)).reshape(s * s, d)


def brute_cdist_l1(X, Y):
    return np.abs(X[:, None, :] - Y[None, :, :]).sum(-1)


TINY = WORKLOADS["tiny_f32"]


# ---- P1: k(x, x) = 1 --------------------------------------------------------------------
def test_kernel_diagonal_is_one(oracle_mod):
    q, k, v = make_inputs(TINY)
    cfg = cfg_of(TINY)
    _, it = run(oracle_mod, cfg, q, k, v)
    dll = it["d_ll"][0, 0]
    w = it["w"][0, 0]
    assert np.all(np.diag(dll) == 0.0)
    assert np.all(np.diag(w) == 1.0 + cfg["eps"])   # exp(0) = 1 exactly, then + eps
    # off-diagonal W entries are exp(-D/lam) in (0, 1)
    off = w[~np.eye(w.shape[0], dtype=bool)]
    assert np.all(off > 0.0) and np.all(off < 1.0)


# ---- P2: W symmetric and positive definite (Laplacian kernel is PD) --------------------
@pytest.mark.parametrize("name", ["tiny_f32", "stage1_f32"])
def test_w_symmetric_positive_definite(oracle_mod, name):
    w0 = WORKLOADS[name]
    w0 = w0.replace(batch=1, heads=1)
    q, k, v = make_inputs(w0)
    _, it = run(oracle_mod, cfg_of(w0), q, k, v)
    W = it["w"][0, 0]
    assert np.array_equal(W, W.T)
    ev = np.linalg.eigvalsh(W)                 # LAPACK, independent of the oracle
    assert ev.min() > 0.0
    np.linalg.cholesky(W)                      # raises if not PD
    # eps shifts the spectrum: eig(W) - eps are the eigenvalues of the pure kernel matrix, > 0
    assert (ev - cfg_of(w0)["eps"]).min() > 0.0


# ---- P3: Newton-Schulz agrees with Gauss-Jordan on tiny m -------------------------------
@pytest.mark.parametrize("m,grid", [(1, 4), (4, 8), (9, 12), (16, 16)])
def test_ns_matches_gauss_jordan(oracle_mod, m, grid):
    w0 = TINY.replace(grid_h=grid, grid_w=grid, num_landmarks=m, ns_steps=20)
    q, k, v = make_inputs(w0)
    _, it = run(oracle_mod, cfg_of(w0), q, k, v)
    W, X = it["w"][0, 0], it["x"][0, 0]
    gj = gauss_jordan_inverse(W)
    assert np.max(np.abs(X - gj)) <= 1e-10 * np.max(np.abs(gj))
    assert np.allclose(gj, np.linalg.inv(W), rtol=1e-12, atol=1e-14)


# ---- P4: algebra of the iteration: R_{t+1} = R_t^2, X_t symmetric, X_t W = W X_t -------
def test_ns_residual_squares(oracle_mod):
    w0 = WORKLOADS["stage1_f32"].replace(batch=1, heads=1)   # kappa(W) ~ 65: slow start
    q, k, v = make_inputs(w0)
    Xs, W = [], None
    for t in range(0, 6):
        _, it = run(oracle_mod, cfg_of(w0, ns_steps=t), q, k, v)
        Xs.append(it["x"][0, 0])
        W = it["w"][0, 0]
        resid = it["ns_resid"][0, 0]
        assert resid.shape == (t + 1,)
    m = W.shape[0]
    I = np.eye(m)
    for t in range(5):
        R0 = I - W @ Xs[t]
        R1 = I - W @ Xs[t + 1]
        assert np.max(np.abs(R1 - R0 @ R0)) < 1e-12
        assert np.max(np.abs(Xs[t] - Xs[t].T)) < 1e-12
        assert np.max(np.abs(Xs[t] @ W - W @ Xs[t])) < 1e-12
    # reported residual norms are those of the returned iterates
    _, it = run(oracle_mod, cfg_of(w0, ns_steps=5), q, k, v)
    assert abs(it["ns_resid"][0, 0, 5] - np.linalg.norm(I - W @ Xs[5])) < 1e-12
    # not yet converged after 5 steps at this conditioning: the step count matters
    assert it["ns_resid"][0, 0, 5] > 0.5


def test_ns_step_zero_and_constant_keys_closed_form(oracle_mod):
    """Constant K: every landmark equals the same vector, so W = J + eps*I (J all ones).
    |W|_1 = |W|_inf = m + eps, hence X0 = (J + eps I)/(m + eps)^2, and by Sherman-Morrison
    W^-1 = (I - J/(m + eps)) / eps."""
    m, eps = 16, 1.0
    w0 = TINY.replace(eps=eps)
    q, k, v = make_inputs(w0)
    k = np.broadcast_to(k[:, :, :1, :], k.shape).copy()     # all keys equal
    J = np.ones((m, m))
    I = np.eye(m)
    _, it = run(oracle_mod, cfg_of(w0, ns_steps=0), q, k, v)
    assert np.allclose(it["w"][0, 0], J + eps * I, rtol=0, atol=1e-15)
    assert np.allclose(it["x"][0, 0], (J + eps * I) / (m + eps) ** 2, rtol=1e-14, atol=0)
    _, it = run(oracle_mod, cfg_of(w0, ns_steps=20), q, k, v)
    sm = (I - J / (m + eps)) / eps
    assert np.max(np.abs(it["x"][0, 0] - sm)) < 1e-10


def test_constant_keys_full_output_closed_form(oracle_mod):
    """With constant K, B = 1 everywhere and every column of A equals a_i = exp(-|q_i-c|_1/lam).
    Then BV_j = sum_n V_n, M_j = sum_n V_n / (m + eps) (row sums of W^-1 are 1/(m+eps)), and
    O_i = m (a_i - mean a) / sqrt(var a + delta) * sum_n V_n / (m + eps)."""
    m, eps, lam, delta = 16, 1.0, 4.0, 1e-5
    w0 = TINY.replace(eps=eps)
    q, k, v = make_inputs(w0)
    k = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    cfg = cfg_of(w0, ns_steps=30)
    out, _ = run(oracle_mod, cfg, q, k, v, inter=False)
    c = k[0, 0, 0].astype(np.float64)
    a = np.exp(-np.abs(q[0, 0].astype(np.float64) - c).sum(-1) / lam)
    z = (a - a.mean()) / math.sqrt(a.var() + cfg["delta"])
    sv = v[0, 0].astype(np.float64).sum(0)
    expect = m * z[:, None] * sv[None, :] / (m + eps)
    assert np.max(np.abs(out[0, 0] - expect)) <= 1e-9 * np.max(np.abs(expect))


# ---- P5: whitening invariants --------------------------------------------------------------
def test_whitening_invariants(oracle_mod):
    w0 = WORKLOADS["stage1_f32"].replace(batch=1, heads=2)
    q, k, v = make_inputs(w0)
    cfg = cfg_of(w0)
    out, it = run(oracle_mod, cfg, q, k, v)
    for h in range(2):
        A, Ah = it["a"][0, h], it["a_hat"][0, h]
        N = A.shape[0]
        var = A.var(axis=0)                                     # ddof=0: divide by N
        assert np.allclose(it["mu"][0, h], A.mean(axis=0), rtol=1e-13, atol=0)
        assert np.allclose(it["var"][0, h], var, rtol=1e-10, atol=1e-300)
        assert np.max(np.abs(Ah.sum(axis=0))) < 1e-9 * N
        assert np.allclose((Ah ** 2).mean(axis=0), var / (var + cfg["delta"]), rtol=1e-9)
        # every output column sums to zero over the tokens
        assert np.max(np.abs(out[0, h].sum(axis=0))) < 1e-9 * np.max(np.abs(out[0, h])) * N


def test_bias_is_column_mean_of_whitened_block(oracle_mod):
    w0 = TINY.replace(heads=3)
    q, k, v = make_inputs(w0)
    bias = make_bias(w0)
    _, it = run(oracle_mod, cfg_of(w0), q, k, v, bias=bias)
    for h in range(3):
        assert np.allclose(it["a_hat"][0, h].mean(axis=0), bias[h], rtol=0, atol=1e-12)


def test_whiten_off_passes_a_through(oracle_mod):
    q, k, v = make_inputs(TINY)
    _, it = run(oracle_mod, cfg_of(TINY, whiten=0), q, k, v, bias=make_bias(TINY))
    assert np.array_equal(it["a_hat"], it["a"])


# ---- P6: landmarks = all keys gives exact kernel attention ------------------------------
@pytest.mark.parametrize("grid", [8, 16])
def test_m_equals_n_is_exact_kernel_attention(oracle_mod, grid):
    n = grid * grid
    w0 = TINY.replace(grid_h=grid, grid_w=grid, num_landmarks=n, eps=0.0, whiten=0,
                      ns_steps=30)
    q, k, v = make_inputs(w0)
    out, it = run(oracle_mod, cfg_of(w0), q, k, v)
    Q, K, V = (x[0, 0].astype(np.float64) for x in (q, k, v))
    assert np.array_equal(it["landmarks"][0, 0], K)            # 1x1 pooling keeps every key
    exact = np.exp(-brute_cdist_l1(Q, K) / 4.0) @ V
    assert np.max(np.abs(out[0, 0] - exact)) <= 1e-10 * np.max(np.abs(exact))


def test_m_equals_n_with_eps_closed_form(oracle_mod):
    """With eps > 0: O = k(Q,K) (k(K,K) + eps I)^-1 k(K,K) V = k(Q,K) (I - eps (k(K,K)+eps I)^-1) V."""
    grid, eps = 8, 1e-3
    w0 = TINY.replace(grid_h=grid, grid_w=grid, num_landmarks=grid * grid, eps=eps, whiten=0,
                      ns_steps=30)
    q, k, v = make_inputs(w0)
    out, _ = run(oracle_mod, cfg_of(w0), q, k, v, inter=False)
    Q, K, V = (x[0, 0].astype(np.float64) for x in (q, k, v))
    kqk = np.exp(-brute_cdist_l1(Q, K) / 4.0)
    kkk = np.exp(-brute_cdist_l1(K, K) / 4.0)
    eps_used = cfg_of(w0)["eps"]
    n = K.shape[0]
    expect = kqk @ (V - eps_used * np.linalg.solve(kkk + eps_used * np.eye(n), V))
    assert np.max(np.abs(out[0, 0] - expect)) <= 1e-10 * np.max(np.abs(expect))


# ---- P8: pooling windows, landmark order, permutation structure -------------------------
def test_pooling_matches_reshape_mean(oracle_mod):
    for name in ["tiny_f32", "stage1_f32"]:
        w0 = WORKLOADS[name].replace(batch=1, heads=1)
        q, k, v = make_inputs(w0)
        _, it = run(oracle_mod, cfg_of(w0), q, k, v)
        s = int(round(math.sqrt(w0.num_landmarks)))
        expect = brute_pool(k[0, 0].astype(np.float64), w0.grid_h, w0.grid_w, s)
        assert np.allclose(it["landmarks"][0, 0], expect, rtol=1e-14, atol=1e-15)


def test_piecewise_constant_keys_give_window_values(oracle_mod):
    """Non-square grid 8x12, s=4, windows 2x3: K = landmark index of its window."""
    w0 = TINY.replace(grid_h=8, grid_w=12, num_landmarks=16)
    q, k, v = make_inputs(w0)
    rows = np.arange(8)[:, None] // 2
    cols = np.arange(12)[None, :] // 3
    win = (rows * 4 + cols).reshape(-1).astype(np.float32)            # row-major landmarks
    k = np.broadcast_to(win[None, None, :, None], k.shape).copy()
    _, it = run(oracle_mod, cfg_of(w0), q, k, v)
    L = it["landmarks"][0, 0]
    assert np.array_equal(L, np.broadcast_to(np.arange(16.0)[:, None], L.shape))


def test_permutation_structure(oracle_mod):
    w0 = TINY.replace(grid_h=8, grid_w=8, num_landmarks=4)     # windows 4x4
    q, k, v = make_inputs(w0)
    cfg = cfg_of(w0)
    out, _ = run(oracle_mod, cfg, q, k, v, inter=False)
    rng = np.random.default_rng(5)
    # permute Q rows: O rows permute the same way
    perm = rng.permutation(64)
    out_q, _ = run(oracle_mod, cfg, q[:, :, perm], k, v, inter=False)
    assert np.allclose(out_q, out[:, :, perm], rtol=0, atol=1e-12 * np.abs(out).max())
    # permute K and V tokens jointly inside each pooling window: O unchanged
    idx = np.arange(64).reshape(8, 8)
    new = idx.copy()
    for wr in range(2):
        for wc in range(2):
            blk = idx[wr * 4:(wr + 1) * 4, wc * 4:(wc + 1) * 4].reshape(-1)
            new[wr * 4:(wr + 1) * 4, wc * 4:(wc + 1) * 4] = rng.permutation(blk).reshape(4, 4)
    p2 = new.reshape(-1)
    out_kv, _ = run(oracle_mod, cfg, q, k[:, :, p2], v[:, :, p2], inter=False)
    assert np.allclose(out_kv, out, rtol=0, atol=1e-12 * np.abs(out).max())
    # but moving a key across windows changes the output
    p3 = np.arange(64)
    p3[[0, 63]] = p3[[63, 0]]
    out_x, _ = run(oracle_mod, cfg, q, k[:, :, p3], v, inter=False)
    assert np.abs(out_x - out).max() > 1e-6 * np.abs(out).max()


# ---- P9: hand example, d = 1, 2x2 grid, one landmark -----------------------------------
def test_hand_example_one_landmark(oracle_mod):
    """d=1, N=4 (2x2 grid), m=1 (2x2 window), lam=4, eps=0.5, delta=0.25, T=3.
    K = [1,3,5,7] -> L = 4; W = 1 + eps = 1.5; X0 = W/(W*W) = 1/1.5 (already exact);
    Q = [0,2,4,8] -> D_QL = [4,2,0,4] -> A = [e^-1, e^-.5, 1, e^-1];
    D_LK = [3,1,1,3] -> B = [e^-.75, e^-.25, e^-.25, e^-.75]; V = [1,-1,2,.5];
    BV = 1.5 e^-.75 + e^-.25; M = BV / 1.5; O_i = (A_i - mean A)/sqrt(var A + .25) * M."""
    import oracle
    cfg = dict(batch=1, heads=1, grid_h=2, grid_w=2, head_dim=1, num_landmarks=1, lam=4.0,
               eps=0.5, delta=0.25, ns_steps=3, whiten=1)
    q = np.array([0, 2, 4, 8.0]).reshape(1, 1, 4, 1)
    k = np.array([1, 3, 5, 7.0]).reshape(1, 1, 4, 1)
    v = np.array([1, -1, 2, 0.5]).reshape(1, 1, 4, 1)
    out, it = oracle.forward(cfg, q, k, v, intermediates=True)
    e = math.exp
    A = np.array([e(-1), e(-0.5), 1.0, e(-1)])
    Bv = np.array([e(-0.75), e(-0.25), e(-0.25), e(-0.75)])
    assert it["landmarks"].ravel()[0] == 4.0
    assert np.array_equal(it["d_ql"].ravel(), [4.0, 2.0, 0.0, 4.0])
    assert np.array_equal(it["d_lk"].ravel(), [3.0, 1.0, 1.0, 3.0])
    assert it["w"].ravel()[0] == 1.5
    assert abs(it["x"].ravel()[0] - 1 / 1.5) < 1e-15
    assert np.allclose(it["a"].ravel(), A, rtol=1e-15)
    assert np.allclose(it["b"].ravel(), Bv, rtol=1e-15)
    bv = 1.5 * e(-0.75) + e(-0.25)
    assert abs(it["bv"].ravel()[0] - bv) < 1e-14
    mean = A.mean()
    var = ((A - mean) ** 2).mean()
    expect = (A - mean) / math.sqrt(var + 0.25) * (bv / 1.5)
    assert np.allclose(out.ravel(), expect, rtol=1e-13, atol=1e-15)


# ---- P10: limits -------------------------------------------------------------------------
def test_large_lambda_limit(oracle_mod):
    """lam -> inf: every kernel value -> 1; with whitening off all rows of O coincide."""
    q, k, v = make_inputs(TINY)
    cfg = cfg_of(TINY, lam=1e12, whiten=0, eps=1.0, ns_steps=30)
    out, it = run(oracle_mod, cfg, q, k, v)
    assert np.allclose(it["a"], 1.0, atol=1e-9) and np.allclose(it["b"], 1.0, atol=1e-9)
    assert np.max(np.abs(out[0, 0] - out[0, 0, :1])) < 1e-8 * np.abs(out).max()


# ---- P11: integer inputs, exact distances ------------------------------------------------
def test_integer_distances_exact(oracle_mod):
    w0 = WORKLOADS["tiny_int"]
    q, k, v = make_inputs(w0)
    _, it = run(oracle_mod, cfg_of(w0), q, k, v)
    # in units of 1/16 every pooled value is an integer (16 keys per window)
    Q16 = (q[0, 0].astype(np.int64) * 16)
    K = k[0, 0].astype(np.int64)
    L16 = K.reshape(4, 4, 4, 4, 32).sum(axis=(1, 3)).reshape(16, 32)      # 16 * window mean
    K16 = K * 16
    dql16 = np.abs(Q16[:, None, :] - L16[None, :, :]).sum(-1)
    dlk16 = np.abs(L16[:, None, :] - K16[None, :, :]).sum(-1)
    dll16 = np.abs(L16[:, None, :] - L16[None, :, :]).sum(-1)
    assert np.array_equal(it["landmarks"][0, 0] * 16, L16.astype(np.float64))
    assert np.array_equal(it["d_ql"][0, 0] * 16, dql16.astype(np.float64))
    assert np.array_equal(it["d_lk"][0, 0] * 16, dlk16.astype(np.float64))
    assert np.array_equal(it["d_ll"][0, 0] * 16, dll16.astype(np.float64))


def test_exp_of_distances(oracle_mod):
    """A, B, W are exp(-D/lam) of the reported distances (libm exp vs numpy exp)."""
    q, k, v = make_inputs(TINY)
    cfg = cfg_of(TINY)
    _, it = run(oracle_mod, cfg, q, k, v)
    assert np.allclose(it["a"], np.exp(-it["d_ql"] / cfg["lam"]), rtol=1e-15, atol=0)
    assert np.allclose(it["b"], np.exp(-it["d_lk"] / cfg["lam"]), rtol=1e-15, atol=0)
    # the distances themselves against a brute-force numpy cdist
    L = it["landmarks"][0, 0]
    Q, K = q[0, 0].astype(np.float64), k[0, 0].astype(np.float64)
    assert np.allclose(it["d_ql"][0, 0], brute_cdist_l1(Q, L), rtol=1e-14, atol=1e-13)
    assert np.allclose(it["d_lk"][0, 0], brute_cdist_l1(L, K), rtol=1e-14, atol=1e-13)


# ---- interface behaviour -------------------------------------------------------------------
def test_rejects_bad_configs(oracle_mod):
    q, k, v = make_inputs(TINY)
    for bad in [dict(num_landmarks=15), dict(num_landmarks=9), dict(lam=0.0), dict(ns_steps=-1),
                dict(delta=0.0)]:
        with pytest.raises(oracle_mod.OracleError):
            oracle_mod.forward(cfg_of(TINY, **bad), q, k, v)


def test_empty_batch(oracle_mod):
    w0 = TINY.replace(batch=0)
    z = np.zeros((0, 1, 256, 32), dtype=np.float32)
    out, _ = oracle_mod.forward(cfg_of(w0), z, z, z)
    assert out.shape == (0, 1, 256, 32)


def test_slices_match_full_run(oracle_mod):
    w0 = TINY.replace(batch=2, heads=3)
    q, k, v = make_inputs(w0)
    cfg = cfg_of(w0)
    full, _ = oracle_mod.forward(cfg, q, k, v)
    part, _ = oracle_mod.forward(cfg, q, k, v, slices=(2, 3))
    flat_f, flat_p = full.reshape(6, -1), part.reshape(6, -1)
    assert np.array_equal(flat_p[2:5], flat_f[2:5])
    assert not flat_p[:2].any() and not flat_p[5:].any()
