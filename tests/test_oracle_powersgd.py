"""Pins of the oracle's PowerSGD step: exact reconstruction of a matrix of
rank <= r, orthonormality, agreement with numpy's QR (a library routine)
on the orthogonalisation, and the error-feedback identity."""
import numpy as np

import oracle
from gradient_compression_ef_gb300 import inputs


def test_exact_low_rank_is_reconstructed():
    r = np.random.default_rng(1)
    m, n, rank = 60, 45, 4
    M = (r.standard_normal((m, rank)) @ r.standard_normal((rank, n))).astype(np.float32)
    Q = r.standard_normal((n, rank)).astype(np.float32)
    P, Q2, E = oracle.powersgd_step(M, np.zeros_like(M), Q, rank)
    approx = P.astype(np.float64) @ Q2.astype(np.float64).T
    assert np.linalg.norm(approx - M) <= 1e-5 * np.linalg.norm(M)
    assert np.abs(E).max() <= 1e-5 * np.abs(M).max()


def test_orthonormal_and_matches_numpy_qr():
    r = np.random.default_rng(2)
    m, n, rank = 80, 50, 5
    G = r.standard_normal((m, n)).astype(np.float32)
    E = (0.1 * r.standard_normal((m, n))).astype(np.float32)
    Q = r.standard_normal((n, rank)).astype(np.float32)
    P, Q2, E2 = oracle.powersgd_step(G, E, Q, rank)
    Pd = P.astype(np.float64)
    assert np.abs(Pd.T @ Pd - np.eye(rank)).max() < 1e-6
    M = G.astype(np.float64) + E.astype(np.float64)
    qr_q, qr_r = np.linalg.qr(M @ Q.astype(np.float64))
    qr_q = qr_q * np.sign(np.diag(qr_r))  # Gram-Schmidt has R_ii > 0
    assert np.abs(Pd - qr_q).max() < 1e-6
    # Q' = M^T P_hat and E' = M - P_hat Q'^T
    assert np.abs(Q2 - (M.T @ Pd)).max() < 1e-5 * np.abs(M.T @ Pd).max()
    assert np.abs(E2 - (M - Pd @ (M.T @ Pd).T)).max() < 1e-5 * np.abs(M).max()


def test_zero_gradient():
    G = np.zeros((7, 9), np.float32)
    P, Q2, E = oracle.powersgd_step(G, G, np.ones((9, 2), np.float32), 2)
    assert not P.any() and not Q2.any() and not E.any()


def test_power_iteration_on_workload_shape():
    """Repeated steps on the rank-16 workload: the carried Q converges
    towards the top singular subspace, so the residual energy after 5 steps
    with a fresh error each step is below the rank-4 truncation bound."""
    M, Q0 = inputs.low_rank_matrix(256, 192, r=4)
    Q = Q0
    for _ in range(5):
        P, Q, _ = oracle.powersgd_step(M, np.zeros_like(M), Q, 4)
    approx = P.astype(np.float64) @ Q.astype(np.float64).T
    s = np.linalg.svd(M.astype(np.float64), compute_uv=False)
    best = np.sqrt(np.sum(s[4:] ** 2))  # Eckart-Young optimum for rank 4
    resid = np.linalg.norm(M - approx)
    assert resid <= 1.05 * best
