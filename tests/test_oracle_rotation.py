"""Pins of the oracle's offline rotation builder R = U·H_Had·P_br and the key error identity."""
import numpy as np

import oracle
import oscar_synthetic as syn
from tests.helpers import bf16_bits


def test_hadamard_closed_form():
    H2 = oracle.hadamard(2) * np.sqrt(2)
    assert np.array_equal(H2, np.array([[1, 1], [1, -1]]))
    H = oracle.hadamard(128)
    assert np.allclose(np.abs(H), 1 / np.sqrt(128), atol=0, rtol=1e-15)
    assert np.abs(H @ H.T - np.eye(128)).max() < 1e-13
    # Sylvester: entry (i, j) = (-1)^popcount(i & j) / sqrt(n)
    for i, j in [(0, 0), (1, 1), (3, 5), (127, 127), (64, 65)]:
        assert np.sign(H[i, j]) == (-1) ** bin(i & j).count("1")


def test_bit_reversal_permutation():
    P = oracle.bit_reversal_permutation(128)
    assert np.array_equal(P @ P, np.eye(128))          # involution
    assert np.array_equal(P, P.T)
    assert P[1, 64] == 1 and P[2, 32] == 1 and P[3, 96] == 1 and P[127, 127] == 1
    # The permutation sends each group of 4 consecutive output channels to
    # channels spread across the whole range (one per importance quarter).
    x = np.arange(128.0)
    y = x @ P                                           # y[j] = x[br(j)]
    assert list(y[:4]) == [0, 64, 32, 96]


def test_eig_basis_diagonal_and_2x2():
    C = np.diag([1.0, 5.0, 3.0])
    U = oracle.eig_basis(C)
    assert np.array_equal(U, np.array([[0, 0, 1], [1, 0, 0], [0, 1, 0]], float))
    U2 = oracle.eig_basis(np.array([[2.0, 1.0], [1.0, 2.0]]))
    s = 1 / np.sqrt(2)
    assert np.allclose(U2, np.array([[s, s], [s, -s]]), atol=1e-15)


def test_rotation_orthogonal_and_diagonalises():
    prof = syn.channel_profile(0, 0, 2)
    q, k, v = syn.calibration_set(0, 0, 4, prof)
    qd = oracle.bf16_to_f64(bf16_bits(q[0]))
    C = oracle.query_covariance(qd)
    U = oracle.eig_basis(C)
    Dg = U.T @ C @ U
    off = Dg - np.diag(np.diag(Dg))
    assert np.abs(off).max() < 1e-9 * np.abs(Dg).max()
    assert np.all(np.diff(np.diag(Dg)) <= 1e-9)        # descending
    R = oracle.rotation_from_covariance(C)
    assert np.abs(R @ R.T - np.eye(128)).max() < 1e-12
    R32 = R.astype(np.float32).astype(np.float64)
    assert np.abs(R32 @ R32.T - np.eye(128)).max() < 1e-6


def test_score_weighted_covariance_uniform_attention_is_rank_one():
    """q = 0 gives uniform S = 1/T, so S V = mean(V) in every row and C_S = vbar vbar^T."""
    rng = np.random.default_rng(3)
    v = rng.normal(size=(50, 8))
    k = rng.normal(size=(50, 8))
    q = np.zeros((7, 8))
    C = oracle.score_weighted_value_covariance(q, k, v, 0.3)
    vbar = v.mean(axis=0)
    assert np.allclose(C, np.outer(vbar, vbar), rtol=1e-12, atol=1e-14)


def test_score_weighted_covariance_one_hot_attention():
    """A query aligned with one key by a huge margin attends to it alone: C_S = (1/N) sum v_a v_a^T."""
    rng = np.random.default_rng(4)
    k = np.eye(6)
    v = rng.normal(size=(6, 5))
    picks = [0, 3, 3, 5]
    q = np.stack([1e4 * k[i] for i in picks])
    C = oracle.score_weighted_value_covariance(q, k, v, 1.0)
    ref = sum(np.outer(v[i], v[i]) for i in picks) / len(picks)
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-14)


def test_query_covariance_two_samples():
    # (1/2)[(1,2)^T(1,2) + (3,-1)^T(3,-1)] = (1/2)[[1+9, 2-3], [2-3, 4+1]]
    q = np.array([[1.0, 2.0], [3.0, -1.0]])
    assert np.array_equal(oracle.query_covariance(q), np.array([[5.0, -0.5], [-0.5, 2.5]]))


def test_joint_rotation_preserves_logits():
    rng = np.random.default_rng(7)
    R = oracle.rotation_from_covariance(np.cov(rng.normal(size=(128, 400))))
    q = rng.normal(size=(3, 128))
    k = rng.normal(size=(9, 128))
    assert np.allclose((q @ R) @ (k @ R).T, q @ k.T, rtol=1e-12, atol=1e-10)


def test_key_error_identity():
    """||QK^T - QK_hat^T||_F^2 = tr((K-K_hat) Q^T Q (K-K_hat)^T) on random and on quantized keys."""
    rng = np.random.default_rng(11)
    Q = rng.normal(size=(40, 128))
    K = rng.normal(size=(30, 128))
    Kh = K + 0.1 * rng.normal(size=K.shape)
    a, b = oracle.key_logit_error(Q, K, Kh), oracle.key_logit_error_trace(Q, K, Kh)
    assert abs(a - b) <= 1e-10 * a
    packed, z, s = oracle.quantize_rows(K.astype(np.float32), 128, 0.96)
    Kq = np.stack([oracle.dequant_row(packed[i], z[i], s[i], 128, 128) for i in range(K.shape[0])])
    a, b = oracle.key_logit_error(Q, K, Kq), oracle.key_logit_error_trace(Q, K, Kq)
    assert abs(a - b) <= 1e-10 * a
