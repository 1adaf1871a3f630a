"""Pins for the other feature maps of the oracle: the identity path (the recurrence on
feature values the caller has mapped already), the positive random-feature map and the
orthogonal random-feature construction. Each is pinned to something other than itself:
the elu + 1 path, a closed form on hand-picked values, the unbiasedness of the estimator
(E[phi(q) . phi(k)] = exp(q . k) over Gaussian rows) within a bound of the central limit
theorem, and the orthogonality and row lengths of the ORF matrix."""
import math

import numpy as np
import pytest

import oracle
import synthetic


def test_identity_path_equals_elu1_path_on_premapped_inputs():
    q, k, v = (synthetic.normal(11, i, (2, 3, 70, 16), 1.0, "f32") for i in range(3))
    a = oracle.causal_fwd(q, k, v)
    fq, fk = oracle.phi(q.astype(np.float64)), oracle.phi(k.astype(np.float64))
    b = oracle.causal_fwd(fq, fk, v.astype(np.float64), phi="identity")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # and the identity path does not apply elu + 1 again
    c = oracle.causal_fwd(q.astype(np.float64) + 3.0, k.astype(np.float64) + 3.0, v.astype(np.float64),
                          phi="identity")
    d = oracle.causal_fwd(q + np.float32(3.0), k + np.float32(3.0), v)
    assert not np.allclose(c[0], d[0])


def test_prf_closed_form():
    x = np.array([[0.5], [-1.0]])          # two tokens, d = 1
    W = np.array([[1.0], [2.0], [0.0]])    # m = 3
    got = oracle.phi_prf(x, W)
    want = np.array([[math.exp(0.5 - 0.125), math.exp(1.0 - 0.125), math.exp(-0.125)],
                     [math.exp(-1.0 - 0.5), math.exp(-2.0 - 0.5), math.exp(-0.5)]]) / math.sqrt(3.0)
    np.testing.assert_allclose(got, want, rtol=1e-15)


def _unbiased(W, q, k):
    fq, fk = oracle.phi_prf(q, W), oracle.phi_prf(k, W)
    terms = fq * fk * W.shape[0]            # m phi_i(q) phi_i(k): the per-feature estimates
    return terms.mean(), terms.std() / math.sqrt(W.shape[0]), math.exp(float(q @ k))


@pytest.mark.parametrize("kind", ["prf", "orf"])
def test_random_features_estimate_the_exponential_kernel(kind):
    d, m = 8, 1 << 16
    G = synthetic.normal(21, 0, (m, d), 1.0, "f32").astype(np.float64)
    W = G if kind == "prf" else oracle.orf_matrix(G, synthetic.normal(21, 1, (m, d), 1.0, "f32"))
    q = synthetic.normal(22, 0, (d,), 0.4, "f32").astype(np.float64)
    k = synthetic.normal(22, 1, (d,), 0.4, "f32").astype(np.float64)
    mean, se, want = _unbiased(W, q, k)
    assert abs(mean - want) < 5 * se, (mean, want, se)
    # a planted slip (the -|x|^2 / 2 term dropped) is far outside that bound
    fq = np.exp(q @ W.T) / math.sqrt(m)
    fk = np.exp(k @ W.T) / math.sqrt(m)
    assert abs((fq * fk).sum() - want) > 50 * se


def test_orf_rows_are_orthogonal_within_blocks_with_gaussian_lengths():
    d, m = 16, 64
    G = synthetic.normal(31, 0, (m, d), 1.0, "f32")
    N = synthetic.normal(31, 1, (m, d), 1.0, "f32")
    W = oracle.orf_matrix(G, N)
    for b0 in range(0, m, d):
        blk = W[b0:b0 + d]
        gram = blk @ blk.T
        np.testing.assert_allclose(gram - np.diag(np.diag(gram)), 0.0, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(W, axis=1), np.linalg.norm(N.astype(np.float64), axis=1), rtol=1e-12)


def test_prf_features_through_the_recurrence_match_the_all_pairs_form():
    """Causal linear attention on PRF features equals the masked all-pairs form with the
    kernel phi(q).phi(k) (the recurrence and the pairwise form agree for any feature map)."""
    B, H, T, d, m = 1, 2, 40, 8, 16
    q, k, v = (synthetic.normal(41, i, (B, H, T, d), 0.5, "f32") for i in range(3))
    W = synthetic.normal(41, 5, (m, d), 1.0, "f32")
    fq, fk = oracle.phi_prf(q, W), oracle.phi_prf(k, W)
    out, _, _ = oracle.causal_fwd(fq, fk, v.astype(np.float64), phi="identity")
    A = np.einsum("bhtm,bhsm->bhts", fq, fk) * np.tril(np.ones((T, T)))
    ref = np.einsum("bhts,bhsv->bhtv", A, v.astype(np.float64)) / (A.sum(-1) + 1e-6)[..., None]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
