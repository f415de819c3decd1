"""Pins for the oracle's q/k L2 normalisation (oracle/norm.py), checked against
what the mathematics fixes rather than against a second copy of the formula.

Source: the sliding-window paragraph of the talk "Qwen系列模型线性注意力高性能优化实践"
takes every key to have unit L2 norm, which is what bounds the factor
I - beta k k^T; the epsilon 1e-6 under the square root is this library's
reading (the pages give none)."""
import numpy as np

from oracle.norm import L2NORM_EPS, l2_normalize, l2_normalize_backward


def rows(n=200, d=64, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d)) * np.exp(rng.standard_normal((n, 1)))   # norms spread over decades
    return x


def test_rows_have_unit_norm():
    x = rows()
    y = l2_normalize(x)
    ss = np.sum(x * x, axis=1)
    norms = np.sqrt(np.sum(y * y, axis=1))
    # exact value: sqrt(ss / (ss + eps))
    assert np.all(np.abs(norms - 1.0) <= L2NORM_EPS / ss + 1e-14)


def test_direction_is_kept():
    x = rows(seed=1)
    y = l2_normalize(x)
    # y is a positive multiple of x: same signs, and |x . y| = |x| |y|
    assert np.all(np.sign(y) == np.sign(x))
    cos = np.sum(x * y, axis=1) / (np.linalg.norm(x, axis=1) * np.linalg.norm(y, axis=1))
    assert np.all(np.abs(cos - 1.0) < 1e-13)


def test_hand_computed_values():
    # (3, 4) has norm 5; (0, 0, 2) has norm 2; a zero row stays zero
    y = l2_normalize(np.array([[3.0, 4.0, 0.0], [0.0, 0.0, 2.0], [0.0, 0.0, 0.0]]), eps=0.0 + 1e-300)
    np.testing.assert_allclose(y[0], [0.6, 0.8, 0.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(y[1], [0.0, 0.0, 1.0], rtol=0, atol=1e-15)
    assert np.all(y[2] == 0.0)
    z = l2_normalize(np.zeros((2, 8)))
    assert np.all(z == 0.0)


def test_epsilon_enters_under_the_square_root():
    # one row of squared norm eps: x / sqrt(2 eps)
    x = np.zeros((1, 4))
    x[0, 0] = np.sqrt(L2NORM_EPS)
    y = l2_normalize(x)
    assert abs(y[0, 0] - np.sqrt(L2NORM_EPS) / np.sqrt(2 * L2NORM_EPS)) < 1e-15


def test_positive_scale_invariance():
    # exact up to the epsilon: y(c x) / y(x) = sqrt((ss + eps) / (ss + eps / c^2))
    x = rows(seed=2)
    ss = np.sum(x * x, axis=1, keepdims=True)
    for c in (1e-1, 3.0, 250.0):
        bound = L2NORM_EPS / np.minimum(ss, c * c * ss) + 1e-14
        rel = np.abs(l2_normalize(c * x) - l2_normalize(x)) / np.abs(l2_normalize(x))
        assert np.all(rel <= bound)


def test_normalised_keys_bound_the_transition():
    """The property the normalisation is there for: with |k| = 1 and beta in
    (0, 1), I - beta k k^T has eigenvalues 1 (multiplicity d-1) and 1 - beta,
    so its spectral norm is exactly 1 and its determinant 1 - beta."""
    rng = np.random.default_rng(3)
    raw = rng.standard_normal((20, 16)) * 7.0
    k = l2_normalize(raw)
    tol = 2 * L2NORM_EPS / np.min(np.sum(raw * raw, axis=1)) + 1e-12   # |k|^2 = ss / (ss + eps)
    for t in range(20):
        beta = rng.uniform(0.05, 0.95)
        m = np.eye(16) - beta * np.outer(k[t], k[t])
        ev = np.sort(np.linalg.eigvalsh(m))
        assert abs(ev[0] - (1 - beta)) < tol and np.all(np.abs(ev[1:] - 1) < 1e-12)
        assert abs(np.linalg.det(m) - (1 - beta)) < tol


def test_batched_shapes_normalise_the_last_axis():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 5, 3, 32))
    y = l2_normalize(x)
    assert y.shape == x.shape
    for idx in np.ndindex(*x.shape[:-1]):
        np.testing.assert_allclose(y[idx], l2_normalize(x[idx][None])[0], rtol=0, atol=1e-15)


def test_backward_matches_finite_differences():
    """The backward against central differences of the forward: a code path
    that shares nothing with the Jacobian's closed form (a dropped x x^T term
    or a wrong power of n misses by far more than the differencing error)."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 6)) * np.array([[1e-2], [0.3], [1.0], [7.0], [40.0]])
    dy = rng.standard_normal((5, 6))
    got = l2_normalize_backward(x, dy)
    num = np.zeros_like(x)
    for i in range(x.shape[0]):
        h = 1e-6 * max(1.0, np.abs(x[i]).max())
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num[i, j] = (np.sum(l2_normalize(xp[i]) * dy[i]) - np.sum(l2_normalize(xm[i]) * dy[i])) / (2 * h)
    for i in range(x.shape[0]):
        scale = max(1.0, np.abs(num[i]).max())
        assert np.abs(got[i] - num[i]).max() <= 1e-6 * scale, i


def test_backward_is_orthogonal_to_the_row_and_scales_inversely():
    """x . dx = (x . dy) eps / n^3 (zero as eps -> 0: the output cannot grow
    along x); and dx at c x is dx at x divided by c (the map is scale-free)."""
    x = rows(n=50, d=32, seed=3)
    dy = np.random.default_rng(4).standard_normal(x.shape)
    dx = l2_normalize_backward(x, dy)
    n = np.sqrt(np.sum(x * x, axis=1) + L2NORM_EPS)
    np.testing.assert_allclose(np.sum(x * dx, axis=1), np.sum(x * dy, axis=1) * L2NORM_EPS / n ** 3,
                               rtol=1e-6, atol=1e-12)
    sel = n > 1.0                                    # rows where eps is negligible
    big, dyb = x[sel], dy[sel]
    assert len(big) > 10
    ref = l2_normalize_backward(big, dyb) / 3.0
    # eps shifts both sides by about eps / n^2 relative to the size of the terms
    # that cancel inside dx, hence an absolute floor at that scale
    np.testing.assert_allclose(l2_normalize_backward(3.0 * big, dyb), ref, rtol=1e-5,
                               atol=1e-5 * np.abs(ref).max())
