"""Pins for the oracle's backward pass (oracle/backward.py).

The gradients are pinned to central finite differences of the forward oracle
(the token-by-token recurrence of the talk "Qwen系列模型线性注意力高性能优化实践",
itself pinned in test_oracle_pins.py) on tiny problems: a code path that shares
nothing with the backward's derivation.  A dropped or mis-signed term moves some
gradient far outside the finite-difference error, which the last test checks
for the terms that are easiest to get wrong."""
import numpy as np
import pytest

import oracle
from oracle.backward import _unit_backward, gdn_backward_reference

EPS = 1e-6


def tiny(seed=0, lens=(6,), H=2, dk=3, dv=4):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = len(lens)
    return dict(
        q=rng.standard_normal((T, H, dk)), k=rng.standard_normal((T, H, dk)) * 0.6,
        v=rng.standard_normal((T, H, dv)), g=-rng.uniform(0.01, 0.7, (T, H)), beta=rng.uniform(0.1, 0.9, (T, H)),
        s0=rng.standard_normal((N, H, dk, dv)) * 0.5, cu=cu,
        do=rng.standard_normal((T, H, dv)), dsT=rng.standard_normal((N, H, dk, dv)), scale=0.7)


def loss(p):
    o, sf = oracle.gdn_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["s0"], p["cu"], scale=p["scale"])
    return float(np.sum(o * p["do"]) + np.sum(sf * p["dsT"]))


def numeric_grad(p, name):
    x = p[name]
    grad = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        orig = x[idx]
        x[idx] = orig + EPS
        lp = loss(p)
        x[idx] = orig - EPS
        lm = loss(p)
        x[idx] = orig
        grad[idx] = (lp - lm) / (2 * EPS)
    return grad


def analytic(p):
    return gdn_backward_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["s0"], p["cu"], scale=p["scale"],
                                  do=p["do"], d_final_state=p["dsT"])


@pytest.mark.parametrize("lens", [(6,), (4, 1, 5)])
def test_gradients_match_finite_differences(lens):
    p = tiny(seed=len(lens), lens=lens)
    got = dict(zip(["q", "k", "v", "g", "beta", "s0"], analytic(p)))
    for name in ["q", "k", "v", "g", "beta", "s0"]:
        num = numeric_grad(p, name)
        scale = max(1.0, float(np.abs(num).max()))
        assert np.abs(got[name] - num).max() <= 1e-6 * scale, name


def test_no_upstream_gradient_gives_zero():
    p = tiny(seed=3)
    p["do"] = np.zeros_like(p["do"])
    p["dsT"] = np.zeros_like(p["dsT"])
    for x in analytic(p):
        assert np.all(x == 0.0)


def test_linear_in_the_upstream_gradients():
    p = tiny(seed=4)
    a = analytic(p)
    p2 = dict(p, do=np.random.default_rng(9).standard_normal(p["do"].shape), dsT=np.zeros_like(p["dsT"]))
    b = analytic(p2)
    p3 = dict(p, do=2.0 * p["do"] - 3.0 * p2["do"], dsT=2.0 * p["dsT"])
    c = analytic(p3)
    for x, y, z in zip(a, b, c):
        np.testing.assert_allclose(z, 2.0 * x - 3.0 * y, rtol=1e-10, atol=1e-12)


def test_zero_beta_closed_forms():
    """beta = 0: S_t = gamma_t S_0, so dv = dk = 0, dq_t = scale gamma_t S_0^T do_t
    and dS_0 = sum_t scale gamma_t do_t q_t^T + gamma_T dS_T."""
    p = tiny(seed=5, lens=(7,), H=1)
    p["beta"] = np.zeros_like(p["beta"])
    dq, dk, dv, dg, db, ds0 = analytic(p)
    assert np.all(dk == 0.0) and np.all(dv == 0.0)
    gam = np.exp(np.cumsum(p["g"][:, 0]))
    S0 = p["s0"][0, 0].T                                     # dv x dk
    dq_ref = p["scale"] * gam[:, None] * (p["do"][:, 0] @ S0)
    np.testing.assert_allclose(dq[:, 0], dq_ref, rtol=1e-12, atol=1e-12)
    dS0 = p["scale"] * np.einsum("t,ti,tj->ij", gam, p["do"][:, 0], p["q"][:, 0]) + gam[-1] * p["dsT"][0, 0].T
    np.testing.assert_allclose(ds0[0, 0], dS0.T, rtol=1e-12, atol=1e-12)


def test_finite_differences_catch_a_dropped_term():
    """The check above is sharp: dk without the dA^T half of the symmetric term,
    or dbeta without its decay term, misses the finite differences by far more
    than their error."""
    p = tiny(seed=6, lens=(5,), H=1)
    num_k = numeric_grad(p, "k")[:, 0]
    num_b = numeric_grad(p, "beta")[:, 0]
    q, k, v, g, b = (p[n][:, 0] for n in ("q", "k", "v", "g", "beta"))
    dq, dk, dv, dg, db, _ = _unit_backward(q, k, v, g, b, p["s0"][0, 0].T, p["do"][:, 0], p["dsT"][0, 0].T,
                                           p["scale"])
    assert np.abs(dk - num_k).max() < 1e-6 and np.abs(db - num_b).max() < 1e-6
    # rebuild the two terms and drop them
    alpha = np.exp(g)
    S = [p["s0"][0, 0].T]
    for t in range(len(g)):
        A = alpha[t] * (np.eye(3) - b[t] * np.outer(k[t], k[t]))
        S.append(S[-1] @ A + b[t] * np.outer(v[t], k[t]))
    G = p["dsT"][0, 0].T.copy()
    wrong_k, wrong_b = dk.copy(), db.copy()
    for t in range(len(g) - 1, -1, -1):
        G = G + p["scale"] * np.outer(p["do"][t, 0], q[t])
        dA = S[t].T @ G
        wrong_k[t] += alpha[t] * b[t] * (dA.T @ k[t])          # removes the dA^T k half
        wrong_b[t] += alpha[t] * (k[t] @ dA @ k[t])            # removes the decay term
        G = G @ (alpha[t] * (np.eye(3) - b[t] * np.outer(k[t], k[t]))).T
    assert np.abs(wrong_k - num_k).max() > 1e-3
    assert np.abs(wrong_b - num_b).max() > 1e-3


@pytest.mark.parametrize("lens,C", [((6,), 64), ((13,), 4), ((9, 1, 7), 3), ((70,), 16)])
def test_chunked_form_matches_the_token_backward(lens, C):
    """The chunked (WY) backward — the algebra a chunked kernel runs, one chunk
    at a time with the start states of a forward sweep and dS0 handed to the
    chunk before — gives the token recurrence's gradients to rounding, with
    ragged last chunks and packed sequences."""
    from oracle.backward import gdn_backward_chunked
    p = tiny(seed=len(lens) + C, lens=lens, dk=5, dv=4)
    args = (p["q"], p["k"], p["v"], p["g"], p["beta"], p["s0"], p["cu"])
    kw = dict(scale=p["scale"], do=p["do"], d_final_state=p["dsT"])
    a = gdn_backward_reference(*args, **kw)
    b = gdn_backward_chunked(*args, C=C, **kw)
    for x, y in zip(a, b):
        assert np.abs(x - y).max() <= 1e-11 * max(1.0, float(np.abs(x).max()))


def test_value_column_slices_sum_to_the_gradients():
    """The state's value rows evolve independently (S_t's row i sees only
    v_t[i] and its own past), so the problem restricted to a set of value
    columns (v, S0, dO, dS_T cut to those columns) is a GDN problem of its own:
    its dv and dS0 are the full problem's columns, and the full dq, dk, dg and
    dbeta are the sums of the slices' — the decomposition a backward that
    splits the value dimension across workers relies on."""
    p = tiny(seed=11, lens=(9, 4), H=2, dk=3, dv=6)
    args = (p["q"], p["k"], p["v"], p["g"], p["beta"], p["s0"], p["cu"])
    full = gdn_backward_reference(*args, scale=p["scale"], do=p["do"], d_final_state=p["dsT"])
    sums = [np.zeros_like(full[i]) for i in (0, 1, 3, 4)]
    for cols in (slice(0, 2), slice(2, 5), slice(5, 6)):
        part = gdn_backward_reference(p["q"], p["k"], p["v"][..., cols], p["g"], p["beta"], p["s0"][..., cols],
                                      p["cu"], scale=p["scale"], do=p["do"][..., cols],
                                      d_final_state=p["dsT"][..., cols])
        np.testing.assert_allclose(part[2], full[2][..., cols], rtol=1e-12, atol=1e-12)   # dv
        np.testing.assert_allclose(part[5], full[5][..., cols], rtol=1e-12, atol=1e-12)   # dS0
        for acc, i in zip(sums, (0, 1, 3, 4)):
            acc += part[i]
    for acc, i in zip(sums, (0, 1, 3, 4)):
        np.testing.assert_allclose(acc, full[i], rtol=1e-10, atol=1e-12)


def test_zero_padding_leaves_the_real_gradients_unchanged():
    """Tokens with q = k = v = 0, beta = 0, g = 0 and dO = 0 appended to a
    sequence are identity steps (A_t = I, no write, no output), so the real
    tokens' gradients and dS0 do not change — the padding a chunked kernel
    applies to a short last chunk.  (The padded tokens' own dg need not be zero:
    their gate still scales the state; a kernel never writes those rows.)"""
    p = tiny(seed=12, lens=(7,), H=2, dk=3, dv=4)
    base = gdn_backward_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["s0"], p["cu"], scale=p["scale"],
                                  do=p["do"], d_final_state=p["dsT"])
    pad = 5
    z = lambda a: np.concatenate([a, np.zeros((pad,) + a.shape[1:])])
    cu = np.array([0, 7 + pad], dtype=np.int64)
    padded = gdn_backward_reference(z(p["q"]), z(p["k"]), z(p["v"]), z(p["g"]), z(p["beta"]), p["s0"], cu,
                                    scale=p["scale"], do=z(p["do"]), d_final_state=p["dsT"])
    for i in range(5):
        np.testing.assert_allclose(padded[i][:7], base[i], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(padded[5], base[5], rtol=1e-12, atol=1e-12)


def test_chunked_form_without_initial_state_or_final_gradient():
    """initial_state = None (zero) and d_final_state = None (zero) take the
    same paths in both forms, as the full-size GPU check uses them."""
    from oracle.backward import gdn_backward_chunked
    p = tiny(seed=13, lens=(21, 2), dk=4, dv=3)
    args = (p["q"], p["k"], p["v"], p["g"], p["beta"], None, p["cu"])
    a = gdn_backward_reference(*args, scale=p["scale"], do=p["do"], d_final_state=None)
    b = gdn_backward_chunked(*args, scale=p["scale"], do=p["do"], d_final_state=None, C=8)
    z = gdn_backward_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], np.zeros_like(p["s0"]), p["cu"],
                               scale=p["scale"], do=p["do"], d_final_state=np.zeros_like(p["dsT"]))
    for x, y, w in zip(a, b, z):
        assert np.abs(x - y).max() <= 1e-11 * max(1.0, float(np.abs(x).max()))
        np.testing.assert_array_equal(x, w)
