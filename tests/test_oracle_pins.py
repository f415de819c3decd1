"""Pins for the fp64 oracle: closed forms, invariants and an independent
algorithm, chosen so that a plausible mistake in the oracle fails at least one
of them (test_planted_mistakes_are_caught plants each mistake in the oracle and
checks exactly that).

Sources: the recurrence S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) +
beta_t v_t k_t^T, o_t = scale S_t q_t, alpha_t = exp(g_t) (FlashQLA talk
"Qwen系列模型线性注意力高性能优化实践", recurrent-form and GDN paragraphs); the
chunked four-step method, Gamma-extraction, forward merge, difference recursion
and compute-for-memory sequence parallelism (same talk, the paragraphs of those
names); the sliding-window property (same talk, sliding-window paragraph).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import chunked, gate

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def problem(T, H=1, dk=8, dv=6, seed=0, gate_scale=0.3, n_seqs=1, s0=True, lens=None):
    """Small fp64 problem, packed layout; keys are unit norm."""
    rng = np.random.default_rng(seed)
    if lens is None:
        lens = [T // n_seqs + (1 if i < T % n_seqs else 0) for i in range(n_seqs)]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -gate_scale * rng.random((T, H))
    b = rng.random((T, H))
    S0 = rng.standard_normal((len(lens), H, dk, dv)) if s0 else None
    return dict(q=q, k=k, v=v, g=g, beta=b, initial_state=S0, cu_seqlens=cu)


def run(p, scale=0.7, mutation=0, **kw):
    return oracle.gdn_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["initial_state"],
                                p["cu_seqlens"], scale=scale, mutation=mutation, **kw)


def math_state(sf_nh):
    """stored [dk, dv] -> math orientation S [dv, dk]."""
    return sf_nh.T


# ---------------------------------------------------------------- pin checks
# Each returns the max deviation from what the mathematics fixes; the tests
# assert it is tiny, and the planted-mistake test asserts some check is not.

def pin_beta0_gate0(mutation=0):
    p = problem(23, dk=5, dv=4, seed=1)
    p["beta"][:] = 0.0
    p["g"][:] = 0.0
    o, sf = run(p, mutation=mutation)
    S0 = math_state(p["initial_state"][0, 0])
    want_o = 0.7 * (p["q"][:, 0] @ S0.T)
    return max(np.abs(sf - p["initial_state"]).max(), np.abs(o[:, 0] - want_o).max())


def pin_beta0_decay(mutation=0):
    p = problem(23, dk=5, dv=4, seed=2, gate_scale=0.5)
    p["beta"][:] = 0.0
    o, sf = run(p, mutation=mutation)
    G = np.cumsum(p["g"][:, 0])
    S0 = math_state(p["initial_state"][0, 0])
    want_o = 0.7 * np.exp(G)[:, None] * (p["q"][:, 0] @ S0.T)
    want_s = np.exp(G[-1]) * p["initial_state"]
    return max(np.abs(sf - want_s).max(), np.abs(o[:, 0] - want_o).max())


def pin_single_token(mutation=0):
    p = problem(1, dk=5, dv=4, seed=3, s0=False)
    o, sf = run(p, scale=0.37, mutation=mutation)
    k, q, v, b = p["k"][0, 0], p["q"][0, 0], p["v"][0, 0], p["beta"][0, 0]
    want_S = b * np.outer(v, k)                    # S_1 = beta v k^T
    want_o = 0.37 * b * (k @ q) * v                # o_1 = scale S_1 q
    return max(np.abs(math_state(sf[0, 0]) - want_S).max(), np.abs(o[0, 0] - want_o).max())


def pin_orthonormal_overwrite(mutation=0, decay=False):
    """beta = 1 and orthonormal keys: the state maps each key exactly to its
    value, scaled by the forget gates applied after it was written."""
    rng = np.random.default_rng(4)
    dk = dv = 6
    T = 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm.T[:T][:, None, :]                       # rows orthonormal
    p = dict(q=rng.standard_normal((T, 1, dk)), k=k, v=rng.standard_normal((T, 1, dv)),
             g=(-0.4 * rng.random((T, 1)) if decay else np.zeros((T, 1))), beta=np.ones((T, 1)),
             initial_state=rng.standard_normal((1, 1, dk, dv)), cu_seqlens=np.array([0, T]))
    _, sf = run(p, mutation=mutation)
    S = math_state(sf[0, 0])
    dev = 0.0
    for t in range(T):
        after = float(np.exp(p["g"][t + 1:, 0].sum()))
        dev = max(dev, np.abs(S @ k[t, 0] - after * p["v"][t, 0]).max())
    return dev


def pin_chunked_algorithm(mutation=0):
    """The chunked WY method (explicit inverse, Gamma-extraction, merge) is a
    different algorithm reaching the same result."""
    p = problem(70, dk=7, dv=5, seed=5, gate_scale=0.4)
    o, sf = run(p, mutation=mutation)
    o2, S2 = chunked.wy_forward(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["g"][:, 0],
                                p["beta"][:, 0], math_state(p["initial_state"][0, 0]), 0.7, 16)
    return max(np.abs(o[:, 0] - o2).max(), np.abs(math_state(sf[0, 0]) - S2).max())


PINS = {
    "beta0_gate0": pin_beta0_gate0,
    "beta0_decay": pin_beta0_decay,
    "single_token": pin_single_token,
    "overwrite": pin_orthonormal_overwrite,
    "overwrite_decay": lambda m=0: pin_orthonormal_overwrite(m, decay=True),
    "chunked": pin_chunked_algorithm,
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    assert PINS[name]() < 1e-12


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5, 6, 7])
def test_planted_mistakes_are_caught(mutation):
    failing = []
    for n, f in PINS.items():
        try:
            dev = f(mutation)
        except RuntimeError:      # mutation 5 (transposed state) needs dk == dv
            continue
        if not dev < 1e-9:
            failing.append(n)
    assert failing, "mutation %d passes every pin" % mutation


# ------------------------------------------------------ algebra of the method

@pytest.mark.parametrize("C", [4, 16, 64])
@pytest.mark.parametrize("T", [1, 37, 130])
@pytest.mark.parametrize("gx,merged", [(True, True), (False, True), (True, False), (False, False)])
def test_chunked_forms_match_recurrence(C, T, gx, merged):
    p = problem(T, dk=8, dv=6, seed=T + C, gate_scale=0.5)
    o, sf = run(p)
    o2, S2 = chunked.wy_forward(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["g"][:, 0],
                                p["beta"][:, 0], math_state(p["initial_state"][0, 0]), 0.7, C,
                                gamma_extraction=gx, merged=merged)
    assert np.abs(o[:, 0] - o2).max() < 1e-12
    assert np.abs(math_state(sf[0, 0]) - S2).max() < 1e-12


def test_gamma_extraction_identity():
    """(I + A)^{-1} = Gamma ⊙ (I + A')^{-1} (Gamma-extraction paragraph)."""
    rng = np.random.default_rng(7)
    L, dk = 64, 16
    K = rng.standard_normal((L, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    b = rng.random(L)
    G = np.cumsum(-0.3 * rng.random(L))
    full = chunked.chunk_inverse(K, b, G)
    gam = chunked._gamma_matrix(G)
    assert np.abs(full - gam * chunked.chunk_inverse(K, b)).max() < 1e-12
    # and the Gamma-free inverse really is the inverse of I + A'
    Tp = chunked.chunk_inverse(K, b)
    assert np.abs(Tp @ (np.eye(L) + b[:, None] * np.tril(K @ K.T, -1)) - np.eye(L)).max() < 1e-12


def test_correction_matrix_is_recurrence_from_identity():
    """M (difference paragraph) is the product of alpha (I - beta k k^T); it is
    also what the recurrence gives with v = 0 started from S = I, and the chunk
    map is affine: S_T(S0) = S0 M + S_T(0)."""
    p = problem(45, dk=6, dv=5, seed=8, gate_scale=0.3)
    T, dk = 45, 6
    M = chunked.correction_product(p["k"][:, 0], p["g"][:, 0], p["beta"][:, 0])
    pm = dict(p, v=np.zeros((T, 1, dk)), initial_state=np.eye(dk)[None, None].transpose(0, 1, 3, 2))
    _, sfm = run(pm)
    assert np.abs(math_state(sfm[0, 0]) - M).max() < 1e-12
    _, sf = run(p)
    _, sf0 = run(dict(p, initial_state=None))
    S0 = math_state(p["initial_state"][0, 0])
    assert np.abs(math_state(sf[0, 0]) - (S0 @ M + math_state(sf0[0, 0]))).max() < 1e-12


@pytest.mark.parametrize("L", [1, 2, 3, 5])
def test_sequence_parallel_matches(L):
    p = problem(330, dk=8, dv=6, seed=9, gate_scale=0.05)
    o, sf = run(p)
    o2, S2 = chunked.cp_forward(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["g"][:, 0],
                                p["beta"][:, 0], math_state(p["initial_state"][0, 0]), 0.7, 16, L)
    assert np.abs(o[:, 0] - o2).max() < 1e-11
    assert np.abs(math_state(sf[0, 0]) - S2).max() < 1e-11


def test_sequence_parallel_alpha_one():
    p = problem(300, dk=8, dv=6, seed=10)
    p["g"][:] = 0.0
    o, sf = run(p)
    o2, S2 = chunked.cp_forward(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["g"][:, 0],
                                p["beta"][:, 0], math_state(p["initial_state"][0, 0]), 0.7, 16, 3)
    assert np.abs(o[:, 0] - o2).max() < 1e-11
    assert np.abs(math_state(sf[0, 0]) - S2).max() < 1e-11


def test_resume_equals_one_call():
    """Chunked prefill continues across calls through initial/final state."""
    p = problem(150, H=2, dk=8, dv=6, seed=11)
    o, sf = run(p)
    a = {k: (v[:61] if k in ("q", "k", "v", "g", "beta") else v) for k, v in p.items()}
    a["cu_seqlens"] = np.array([0, 61])
    oa, sfa = run(a)
    b = {k: (v[61:] if k in ("q", "k", "v", "g", "beta") else v) for k, v in p.items()}
    b["cu_seqlens"] = np.array([0, 89])
    b["initial_state"] = sfa
    ob, sfb = run(b)
    assert np.abs(np.concatenate([oa, ob]) - o).max() < 1e-12
    assert np.abs(sfb - sf).max() < 1e-12


def test_decay_bound():
    """The sliding-window paragraph: an old state's influence decays at least
    geometrically, ||S_T(S0 + d) - S_T(S0)|| <= exp(sum g) ||d||."""
    p = problem(200, dk=8, dv=6, seed=12, gate_scale=0.05)
    _, sf = run(p)
    rng = np.random.default_rng(13)
    d = rng.standard_normal(p["initial_state"].shape)
    _, sf2 = run(dict(p, initial_state=p["initial_state"] + d))
    lhs = np.linalg.norm(math_state((sf2 - sf)[0, 0]), 2)
    rhs = math.exp(p["g"][:, 0].sum()) * np.linalg.norm(math_state(d[0, 0]), 2)
    assert lhs <= rhs * (1 + 1e-9)
    # and with alpha == 1 the bound is 1 (no growth)
    p["g"][:] = 0
    _, sfa = run(p)
    _, sfb = run(dict(p, initial_state=p["initial_state"] + d))
    assert np.linalg.norm(math_state((sfb - sfa)[0, 0]), 2) <= np.linalg.norm(math_state(d[0, 0]), 2) * (1 + 1e-9)


@pytest.mark.parametrize("ln_eps", [-4.0, -8.0, -16.0])
def test_sliding_restart_error_bound(ln_eps):
    p = problem(640, dk=8, dv=6, seed=14, gate_scale=0.2)
    o, sf = run(p)
    o2, S2 = chunked.sliding_forward(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], p["g"][:, 0],
                                     p["beta"][:, 0], math_state(p["initial_state"][0, 0]), 0.7, 16, 4,
                                     ln_eps)
    # state norms along the way bound the restart error
    smax = 0.0
    for t in range(0, 641, 16):
        _, st = run(dict(p, q=p["q"][:t], k=p["k"][:t], v=p["v"][:t], g=p["g"][:t], beta=p["beta"][:t],
                         cu_seqlens=np.array([0, t])))
        smax = max(smax, np.linalg.norm(math_state(st[0, 0]), 2))
    eps = math.exp(ln_eps)
    assert np.linalg.norm(math_state(sf[0, 0]) - S2, 2) <= eps * smax * (1 + 1e-6)
    qn = np.linalg.norm(p["q"][:, 0], axis=1).max()
    assert np.abs(o[:, 0] - o2).max() <= 0.7 * qn * eps * smax * (1 + 1e-6)
    if ln_eps <= -16.0:
        assert np.abs(o[:, 0] - o2).max() < 1e-6


def test_varlen_equals_separate_calls():
    p = problem(0, H=2, dk=6, dv=5, seed=15, lens=[5, 64, 1, 70])
    o, sf = run(p)
    cu = p["cu_seqlens"]
    for n in range(4):
        sl = slice(cu[n], cu[n + 1])
        one = dict(q=p["q"][sl], k=p["k"][sl], v=p["v"][sl], g=p["g"][sl], beta=p["beta"][sl],
                   initial_state=p["initial_state"][n:n + 1], cu_seqlens=np.array([0, cu[n + 1] - cu[n]]))
        o1, sf1 = run(one)
        assert np.abs(o1 - o[sl]).max() < 1e-13
        assert np.abs(sf1 - sf[n:n + 1]).max() < 1e-13


def test_batched_layout_equals_packed():
    p = problem(0, H=3, dk=6, dv=5, seed=16, lens=[40, 40])
    o, sf = run(p)
    B = dict(q=p["q"].reshape(2, 40, 3, 6), k=p["k"].reshape(2, 40, 3, 6), v=p["v"].reshape(2, 40, 3, 5),
             g=p["g"].reshape(2, 40, 3), beta=p["beta"].reshape(2, 40, 3),
             initial_state=p["initial_state"], cu_seqlens=None)
    ob, sfb = run(B)
    assert np.abs(ob - o).max() == 0 and np.abs(sfb - sf).max() == 0


def test_subset_selection_is_exact():
    p = problem(0, H=3, dk=6, dv=5, seed=17, lens=[20, 33, 9])
    o, sf = run(p)
    o2, sf2 = run(p, seqs=[1, 2], heads=[2, 0], rows=[4, 1])
    cu = p["cu_seqlens"]
    sel = np.concatenate([np.arange(cu[1], cu[2]), np.arange(cu[2], cu[3])])
    assert np.abs(o2 - o[sel][:, [2, 0]][:, :, [4, 1]]).max() == 0
    assert np.abs(sf2 - sf[[1, 2]][:, [2, 0]][..., [4, 1]]).max() == 0


def test_threads_do_not_change_results():
    p = problem(0, H=2, dk=6, dv=5, seed=18, lens=[50, 17])
    o1, s1 = run(p, threads=1)
    o2, s2 = run(p, threads=3, row_block=2)
    assert np.abs(o1 - o2).max() == 0 and np.abs(s1 - s2).max() == 0


def test_linear_in_values_and_state():
    p = problem(90, H=1, dk=6, dv=5, seed=19)
    r = np.random.default_rng(20)
    p2 = dict(p, v=r.standard_normal(p["v"].shape), initial_state=r.standard_normal(p["initial_state"].shape))
    mix = dict(p, v=2.0 * p["v"] - 3.0 * p2["v"], initial_state=2.0 * p["initial_state"] - 3.0 * p2["initial_state"])
    o1, s1 = run(p)
    o2, s2 = run(p2)
    om, sm = run(mix)
    assert np.abs(om - (2 * o1 - 3 * o2)).max() < 1e-12
    assert np.abs(sm - (2 * s1 - 3 * s2)).max() < 1e-12


# ----------------------------------------------------------- gate quantities

def test_gate_cumsum_and_totals_closed_form():
    cu = np.array([0, 100, 101, 230])
    g = np.full((230, 2), -0.25)
    G = gate.chunk_local_cumsum(g, cu, 64)
    for n, t0, L in gate.chunk_table(cu, 64):
        assert np.allclose(G[t0:t0 + L, 0], -0.25 * np.arange(1, L + 1))
    tot = gate.chunk_totals(g, cu, 64)
    assert [round(x, 9) for x in tot[:, 1]] == [-16.0, -9.0, -0.25, -16.0, -16.0, -0.25]


def test_head_flags_and_lookback():
    cu = np.array([0, 10, 20])
    g = np.zeros((20, 3))
    g[3, 1] = -1e-30
    g[15, 2] = -0.5
    assert gate.head_flags(g, cu).tolist() == [[0, 1, 0], [0, 0, 1]]
    tot = np.array([-1.0, -2.0, -4.0, -8.0])
    assert gate.lookback_chunks(tot, 4, -7.0) == 1
    assert gate.lookback_chunks(tot, 4, -12.0) == 2
    assert gate.lookback_chunks(tot, 3, -100.0) == 3   # reaches the sequence start
    assert gate.lookback_chunks(tot, 0, -1.0) == 0


def test_inverse_rows():
    p = problem(0, H=2, dk=8, dv=4, seed=21, lens=[70, 5])
    Tp = chunked.inverse_rows(p["k"], p["beta"], p["cu_seqlens"], 64)
    for n, t0, L in gate.chunk_table(p["cu_seqlens"], 64):
        for h in range(2):
            K = p["k"][t0:t0 + L, h]
            A = p["beta"][t0:t0 + L, h][:, None] * np.tril(K @ K.T, -1)
            X = Tp[t0:t0 + L, h, :L]
            assert np.abs(X @ (np.eye(L) + A) - np.eye(L)).max() < 1e-12
            assert np.allclose(np.triu(X, 1), 0) and np.allclose(np.diag(X), 1)
    zb = chunked.inverse_rows(p["k"], np.zeros_like(p["beta"]), p["cu_seqlens"], 64)
    assert np.allclose(zb[:64, :, :64], np.eye(64)[:, None, :])


# ------------------------------------------------------------- golden fixture

def test_golden_small_case():
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    with open(os.path.join(GOLDEN, "oracle_small.json")) as f:
        fx = json.load(f)
    inp = {k: np.array(v, dtype=np.float64) for k, v in fx["inputs"].items()}
    o, sf = oracle.gdn_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                 inp["initial_state"], np.array(fx["cu_seqlens"]), scale=fx["scale"])
    assert np.abs(o - np.array(fx["o"])).max() < 1e-13
    assert np.abs(sf - np.array(fx["final_state"])).max() < 1e-13
