"""Pins of the oracle's backward pass (gradients of L = sum(dout * O)).

The backward oracle is checked against things other than itself:
  * central finite differences of the forward oracle (already pinned by its own
    tests), every coordinate of every input on tiny problems;
  * a = 1, lambda = 1: causal linear attention, whose gradients are the
    textbook matrix formulas (numpy, independent of the oracle's loops);
  * T = 1 closed form; linearity in dout.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _problem(rng, B, H, T, dk, dv):
    L = oracle.num_levels(T)
    q = rng.normal(size=(B, H, T, dk))
    k = rng.normal(size=(B, H, T, dk))
    v = rng.normal(size=(B, H, T, dv))
    log_a = -np.log1p(np.exp(rng.normal(size=(B, H, T))))
    lam = np.log1p(np.exp(rng.normal(size=(B, H, T, L))))
    dout = rng.normal(size=(B, H, T, dv))
    return q, k, v, log_a, lam, dout


def _loss(args, dout):
    return float((oracle.explicit(*args) * dout).sum())


@pytest.mark.parametrize("B,H,T,dk,dv,seed", [(1, 1, 9, 3, 2, 0), (1, 2, 17, 2, 3, 1), (2, 1, 6, 4, 1, 2)])
def test_backward_matches_finite_differences(B, H, T, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q, k, v, log_a, lam, dout = _problem(rng, B, H, T, dk, dv)
    args = [q, k, v, log_a, lam]
    grads = oracle.backward(q, k, v, log_a, lam, dout)
    h = 1e-6
    for i, (x, g) in enumerate(zip(args, grads)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            ap = list(args); ap[i] = xp
            am = list(args); am[i] = xm
            num[idx] = (_loss(ap, dout) - _loss(am, dout)) / (2 * h)
        scale = max(np.abs(num).max(), 1e-12)
        assert np.abs(num - g).max() / scale < 1e-7, ["dq", "dk", "dv", "dlog_a", "dlambda"][i]


def test_backward_linear_attention_closed_form():
    """a = 1 and lambda = 1: O = tril(Q K^T) V, gradients by matrix algebra."""
    rng = np.random.default_rng(3)
    B, H, T, dk, dv = 1, 2, 40, 5, 3
    q, k, v, _, _, dout = _problem(rng, B, H, T, dk, dv)
    L = oracle.num_levels(T)
    log_a = np.zeros((B, H, T))
    lam = np.ones((B, H, T, L))
    dq, dk_, dv_, dla, dlam = oracle.backward(q, k, v, log_a, lam, dout)
    lv = np.array([[oracle.level(t, s) for s in range(T)] for t in range(T)])
    for h in range(H):
        Q, K, V, G = q[0, h], k[0, h], v[0, h], dout[0, h]
        mask = np.tril(np.ones((T, T)))
        A = (Q @ K.T) * mask
        dA = (G @ V.T) * mask
        np.testing.assert_allclose(dv_[0, h], A.T @ G, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dq[0, h], dA @ K, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dk_[0, h], dA.T @ Q, rtol=1e-10, atol=1e-10)
        E = A * (G @ V.T)
        want_la = np.array([E[r:, :r].sum() for r in range(T)])
        np.testing.assert_allclose(dla[0, h], want_la, rtol=1e-9, atol=1e-9)
        want_lam = np.zeros((T, L))
        for t in range(T):
            for s in range(t + 1):
                want_lam[t, lv[t, s]] += E[t, s]
        np.testing.assert_allclose(dlam[0, h], want_lam, rtol=1e-10, atol=1e-10)


def test_backward_single_token():
    rng = np.random.default_rng(4)
    q, k, v, log_a, lam, dout = _problem(rng, 1, 1, 1, 4, 3)
    dq, dk_, dv_, dla, dlam = oracle.backward(q, k, v, log_a, lam, dout)
    l0 = lam[0, 0, 0, 0]
    qk = q[0, 0, 0] @ k[0, 0, 0]
    gv = dout[0, 0, 0] @ v[0, 0, 0]
    np.testing.assert_allclose(dq[0, 0, 0], l0 * gv * k[0, 0, 0], rtol=1e-12)
    np.testing.assert_allclose(dk_[0, 0, 0], l0 * gv * q[0, 0, 0], rtol=1e-12)
    np.testing.assert_allclose(dv_[0, 0, 0], l0 * qk * dout[0, 0, 0], rtol=1e-12)
    assert dla[0, 0, 0] == 0.0
    np.testing.assert_allclose(dlam[0, 0, 0, 0], qk * gv, rtol=1e-12)


def test_backward_linear_in_dout():
    rng = np.random.default_rng(5)
    q, k, v, log_a, lam, dout = _problem(rng, 1, 1, 33, 3, 2)
    g1 = oracle.backward(q, k, v, log_a, lam, dout)
    g2 = oracle.backward(q, k, v, log_a, lam, -2.5 * dout)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(b, -2.5 * a, rtol=1e-12, atol=1e-14)


def test_backward_rows_match_full_backward():
    """The per-position backward (used for spot checks of long sequences) against the
    full backward: dq/dk/dv/dlambda rows, and dcum_x = dlog_a_x - dlog_a_{x+1}."""
    rng = np.random.default_rng(6)
    B, H, T, dk, dv = 2, 2, 70, 5, 4
    q, k, v, log_a, lam, dout = _problem(rng, B, H, T, dk, dv)
    dq, dk_, dv_, dla, dlam = oracle.backward(q, k, v, log_a, lam, dout)
    rows = [0, 1, 31, 32, 63, 69]
    for b, h in ((0, 1), (1, 0)):
        rq, rk, rv, rl, rc = oracle.backward_rows(q, k, v, log_a, lam, dout, b, h, rows)
        np.testing.assert_allclose(rq, dq[b, h, rows], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(rk, dk_[b, h, rows], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(rv, dv_[b, h, rows], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(rl, dlam[b, h, rows], rtol=1e-11, atol=1e-12)
        nxt = np.append(dla[b, h], 0.0)
        np.testing.assert_allclose(rc, nxt[rows] - nxt[np.array(rows) + 1], rtol=1e-9, atol=1e-10)
