"""Pins of the log-linear Gated DeltaNet oracle against what the pages and the mathematics fix.

The pages name the variant (pt §2 "Generalizacao", fr §3 "Etudes de Cas": the hierarchical mask
applied to Gated DeltaNet) and its two forms (pt §2 "Forma Recorrente e Paralela"); Gated DeltaNet
itself is the published gated delta rule, S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T.
Each pin would catch a plausible mistake: a wrong transition sign or a missing beta (hand-worked
values), a transposed or reordered transition product (two independent forms), a wrong hierarchy
(reduction to the pinned Mamba-2 oracle and to the plain Gated DeltaNet recurrence).
"""
import math
import os

import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gdn_hand_examples.txt")


def _problem(rng, B, H, T, dk, dv, L=None, unit_keys=True):
    L = inputs.num_levels(T) if L is None else L
    q = rng.standard_normal((B, H, T, dk)) / np.sqrt(dk)
    k = rng.standard_normal((B, H, T, dk))
    k = k / np.linalg.norm(k, axis=-1, keepdims=True) if unit_keys else k / np.sqrt(dk)
    v = rng.standard_normal((B, H, T, dv))
    log_a = -np.logaddexp(0.0, rng.standard_normal((B, H, T)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T))))
    lam = np.logaddexp(0.0, rng.standard_normal((B, H, T, L)))
    return q, k, v, log_a, beta, lam


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _golden_inputs(name):
    if name == "G1":
        T = 4
        q = np.ones((1, 1, T, 1))
        k = np.ones((1, 1, T, 1))
        v = np.array([1.0, 2.0, 4.0, 8.0]).reshape(1, 1, T, 1)
        log_a = np.zeros((1, 1, T))
        beta = np.full((1, 1, T), 0.5)
        L = inputs.num_levels(T)
        lam = np.tile(10.0 ** np.arange(L), (1, 1, T, 1))
    elif name == "G2":
        q = np.array([[1.0, 0.0], [1.0, 1.0]]).reshape(1, 1, 2, 2)
        k = np.array([[1.0, 0.0], [1.0, 0.0]]).reshape(1, 1, 2, 2)
        v = np.array([3.0, 5.0]).reshape(1, 1, 2, 1)
        log_a = np.zeros((1, 1, 2))
        beta = np.ones((1, 1, 2))
        lam = np.ones((1, 1, 2, inputs.num_levels(2)))
    else:  # G3
        q = np.array([[1.0, 0.0], [1.0, 1.0]]).reshape(1, 1, 2, 2)
        k = np.array([[1.0, 0.0], [0.0, 1.0]]).reshape(1, 1, 2, 2)
        v = np.array([3.0, 5.0]).reshape(1, 1, 2, 1)
        log_a = np.array([0.0, -math.log(2.0)]).reshape(1, 1, 2)
        beta = np.ones((1, 1, 2))
        lam = np.array([[1.0, 10.0], [1.0, 10.0]]).reshape(1, 1, 2, 2)
    return q, k, v, log_a, beta, lam


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, t, want = line.split()
        rows.append((name, int(t), float(want)))
    return rows


@pytest.mark.parametrize("name,t,want", _golden_rows())
@pytest.mark.parametrize("form", ["explicit", "recurrent"])
def test_gdn_hand_worked_values(name, t, want, form):
    args = _golden_inputs(name)
    f = oracle.gdn_explicit if form == "explicit" else oracle.gdn_recurrent
    got = f(*args)[0, 0, t, 0]
    assert abs(got - want) <= 1e-12 * max(1.0, abs(want)), (name, t, got, want)


@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 1, 1, 3, 2), (1, 2, 37, 5, 3), (2, 1, 128, 8, 4), (1, 1, 301, 6, 5),
                                         (1, 1, 64, 16, 16)])
def test_gdn_explicit_equals_recurrent(B, H, T, dk, dv):
    """The attention-matrix walk and the bucket recurrence are independent computations of the
    same operator (the recurrence never evaluates l(t,s) or a pairwise coefficient)."""
    rng = np.random.default_rng(T * 7 + dk)
    args = _problem(rng, B, H, T, dk, dv)
    assert _rel(oracle.gdn_explicit(*args), oracle.gdn_recurrent(*args)) <= 1e-12


def test_gdn_non_unit_keys_two_forms_agree():
    rng = np.random.default_rng(3)
    args = _problem(rng, 1, 1, 90, 7, 3, unit_keys=False)
    assert _rel(oracle.gdn_explicit(*args), oracle.gdn_recurrent(*args)) <= 1e-12


def test_gdn_equal_lambda_is_lambda_times_textbook_gated_deltanet():
    """lambda_t^(l) = lambda_t for every level: o_t = lambda_t * (Gated DeltaNet output), by the plain
    recurrence S = alpha (I - beta k k^T) S + beta k v^T, o = S^T q, written here in numpy."""
    rng = np.random.default_rng(5)
    B, H, T, dk, dv = 1, 2, 70, 6, 4
    q, k, v, log_a, beta, lam = _problem(rng, B, H, T, dk, dv)
    lam_t = np.logaddexp(0.0, rng.standard_normal((B, H, T)))
    lam = np.repeat(lam_t[..., None], lam.shape[-1], axis=-1)
    got = oracle.gdn_explicit(q, k, v, log_a, beta, lam)
    want = np.zeros_like(got)
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv))
            for t in range(T):
                kt = k[b, h, t]
                A = math.exp(log_a[b, h, t]) * (np.eye(dk) - beta[b, h, t] * np.outer(kt, kt))
                S = A @ S + beta[b, h, t] * np.outer(kt, v[b, h, t])
                want[b, h, t] = lam_t[b, h, t] * (S.T @ q[b, h, t])
    assert _rel(got, want) <= 1e-12


def test_gdn_orthonormal_keys_reduce_to_log_linear_mamba2():
    """Mutually orthogonal unit keys (T <= dk): every transition acts on an earlier key as the scalar
    alpha_r, so A[t,s] = beta_s prod_{r=s+1..t} alpha_r (q_t . k_s), which is the pinned log-linear
    Mamba-2 oracle with values beta_s v_s."""
    rng = np.random.default_rng(9)
    T, dk, dv = 24, 32, 3
    q, _, v, log_a, beta, lam = _problem(rng, 1, 1, T, dk, dv)
    basis, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = basis[:T].reshape(1, 1, T, dk)
    got = oracle.gdn_explicit(q, k, v, log_a, beta, lam)
    want = oracle.explicit(q, k, v * beta[..., None], log_a, lam)
    assert _rel(got, want) <= 1e-12
    assert _rel(oracle.gdn_recurrent(q, k, v, log_a, beta, lam), want) <= 1e-12


def test_gdn_beta_zero_writes_nothing():
    rng = np.random.default_rng(10)
    q, k, v, log_a, beta, lam = _problem(rng, 1, 1, 33, 4, 2)
    beta[:] = 0.0
    assert np.all(oracle.gdn_explicit(q, k, v, log_a, beta, lam) == 0.0)
    assert np.all(oracle.gdn_recurrent(q, k, v, log_a, beta, lam) == 0.0)


def test_gdn_single_token():
    rng = np.random.default_rng(11)
    q, k, v, log_a, beta, lam = _problem(rng, 1, 1, 1, 5, 3)
    want = lam[0, 0, 0, 0] * beta[0, 0, 0] * float(q[0, 0, 0] @ k[0, 0, 0]) * v[0, 0, 0]
    assert np.allclose(oracle.gdn_explicit(q, k, v, log_a, beta, lam)[0, 0, 0], want, rtol=1e-14, atol=0)


def test_gdn_linear_in_v_and_lambda():
    rng = np.random.default_rng(12)
    q, k, v, log_a, beta, lam = _problem(rng, 1, 1, 45, 4, 3)
    v2 = rng.standard_normal(v.shape)
    lam2 = np.logaddexp(0.0, rng.standard_normal(lam.shape))
    f = oracle.gdn_explicit
    assert _rel(f(q, k, v + 2 * v2, log_a, beta, lam),
                f(q, k, v, log_a, beta, lam) + 2 * f(q, k, v2, log_a, beta, lam)) <= 1e-12
    assert _rel(f(q, k, v, log_a, beta, lam + lam2),
                f(q, k, v, log_a, beta, lam) + f(q, k, v, log_a, beta, lam2)) <= 1e-12


def test_gdn_decode_steps_reproduce_recurrent_rows():
    """Stepping the decode oracle token by token from empty states gives the recurrent form's rows."""
    rng = np.random.default_rng(13)
    B, H, T, dk, dv = 2, 2, 40, 4, 3
    q, k, v, log_a, beta, lam = _problem(rng, B, H, T, dk, dv)
    ref = oracle.gdn_recurrent(q, k, v, log_a, beta, lam)
    Lmax = lam.shape[-1]
    states = np.zeros((B, H, Lmax, dk, dv))
    for t in range(T):
        o = oracle.gdn_decode_step(q[:, :, t], k[:, :, t], v[:, :, t], log_a[:, :, t], beta[:, :, t],
                                   lam[:, :, t], states, np.full(B, t))
        assert _rel(o, ref[:, :, t]) <= 1e-12


def test_gdn_rows_form_equals_full_explicit():
    rng = np.random.default_rng(14)
    q, k, v, log_a, beta, lam = _problem(rng, 2, 2, 77, 5, 3)
    full = oracle.gdn_explicit(q, k, v, log_a, beta, lam)
    rows = [0, 1, 31, 32, 63, 76]
    got = oracle.gdn_explicit_rows(q, k, v, log_a, beta, lam, 1, 0, rows)
    assert np.max(np.abs(got - full[1, 0, rows])) == 0.0
