"""Pins for the CPU oracle against what the pages and the mathematics fix.

The pages ("Log-Linear Attention", gist.science summaries of arXiv 2506.04761,
Portuguese and French §2) print no worked numeric example. The oracle is pinned
instead by: the Fenwick bucket structure (sizes 1, 2, 4, ...; O(log T) buckets;
the level counts 7/12/14/17 of the benchmark shapes), agreement of two forms
written independently (explicit mask vs token recurrence), the special cases
that collapse to textbook operators (gated linear attention / Mamba-2 when
lambda is level-independent; causal linear attention when a = 1 and
lambda = 1), one-hot lambda isolating a single bucket, linearity, and
hand-worked values in tests/golden/.
"""
import os

import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, B, H, T, dk, dv, L=None):
    L = inputs.num_levels(T) if L is None else L
    q = rng.standard_normal((B, H, T, dk)) / np.sqrt(dk)
    k = rng.standard_normal((B, H, T, dk)) / np.sqrt(dk)
    v = rng.standard_normal((B, H, T, dv))
    log_a = -np.logaddexp(0.0, rng.standard_normal((B, H, T)))
    lam = np.logaddexp(0.0, rng.standard_normal((B, H, T, L)))
    return q, k, v, log_a, lam


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------- Fenwick structure

def test_level_matches_xor_closed_form():
    """Fenwick bucket walk == 1 + floor(log2(t xor s)) for s < t, 0 for s == t."""
    for t in range(0, 300):
        for s in range(0, t + 1):
            want = 0 if s == t else (t ^ s).bit_length()
            assert oracle.level(t, s) == want, (t, s)
    # far positions, spot-checked
    rng = np.random.default_rng(1)
    for _ in range(2000):
        t = int(rng.integers(0, 1 << 20))
        s = int(rng.integers(0, t + 1))
        assert oracle.level(t, s) == (0 if s == t else (t ^ s).bit_length())
    assert oracle.level(3, 4) == -1


def test_bucket_sizes_are_powers_of_two_and_logarithmic():
    """For every query t the keys 0..t split into one bucket per level l with
    size 2^(l-1) (level 0 = the token itself), nonempty exactly for the set bits
    of t: popcount(t) + 1 buckets, i.e. O(log T)."""
    for t in range(0, 260):
        sizes = {}
        for s in range(t + 1):
            l = oracle.level(t, s)
            sizes[l] = sizes.get(l, 0) + 1
        assert sizes[0] == 1
        for l, n in sizes.items():
            if l > 0:
                assert n == 1 << (l - 1)
                assert (t >> (l - 1)) & 1 == 1
        assert len(sizes) == bin(t).count("1") + 1
        # buckets are contiguous, nearer keys never sit in a coarser bucket than farther ones
        levels = [oracle.level(t, s) for s in range(t, -1, -1)]
        assert all(levels[i] <= levels[i + 1] for i in range(len(levels) - 1))


@pytest.mark.parametrize("T,want", [(64, 7), (2048, 12), (8192, 14)])
def test_level_count_by_enumeration(T, want):
    """The benchmark shapes state 7/12/14 levels for T = 64/2048/8192."""
    assert oracle.num_levels(T) == want
    assert inputs.num_levels(T) == want


def test_level_count_long():
    """T = 65536 states 17 levels: the deepest pair is (T-1, 0)."""
    assert oracle.level(65535, 0) + 1 == 17
    assert inputs.num_levels(65536) == 17


# ---------------------------------------------------------------- two forms agree

@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 1, 1, 3, 2), (1, 2, 2, 4, 3), (2, 1, 3, 2, 5),
                                         (1, 1, 17, 8, 4), (1, 2, 64, 16, 16), (1, 1, 200, 4, 6),
                                         (1, 1, 513, 3, 2)])
def test_explicit_equals_recurrent(B, H, T, dk, dv):
    rng = np.random.default_rng(T * 7 + dk)
    args = _rand_problem(rng, B, H, T, dk, dv)
    e = oracle.explicit(*args)
    r = oracle.recurrent(*args)
    assert _rel(r, e) <= 1e-12


# ---------------------------------------------------------------- special cases

def test_level_independent_lambda_is_gated_linear_attention():
    """lambda_t^(l) = c_t for every l: o_t = c_t * (Mamba-2 / gated linear attention)
    o_t, computed by the textbook recurrence S_t = a_t S_{t-1} + k_t v_t^T, o_t = S_t^T q_t."""
    rng = np.random.default_rng(5)
    B, H, T, dk, dv = 1, 2, 97, 5, 3
    q, k, v, log_a, _ = _rand_problem(rng, B, H, T, dk, dv)
    c = np.exp(rng.standard_normal((B, H, T)))
    lam = np.repeat(c[..., None], inputs.num_levels(T), axis=-1)
    want = np.zeros((B, H, T, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv))
            for t in range(T):
                S = np.exp(log_a[b, h, t]) * S + np.outer(k[b, h, t], v[b, h, t])
                want[b, h, t] = c[b, h, t] * (S.T @ q[b, h, t])
    for form in (oracle.explicit, oracle.recurrent):
        assert _rel(form(q, k, v, log_a, lam), want) <= 1e-12


def test_unit_decay_unit_lambda_is_causal_linear_attention():
    """a = 1 and lambda = 1: o = tril(Q K^T) V."""
    rng = np.random.default_rng(6)
    B, H, T, dk, dv = 2, 1, 70, 6, 4
    q, k, v, _, _ = _rand_problem(rng, B, H, T, dk, dv)
    log_a = np.zeros((B, H, T))
    lam = np.ones((B, H, T, inputs.num_levels(T)))
    want = np.tril(q @ np.swapaxes(k, -1, -2)) @ v
    for form in (oracle.explicit, oracle.recurrent):
        assert _rel(form(q, k, v, log_a, lam), want) <= 1e-12


@pytest.mark.parametrize("lvl", [0, 1, 2, 3, 5])
def test_one_hot_lambda_isolates_one_bucket(lvl):
    """lambda one-hot on level l: o_t sums exactly the keys s with t xor s in [2^(l-1), 2^l)
    (s = t for l = 0), each decayed by prod_{r in (s,t]} a_r."""
    rng = np.random.default_rng(10 + lvl)
    B, H, T, dk, dv = 1, 1, 45, 3, 2
    q, k, v, log_a, _ = _rand_problem(rng, B, H, T, dk, dv)
    L = inputs.num_levels(T)
    lam = np.zeros((B, H, T, L))
    lam[..., lvl] = 1.0
    a = np.exp(log_a[0, 0])
    want = np.zeros((B, H, T, dv))
    for t in range(T):
        for s in range(t + 1):
            in_bucket = (s == t) if lvl == 0 else ((1 << (lvl - 1)) <= (t ^ s) < (1 << lvl))
            if in_bucket:
                decay = np.prod(a[s + 1:t + 1])
                want[0, 0, t] += decay * (q[0, 0, t] @ k[0, 0, s]) * v[0, 0, s]
    for form in (oracle.explicit, oracle.recurrent):
        got = form(q, k, v, log_a, lam)
        assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_single_token():
    rng = np.random.default_rng(7)
    q, k, v, log_a, lam = _rand_problem(rng, 1, 1, 1, 4, 3)
    want = lam[0, 0, 0, 0] * (q[0, 0, 0] @ k[0, 0, 0]) * v[0, 0, 0]
    for form in (oracle.explicit, oracle.recurrent):
        assert np.allclose(form(q, k, v, log_a, lam)[0, 0, 0], want, rtol=1e-14, atol=0)


def test_linearity_in_v_and_lambda():
    rng = np.random.default_rng(8)
    q, k, v, log_a, lam = _rand_problem(rng, 1, 1, 33, 4, 3)
    _, _, v2, _, lam2 = _rand_problem(rng, 1, 1, 33, 4, 3)
    f = oracle.recurrent
    assert _rel(f(q, k, 2.0 * v - 3.0 * v2, log_a, lam),
                2.0 * f(q, k, v, log_a, lam) - 3.0 * f(q, k, v2, log_a, lam)) <= 1e-12
    assert _rel(f(q, k, v, log_a, lam + lam2),
                f(q, k, v, log_a, lam) + f(q, k, v, log_a, lam2)) <= 1e-12


def test_hand_worked_examples():
    rows = []
    with open(os.path.join(GOLDEN, "fenwick_hand_examples.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    assert len(rows) == 6
    for name, T, t, vs, expected in rows:
        T, t, expected = int(T), int(t), float(expected)
        vals = np.array([float(x) for x in vs.split(",")]).reshape(1, 1, T, 1)
        ones = np.ones((1, 1, T, 1))
        log_a = np.full((1, 1, T), -np.log(2.0))
        L = inputs.num_levels(T)
        lam = np.broadcast_to(10.0 ** np.arange(L), (1, 1, T, L)).copy()
        for form in (oracle.explicit, oracle.recurrent):
            got = form(ones, ones, vals, log_a, lam)[0, 0, t, 0]
            assert abs(got - expected) <= 1e-12 * expected, (name, t, got, expected)


# ---------------------------------------------------------------- decode step

def test_decode_steps_reproduce_recurrent_form():
    """Stepping the batched decode from empty states over a sequence gives the
    recurrent form's rows, with per-sequence positions offset."""
    rng = np.random.default_rng(9)
    B, H, T, dk, dv = 2, 2, 40, 4, 3
    q, k, v, log_a, lam = _rand_problem(rng, B, H, T, dk, dv, L=7)
    want = oracle.recurrent(q, k, v, log_a, lam[..., :inputs.num_levels(T)])
    Lmax = 7
    states = np.zeros((B, H, Lmax, dk, dv))
    for t in range(T):
        out = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], log_a[:, :, t],
                                 lam[:, :, t, :Lmax], states, np.full(B, t))
        assert _rel(out, want[:, :, t]) <= 1e-12


def test_decode_rejects_too_few_levels():
    B, H, dk, dv, Lmax = 1, 1, 2, 2, 3
    z = np.zeros
    with pytest.raises(ValueError):
        oracle.decode_step(z((B, H, dk)), z((B, H, dk)), z((B, H, dv)), z((B, H)), z((B, H, Lmax)),
                           z((B, H, Lmax, dk, dv)), np.array([4]))


def test_explicit_rows_matches_full_explicit():
    rng = np.random.default_rng(11)
    q, k, v, log_a, lam = _rand_problem(rng, 2, 2, 70, 5, 3)
    full = oracle.explicit(q, k, v, log_a, lam)
    rows = [0, 1, 31, 32, 69]
    got = oracle.explicit_rows(q, k, v, log_a, lam, 1, 0, rows)
    assert np.array_equal(got, full[1, 0, rows])
