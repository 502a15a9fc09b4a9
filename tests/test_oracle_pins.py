"""Pins of the float64 oracle against what the pages and mathematics fix.

Each test targets a mistake that would otherwise go unnoticed in the oracle
(a dropped term, a transposed operand, a wrong exponent or sign); none of them
re-types the function it checks.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "shampoo_hand_example.json")


@pytest.fixture(scope="module")
def hand():
    with open(GOLD) as f:
        return json.load(f)


def _sv(X):
    return np.sort(np.linalg.svd(np.asarray(X, dtype=np.float64), compute_uv=False))[::-1]


# --------------------------------------------------------------- hand example

def test_hand_example_factors(hand):
    """L = G G^T printed on the page; the factor EMA with beta2 = 0, P = I,
    eps = 0 must give n S_a = G G^T and m S_b = G^T G."""
    G = np.array(hand["G"], dtype=np.float64)
    m, n = G.shape
    Sa = O.factor_ema(np.zeros((m, m)), G @ np.eye(n), 0.0, n, 0.0)
    Sb = O.factor_ema(np.zeros((n, n)), (np.eye(m) @ G).T, 0.0, m, 0.0)
    assert np.array_equal(n * Sa, np.array(hand["L_equals_GGt"], dtype=np.float64))
    # G^T G of the page's G, entry by entry
    assert np.allclose(m * Sb, [[10, 2, 3], [2, 4, 0], [3, 0, 1]], atol=1e-12)
    assert np.allclose(_sv(G), hand["singular_values_G"], atol=hand["printed_precision"])


@pytest.mark.parametrize("acc,key", [(1, "shampoo_quarter_root_step_singular_values"),
                                     (4, "shampoo_quarter_root_after_4_accumulations"),
                                     (100, "shampoo_quarter_root_after_100_accumulations")])
def test_hand_example_quarter_root(hand, acc, key):
    """sigma(L^-1/4 G R^-1/4) = 1, 1 for one gradient, 0.5 after four identical
    accumulations and 0.1 after a hundred (R is rank 2: pseudo-inverse)."""
    G = np.array(hand["G"], dtype=np.float64)
    L, R = acc * (G @ G.T), acc * (G.T @ G)
    step = O.sym_power(L, -0.25, rcond=1e-12) @ G @ O.sym_power(R, -0.25, rcond=1e-12)
    assert np.allclose(_sv(step)[:2], hand[key], atol=hand["printed_precision"])


def test_problem14_half_roots(hand):
    """Problem 14: with -1/2 on both sides the step's singular values are
    0.527 / 0.296, and 0.0527 / 0.0296 for 10 G; with -1/4, 10 G keeps 1, 1."""
    G = np.array(hand["G"], dtype=np.float64)
    tol = hand["printed_precision"]
    for c, key in [(1.0, "problem14_half_root_G"), (10.0, "problem14_half_root_10G")]:
        Gc = c * G
        L, R = Gc @ Gc.T, Gc.T @ Gc
        step = O.inv_root_exact(L) @ Gc @ O.sym_power(R, -0.5, rcond=1e-12)
        want = np.array(hand[key])
        assert np.allclose(_sv(step)[:2], want, rtol=tol / want.min() * 0.6)
    G10 = 10 * G
    step = (O.sym_power(G10 @ G10.T, -0.25) @ G10
            @ O.sym_power(G10.T @ G10, -0.25, rcond=1e-12))
    assert np.allclose(_sv(step)[:2], hand["problem14_quarter_root_10G"], atol=tol)


def test_eps_regularised_rank_deficient_right_factor(hand):
    """With +eps I instead of a pseudo-inverse, G annihilates R's null
    direction, so the -1/2 step keeps Problem 14's singular values."""
    G = np.array(hand["G"], dtype=np.float64)
    R = G.T @ G + 1e-9 * np.eye(3)
    step = O.inv_root_exact(G @ G.T) @ G @ O.inv_root_exact(R)
    assert np.allclose(_sv(step)[:2], [0.527, 0.296], atol=1e-3)


# --------------------------------------------------------------- schedule

def test_schedule_textbook_special_case():
    """On [1, 1] the minimax cubic is the textbook Newton-Schulz step."""
    (a, b, _l, _u), = O.cans_schedule(1, lo=1.0, hi=1.0)
    assert abs(a - 1.5) < 1e-15 and abs(b + 0.5) < 1e-15


def test_schedule_is_minimax_by_brute_force():
    """For each step, no (a, b) on a fine grid around the schedule's pair has
    a smaller worst error max|1 - q(s)| on [l, u], and the error
    equioscillates at l, s* and u."""
    sch = O.cans_schedule(10, 1e-3)
    for (a, b, l, u) in sch[:6]:
        s = np.concatenate([np.linspace(l, u, 20001), np.geomspace(l, u, 20001)])
        err = lambda A, B: np.max(np.abs(1 - (A * s + B * s ** 3)))  # noqa: E731
        e0 = err(a, b)
        for da in np.linspace(-0.02, 0.02, 21):
            for db in np.linspace(-0.02, 0.02, 21):
                if da == 0 and db == 0:
                    continue
                assert err(a * (1 + da), b * (1 + db)) >= e0 - 1e-12
        s_star = math.sqrt(-a / (3 * b))
        e_l, e_s, e_u = 1 - (a * l + b * l ** 3), 1 - (a * s_star + b * s_star ** 3), \
            1 - (a * u + b * u ** 3)
        assert abs(e_l - e_u) < 1e-9 and abs(e_l + e_s) < 1e-9


def test_schedule_convergence_window():
    """After ten steps from [1e-3, 1] every sqrt-eigenvalue lies within 1e-5
    of 1 (scalar map checked on a dense grid, independent of the interval
    bookkeeping)."""
    sch = O.cans_schedule(10, 1e-3)
    s = np.geomspace(1e-3, 1.0, 200001)
    mu = s ** 2
    y, z = O.ns_scalar_map(mu, sch)
    assert np.max(np.abs(np.sqrt(y * z) - 1)) < 1e-5
    # z converges to mu^-1/2 with the same relative error
    assert np.max(np.abs(z * np.sqrt(mu) - 1)) < 1e-5


def test_scale_exponents_bound_z():
    """Entries of Z_k of the float64 iteration never exceed 2**z_k."""
    rng = np.random.default_rng(3)
    sch = O.cans_schedule(10, 1e-3)
    z = O.ns_exponents(sch)
    d = 24
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    S = (Q * np.geomspace(1e-6, 1, d)) @ Q.T
    cp = np.linalg.norm(S) * (1 + O.NS_MARGIN)
    Y, Z = S / cp, np.eye(d)
    for k, (a, b, _l, _u) in enumerate(sch):
        assert np.max(np.abs(Z)) <= 2.0 ** z[k]
        T = a * np.eye(d) + b * Z @ Y
        Y, Z = Y @ T, T @ Z
    assert np.max(np.abs(Z)) <= 2.0 ** z[len(sch)]


# --------------------------------------------------------------- NS chain

def _spd(d, cond, seed):
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    w = np.geomspace(1.0, cond, d)
    return (Q * w) @ Q.T


def test_matrix_iteration_equals_scalar_polynomial():
    """Coupled matrix iteration (float64) = eigen-wise scalar recursion."""
    S = _spd(40, 1e3, 1)
    sch = O.cans_schedule(10, 1e-3)
    P1, R1 = O.ns_matrix_float64(S, sch)
    P2, R2 = O.ns_exact(S, sch)
    assert O.rel_fro(P1, P2) < 1e-10 and O.rel_fro(R1, R2) < 1e-10


def test_ns_reaches_exact_root_within_schedule_bound():
    """For spectra inside the converging window the 10-step result equals
    S^-1/2 and S^1/2 (eigendecomposition) within the schedule's error."""
    sch = O.cans_schedule(10, 1e-3)
    for cond in [1.0, 1e2, 1e4]:
        S = _spd(32, cond, 2)
        P, R = O.ns_exact(S, sch)
        assert O.rel_fro(P, O.inv_root_exact(S)) < 2e-5
        assert O.rel_fro(R, O.sym_power(S, 0.5)) < 2e-5
        assert np.allclose(P @ S @ P, np.eye(32), atol=5e-5)


def test_ridge_is_root_of_shifted_matrix():
    S = _spd(20, 1e5, 4)
    rho = 1e-3
    c = np.linalg.norm(S)
    want = O.sym_power(S + rho * c * np.eye(20), -0.5)
    assert O.rel_fro(O.inv_root_exact(S, rho), want) < 1e-12
    assert O.rel_fro(O.ns_exact(S, O.cans_schedule(10, 1e-3), rho)[0], want) < 2e-5


def test_roots_for_several_ridges_from_one_decomposition():
    S = _spd(40, 1e3, 12)
    got = O.inv_roots_exact(S, [0.0, 1e-4, 1e-3])
    for P, rho in zip(got, [0.0, 1e-4, 1e-3]):
        assert O.rel_fro(P, O.inv_root_exact(S, rho)) < 1e-12


def test_replay_without_rounding_is_the_float64_iteration():
    S = _spd(48, 1e3, 5)
    sch = O.cans_schedule(10, 1e-3)
    r = O.ns_replay(S, sch, rounding=False)
    assert O.rel_fro(r["P"], O.ns_matrix_float64(S, sch)[0]) < 1e-11
    assert O.rel_fro(r["pi"] * r["P_hat"], r["P"]) < 1e-12
    rs = O.ns_replay(S, sch, rounding=False, split_iters=4)
    assert O.rel_fro(rs["P"], r["P"]) < 1e-11


def test_replay_with_binary16_rounding_is_accurate_when_well_conditioned():
    sch = O.cans_schedule(10, 1e-3)
    S = _spd(64, 10.0, 6)
    r = O.ns_replay(S, sch)
    assert 1e-6 < O.rel_fro(r["P"], O.inv_root_exact(S)) < 5e-3
    # the split mode cuts the error of an ill-conditioned factor
    S4 = _spd(64, 1e4, 7)
    e0 = O.rel_fro(O.ns_replay(S4, sch)["P"], O.inv_root_exact(S4))
    e3 = O.rel_fro(O.ns_replay(S4, sch, split_iters=3)["P"], O.inv_root_exact(S4))
    assert e3 < 1e-2 and e3 < 0.5 * e0


def test_replay_float32_accumulation_is_the_same_chain():
    """accumulate="float32" changes only the summation precision: without
    binary16 rounding it is the float64 iteration to float32 accuracy; with
    rounding it still reaches the exact root, and it moves the end-to-end
    result by a small but non-zero amount (the accumulation-order floor)."""
    sch = O.cans_schedule(10, 1e-3)
    S = _spd(96, 1e2, 9)
    r64 = O.ns_replay(S, sch, rounding=False)
    r32 = O.ns_replay(S, sch, rounding=False, accumulate="float32")
    assert O.rel_fro(r32["P"], r64["P"]) < 1e-5
    q64 = O.ns_replay(S, sch)
    q32 = O.ns_replay(S, sch, accumulate="float32")
    assert O.rel_fro(q32["P"], O.inv_root_exact(S)) < 1e-2
    assert 0.0 < O.rel_fro(q32["P"], q64["P"]) < 5e-3
    with pytest.raises(ValueError):
        O.ns_replay(S, sch, accumulate="float16")


def test_replay_iteration_matches_trace():
    sch = O.cans_schedule(10, 1e-3)
    S = _spd(32, 1e2, 8)
    r = O.ns_replay(S, sch, trace=True)
    for k in range(1, 10):
        T, Yn, Zn = O.ns_replay_iteration(k, r["Y"][k], r["Z"][k], sch)
        assert np.array_equal(T, r["T"][k])
        if k < 9:
            assert np.array_equal(Yn, r["Y"][k + 1]) and np.array_equal(Zn, r["Z"][k + 1])
        else:
            assert np.array_equal(Zn, r["P_hat"])


def test_binary16_rounding_is_round_to_nearest_even():
    one = 1.0
    assert O.f16(one + 2 ** -11) == 1.0                      # tie -> even
    assert O.f16(one + 3 * 2 ** -11) == one + 2 ** -9        # tie -> even
    assert O.f16(one + 2 ** -11 + 2 ** -40) == one + 2 ** -10  # no double rounding
    assert O.f16(65519.0) == 65504.0 and np.isinf(O.f16(65520.0))
    assert O.f16(2 ** -25) == 0.0 and O.f16(3 * 2 ** -25) == 2 ** -23  # subnormals
    # at the operands' headroom scale (2**12) the low half stays normal and
    # the pair carries ~22 bits
    x = np.random.default_rng(0).standard_normal(1000) * 2.0 ** 12
    x = x[np.abs(x) > 1.0]
    hi, lo = O.split16(x)
    assert np.max(np.abs(hi + lo - x) / np.abs(x)) < 2 ** -21


# --------------------------------------------------------------- step pieces

def test_factor_ema_brute_force_loops():
    """Element-by-element sums on tiny inputs, including non-identity roots."""
    rng = np.random.default_rng(9)
    m, n = 4, 3
    G = rng.standard_normal((m, n))
    Pa = _spd(m, 5.0, 10)
    Pb = _spd(n, 3.0, 11)
    Sa0, Sb0 = _spd(m, 2.0, 12), _spd(n, 2.0, 13)
    b2, eps = 0.7, 1e-3
    Sa = np.zeros((m, m))
    for i in range(m):
        for j in range(m):
            acc = 0.0
            for k in range(n):
                xi = sum(G[i, l] * Pb[l, k] for l in range(n))
                xj = sum(G[j, l] * Pb[l, k] for l in range(n))
                acc += xi * xj
            Sa[i, j] = b2 * Sa0[i, j] + (1 - b2) / n * acc + (eps if i == j else 0.0)
    Sb = np.zeros((n, n))
    for i in range(n):
        for j in range(n):
            acc = 0.0
            for k in range(m):
                xi = sum(Pa[k, l] * G[l, i] for l in range(m))
                xj = sum(Pa[k, l] * G[l, j] for l in range(m))
                acc += xi * xj
            Sb[i, j] = b2 * Sb0[i, j] + (1 - b2) / m * acc + (eps if i == j else 0.0)
    assert np.allclose(O.factor_ema(Sa0, G @ Pb, b2, n, eps), Sa, atol=1e-12)
    assert np.allclose(O.factor_ema(Sb0, (Pa @ G).T, b2, m, eps), Sb, atol=1e-12)


def test_c_shape_closed_forms():
    assert abs(O.c_shape(16, 16) - 1 / (2 * 4)) < 1e-15
    assert abs(O.c_shape(4, 1) - 2 / 3) < 1e-15
    assert abs(O.c_shape(1, 4) - (0.5 / 3)) < 1e-15


def test_variance_correction_monte_carlo():
    """N_t * kappa_t has unit variance for iid unit gradients (the reading's
    definition), checked by simulation, not by the closed form."""
    rng = np.random.default_rng(14)
    b1 = 0.9684
    trials, T = 200000, 12
    M = np.zeros(trials)
    for t in range(1, T + 1):
        g = rng.standard_normal(trials)
        M = b1 * M + (1 - b1) * g
        N = b1 * M + (1 - b1) * g
        std = np.std(N * O.variance_correction(b1, t))
        assert abs(std - 1) < 0.01
    assert O.variance_correction(0.0, 5) == 1.0


def test_nesterov_combination_for_a_constant_gradient():
    """README bullet "Nesterov momentum with variance correction": for a
    constant gradient G and M_0 = 0 the momentum is M_t = (1 - b1^t) G, and
    the Nesterov combination N_t = kappa_t (b1 M_t + (1 - b1) G) sums to the
    closed form kappa_t (1 - b1^(t+1)) G.  N is recovered from the change of
    W through the step's own roots (U = P_a N P_b), so a combination built
    from M_{t-1} (giving 1 - b1^t), a missing or misplaced kappa, or a wrong
    sign of the update fails here."""
    rng = np.random.default_rng(21)
    m, n = 6, 4
    G = rng.standard_normal((m, n))
    hp = O.Hyper()
    st = O.init_state(m, n, hp)
    W = rng.standard_normal((m, n))
    b1 = hp.beta1
    decay = O.adamc_decay(hp.lr, hp.peak, hp.weight_decay)
    c = O.c_shape(m, n)
    for t in range(1, 6):
        W_prev = W
        st, W, U = O.okls_step(st, W, G, hp.lr, hp)
        assert np.allclose(st.M, (1 - b1 ** t) * G, rtol=1e-13, atol=1e-15)
        U_w = ((1 - decay) * W_prev - W) / (hp.lr * c)
        N = np.linalg.solve(st.Pa, np.linalg.solve(st.Pb.T, U_w.T).T)
        # kappa_t from its definition (variance of the unrolled combination
        # for iid unit gradients), summed here term by term
        v = (1 - b1) ** 2 * (1 + b1) ** 2 + sum((1 - b1) ** 2 * b1 ** (2 * k) for k in range(2, t + 1))
        want = (1 - b1 ** (t + 1)) / math.sqrt(v) * G
        assert O.rel_fro(N, want) < 1e-9, t
        assert O.rel_fro(U_w, U) < 1e-9


def test_hyperparameter_defaults_are_the_readme_table():
    hp = O.Hyper()
    assert (hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay) == \
        (0.09434, 0.9684, 0.9482, 1e-9, 0.0303)
    assert hp.ns_iters == 10


def test_weight_decay_closed_form_with_zero_gradients():
    """G = 0: U = 0, so W_t = W_0 prod_t (1 - lr_t^2 wd / lr_peak)."""
    hp = O.Hyper(lr=0.1)
    rng = np.random.default_rng(15)
    W0 = rng.standard_normal((6, 5))
    lrs = [0.1, 0.05, 0.08, 0.1]
    _st, W, Us = O.okls_run(W0, [np.zeros((6, 5))] * 4, hp, lrs=lrs)
    f = np.prod([1 - l * l * hp.weight_decay / 0.1 for l in lrs])
    assert np.allclose(W, W0 * f, atol=1e-14)
    assert all(np.all(U == 0) for U in Us)


def test_first_step_is_a_descent_direction():
    """<W_1 - (1 - decay) W_0, G> < 0: the update moves against G."""
    hp = O.Hyper()
    rng = np.random.default_rng(16)
    G = rng.standard_normal((7, 5))
    W0 = rng.standard_normal((7, 5))
    _st, W1, _U = O.okls_step(O.init_state(7, 5, hp), W0, G, hp.lr, hp)
    decay = O.adamc_decay(hp.lr, hp.peak, hp.weight_decay)
    assert np.sum((W1 - (1 - decay) * W0) * G) < 0


@pytest.mark.parametrize("beta2,steps", [(0.5, 300), (0.9482, 1500)])
def test_square_fixed_gradient_reaches_scaled_polar_factor(beta2, steps):
    """Fed one square G forever, the KL factors reach a fixed point where
    P_a G P_b = sqrt(n) U V^T (G = U Sigma V^T).  A transposed operand, a
    swapped side or a wrong 1/n breaks this limit."""
    rng = np.random.default_rng(17)
    n = 12
    G = rng.standard_normal((n, n))
    hp = O.Hyper(beta1=0.0, beta2=beta2, eps=0.0, lr=0.0, lr_peak=1.0)
    st = O.init_state(n, n, hp)
    st.Sa, st.Sb = np.eye(n) * 1e-3, np.eye(n) * 1e-3
    W = np.zeros((n, n))
    for _ in range(steps):
        st, W, U = O.okls_step(st, W, G, 0.0, hp)
    u, _s, vt = np.linalg.svd(G)
    assert O.rel_fro(st.Pa @ G @ st.Pb, math.sqrt(n) * (u @ vt)) < 1e-8
    assert O.rel_fro(U, math.sqrt(n) * (u @ vt)) < 1e-8


def test_step_root_modes_agree_on_a_benign_case():
    rng = np.random.default_rng(18)
    hp = O.Hyper()
    G = [rng.standard_normal((24, 16)) for _ in range(4)]
    W0 = rng.standard_normal((24, 16)) * 0.01
    _s1, W1, U1 = O.okls_run(W0, G, hp, root="exact")
    _s2, W2, U2 = O.okls_run(W0, G, hp, root="ns_exact")
    assert O.rel_fro(U2[0], U1[0]) < 1e-3


def test_stale_roots_refresh_schedule():
    """root_every = k: the roots are the eigendecomposition roots of the
    current factors at t = 1, 1+k, ... and unchanged in between, while the
    factors keep their per-step EMA; k = 1 is the default method."""
    rng = np.random.default_rng(19)
    G = [rng.standard_normal((10, 6)) for _ in range(7)]
    W0 = rng.standard_normal((10, 6)) * 0.01
    hp3 = O.Hyper(root_every=3)
    st = O.init_state(10, 6, hp3)
    W = W0
    prev = None
    for t, g in enumerate(G, start=1):
        st, W, _U = O.okls_step(st, W, g, hp3.lr, hp3)
        if (t - 1) % 3 == 0:
            assert O.rel_fro(st.Pa, O.inv_root_exact(st.Sa)) < 1e-12
        else:
            assert np.array_equal(st.Pa, prev.Pa) and np.array_equal(st.Pb, prev.Pb)
            assert not np.allclose(st.Sa, prev.Sa)
        prev = st
    _s1, W1, _ = O.okls_run(W0, G, O.Hyper())
    _s2, W2, _ = O.okls_run(W0, G, O.Hyper(root_every=1))
    assert np.array_equal(W1, W2)


# ----------------------------------------------------------- classic Shampoo

def _shampoo_run(G_seq, hp, root="exact", lr=1.0):
    m, n = np.asarray(G_seq[0]).shape
    st = O.shampoo_init(m, n, hp)
    W = np.zeros((m, n))
    Us = []
    for G in G_seq:
        st, W, U = O.shampoo_step(st, W, G, lr, hp, root=root)
        Us.append(U)
    return st, W, Us


@pytest.mark.parametrize("steps,key", [(1, "shampoo_quarter_root_step_singular_values"),
                                       (4, "shampoo_quarter_root_after_4_accumulations"),
                                       (100, "shampoo_quarter_root_after_100_accumulations")])
def test_shampoo_step_hand_example(hand, steps, key):
    """The whole Shampoo step on the page's gradient, fed `steps` times: the
    last step's singular values are 1, 1 / 0.5, 0.5 / 0.1, 0.1.  An EMA in
    place of the plain sum, a -1/2 exponent or momentum in the middle would
    all miss the 4- and 100-step values."""
    G = np.array(hand["G"], dtype=np.float64)
    hp = O.Hyper(eps=1e-9, ridge=0.0, weight_decay=0.0)
    st, W, Us = _shampoo_run([G] * steps, hp)
    assert np.allclose(_sv(Us[-1])[:2], hand[key], atol=hand["printed_precision"])
    # the descent step itself: W moves by -lr U from W = 0 at the first step
    _st1, W1, U1 = _shampoo_run([G], hp, lr=0.25)
    assert np.allclose(W1, -0.25 * U1[0], atol=1e-15)


def test_shampoo_step_is_scale_invariant(hand):
    """Problem 14 (first part): 10 G gives the same step as G."""
    G = np.array(hand["G"], dtype=np.float64)
    hp = O.Hyper(eps=1e-9, ridge=0.0, weight_decay=0.0)
    _s, _w, U1 = _shampoo_run([G], hp)
    _s, _w, U10 = _shampoo_run([10.0 * G], hp)
    assert np.allclose(_sv(U10[0])[:2], hand["problem14_quarter_root_10G"], atol=hand["printed_precision"])
    assert O.rel_fro(U10[0], U1[0]) < 1e-6


def test_shampoo_factor_sums_brute_force():
    """L_t = eps I + sum_s G_s G_s^T and R_t = eps I + sum_s G_s^T G_s,
    entry by entry with explicit loops, over three random gradients."""
    rng = np.random.default_rng(21)
    for m, n in [(2, 3), (4, 3)]:
        Gs = [rng.standard_normal((m, n)) for _ in range(3)]
        hp = O.Hyper(eps=0.5, ridge=0.0, weight_decay=0.0)
        st, _W, _U = _shampoo_run(Gs, hp)
        for i in range(m):
            for j in range(m):
                want = 0.5 * (i == j)
                for G in Gs:
                    for k in range(n):
                        want += G[i, k] * G[j, k]
                assert abs(st.Sa[i, j] - want) < 1e-12
        for i in range(n):
            for j in range(n):
                want = 0.5 * (i == j)
                for G in Gs:
                    for k in range(m):
                        want += G[k, i] * G[k, j]
                assert abs(st.Sb[i, j] - want) < 1e-12


def _spd(d, cond, seed):
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    w = np.exp(rng.uniform(0.0, math.log(cond), d))
    w[0], w[-1] = 1.0, cond
    return (Q * w) @ Q.T


def test_replay_root_output_is_the_float64_square_root():
    """The root output of the replay without rounding equals the plain
    float64 coupled iteration's Y_K sqrt(c'), and squares back to S + rho c I
    once converged (the scales 2^-2h and sqrt(c') are right)."""
    sch = O.cans_schedule(10, 1e-3)
    S = _spd(48, 100.0, 3)
    for ridge in (0.0, 1e-3):
        rep = O.ns_replay(S, sch, ridge, rounding=False)["root"]
        ref = O.ns_matrix_float64(S, sch, ridge)[1]
        assert O.rel_fro(rep, ref) < 1e-12
        c = math.sqrt(float(np.sum(S * S)))
        assert O.rel_fro(rep @ rep, S + ridge * c * np.eye(48)) < 1e-5


@pytest.mark.parametrize("cond", [1e2, 1e4])
@pytest.mark.parametrize("ridge", [0.0, 1e-3])
def test_quarter_root_chain_reaches_the_eigendecomposition_root(cond, ridge):
    """Two chained exact-arithmetic chains give (S + rho ||S||_F I)^-1/4, and
    P^4 (S + rho c I) = I."""
    sch = O.cans_schedule(10, 1e-3)
    S = _spd(64, cond, 4)
    P = O.quarter_root_chain(S, sch, ridge, "ns_exact")
    assert O.rel_fro(P, O.quarter_root_exact(S, ridge)) < 1e-5
    c = math.sqrt(float(np.sum(S * S)))
    P2 = P @ P
    assert O.rel_fro(P2 @ P2 @ (S + ridge * c * np.eye(64)), np.eye(64)) < 1e-4


def test_quarter_root_replay_is_accurate_with_a_ridge():
    """The binary16 replay of both chains stays within 5e-3 of the exact
    quarter root of the ridged factor up to condition number 1e6."""
    sch = O.cans_schedule(10, 1e-3)
    for d, cond in [(64, 1e2), (128, 1e3), (96, 1e6)]:
        S = _spd(d, cond, d)
        P = O.quarter_root_chain(S, sch, 1e-3, "replay")
        assert O.rel_fro(P, O.quarter_root_exact(S, 1e-3)) < 5e-3


def test_shampoo_stale_roots():
    """root_every = k: fresh quarter roots at t = 1, 1+k, ...; the sums and
    the step still run every step."""
    rng = np.random.default_rng(22)
    Gs = [rng.standard_normal((6, 5)) for _ in range(5)]
    hp = O.Hyper(eps=1e-3, ridge=0.0, weight_decay=0.0, root_every=2)
    st = O.shampoo_init(6, 5, hp)
    W = np.zeros((6, 5))
    prev = None
    for t, G in enumerate(Gs, start=1):
        st, W, U = O.shampoo_step(st, W, G, 1.0, hp)
        if (t - 1) % 2 == 0:
            assert O.rel_fro(st.Pa, O.quarter_root_exact(st.Sa)) < 1e-12
        else:
            assert np.array_equal(st.Pa, prev.Pa) and np.array_equal(st.Pb, prev.Pb)
            assert O.rel_fro(U, prev.Pa @ G @ prev.Pb) < 1e-14
        prev = st


# ------------------------------------------------------------------- SOAP

def _adam_loops(Gs, lr, b1, b2, eps):
    """Textbook Adam (both moments bias-corrected), entry by entry."""
    m, n = Gs[0].shape
    M = [[0.0] * n for _ in range(m)]
    V = [[0.0] * n for _ in range(m)]
    W = [[0.0] * n for _ in range(m)]
    for t, G in enumerate(Gs, start=1):
        for i in range(m):
            for j in range(n):
                g = float(G[i, j])
                M[i][j] = b1 * M[i][j] + (1 - b1) * g
                V[i][j] = b2 * V[i][j] + (1 - b2) * g * g
                mh = M[i][j] / (1 - b1 ** t)
                vh = V[i][j] / (1 - b2 ** t)
                W[i][j] -= lr * mh / (math.sqrt(vh) + eps)
    return np.array(W)


def test_soap_without_refresh_is_adam():
    """Before any refresh the bases are the identity (reading p2), so SOAP is
    Adam with both moments bias-corrected (reading p1), entry by entry."""
    rng = np.random.default_rng(31)
    Gs = [rng.standard_normal((5, 3)) for _ in range(6)]
    st = O.soap_init(5, 3)
    W = np.zeros((5, 3))
    for G in Gs:
        st, W, _N = O.soap_step(st, W, G, 0.05, 0.9, 0.99, 1e-8, f=1000)
    assert np.allclose(W, _adam_loops(Gs, 0.05, 0.9, 0.99, 1e-8), atol=1e-13, rtol=0)


def _orth(d, seed):
    q, _ = np.linalg.qr(np.random.default_rng(seed).standard_normal((d, d)))
    return q


def test_soap_in_a_fixed_basis_is_rotated_adam():
    """With bases A, B held fixed, the step is Adam on A^T G B rotated back
    by A (.) B^T: a transposed rotation or a basis on the wrong side fails."""
    rng = np.random.default_rng(32)
    m, n = 5, 4
    A, B = _orth(m, 1), _orth(n, 2)
    Gs = [rng.standard_normal((m, n)) for _ in range(4)]
    st = O.soap_init(m, n)
    st.QL, st.QR = A, B
    W = np.zeros((m, n))
    for G in Gs:
        st, W, _N = O.soap_step(st, W, G, 0.03, 0.8, 0.95, 1e-6, f=1000)
    W_rot = _adam_loops([A.T @ G @ B for G in Gs], 0.03, 0.8, 0.95, 1e-6)
    assert O.rel_fro(W, A @ W_rot @ B.T) < 1e-12


def test_eigenvectors_are_ordered_and_sign_aligned():
    """Reading p3: decreasing eigenvalues, each column signed to agree with
    the previous basis."""
    d = 6
    A = _orth(d, 3)
    lam = np.array([9.0, 7.0, 4.0, 2.5, 1.0, 0.25])
    S = (A * lam) @ A.T
    Q = O.eigenvectors_aligned(S, A)
    assert np.allclose(Q, A, atol=1e-12)
    flips = np.array([1, -1, 1, -1, -1, 1.0])
    assert np.allclose(O.eigenvectors_aligned(S, A * flips), A * flips, atol=1e-12)
    assert np.allclose(np.diag(Q.T @ S @ Q), lam, atol=1e-12)


def test_soap_refresh_schedule():
    """f = 3: the bases change only at the end of steps 3 and 6, to the
    eigenvectors of the factors of that step; L, R are EMAs of G G^T, G^T G."""
    rng = np.random.default_rng(33)
    st = O.soap_init(4, 3)
    W = np.zeros((4, 3))
    L = np.zeros((4, 4))
    for t in range(1, 7):
        G = rng.standard_normal((4, 3))
        prev = st
        st, W, _N = O.soap_step(st, W, G, 0.01, 0.9, 0.95, 1e-8, f=3)
        L = 0.95 * L + 0.05 * G @ G.T
        assert np.allclose(st.L, L, atol=1e-14)
        if t % 3 == 0:
            QL = st.QL
            assert np.allclose(QL.T @ L @ QL, np.diag(np.diag(QL.T @ L @ QL)), atol=1e-12)
        else:
            assert np.array_equal(st.QL, prev.QL) and np.array_equal(st.QR, prev.QR)


# ------------------------------------------------------------------ Clean

def test_eps64_is_the_binary64_spacing():
    """Reading c2: eps(x) = 2^(floor(log2 x) - 52)."""
    from oracle import okls_oracle as OO
    assert OO._eps64(1.0) == 2.0 ** -52 and OO._eps64(3.0) == 2.0 ** -51
    assert OO._eps64(0.75) == 2.0 ** -53 and np.nextafter(8.0, 9.0) - 8.0 == OO._eps64(8.0)


@pytest.mark.parametrize("warm", [False, True])
def test_nystrom_recovers_an_exactly_low_rank_operator(warm):
    """Algorithm 3 on a rank-r PSD matrix returns its eigenpairs (decreasing;
    with a warm start, signs aligned to it) to rounding."""
    rng = np.random.default_rng(41)
    d, r, p = 30, 5, 4
    U0 = _orth(d, 9)[:, :r]
    lam0 = np.array([9.0, 6.0, 4.0, 2.0, 1.0])
    A = (U0 * lam0) @ U0.T
    prev = U0 * np.array([1, -1, 1, 1, -1.0]) if warm else None
    psi = rng.standard_normal((d, p if warm else r + p))
    U, lam = O.nystrom_warm(lambda X: A @ X, r, p, 1, prev, psi)
    assert np.allclose(lam, lam0, rtol=1e-10)
    if warm:
        assert np.allclose(U, prev, atol=1e-10)
    else:
        assert np.allclose(np.abs(U.T @ U0), np.eye(r), atol=1e-10)


def test_nystrom_with_power_iterations_tracks_the_top_eigenpairs():
    rng = np.random.default_rng(42)
    d, r, p = 40, 4, 6
    Q = _orth(d, 10)
    lam_all = 0.5 ** np.arange(d)
    A = (Q * lam_all) @ Q.T
    U, lam = O.nystrom_warm(lambda X: A @ X, r, p, 3, None, rng.standard_normal((d, r + p)))
    assert np.allclose(lam, lam_all[:r], rtol=1e-6)
    assert np.allclose(np.abs(U.T @ Q[:, :r]), np.eye(r), atol=1e-6)


def test_clean_blocks_partition_the_gradient():
    """Eqn. (10) with the scalings dropped: U_L S U_R^T + G_A U_R^T + U_L G_B
    + C = G for orthonormal U_L, U_R (a projector on the wrong side breaks it)."""
    rng = np.random.default_rng(43)
    m, n, r = 9, 7, 3
    UL, UR = _orth(m, 11)[:, :r], _orth(n, 12)[:, :r]
    G = rng.standard_normal((m, n))
    PL, PR = np.eye(m) - UL @ UL.T, np.eye(n) - UR @ UR.T
    S, GA, GB, C = UL.T @ G @ UR, PL @ G @ UR, UL.T @ G @ PR, PL @ G @ PR
    assert O.rel_fro(UL @ S @ UR.T + GA @ UR.T + UL @ GB + C, G) < 1e-14


def test_clean_moments_by_entry_loops():
    """Table 1 / Eqns. (12)-(13): first moments EMAs of S, G_A, G_B; second
    moments V entry-wise, v_A summed over rows, v_B over columns, v_C the
    squared Frobenius norm of C (sums as printed, reading c6)."""
    rng = np.random.default_rng(44)
    m, n, r, p = 8, 6, 2, 2
    b1, b2 = 0.8, 0.9
    st = O.clean_init(m, n, r)
    G1 = rng.standard_normal((m, n))
    st, _W, _Gt = O.clean_step(st, np.zeros((m, n)), G1, 0.1, b1, b2, 1e-8, r, p, 1, 100,
                               rng.standard_normal((m, r + p)), rng.standard_normal((n, r + p)))
    UL, UR = st.UL, st.UR
    G2 = rng.standard_normal((m, n))
    prev = st
    st, _W, _Gt = O.clean_step(prev, np.zeros((m, n)), G2, 0.1, b1, b2, 1e-8, r, p, 1, 100)
    PL, PR = np.eye(m) - UL @ UL.T, np.eye(n) - UR @ UR.T
    GA, GB, C = PL @ G2 @ UR, UL.T @ G2 @ PR, PL @ G2 @ PR
    for j in range(r):
        s = sum(GA[i, j] ** 2 for i in range(m))
        assert abs(st.vA[j] - (b2 * prev.vA[j] + (1 - b2) * s)) < 1e-12
    for i in range(r):
        s = sum(GB[i, j] ** 2 for j in range(n))
        assert abs(st.vB[i] - (b2 * prev.vB[i] + (1 - b2) * s)) < 1e-12
    s = sum(C[i, j] ** 2 for i in range(m) for j in range(n))
    assert abs(st.vC - (b2 * prev.vC + (1 - b2) * s)) < 1e-12
    assert np.allclose(st.MA, b1 * prev.MA + (1 - b1) * GA, atol=1e-14)


def test_clean_full_rank_bases_are_rotated_adam():
    """r = m = n: the complements vanish, blocks A, B, C are zero, and with
    the bases of the first refresh kept the whole run is Adam on
    S_t = U_L^T G_t U_R rotated back by U_L (.) U_R^T."""
    rng = np.random.default_rng(45)
    d, r, p, lr, b1, b2, eps = 5, 5, 0, 0.05, 0.9, 0.95, 1e-8
    st = O.clean_init(d, d, r)
    W = np.zeros((d, d))
    Gs = [rng.standard_normal((d, d)) for _ in range(4)]
    for t, G in enumerate(Gs, start=1):
        psi = (rng.standard_normal((d, r)), rng.standard_normal((d, r))) if t == 1 else (None, None)
        st, W, _ = O.clean_step(st, W, G, lr, b1, b2, eps, r, p, 1, 1000, *psi)
    assert np.abs(st.MA).max() < 1e-12 and np.abs(st.MB).max() < 1e-12 and st.vC < 1e-20
    W_rot = _adam_loops([st.UL.T @ G @ st.UR for G in Gs], lr, b1, b2, eps)
    # the complement blocks are rounding-level (~1e-16) but block C divides by
    # sqrt(v_C) + eps, lifting them to ~1e-16 / eps = 1e-8
    assert O.rel_fro(W, st.UL @ W_rot @ st.UR.T) < 1e-6


def test_clean_moment_transport_is_identity_for_an_unchanged_basis():
    """Eqns. (14)-(15): a refresh that returns the same bases leaves every
    moment as it was."""
    rng = np.random.default_rng(46)
    m, n, r, p = 10, 8, 3, 2
    UL0, UR0 = _orth(m, 13)[:, :r], _orth(n, 14)[:, :r]
    st = O.clean_init(m, n, r)
    st.UL, st.lamL, st.UR, st.lamR = UL0, np.array([3.0, 2.0, 1.0]), UR0, np.array([3.0, 2.0, 1.0])
    st.M = rng.standard_normal((r, r))
    st.MA = (np.eye(m) - UL0 @ UL0.T) @ rng.standard_normal((m, r))
    st.MB = rng.standard_normal((r, n)) @ (np.eye(n) - UR0 @ UR0.T)
    st.vA, st.vB = rng.random(r), rng.random(r)
    st.t = 3   # the next step (t = 4) refreshes with T = 3
    # a gradient that keeps the factors' eigenvectors: G = U_L diag U_R^T
    G = UL0 @ np.diag([1.0, 0.8, 0.6]) @ UR0.T
    new, _W, _ = O.clean_step(st, np.zeros((m, n)), G, 0.0, 0.0, 0.5, 1e-8, r, p, 2, 3,
                              rng.standard_normal((m, p)), rng.standard_normal((n, p)))
    assert np.allclose(new.UL, UL0, atol=1e-10) and np.allclose(new.UR, UR0, atol=1e-10)
    # with beta1 = 0 the first moments are this step's blocks; v_A, v_B decay with beta2 only
    assert np.allclose(new.vA, 0.5 * st.vA + 0.5 * np.sum(((np.eye(m) - UL0 @ UL0.T) @ G @ UR0) ** 2, axis=0),
                       atol=1e-10)
    assert np.allclose(new.vB, 0.5 * st.vB, atol=1e-10)
