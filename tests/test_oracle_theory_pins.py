"""Pins of the oracle's step-time theory ("Speculative Decoding for Mixture-of-Experts
Models" (Lan), §3.2-3.5, App. B.1-B.3 and C) to closed forms, brute force and the pages'
printed examples (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import load_golden


def _rand_V(rng, kmax, kind="any"):
    if kind == "convex":
        c = np.sort(rng.uniform(0.0, 1.0, kmax))
        v0 = rng.uniform(0.5, 2.0)
        return np.concatenate([[v0], v0 + np.cumsum(c)])
    return rng.uniform(0.2, 3.0, kmax + 1)


def _G(a, k):
    return sum(a ** i for i in range(k + 1))


# ------------------------------------------------------------------ alpha_{k,i}

def test_alpha_closed_forms(oracle_mod):
    """(1,0): T_a(1) > T_a(0) iff a > V1/V0 - 1 (B.4).  (2,0) and (2,1): the positive roots of
    the quadratics 1 + a + a^2 = V2/V0 and (1 + a + a^2) V1 = (1 + a) V2, clamped to [0, 1]."""
    rng = np.random.default_rng(100)
    for _ in range(400):
        V = _rand_V(rng, 2)
        a0 = V[1] / V[0] - 1
        assert oracle_mod.alpha(V, 1, 0) == pytest.approx(min(max(a0, 0.0), 1.0), abs=1e-12)
        R = V[2] / V[0]
        want = 0.0 if R <= 1 else (1.0 if R >= 3 else (-1 + math.sqrt(4 * R - 3)) / 2)
        assert oracle_mod.alpha(V, 2, 0) == pytest.approx(want, abs=1e-12)
        R = V[2] / V[1]
        want = 0.0 if R <= 1 else (1.0 if R >= 1.5 else ((R - 1) + math.sqrt((R - 1) * (R + 3))) / 2)
        assert oracle_mod.alpha(V, 2, 1) == pytest.approx(want, abs=1e-10)


def test_alpha_matches_polynomial_roots(oracle_mod):
    """alpha_{k,i} is the largest root in [0, 1) of G_a(k) V(i) - G_a(i) V(k) where it turns
    positive (numpy.roots of the polynomial), 0 if positive at a = 0, 1 if never positive."""
    rng = np.random.default_rng(101)
    for _ in range(300):
        kmax = int(rng.integers(1, 8))
        V = _rand_V(rng, kmax)
        for k in range(1, kmax + 1):
            for i in range(k):
                # coefficients of V(i) G_a(k) - V(k) G_a(i), lowest degree first
                c = np.zeros(k + 1)
                c[:k + 1] += V[i]
                c[:i + 1] -= V[k]
                P = np.polynomial.Polynomial(c)
                if P(0.0) > 0:
                    want = 0.0
                else:
                    r = [x.real for x in P.roots() if abs(x.imag) < 1e-9 and 0 <= x.real < 1]
                    r = [x for x in r if P(min(x + 1e-7, 1 - 1e-12)) > 0]
                    want = max(r) if r else 1.0
                assert oracle_mod.alpha(V, k, i) == pytest.approx(want, abs=1e-7), (V, k, i)


# ------------------------------------------------------------------ step points

def test_step_points_match_the_brute_force_staircase(oracle_mod):
    """(B.31): k*(a) >= j for a > a_j and k*(a) < j for a < a_j, with k*(a) the smallest
    maximiser of G_a(k)/V(k) evaluated directly on a grid."""
    rng = np.random.default_rng(102)
    grid = np.linspace(0.0, 0.9995, 2001)
    for _ in range(120):
        kmax = int(rng.integers(1, 7))
        V = _rand_V(rng, kmax, kind=("convex" if rng.random() < 0.5 else "any"))
        steps = oracle_mod.step_points(V)
        ks = np.array([oracle_mod.best_draft_length(V, a) for a in grid])
        for j in range(1, kmax + 1):
            above = grid > steps[j] + 1e-9
            below = grid < steps[j] - 1e-9
            assert np.all(ks[above] >= j), (V, j, steps)
            assert np.all(ks[below] < j), (V, j, steps)
        # monotone staircase (B.28)
        assert np.all(np.diff(ks) >= 0)


def test_step_points_of_the_jump_example(oracle_mod):
    """App. B.3 'Jumps': V = (1, 2, 2) jumps from 0 to 2; alpha_{1,0} = 1 (one draft never
    helps), a_1 = a_2 = alpha_{2,0} = (sqrt(5) - 1)/2 from 1 + a + a^2 = 2."""
    g = load_golden("staircase_jump.json")
    V = np.array(g["V"])
    steps = oracle_mod.step_points(V)
    phi = (math.sqrt(5) - 1) / 2
    assert oracle_mod.alpha(V, 1, 0) == 1.0
    assert steps[1] == pytest.approx(phi, abs=1e-14) and steps[2] == pytest.approx(phi, abs=1e-14)
    for a, k in g["cases"]:
        assert (a > steps[1]) == (k >= 1)


def test_first_threshold_and_speedup(oracle_mod):
    """(B.4) a0 = V(1)/V(0) - 1 decides T_a(1) > T_a(0); (9) the speedup G_a(k) V(0)/V(k)."""
    rng = np.random.default_rng(103)
    for _ in range(200):
        V = _rand_V(rng, 4)
        a0 = oracle_mod.first_threshold(V)
        for a in rng.uniform(0, 1, 5):
            assert (oracle_mod.throughput(V, 1, a) > oracle_mod.throughput(V, 0, a)) == (a > a0)
            for k in range(5):
                assert oracle_mod.speedup(V, k, a) == pytest.approx(_G(a, k) * V[0] / V[k], rel=1e-14)


def test_convex_step_points(oracle_mod):
    """(10), (B.35)-(B.36): for a convex non-decreasing step time, k*(a) >= j iff
    a^j V(j-1) > G_a(j-1) c_j, its step point equals (B.31), and a_1 = min(c_1/V(0), 1)."""
    rng = np.random.default_rng(104)
    grid = np.linspace(0.0, 0.999, 500)
    for _ in range(100):
        kmax = int(rng.integers(1, 7))
        V = _rand_V(rng, kmax, kind="convex")
        assert oracle_mod.convex_nondecreasing(V)
        steps = oracle_mod.step_points(V)
        for j in range(1, kmax + 1):
            assert oracle_mod.convex_step_point(V, j) == pytest.approx(steps[j], abs=1e-9)
            c = V[j] - V[j - 1]
            for a in grid[::25]:
                assert (oracle_mod.best_draft_length(V, a) >= j) == (a ** j * V[j - 1] > _G(a, j - 1) * c)
        assert oracle_mod.convex_step_point(V, 1) == pytest.approx(min((V[1] - V[0]) / V[0], 1.0), abs=1e-15)
    assert not oracle_mod.convex_nondecreasing([1.0, 3.0, 4.0])      # c_2 < c_1
    assert not oracle_mod.convex_nondecreasing([2.0, 1.0, 3.0])      # c_1 < 0
    assert oracle_mod.convex_nondecreasing([1.0, 1.0, 1.0])


# ------------------------------------------------------------------ reuse threshold

def _periodic_reuse(oracle_mod, pattern, n):
    """rho(n) of a pattern repeated from a uniformly random phase: the reuse estimate over
    exactly one window per phase (T = P*R + n - 1 tokens)."""
    P = len(pattern)
    R = 4
    T = P * R + n - 1
    sets = np.array([[int(pattern[t % P])] for t in range(T)], dtype=np.int32)
    return oracle_mod.reuse_estimate(sets, 3, n), sets


def test_no_single_threshold_counterexample(oracle_mod):
    """App. B.2: rho*_1 = 7/20, rho*_2 = 371/800 from (16), and the three patterns' mean
    reuses and speedup decisions, each checked by brute force on the union step time too."""
    g = load_golden("no_single_threshold.json")
    a = g["a"][0] / g["a"][1]
    rs = [oracle_mod.reuse_threshold_bytes(k, a, 1.0) for k in (1, 2)]
    for got, (p, q) in zip(rs, g["rho_star"]):
        assert got == pytest.approx(p / q, abs=1e-15)
    for pat in g["patterns"]:
        rho = np.zeros((1, 4))
        for n in (2, 3):
            rho[0, n], _ = _periodic_reuse(oracle_mod, pat["pattern"], n)
        rb = [oracle_mod.mean_reuse([1.0], rho, k) for k in (1, 2)]
        for got, (p, q) in zip(rb, pat["rho_bar"]):
            assert got == pytest.approx(p / q, abs=1e-12), pat
        faster = [rb[k - 1] > rs[k - 1] for k in (1, 2)]
        assert any(faster) == pat["speedup"]
        if pat["k"] is not None:
            assert faster[pat["k"] - 1]
        # one bandwidth, t0 = phi = 0: V(k) = E_dedup(k+1) = mean union of k+1 tokens
        V = []
        for k in range(3):
            n = k + 1
            _, sets = _periodic_reuse(oracle_mod, pat["pattern"], n)
            T = len(sets)
            V.append(np.mean([oracle_mod.union_size(sets, 3, t0, n) for t0 in range(T - n + 1)]))
        assert (oracle_mod.best_draft_length(V, a) >= 1) == pat["speedup"]


def test_time_threshold_identity(oracle_mod):
    """(B.13): V(k) - V(0) - (G_a(k) - 1) V(0) = (m W k / B_k)(rho*_k(a) - rho_bar_k) with
    V(0), V(k) from (B.10); hence T_a(k) > T_a(0) iff rho_bar_k > rho*_k(a) (B.14)."""
    rng = np.random.default_rng(105)
    for _ in range(500):
        k = int(rng.integers(1, 8))
        a = rng.uniform(0, 1)
        mW, Bk, b1, bD = rng.uniform(1, 10), rng.uniform(0.5, 2), rng.uniform(0.5, 2), rng.uniform(0.5, 2)
        t0, D1, dD, phi1, dphi = rng.uniform(0, 2), rng.uniform(0, 5), rng.uniform(0, 3), rng.uniform(0, 1), rng.uniform(-0.5, 1)
        phik = phi1 + dphi
        if phik < 0:
            continue
        rb = rng.uniform(0, 1)
        V0 = t0 + D1 / bD + mW / b1 + phi1
        Vk = t0 + (D1 + dD) / bD + (mW + mW * k * (1 - rb)) / Bk + phik
        rs = oracle_mod.reuse_threshold(k, a, mW, Bk, b1, V0, dD / bD, dphi)
        lhs = Vk - V0 - (_G(a, k) - 1) * V0
        assert lhs == pytest.approx(mW * k / Bk * (rs - rb), rel=1e-9, abs=1e-9)
        V = np.array([V0] + [Vk] * k)
        assert (_G(a, k) / Vk > 1 / V0) == (rb > rs) or abs(rb - rs) < 1e-12


def test_byte_form_is_the_one_bandwidth_time_form(oracle_mod):
    """(16) is (14) with beta_D = B_k = beta(1) = beta and t0 = phi = 0 (B.16)."""
    rng = np.random.default_rng(106)
    for _ in range(300):
        k, a = int(rng.integers(1, 8)), rng.uniform(0, 1)
        mW, beta, D1, Dk1 = rng.uniform(1, 10), rng.uniform(0.1, 5), rng.uniform(0, 5), 0.0
        Dk1 = D1 + rng.uniform(0, 3)
        t = oracle_mod.reuse_threshold(k, a, mW, beta, beta, (D1 + mW) / beta, (Dk1 - D1) / beta, 0.0)
        assert t == pytest.approx(oracle_mod.reuse_threshold_bytes(k, a, mW, D1, Dk1), rel=1e-12, abs=1e-12)


def test_threshold_falls_with_acceptance(oracle_mod):
    """(B.19): rho*_k(a) strictly decreases in a (and in D for a > 0)."""
    rng = np.random.default_rng(107)
    for _ in range(200):
        k, mW = int(rng.integers(1, 6)), rng.uniform(1, 5)
        a, a2 = np.sort(rng.uniform(0, 1, 2))
        D, D2 = np.sort(rng.uniform(0, 5, 2))
        assert oracle_mod.reuse_threshold_bytes(k, a2, mW, D, D) < oracle_mod.reuse_threshold_bytes(k, a, mW, D, D)
        assert oracle_mod.reuse_threshold_bytes(k, a2, mW, D2, D2) < oracle_mod.reuse_threshold_bytes(k, a2, mW, D, D)


# ------------------------------------------------------------------ error bounds

def test_error_bounds_hold_under_random_bandwidth_errors(oracle_mod):
    """Table 2 / App. C: with every bandwidth of (5) estimated as beta (1 + e), |e| <= eps,
    the verify time, the saving, the faster kernel, the best draft length and the best
    speedup move no more than (17)-(21) allow; delta = eps/(1 - eps)."""
    rng = np.random.default_rng(108)
    for _ in range(400):
        eps = rng.uniform(0.01, 0.3)
        f = oracle_mod.err_verify_factor(eps)
        assert f == pytest.approx(eps / (1 - eps))
        e = lambda: rng.uniform(-eps, eps)
        # (17), (18): one pass, both kernels
        t0, D, bD, phi = rng.uniform(0, 1), rng.uniform(0, 5), rng.uniform(0.5, 2), rng.uniform(0, 1)
        Es, Ed = rng.uniform(1, 10), rng.uniform(0.5, 10)
        bs, bd = rng.uniform(0.5, 2), rng.uniform(0.3, 2)
        eD, es, ed = e(), e(), e()
        tau_s, tau_d = t0 + D / bD + Es / bs + phi, t0 + D / bD + Ed / bd + phi
        that_s = t0 + D / (bD * (1 + eD)) + Es / (bs * (1 + es)) + phi
        that_d = t0 + D / (bD * (1 + eD)) + Ed / (bd * (1 + ed)) + phi
        assert abs(that_s - tau_s) <= f * (D / bD + Es / bs) + 1e-12
        assert abs(that_s - tau_s) <= f * tau_s + 1e-12
        S, Shat = tau_s - tau_d, that_s - that_d
        assert abs(Shat - S) <= oracle_mod.err_saving_bound(eps, Es / bs, Ed / bd) + 1e-12
        # (19): ubar = Ed/Es, r = bd/bs
        if oracle_mod.err_decision_agrees(bd / bs, Ed / Es, eps):
            assert (Es / (bs * (1 + es)) > Ed / (bd * (1 + ed))) == (Es / bs > Ed / bd)
        # (20), (21): step times with bandwidth errors only, delta = eps/(1-eps)
        kmax = int(rng.integers(1, 6))
        mem = rng.uniform(0.5, 3, kmax + 1)
        fixed = rng.uniform(0, 1, kmax + 1)
        V = mem + fixed
        Vhat = mem / (1 + rng.uniform(-eps, eps, kmax + 1)) + fixed
        delta = f
        assert np.all((1 - delta) * V <= Vhat + 1e-12) and np.all(Vhat <= (1 + delta) * V + 1e-12)
        a = rng.uniform(0, 1)
        ks, kh = oracle_mod.best_draft_length(V, a), oracle_mod.best_draft_length(Vhat, a)
        T = lambda W, k: _G(a, k) / W[k]
        assert T(V, kh) >= oracle_mod.err_regret_factor(delta) * T(V, ks) - 1e-12
        if oracle_mod.err_kstar_separated(V, a, delta):
            assert kh == ks
        lo, hi = oracle_mod.err_speedup_interval(delta)
        ratio = (T(Vhat, kh) / T(Vhat, 0)) / (T(V, ks) / T(V, 0))
        assert lo - 1e-12 <= ratio <= hi + 1e-12


def test_error_bound_factor_at_ten_percent(oracle_mod):
    """§3.5 and (C.7): a 10% bandwidth error moves the predicted speedup by at most 25%."""
    delta = oracle_mod.err_verify_factor(0.1)
    lo, hi = oracle_mod.err_speedup_interval(delta)
    assert hi == pytest.approx(1.25, rel=1e-14) and lo == pytest.approx(0.8, rel=1e-14)
    assert oracle_mod.err_decision_agrees(1.0, 0.8, 0.1) is True     # |ln 1.25| > ln(1.1/0.9)
    assert oracle_mod.err_decision_agrees(1.0, 0.85, 0.1) is False


# ------------------------------------------------------------------ chosen ids and fits

def test_chosen_ids_name_exactly_U_experts(oracle_mod):
    from moe_speculative_decoding_gb300 import synth
    rng = np.random.default_rng(110)
    for _ in range(300):
        N, m = int(rng.integers(2, 130)), 0
        m = int(rng.integers(1, min(N, 9) + 1))
        n = int(rng.integers(1, 17))
        U = int(rng.integers(m, min(N, n * m) + 1))
        ids = synth.chosen_ids(n, m, N, U, seed=int(rng.integers(1 << 30)))
        assert ids.shape == (n, m) and ids.min() >= 0 and ids.max() < N
        assert all(len(set(row)) == m for row in ids.tolist())
        assert len(set(ids.ravel().tolist())) == U
        assert oracle_mod.pass_bytes(64, 64, N, ids)["U"] == U
    with pytest.raises(ValueError):
        synth.chosen_ids(2, 4, 128, 3, 0)


def test_fits_recover_known_coefficients(oracle_mod):
    """(4) and (E.1) on noise-free times built from known constants return them; on noisy
    times the residual is orthogonal to every regressor (least squares)."""
    rng = np.random.default_rng(111)
    m, b = 8, 9.437184e6
    n = np.repeat(np.arange(2, 10), 5)
    U = np.array([int(rng.integers(m, n_ * m + 1)) for n_ in n])
    t_op, cu, cre = 12e-6, 1.4e-13, 0.3e-13
    t = t_op + cu * U * b + cre * (n * m - U) * b
    got = oracle_mod.fit_slot(n, U, t, m, b)
    assert got == pytest.approx((t_op, cu, cre), rel=1e-9)
    tg, cg, ct = 9e-6, 1.6e-13, 2e-7
    got = oracle_mod.fit_dedup(n, U, tg + cg * U * b + ct * n, b)
    assert got == pytest.approx((tg, cg, ct), rel=1e-9)
    noisy = t * (1 + rng.normal(0, 0.02, t.size))
    c = oracle_mod.fit_slot(n, U, noisy, m, b)
    res = noisy - (c[0] + c[1] * U * b + c[2] * (n * m - U) * b)
    for col in (np.ones_like(U), U * b, (n * m - U) * b):
        assert abs(np.dot(res, col)) <= 1e-9 * np.linalg.norm(col) * np.linalg.norm(noisy)
    assert oracle_mod.fit_error([1.1, 0.9, 1.0], [1.0, 1.0, 1.0]) == pytest.approx(0.1)
