"""Pins of the oracle's verify-side neighbours to what the pages fix.

Speculative sampling ("Lossless but Not Free: An Empirical Anatomy of Speculative Decoding on
Consumer Hardware", §3.1-3.2): Proposition 1 (the emitted token is distributed as the target's
p) by exact enumeration of the draft token and of fine grids of the uniform draws; the greedy
special case as the general rule on one-hot distributions; the expected yield
(1 - a^{K+1})/(1 - a) under a position-independent acceptance rate; hand cases and the edge
cases the readings define.  Expert-union cost ("SpecFit", §3.2 eqs (3)-(5)): per-layer set
unions in Python, monotone and submodular F, additive R, brute-force argmax of R/T."""
import itertools

import numpy as np
import pytest

import oracle


def _dist(rng, V, zeros=0):
    w = rng.random(V).astype(np.float64) + 0.05
    if zeros:
        w[rng.choice(V, zeros, replace=False)] = 0.0
    return (w / w.sum()).astype(np.float32)


def _first_token(draft, na, tok):
    return np.where(na >= 1, draft[:, 0], tok)


@pytest.mark.parametrize("seed,V,zeros", [(0, 5, 0), (1, 6, 2), (2, 4, 1)])
def test_proposition_1_exact_enumeration(seed, V, zeros):
    """P[Y = y] = p_1(y) for the first emitted token: x_1 ~ q_1 enumerated exactly, r and u on
    midpoint grids of 512 and 1024 points (discretisation error below 3e-3)."""
    rng = np.random.default_rng(seed)
    p1, p2, q1 = _dist(rng, V, zeros), _dist(rng, V), _dist(rng, V, zeros)
    R, U = 512, 1024
    rs = ((np.arange(R) + 0.5) / R).astype(np.float32)
    us = ((np.arange(U) + 0.5) / U).astype(np.float32)
    prob = np.zeros(V)
    for x in range(V):
        if q1[x] == 0.0:
            continue
        # every (r, u) pair as one sequence of a batch
        B = R * U
        draft = np.full((B, 1), x, np.int32)
        q = np.broadcast_to(q1, (B, 1, V))
        p = np.broadcast_to(np.stack([p1, p2]), (B, 2, V))
        r = np.repeat(rs, U).reshape(B, 1)
        u = np.tile(us, R)
        na, tok = oracle.spec_accept(draft, q, p, r, u)
        y = _first_token(draft, na, tok)
        prob += q1[x] * np.bincount(y, minlength=V) / B
    assert np.max(np.abs(prob - p1)) < 3e-3, (prob, p1)
    # a planted mistake would show: resampling from p instead of max(0, p - q) overweights
    # the tokens the draft already covers
    assert np.max(np.abs(np.minimum(p1, q1) + p1 * (1 - np.minimum(p1, q1).sum()) - p1)) > 1e-2


def test_greedy_is_the_general_rule_on_one_hots():
    """[Anatomy] §3.2: as T -> 0 both distributions are one-hot and the general rule is
    'accept iff argmax p_i = x_i, else emit argmax p_i' (no draw consumed)."""
    rng = np.random.default_rng(5)
    B, K, V = 64, 6, 40
    logits = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    p = np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)
    am = p.argmax(-1)
    # drafts: the target's argmax for a random number of leading positions, then a miss
    lead = rng.integers(0, K + 1, size=B)
    draft = am[:, :K].copy().astype(np.int32)
    for b in range(B):
        if lead[b] < K:
            draft[b, lead[b]] = (am[b, lead[b]] + 1 + rng.integers(0, V - 1)) % V
    onehot_p = np.eye(V, dtype=np.float32)[am]
    onehot_q = np.eye(V, dtype=np.float32)[draft]
    r = rng.random((B, K)).astype(np.float32)
    u = rng.random(B).astype(np.float32)
    na_g, tok_g = oracle.spec_accept(draft, None, p, None, None, greedy=True)
    na_1, tok_1 = oracle.spec_accept(draft, onehot_q, onehot_p, r, u)
    na_h, tok_h = oracle.spec_accept(draft, None, onehot_p, None, None, greedy=True)
    assert np.array_equal(na_g, lead) and np.array_equal(na_g, na_1) and np.array_equal(na_g, na_h)
    assert np.array_equal(tok_g, am[np.arange(B), lead]) and np.array_equal(tok_g, tok_1)
    assert np.array_equal(tok_g, tok_h)


@pytest.mark.parametrize("alpha,K", [(0.6, 4), (0.85, 7), (0.3, 2)])
def test_expected_yield(alpha, K):
    """Position-independent acceptance a = sum min(p_i, q_i): the mean tokens per round is
    (1 - a^{K+1})/(1 - a) ([Anatomy] §3.2, "Expected yield"); Monte Carlo within 4 SE."""
    rng = np.random.default_rng(11)
    V, B = 12, 40000
    c = np.zeros(V)
    c[2:] = rng.random(V - 2) + 0.1
    c /= c.sum()
    p_row = (alpha * c + (1 - alpha) * np.eye(V)[0]).astype(np.float32)
    q_row = (alpha * c + (1 - alpha) * np.eye(V)[1]).astype(np.float32)
    assert abs(np.minimum(p_row, q_row).sum() - alpha) < 1e-6
    qd = q_row.astype(np.float64)
    qd /= qd.sum()
    draft = np.searchsorted(np.cumsum(qd), rng.random((B, K)) * np.cumsum(qd)[-1], side="right")
    draft = np.minimum(draft, V - 1).astype(np.int32)
    q = np.broadcast_to(q_row, (B, K, V))
    p = np.broadcast_to(p_row, (B, K + 1, V))
    r = rng.random((B, K)).astype(np.float32)
    u = rng.random(B).astype(np.float32)
    na, _ = oracle.spec_accept(draft, q, p, r, u)
    got = (na + 1).astype(np.float64)
    want = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(got.mean() - want) < 4 * got.std() / np.sqrt(B) + 1e-3, (got.mean(), want)


def test_accept_test_hand_cases():
    """r < min(1, p(x)/q(x)) in single precision; p >= q always accepts; a zero-probability
    draft (q(x) = 0) is accepted iff p(x) > 0; ids outside [0, V) are rejected."""
    V = 4
    p = np.array([[[0.1, 0.4, 0.3, 0.2], [0.25, 0.25, 0.25, 0.25]]], np.float32)
    q = np.array([[[0.2, 0.2, 0.3, 0.3]]], np.float32)
    u = np.array([0.0], np.float32)
    ratio = np.float32(0.2) / np.float32(0.3)          # x = 3: p/q = 2/3
    below = np.nextafter(ratio, np.float32(0))
    assert oracle.spec_accept([[3]], q, p, [[below]], u)[0][0] == 1
    assert oracle.spec_accept([[3]], q, p, [[ratio]], u)[0][0] == 0
    assert oracle.spec_accept([[1]], q, p, [[0.999999]], u)[0][0] == 1      # p >= q
    q0 = q.copy(); q0[0, 0, 2] = 0.0
    assert oracle.spec_accept([[2]], q0, p, [[0.999999]], u)[0][0] == 1     # q(x) = 0, p(x) > 0
    p0 = p.copy(); p0[0, 0, 2] = 0.0
    assert oracle.spec_accept([[2]], q0, p0, [[0.0]], u)[0][0] == 0         # both zero
    assert oracle.spec_accept([[V]], q, p, [[0.0]], u)[0][0] == 0           # bad id
    assert oracle.spec_accept([[-1]], q, p, [[0.0]], u)[0][0] == 0


def test_resample_and_bonus_edges():
    """The adjusted draw never picks a token with p <= q; K = 0 is a bonus draw only; all-zero
    adjusted weights fall back to p, an all-zero p to its argmax (index 0)."""
    p = np.array([[[0.5, 0.1, 0.4], [0.2, 0.3, 0.5]]], np.float32)
    q = np.array([[[0.2, 0.6, 0.2]]], np.float32)   # adjusted weights: [0.3, 0, 0.2]
    for uu in np.linspace(0, 0.999, 50, dtype=np.float32):
        na, tok = oracle.spec_accept([[1]], q, p, [[0.99]], [uu])
        assert na[0] == 0 and tok[0] in (0, 2)
        assert tok[0] == (0 if uu < np.float32(0.3) / np.float32(0.5) - 1e-6 else tok[0])
    na, tok = oracle.spec_accept(np.zeros((1, 0), np.int32), None, p[:, 1:], None, [0.1])
    assert na[0] == 0 and tok[0] == 0
    na, tok = oracle.spec_accept(np.zeros((1, 0), np.int32), None, p[:, 1:], None, [0.99])
    assert tok[0] == 2
    same = np.array([[[0.2, 0.3, 0.5], [0.0, 1.0, 0.0]]], np.float32)
    # p == q at the rejected position (reject needs r >= 1 here): fallback to p itself
    na, tok = oracle.spec_accept([[0]], same[:, :1], same, [[1.0]], [0.95])
    assert na[0] == 0 and tok[0] == 2
    zero = np.zeros((1, 1, 3), np.float32)
    assert oracle.spec_accept(np.zeros((1, 0), np.int32), None, zero, None, [0.5])[1][0] == 0


def test_fixed_point_draw():
    """Frequencies over a uniform u grid equal the weights' shares within the grid step;
    u = 0 gives the first positive weight, u near 1 the last; zero weights are never drawn;
    a boundary case worked by hand (w = [1/4, 0, 3/4]: u = 1/4 lands on the boundary and goes
    to token 2, the largest u below 1/4 to token 0)."""
    rng = np.random.default_rng(3)
    w = rng.random(9).astype(np.float32) * 0.1
    w[[2, 5]] = 0.0
    G = 4096
    draws = np.array([oracle.fx_draw(w, np.float32((k + 0.5) / G)) for k in range(G)])
    freq = np.bincount(draws, minlength=w.size) / G
    share = w.astype(np.float64) / w.sum()
    assert np.max(np.abs(freq - share)) <= 1.0 / G + 1e-6
    assert freq[2] == 0 and freq[5] == 0
    assert oracle.fx_draw(w, 0.0) == 0
    assert oracle.fx_draw(w, np.nextafter(np.float32(1), np.float32(0))) == 8
    hand = np.array([0.25, 0.0, 0.75], np.float32)
    assert oracle.fx_draw(hand, np.float32(0.25)) == 2
    assert oracle.fx_draw(hand, np.nextafter(np.float32(0.25), np.float32(0))) == 0
    assert oracle.fx_draw(np.zeros(4, np.float32), 0.5) == -1


def _bitmaps(rng, nodes, L, N, m):
    W = (N + 63) // 64
    bm = np.zeros((nodes + 1, L, W), np.uint64)
    sets = [[set(rng.choice(N, m, replace=False).tolist()) for _ in range(L)] for _ in range(nodes + 1)]
    for v in range(nodes + 1):
        for l in range(L):
            for e in sets[v][l]:
                bm[v, l, e // 64] |= np.uint64(1) << np.uint64(e % 64)
    return bm, sets


def test_union_cost_against_set_unions_and_properties():
    """F(S) = sum_l |E_{l,s} u U_{v in S} E_{l,v}| by Python set unions; F monotone and
    submodular ([SpecFit] §3.2); R(S) - 1 additive over disjoint sets; best = the lowest index
    of the largest R/T by brute force."""
    rng = np.random.default_rng(8)
    nodes, L, N, m = 10, 6, 128, 8
    bm, sets = _bitmaps(rng, nodes, L, N, m)
    pv = rng.random(nodes)
    bcoef = np.sort(rng.random(nodes + 1)) * 5
    beta = 0.3
    subsets = np.array(rng.integers(0, 1 << nodes, size=400), np.uint32)
    subsets[:2] = [0, (1 << nodes) - 1]
    out = oracle.union_cost(bm, subsets, pv, bcoef, beta)
    for c, mask in enumerate(subsets.tolist()):
        members = [v for v in range(1, nodes + 1) if (mask >> (v - 1)) & 1]
        F = sum(len(set(sets[0][l]).union(*[sets[v][l] for v in members])) for l in range(L))
        assert out["F"][c] == F and out["size"][c] == len(members)
        assert abs(out["R"][c] - (1 + sum(pv[v - 1] for v in members))) < 1e-12
        assert abs(out["T"][c] - (bcoef[len(members)] + beta * F)) < 1e-12
    ratio = out["R"] / out["T"]
    assert out["best"] == int(np.argmax(ratio))
    assert out["F"][0] == L * m            # the root alone
    # bits beyond the pool name no node
    extra = oracle.union_cost(bm, np.array([subsets[5] | (1 << nodes) | (1 << 31)], np.uint32), pv, bcoef, beta)
    assert extra["F"][0] == out["F"][5] and extra["size"][0] == out["size"][5]
    # monotone, submodular
    for _ in range(200):
        a = int(rng.integers(0, 1 << nodes))
        b = a | int(rng.integers(0, 1 << nodes))
        v = int(rng.integers(0, nodes))
        sub = np.array([a, a | (1 << v), b, b | (1 << v)], np.uint32)
        F = oracle.union_cost(bm, sub, pv, bcoef, beta)["F"]
        assert F[1] >= F[0] and F[3] >= F[2] and F[2] >= F[0]
        assert F[1] - F[0] >= F[3] - F[2]
    # R - 1 is additive over disjoint subsets
    a, b = 0b0000011111, 0b1111100000
    R = oracle.union_cost(bm, np.array([a, b, a | b], np.uint32), pv, bcoef, beta)["R"]
    assert abs((R[2] - 1) - ((R[0] - 1) + (R[1] - 1))) < 1e-12


def test_union_cost_exhaustive_small_tree():
    """Every subset of a 5-node pool: F by set unions, and a bit pattern per expert word
    boundary (experts 63, 64, 127)."""
    L = 2
    sets = [[{63, 64}, {0}], [{127}, {0, 1}], [{64}, {2}], [{1, 2, 3}, {127}], [set(), {63}], [{100}, set()]]
    nodes = len(sets) - 1
    bm = np.zeros((nodes + 1, L, 2), np.uint64)
    for v in range(nodes + 1):
        for l in range(L):
            for e in sets[v][l]:
                bm[v, l, e // 64] |= np.uint64(1) << np.uint64(e % 64)
    subsets = np.arange(1 << nodes, dtype=np.uint32)
    out = oracle.union_cost(bm, subsets, np.full(nodes, 0.5), np.arange(nodes + 1, dtype=np.float64), 1.0)
    for mask in range(1 << nodes):
        members = [v for v in range(1, nodes + 1) if (mask >> (v - 1)) & 1]
        F = sum(len(set(sets[0][l]).union(*[sets[v][l] for v in members])) for l in range(L))
        assert out["F"][mask] == F
