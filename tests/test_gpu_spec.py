"""Parity of the verify-side kernels with the oracle, bit for bit.

moe_spec_accept (speculative sampling, "Lossless but Not Free" §3.1-3.2): accepted counts and
emitted tokens equal the oracle's on the same inputs and draws, in sampling and greedy mode, for
vocabularies from 1 to the Qwen3 vocabulary (151,936, several clusters' worth of ragged
segments), K from 0 to 31, and the edge cases the readings define.  moe_union_cost (SpecFit
§3.2 eqs (3)-(5)): F, |S|, R, T and the best index equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from moe_speculative_decoding_gb300 import api

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _softmax(z):
    z = z - z.max(-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def _case(seed, B, K, V, sharp=2.0, agree=0.7):
    """Target p and draft q distributions with overlapping mass; drafts sampled from q."""
    rng = np.random.default_rng(seed)
    zt = rng.normal(scale=sharp, size=(B, K + 1, V))
    zd = agree * zt[:, :K] + (1 - agree) * rng.normal(scale=sharp, size=(B, K, V))
    p, q = _softmax(zt), _softmax(zd)
    cq = np.cumsum(q.astype(np.float64), -1)
    draft = np.empty((B, K), np.int32)
    for b in range(B):
        for i in range(K):
            draft[b, i] = min(V - 1, int(np.searchsorted(cq[b, i], rng.random() * cq[b, i, -1], side="right")))
    r = rng.random((B, K)).astype(np.float32)
    u = rng.random(B).astype(np.float32)
    return draft, q, p, r, u


def _gpu(draft, q, p, r, u, greedy=False):
    t = lambda a, dt: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    na, tok = api.spec_accept(t(draft, None), t(q, None), t(p, None), t(r, None), t(u, None), greedy=greedy)
    torch.cuda.synchronize()
    return na.cpu().numpy(), tok.cpu().numpy()


# V % 4 = 0 runs the float4 loads (up to the largest vocabularies: 151936, 240000), the
# other V the scalar loads
@pytest.mark.parametrize("B,K,V", [(37, 5, 1000), (8, 0, 4097), (5, 31, 257), (16, 8, 32000), (3, 1, 1),
                                   (16, 8, 151936), (64, 3, 7), (3, 3, 240000)])
def test_sampling_matches_oracle(B, K, V):
    draft, q, p, r, u = _case(B * 1000 + K * 10 + V % 97, B, K, V)
    na_o, tok_o = oracle.spec_accept(draft, q, p, r, u)
    na_g, tok_g = _gpu(draft, q, p, r, u)
    assert np.array_equal(na_g, na_o)
    assert np.array_equal(tok_g, tok_o)
    if K:
        assert 0 < na_o.sum() < B * K or B < 4   # the cases exercise both outcomes


@pytest.mark.parametrize("B,K,V", [(37, 5, 1000), (16, 8, 151936), (4, 31, 300), (6, 0, 50), (3, 3, 240000)])
def test_greedy_matches_oracle(B, K, V):
    draft, q, p, r, u = _case(7 + B + K, B, K, V)
    am = p.argmax(-1)
    rng = np.random.default_rng(3)
    lead = rng.integers(0, K + 1, size=B)
    for b in range(B):
        draft[b, :lead[b]] = am[b, :lead[b]]
    na_o, tok_o = oracle.spec_accept(draft, None, p, None, None, greedy=True)
    na_g, tok_g = _gpu(draft, None, p, None, None, greedy=True)
    assert np.array_equal(na_g, na_o) and np.array_equal(tok_g, tok_o)
    first_miss = [next((i for i in range(K) if draft[b, i] != am[b, i]), K) for b in range(B)]
    assert np.array_equal(na_o, first_miss) and np.all(na_o >= lead)


def test_edge_cases_match_oracle():
    """q(x) = 0 drafts, ids outside [0, V), p = q rows (all-zero adjusted weights: the draw
    falls back to p), an all-zero bonus row (argmax), draws at u = 0 and just below 1, ties in
    the greedy argmax (lowest index)."""
    B, K, V = 12, 3, 600
    draft, q, p, r, u = _case(99, B, K, V)
    q[0, 0, draft[0, 0]] = 0.0                      # accepted iff p > 0
    draft[1, 0] = V                                 # rejected
    draft[2, 1] = -5
    q[3, 0] = p[3, 0]; r[3, 0] = 1.0                # rejected at a row with p = q
    p[4, K] = 0.0; r[4] = 0.0                       # all accepted, bonus row all zero
    u[5] = 0.0
    u[6] = np.nextafter(np.float32(1), np.float32(0))
    p[7, :, 10] = p[7, :, 20] = p[7].max() + 1      # ties for the argmax
    na_o, tok_o = oracle.spec_accept(draft, q, p, r, u)
    na_g, tok_g = _gpu(draft, q, p, r, u)
    assert np.array_equal(na_g, na_o) and np.array_equal(tok_g, tok_o)
    assert na_o[1] == 0 and na_o[2] <= 1 and na_o[3] == 0 and tok_o[4] == 0
    na_o, tok_o = oracle.spec_accept(draft, None, p, None, None, greedy=True)
    na_g, tok_g = _gpu(draft, None, p, None, None, greedy=True)
    assert np.array_equal(na_g, na_o) and np.array_equal(tok_g, tok_o)
    assert tok_o[7] == 10 or na_o[7] > 0


def test_draws_match_over_a_u_grid():
    """The emitted token for 512 evenly spaced u on one rejected row: every draw equal."""
    B, K, V = 512, 1, 20000
    draft, q, p, r, u = _case(5, 1, K, V)
    draft = np.repeat(draft, B, 0); q = np.repeat(q, B, 0); p = np.repeat(p, B, 0)
    r = np.ones((B, K), np.float32) * np.float32(0.999999)
    u = ((np.arange(B) + 0.5) / B).astype(np.float32)
    na_o, tok_o = oracle.spec_accept(draft, q, p, r, u)
    na_g, tok_g = _gpu(draft, q, p, r, u)
    assert np.array_equal(na_g, na_o) and np.array_equal(tok_g, tok_o)
    assert len(np.unique(tok_o)) > 50


def _pool(seed, nodes, L, N, m):
    rng = np.random.default_rng(seed)
    W = (N + 63) // 64
    bm = np.zeros((nodes + 1, L, W), np.uint64)
    for v in range(nodes + 1):
        for l in range(L):
            for e in rng.choice(N, m, replace=False):
                bm[v, l, e // 64] |= np.uint64(1) << np.uint64(e % 64)
    pv = rng.random(nodes)
    bcoef = np.sort(rng.random(nodes + 1)) * 3
    return bm, pv, bcoef


@pytest.mark.parametrize("nodes,L,N,m,S", [(18, 48, 128, 8, 20000), (10, 27, 64, 6, 1 << 10), (32, 4, 200, 5, 3000),
                                           (7, 9, 128, 4, 500), (12, 400, 128, 6, 800), (0, 3, 64, 2, 1)])
def test_union_cost_matches_oracle(nodes, L, N, m, S):
    # L*W even with the node-triple table (18/48, 32/4, 7/9), odd (10/27, 0/3), and even with a
    # table too large for shared memory beside the bitmaps (12/400: the broadcast node loop)
    bm, pv, bcoef = _pool(nodes * 7 + L, nodes, L, N, m)
    rng = np.random.default_rng(1)
    if S == 1 << nodes:
        subsets = np.arange(S, dtype=np.uint32)
    else:
        subsets = rng.integers(0, 1 << 32, size=S, dtype=np.uint64).astype(np.uint32)
    ref = oracle.union_cost(bm, subsets, pv, bcoef, 0.37)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = api.union_cost(t(bm.view(np.int64)), t(subsets.view(np.int32)), t(pv) if nodes else None, t(bcoef), 0.37)
    torch.cuda.synchronize()
    assert np.array_equal(out["F"].cpu().numpy(), ref["F"])
    assert np.array_equal(out["size"].cpu().numpy(), ref["size"])
    assert np.array_equal(out["R"].cpu().numpy(), ref["R"])
    assert np.array_equal(out["T"].cpu().numpy(), ref["T"])
    assert int(out["best"].item()) == ref["best"]

def test_union_cost_negative_costs():
    """Negative b coefficients make every T negative: the best is still the oracle's (its first
    subset, then any strictly larger R/T)."""
    bm, pv, bcoef = _pool(3, 9, 12, 128, 6)
    bcoef = bcoef - 50.0
    subsets = np.random.default_rng(2).integers(0, 1 << 9, size=700, dtype=np.uint64).astype(np.uint32)
    ref = oracle.union_cost(bm, subsets, pv, bcoef, 0.01)
    assert (ref["T"] < 0).all()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out = api.union_cost(t(bm.view(np.int64)), t(subsets.view(np.int32)), t(pv), t(bcoef), 0.01)
    torch.cuda.synchronize()
    assert np.array_equal(out["F"].cpu().numpy(), ref["F"])
    assert np.array_equal(out["T"].cpu().numpy(), ref["T"])
    assert int(out["best"].item()) == ref["best"]
