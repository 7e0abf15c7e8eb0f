"""CPU oracle for the MoE verify-pass expert operation (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of ``bench.py``
import this package.  The product library never loads it, and the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 accumulation; every function
cites the passage of "Speculative Decoding for Mixture-of-Experts Models" (Lan) it
follows).  This module compiles it with gcc into ``oracle/_build/`` and wraps it with
ctypes and numpy arrays.  Parity of every function here is pinned by
``tests/test_oracle_pins.py``; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")

F32, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared object (gcc, -O2, no fast-math).  Returns its path."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", "-fopenmp",
                            "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.oracle_route_topm.argtypes = [P, I, I, I, I, P, P]
        lib.oracle_group_slots.argtypes = [P, I, I, I, P, P, P, P]
        lib.oracle_expert_op_perslot.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, I, P]
        lib.oracle_expert_op_dedup.argtypes = [I, I, I, I, I, I, P, P, P, P, P, I, I, P, P, P, P]
        lib.oracle_expert_op_token.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, I, P]
        lib.oracle_pass_bytes.argtypes = [I, I, I, I, I, I, P, I, P, P, P]
        lib.oracle_union_size.argtypes = [P, I, I, I, I, I]
        lib.oracle_reuse_estimate.argtypes = [P, I, I, I, I]
        lib.oracle_reuse_estimate.restype = D
        lib.oracle_expected_union.argtypes = [I, I, I]
        lib.oracle_expected_union.restype = D
        lib.oracle_expected_tokens.argtypes = [D, I]
        lib.oracle_expected_tokens.restype = D
        lib.oracle_best_draft_length.argtypes = [P, I, D]
        lib.oracle_crossover.argtypes = [P, P, I, I]
        lib.oracle_bandwidth_report.argtypes = [I, I, P, P, P, P, P, P, P, P, P, P]
        for name, args in (("oracle_throughput", [P, I, D]), ("oracle_first_threshold", [P]),
                           ("oracle_speedup", [P, I, D]), ("oracle_alpha", [P, I, I]),
                           ("oracle_convex_step_point", [P, I]), ("oracle_mean_reuse", [I, P, P, I, I]),
                           ("oracle_reuse_threshold", [I, D, D, D, D, D, D, D]),
                           ("oracle_reuse_threshold_bytes", [I, D, D, D, D]),
                           ("oracle_err_verify_factor", [D]), ("oracle_err_saving_bound", [D, D, D]),
                           ("oracle_err_regret_factor", [D])):
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = D
        lib.oracle_step_points.argtypes = [P, I, P]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = D
        lib.oracle_e4m3_encode.argtypes = [D]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_rows_e4m3.argtypes = [P, I, I, I, P, P]
        lib.oracle_expert_op_token_fp8.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P, I, P]
        lib.oracle_convex_nondecreasing.argtypes = [P, I]
        lib.oracle_err_decision_agrees.argtypes = [D, D, D]
        lib.oracle_err_kstar_separated.argtypes = [P, I, D, D]
        lib.oracle_err_speedup_interval.argtypes = [D, P, P]
        lib.oracle_spec_accept.argtypes = [P, P, P, P, P, I, I, I, I, P, P]
        lib.oracle_fx_draw.argtypes = [P, I, ctypes.c_float]
        lib.oracle_fx_draw.restype = ctypes.c_int32
        lib.oracle_union_cost.argtypes = [P, I, I, I, P, I, P, P, D, P, P, P, P, P]
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_set_threads(1)   # single-threaded unless a caller asks for more
        _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Threads of the expert-operation loops (OpenMP over output rows, which never changes a
    result bit).  Returns the count in force."""
    return int(_load().oracle_set_threads(int(n)))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _wcode(a: np.ndarray) -> int:
    """Weights/activations: float32 arrays are fp32, uint16 arrays hold bf16 bit patterns."""
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or bf16-as-uint16 arrays, got {a.dtype}")


def route_topm(logits: np.ndarray, m: int, renorm: bool = True):
    """Top-m routing: returns (ids int32 [n, m], gates float64 [n, m])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    n, N = logits.shape
    ids = np.zeros((n, m), np.int32)
    gates = np.zeros((n, m), np.float64)
    rc = _load().oracle_route_topm(_ptr(logits), n, N, m, int(bool(renorm)), _ptr(ids), _ptr(gates))
    if rc != 0:
        raise ValueError("oracle_route_topm: bad arguments or NaN logit")
    return ids, gates


def group_slots(ids: np.ndarray, N: int):
    """Counting sort of slots by expert: returns (U, expert_list[U], offsets[U+1], order[n*m])."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n, m = ids.shape
    cap = min(N, n * m)
    U = np.zeros(1, np.int32)
    lst = np.zeros(max(cap, 1), np.int32)
    off = np.zeros(cap + 1, np.int32)
    order = np.zeros(max(n * m, 1), np.int32)
    rc = _load().oracle_group_slots(_ptr(ids), n, m, N, _ptr(U), _ptr(lst), _ptr(off), _ptr(order))
    if rc != 0:
        raise ValueError("oracle_group_slots: expert id out of range")
    u = int(U[0])
    return u, lst[:u].copy(), off[:u + 1].copy(), order[:n * m].copy()


def _check_layer(wg, wu, wd, x):
    N, f, d = wg.shape
    assert wu.shape == (N, f, d) and wd.shape == (N, d, f) and x.shape[1] == d
    assert wg.dtype == wu.dtype == wd.dtype
    return N, f, d


def expert_op_perslot(wg, wu, wd, x, ids, gates):
    """Per-slot expert op + combine.  Weights [N,f,d],[N,f,d],[N,d,f]; x [n,d].  Returns y float64 [n,d]."""
    wg, wu, wd, x = (np.ascontiguousarray(a) for a in (wg, wu, wd, x))
    N, f, d = _check_layer(wg, wu, wd, x)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    n, m = ids.shape
    y = np.zeros((n, d), np.float64)
    rc = _load().oracle_expert_op_perslot(d, f, N, m, _wcode(wg), _wcode(x), _ptr(wg), _ptr(wu),
                                          _ptr(wd), _ptr(x), _ptr(ids), _ptr(gates), n, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_expert_op_perslot: expert id out of range")
    return y


def expert_op_dedup(wg, wu, wd, x, gates, m, grouping):
    """Deduplicating expert op + combine over a grouping (U, list, offsets, order)."""
    wg, wu, wd, x = (np.ascontiguousarray(a) for a in (wg, wu, wd, x))
    N, f, d = _check_layer(wg, wu, wd, x)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    n = gates.shape[0]
    U, lst, off, order = grouping
    lst = np.ascontiguousarray(lst, dtype=np.int32)
    off = np.ascontiguousarray(off, dtype=np.int32)
    order = np.ascontiguousarray(order, dtype=np.int32)
    y = np.zeros((n, d), np.float64)
    rc = _load().oracle_expert_op_dedup(d, f, N, m, _wcode(wg), _wcode(x), _ptr(wg), _ptr(wu),
                                        _ptr(wd), _ptr(x), _ptr(gates), n, int(U), _ptr(lst),
                                        _ptr(off), _ptr(order), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_expert_op_dedup: expert id out of range")
    return y


def expert_op_token(wg, wu, wd, x, ids, gates, t):
    """Layer output of token t alone (for spot checks of large passes).  Returns float64 [d]."""
    wg, wu, wd, x = (np.ascontiguousarray(a) for a in (wg, wu, wd, x))
    N, f, d = _check_layer(wg, wu, wd, x)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    m = ids.shape[1]
    y = np.zeros(d, np.float64)
    rc = _load().oracle_expert_op_token(d, f, N, m, _wcode(wg), _wcode(x), _ptr(wg), _ptr(wu),
                                        _ptr(wd), _ptr(x), _ptr(ids), _ptr(gates), int(t), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_expert_op_token: expert id out of range")
    return y


def pass_bytes(d, f, N, ids, w_dtype=BF16, x_dtype=BF16):
    """Bytes of one pass: dict(expert_bytes, slot_bytes, dedup_bytes, act_bytes, U, ubar)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n, m = ids.shape
    out = np.zeros(4, np.uint64)
    U = np.zeros(1, np.int32)
    ubar = np.zeros(1, np.float64)
    rc = _load().oracle_pass_bytes(d, f, N, m, w_dtype, x_dtype, _ptr(ids), n, _ptr(out), _ptr(U), _ptr(ubar))
    if rc != 0:
        raise ValueError("oracle_pass_bytes: expert id out of range")
    return dict(expert_bytes=int(out[0]), slot_bytes=int(out[1]), dedup_bytes=int(out[2]),
                act_bytes=int(out[3]), U=int(U[0]), ubar=float(ubar[0]))


def union_size(sets: np.ndarray, N: int, t0: int, n: int) -> int:
    sets = np.ascontiguousarray(sets, dtype=np.int32)
    T, m = sets.shape
    r = _load().oracle_union_size(_ptr(sets), T, m, N, t0, n)
    if r < 0:
        raise ValueError("oracle_union_size: bad arguments")
    return int(r)


def reuse_estimate(sets: np.ndarray, N: int, n: int) -> float:
    sets = np.ascontiguousarray(sets, dtype=np.int32)
    T, m = sets.shape
    return float(_load().oracle_reuse_estimate(_ptr(sets), T, m, N, n))


def expected_union(N: int, m: int, n: int) -> float:
    return float(_load().oracle_expected_union(N, m, n))


def expected_tokens(a: float, k: int) -> float:
    return float(_load().oracle_expected_tokens(float(a), int(k)))


def best_draft_length(V, a: float) -> int:
    V = np.ascontiguousarray(V, dtype=np.float64)
    return int(_load().oracle_best_draft_length(_ptr(V), len(V) - 1, float(a)))


def crossover(t_slot, t_dedup, n_lo: int):
    """Smallest n from which t_slot - t_dedup stays positive, or None."""
    t_slot = np.ascontiguousarray(t_slot, dtype=np.float64)
    t_dedup = np.ascontiguousarray(t_dedup, dtype=np.float64)
    n_hi = n_lo + len(t_slot) - 1
    r = _load().oracle_crossover(_ptr(t_slot), _ptr(t_dedup), n_lo, n_hi)
    return None if r < 0 else int(r)


def bandwidth_report(n_lo, slot_bytes, dedup_bytes, t_slot, t_dedup):
    """dict of beta_slot, beta_dedup, ubar, r, saving (arrays) and crossover (int or None)."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (slot_bytes, dedup_bytes, t_slot, t_dedup)]
    count = len(arrs[0])
    outs = [np.zeros(count, np.float64) for _ in range(5)]
    cross = np.zeros(1, np.int32)
    rc = _load().oracle_bandwidth_report(int(n_lo), count, *[_ptr(a) for a in arrs],
                                         *[_ptr(o) for o in outs], _ptr(cross))
    if rc != 0:
        raise ValueError("oracle_bandwidth_report: non-positive time or bytes")
    res = dict(zip(("beta_slot", "beta_dedup", "ubar", "r", "saving"), outs))
    res["crossover"] = None if cross[0] < 0 else int(cross[0])
    return res


# ---------------------------------------------------------------- step-time theory
def _V(V):
    return np.ascontiguousarray(V, dtype=np.float64)


def throughput(V, k: int, a: float) -> float:
    V = _V(V)
    return float(_load().oracle_throughput(_ptr(V), int(k), float(a)))


def first_threshold(V) -> float:
    V = _V(V)
    return float(_load().oracle_first_threshold(_ptr(V)))


def speedup(V, k: int, a: float) -> float:
    V = _V(V)
    return float(_load().oracle_speedup(_ptr(V), int(k), float(a)))


def alpha(V, k: int, i: int) -> float:
    V = _V(V)
    return float(_load().oracle_alpha(_ptr(V), int(k), int(i)))


def step_points(V) -> np.ndarray:
    """a_step[0..kmax], a_step[0] = 0 (B.31)."""
    V = _V(V)
    out = np.zeros(len(V), np.float64)
    if _load().oracle_step_points(_ptr(V), len(V) - 1, _ptr(out)) != 0:
        raise ValueError("oracle_step_points: kmax < 1 or a non-positive step time")
    return out


def convex_nondecreasing(V) -> bool:
    V = _V(V)
    return bool(_load().oracle_convex_nondecreasing(_ptr(V), len(V) - 1))


def convex_step_point(V, j: int) -> float:
    V = _V(V)
    return float(_load().oracle_convex_step_point(_ptr(V), int(j)))


def mean_reuse(w, rho, k: int) -> float:
    """rho_bar_k of (11): w [L], rho [L, jmax+1]."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    rho = np.ascontiguousarray(rho, dtype=np.float64)
    return float(_load().oracle_mean_reuse(len(w), _ptr(w), _ptr(rho), rho.shape[1] - 1, int(k)))


def reuse_threshold(k, a, mW, Bk, beta1, tau1, dD_bD=0.0, dphi=0.0) -> float:
    return float(_load().oracle_reuse_threshold(int(k), float(a), float(mW), float(Bk), float(beta1),
                                                float(tau1), float(dD_bD), float(dphi)))


def reuse_threshold_bytes(k, a, mW, D1=0.0, Dk1=0.0) -> float:
    return float(_load().oracle_reuse_threshold_bytes(int(k), float(a), float(mW), float(D1), float(Dk1)))


def err_verify_factor(eps) -> float:
    return float(_load().oracle_err_verify_factor(float(eps)))


def err_saving_bound(eps, Me_slot, Me_dedup) -> float:
    return float(_load().oracle_err_saving_bound(float(eps), float(Me_slot), float(Me_dedup)))


def err_decision_agrees(r, ubar, eps) -> bool:
    return bool(_load().oracle_err_decision_agrees(float(r), float(ubar), float(eps)))


def err_regret_factor(delta) -> float:
    return float(_load().oracle_err_regret_factor(float(delta)))


def err_kstar_separated(V, a, delta) -> bool:
    V = _V(V)
    return bool(_load().oracle_err_kstar_separated(_ptr(V), len(V) - 1, float(a), float(delta)))


def err_speedup_interval(delta):
    lo = np.zeros(1, np.float64)
    hi = np.zeros(1, np.float64)
    _load().oracle_err_speedup_interval(float(delta), _ptr(lo), _ptr(hi))
    return float(lo[0]), float(hi[0])


# ---------------------------------------------------------------- operation-time fits
def fit_slot(n, U, t, m: int, b: float):
    """Least-squares fit (4) of the per-slot operation time on passes with chosen ids
    [Lan, §2 "Effective bandwidth"]: t = t_op + c_u U b + c_re (n m - U) b.
    Returns (t_op, c_u, c_re)."""
    n, U, t = (np.asarray(v, dtype=np.float64) for v in (n, U, t))
    A = np.stack([np.ones_like(U), U * b, (n * m - U) * b], axis=1)
    coef, *_ = np.linalg.lstsq(A, t, rcond=None)
    return tuple(float(c) for c in coef)


def fit_dedup(n, U, t, b: float):
    """Least-squares fit (E.1) of the deduplicating operation time on passes with chosen ids
    [Lan, App. E "Deduplicating fit"]: t = t_op + c_g U b + c_t n.  Returns (t_op, c_g, c_t)."""
    n, U, t = (np.asarray(v, dtype=np.float64) for v in (n, U, t))
    A = np.stack([np.ones_like(U), U * b, n], axis=1)
    coef, *_ = np.linalg.lstsq(A, t, rcond=None)
    return tuple(float(c) for c in coef)


def fit_error(predicted, measured) -> float:
    """A fit's error on windows of recorded routing [Lan, §4: the median relative error of
    the fit's time on the windows it did not see]."""
    p, q = np.asarray(predicted, np.float64), np.asarray(measured, np.float64)
    return float(np.median(np.abs(p - q) / q))


# ---------------------------------------------------------------- FP8 (e4m3) experts
def e4m3_decode(c: int) -> float:
    return float(_load().oracle_e4m3_decode(int(c)))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def quantize_rows_e4m3(src: np.ndarray):
    """src [rows, cols] float32 or bf16-as-uint16 -> (codes uint8 [rows, cols], scale float32 [rows])."""
    src = np.ascontiguousarray(src)
    rows, cols = src.shape
    q = np.zeros((rows, cols), np.uint8)
    sc = np.zeros(rows, np.float32)
    _load().oracle_quantize_rows_e4m3(_ptr(src), _wcode(src), rows, cols, _ptr(q), _ptr(sc))
    return q, sc


def expert_op_token_fp8(wg, wu, wd, sg, su, sd, x, sx, ids, gates, t):
    """y_t [d] of the e4m3 expert operation; weights [E, f, d] / [E, d, f] uint8 codes with
    row scales [E, f] / [E, d]; x [n, d] codes with row scales sx [n]; ids index the E experts."""
    E, f, d = wg.shape
    arrs = [np.ascontiguousarray(a) for a in (wg, wu, wd)]
    scs = [np.ascontiguousarray(a, dtype=np.float32) for a in (sg, su, sd)]
    x = np.ascontiguousarray(x, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    y = np.zeros(d, np.float64)
    rc = _load().oracle_expert_op_token_fp8(d, f, E, ids.shape[1], *[_ptr(a) for a in arrs],
                                            *[_ptr(a) for a in scs], _ptr(x), _ptr(sx), _ptr(ids),
                                            _ptr(gates), int(t), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_expert_op_token_fp8: bad arguments")
    return y


# ---------------------------------------------------------------- verify-side neighbours
def spec_accept(draft, q, p, r, u, greedy: bool = False):
    """One round of speculative sampling for B sequences ("Lossless but Not Free", §3.1,
    Algorithm 1).  draft [B, K] int32, q [B, K, V] and p [B, K+1, V] float32, r [B, K] and
    u [B] float32 uniforms.  Returns (n_accepted int32 [B], token int32 [B])."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    B, K1, V = p.shape
    K = K1 - 1
    draft = np.ascontiguousarray(np.asarray(draft, np.int32).reshape(B, K))
    dummy = np.zeros(1, np.float32)
    # the greedy rule reads neither q nor the draws
    q = dummy if (q is None or K == 0) else np.ascontiguousarray(np.asarray(q, np.float32).reshape(B, K, V))
    r = dummy if (r is None or K == 0) else np.ascontiguousarray(np.asarray(r, np.float32).reshape(B, K))
    u = np.zeros(B, np.float32) if u is None else np.ascontiguousarray(np.asarray(u, np.float32).reshape(B))
    if not greedy and K and (q is dummy or r is dummy):
        raise ValueError("spec_accept: sampling needs q and r")
    na = np.zeros(B, np.int32)
    tok = np.zeros(B, np.int32)
    rc = _load().oracle_spec_accept(_ptr(draft) if K else _ptr(np.zeros(1, np.int32)), _ptr(q), _ptr(p), _ptr(r),
                                    _ptr(u), B, K, V, int(bool(greedy)), _ptr(na), _ptr(tok))
    if rc != 0:
        raise ValueError("oracle_spec_accept: bad arguments")
    return na, tok


def fx_draw(w, u: float) -> int:
    """The fixed-point inverse-CDF draw alone (weights clamped to [0, 1]); -1 if all zero."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    return int(_load().oracle_fx_draw(_ptr(w), int(w.size), float(u)))


def union_cost(bitmaps, subsets, pv, bcoef, beta: float):
    """SpecFit §3.2 eqs (3)-(5): bitmaps uint64 [nodes+1, L, W] (node 0 the root), subsets
    uint32 [S] node masks.  Returns dict(F, size, R, T, best)."""
    bm = np.ascontiguousarray(bitmaps, dtype=np.uint64)
    nodes1, L, W = bm.shape
    sub = np.ascontiguousarray(subsets, dtype=np.uint32).reshape(-1)
    pv = np.ascontiguousarray(pv, dtype=np.float64).reshape(nodes1 - 1) if nodes1 > 1 else np.zeros(1)
    bc = np.ascontiguousarray(bcoef, dtype=np.float64)
    S = sub.size
    F = np.zeros(S, np.int32)
    size = np.zeros(S, np.int32)
    R = np.zeros(S, np.float64)
    T = np.zeros(S, np.float64)
    best = np.zeros(1, np.int32)
    rc = _load().oracle_union_cost(_ptr(bm), nodes1 - 1, L, W, _ptr(sub) if S else _ptr(np.zeros(1, np.uint32)), S,
                                   _ptr(pv), _ptr(bc), float(beta), _ptr(F), _ptr(size), _ptr(R), _ptr(T), _ptr(best))
    if rc != 0:
        raise ValueError("oracle_union_cost: bad arguments")
    return dict(F=F, size=size, R=R, T=T, best=int(best[0]))
