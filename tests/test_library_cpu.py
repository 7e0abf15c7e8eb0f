"""The C-ABI library on the CPU: it builds, loads, exports every declared symbol, and its
host-only calls (bytes, report math) agree with the oracle.  No kernel is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT, load_golden
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300 import build as mbuild


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return api.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe_verify.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(api.EXPORTED)
    assert lib.moe_abi_version() == 2


def test_status_strings(lib):
    for code in range(7):
        assert len(lib.moe_status_str(code)) > 0
    assert lib.moe_status_str(99) == b"unknown status"


def test_argument_validation_before_any_launch(lib):
    """Invalid arguments are rejected on the host, before anything touches the GPU."""
    st = lib.moe_route_topm(None, 4, 8, 2, 1, None, None, None)
    assert st == 1  # MOE_ERR_ARG
    assert lib.moe_route_topm(None, 4, 8, 9, 1, None, None, None) == 2   # m > N
    assert lib.moe_route_topm(None, 4, 2048, 2, 1, None, None, None) == 2  # N > 1024
    assert lib.moe_group_slots(None, 64, 128, 8, None, None, None, None, None, None) == 2  # > 4096 slots
    L = api.make_layer(2048, 768, 128, 8)
    bad = api.make_layer(2048, 700, 128, 8)   # f not a multiple of 64
    args = [None] * 6
    assert lib.moe_expert_op_perslot(ctypes.byref(bad), *args, 4, 0, None, None, 0, None) == 2
    # n above the pass limit (64) is unsupported in every form; up to 64 the null pointers are
    # the error (the per-slot calls split 17..64 into launches of up to 16 tokens, the
    # deduplicating ones take them in one launch)
    assert lib.moe_expert_op_perslot(ctypes.byref(L), *args, 65, 0, None, None, 0, None) == 2
    assert lib.moe_expert_op_perslot(ctypes.byref(L), *args, 17, 0, None, None, 0, None) == 1
    assert lib.moe_expert_op_perslot(ctypes.byref(L), *args, 64, 0, None, None, 0, None) == 1
    assert lib.moe_expert_op_dedup_ids(ctypes.byref(L), *args, 17, 0, None, None, 0, None) == 1
    assert lib.moe_expert_op_dedup_ids(ctypes.byref(L), *args, 64, 0, None, None, 0, None) == 1
    assert lib.moe_expert_op_dedup_ids(ctypes.byref(L), *args, 65, 0, None, None, 0, None) == 2
    assert lib.moe_expert_op_dedup(ctypes.byref(L), *[None] * 5, 65, *[None] * 4, 0, None, None, 0, None) == 2
    # null pointers
    assert lib.moe_expert_op_perslot(ctypes.byref(L), *args, 4, 0, None, None, 0, None) == 1
    mixed = api.Layer(2048, 768, 128, 8, 1, 0, 0)   # bf16 weights with fp32 x
    assert lib.moe_expert_op_dedup(ctypes.byref(mixed), *[None] * 5, 4, *[None] * 4, 0, None, None, 0,
                                   None) == 2
    assert lib.moe_workspace_init(None, 256, None) == 4


def test_workspace_bytes(lib):
    """256 header bytes, plus for the tensor-core path its flag region (4 words per CTA for
    the zeroing of y, 256 CTAs) and 3 CTA shares x 128 tagged 64-bit partial sums (value and
    the call's ticket) per (slot, 64-row f tile): the gate/up shares' hand-off to the h formers."""
    r256 = lambda b: (b + 255) // 256 * 256
    for (d, f, N, m) in [(2048, 768, 128, 8), (2048, 1408, 64, 6), (4096, 14336, 8, 2), (256, 128, 8, 2)]:
        L = api.make_layer(d, f, N, m, "bf16")
        flags = r256(256 * 4 * 4)
        for n in (1, 5, 16, 17, 40, 64):
            part = n * m * (f // 64) * 3 * 128 * 8
            # a pass of more than 256 slots keeps its grouping (count, N ids, N + 1 offsets,
            # n*m slots) for the deduplicating call from ids
            grouping = r256(4 * (2 * N + n * m + 2)) if n * m > 256 else 0
            assert lib.moe_workspace_bytes(ctypes.byref(L), n) == 256 + flags + r256(part) + grouping
        # passes cap at MOE_MAX_PASS_TOKENS
        assert lib.moe_workspace_bytes(ctypes.byref(L), 100) == lib.moe_workspace_bytes(ctypes.byref(L), 64)
    assert lib.moe_workspace_bytes(ctypes.byref(api.make_layer(2048, 768, 128, 8)), 16) == 256 + 4096 + 4718592
    # the SIMT kernel and fp32 layers keep only the header
    assert lib.moe_workspace_bytes(ctypes.byref(api.make_layer(256, 512, 8, 2, "f32")), 16) == 256
    assert lib.moe_workspace_bytes(ctypes.byref(api.make_layer(256, 512, 8, 2, "bf16", simt=True)), 16) == 256
    assert lib.moe_workspace_bytes(None, 16) == 256


def test_noalloc_rejects_layers_beyond_its_scratch(lib):
    """The 32 MiB library scratch holds 22 MB for d=4096, f=14336, top-2 at 16 tokens; a
    layer needing more is refused before any device work (no GPU needed for that)."""
    fn = lib.moe_expert_op_perslot_noalloc
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(api.Layer), P, P, P, P, P, P, I32, I32, P, P, P]
    fn.restype = I32
    # aligned stand-in addresses: every check runs on the host, before any CUDA call (there
    # is no GPU here, so a call that reached the device would return MOE_ERR_CUDA)
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(7)]
    big = api.make_layer(4096, 65536, 128, 64)   # 16 * 64 * 1024 * 3072 bytes of partial sums
    assert lib.moe_workspace_bytes(ctypes.byref(big), 16) > 32 << 20
    assert fn(ctypes.byref(big), *fake[:6], 16, 0, fake[6], None, None) == 4   # MOE_ERR_WORKSPACE
    assert fn(None, *fake[:6], 1, 0, fake[6], None, None) == 1
    # invalid layers and arguments get the workspace call's statuses, also before any CUDA call
    assert fn(ctypes.byref(api.make_layer(256, 128, 2, 3)), *fake[:6], 1, 0, fake[6], None, None) == 2   # m > N
    assert fn(ctypes.byref(api.make_layer(256, 96, 8, 2)), *fake[:6], 1, 0, fake[6], None, None) == 2    # f % 64
    assert fn(ctypes.byref(api.make_layer(256, 128, 8, 2)), *fake[:6], 65, 0, fake[6], None, None) == 2  # n > 64
    assert fn(ctypes.byref(api.make_layer(256, 128, 8, 2)), *fake[:6], 0, 0, fake[6], None, None) == 1   # n < 1
    assert fn(ctypes.byref(api.make_layer(256, 128, 8, 2)), *fake[:3], None, *fake[4:6], 1, 0, fake[6],
              None, None) == 1   # x missing
    # a CUDA-core layer needs the header alone, however large its tensor-core flag region would be
    wide = api.make_layer(64, 65536, 24, 22, "bf16", simt=True)
    assert lib.moe_workspace_bytes(ctypes.byref(wide), 16) == 256
    mixtral = api.make_layer(4096, 14336, 8, 2)
    assert lib.moe_workspace_bytes(ctypes.byref(mixtral), 16) <= 32 << 20


def test_pass_bytes_matches_oracle(lib, oracle_mod):
    rng = np.random.default_rng(40)
    for (d, f, N, m, dt) in [(2048, 768, 128, 8, "bf16"), (2048, 1408, 64, 6, "bf16"),
                             (4096, 14336, 8, 2, "bf16"), (256, 512, 8, 2, "f32"), (2048, 768, 128, 8, "e4m3")]:
        L = api.make_layer(d, f, N, m, dt)
        for n in (1, 3, 8, 16):
            sets, _ = synth.routing_traces(1, n, N, m, float(rng.uniform(0, 1)), seed=int(rng.integers(1e9)))
            ids = sets[0]
            got = api.pass_bytes(L, ids)
            code = {"bf16": 1, "f32": 0, "e4m3": 2}[dt]
            ref = oracle_mod.pass_bytes(d, f, N, ids, code, code)
            for k in ("expert_bytes", "slot_bytes", "dedup_bytes", "act_bytes", "U"):
                assert got[k] == ref[k], k
            assert got["ubar"] == ref["ubar"]
    with pytest.raises(api.MoeError):
        api.pass_bytes(api.make_layer(256, 512, 8, 2, "f32"), np.array([[0, 8]], np.int32))


def test_bandwidth_report_matches_oracle(lib, oracle_mod):
    rng = np.random.default_rng(41)
    for _ in range(50):
        k = int(rng.integers(1, 17))
        sb = rng.uniform(1e7, 1e9, k)
        db = sb * rng.uniform(0.2, 1.0, k)
        ts = rng.uniform(1e-6, 1e-3, k)
        td = ts * rng.uniform(0.5, 1.5, k)
        got = api.bandwidth_report(1, sb, db, ts, td)
        ref = oracle_mod.bandwidth_report(1, sb, db, ts, td)
        for key in ("beta_slot", "beta_dedup", "ubar", "r", "saving"):
            assert np.allclose(got[key], ref[key], rtol=1e-15, atol=0), key
        assert got["crossover"] == ref["crossover"]
    g = load_golden("table1_effective_bandwidth.json")
    for row in g["rows"]:
        _, _, bs, bd, r, u = row[:6]
        rep = api.bandwidth_report(2, [1e9], [u * 1e9], [1e9 / bs], [u * 1e9 / bd])
        assert abs(rep["r"][0] - r) <= g["rounding"]


def test_expected_union_and_best_draft_length_match_oracle(lib, oracle_mod):
    for (N, m) in [(128, 8), (64, 6), (8, 2), (4, 2)]:
        for n in range(0, 17):
            assert abs(api.expected_union(N, m, n) - oracle_mod.expected_union(N, m, n)) < 1e-12
    g = load_golden("staircase_jump.json")
    for a, kstar in g["cases"]:
        assert api.best_draft_length(g["V"], a) == kstar
    rng = np.random.default_rng(42)
    for _ in range(200):
        V = rng.uniform(0.2, 5.0, size=int(rng.integers(1, 10)))
        a = float(rng.uniform(0, 0.99))
        assert api.best_draft_length(V, a) == oracle_mod.best_draft_length(V, a)
    with pytest.raises(api.MoeError):
        api.best_draft_length([1.0, -1.0], 0.5)


# ------------------------------------------------------------------ step-time theory (host)

def _rand_V(rng, kmax):
    if rng.random() < 0.5:
        c = np.sort(rng.uniform(0.0, 1.0, kmax))
        v0 = rng.uniform(0.5, 2.0)
        return np.concatenate([[v0], v0 + np.cumsum(c)])
    return rng.uniform(0.2, 3.0, kmax + 1)


def test_staircase_matches_oracle(lib, oracle_mod):
    rng = np.random.default_rng(60)
    for _ in range(300):
        kmax = int(rng.integers(1, 9))
        V = _rand_V(rng, kmax)
        got = api.staircase(V)
        assert np.allclose(got["a_step"], oracle_mod.step_points(V), rtol=0, atol=1e-12)
        for k in range(1, kmax + 1):
            for i in range(k):
                assert abs(got["alpha"][k, i] - oracle_mod.alpha(V, k, i)) <= 1e-12
        assert got["a0"] == oracle_mod.first_threshold(V)
        assert got["convex"] == oracle_mod.convex_nondecreasing(V)
        for a in rng.uniform(0, 1, 3):
            for k in range(kmax + 1):
                assert api.speedup(V, k, a) == pytest.approx(oracle_mod.speedup(V, k, a), rel=1e-14)
    g = load_golden("staircase_jump.json")
    st = api.staircase(g["V"])
    assert st["a_step"][1] == pytest.approx((5 ** 0.5 - 1) / 2, abs=1e-14) and st["alpha"][1, 0] == 1.0


def test_reuse_thresholds_match_oracle(lib, oracle_mod):
    rng = np.random.default_rng(61)
    for _ in range(300):
        k, a = int(rng.integers(1, 9)), float(rng.uniform(0, 1))
        args = [float(x) for x in (rng.uniform(1, 10), rng.uniform(0.3, 3), rng.uniform(0.3, 3), rng.uniform(1, 20),
                                   rng.uniform(0, 2), rng.uniform(-1, 1))]
        assert api.reuse_threshold(k, a, *args) == pytest.approx(oracle_mod.reuse_threshold(k, a, *args), rel=1e-13, abs=1e-13)
        mW, D1 = float(rng.uniform(1, 10)), float(rng.uniform(0, 5))
        Dk1 = D1 + float(rng.uniform(0, 3))
        assert api.reuse_threshold_bytes(k, a, mW, D1, Dk1) == pytest.approx(
            oracle_mod.reuse_threshold_bytes(k, a, mW, D1, Dk1), rel=1e-13, abs=1e-13)
    g = load_golden("no_single_threshold.json")
    a = g["a"][0] / g["a"][1]
    for k, (p, q) in zip((1, 2), g["rho_star"]):
        assert api.reuse_threshold_bytes(k, a, 1.0) == pytest.approx(p / q, abs=1e-15)
    assert np.isnan(api.reuse_threshold_bytes(0, a, 1.0)) and np.isnan(api.reuse_threshold(1, 1.0, 1, 1, 1, 1))


def test_error_bounds_and_separation_match_oracle(lib, oracle_mod):
    rng = np.random.default_rng(62)
    for eps in (0.0, 0.05, 0.1, 0.3, 0.49):
        b = api.error_bounds(eps)
        d = oracle_mod.err_verify_factor(eps)
        assert b["delta"] == pytest.approx(d, rel=1e-15) and b["verify_factor"] == pytest.approx(d, rel=1e-15)
        assert b["regret_factor"] == pytest.approx(oracle_mod.err_regret_factor(d), rel=1e-14)
        lo, hi = oracle_mod.err_speedup_interval(d)
        assert b["speedup_lo"] == pytest.approx(lo, rel=1e-14) and b["speedup_hi"] == pytest.approx(hi, rel=1e-14)
        for _ in range(20):
            r, u = float(rng.uniform(0.2, 1.5)), float(rng.uniform(0.2, 1.0))
            assert (abs(np.log(r) - np.log(u)) > b["decision_log_margin"]) == oracle_mod.err_decision_agrees(r, u, eps)
    for _ in range(200):
        V = _rand_V(rng, int(rng.integers(1, 8)))
        a, delta = float(rng.uniform(0, 1)), float(rng.uniform(0, 0.3))
        assert api.kstar_separated(V, a, delta) == oracle_mod.err_kstar_separated(V, a, delta)
    with pytest.raises(api.MoeError):
        api.error_bounds(0.5)
    with pytest.raises(api.MoeError):
        api.staircase([1.0])
    with pytest.raises(api.MoeError):
        api.staircase([1.0, -2.0])


def test_fit_op_times_matches_oracle(lib, oracle_mod):
    rng = np.random.default_rng(63)
    m, b = 8, 9.437184e6
    for _ in range(50):
        n = np.repeat(np.arange(2, 17), 4)
        U = np.array([int(rng.integers(m, min(128, k * m) + 1)) for k in n])
        t = 1e-5 + 1.3e-13 * U * b + 0.4e-13 * (n * m - U) * b
        t = t * (1 + rng.normal(0, 0.03, t.size))
        for form, fit in (("slot", lambda: oracle_mod.fit_slot(n, U, t, m, b)), ("dedup", lambda: oracle_mod.fit_dedup(n, U, t, b))):
            got, want = api.fit_op_times(n, U, t, m, b, form), fit()
            for g_, w_ in zip(got, want):
                assert g_ == pytest.approx(w_, rel=1e-7, abs=1e-22)
    with pytest.raises(api.MoeError):
        api.fit_op_times([2, 2, 2], [8, 8, 8], [1.0, 1.0, 1.0], m, b, "slot")   # rank 1


def test_fp8_entry_points_validate(lib):
    """e4m3 layers need the _fp8 calls (their scales); bf16 layers are refused there; NULL
    scales or misaligned pointers are argument errors - all before any device work."""
    P = ctypes.c_void_p
    L8 = api.make_layer(2048, 768, 128, 8, "e4m3")
    Lb = api.make_layer(2048, 768, 128, 8, "bf16")
    fake = P(1 << 20)   # aligned, never dereferenced: validation fails first
    ws = P(1 << 21)
    wsb = lib.moe_workspace_bytes(ctypes.byref(L8), 16)
    assert wsb == lib.moe_workspace_bytes(ctypes.byref(Lb), 16)
    sc = api.WeightScales(fake, fake, fake)
    args = (fake, fake, fake)
    # plain call with an e4m3 layer
    assert lib.moe_expert_op_perslot(ctypes.byref(L8), *args, fake, fake, fake, 4, 0, fake, ws, wsb, None) == 2
    # fp8 call with a bf16 layer
    assert lib.moe_expert_op_perslot_fp8(ctypes.byref(Lb), *args, ctypes.byref(sc), fake, fake, fake, fake, 4, 0,
                                         fake, ws, wsb, None) == 2
    # missing scales
    assert lib.moe_expert_op_perslot_fp8(ctypes.byref(L8), *args, None, fake, fake, fake, fake, 4, 0, fake, ws,
                                         wsb, None) == 1
    bad = api.WeightScales(fake, None, fake)
    assert lib.moe_expert_op_dedup_fp8(ctypes.byref(L8), *args, ctypes.byref(bad), fake, fake, fake, 4, fake, fake,
                                       fake, fake, 0, fake, ws, wsb, None) == 1
    # e4m3 needs d and f multiples of 128
    L8b = api.make_layer(2048, 704, 128, 8, "e4m3")
    assert lib.moe_expert_op_perslot_fp8(ctypes.byref(L8b), *args, ctypes.byref(sc), fake, fake, fake, fake, 4, 0,
                                         fake, ws, wsb, None) == 2
    assert lib.moe_quantize_rows_e4m3(None, 1, 4, 64, None, None, None) == 1
    assert lib.moe_quantize_rows_e4m3(fake, 7, 4, 64, fake, fake, None) == 1
    assert lib.moe_quantize_rows_e4m3(None, 1, 0, 64, None, None, None) == 0


def test_verify_side_calls_validate_on_the_host(lib):
    """moe_spec_accept and moe_union_cost reject bad sizes and pointers before any device work."""
    P = ctypes.c_void_p
    good = P(64)
    # K above one warp's walk, V above the fixed-point range
    assert lib.moe_spec_accept(good, good, good, good, good, 4, 32, 1000, 0, good, good, None) == 2
    assert lib.moe_spec_accept(good, good, good, good, good, 4, 8, 262145, 0, good, good, None) == 2
    assert lib.moe_spec_accept(good, good, good, good, good, -1, 8, 1000, 0, good, good, None) == 1
    assert lib.moe_spec_accept(good, good, good, good, good, 4, 8, 0, 0, good, good, None) == 1
    assert lib.moe_spec_accept(None, None, None, None, None, 0, 8, 1000, 0, None, None, None) == 0   # B == 0
    assert lib.moe_spec_accept(good, good, None, good, good, 4, 8, 1000, 0, good, good, None) == 1   # p
    assert lib.moe_spec_accept(good, None, good, good, good, 4, 8, 1000, 0, good, good, None) == 1   # q
    assert lib.moe_spec_accept(good, good, good, good, P(66), 4, 8, 1000, 0, good, good, None) == 1  # u align
    # union cost: pool size, shared-memory bound, workspace
    assert lib.moe_union_cost(good, 33, 4, 2, good, 10, good, good, 0.5, good, good, good, good, good, good,
                              4096, None) == 2
    assert lib.moe_union_cost(good, 32, 1000, 4, good, 10, good, good, 0.5, good, good, good, good, good, good,
                              4096, None) == 2
    assert lib.moe_union_cost(good, 8, 4, 2, good, 10, good, good, 0.5, good, good, good, good, good, None,
                              4096, None) == 1
    assert lib.moe_union_cost(good, 8, 4, 2, good, 1000, good, good, 0.5, good, good, good, good, good, good,
                              16, None) == 4
    assert lib.moe_union_cost_workspace_bytes(1000) >= 4 * 12


def test_wait_limit_setter(lib):
    """moe_set_wait_limit is host only: negative limits are refused, 0 restores the default."""
    assert lib.moe_set_wait_limit(ctypes.c_int64(-1)) == 1
    assert lib.moe_set_wait_limit(ctypes.c_int64(2000)) == 0
    assert lib.moe_set_wait_limit(ctypes.c_int64(0)) == 0
