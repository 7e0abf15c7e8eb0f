"""GPU parity: every kernel through the C ABI against the CPU oracle on the same seeded
inputs.  Routing ids, groupings and byte counts bit-exact; outputs within
max|y - y_ref| <= 2e-2 * rms(y_ref) (bf16 weights, fp32 accumulation)."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16, TOL_F32, DeviceLayer, rel_max_err, route
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300.configs import DSV2_LITE, MIXTRAL, QWEN3, TINY

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_speculative_decoding_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    api.lib()


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("n,N,m,rho", [(16, 128, 8, 0.5), (8, 64, 6, 0.3), (8, 8, 2, 0.8), (4, 8, 2, 0.0),
                                       (1, 2, 1, 0.0), (37, 1024, 32, 0.2), (300, 100, 7, 0.0)])
def test_route_matches_oracle(oracle_mod, n, N, m, rho):
    sets, logits = synth.routing_traces(1, n, N, m, rho, seed=100 + N)
    ids, gates = route(logits[0], m)
    ref_ids, ref_gates = oracle_mod.route_topm(logits[0], m)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(gates.cpu().numpy(), ref_gates, rtol=2e-6, atol=1e-7)


def test_route_ties_and_full_softmax(oracle_mod):
    rng = np.random.default_rng(101)
    z = rng.integers(-3, 4, size=(64, 40)).astype(np.float32)     # many exact ties
    z[0] = 0.0
    z[1, :] = -0.0
    z[2, 5] = np.float32(-np.inf)
    for m in (1, 3, 8, 32):
        ids, gates = route(z, m)
        ref_ids, ref_gates = oracle_mod.route_topm(z, m)
        assert np.array_equal(ids.cpu().numpy(), ref_ids)
        assert np.allclose(gates.cpu().numpy(), ref_gates, rtol=2e-6, atol=1e-7)
    logits = torch.from_numpy(z).cuda()
    ids, gates = api.route_topm(logits, 4, renorm=False)
    ref_ids, ref_gates = oracle_mod.route_topm(z, 4, renorm=False)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(gates.cpu().numpy(), ref_gates, rtol=2e-6, atol=1e-7)
    # n = 0 enqueues nothing
    e = torch.empty((0, 40), device="cuda")
    api.route_topm(e, 4)


@pytest.mark.parametrize("N,m", [(128, 8), (64, 6)])
def test_route_near_ties_at_config_size(oracle_mod, N, m):
    """Normal logits at the configs' expert counts, with the m-th and (m+1)-th largest made
    equal, one ulp apart either way, or +0/-0, and an exact tie inside the selected set."""
    rng = np.random.default_rng(1000 + N + m)
    n = 96
    z = rng.standard_normal((n, N)).astype(np.float32)
    for t in range(n):
        order = np.argsort(-z[t].astype(np.float64), kind="stable")
        a, b = order[m - 1], order[m]
        kind = t % 4
        if kind == 0:
            z[t, b] = z[t, a]                                      # exact tie at the boundary
        elif kind == 1:
            z[t, b] = np.nextafter(z[t, a], np.float32(-np.inf))   # one ulp below
        elif kind == 2:
            z[t, b] = np.nextafter(z[t, a], np.float32(np.inf))    # one ulp above: they swap
        else:
            z[t, a], z[t, b] = np.float32(0.0), np.float32(-0.0)   # +0 and -0 compare equal
            z[t, order[m + 1:]] = -np.abs(z[t, order[m + 1:]]) - 1.0
            z[t, order[:m - 1]] = np.abs(z[t, order[:m - 1]]) + 1.0
        if m >= 3:
            z[t, order[1]] = z[t, order[2]]                        # a tie inside the selected set
    ids, gates = route(z, m)
    ref_ids, ref_gates = oracle_mod.route_topm(z, m)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(gates.cpu().numpy(), ref_gates, rtol=2e-6, atol=1e-7)


def test_route_nan_logits_stay_valid():
    z = np.random.default_rng(102).standard_normal((8, 16)).astype(np.float32)
    z[:, ::2] = np.nan
    z[7, :] = np.nan
    ids, _ = route(z, 10)
    ids = ids.cpu().numpy()
    for t in range(8):
        assert len(set(ids[t].tolist())) == 10 and ids[t].min() >= 0 and ids[t].max() < 16


# ------------------------------------------------------------------ grouping

@pytest.mark.parametrize("n,m,N", [(1, 1, 2), (4, 2, 8), (16, 8, 128), (8, 6, 64), (8, 2, 8),
                                   (16, 32, 256), (64, 64, 1024), (13, 3, 5)])
def test_group_matches_oracle(oracle_mod, n, m, N):
    sets, _ = synth.routing_traces(1, n, N, m, 0.5, seed=103 + n)
    ids = torch.from_numpy(sets[0]).cuda()
    g = api.group_slots(ids, N)
    U, lst, off, order = oracle_mod.group_slots(sets[0], N)
    assert int(g.num_distinct.item()) == U
    assert np.array_equal(g.expert_list[:U].cpu().numpy(), lst)
    assert np.array_equal(g.offsets[:U + 1].cpu().numpy(), off)
    assert np.array_equal(g.slot_order.cpu().numpy(), order)
    # the grouping's U is the byte count's U
    assert U == api.pass_bytes(api.make_layer(64, 64, N, m), sets[0])["U"]


def test_group_bad_ids_flagged_and_skipped():
    L = api.make_layer(64, 64, 8, 2)
    ws = api.workspace(L)
    ids = torch.tensor([[0, 3], [9, 3], [-1, 2]], dtype=torch.int32, device="cuda")
    g = api.group_slots(ids, 8, ws=ws)
    assert api.last_device_error(ws) == 5
    U = int(g.num_distinct.item())
    assert U == 3
    assert g.expert_list[:U].tolist() == [0, 2, 3]
    assert g.offsets[:U + 1].tolist() == [0, 1, 2, 4]
    assert g.slot_order[:4].tolist() == [0, 5, 1, 3]


# ------------------------------------------------------------- expert op helpers

def _run_both(dl, x, logits_np, seed_grp=None):
    ids, gates = route(logits_np, dl.m)
    y_slot = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws)
    grp = api.group_slots(ids, dl.N, ws=dl.ws)
    y_dedup = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=dl.ws)
    assert api.last_device_error(dl.ws) == 0
    yd = y_dedup.cpu().numpy()
    # the deduplicating form from ids in one launch (grouping inside the kernel), where the
    # tensor-core kernel runs the layer: the same result as the two calls
    if dl.tdtype == torch.bfloat16 and dl.d % 128 == 0 and x.shape[0] * dl.m <= 256:
        y_ids = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
        assert api.last_device_error(dl.ws) == 0
        assert rel_max_err(y_ids, yd) <= 1e-4, rel_max_err(y_ids, yd)
    return ids, gates, grp, y_slot.cpu().numpy(), yd


def _oracle_full(oracle_mod, dl, x, logits_np):
    ids, gates = oracle_mod.route_topm(logits_np, dl.m)
    xh = synth.host_array(x)
    y1 = oracle_mod.expert_op_perslot(*dl.host(), xh, ids, gates)
    y2 = oracle_mod.expert_op_dedup(*dl.host(), xh, gates, dl.m, oracle_mod.group_slots(ids, dl.N))
    assert np.array_equal(y1, y2)
    return ids, y1


# ------------------------------------------------------------- tiny fp32 layer

def test_tiny_fp32_layer(oracle_mod):
    """The tiny fp32 layer: N=8, m=2, d=256, f=512, n=4, router logits x W_r^T, seed 0."""
    w = TINY
    dl = DeviceLayer(w.d, w.f, w.N, w.m, "f32", seed=synth.seed_for(w.index, stream=0))
    x_cpu = synth.activations(4, w.d, torch.float32, seed=synth.seed_for(w.index, stream=1))
    w_r = synth.tiny_router(w.N, w.d, seed=synth.seed_for(w.index, stream=2))
    logits = synth.tiny_logits(x_cpu, w_r).numpy()
    x = x_cpu.cuda()
    ids, gates, grp, ys, yd = _run_both(dl, x, logits)
    ref_ids, ref = _oracle_full(oracle_mod, dl, x, logits)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert rel_max_err(ys, ref) <= TOL_F32
    assert rel_max_err(yd, ref) <= TOL_F32


# ------------------------------------------------------ bf16: several tiles, ragged

SMALL = [
    # d, f, N, m, n, rho
    (128, 64, 4, 1, 1, 0.0),       # one tile, one down block, single expert
    (256, 192, 8, 2, 5, 0.3),      # 3 f tiles, 2 down blocks
    (384, 128, 16, 4, 16, 0.5),    # odd number of down blocks, full pass
    (512, 256, 8, 8, 3, 0.0),      # m = N: every token takes every expert
    (256, 128, 32, 3, 16, 0.9),    # heavy reuse
    (1024, 320, 12, 5, 7, 0.2),    # 5 f tiles, ragged n
    (4096, 128, 4, 2, 9, 0.5),     # largest d of the tensor-core kernel (5 stages)
]


@pytest.mark.parametrize("d,f,N,m,n,rho", SMALL)
def test_bf16_small_layers_match_oracle(oracle_mod, d, f, N, m, n, rho):
    dl = DeviceLayer(d, f, N, m, "bf16", seed=200 + d + f)
    x = dl.activations(n, seed=201)
    _, logits = synth.routing_traces(1, n, N, m, rho, seed=202 + n)
    ids, gates, grp, ys, yd = _run_both(dl, x, logits[0])
    ref_ids, ref = _oracle_full(oracle_mod, dl, x, logits[0])
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    e_s, e_d = rel_max_err(ys, ref), rel_max_err(yd, ref)
    assert e_s <= TOL_BF16 and e_d <= TOL_BF16, (e_s, e_d)
    assert rel_max_err(ys, yd) <= TOL_BF16
    # the CUDA-core kernel on the same bf16 layer
    simt = api.make_layer(d, f, N, m, "bf16", simt=True)
    y_simt = api.expert_op_perslot(simt, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    y_simt_d = api.expert_op_dedup(simt, dl.w, x, gates, grp, ws=dl.ws).cpu().numpy()
    assert rel_max_err(y_simt, ref) <= 1e-3 and rel_max_err(y_simt_d, ref) <= 1e-3


def test_single_token_single_expert_is_one_ffn(oracle_mod):
    dl = DeviceLayer(256, 128, 3, 1, "bf16", seed=210)
    x = dl.activations(1, seed=211)
    for e in range(3):
        ids = torch.tensor([[e]], dtype=torch.int32, device="cuda")
        gates = torch.ones((1, 1), device="cuda")
        y = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
        ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), np.ones((1, 1)))
        assert rel_max_err(y, ref) <= TOL_BF16


def test_same_set_every_token_and_all_distinct(oracle_mod):
    dl = DeviceLayer(256, 128, 64, 4, "bf16", seed=220)
    n = 16
    x = dl.activations(n, seed=221)
    # rho = 1: every token selects the same set -> U = m
    _, logits = synth.routing_traces(1, n, 64, 4, 1.0, seed=222)
    ids, gates, grp, ys, yd = _run_both(dl, x, logits[0])
    assert int(grp.num_distinct.item()) == 4
    _, ref = _oracle_full(oracle_mod, dl, x, logits[0])
    assert rel_max_err(yd, ref) <= TOL_BF16 and rel_max_err(ys, ref) <= TOL_BF16
    # all slots distinct -> U = n m
    z = np.full((n, 64), -5.0, np.float32)
    for t in range(n):
        z[t, 4 * t:4 * t + 4] = [3.0, 2.0, 1.0, 0.5]
    ids, gates, grp, ys, yd = _run_both(dl, x, z)
    assert int(grp.num_distinct.item()) == 64
    _, ref = _oracle_full(oracle_mod, dl, x, z)
    assert rel_max_err(yd, ref) <= TOL_BF16 and rel_max_err(ys, ref) <= TOL_BF16


def test_accumulate_adds_and_bad_ids_are_skipped(oracle_mod):
    dl = DeviceLayer(256, 128, 8, 2, "bf16", seed=230)
    x = dl.activations(3, seed=231)
    ids = torch.tensor([[0, 1], [2, 3], [4, 5]], dtype=torch.int32, device="cuda")
    gates = torch.full((3, 2), 0.5, device="cuda")
    y0 = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws)
    y = y0.clone()
    api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, y=y, accumulate=True, ws=dl.ws)
    assert rel_max_err(y.cpu().numpy(), 2 * y0.cpu().numpy()) <= 1e-5
    bad = torch.tensor([[0, 11], [2, 3], [-3, 5]], dtype=torch.int32, device="cuda")
    yb = api.expert_op_perslot(dl.layer, dl.w, x, bad, gates, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == 5
    ok_ids = np.array([[0, 0], [2, 3], [0, 5]], np.int32)
    g = np.array([[0.5, 0.0], [0.5, 0.5], [0.0, 0.5]])
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ok_ids, g)
    assert rel_max_err(yb, ref) <= TOL_BF16


# ------------------------------------------------- the workloads at full size, every token

def _full_size(oracle_mod, wl, n, rho_index):
    """A full-size layer of the workload, both forms, every token of the pass against the
    oracle (each token's output from host copies of its own m experts)."""
    dl = DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=synth.seed_for(wl.index, rho_index=rho_index))
    x = dl.activations(n, seed=synth.seed_for(wl.index, rho_index=rho_index, stream=1))
    _, logits = synth.routing_traces(1, n, wl.N, wl.m, wl.rhos[rho_index],
                                     seed=synth.seed_for(wl.index, rho_index=rho_index, stream=2))
    ids, gates, grp, ys, yd = _run_both(dl, x, logits[0])
    ref_ids, ref_gates = oracle_mod.route_topm(logits[0], wl.m)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert int(grp.num_distinct.item()) == oracle_mod.pass_bytes(wl.d, wl.f, wl.N, ref_ids)["U"]
    xh = synth.host_array(x)
    local = np.arange(wl.m, dtype=np.int32)[None, :].repeat(n, axis=0)
    refs = {}
    for t in range(n):
        y_ref = oracle_mod.expert_op_token(*dl.host_experts(ref_ids[t]), xh, local, ref_gates, t)
        refs[t] = y_ref
        rms = np.sqrt(np.mean(y_ref ** 2))
        for y in (ys, yd):
            assert np.max(np.abs(y[t] - y_ref)) <= TOL_BF16 * rms, t
    return dl, x, ys, yd, refs


@pytest.mark.parametrize("rho_index", [0, 2])
def test_deepseek_v2_lite_layer_with_shared_experts(oracle_mod, rho_index):
    wl = DSV2_LITE
    n = 8
    dl, x, ys, yd, refs = _full_size(oracle_mod, wl, n, rho_index)
    # two always-on shared experts through the deduplicating call: ids [0, 1], gates 1
    sh = DeviceLayer(wl.d, wl.f_shared, wl.n_shared, wl.n_shared, "bf16",
                     seed=synth.seed_for(wl.index, stream=9))
    sids = torch.tensor([[0, 1]] * n, dtype=torch.int32, device="cuda")
    sgates = torch.ones((n, 2), device="cuda")
    sgrp = api.group_slots(sids, 2)
    y = torch.from_numpy(yd).cuda()
    api.expert_op_dedup(sh.layer, sh.w, x, sgates, sgrp, y=y, accumulate=True, ws=sh.ws)
    y = y.cpu().numpy()
    xh = synth.host_array(x)
    for t in range(n):
        # the layer's output of token t: routed experts plus both shared experts
        y_sh = oracle_mod.expert_op_token(*sh.host(), xh, np.array([[0, 1]] * n, np.int32), np.ones((n, 2)), t)
        full = refs[t] + y_sh
        assert np.max(np.abs(y[t] - full)) <= TOL_BF16 * np.sqrt(np.mean(full ** 2)), t
        shared_part = y[t] - yd[t]
        assert np.max(np.abs(shared_part - y_sh)) <= TOL_BF16 * np.sqrt(np.mean(y_sh ** 2)), t


@pytest.mark.parametrize("rho_index", [0, 1])
def test_qwen3_layer_full_pass(oracle_mod, rho_index):
    _full_size(oracle_mod, QWEN3, 16, rho_index)


@pytest.mark.parametrize("rho_index", [0, 1])
def test_mixtral_layer(oracle_mod, rho_index):
    _full_size(oracle_mod, MIXTRAL, 8, rho_index)


@pytest.mark.parametrize("n", [1, 2, 11])
def test_qwen3_each_pass_size_forms_agree(oracle_mod, n):
    """Per-slot and dedup agree at every pass size; n = 1 gives U = m."""
    wl = QWEN3
    dl = DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=300)
    x = dl.activations(n, seed=301)
    _, logits = synth.routing_traces(1, n, wl.N, wl.m, 0.5, seed=302)
    ids, gates, grp, ys, yd = _run_both(dl, x, logits[0])
    assert rel_max_err(ys, yd) <= TOL_BF16
    if n == 1:
        assert int(grp.num_distinct.item()) == wl.m
    ref_ids, ref_gates = oracle_mod.route_topm(logits[0], wl.m)
    t = n - 1
    sub = dl.host_experts(ref_ids[t])
    local = np.arange(wl.m, dtype=np.int32)[None, :].repeat(n, axis=0)
    y_ref = oracle_mod.expert_op_token(*sub, synth.host_array(x), local, ref_gates, t)
    assert np.max(np.abs(yd[t] - y_ref)) <= TOL_BF16 * np.sqrt(np.mean(y_ref ** 2))


# ------------------------------------------------------- calls in a row, small passes

@pytest.mark.parametrize("n,rho", [(1, 0.0), (2, 0.5), (3, 0.0), (5, 0.4)])
def test_repeated_calls_same_workspace(oracle_mod, n, rho):
    """Calls in a row on one workspace stay within tolerance of the oracle and of each other."""
    wl = QWEN3
    dl = DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=400 + n)
    x = dl.activations(n, seed=401)
    _, logits = synth.routing_traces(1, n, wl.N, wl.m, rho, seed=402 + n)
    ids, gates = route(logits[0], wl.m)
    grp = api.group_slots(ids, wl.N, ws=dl.ws)
    ref_ids, ref_gates = oracle_mod.route_topm(logits[0], wl.m)
    t = n - 1
    sub = dl.host_experts(ref_ids[t])
    local = np.arange(wl.m, dtype=np.int32)[None, :].repeat(n, axis=0)
    y_ref = oracle_mod.expert_op_token(*sub, synth.host_array(x), local, ref_gates, t)
    rms = np.sqrt(np.mean(y_ref ** 2))
    outs = []
    for rep in range(3):
        ys = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws)
        yd = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=dl.ws)
        outs.append((ys.cpu().numpy(), yd.cpu().numpy()))
    assert api.last_device_error(dl.ws) == 0
    for ys, yd in outs:
        assert np.max(np.abs(ys[t] - y_ref)) <= TOL_BF16 * rms
        assert np.max(np.abs(yd[t] - y_ref)) <= TOL_BF16 * rms
        # the fp32 atomics of the combine add in run-dependent order
        assert rel_max_err(ys, outs[0][0]) <= 1e-4 and rel_max_err(yd, outs[0][1]) <= 1e-4
