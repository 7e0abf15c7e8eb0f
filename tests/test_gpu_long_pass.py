"""Passes above 16 tokens.  The per-slot calls (and their e4m3 form) run them as consecutive
launches of up to 16 tokens on one workspace sized for 16; the deduplicating calls take up to 64
tokens in one launch of the 32- or 64-token instantiation (32 or 64 TMEM columns per
accumulator, wider token masks), so each distinct expert is still read once.  Everything against
the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16, TOL_F32, DeviceLayer, rel_max_err, route
from moe_speculative_decoding_gb300 import api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_speculative_decoding_gb300 import build
    build.build()
    api.lib()


@pytest.mark.parametrize("n", [17, 40, 64])
def test_bf16_long_pass_matches_oracle(oracle_mod, n):
    dl = DeviceLayer(512, 256, 16, 4, "bf16", seed=800 + n)
    x = dl.activations(n, seed=801 + n)
    _, logits = synth.routing_traces(1, n, 16, 4, 0.4, seed=802 + n)
    ids, gates = route(logits[0], 4)
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), gates.cpu().numpy())
    y = torch.full((n, 512), 3.0, device="cuda")
    api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, y=y, ws=dl.ws)   # overwrite
    assert api.last_device_error(dl.ws) == 0
    assert rel_max_err(y.cpu().numpy(), ref) <= TOL_BF16
    api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, y=y, accumulate=True, ws=dl.ws)
    assert rel_max_err(y.cpu().numpy(), 2 * ref) <= TOL_BF16


def test_e4m3_long_pass_matches_oracle(oracle_mod):
    d, f, N, m, n = 256, 256, 16, 4, 40
    dl = DeviceLayer(d, f, N, m, "bf16", seed=820)
    l8 = api.make_layer(d, f, N, m, "e4m3")
    ws8 = api.workspace(l8, 16, "cuda")
    w8, sc = api.quantize_experts(dl.w)
    x = dl.activations(n, seed=821)
    xq, sx = api.quantize_rows_e4m3(x)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=822)
    ids, gates = route(logits[0], m)
    y = api.expert_op_perslot_fp8(l8, w8, sc, xq, sx, ids, gates, ws=ws8).cpu().numpy()
    assert api.last_device_error(ws8) == 0
    ids_h, g_h = ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64)
    xq_h, sx_h = xq.cpu().numpy(), sx.cpu().numpy()
    for t in (0, 15, 16, 17, 31, 32, 39):   # both sides of every launch boundary
        idx = torch.as_tensor(ids_h[t].astype(np.int64), device="cuda")
        cg, cu, cd = (w.index_select(0, idx).cpu().numpy() for w in w8)
        sg, su, sd = (s.index_select(0, idx).cpu().numpy() for s in sc)
        local = np.arange(m, dtype=np.int32)[None, :].repeat(n, axis=0)
        y_ref = oracle_mod.expert_op_token_fp8(cg, cu, cd, sg, su, sd, xq_h, sx_h, local, g_h, t)
        assert np.max(np.abs(y[t] - y_ref)) <= TOL_BF16 * np.sqrt(np.mean(y_ref ** 2)), t


def _check_rows(y, ref_rows):
    for t, yr in ref_rows.items():
        assert np.max(np.abs(y[t] - yr)) <= TOL_BF16 * np.sqrt(np.mean(yr ** 2)), t


@pytest.mark.parametrize("n", [17, 32, 33, 40, 64])
@pytest.mark.parametrize("shape", [(512, 256, 16, 4), (512, 384, 32, 8)])
def test_bf16_dedup_long_pass_matches_oracle(oracle_mod, n, shape):
    """Both deduplicating calls at 17 (one token past the first 16 columns) and 32 tokens (the
    32-token instantiation), 33, 40 and 64 tokens (the 64-token one).
    Top-4 of 16 gives 68..256 slots (grouping inside the kernel); top-8 of 32 gives 136..512
    (above 256 slots the call from ids groups with moe_group_slots into the workspace first).
    Overwrite and accumulate, against the oracle on every token."""
    d, f, N, m = shape
    dl = DeviceLayer(d, f, N, m, "bf16", seed=840 + n + N)
    ws = api.workspace(dl.layer, n, "cuda")
    x = dl.activations(n, seed=841 + n)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=842 + n)
    ids, gates = route(logits[0], m)
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), gates.cpu().numpy())
    y = torch.full((n, d), 3.0, device="cuda")
    api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, y=y, ws=ws)   # overwrite
    assert api.last_device_error(ws) == 0
    assert rel_max_err(y.cpu().numpy(), ref) <= TOL_BF16
    api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, y=y, accumulate=True, ws=ws)
    assert rel_max_err(y.cpu().numpy(), 2 * ref) <= TOL_BF16
    grp = api.group_slots(ids, N, ws=ws)
    yd = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=ws).cpu().numpy()
    assert api.last_device_error(ws) == 0
    assert rel_max_err(yd, ref) <= TOL_BF16
    # per-slot on the same pass (launches of 16) agrees as well
    ys = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
    assert rel_max_err(ys, yd) <= 2 * TOL_BF16


def test_every_token_in_one_group_and_repeated_ids(oracle_mod):
    """64 tokens naming the same four experts: groups of all 64 tokens, whose masks fill all four
    16-token column blocks and whose h is formed by every h-former warp; then a pass where some
    tokens name an expert twice (their gates add) and one token alone holds an expert in the
    last column block."""
    d, f, N, m, n = 256, 256, 16, 4, 64
    dl = DeviceLayer(d, f, N, m, "bf16", seed=860)
    ws = api.workspace(dl.layer, n, "cuda")
    x = dl.activations(n, seed=861)
    rng = np.random.default_rng(862)
    gates_np = rng.random((n, m)).astype(np.float32)
    gates = torch.from_numpy(gates_np).cuda()
    same = np.array([[2, 7, 11, 0]] * n, np.int32)
    rep = np.array([[(t + j) % 12 for j in range(m)] for t in range(n)], np.int32)
    rep[5] = [3, 3, 3, 9]
    rep[40] = [1, 1, 6, 6]
    rep[63] = [15, 14, 13, 12]   # experts 12..15: token 63 only
    for ids_np in (same, rep):
        ids = torch.from_numpy(ids_np).cuda()
        ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids_np, gates_np)
        y1 = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
        assert api.last_device_error(ws) == 0
        assert rel_max_err(y1, ref) <= TOL_BF16
        grp = api.group_slots(ids, N, ws=ws)
        y2 = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=ws).cpu().numpy()
        assert rel_max_err(y2, y1) <= 1e-4


def test_qwen3_layer_at_64_tokens_every_token(oracle_mod):
    """The full Qwen3-30B-A3B layer shape (d 2048, f 768, 128 experts, top-8) at 64 tokens: 512
    slots, grouped by moe_group_slots inside the call from ids; every token against the oracle."""
    d, f, N, m, n = 2048, 768, 128, 8, 64
    dl = DeviceLayer(d, f, N, m, "bf16", seed=870)
    ws = api.workspace(dl.layer, n, "cuda")
    x = dl.activations(n, seed=871)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=872)
    ids, gates = route(logits[0], m)
    y1 = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
    assert api.last_device_error(ws) == 0
    grp = api.group_slots(ids, N, ws=ws)
    y2 = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=ws).cpu().numpy()
    assert rel_max_err(y2, y1) <= 1e-4
    ids_h, g_h = ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64)
    xh = synth.host_array(x)
    local = np.arange(m, dtype=np.int32)[None, :].repeat(n, axis=0)
    refs = {t: oracle_mod.expert_op_token(*dl.host_experts(ids_h[t]), xh, local, g_h, t) for t in range(n)}
    _check_rows(y1, refs)


@pytest.mark.parametrize("n,N,m", [(24, 16, 4), (40, 16, 4), (64, 32, 8)])
def test_e4m3_dedup_long_pass_matches_oracle(oracle_mod, n, N, m):
    """The e4m3 deduplicating calls at 24 tokens (the 32-token instantiation), 40 tokens (160
    slots, grouping in the kernel) and 64 (512 slots, moe_group_slots first), against the e4m3
    oracle on every token."""
    d, f = 256, 256
    dl = DeviceLayer(d, f, N, m, "bf16", seed=880 + n)
    l8 = api.make_layer(d, f, N, m, "e4m3")
    ws8 = api.workspace(l8, n, "cuda")
    w8, sc = api.quantize_experts(dl.w)
    x = dl.activations(n, seed=881 + n)
    xq, sx = api.quantize_rows_e4m3(x)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=882 + n)
    ids, gates = route(logits[0], m)
    y1 = api.expert_op_dedup_ids_fp8(l8, w8, sc, xq, sx, ids, gates, ws=ws8).cpu().numpy()
    assert api.last_device_error(ws8) == 0
    grp = api.group_slots(ids, N, ws=ws8)
    y2 = api.expert_op_dedup_fp8(l8, w8, sc, xq, sx, gates, grp, ws=ws8).cpu().numpy()
    assert rel_max_err(y2, y1) <= 1e-4
    ids_h, g_h = ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64)
    xq_h, sx_h = xq.cpu().numpy(), sx.cpu().numpy()
    local = np.arange(m, dtype=np.int32)[None, :].repeat(n, axis=0)
    refs = {}
    for t in range(n):
        idx = torch.as_tensor(ids_h[t].astype(np.int64), device="cuda")
        cg, cu, cd = (w.index_select(0, idx).cpu().numpy() for w in w8)
        sg, su, sd = (s.index_select(0, idx).cpu().numpy() for s in sc)
        refs[t] = oracle_mod.expert_op_token_fp8(cg, cu, cd, sg, su, sd, xq_h, sx_h, local, g_h, t)
    _check_rows(y1, refs)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cuda_core_kernel_long_dedup_pass(oracle_mod, dtype):
    """The CUDA-core kernel (fp32 layers, and bf16 layers that ask for it) takes a group's tokens
    in windows of 16: the deduplicating call at 64 tokens, against the oracle."""
    d, f, N, m, n = 256, 128, 8, 2, 64
    dl = DeviceLayer(d, f, N, m, dtype, seed=890, simt=True)
    ws = api.workspace(dl.layer, n, "cuda")
    x = dl.activations(n, seed=891)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=892)
    ids, gates = route(logits[0], m)
    grp = api.group_slots(ids, N, ws=ws)
    y = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=ws).cpu().numpy()
    assert api.last_device_error(ws) == 0
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), gates.cpu().numpy())
    assert rel_max_err(y, ref) <= (TOL_F32 if dtype == "f32" else TOL_BF16)


def test_largest_pass_of_the_largest_routing(oracle_mod):
    """The supported maxima of the routing side at once: N = 1024 experts, top-32, 64 tokens
    (2,048 slots, grouped with moe_group_slots into the workspace), both deduplicating calls and
    the per-slot call, sampled tokens against the oracle."""
    d, f, N, m, n = 256, 128, 1024, 32, 64
    dl = DeviceLayer(d, f, N, m, "bf16", seed=900)
    ws = api.workspace(dl.layer, n, "cuda")
    x = dl.activations(n, seed=901)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=902)
    ids, gates = route(logits[0], m)
    y1 = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
    grp = api.group_slots(ids, N, ws=ws)
    y2 = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=ws).cpu().numpy()
    y3 = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
    assert api.last_device_error(ws) == 0
    assert rel_max_err(y2, y1) <= 1e-4
    ids_h, g_h = ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64)
    xh = synth.host_array(x)
    local = np.arange(m, dtype=np.int32)[None, :].repeat(n, axis=0)
    rows = {t: oracle_mod.expert_op_token(*dl.host_experts(ids_h[t]), xh, local, g_h, t) for t in (0, 21, 42, 63)}
    _check_rows(y1, rows)
    _check_rows(y3, rows)


def test_largest_layer_dimensions(oracle_mod):
    """d = 8192 and f = 65536, the largest the library takes (two experts of 3.2 GB each, top-1,
    two tokens), both forms against the oracle on every token."""
    d, f, N, m, n = 8192, 65536, 2, 1, 2
    dl = DeviceLayer(d, f, N, m, "bf16", seed=910)
    x = dl.activations(n, seed=911)
    ids = torch.tensor([[1], [0]], dtype=torch.int32, device="cuda")
    gates = torch.tensor([[0.75], [1.25]], device="cuda")
    ws = api.workspace(dl.layer, n, "cuda")
    ys = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
    yd = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=ws).cpu().numpy()
    assert api.last_device_error(ws) == 0
    ids_h, g_h = ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64)
    xh = synth.host_array(x)
    local = np.zeros((n, 1), np.int32)
    rows = {t: oracle_mod.expert_op_token(*dl.host_experts(ids_h[t]), xh, local, g_h, t) for t in range(n)}
    _check_rows(ys, rows)
    _check_rows(yd, rows)


@pytest.mark.parametrize("n", [17, 32, 33, 64])
def test_perslot_long_pass_in_one_launch(oracle_mod, n):
    """A per-slot pass above 16 tokens runs as equal launches of up to 32 tokens (the 32-token
    form) when the workspace holds 32 tokens, and of up to 16 when it holds 16: the same result,
    bf16 and e4m3, against the oracle.  The two agree to 2e-3 of the output's scale, not to the
    last bit: launches of different sizes split each gate/up sum over CTAs differently, so its
    fp32 shares add in another order and h's rounding to bf16 (e4m3) can differ by one step."""
    d, f, N, m = 512, 256, 32, 8
    dl = DeviceLayer(d, f, N, m, "bf16", seed=920 + n)
    x = dl.activations(n, seed=921 + n)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=922 + n)
    ids, gates = route(logits[0], m)
    ws_n, ws_16 = api.workspace(dl.layer, n, "cuda"), api.workspace(dl.layer, 16, "cuda")
    y1 = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=ws_n).cpu().numpy()
    y2 = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=ws_16).cpu().numpy()
    assert api.last_device_error(ws_n) == 0 and api.last_device_error(ws_16) == 0
    assert rel_max_err(y1, y2) <= 2e-3
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), gates.cpu().numpy())
    assert rel_max_err(y1, ref) <= TOL_BF16
    l8 = api.make_layer(d, f, N, m, "e4m3")
    w8, sc = api.quantize_experts(dl.w)
    xq, sx = api.quantize_rows_e4m3(x)
    w8n, w816 = api.workspace(l8, n, "cuda"), api.workspace(l8, 16, "cuda")
    z1 = api.expert_op_perslot_fp8(l8, w8, sc, xq, sx, ids, gates, ws=w8n).cpu().numpy()
    z2 = api.expert_op_perslot_fp8(l8, w8, sc, xq, sx, ids, gates, ws=w816).cpu().numpy()
    assert api.last_device_error(w8n) == 0 and api.last_device_error(w816) == 0
    assert rel_max_err(z1, z2) <= 2e-3
