"""The deduplicating form from ids in one launch (moe_expert_op_dedup_ids and its e4m3 form):
the grouping built inside the tensor-core kernel gives the result of moe_group_slots followed
by moe_expert_op_dedup, including repeated and out-of-range ids, and the oracle's per token."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16, DeviceLayer, rel_max_err, route
from moe_speculative_decoding_gb300 import api, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_speculative_decoding_gb300 import build
    build.build()
    api.lib()


def test_repeated_and_bad_ids_match_the_two_calls(oracle_mod):
    """A token naming one expert twice (its gates add), ids N and -1 (skipped, MOE_ERR_BAD_ID)."""
    dl = DeviceLayer(256, 256, 16, 4, "bf16", seed=700)
    n = 6
    x = dl.activations(n, seed=701)
    ids_np = np.array([[0, 1, 2, 3], [3, 3, 5, 7], [15, 14, 0, 1], [16, 2, -1, 9], [8, 8, 8, 8], [1, 4, 6, 12]],
                      np.int32)
    gates = torch.from_numpy(np.random.default_rng(2).random((n, 4)).astype(np.float32)).cuda()
    ids = torch.from_numpy(ids_np).cuda()
    grp = api.group_slots(ids, dl.N, ws=dl.ws)
    y2 = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == 5
    y1 = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == 5
    assert rel_max_err(y1, y2) <= 1e-4
    ok = np.where((ids_np >= 0) & (ids_np < dl.N), ids_np, 0)
    g = np.where((ids_np >= 0) & (ids_np < dl.N), gates.cpu().numpy(), 0.0)
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ok, g)
    assert rel_max_err(y1, ref) <= TOL_BF16


@pytest.mark.parametrize("row", [[3, 0, 15, 7], [3, 3, 5, 7], [2, 16, 1, 0], [9, -1, 9, 4]])
def test_one_token_pass_with_and_without_distinct_ids(oracle_mod, row):
    """A one-token pass with distinct ids needs no grouping (each slot is its own group); a
    repeated id (gates added, read once) or an id out of range (skipped, MOE_ERR_BAD_ID) takes
    the grouping path.  Every case matches the two calls and the oracle."""
    dl = DeviceLayer(256, 256, 16, 4, "bf16", seed=705)
    x = dl.activations(1, seed=706)
    ids_np = np.array([row], np.int32)
    gates = torch.tensor([[0.4, 0.3, 0.2, 0.1]], device="cuda")
    ids = torch.from_numpy(ids_np).cuda()
    bad = bool(((ids_np < 0) | (ids_np >= dl.N)).any())
    grp = api.group_slots(ids, dl.N, ws=dl.ws)
    y2 = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == (5 if bad else 0)
    y1 = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == (5 if bad else 0)
    assert rel_max_err(y1, y2) <= 1e-4
    ok = np.where((ids_np >= 0) & (ids_np < dl.N), ids_np, 0)
    g = np.where((ids_np >= 0) & (ids_np < dl.N), gates.cpu().numpy(), 0.0)
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ok, g)
    assert rel_max_err(y1, ref) <= TOL_BF16


@pytest.mark.parametrize("n", [1, 3, 16])
def test_qwen3_shape_matches_oracle_and_overwrite(oracle_mod, n):
    """N = 128 experts, m = 8, d = 2048, f = 768 (smaller N for host copies: 32 experts)."""
    dl = DeviceLayer(2048, 768, 32, 8, "bf16", seed=710 + n)
    x = dl.activations(n, seed=711)
    _, logits = synth.routing_traces(1, n, 32, 8, 0.4, seed=712 + n)
    ids, gates = route(logits[0], 8)
    y = torch.full((n, 2048), 7.0, device="cuda")
    api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, y=y, ws=dl.ws)   # overwrite
    y1 = y.cpu().numpy()
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), gates.cpu().numpy())
    assert rel_max_err(y1, ref) <= TOL_BF16
    api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, y=y, accumulate=True, ws=dl.ws)
    assert rel_max_err(y.cpu().numpy(), 2 * ref) <= TOL_BF16


def test_e4m3_matches_the_two_calls():
    d, f, N, m, n = 2048, 768, 32, 8, 16
    dl = DeviceLayer(d, f, N, m, "bf16", seed=720)
    l8 = api.make_layer(d, f, N, m, "e4m3")
    ws8 = api.workspace(l8, 16, "cuda")
    w8, sc = api.quantize_experts(dl.w)
    x = dl.activations(n, seed=721)
    xq, sx = api.quantize_rows_e4m3(x)
    _, logits = synth.routing_traces(1, n, N, m, 0.4, seed=722)
    ids, gates = route(logits[0], m)
    grp = api.group_slots(ids, N)
    y2 = api.expert_op_dedup_fp8(l8, w8, sc, xq, sx, gates, grp, ws=ws8).cpu().numpy()
    y1 = api.expert_op_dedup_ids_fp8(l8, w8, sc, xq, sx, ids, gates, ws=ws8).cpu().numpy()
    assert api.last_device_error(ws8) == 0
    assert rel_max_err(y1, y2) <= 1e-4


def test_unsupported_shapes():
    f32 = api.make_layer(256, 512, 8, 2, "f32")
    dl = DeviceLayer(256, 512, 8, 2, "f32", seed=730)
    x = dl.activations(4, seed=731)
    ids = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    gates = torch.ones((4, 2), device="cuda")
    with pytest.raises(api.MoeError):
        api.expert_op_dedup_ids(f32, dl.w, x, ids, gates, ws=dl.ws)
    with pytest.raises(api.MoeError):   # above 64 tokens
        bf = DeviceLayer(256, 128, 8, 2, "bf16", seed=734)
        api.expert_op_dedup_ids(bf.layer, bf.w, bf.activations(65, seed=735),
                                torch.zeros((65, 2), dtype=torch.int32, device="cuda"),
                                torch.ones((65, 2), device="cuda"), ws=api.workspace(bf.layer, 64, "cuda"))


def test_more_than_256_slots_group_in_the_workspace(oracle_mod):
    """9 tokens of top-32: 288 slots, more than the kernel groups in shared memory, so the call
    from ids groups them with moe_group_slots into the workspace first.  Every slot names expert
    0 (one group of 9 tokens, each token's 32 gates added), then random routing."""
    big = DeviceLayer(256, 128, 64, 32, "bf16", seed=732)
    n = 9
    xb = big.activations(n, seed=733)
    rng = np.random.default_rng(736)
    gates_np = rng.random((n, 32)).astype(np.float32)
    gates = torch.from_numpy(gates_np).cuda()
    for ids_np in (np.zeros((n, 32), np.int32), np.stack([rng.permutation(64)[:32] for _ in range(n)]).astype(np.int32)):
        ids = torch.from_numpy(ids_np).cuda()
        y = api.expert_op_dedup_ids(big.layer, big.w, xb, ids, gates, ws=big.ws).cpu().numpy()
        assert api.last_device_error(big.ws) == 0
        ref = oracle_mod.expert_op_perslot(*big.host(), synth.host_array(xb), ids_np, gates_np)
        assert rel_max_err(y, ref) <= TOL_BF16


def test_routing_slices_need_only_element_alignment(oracle_mod):
    """Per-layer slices of one ids / gates array start 8 bytes apart when m = 2 and n is odd:
    every form takes them (the kernels read routing arrays one element at a time)."""
    dl = DeviceLayer(512, 256, 8, 2, "bf16", seed=740)
    n = 3
    x = dl.activations(n, seed=741)
    _, logits = synth.routing_traces(1, 2 * n, 8, 2, 0.3, seed=742)
    ids_all, gates_all = route(logits[0], 2)
    ids, gates = ids_all[n:], gates_all[n:]             # 24-byte offset: 8-byte aligned only
    assert ids.data_ptr() % 16 == 8
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids.cpu().numpy(), gates.cpu().numpy())
    ys = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    grp = api.group_slots(ids, 8, ws=dl.ws)
    yd = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=dl.ws).cpu().numpy()
    yi = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == 0
    for y in (ys, yd, yi):
        assert rel_max_err(y, ref) <= TOL_BF16


def test_groups_larger_than_their_tokens_split_over_warps(oracle_mod):
    """Two tokens naming one expert in all 8 slots: a group of 16 slots but 2 tokens, whose h is
    formed by four h-former warps of which two hold no token, beside groups of 1 to 2 tokens;
    bf16 and e4m3, against the oracle per token."""
    d, f, N, m, n = 256, 256, 16, 8, 4
    dl = DeviceLayer(d, f, N, m, "bf16", seed=750)
    x = dl.activations(n, seed=751)
    ids_np = np.array([[5] * 8, [5] * 8, list(range(8)), list(range(8, 16))], np.int32)
    gates_np = np.random.default_rng(752).random((n, m)).astype(np.float32)
    ids, gates = torch.from_numpy(ids_np).cuda(), torch.from_numpy(gates_np).cuda()
    y1 = api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    assert api.last_device_error(dl.ws) == 0
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ids_np, gates_np)
    assert rel_max_err(y1, ref) <= TOL_BF16
    grp = api.group_slots(ids, N, ws=dl.ws)
    y2 = api.expert_op_dedup(dl.layer, dl.w, x, gates, grp, ws=dl.ws).cpu().numpy()
    assert rel_max_err(y1, y2) <= 1e-4
    # e4m3: the same grouping on the FP8 kernel (TK = 2 tokens per round: four warps as well)
    l8 = api.make_layer(d, f, N, m, "e4m3")
    ws8 = api.workspace(l8, 16, "cuda")
    w8, sc = api.quantize_experts(dl.w)
    xq, sx = api.quantize_rows_e4m3(x)
    y8 = api.expert_op_dedup_ids_fp8(l8, w8, sc, xq, sx, ids, gates, ws=ws8).cpu().numpy()
    assert api.last_device_error(ws8) == 0
    xq_h, sx_h = xq.cpu().numpy(), sx.cpu().numpy()
    for t in range(n):
        idx = torch.as_tensor(ids_np[t].astype(np.int64), device="cuda")
        cg, cu, cd = (w.index_select(0, idx).cpu().numpy() for w in w8)
        sg, su, sd = (s.index_select(0, idx).cpu().numpy() for s in sc)
        local = np.arange(m, dtype=np.int32)[None, :].repeat(n, axis=0)
        y_ref = oracle_mod.expert_op_token_fp8(cg, cu, cd, sg, su, sd, xq_h, sx_h, local,
                                               gates_np.astype(np.float64), t)
        assert np.max(np.abs(y8[t] - y_ref)) <= TOL_BF16 * np.sqrt(np.mean(y_ref ** 2)), t
