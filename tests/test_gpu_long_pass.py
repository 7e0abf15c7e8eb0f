"""Per-slot passes above 16 tokens (moe_expert_op_perslot and its e4m3 form): consecutive launches
of up to 16 tokens on one workspace sized for 16, against the oracle per token."""
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


def test_deduplicating_forms_stop_at_16_tokens():
    dl = DeviceLayer(256, 256, 16, 4, "bf16", seed=830)
    x = dl.activations(17, seed=831)
    ids = torch.zeros((17, 4), dtype=torch.int32, device="cuda")
    gates = torch.ones((17, 4), device="cuda")
    with pytest.raises(api.MoeError):
        api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws)
