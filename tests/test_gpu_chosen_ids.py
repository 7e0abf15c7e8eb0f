"""Passes with chosen ids on the Qwen3-30B-A3B-shaped layer: the n*m slots name exactly U
distinct experts, from heavy repetition (U = m) to none (U = min(N, n*m)) ([Lan], §2
"Effective bandwidth": the passes the fits (4) and (E.1) are made on).  The grouping's U is
exact and both forms match the oracle on sampled tokens."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16, DeviceLayer
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300.configs import QWEN3

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    wl = QWEN3
    return DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=synth.seed_for(wl.index, stream=40))


@pytest.mark.parametrize("n,which", [(2, "min"), (2, "max"), (9, "min"), (9, "mid"), (9, "max"),
                                     (16, "min"), (16, "mid"), (16, "max")])
def test_chosen_ids_pass(oracle_mod, layer, n, which):
    wl = QWEN3
    m, N = wl.m, wl.N
    U = {"min": m, "max": min(N, n * m), "mid": (m + min(N, n * m)) // 2}[which]
    ids_h = synth.chosen_ids(n, m, N, U, seed=1000 + 17 * n + U)
    rng = np.random.default_rng(n * 131 + U)
    g = rng.uniform(0.1, 1.0, (n, m)).astype(np.float32)
    g /= g.sum(axis=1, keepdims=True)
    ids = torch.from_numpy(ids_h).cuda()
    gates = torch.from_numpy(g).cuda()
    x = layer.activations(n, seed=2000 + n)
    grp = api.group_slots(ids, N, ws=layer.ws)
    ys = api.expert_op_perslot(layer.layer, layer.w, x, ids, gates, ws=layer.ws)
    yd = api.expert_op_dedup(layer.layer, layer.w, x, gates, grp, ws=layer.ws)
    torch.cuda.synchronize()
    assert api.last_device_error(layer.ws) == 0
    assert int(grp.num_distinct.item()) == U == oracle_mod.pass_bytes(wl.d, wl.f, N, ids_h)["U"]
    ys, yd = ys.cpu().numpy(), yd.cpu().numpy()
    xh = synth.host_array(x)
    for t in sorted({0, n // 2, n - 1}):
        sub = layer.host_experts(ids_h[t])
        local = np.arange(m, dtype=np.int32)[None, :].repeat(n, axis=0)
        y_ref = oracle_mod.expert_op_token(*sub, xh, local, g.astype(np.float64), t)
        rms = np.sqrt(np.mean(y_ref ** 2))
        for y in (ys, yd):
            assert np.max(np.abs(y[t] - y_ref)) <= TOL_BF16 * rms
