"""Failure detection without a GPU fault.

Every pipeline wait of the expert kernel is bounded.  A wait that runs out raises the CTA's
abort flag, records MOE_ERR_DEVICE_TIMEOUT in the workspace's error word, waits (bounded)
for the copies and tensor-core operations in flight, frees its tensor memory and returns;
CTAs waiting for an aborted CTA's flags run out in turn.  Here the limit is made far shorter
than the call's normal waits (moe_set_wait_limit), so that the call gives up, and the next
ordinary call on the same workspace must still match the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16, DeviceLayer, route
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300.configs import QWEN3

pytestmark = pytest.mark.gpu

# about 1 us at the maximum SM clock: shorter than the first weight copy's arrival, so some
# wait of every CTA runs out
SHORT_LIMIT_CYCLES = 2000


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_speculative_decoding_gb300 import build
    build.build()
    api.lib()


def _oracle_rows(oracle_mod, dl, x, ids, gates, tokens):
    ids_h = ids.cpu().numpy()
    gates_h = gates.cpu().numpy().astype(np.float64)
    xh = synth.host_array(x)
    local = np.arange(dl.m, dtype=np.int32)[None, :].repeat(x.shape[0], axis=0)
    return {t: oracle_mod.expert_op_token(*dl.host_experts(ids_h[t]), xh, local, gates_h, t) for t in tokens}


@pytest.mark.parametrize("form", ["perslot", "dedup_ids"])
def test_wait_that_runs_out_reports_timeout_then_next_call_matches_oracle(oracle_mod, form):
    wl = QWEN3
    dl = DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=600)
    n = 16
    x = dl.activations(n, seed=601)
    _, logits = synth.routing_traces(1, n, wl.N, wl.m, 0.4, seed=602)
    ids, gates = route(logits[0], wl.m)

    def call():
        if form == "perslot":
            return api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws)
        return api.expert_op_dedup_ids(dl.layer, dl.w, x, ids, gates, ws=dl.ws)

    assert api.last_device_error(dl.ws) == 0
    try:
        api.set_wait_limit(SHORT_LIMIT_CYCLES)
        call()
        code = api.last_device_error(dl.ws)   # synchronises: the aborted call has returned
    finally:
        api.set_wait_limit(0)
    assert code == 6   # MOE_ERR_DEVICE_TIMEOUT
    # the context and the workspace stay usable: the next call is exact to tolerance
    ref = _oracle_rows(oracle_mod, dl, x, ids, gates, (0, 7, 15))
    for _ in range(2):
        y = call().cpu().numpy()
        assert api.last_device_error(dl.ws) == 0
        for t, yr in ref.items():
            assert np.max(np.abs(y[t] - yr)) <= TOL_BF16 * np.sqrt(np.mean(yr ** 2))

