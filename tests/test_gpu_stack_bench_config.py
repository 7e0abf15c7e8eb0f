"""Parity at the bench's full size and in the launch configuration bench.py times: the
48-layer Qwen3-30B-A3B-shaped stack (57.98 GB resident), CUDA-graph replays of the timed
phases (route over all layers' tokens, 48 per-slot launches, 48 deduplicating launches that
group their slots themselves), checked on sampled layers and tokens against the oracle one
token at a time; the standalone grouping of the same window checks U."""
import os
import sys

import numpy as np
import pytest
import torch

from conftest import ROOT
from gpu_util import TOL_BF16
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300.configs import QWEN3_STACK

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def stack():
    from moe_speculative_decoding_gb300 import build
    build.build()
    sys.path.insert(0, ROOT)
    import bench
    b = bench.StackBench(QWEN3_STACK, QWEN3_STACK.layers, [1, 8, 16], windows=2,
                         device=torch.device("cuda", 0), use_graph=True)
    b.capture()
    b.step(1)               # the second window, as a timed step would
    for n in b.n_values:    # the standalone grouping of the same window, for the U check
        b._run(n, "group")
    torch.cuda.synchronize()
    assert api.last_device_error(b.ws) == 0
    yield b
    del b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [1, 8, 16])
def test_stack_graph_replay_matches_oracle(oracle_mod, stack, n):
    b = stack
    wl = b.wl
    st = b.per_n[n]
    ids_all = st["ids"].cpu().numpy()
    logits = st["logits"].cpu().numpy()
    x_host = synth.host_array(st["x"])
    for layer in (0, 23, 47):
        lg = logits[layer * n:(layer + 1) * n]
        ref_ids, ref_gates = oracle_mod.route_topm(lg, wl.m)
        assert np.array_equal(ids_all[layer * n:(layer + 1) * n], ref_ids)
        # the ids are the trace's sets for this window
        for t in range(n):
            assert set(ref_ids[t].tolist()) == set(b.sets[layer, n + t].tolist())
        U = int(st["groups"][layer].num_distinct.item())
        assert U == oracle_mod.pass_bytes(wl.d, wl.f, wl.N, ref_ids)["U"]
        ys = st["y_slot"][layer].cpu().numpy()
        yd = st["y_dedup"][layer].cpu().numpy()
        for t in sorted({0, n - 1}):
            idx = torch.as_tensor(ref_ids[t].astype(np.int64), device=b.weights[layer][0].device)
            sub = tuple(synth.host_array(w.index_select(0, idx)) for w in b.weights[layer])
            local = np.arange(wl.m, dtype=np.int32)[None, :].repeat(n, axis=0)
            y_ref = oracle_mod.expert_op_token(*sub, x_host, local, ref_gates, t)
            rms = np.sqrt(np.mean(y_ref ** 2))
            assert np.max(np.abs(ys[t] - y_ref)) <= TOL_BF16 * rms
            assert np.max(np.abs(yd[t] - y_ref)) <= TOL_BF16 * rms
