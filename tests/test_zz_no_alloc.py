"""The entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: code running under a memory manager that owns every
device byte (a serving framework's caching allocator, a fixed arena budgeted ahead of
time) and code on a latency-critical path, where allocation synchronises the device.
moe_expert_op_perslot_noalloc runs the per-slot expert operation with its scratch in a
static array inside the library.  This file is collected last so that a run stopping at
its first failure has already run every other test; it also passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import DeviceLayer, rel_max_err, route
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300 import build as mbuild
from moe_speculative_decoding_gb300.configs import QWEN3

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def noalloc():
    mbuild.build()
    fn = api.lib().moe_expert_op_perslot_noalloc
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(api.Layer), P, P, P, P, P, P, I32, I32, P, P, P]
    fn.restype = I32
    return fn


def _call(fn, layer, w, x, ids, gates, y, status):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.byref(layer), *(ctypes.c_void_p(t.data_ptr()) for t in w), ctypes.c_void_p(x.data_ptr()),
              ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(gates.data_ptr()), x.shape[0], 0,
              ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(status.data_ptr()), stream)


def test_no_alloc_entry_point_matches_workspace_entry_point(noalloc):
    wl = QWEN3
    dl = DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=500)
    n = 6
    x = dl.activations(n, seed=501)
    _, logits = synth.routing_traces(1, n, wl.N, wl.m, 0.5, seed=502)
    ids, gates = route(logits[0], wl.m)
    y_ref = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):   # two calls in a row share the library's scratch
        y = torch.full((n, wl.d), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(noalloc, dl.layer, dl.w, x, ids, gates, y, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # same kernels as the workspace call; the fp32 atomics of the combine add in
        # run-dependent order
        assert rel_max_err(y.cpu().numpy(), y_ref) <= 1e-4


def test_no_alloc_reports_device_errors_per_call(noalloc):
    dl = DeviceLayer(256, 128, 8, 2, "bf16", seed=510)
    x = dl.activations(2, seed=511)
    gates = torch.full((2, 2), 0.5, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.zeros((2, 256), dtype=torch.float32, device="cuda")
    bad = torch.tensor([[0, 9], [1, 2]], dtype=torch.int32, device="cuda")
    assert _call(noalloc, dl.layer, dl.w, x, bad, gates, y, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 5          # MOE_ERR_BAD_ID, the bad slot skipped
    good = torch.tensor([[0, 3], [1, 2]], dtype=torch.int32, device="cuda")
    assert _call(noalloc, dl.layer, dl.w, x, good, gates, y, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0          # cleared at the start of the next call
    y_ws = api.expert_op_perslot(dl.layer, dl.w, x, good, gates, ws=dl.ws).cpu().numpy()
    assert rel_max_err(y.cpu().numpy(), y_ws) <= 1e-4


def test_no_alloc_alternating_layer_shapes(noalloc):
    """Calls that alternate between layers of different (f, m) share the scratch: its
    tensor-core flag region moves with the shape and starts from zero after every change, so
    every call still matches the workspace call."""
    a = DeviceLayer(1024, 768, 32, 8, "bf16", seed=520)
    b = DeviceLayer(1024, 256, 16, 2, "bf16", seed=521)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rep in range(3):
        for dl, n in ((a, 16), (b, 5), (a, 3), (b, 16)):
            x = dl.activations(n, seed=522 + rep + n)
            _, logits = synth.routing_traces(1, n, dl.N, dl.m, 0.4, seed=523 + rep + n)
            ids, gates = route(logits[0], dl.m)
            y_ref = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
            y = torch.full((n, dl.d), float("nan"), dtype=torch.float32, device="cuda")
            assert _call(noalloc, dl.layer, dl.w, x, ids, gates, y, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert rel_max_err(y.cpu().numpy(), y_ref) <= 1e-4
