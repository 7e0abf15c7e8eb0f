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

from gpu_util import TOL_BF16, TOL_F32, DeviceLayer, rel_max_err, route
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


def _oracle_tokens(oracle_mod, dl, x, ids, gates, tokens):
    """The oracle's output rows for the listed tokens, from host copies of their experts."""
    ids_h = ids.cpu().numpy()
    gates_h = gates.cpu().numpy().astype(np.float64)
    xh = synth.host_array(x)
    local = np.arange(dl.m, dtype=np.int32)[None, :].repeat(x.shape[0], axis=0)
    return {t: oracle_mod.expert_op_token(*dl.host_experts(ids_h[t]), xh, local, gates_h, t) for t in tokens}


def test_no_alloc_entry_point_matches_workspace_entry_point(noalloc, oracle_mod):
    wl = QWEN3
    dl = DeviceLayer(wl.d, wl.f, wl.N, wl.m, "bf16", seed=500)
    n = 6
    x = dl.activations(n, seed=501)
    _, logits = synth.routing_traces(1, n, wl.N, wl.m, 0.5, seed=502)
    ids, gates = route(logits[0], wl.m)
    y_ref = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    ref = _oracle_tokens(oracle_mod, dl, x, ids, gates, range(n))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):   # two calls in a row share the library's scratch
        y = torch.full((n, wl.d), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(noalloc, dl.layer, dl.w, x, ids, gates, y, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        yh = y.cpu().numpy()
        # same kernels as the workspace call; the fp32 atomics of the combine add in
        # run-dependent order
        assert rel_max_err(yh, y_ref) <= 1e-4
        # and every token within the output tolerance of the oracle
        for t, yr in ref.items():
            assert np.max(np.abs(yh[t] - yr)) <= TOL_BF16 * np.sqrt(np.mean(yr ** 2))


@pytest.mark.parametrize("dtype,simt,tol", [("f32", False, TOL_F32), ("bf16", True, 1e-3)])
def test_no_alloc_layers_off_the_tensor_core_path(noalloc, oracle_mod, dtype, simt, tol):
    """fp32 layers and bf16 layers with MOE_FLAG_SIMT run the CUDA-core kernel, whose
    workspace is the header alone: the entry point clears no flag region for them, and
    their results match the workspace call and the oracle.  A tensor-core call after them
    still matches its workspace call."""
    dl = DeviceLayer(256, 512, 8, 2, dtype, seed=530, simt=simt)
    n = 4
    x = dl.activations(n, seed=531)
    _, logits = synth.routing_traces(1, n, dl.N, dl.m, 0.3, seed=532)
    ids, gates = route(logits[0], dl.m)
    y_ws = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    ref_ids, ref_gates = oracle_mod.route_topm(logits[0], dl.m)
    ref = oracle_mod.expert_op_perslot(*dl.host(), synth.host_array(x), ref_ids, ref_gates)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        y = torch.full((n, dl.d), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(noalloc, dl.layer, dl.w, x, ids, gates, y, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_max_err(y.cpu().numpy(), y_ws) <= 1e-4
        assert rel_max_err(y.cpu().numpy(), ref) <= tol
    tc = DeviceLayer(256, 512, 8, 2, "bf16", seed=533)
    y_tc_ws = api.expert_op_perslot(tc.layer, tc.w, x.to(torch.bfloat16), ids, gates, ws=tc.ws).cpu().numpy()
    y = torch.full((n, tc.d), float("nan"), dtype=torch.float32, device="cuda")
    assert _call(noalloc, tc.layer, tc.w, x.to(torch.bfloat16), ids, gates, y, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rel_max_err(y.cpu().numpy(), y_tc_ws) <= 1e-4


def _graph_node_count(graph):
    """Nodes of a captured graph, through the driver API (libcuda is on every GPU machine)."""
    cu = ctypes.CDLL("libcuda.so.1")
    count = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(ctypes.c_void_p(graph.raw_cuda_graph()), None, ctypes.byref(count)) == 0
    return count.value


def test_no_alloc_rejects_bad_layers_before_any_device_work(noalloc):
    """A layer the library does not support (m > N, f not a multiple of 64, a huge f) or an
    unsupported pass size is rejected with the status the workspace call gives, and the
    rejected call enqueues nothing: captured on a stream, it leaves an empty graph, and the
    status word it was given keeps its value."""
    good = DeviceLayer(256, 128, 8, 2, "bf16", seed=540)
    x = good.activations(2, seed=541)
    ids = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    gates = torch.full((2, 2), 0.5, device="cuda")
    y = torch.zeros((2, 256), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    assert _call(noalloc, good.layer, good.w, x, ids, gates, y, status) == 0   # sets up the device
    torch.cuda.synchronize()
    bad_layers = [api.make_layer(256, 128, 2, 3),        # m > N
                  api.make_layer(256, 96, 8, 2),         # f not a multiple of 64
                  api.make_layer(256, 1 << 20, 8, 2)]    # f beyond the supported range
    for L in bad_layers:
        want = api.lib().moe_expert_op_perslot(ctypes.byref(L), *(ctypes.c_void_p(t.data_ptr()) for t in good.w),
                                              ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                                              ctypes.c_void_p(gates.data_ptr()), 2, 0, ctypes.c_void_p(y.data_ptr()),
                                              ctypes.c_void_p(good.ws.data_ptr()), good.ws.numel(),
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert want in (1, 2)   # MOE_ERR_ARG or MOE_ERR_UNSUPPORTED
        status.fill_(-7)
        torch.cuda.synchronize()
        try:
            g = torch.cuda.CUDAGraph(keep_graph=True)
        except TypeError:
            g = None
        if g is not None:
            with torch.cuda.graph(g):
                got = _call(noalloc, L, good.w, x, ids, gates, y, status)
            assert _graph_node_count(g) == 0
        else:
            got = _call(noalloc, L, good.w, x, ids, gates, y, status)
        torch.cuda.synchronize()
        assert got == want
        assert int(status.item()) == -7
    # a pass size outside the per-slot range
    big = torch.zeros((65, 256), dtype=torch.bfloat16, device="cuda")
    assert _call(noalloc, good.layer, good.w, big, ids, gates, y, status) == 2


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


def test_no_alloc_wide_simt_layer_clears_nothing_beyond_the_header(noalloc):
    """A CUDA-core layer whose tensor-core flag region would exceed the scratch (f = 65536,
    top-22) needs only the workspace header: the call runs and matches the workspace call."""
    dl = DeviceLayer(64, 65536, 24, 22, "bf16", seed=550, simt=True)
    x = dl.activations(1, seed=551)
    ids = torch.arange(22, dtype=torch.int32, device="cuda").reshape(1, 22)
    gates = torch.full((1, 22), 1.0 / 22, device="cuda")
    y_ws = api.expert_op_perslot(dl.layer, dl.w, x, ids, gates, ws=dl.ws).cpu().numpy()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = torch.full((1, 64), float("nan"), dtype=torch.float32, device="cuda")
    assert _call(noalloc, dl.layer, dl.w, x, ids, gates, y, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rel_max_err(y.cpu().numpy(), y_ws) <= 1e-4
