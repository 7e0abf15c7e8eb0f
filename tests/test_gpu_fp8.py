"""The e4m3 (FP8) expert operation against the oracle: the device quantization is bit-exact,
and both forms match the oracle's FP8 expert operation on a small layer (every token) and on
the Qwen3-30B-A3B-shaped layer (sampled tokens)."""
import numpy as np
import pytest
import torch

from gpu_util import TOL_BF16, route
from moe_speculative_decoding_gb300 import api, synth
from moe_speculative_decoding_gb300.configs import QWEN3

pytestmark = pytest.mark.gpu


def test_quantize_rows_matches_oracle(oracle_mod):
    rng = np.random.default_rng(200)
    for dt in (torch.float32, torch.bfloat16):
        src = torch.from_numpy((rng.normal(0, 1, (70, 384)) * rng.uniform(1e-3, 30, (70, 1))).astype(np.float32))
        src[5] = 0.0
        src[9, 7] = 1e4
        src = src.to(dt)
        q, sc = api.quantize_rows_e4m3(src.cuda())
        host = src.float().numpy() if dt == torch.float32 else synth.bf16_bits(src)
        q_ref, sc_ref = oracle_mod.quantize_rows_e4m3(host)
        assert np.array_equal(q.cpu().numpy(), q_ref)
        assert np.array_equal(sc.cpu().numpy(), sc_ref)


class Fp8Layer:
    def __init__(self, d, f, N, m, seed):
        self.d, self.f, self.N, self.m = d, f, N, m
        self.layer = api.make_layer(d, f, N, m, "e4m3")
        gen = "cuda" if d * f * N * 6 > (64 << 20) else "cpu"
        w = tuple(t.cuda() for t in synth.expert_weights(N, f, d, torch.bfloat16, seed, device=gen))
        self.wq, self.ws_ = api.quantize_experts(w)
        self.ws = api.workspace(self.layer, 16, "cuda")

    def host_experts(self, experts):
        idx = torch.as_tensor(np.asarray(experts, np.int64), device="cuda")
        codes = tuple(t.index_select(0, idx).cpu().numpy() for t in self.wq)
        scales = tuple(t.index_select(0, idx).cpu().numpy() for t in self.ws_)
        return codes, scales


def _run_and_check(oracle_mod, L, n, ids, gates, x, tokens):
    xq, sx = api.quantize_rows_e4m3(x)
    grp = api.group_slots(ids, L.N, ws=L.ws)
    ys = api.expert_op_perslot_fp8(L.layer, L.wq, L.ws_, xq, sx, ids, gates, ws=L.ws)
    yd = api.expert_op_dedup_fp8(L.layer, L.wq, L.ws_, xq, sx, gates, grp, ws=L.ws)
    torch.cuda.synchronize()
    assert api.last_device_error(L.ws) == 0
    ys, yd = ys.cpu().numpy(), yd.cpu().numpy()
    ids_h, g_h = ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64)
    xq_h, sx_h = xq.cpu().numpy(), sx.cpu().numpy()
    worst = 0.0
    for t in tokens:
        (cg, cu, cd), (sg, su, sd) = L.host_experts(ids_h[t])
        local = np.arange(L.m, dtype=np.int32)[None, :].repeat(n, axis=0)
        y_ref = oracle_mod.expert_op_token_fp8(cg, cu, cd, sg, su, sd, xq_h, sx_h, local, g_h, t)
        rms = np.sqrt(np.mean(y_ref ** 2))
        for y in (ys, yd):
            err = np.max(np.abs(y[t] - y_ref)) / rms
            worst = max(worst, err)
            assert err <= TOL_BF16, (t, err)
    return ys, yd, worst


def test_fp8_small_layer_every_token(oracle_mod):
    d, f, N, m, n = 256, 256, 16, 4, 6
    L = Fp8Layer(d, f, N, m, seed=210)
    _, lg = synth.routing_traces(1, n, N, m, 0.5, seed=211)
    ids, gates = route(lg[0], m)
    x = synth.activations(n, d, torch.bfloat16, 212, device="cuda")
    _run_and_check(oracle_mod, L, n, ids, gates, x, range(n))


@pytest.mark.parametrize("n,which", [(1, "rho"), (16, "rho"), (16, "min"), (16, "max"), (7, "rho")])
def test_fp8_qwen3_layer(oracle_mod, n, which):
    wl = QWEN3
    L = Fp8Layer(wl.d, wl.f, wl.N, wl.m, seed=synth.seed_for(wl.index, stream=50))
    if which == "rho":
        _, lg = synth.routing_traces(1, n, wl.N, wl.m, 0.5, seed=220 + n)
        ids, gates = route(lg[0], wl.m)
    else:
        U = wl.m if which == "min" else min(wl.N, n * wl.m)
        ids = torch.from_numpy(synth.chosen_ids(n, wl.m, wl.N, U, seed=230 + U)).cuda()
        gates = torch.full((n, wl.m), 1.0 / wl.m, device="cuda")
    x = synth.activations(n, wl.d, torch.bfloat16, 240 + n, device="cuda")
    _run_and_check(oracle_mod, L, n, ids, gates, x, sorted({0, n // 2, n - 1}))


def test_fp8_close_to_bf16():
    """The e4m3 operation stays within its quantization error of the bf16 one."""
    wl = QWEN3
    n = 8
    w = tuple(t.cuda() for t in synth.expert_weights(wl.N, wl.f, wl.d, torch.bfloat16, 260, device="cuda"))
    Lb = api.make_layer(wl.d, wl.f, wl.N, wl.m, "bf16")
    L8 = api.make_layer(wl.d, wl.f, wl.N, wl.m, "e4m3")
    wq, sc = api.quantize_experts(w)
    _, lg = synth.routing_traces(1, n, wl.N, wl.m, 0.3, seed=261)
    ids, gates = route(lg[0], wl.m)
    x = synth.activations(n, wl.d, torch.bfloat16, 262, device="cuda")
    xq, sx = api.quantize_rows_e4m3(x)
    yb = api.expert_op_perslot(Lb, w, x, ids, gates).cpu().numpy()
    y8 = api.expert_op_perslot_fp8(L8, wq, sc, xq, sx, ids, gates).cpu().numpy()
    rel = np.sqrt(np.mean((y8 - yb) ** 2)) / np.sqrt(np.mean(yb ** 2))
    assert 1e-4 < rel < 0.1, rel
