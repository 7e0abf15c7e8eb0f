"""Helpers shared by the GPU parity tests: seeded layers on the device, oracle calls on
host copies, and the output tolerance."""
import numpy as np
import torch

from moe_speculative_decoding_gb300 import api, synth

# Output tolerance of the expert operation: max|y - y_ref| <= 2e-2 * rms(y_ref) for bf16
# weights with fp32 accumulation (the stated target).  fp32 layers must meet a far
# tighter bound: both sides use the same fp32 inputs, only summation order and
# precision (fp32 vs fp64) differ.
TOL_BF16 = 2e-2
TOL_F32 = 1e-4


def rel_max_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(y - ref))) / max(rms, 1e-30)


class DeviceLayer:
    """A seeded layer resident on the GPU, plus host copies on demand."""

    def __init__(self, d, f, N, m, dtype="bf16", seed=0, simt=False, device="cuda"):
        self.d, self.f, self.N, self.m = d, f, N, m
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.layer = api.make_layer(d, f, N, m, dtype, simt=simt)
        gen_dev = device if d * f * N * 6 > (64 << 20) else "cpu"
        w = synth.expert_weights(N, f, d, self.tdtype, seed, device=gen_dev)
        self.w = tuple(t.to(device) for t in w)
        self.ws = api.workspace(self.layer, 16, device)
        self._host = None

    def host(self):
        if self._host is None:
            self._host = tuple(synth.host_array(t) for t in self.w)
        return self._host

    def host_experts(self, experts):
        """Host copies of only the listed experts (for large layers)."""
        idx = torch.as_tensor(np.asarray(experts, np.int64), device=self.w[0].device)
        return tuple(synth.host_array(t.index_select(0, idx)) for t in self.w)

    def activations(self, n, seed):
        return synth.activations(n, self.d, self.tdtype, seed, device="cuda")


def route(logits_np, m):
    logits = torch.from_numpy(np.ascontiguousarray(logits_np)).cuda()
    return api.route_topm(logits, m)
