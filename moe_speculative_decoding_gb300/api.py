"""Python binding of libmoeverify.so: argument marshalling only.

Every step of the verify-pass expert operation runs in the library's CUDA kernels; this
module checks tensor devices, dtypes and shapes, passes raw pointers and the current
torch stream, and turns status codes into exceptions.  There is no fallback: if the
library is missing, every call raises MoeError.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

from . import build as _build

MOE_F32, MOE_BF16, MOE_E4M3 = 0, 1, 2
MOE_FLAG_SIMT = 1
MAX_PASS_TOKENS = 64        # tokens per pass of every expert-operation call
PERSLOT_LAUNCH_TOKENS = 16  # tokens per launch of the per-slot calls (a longer pass is split)
MAX_PERSLOT_TOKENS = 64     # tokens per per-slot call
STATUS = {0: "MOE_OK", 1: "MOE_ERR_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_BAD_ID", 6: "MOE_ERR_DEVICE_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class Layer(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("N", ctypes.c_int32),
                ("m", ctypes.c_int32), ("w_dtype", ctypes.c_int32), ("x_dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]

    @property
    def torch_dtype(self):
        if self.w_dtype == MOE_E4M3:
            return torch.uint8   # e4m3 codes
        return torch.bfloat16 if self.w_dtype == MOE_BF16 else torch.float32


class _PassBytes(ctypes.Structure):
    _fields_ = [("expert_bytes", ctypes.c_uint64), ("slot_bytes", ctypes.c_uint64),
                ("dedup_bytes", ctypes.c_uint64), ("act_bytes", ctypes.c_uint64),
                ("n", ctypes.c_int32), ("m", ctypes.c_int32), ("U", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("ubar", ctypes.c_double)]


class WeightScales(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p)]


class ThresholdIn(ctypes.Structure):
    _fields_ = [(f, ctypes.c_double) for f in ("mW", "B_k", "beta_1", "tau_1", "dD_over_betaD", "dphi")]


class _ErrorBounds(ctypes.Structure):
    _fields_ = [(f, ctypes.c_double) for f in ("delta", "verify_factor", "decision_log_margin", "regret_factor",
                                               "speedup_lo", "speedup_hi")]


EXPORTED = ("moe_abi_version", "moe_status_str", "moe_workspace_bytes", "moe_workspace_init",
            "moe_route_topm", "moe_group_slots", "moe_expert_op_perslot", "moe_expert_op_dedup",
            "moe_pass_bytes", "moe_bandwidth_report", "moe_expected_union",
            "moe_best_draft_length", "moe_last_device_error", "moe_expert_op_perslot_noalloc",
            "moe_staircase", "moe_speedup", "moe_reuse_threshold", "moe_reuse_threshold_bytes",
            "moe_error_bounds", "moe_kstar_separated", "moe_fit_op_times", "moe_expert_op_perslot_fp8",
            "moe_expert_op_dedup_fp8", "moe_quantize_rows_e4m3", "moe_spec_accept",
            "moe_union_cost_workspace_bytes", "moe_union_cost", "moe_expert_op_dedup_ids",
            "moe_expert_op_dedup_ids_fp8", "moe_read_probe", "moe_set_wait_limit")

_lib = None


def lib_path() -> str:
    """Path of the in-tree libmoeverify.so (library infrastructure)."""
    return _build.LIB


def lib():
    """The loaded library.  Raises MoeError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise MoeError(-1, f"libmoeverify.so not built at {path} "
                           "(run python -m moe_speculative_decoding_gb300.build)")
    L = ctypes.CDLL(path)
    P, I32, SZ, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_double
    LP = ctypes.POINTER(Layer)
    sig = {
        "moe_abi_version": ([], I32),
        "moe_status_str": ([I32], ctypes.c_char_p),
        "moe_workspace_bytes": ([LP, I32], SZ),
        "moe_workspace_init": ([P, SZ, P], I32),
        "moe_route_topm": ([P, I32, I32, I32, I32, P, P, P], I32),
        "moe_group_slots": ([P, I32, I32, I32, P, P, P, P, P, P], I32),
        "moe_expert_op_perslot": ([LP, P, P, P, P, P, P, I32, I32, P, P, SZ, P], I32),
        "moe_expert_op_dedup": ([LP, P, P, P, P, P, I32, P, P, P, P, I32, P, P, SZ, P], I32),
        "moe_pass_bytes": ([LP, P, I32, ctypes.POINTER(_PassBytes)], I32),
        "moe_bandwidth_report": ([I32, I32, P, P, P, P, P, P, P, P, P, P], I32),
        "moe_expected_union": ([I32, I32, I32], D),
        "moe_best_draft_length": ([P, I32, D], I32),
        "moe_last_device_error": ([P, P, P], I32),
        "moe_set_wait_limit": ([ctypes.c_int64], I32),
        "moe_staircase": ([P, I32, P, P, P, P], I32),
        "moe_speedup": ([P, I32, I32, D], D),
        "moe_reuse_threshold": ([I32, D, ctypes.POINTER(ThresholdIn)], D),
        "moe_reuse_threshold_bytes": ([I32, D, D, D, D], D),
        "moe_error_bounds": ([D, ctypes.POINTER(_ErrorBounds)], I32),
        "moe_kstar_separated": ([P, I32, D, D], I32),
        "moe_fit_op_times": ([I32, P, P, P, I32, D, I32, P], I32),
        "moe_expert_op_perslot_fp8": ([LP, P, P, P, ctypes.POINTER(WeightScales), P, P, P, P, I32, I32, P, P, SZ, P],
                                      I32),
        "moe_expert_op_dedup_fp8": ([LP, P, P, P, ctypes.POINTER(WeightScales), P, P, P, I32, P, P, P, P, I32, P,
                                     P, SZ, P], I32),
        "moe_quantize_rows_e4m3": ([P, I32, I32, I32, P, P, P], I32),
        "moe_spec_accept": ([P, P, P, P, P, I32, I32, I32, I32, P, P, P], I32),
        "moe_expert_op_dedup_ids": ([LP, P, P, P, P, P, P, I32, I32, P, P, SZ, P], I32),
        "moe_expert_op_dedup_ids_fp8": ([LP, P, P, P, ctypes.POINTER(WeightScales), P, P, P, P, I32, I32, P, P, SZ, P],
                                        I32),
        "moe_union_cost_workspace_bytes": ([I32], SZ),
        "moe_read_probe": ([P, SZ, P, P], I32),
        "moe_union_cost": ([P, I32, I32, I32, P, I32, P, P, D, P, P, P, P, P, P, SZ, P], I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(code: int, what: str):
    if code != 0:
        raise MoeError(code, what)


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------- layer + workspace

def make_layer(d: int, f: int, N: int, m: int, dtype: str = "bf16", simt: bool = False) -> Layer:
    """A moe_layer_t: hidden size d, expert size f, N experts, top-m, weight/activation dtype ([Lan] §1: the expert operation's shapes)."""
    code = {"bf16": MOE_BF16, "f32": MOE_F32, "e4m3": MOE_E4M3}[dtype]
    return Layer(d, f, N, m, code, code, MOE_FLAG_SIMT if simt else 0)


def workspace(layer: Layer, n_max: int = PERSLOT_LAUNCH_TOKENS, device=None) -> torch.Tensor:
    """A zeroed device workspace for passes of up to n_max tokens (moe_workspace_bytes, moe_workspace_init; infrastructure).

    The default serves per-slot calls of any size (they launch 16 tokens at a time); a
    deduplicating call of n > 16 tokens needs n_max >= n."""
    nbytes = int(lib().moe_workspace_bytes(ctypes.byref(layer), n_max))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    _check(lib().moe_workspace_init(ctypes.c_void_p(ws.data_ptr()), nbytes, _stream(ws.device)),
           "moe_workspace_init")
    return ws


def last_device_error(ws: torch.Tensor) -> int:
    """moe_last_device_error: synchronise, return and clear the workspace's device error code (infrastructure)."""
    code = ctypes.c_int32(0)
    _check(lib().moe_last_device_error(ctypes.c_void_p(ws.data_ptr()), _stream(ws.device),
                                       ctypes.byref(code)), "moe_last_device_error")
    return int(code.value)


def set_wait_limit(cycles: int) -> None:
    """moe_set_wait_limit: SM cycles one device pipeline wait of later expert calls may take
    before the call records MOE_ERR_DEVICE_TIMEOUT and returns (0: the default; infrastructure)."""
    _check(lib().moe_set_wait_limit(int(cycles)), "moe_set_wait_limit")


# ---------------------------------------------------------------- the hot path

def route_topm(logits: torch.Tensor, m: int, renorm: bool = True, ids=None, gates=None):
    """Top-m routing of fp32 logits [n, N] -> (ids int32 [n, m], gates fp32 [n, m])."""
    n, N = logits.shape
    if ids is None:
        ids = torch.empty((n, m), dtype=torch.int32, device=logits.device)
    if gates is None:
        gates = torch.empty((n, m), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topm(_dev(logits, "logits", torch.float32), n, N, m, int(bool(renorm)),
                                _dev(ids, "ids", torch.int32, (n, m)),
                                _dev(gates, "gates", torch.float32, (n, m)), _stream(logits.device)),
           "moe_route_topm")
    return ids, gates


@dataclass
class Grouping:
    num_distinct: torch.Tensor   # int32 [1]
    expert_list: torch.Tensor    # int32 [min(N, n*m)]
    offsets: torch.Tensor        # int32 [min(N, n*m) + 1]
    slot_order: torch.Tensor     # int32 [n*m]

    @staticmethod
    def empty(n: int, m: int, N: int, device) -> "Grouping":
        cap = min(N, n * m)
        z = lambda k: torch.zeros(k, dtype=torch.int32, device=device)
        return Grouping(z(1), z(max(cap, 1)), z(cap + 1), z(n * m))


def group_slots(ids: torch.Tensor, N: int, out: Grouping | None = None, ws=None) -> Grouping:
    """moe_group_slots: the pass's slots grouped by expert, a counting sort ([Lan] §1, App. E): U, expert list, offsets, slot order."""
    n, m = ids.shape
    g = out or Grouping.empty(n, m, N, ids.device)
    _check(lib().moe_group_slots(_dev(ids, "ids", torch.int32), n, m, N,
                                 _dev(g.num_distinct, "num_distinct"), _dev(g.expert_list, "expert_list"),
                                 _dev(g.offsets, "offsets"), _dev(g.slot_order, "slot_order"),
                                 ctypes.c_void_p(ws.data_ptr()) if ws is not None else None,
                                 _stream(ids.device)), "moe_group_slots")
    return g


def _weights(layer: Layer, weights):
    wg, wu, wd = weights
    dt = layer.torch_dtype
    return (_dev(wg, "w_gate", dt, (layer.N, layer.f, layer.d)),
            _dev(wu, "w_up", dt, (layer.N, layer.f, layer.d)),
            _dev(wd, "w_down", dt, (layer.N, layer.d, layer.f)))


def _y(layer, x, y):
    n = x.shape[0]
    if y is None:
        y = torch.empty((n, layer.d), dtype=torch.float32, device=x.device)
    return y, _dev(y, "y", torch.float32, (n, layer.d))


def expert_op_perslot(layer: Layer, weights, x: torch.Tensor, ids: torch.Tensor, gates: torch.Tensor,
                      y=None, accumulate: bool = False, ws=None):
    """moe_expert_op_perslot: the per-slot form of the expert operation, one expert read per slot ([Lan] §1)."""
    n = x.shape[0]
    ws = ws if ws is not None else workspace(layer, n, x.device)
    y, yp = _y(layer, x, y)
    _check(lib().moe_expert_op_perslot(ctypes.byref(layer), *_weights(layer, weights),
                                       _dev(x, "x", layer.torch_dtype, (n, layer.d)),
                                       _dev(ids, "ids", torch.int32, (n, layer.m)),
                                       _dev(gates, "gates", torch.float32, (n, layer.m)), n,
                                       int(bool(accumulate)), yp, ctypes.c_void_p(ws.data_ptr()),
                                       ws.numel(), _stream(x.device)), "moe_expert_op_perslot")
    return y


def expert_op_dedup_ids(layer: Layer, weights, x: torch.Tensor, ids: torch.Tensor, gates: torch.Tensor,
                        y=None, accumulate: bool = False, ws=None):
    """The deduplicating form from ids in one launch (the grouping built inside the kernel)."""
    n = x.shape[0]
    ws = ws if ws is not None else workspace(layer, n, x.device)
    y, yp = _y(layer, x, y)
    _check(lib().moe_expert_op_dedup_ids(ctypes.byref(layer), *_weights(layer, weights),
                                         _dev(x, "x", layer.torch_dtype, (n, layer.d)),
                                         _dev(ids, "ids", torch.int32, (n, layer.m)),
                                         _dev(gates, "gates", torch.float32, (n, layer.m)), n,
                                         int(bool(accumulate)), yp, ctypes.c_void_p(ws.data_ptr()),
                                         ws.numel(), _stream(x.device)), "moe_expert_op_dedup_ids")
    return y


def expert_op_dedup(layer: Layer, weights, x: torch.Tensor, gates: torch.Tensor, grouping: Grouping,
                    y=None, accumulate: bool = False, ws=None):
    """moe_expert_op_dedup: the deduplicating form on a precomputed grouping, each distinct expert read once ([Lan] §1)."""
    n = x.shape[0]
    ws = ws if ws is not None else workspace(layer, n, x.device)
    y, yp = _y(layer, x, y)
    _check(lib().moe_expert_op_dedup(ctypes.byref(layer), *_weights(layer, weights),
                                     _dev(x, "x", layer.torch_dtype, (n, layer.d)),
                                     _dev(gates, "gates", torch.float32, (n, layer.m)), n,
                                     _dev(grouping.num_distinct, "num_distinct"),
                                     _dev(grouping.expert_list, "expert_list"),
                                     _dev(grouping.offsets, "offsets"),
                                     _dev(grouping.slot_order, "slot_order"),
                                     int(bool(accumulate)), yp, ctypes.c_void_p(ws.data_ptr()),
                                     ws.numel(), _stream(x.device)), "moe_expert_op_dedup")
    return y


# ---------------------------------------------------------------- host-side report

def pass_bytes(layer: Layer, ids_host) -> dict:
    """moe_pass_bytes: E_slot = n m w, E_dedup = U w and u-bar of one pass, on the host ([Lan] §1 "Bytes", §2 "Effective bandwidth")."""
    ids = np.ascontiguousarray(np.asarray(ids_host, dtype=np.int32))
    n = ids.shape[0] if ids.ndim == 2 else ids.size // layer.m
    out = _PassBytes()
    _check(lib().moe_pass_bytes(ctypes.byref(layer), ctypes.c_void_p(ids.ctypes.data), n,
                                ctypes.byref(out)), "moe_pass_bytes")
    return dict(expert_bytes=out.expert_bytes, slot_bytes=out.slot_bytes, dedup_bytes=out.dedup_bytes,
                act_bytes=out.act_bytes, n=out.n, m=out.m, U=out.U, ubar=out.ubar)


def bandwidth_report(n_lo: int, slot_bytes, dedup_bytes, t_slot, t_dedup) -> dict:
    """moe_bandwidth_report: u-bar(n), beta_p, r(n), S(n) and the crossover from bytes and times ([Lan] §2 "Effective bandwidth", §3.1, §2 "Testing the inputs")."""
    arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.float64)) for a in
            (slot_bytes, dedup_bytes, t_slot, t_dedup)]
    count = arrs[0].size
    outs = [np.zeros(count, np.float64) for _ in range(5)]
    cross = ctypes.c_int32(0)
    _check(lib().moe_bandwidth_report(n_lo, count, *[ctypes.c_void_p(a.ctypes.data) for a in arrs],
                                      *[ctypes.c_void_p(o.ctypes.data) for o in outs],
                                      ctypes.byref(cross)), "moe_bandwidth_report")
    res = dict(zip(("beta_slot", "beta_dedup", "ubar", "r", "saving"), outs))
    res["crossover"] = None if cross.value < 0 else int(cross.value)
    return res


def expected_union(N: int, m: int, n: int) -> float:
    """moe_expected_union: E[U] = N (1 - q^n) under uniform routing ([Lan] §1)."""
    return float(lib().moe_expected_union(N, m, n))


def best_draft_length(V, a: float) -> int:
    """moe_best_draft_length: the smallest maximiser k* of G_a(k) / V(k) ([Lan] §1 "Speculative decoding")."""
    V = np.ascontiguousarray(np.asarray(V, dtype=np.float64))
    k = int(lib().moe_best_draft_length(ctypes.c_void_p(V.ctypes.data), V.size - 1, float(a)))
    if k < 0:
        raise MoeError(1, "moe_best_draft_length")
    return k


# ---------------------------------------------------------------- step-time theory
def _times(V) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(V, dtype=np.float64))


def staircase(V) -> dict:
    """a0, the step points a_step[0..kmax] (a_step[0] = 0), alpha[k, i] and the convex flag."""
    V = _times(V)
    K = V.size
    a0 = ctypes.c_double(0.0)
    steps = np.zeros(K, np.float64)
    alpha = np.zeros((K, K), np.float64)
    convex = ctypes.c_int32(0)
    _check(lib().moe_staircase(ctypes.c_void_p(V.ctypes.data), K - 1, ctypes.byref(a0),
                               ctypes.c_void_p(steps.ctypes.data), ctypes.c_void_p(alpha.ctypes.data),
                               ctypes.byref(convex)), "moe_staircase")
    return dict(a0=a0.value, a_step=steps, alpha=alpha, convex=bool(convex.value))


def speedup(V, k: int, a: float) -> float:
    """moe_speedup: T_a(k) / T_a(0) = G_a(k) V(0) / V(k), the speed-up of draft length k ([Lan] §3.2 (9))."""
    V = _times(V)
    return float(lib().moe_speedup(ctypes.c_void_p(V.ctypes.data), V.size - 1, int(k), float(a)))


def reuse_threshold(k: int, a: float, mW: float, B_k: float, beta_1: float, tau_1: float,
                    dD_over_betaD: float = 0.0, dphi: float = 0.0) -> float:
    """moe_reuse_threshold: the deduplicating engine's reuse threshold rho*_k(a) in time ([Lan] §3.4 (14), App. B.2 (B.12)-(B.14))."""
    t = ThresholdIn(mW, B_k, beta_1, tau_1, dD_over_betaD, dphi)
    return float(lib().moe_reuse_threshold(int(k), float(a), ctypes.byref(t)))


def reuse_threshold_bytes(k: int, a: float, mW: float, D_1: float = 0.0, D_k1: float = 0.0) -> float:
    """moe_reuse_threshold_bytes: the same threshold with one bandwidth and no fixed time ([Lan] §3.4 (16), (B.16))."""
    return float(lib().moe_reuse_threshold_bytes(int(k), float(a), float(mW), float(D_1), float(D_k1)))


def error_bounds(eps: float) -> dict:
    """moe_error_bounds: delta, the verify factor of (17)-(18) and the decision margin for a relative bandwidth error eps ([Lan] §3.5, Table 2, App. C)."""
    out = _ErrorBounds()
    _check(lib().moe_error_bounds(float(eps), ctypes.byref(out)), "moe_error_bounds")
    return {f: getattr(out, f) for f, _ in _ErrorBounds._fields_}


def kstar_separated(V, a: float, delta: float) -> bool:
    """moe_kstar_separated: the separation condition of (20), under which the predicted k* is the true one ([Lan] §3.5, Table 2)."""
    V = _times(V)
    r = int(lib().moe_kstar_separated(ctypes.c_void_p(V.ctypes.data), V.size - 1, float(a), float(delta)))
    if r < 0:
        raise MoeError(1, "moe_kstar_separated")
    return bool(r)


def fit_op_times(n, U, t, m: int, b: float, form: str) -> tuple:
    """Fit (4) (form 'slot': t_op, c_u, c_re) or (E.1) (form 'dedup': t_op, c_g, c_t)."""
    n = np.ascontiguousarray(np.asarray(n, dtype=np.int32))
    U = np.ascontiguousarray(np.asarray(U, dtype=np.int32))
    t = np.ascontiguousarray(np.asarray(t, dtype=np.float64))
    coef = np.zeros(3, np.float64)
    _check(lib().moe_fit_op_times(n.size, ctypes.c_void_p(n.ctypes.data), ctypes.c_void_p(U.ctypes.data),
                                  ctypes.c_void_p(t.ctypes.data), int(m), float(b), 0 if form == "slot" else 1,
                                  ctypes.c_void_p(coef.ctypes.data)), "moe_fit_op_times")
    return tuple(float(c) for c in coef)


# ---------------------------------------------------------------- FP8 (e4m3) experts
def quantize_rows_e4m3(src: torch.Tensor):
    """Row-wise e4m3 codes (uint8, same shape) and fp32 row scales of a 2-D or 3-D fp32/bf16
    CUDA tensor (rows = all leading dimensions)."""
    if src.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("quantize_rows_e4m3 takes fp32 or bf16")
    cols = src.shape[-1]
    rows = src.numel() // cols
    q = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scale = torch.empty(src.shape[:-1], dtype=torch.float32, device=src.device)
    _check(lib().moe_quantize_rows_e4m3(_dev(src, "src"), MOE_F32 if src.dtype == torch.float32 else MOE_BF16,
                                        rows, cols, ctypes.c_void_p(q.data_ptr()),
                                        ctypes.c_void_p(scale.data_ptr()), _stream(src.device)),
           "moe_quantize_rows_e4m3")
    return q, scale


def quantize_experts(weights):
    """(w_gate, w_up, w_down) bf16/fp32 -> (codes, row scales) for an e4m3 layer."""
    qs = [quantize_rows_e4m3(w) for w in weights]
    return tuple(q for q, _ in qs), tuple(s for _, s in qs)


def _scales(layer: Layer, scales) -> WeightScales:
    sg, su, sd = scales
    return WeightScales(_dev(sg, "s_gate", torch.float32, (layer.N, layer.f)),
                        _dev(su, "s_up", torch.float32, (layer.N, layer.f)),
                        _dev(sd, "s_down", torch.float32, (layer.N, layer.d)))


def expert_op_perslot_fp8(layer: Layer, weights, scales, xq: torch.Tensor, x_scale: torch.Tensor, ids: torch.Tensor,
                          gates: torch.Tensor, y=None, accumulate: bool = False, ws=None):
    """moe_expert_op_perslot_fp8: the per-slot form on e4m3 experts with row scales (the quantized experts of [Lan] App. E Table 6)."""
    n = xq.shape[0]
    ws = ws if ws is not None else workspace(layer, n, xq.device)
    y, yp = _y(layer, xq, y)
    sc = _scales(layer, scales)
    _check(lib().moe_expert_op_perslot_fp8(ctypes.byref(layer), *_weights(layer, weights), ctypes.byref(sc),
                                           _dev(xq, "x", torch.uint8, (n, layer.d)),
                                           _dev(x_scale, "x_scale", torch.float32, (n,)),
                                           _dev(ids, "ids", torch.int32, (n, layer.m)),
                                           _dev(gates, "gates", torch.float32, (n, layer.m)), n,
                                           int(bool(accumulate)), yp, ctypes.c_void_p(ws.data_ptr()),
                                           ws.numel(), _stream(xq.device)), "moe_expert_op_perslot_fp8")
    return y


def expert_op_dedup_ids_fp8(layer: Layer, weights, scales, xq: torch.Tensor, x_scale: torch.Tensor, ids: torch.Tensor,
                            gates: torch.Tensor, y=None, accumulate: bool = False, ws=None):
    """moe_expert_op_dedup_ids_fp8: the deduplicating form from ids on e4m3 experts, the grouping built in the kernel ([Lan] §1; App. E Table 6)."""
    n = xq.shape[0]
    ws = ws if ws is not None else workspace(layer, n, xq.device)
    y, yp = _y(layer, xq, y)
    sc = _scales(layer, scales)
    _check(lib().moe_expert_op_dedup_ids_fp8(ctypes.byref(layer), *_weights(layer, weights), ctypes.byref(sc),
                                             _dev(xq, "x", torch.uint8, (n, layer.d)),
                                             _dev(x_scale, "x_scale", torch.float32, (n,)),
                                             _dev(ids, "ids", torch.int32, (n, layer.m)),
                                             _dev(gates, "gates", torch.float32, (n, layer.m)), n,
                                             int(bool(accumulate)), yp, ctypes.c_void_p(ws.data_ptr()),
                                             ws.numel(), _stream(xq.device)), "moe_expert_op_dedup_ids_fp8")
    return y


def expert_op_dedup_fp8(layer: Layer, weights, scales, xq: torch.Tensor, x_scale: torch.Tensor, gates: torch.Tensor,
                        grouping: Grouping, y=None, accumulate: bool = False, ws=None):
    """moe_expert_op_dedup_fp8: the deduplicating form on e4m3 experts and a precomputed grouping ([Lan] §1; App. E Table 6)."""
    n = xq.shape[0]
    ws = ws if ws is not None else workspace(layer, n, xq.device)
    y, yp = _y(layer, xq, y)
    sc = _scales(layer, scales)
    _check(lib().moe_expert_op_dedup_fp8(ctypes.byref(layer), *_weights(layer, weights), ctypes.byref(sc),
                                         _dev(xq, "x", torch.uint8, (n, layer.d)),
                                         _dev(x_scale, "x_scale", torch.float32, (n,)),
                                         _dev(gates, "gates", torch.float32, (n, layer.m)), n,
                                         _dev(grouping.num_distinct, "num_distinct"),
                                         _dev(grouping.expert_list, "expert_list"),
                                         _dev(grouping.offsets, "offsets"),
                                         _dev(grouping.slot_order, "slot_order"),
                                         int(bool(accumulate)), yp, ctypes.c_void_p(ws.data_ptr()),
                                         ws.numel(), _stream(xq.device)), "moe_expert_op_dedup_fp8")
    return y


# ---------------------------------------------------------------- verify-side neighbours
def spec_accept(draft, q, p, r, u, greedy: bool = False, n_accepted=None, token=None):
    """One round of speculative sampling for B sequences ("Lossless but Not Free", §3.1,
    Algorithm 1) on the device.  draft int32 [B, K], q fp32 [B, K, V], p fp32 [B, K+1, V],
    r fp32 [B, K], u fp32 [B] (q, r, u may be None when greedy).  Returns (n_accepted, token),
    int32 [B] each."""
    B, K1, V = p.shape
    K = K1 - 1
    dev = p.device
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=dev)
    dptr = lambda t, name, dt: None if t is None else _dev(t, name, dt)
    _check(lib().moe_spec_accept(dptr(draft, "draft", torch.int32) if K else None, dptr(q, "q", torch.float32),
                                 _dev(p, "p", torch.float32), dptr(r, "r", torch.float32), dptr(u, "u", torch.float32),
                                 B, K, V, int(bool(greedy)), _dev(n_accepted, "n_accepted", torch.int32),
                                 _dev(token, "token", torch.int32), _stream(dev)), "moe_spec_accept")
    return n_accepted, token


def union_cost(bitmaps, subsets, pv, bcoef, beta: float, out=None, ws=None):
    """SpecFit §3.2 eqs (3)-(5) on the device: bitmaps uint64-as-int64 [nodes+1, L, W], subsets
    int32/uint32 bits [S], pv float64 [nodes], bcoef float64 [nodes+1].  Returns dict(F, size,
    R, T, best) of device tensors."""
    nodes1, L, W = bitmaps.shape
    S = subsets.numel()
    dev = bitmaps.device
    if out is None:
        out = dict(F=torch.empty(S, dtype=torch.int32, device=dev), size=torch.empty(S, dtype=torch.int32, device=dev),
                   R=torch.empty(S, dtype=torch.float64, device=dev), T=torch.empty(S, dtype=torch.float64, device=dev),
                   best=torch.empty(1, dtype=torch.int32, device=dev))
    if ws is None:
        ws = torch.empty(int(lib().moe_union_cost_workspace_bytes(S)), dtype=torch.uint8, device=dev)
    _check(lib().moe_union_cost(_dev(bitmaps, "bitmaps", torch.int64), nodes1 - 1, L, W,
                                _dev(subsets, "subsets", torch.int32), S,
                                _dev(pv, "pv", torch.float64) if nodes1 > 1 else None,
                                _dev(bcoef, "bcoef", torch.float64), float(beta),
                                _dev(out["F"], "F", torch.int32), _dev(out["size"], "size", torch.int32),
                                _dev(out["R"], "R", torch.float64), _dev(out["T"], "T", torch.float64),
                                _dev(out["best"], "best", torch.int32), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                _stream(dev)), "moe_union_cost")
    return out


def read_probe(buf: torch.Tensor, ws: torch.Tensor) -> int:
    """Enqueue the read-only streaming probe over buf (a CUDA tensor); returns the bytes it reads."""
    nbytes = buf.numel() * buf.element_size()
    _check(lib().moe_read_probe(ctypes.c_void_p(buf.data_ptr()), nbytes, ctypes.c_void_p(ws.data_ptr()),
                                _stream(buf.device)), "moe_read_probe")
    return nbytes // 32768 * 32768
