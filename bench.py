#!/usr/bin/env python3
"""Benchmark of the MoE verify-pass expert operation on GB300.

Metric: expert-operation µs per pass and achieved HBM TB/s on requested expert bytes,
against the pass size n = 1..16, for the per-slot and the deduplicating forms.

Workload (default): a 48-layer Qwen3-30B-A3B-shaped expert stack (d=2048, N=128 experts,
top-8, f=768, bf16; 57.98 GB resident), per-layer seeded routing traces with reuse 0.4,
one shared pass x for every layer.  One *step* is one verification pass at every
n = 1..16 through all 48 layers in both forms:
    route (top-m of the 48*n router logits, one launch)
    per-slot pass   (48 expert launches)
    grouping        (48 counting sorts)
    dedup pass      (48 expert launches)
Each (n, phase) is a CUDA graph of the library's own kernels; events between the phases
give the per-form times.  The weights (58 GB) are far larger than L2, and the layers run
one after another, so no pass finds its weights in L2 from a previous pass.

value    = expert bytes requested by both forms in the step / step time (TB/s, decimal).
e2e      = the same with the step's inputs copied from pinned host memory and the outputs
           copied back inside the timed region.
roofline = the expert kernel: requested bytes per launch / its mean launch time, against
           the measured HBM copy bandwidth.

--impl reference times the CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_speculative_decoding_gb300 import api, synth  # noqa: E402
from moe_speculative_decoding_gb300 import build as mbuild  # noqa: E402
from moe_speculative_decoding_gb300.configs import BY_NAME, DSV2_LITE, MIXTRAL, QWEN3, QWEN3_STACK  # noqa: E402

METRIC = "MoE verify-pass expert-op µs and achieved HBM TB/s vs pass size n=1..16"
UNIT = "TB/s"
EXPERT_OP = "expert_tc_kernel"
A_GRID = [round(0.10 + 0.05 * i, 2) for i in range(18)]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=QWEN3_STACK.name, choices=sorted(BY_NAME))
    p.add_argument("--layers", type=int, default=None, help="override the stack depth (smaller test runs)")
    p.add_argument("--n-min", type=int, default=None)
    p.add_argument("--n-max", type=int, default=None)
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-fit", action="store_true", help="skip the chosen-id fits (4) and (E.1)")
    p.add_argument("--no-fp8", action="store_true", help="skip the e4m3 (FP8) expert step")
    p.add_argument("--fit-only", action="store_true",
                   help="only the chosen-id fits, on one freshly generated layer (prints their JSON)")
    p.add_argument("--fit-reps", type=int, default=7)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-verify-side", action="store_true", help="skip the accept/reject and union-cost leg")
    p.add_argument("--verify-side-only", action="store_true", help="run only the accept/reject and union-cost leg")
    p.add_argument("--verify-reps", type=int, default=20)
    p.add_argument("--no-configs", action="store_true",
                   help="skip the page-shaped single-layer workloads (DeepSeek-V2-Lite, Qwen3, Mixtral at each reuse)")
    p.add_argument("--no-long", action="store_true", help="skip the passes of 17..64 tokens")
    p.add_argument("--profile-layer", default=None,
                   help="comma-separated pass sizes, each n (two deduplicating calls from ids) or sn (two per-slot "
                        "calls), on one layer of the workload's shape (a small case for ncu captures; prints ok)")
    p.add_argument("--long-only", action="store_true",
                   help="only the passes of 17..64 tokens on 8 freshly generated layers (prints their JSON)")
    p.add_argument("--configs-only", default=None,
                   help="only the configs leg, for the listed workloads (comma-separated names; prints their JSON)")
    return p.parse_args()


# --------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def step_time_theory(n_values, Vs, Vd, Vw, bytes_slot, bytes_dedup, K):
    """The step-time theory of the pages on the measured expert times (all 48 layers):
    a0, the step points and the convexity test for each engine; for the deduplicating one,
    the mean reuse of the drafted tokens from the union bytes (12) and the reuse threshold in
    time (14) from the measured bandwidths, with the speedup decision (B.14) beside the one
    the step times give directly; and the error bounds at a 10% bandwidth error."""
    out = {}
    for name, V in (("slot", Vs), ("dedup", Vd), ("switched", Vw)):
        st = api.staircase(V)
        out[name] = dict(a0=round(st["a0"], 6), a_step=[round(float(x), 6) for x in st["a_step"]],
                         convex=st["convex"])
    # dedup engine: one-token pass on the per-slot kernel (tau(1) = V(0)), B_k = beta_dedup(k+1)
    mW = bytes_dedup[n_values[0]] / K
    tau1 = Vd[0]
    beta1 = mW / tau1
    kmax = len(n_values) - 1
    rho_bar, B = [], []
    for k in range(1, kmax + 1):
        E = bytes_dedup[n_values[k]] / K
        rho_bar.append(1.0 - (E - mW) / (mW * k))
        B.append(E / Vd[k])
    decisions = {}
    agree = True
    for a in A_GRID:
        thr = [api.reuse_threshold(k, a, mW, B[k - 1], beta1, tau1) for k in range(1, kmax + 1)]
        by_reuse = any(rb > t for rb, t in zip(rho_bar, thr))
        by_time = api.best_draft_length(Vd, a) >= 1
        agree = agree and (by_reuse == by_time)
        decisions[str(a)] = dict(speedup=by_reuse, rho_star=[round(t, 5) for t in thr[:4]])
    out["dedup_reuse"] = dict(rho_bar=[round(x, 5) for x in rho_bar], decisions=decisions,
                              agrees_with_step_times=agree)
    eb = api.error_bounds(0.10)
    out["error_bounds_eps_0.10"] = {k: round(v, 6) for k, v in eb.items()}
    return out


def fp8_leg(b: "StackBench", args, device, per_n_bf16):
    """The same step with e4m3 experts (GB300's FP8 in place of the quantized experts the
    pages' engines run): the stack quantized once, then per n and layer one activation quantization and
    the FP8 expert operation, per-slot and dedup (one launch each; the dedup launch groups the slots).  Timed over the same
    windows after the bf16 measurement; value = FP8 expert bytes requested / time."""
    wl, L = b.wl, b.L
    layer8 = api.make_layer(wl.d, wl.f, wl.N, wl.m, "e4m3")
    ws8 = api.workspace(layer8, 16, device)
    t0 = time.time()
    w8 = [api.quantize_experts(w) for w in b.weights]
    torch.cuda.synchronize(device)
    t_quant = time.time() - t0
    bufs = {}
    for n in b.n_values:
        bufs[n] = dict(xq=torch.empty((L, n, wl.d), dtype=torch.uint8, device=device),
                       sx=torch.empty((L, 16), dtype=torch.float32, device=device),
                       ys=torch.zeros((L, n, wl.d), dtype=torch.float32, device=device),
                       yd=torch.zeros((L, n, wl.d), dtype=torch.float32, device=device))

    def slot8(n):
        st, bf = b.per_n[n], bufs[n]
        for l in range(L):
            xq, sx = bf["xq"][l], bf["sx"][l, :n]
            api._check(api.lib().moe_quantize_rows_e4m3(ctypes.c_void_p(st["x"].data_ptr()), api.MOE_BF16, n, wl.d,
                                                        ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(sx.data_ptr()),
                                                        api._stream(device)), "moe_quantize_rows_e4m3")
            api.expert_op_perslot_fp8(layer8, w8[l][0], w8[l][1], xq, sx, st["ids"][l * n:(l + 1) * n],
                                      st["gates"][l * n:(l + 1) * n], y=bf["ys"][l], accumulate=True, ws=ws8)

    def dedup8(n):
        st, bf = b.per_n[n], bufs[n]
        for l in range(L):
            xq, sx = bf["xq"][l], bf["sx"][l, :n]
            api._check(api.lib().moe_quantize_rows_e4m3(ctypes.c_void_p(st["x"].data_ptr()), api.MOE_BF16, n, wl.d,
                                                        ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(sx.data_ptr()),
                                                        api._stream(device)), "moe_quantize_rows_e4m3")
            api.expert_op_dedup_ids_fp8(layer8, w8[l][0], w8[l][1], xq, sx, st["ids"][l * n:(l + 1) * n],
                                        st["gates"][l * n:(l + 1) * n], y=bf["yd"][l], accumulate=True, ws=ws8)

    graphs = {}
    for n in b.n_values:
        slot8(n), dedup8(n)
        torch.cuda.synchronize(device)
        for ph, fn in (("slot8", slot8), ("dedup8", dedup8)):
            if b.use_graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn(n)
                graphs[(n, ph)] = g
            else:
                graphs[(n, ph)] = (lambda fn=fn, n=n: fn(n))

    def run(n, ph):
        g = graphs[(n, ph)]
        g.replay() if b.use_graph else g()

    def step(w, ev=None):
        for n in b.n_values:
            b.stage(n, w)
            b._run(n, "route")
            bufs[n]["ys"].zero_()
            bufs[n]["yd"].zero_()
            if ev is not None:
                ev[(n, "start")].record()
            for ph in ("slot8", "dedup8"):
                run(n, ph)
                if ev is not None:
                    ev[(n, ph)].record()

    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize(device)
    K = args.steps
    evs = [{(n, k): torch.cuda.Event(enable_timing=True) for n in b.n_values for k in ("start", "slot8", "dedup8")}
           for _ in range(K)]
    for k in range(K):
        step(args.warmup + k, evs[k])
    torch.cuda.synchronize(device)
    assert api.last_device_error(ws8) == 0
    tot_b, tot_t, rows = 0.0, 0.0, []
    bf16 = {r["n"]: r for r in per_n_bf16}
    for n in b.n_values:
        ts = sum(evs[k][(n, "start")].elapsed_time(evs[k][(n, "slot8")]) * 1e-3 for k in range(K))
        td = sum(evs[k][(n, "slot8")].elapsed_time(evs[k][(n, "dedup8")]) * 1e-3 for k in range(K))
        bs = bd = 0
        for k in range(K):
            w = args.warmup + k
            for l in range(L):
                pb = api.pass_bytes(layer8, b.sets[l, w * n:(w + 1) * n])
                bs += pb["slot_bytes"]
                bd += pb["dedup_bytes"]
        tot_b += bs + bd
        tot_t += ts + td
        rows.append(dict(n=n, us_slot=round(ts / K * 1e6, 2), us_dedup=round(td / K * 1e6, 2),
                         tbps_slot=round(bs / ts / 1e12, 3), tbps_dedup=round(bd / td / 1e12, 3),
                         speedup_slot=round(bf16[n]["us_slot"] / (ts / K * 1e6), 3),
                         speedup_dedup=round(bf16[n]["us_dedup"] / (td / K * 1e6), 3)))
    # outputs against the bf16 per-slot pass of the same (last) window: quantization error only;
    # the FP8 forms against each other: accumulation order only
    worst, worst_forms = 0.0, 0.0
    for n in b.n_values:
        b.stage(n, args.warmup + K - 1)
        b._run(n, "route")
        b._run(n, "slot")
        bufs[n]["ys"].zero_()
        bufs[n]["yd"].zero_()
        run(n, "slot8")
        run(n, "dedup8")
        torch.cuda.synchronize(device)
        yb = b.per_n[n]["y_slot"].double()
        y8, y8d = bufs[n]["ys"].double(), bufs[n]["yd"].double()
        rms8 = y8.pow(2).mean().sqrt().clamp_min(1e-30)
        worst = max(worst, float((y8 - yb).pow(2).mean().sqrt() / yb.pow(2).mean().sqrt().clamp_min(1e-30)))
        worst_forms = max(worst_forms, float((y8 - y8d).abs().max() / rms8))
    return dict(value=round(tot_b / tot_t / 1e12, 4), unit="TB/s", dtype="e4m3 weights and activations, fp32 accumulate",
                expert_bytes=int(api.pass_bytes(layer8, b.sets[0, :1])["expert_bytes"]),
                quantize_s=round(t_quant, 2), per_n=rows, rel_rms_vs_bf16=round(worst, 5),
                max_dev_dedup_vs_slot=round(worst_forms, 6),
                launches_per_layer_form=2)


def read_probe_leg(device, gib: int = 4, reps: int = 5):
    """Read-only streaming probe (our TMA bulk-copy kernel) over a 4 GiB buffer: the read
    bandwidth beside the copy peak (read + write) of MEASURED_PEAKS.json."""
    buf = torch.empty(gib << 30, dtype=torch.uint8, device=device)
    buf.fill_(1)
    ws = api.workspace(api.make_layer(256, 256, 8, 2), 1, device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    api.read_probe(buf, ws)
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize(device)
        ev[0].record()
        nbytes = api.read_probe(buf, ws)
        ev[1].record()
        torch.cuda.synchronize(device)
        ts.append(ev[0].elapsed_time(ev[1]) * 1e-3)
    assert api.last_device_error(ws) == 0
    t = float(np.median(ts))
    del buf
    torch.cuda.empty_cache()
    return dict(gbs=round(nbytes / t / 1e9, 1), bytes=int(nbytes), us=round(t * 1e6, 1),
                of_copy_peak=round(nbytes / t / 1e9 / measured_peaks()[0]["hbm_gbs"], 4),
                kernel="read_probe_kernel (1-D TMA bulk copies, one CTA per SM)")


def verify_side_leg(device, reps: int = 20, B: int = 16, K: int = 8, V: int = 151936, nodes: int = 18,
                    layers: int = 48, N: int = 128, m: int = 8):
    """The steps either side of the verification pass, timed on the device.
    Speculative accept/reject ("Lossless but Not Free", §3.1, Algorithm 1) for B sequences of
    K drafts over a V-token vocabulary (Qwen3's 151,936), sampling and greedy; algorithmic bytes
    are the rows each call must read (p and q at the first rejection or p_{K+1}: sampling; the
    K+1 target rows: greedy), and inputs rotate over sets whose total exceeds L2.  The
    expert-union cost ([SpecFit] §3.2 eq. (4)) of every subset of an 18-node pool over 48
    layers of 128 experts: an integer OR/popcount kernel, reported in subsets per second."""
    g = torch.Generator(device=device)
    g.manual_seed(synth.seed_for(0, stream=9001))
    sets = 8
    cases = []
    for _ in range(sets):
        zt = torch.randn((B, K + 1, V), generator=g, device=device) * 2.0
        zd = 0.7 * zt[:, :K] + 0.3 * torch.randn((B, K, V), generator=g, device=device) * 2.0
        p = torch.softmax(zt, -1).contiguous()
        q = torch.softmax(zd, -1).contiguous()
        draft = torch.multinomial(q.reshape(B * K, V), 1, generator=g).reshape(B, K).to(torch.int32).contiguous()
        r = torch.rand((B, K), generator=g, device=device)
        u = torch.rand((B,), generator=g, device=device)
        cases.append((draft, q, p, r, u))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    out = {}
    for greedy in (False, True):
        # one call per input set, eagerly (the rows each call reads), then the same calls in a
        # CUDA graph replayed back to back: device time per call without host launch gaps
        outs = [(torch.empty(B, dtype=torch.int32, device=device), torch.empty(B, dtype=torch.int32, device=device))
                for _ in range(sets)]
        nbytes = 0
        for c, (na, tok) in zip(cases, outs):
            api.spec_accept(*c, greedy=greedy, n_accepted=na, token=tok)
        torch.cuda.synchronize(device)
        for na, _ in outs:
            nbytes += B * (K + 1) * V * 4 if greedy else sum((2 if int(a) < K else 1) for a in na.cpu().tolist()) * V * 4
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c, (na, tok) in zip(cases, outs):
                api.spec_accept(*c, greedy=greedy, n_accepted=na, token=tok)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(device)
        ev[0].record()
        for _ in range(reps):
            graph.replay()
        ev[1].record()
        torch.cuda.synchronize(device)
        t = ev[0].elapsed_time(ev[1]) * 1e-3 / (reps * sets)
        per_call = nbytes / sets
        out["greedy" if greedy else "sampling"] = dict(
            us_per_call=round(t * 1e6, 2), gbps=round(per_call / t / 1e9, 1),
            frac_of_hbm=round(per_call / t / 1e9 / measured_peaks()[0]["hbm_gbs"], 4),
            bytes_per_call=int(per_call), mean_accepted=round(float(np.mean([o[0].float().mean().item() for o in outs])), 3))
    # union cost of every subset of the pool
    W = (N + 63) // 64
    rng = np.random.default_rng(synth.seed_for(0, stream=9002))
    bm = np.zeros((nodes + 1, layers, W), np.uint64)
    for v in range(nodes + 1):
        for l in range(layers):
            for e in rng.choice(N, m, replace=False):
                bm[v, l, e // 64] |= np.uint64(1) << np.uint64(e % 64)
    bmt = torch.from_numpy(bm.view(np.int64)).to(device)
    S = 1 << nodes
    subs = torch.arange(S, dtype=torch.int64, device=device).to(torch.int32)
    pv = torch.from_numpy(rng.random(nodes)).to(device)
    bcoef = torch.from_numpy(np.sort(rng.random(nodes + 1))).to(device)
    res = api.union_cost(bmt, subs, pv, bcoef, 0.4)
    ws = torch.empty(int(api.lib().moe_union_cost_workspace_bytes(S)), dtype=torch.uint8, device=device)
    for _ in range(3):
        api.union_cost(bmt, subs, pv, bcoef, 0.4, out=res, ws=ws)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.union_cost(bmt, subs, pv, bcoef, 0.4, out=res, ws=ws)
    graph.replay()
    torch.cuda.synchronize(device)
    ev[0].record()
    for _ in range(reps):
        graph.replay()
    ev[1].record()
    torch.cuda.synchronize(device)
    t = ev[0].elapsed_time(ev[1]) * 1e-3 / reps
    out["union_cost"] = dict(subsets=S, nodes=nodes, layers=layers, experts=N, us_per_call=round(t * 1e6, 2),
                             subsets_per_s=round(S / t, 1), best=int(res["best"].item()),
                             **union_roofline(nodes, layers, W, S, t, torch.cuda.get_device_properties(device).multi_processor_count))
    out["config"] = dict(B=B, K=K, V=V, input_sets=sets, reps=reps, timing="CUDA-graph replays of one call per input set")
    return out


def fit_leg(wl, weights, device, reps: int = 7, windows: int = 8, n_max: int = 16):
    """Fits (4) and (E.1) of one layer's expert-operation time on passes with chosen ids, and
    their error on windows of the layer's synthetic routing trace, the bandwidth error eps
    ([Lan] §2 "Effective bandwidth", §4, App. E "Deduplicating fit").  Every pass follows a
    write of 512 MiB (four times L2), so no pass finds its weights in L2."""
    layer = api.make_layer(wl.d, wl.f, wl.N, wl.m, "bf16")
    ws = api.workspace(layer, 16, device)
    m, N = wl.m, wl.N
    b = 3.0 * wl.d * wl.f * 2
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    x_all = synth.activations(n_max, wl.d, torch.bfloat16, synth.seed_for(wl.index, stream=77), device=device)
    y = torch.empty((n_max, wl.d), dtype=torch.float32, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(n, ids_h):
        ids = torch.from_numpy(np.ascontiguousarray(ids_h)).to(device)
        gates = torch.full((n, m), 1.0 / m, dtype=torch.float32, device=device)
        x = x_all[:n]
        grp = api.Grouping.empty(n, m, N, device)
        ts, td = [], []
        for _ in range(reps):
            flush.fill_(1)
            ev[0].record()
            api.expert_op_perslot(layer, weights, x, ids, gates, y=y[:n], ws=ws)
            ev[1].record()
            torch.cuda.synchronize(device)
            ts.append(ev[0].elapsed_time(ev[1]) * 1e-3)
            flush.fill_(2)
            ev[0].record()
            api.group_slots(ids, N, out=grp, ws=ws)
            api.expert_op_dedup(layer, weights, x, gates, grp, y=y[:n], ws=ws)
            ev[1].record()
            torch.cuda.synchronize(device)
            td.append(ev[0].elapsed_time(ev[1]) * 1e-3)
        return float(np.median(ts)), float(np.median(td))

    ns, Us, tss, tds = [], [], [], []
    for n in range(2, n_max + 1):
        hi = min(N, n * m)
        for U in sorted(set(int(round(u)) for u in np.linspace(m, hi, 5))):
            t_s, t_d = timed(n, synth.chosen_ids(n, m, N, U, seed=synth.seed_for(wl.index, stream=3000 + 131 * n + U)))
            ns.append(n), Us.append(U), tss.append(t_s), tds.append(t_d)
    slot = api.fit_op_times(ns, Us, tss, m, b, "slot")
    dedup = api.fit_op_times(ns, Us, tds, m, b, "dedup")
    # score on windows of the synthetic trace (the stand-in for recorded routing)
    sets, _ = synth.routing_traces(1, windows * n_max, N, m, wl.rhos[0], seed=synth.seed_for(wl.index, stream=4000))
    err_s, err_d = [], []
    for n in range(2, n_max + 1):
        for w in range(windows):
            ids_h = sets[0, w * n:(w + 1) * n]
            U = api.pass_bytes(layer, ids_h)["U"]
            t_s, t_d = timed(n, ids_h)
            err_s.append(abs(slot[0] + slot[1] * U * b + slot[2] * (n * m - U) * b - t_s) / t_s)
            err_d.append(abs(dedup[0] + dedup[1] * U * b + dedup[2] * n - t_d) / t_d)
    eps_s, eps_d = float(np.median(err_s)), float(np.median(err_d))
    return dict(passes=len(ns), n_values=f"2..{n_max}", reps=reps, flush_bytes=512 << 20, b=int(b),
                slot=dict(t_op_us=round(slot[0] * 1e6, 3), c_u_ps_per_byte=round(slot[1] * 1e12, 5),
                          c_re_ps_per_byte=round(slot[2] * 1e12, 5), re_read_cost=round(slot[2] / slot[1], 4),
                          first_read_tbps=round(1e-12 / slot[1], 3)),
                dedup=dict(t_op_us=round(dedup[0] * 1e6, 3), c_g_ps_per_byte=round(dedup[1] * 1e12, 5),
                           c_t_us_per_token=round(dedup[2] * 1e6, 4), union_tbps=round(1e-12 / dedup[1], 3)),
                eps_slot=round(eps_s, 4), eps_dedup=round(eps_d, 4), eps=round(max(eps_s, eps_d), 4),
                scored_windows=len(err_s))


UNION_SMEM_MAX = 200 * 1024       # shared memory the union-cost kernel may use (its table path's limit)
SMEM_BYTES_PER_CLK = 128          # shared memory delivered to the lanes per clock and SM (32 banks x 4 B)
SM_MAX_CLOCK_HZ = 2.07e9          # GB300's maximum SM clock


def union_roofline(nodes, layers, W, S, t, sms):
    """The union-cost kernel's roofline: the bytes its lanes read from shared memory per call (with
    the node-triple table, one 8-byte word per triple and the root per (layer, word) and subset;
    otherwise one per node and the root) over what the SMs' shared memory delivers at the maximum
    clock.  The kernel takes the table path under the same rule as here."""
    lw = layers * W
    ngroups = (nodes + 2) // 3
    table = lw % 2 == 0 and nodes > 0 and lw * 8 + ngroups * 8 * lw * 8 <= UNION_SMEM_MAX
    words = (ngroups + 1 if table else nodes + 1) * lw
    delivered = S * words * 8
    peak = sms * SMEM_BYTES_PER_CLK * SM_MAX_CLOCK_HZ
    achieved = delivered / t
    return dict(bound="shared-memory delivery", path="node-triple table" if table else "broadcast node loop",
                delivered_bytes_per_call=int(delivered), achieved_tbps=round(achieved / 1e12, 2),
                peak_tbps=round(peak / 1e12, 2), frac=round(achieved / peak, 4),
                peak_source="152 SMs x 128 B per clock x 2.07 GHz (derived)" if sms == 152 else
                f"{sms} SMs x 128 B per clock x 2.07 GHz (derived)")


def kernel_traffic(kernel: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, when it was taken on
    the current source of that kernel; None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        data = json.load(fh)
    ent = data.get(kernel)
    if not ent:
        return None
    import hashlib
    h = hashlib.sha256()
    for src in ent["sources"]:
        with open(os.path.join(ROOT, src), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != ent.get("sources_sha256"):
        return None
    return ent


# --------------------------------------------------------------------- our arm

class StackBench:
    def __init__(self, wl, layers, n_values, windows, device, use_graph=True, rho_index=0, weights=None):
        self.wl, self.L, self.n_values, self.windows, self.dev = wl, layers, n_values, windows, device
        self.layer = api.make_layer(wl.d, wl.f, wl.N, wl.m, "bf16")
        self.use_graph = use_graph
        self.rho = wl.rhos[rho_index]
        t0 = time.time()
        self.weights = weights if weights is not None else [
            synth.expert_weights(wl.N, wl.f, wl.d, torch.bfloat16, synth.seed_for(wl.index, layer=l), device=device)
            for l in range(layers)]
        torch.cuda.synchronize(device)
        self.t_weights = time.time() - t0
        T = windows * max(n_values)
        self.sets, logits = synth.routing_traces(layers, T, wl.N, wl.m, self.rho,
                                                 seed=synth.seed_for(wl.index, rho_index=rho_index, stream=2))
        self.ws = api.workspace(self.layer, max(16, max(n_values)), device)
        self.per_n = {}
        for n in n_values:
            lw = np.stack([logits[:, w * n:(w + 1) * n, :].reshape(layers * n, wl.N) for w in range(windows)])
            xw = torch.stack([synth.activations(n, wl.d, torch.bfloat16,
                                                synth.seed_for(wl.index, stream=1000 + 17 * n + w), device=device)
                              for w in range(windows)])
            st = dict(
                logits_all=torch.from_numpy(np.ascontiguousarray(lw)).to(device),
                x_all=xw.contiguous(),
                logits=torch.empty((layers * n, wl.N), dtype=torch.float32, device=device),
                x=torch.empty((n, wl.d), dtype=torch.bfloat16, device=device),
                ids=torch.empty((layers * n, wl.m), dtype=torch.int32, device=device),
                gates=torch.empty((layers * n, wl.m), dtype=torch.float32, device=device),
                y_slot=torch.zeros((layers, n, wl.d), dtype=torch.float32, device=device),
                y_dedup=torch.zeros((layers, n, wl.d), dtype=torch.float32, device=device),
                groups=[api.Grouping.empty(n, wl.m, wl.N, device) for _ in range(layers)],
            )
            bytes_slot, bytes_dedup = [], []
            for w in range(windows):
                bs = bd = 0
                for l in range(layers):
                    pb = api.pass_bytes(self.layer, self.sets[l, w * n:(w + 1) * n])
                    bs += pb["slot_bytes"]
                    bd += pb["dedup_bytes"]
                bytes_slot.append(bs)
                bytes_dedup.append(bd)
            st["bytes_slot"], st["bytes_dedup"] = bytes_slot, bytes_dedup
            self.per_n[n] = st
        self.graphs = {}
        # per pass size: one route and one kernel per expert op in each form
        self.launches_per_step = sum(1 + 2 * layers for _ in n_values)

    # the four phases of one pass size
    def _route(self, st):
        api.route_topm(st["logits"], self.wl.m, ids=st["ids"], gates=st["gates"])

    def _slot(self, st, n):
        for l in range(self.L):
            api.expert_op_perslot(self.layer, self.weights[l], st["x"], st["ids"][l * n:(l + 1) * n],
                                  st["gates"][l * n:(l + 1) * n], y=st["y_slot"][l], accumulate=True, ws=self.ws)

    def _group(self, st, n):
        for l in range(self.L):
            api.group_slots(st["ids"][l * n:(l + 1) * n], self.wl.N, out=st["groups"][l], ws=self.ws)

    def _dedup(self, st, n):
        # the deduplicating form in one launch per layer: the kernel builds the pass's grouping
        for l in range(self.L):
            api.expert_op_dedup_ids(self.layer, self.weights[l], st["x"], st["ids"][l * n:(l + 1) * n],
                                    st["gates"][l * n:(l + 1) * n], y=st["y_dedup"][l], accumulate=True, ws=self.ws)

    def capture(self):
        phases = ("route", "slot", "group", "dedup")
        for n in self.n_values:
            st = self.per_n[n]
            self.stage(n, 0)
            fns = {"route": lambda st=st: self._route(st), "slot": lambda st=st, n=n: self._slot(st, n),
                   "group": lambda st=st, n=n: self._group(st, n), "dedup": lambda st=st, n=n: self._dedup(st, n)}
            for ph in phases:      # eager run first: lazy initialisation outside capture
                fns[ph]()
            torch.cuda.synchronize(self.dev)
            if self.use_graph:
                for ph in phases:
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        fns[ph]()
                    self.graphs[(n, ph)] = g
            else:
                for ph in phases:
                    self.graphs[(n, ph)] = fns[ph]
        torch.cuda.synchronize(self.dev)
        assert api.last_device_error(self.ws) == 0

    def _run(self, n, ph):
        g = self.graphs[(n, ph)]
        g.replay() if self.use_graph else g()

    def stage(self, n, w):
        st = self.per_n[n]
        st["logits"].copy_(st["logits_all"][w], non_blocking=True)
        st["x"].copy_(st["x_all"][w], non_blocking=True)
        st["y_slot"].zero_()
        st["y_dedup"].zero_()

    # the timed phases of a pass size; "group" (the standalone counting sort) runs only for the
    # checks: the deduplicating launch groups the slots itself
    TIMED = ("route", "slot", "dedup")

    def step(self, w, events=None):
        for n in self.n_values:
            self.stage(n, w)
            if events is not None:
                events[(n, "start")].record()
            for ph in self.TIMED:
                self._run(n, ph)
                if events is not None:
                    events[(n, ph)].record()

    def check_outputs(self):
        """Cheap self-check after timing: ids equal the trace sets, forms agree."""
        worst = 0.0
        for n in self.n_values:
            st = self.per_n[n]
            ys, yd = st["y_slot"].double(), st["y_dedup"].double()
            rms = ys.pow(2).mean().sqrt().clamp_min(1e-30)
            worst = max(worst, float((ys - yd).abs().max() / rms))
        return worst


def run_ours(args, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    mbuild.build()
    api.lib()
    wl = BY_NAME[args.workload]
    if wl.layers < 2 and args.layers is None:
        raise SystemExit("bench.py times the multi-layer stack; single layers are parity-test cases")
    layers = args.layers or wl.layers
    n_max = args.n_max or max(wl.n_values)
    n_values = [n for n in wl.n_values if (args.n_min or 1) <= n <= n_max]
    windows = args.warmup + args.steps
    b = StackBench(wl, layers, n_values, windows, device, use_graph=not args.no_graph)
    b.capture()

    for w in range(args.warmup):
        b.step(w)
    torch.cuda.synchronize(device)

    phases = b.TIMED
    events = [{(n, k): torch.cuda.Event(enable_timing=True) for n in n_values for k in ("start",) + phases}
              for _ in range(args.steps)]
    acc = {(n, ph): 0.0 for n in n_values for ph in phases}
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clk:
        t_start.record()
        for k in range(args.steps):
            b.step(args.warmup + k, events[k])
        t_end.record()
        torch.cuda.synchronize(device)
    barrier(world)
    for k in range(args.steps):
        for n in n_values:
            prev = events[k][(n, "start")]
            for ph in phases:
                acc[(n, ph)] += prev.elapsed_time(events[k][(n, ph)]) * 1e-3
                prev = events[k][(n, ph)]
    total_s = t_start.elapsed_time(t_end) * 1e-3
    total_s = reduce_max(total_s, world, device)
    self_check = b.check_outputs()
    err = api.last_device_error(b.ws)

    # bytes requested in the timed steps
    steps_w = range(args.warmup, args.warmup + args.steps)
    bytes_slot = {n: sum(b.per_n[n]["bytes_slot"][w] for w in steps_w) for n in n_values}
    bytes_dedup = {n: sum(b.per_n[n]["bytes_dedup"][w] for w in steps_w) for n in n_values}
    total_bytes = sum(bytes_slot.values()) + sum(bytes_dedup.values())
    value = world * total_bytes / total_s / 1e12
    t_slot = [acc[(n, "slot")] for n in n_values]
    t_dedup = [acc[(n, "dedup")] for n in n_values]
    rep = api.bandwidth_report(n_values[0], [bytes_slot[n] for n in n_values],
                               [bytes_dedup[n] for n in n_values], t_slot, t_dedup)
    K = args.steps
    per_n = []
    for i, n in enumerate(n_values):
        per_n.append(dict(
            n=n,
            us_slot=round(t_slot[i] / K * 1e6, 2), us_dedup=round(t_dedup[i] / K * 1e6, 2),
            us_route=round(acc[(n, "route")] / K * 1e6, 2),
            tbps_slot=round(rep["beta_slot"][i] / 1e12, 3), tbps_dedup=round(rep["beta_dedup"][i] / 1e12, 3),
            tbps_dedup_kernel=round(bytes_dedup[n] / acc[(n, "dedup")] / 1e12, 3),
            ubar=round(float(rep["ubar"][i]), 4), r=round(float(rep["r"][i]), 4),
            saving_us=round(float(rep["saving"][i]) / K * 1e6, 2)))
    # best draft length: V(k) = expert time of a pass of k+1 tokens (all layers)
    kstar = {}
    # the draft-length report needs the one-token pass and at least one longer one
    if n_values[0] == 1 and len(n_values) > 1:
        Vs = [t / K for t in t_slot]
        Vd = [t_slot[0] / K] + [t / K for t in t_dedup[1:]]
        cross = rep["crossover"]
        Vw = [Vs[i] if (cross is None or n_values[i] < cross) else Vd[i] for i in range(len(n_values))]
        for a in A_GRID:
            kstar[str(a)] = dict(slot=api.best_draft_length(Vs, a), dedup=api.best_draft_length(Vd, a),
                                 switched=api.best_draft_length(Vw, a))
        theory = step_time_theory(n_values, Vs, Vd, Vw, bytes_slot, bytes_dedup, K)
    else:
        theory = None

    # roofline of the expert op (both forms; one launch = one layer's expert op, one
    # persistent kernel streaming its gate/up and then its down weights)
    expert_s = sum(acc[(n, "slot")] + acc[(n, "dedup")] for n in n_values)
    launches = 2 * layers * len(n_values) * K
    peaks, peak_kind = measured_peaks()
    achieved = total_bytes / expert_s / 1e9
    traffic = kernel_traffic(EXPERT_OP)
    roofline = dict(kernel=EXPERT_OP, bound="hbm", achieved=round(achieved, 1),
                    peak=peaks["hbm_gbs"], unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4),
                    peak_source=f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                    bytes_per_launch=round(total_bytes / launches), mean_launch_us=round(expert_s / launches * 1e6, 2),
                    traffic=(traffic or {}).get("dram_bytes_per_launch"),
                    traffic_note=(traffic or {}).get("note"))

    line = dict(metric=METRIC, value=round(value, 4), unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
                ms_per_step=round(total_s / K * 1e3, 3), higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="bf16", data="synthetic",
                config=dict(workload=wl.name, layers=layers, d=wl.d, f=wl.f, N=wl.N, m=wl.m,
                            n_values=f"{n_values[0]}..{n_values[-1]}", rho=wl.rhos[0], parallelism="replicas",
                            windows_per_step=1, graphs=not args.no_graph,
                            l2="inputs larger than L2: 57.98 GB of weights streamed layer after layer"
                            if layers == 48 else f"{layers} layers, no flush"),
                roofline=roofline, gpu_launches=b.launches_per_step * K,
                clocks=clk.summary(), per_n=per_n, crossover=rep["crossover"], kstar=kstar, theory=theory,
                self_check=dict(max_slot_vs_dedup_rel=round(self_check, 6), device_error=err),
                setup_s=dict(weights=round(b.t_weights, 1)))

    if not args.no_e2e:
        line["e2e"] = e2e_run(b, args, world, device, total_bytes_per_step=total_bytes / K)
    if not args.no_fp8:
        line["fp8"] = fp8_leg(b, args, device, per_n)
    if rank == 0 and not args.no_fit:
        line["fits"] = fit_leg(wl, b.weights[0], device, reps=args.fit_reps)
    if rank == 0 and not args.no_configs:
        line["configs"] = configs_leg(device)
    if rank == 0 and not args.no_long:
        line["long_pass"] = long_pass_leg(wl, b.weights[:8], device)
    if rank == 0:
        line["hbm_read_probe"] = read_probe_leg(device)
    if rank == 0 and not args.no_verify_side:
        line["verify_side"] = verify_side_leg(device, reps=args.verify_reps)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(b)
    if rank == 0:
        print(json.dumps(line), flush=True)


# layers of each page-shaped workload in the configs leg: enough that the stack's weights
# exceed L2 (8.9 GB, 9.7 GB and 11.3 GB), so passes run layer after layer without a flush
CONFIG_LAYERS = {DSV2_LITE.name: 8, QWEN3.name: 8, MIXTRAL.name: 4}


def _time_stack(b: StackBench, warmup: int, steps: int, extra=None):
    """Warm-up and timed steps of a captured stack; per-n seconds of each timed phase (and of
    `extra(n)`, a callable that runs one more captured phase after the dedup phase)."""
    for w in range(warmup):
        b.step(w)
        if extra is not None:
            for n in b.n_values:
                extra(n)
    torch.cuda.synchronize(b.dev)
    phases = b.TIMED + (("extra",) if extra is not None else ())
    acc = {(n, ph): 0.0 for n in b.n_values for ph in phases}
    for k in range(steps):
        w = warmup + k
        for n in b.n_values:
            ev = {ph: torch.cuda.Event(enable_timing=True) for ph in ("start",) + phases}
            b.stage(n, w)
            ev["start"].record()
            prev = "start"
            for ph in b.TIMED:
                b._run(n, ph)
                ev[ph].record()
            if extra is not None:
                extra(n)
                ev["extra"].record()
            torch.cuda.synchronize(b.dev)
            for ph in phases:
                acc[(n, ph)] += ev[prev].elapsed_time(ev[ph]) * 1e-3
                prev = ph
    return acc


def configs_leg(device, warmup: int = 2, steps: int = 3, names=None):
    """The page-shaped single-layer workloads at every reuse value ([Lan] Table 1, §2: per-model
    effective bandwidths, u_bar(n), r(n) and the crossover): each as a stack of CONFIG_LAYERS
    layers run layer after layer, like the headline workload.  Per n: microseconds per layer
    pass of each form, TB/s on requested bytes, u_bar, r, and the crossover n*.  The
    DeepSeek-V2-Lite block also times its two always-on shared experts (one deduplicating
    launch per layer on their own weights, ids [0, 1] for every token, gates 1, accumulated),
    which the pages count outside the expert operation's bytes."""
    out = {}
    for wl in (DSV2_LITE, QWEN3, MIXTRAL):
        if names is not None and wl.name not in names:
            continue
        L = CONFIG_LAYERS[wl.name]
        weights = [synth.expert_weights(wl.N, wl.f, wl.d, torch.bfloat16, synth.seed_for(wl.index, layer=l),
                                        device=device) for l in range(L)]
        shared = None
        if wl.n_shared:
            sh_layer = api.make_layer(wl.d, wl.f_shared, wl.n_shared, wl.n_shared, "bf16")
            shared = dict(layer=sh_layer, ws=api.workspace(sh_layer, 16, device),
                          w=[synth.expert_weights(wl.n_shared, wl.f_shared, wl.d, torch.bfloat16,
                                                  synth.seed_for(wl.index, layer=l, stream=9), device=device)
                             for l in range(L)])
        block = dict(layers=L, d=wl.d, f=wl.f, N=wl.N, m=wl.m, n_values=f"{wl.n_values[0]}..{wl.n_values[-1]}",
                     timing="CUDA-graph phases of L expert launches, events between phases; weights > L2",
                     per_rho={})
        for ri, rho in enumerate(wl.rhos):
            b = StackBench(wl, L, list(wl.n_values), warmup + steps, device, rho_index=ri, weights=weights)
            b.capture()
            extra = None
            if shared is not None:
                graphs = {}
                # every tensor a captured graph reads or writes must outlive the graph: the per-n
                # grouping, gates and output stay referenced here until the block is done
                keep = []
                for n in b.n_values:
                    st = b.per_n[n]
                    y_sh = torch.zeros((L, n, wl.d), dtype=torch.float32, device=device)
                    sids = torch.tensor([[0, 1]] * n, dtype=torch.int32, device=device)
                    sg = api.group_slots(sids, wl.n_shared)
                    sgates = torch.ones((n, wl.n_shared), device=device)

                    def run_shared(st=st, sg=sg, sgates=sgates, y_sh=y_sh):
                        for l in range(L):
                            api.expert_op_dedup(shared["layer"], shared["w"][l], st["x"], sgates, sg,
                                                y=y_sh[l], accumulate=True, ws=shared["ws"])
                    keep.append((sids, sg, sgates, y_sh))
                    run_shared()
                    torch.cuda.synchronize(device)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        run_shared()
                    graphs[n] = g
                extra = lambda n: graphs[n].replay()
            acc = _time_stack(b, warmup, steps, extra)
            steps_w = range(warmup, warmup + steps)
            nv = b.n_values
            bs = [sum(b.per_n[n]["bytes_slot"][w] for w in steps_w) for n in nv]
            bd = [sum(b.per_n[n]["bytes_dedup"][w] for w in steps_w) for n in nv]
            ts = [acc[(n, "slot")] for n in nv]
            td = [acc[(n, "dedup")] for n in nv]
            rep = api.bandwidth_report(nv[0], bs, bd, ts, td)
            per_n = []
            for i, n in enumerate(nv):
                row = dict(n=n, us_slot=round(ts[i] / (steps * L) * 1e6, 2), us_dedup=round(td[i] / (steps * L) * 1e6, 2),
                           tbps_slot=round(rep["beta_slot"][i] / 1e12, 3), tbps_dedup=round(rep["beta_dedup"][i] / 1e12, 3),
                           ubar=round(float(rep["ubar"][i]), 4), r=round(float(rep["r"][i]), 4))
                if shared is not None:
                    t_sh = acc[(n, "extra")] / (steps * L)
                    row["us_shared"] = round(t_sh * 1e6, 2)
                    row["tbps_shared"] = round(wl.n_shared * 3 * wl.d * wl.f_shared * 2 / t_sh / 1e12, 3)
                per_n.append(row)
            assert api.last_device_error(b.ws) == 0
            block["per_rho"][str(rho)] = dict(per_n=per_n, crossover=rep["crossover"],
                                             max_slot_vs_dedup_rel=round(b.check_outputs(), 6))
            torch.cuda.synchronize(device)
            if shared is not None:
                assert api.last_device_error(shared["ws"]) == 0
                del graphs, keep, extra
            del b
            torch.cuda.empty_cache()
        out[wl.name] = block
        del weights, shared
        torch.cuda.empty_cache()
    return out


LONG_PASS_N = (17, 24, 32, 40, 48, 64)


def long_pass_leg(wl, weights, device, warmup: int = 2, steps: int = 3):
    """Passes of 17 to 64 tokens on the headline layer shape ([Lan] §1: the deduplicating form
    reads each distinct expert once per pass; §2: effective bandwidth on requested bytes).  A
    stack of len(weights) layers run layer after layer (weights > L2), the per-slot calls as
    launches of up to 16 tokens, the deduplicating call in one launch of the 64-token
    instantiation (above 256 slots after its in-workspace grouping launch).  Per n:
    microseconds per layer pass of each form, TB/s on requested bytes, u_bar and r."""
    L = len(weights)
    b = StackBench(wl, L, list(LONG_PASS_N), warmup + steps, device, weights=weights)
    b.capture()
    acc = _time_stack(b, warmup, steps)
    steps_w = range(warmup, warmup + steps)
    nv = b.n_values
    bs = [sum(b.per_n[n]["bytes_slot"][w] for w in steps_w) for n in nv]
    bd = [sum(b.per_n[n]["bytes_dedup"][w] for w in steps_w) for n in nv]
    ts = [acc[(n, "slot")] for n in nv]
    td = [acc[(n, "dedup")] for n in nv]
    rep = api.bandwidth_report(nv[0], bs, bd, ts, td)
    per_n = [dict(n=n, us_slot=round(ts[i] / (steps * L) * 1e6, 2), us_dedup=round(td[i] / (steps * L) * 1e6, 2),
                  tbps_slot=round(rep["beta_slot"][i] / 1e12, 3), tbps_dedup=round(rep["beta_dedup"][i] / 1e12, 3),
                  ubar=round(float(rep["ubar"][i]), 4), r=round(float(rep["r"][i]), 4))
             for i, n in enumerate(nv)]
    out = dict(layers=L, d=wl.d, f=wl.f, N=wl.N, m=wl.m, rho=b.rho, per_n=per_n,
               max_slot_vs_dedup_rel=round(b.check_outputs(), 6), device_error=api.last_device_error(b.ws),
               timing="CUDA-graph phases of L expert launches, events between phases; weights > L2")
    del b
    torch.cuda.empty_cache()
    return out


def profile_layer(wl, cases):
    """A small case for Nsight Compute: one layer of the workload's shape (1.2 GB of bf16 weights for
    the Qwen3 shape, larger than L2), the reuse-0.4 routing of a pass of each size n, and two calls
    per case on a workspace for the largest n: "n" the deduplicating call from ids, "sn" the
    per-slot call (n <= 16: one launch)."""
    mbuild.build()
    device = torch.device("cuda", 0)
    layer = api.make_layer(wl.d, wl.f, wl.N, wl.m, "bf16")
    w = synth.expert_weights(wl.N, wl.f, wl.d, torch.bfloat16, 11, device=device)
    parsed = [(c.startswith("s"), int(c.lstrip("s"))) for c in cases]
    n_max = max(n for _, n in parsed)
    ws = api.workspace(layer, n_max, device)
    x_all = synth.activations(n_max, wl.d, torch.bfloat16, 2, device=device)
    for perslot, n in parsed:
        _, logits = synth.routing_traces(1, n, wl.N, wl.m, 0.4, seed=3)
        ids, gates = api.route_topm(torch.from_numpy(logits[0]).to(device), wl.m)
        x = x_all[:n].contiguous()
        for _ in range(2):
            if perslot:
                api.expert_op_perslot(layer, w, x, ids, gates, ws=ws)
            else:
                api.expert_op_dedup_ids(layer, w, x, ids, gates, ws=ws)
        torch.cuda.synchronize(device)
    assert api.last_device_error(ws) == 0
    print("ok", flush=True)


def e2e_run(b: StackBench, args, world, device, total_bytes_per_step):
    """The same steps with inputs copied from pinned host memory and outputs copied back."""
    host = {}
    h2d = d2h = 0
    for n in b.n_values:
        st = b.per_n[n]
        host[n] = dict(logits=st["logits_all"].cpu().pin_memory(), x=st["x_all"].cpu().pin_memory(),
                       y_slot=torch.empty(st["y_slot"].shape, dtype=torch.float32).pin_memory(),
                       y_dedup=torch.empty(st["y_dedup"].shape, dtype=torch.float32).pin_memory())
        h2d += st["logits"].numel() * 4 + st["x"].numel() * 2
        d2h += 2 * st["y_slot"].numel() * 4

    def step(w):
        for n in b.n_values:
            st, hs = b.per_n[n], host[n]
            st["logits"].copy_(hs["logits"][w], non_blocking=True)
            st["x"].copy_(hs["x"][w], non_blocking=True)
            st["y_slot"].zero_()
            st["y_dedup"].zero_()
            for ph in b.TIMED:
                b._run(n, ph)
            hs["y_slot"].copy_(st["y_slot"], non_blocking=True)
            hs["y_dedup"].copy_(st["y_dedup"], non_blocking=True)

    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize(device)
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for k in range(args.steps):
        step(args.warmup + k)
    e.record()
    torch.cuda.synchronize(device)
    t = reduce_max(s.elapsed_time(e) * 1e-3, world, device)
    return dict(value=round(world * total_bytes_per_step * args.steps / t / 1e12, 4), unit=UNIT,
                h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h, ms_per_step=round(t / args.steps * 1e3, 3))


# --------------------------------------------------------------------- oracle timing

def _oracle_sample(oracle_mod, wl, host_w, sets_l, x_host, n_list, budget_s, min_s=0.0):
    """Time the oracle (both forms) on passes of layer 0; returns (bytes, seconds, passes).  The
    pass sizes are taken in order, again and again on later windows of the trace, until at
    least min_s seconds were timed, and no new one starts after budget_s."""
    w_bytes = wl.expert_bytes
    done_bytes, done_s, passes = 0, 0.0, []
    order = list(n_list)
    k = 0
    while k < len(order):
        n = order[k]
        k += 1
        if k == len(order) and done_s < min_s:
            order += list(n_list)
        off = (len(passes) // max(1, len(n_list))) * max(n_list)
        ids_set = sets_l[off:off + n] if off + n <= len(sets_l) else sets_l[:n]
        # the oracle routes from logits whose top-m is the set; use its grouping and bytes
        z = np.full((n, wl.N), -10.0, np.float32)
        for t in range(n):
            z[t, ids_set[t]] = np.linspace(1.0, 0.5, wl.m, dtype=np.float32)
        xh = x_host[:n]
        t0 = time.perf_counter()
        ids, gates = oracle_mod.route_topm(z, wl.m)
        oracle_mod.expert_op_perslot(*host_w, xh, ids, gates)
        grp = oracle_mod.group_slots(ids, wl.N)
        oracle_mod.expert_op_dedup(*host_w, xh, gates, wl.m, grp)
        done_s += time.perf_counter() - t0
        done_bytes += n * wl.m * w_bytes + grp[0] * w_bytes
        passes.append(n)
        if done_s > budget_s:
            break
    return done_bytes, done_s, passes


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(b: StackBench):
    """The oracle on layer 0 of the stack, both forms, at n in {1, 4, 8, 16}: on every host core
    (OpenMP over output rows) and single-threaded (results are bit-identical either way)."""
    import oracle
    oracle.build()
    wl = b.wl
    host_w = tuple(synth.host_array(t) for t in b.weights[0])
    x_host = synth.host_array(b.per_n[max(b.n_values)]["x_all"][0])
    n_list = [n for n in (1, 4, 8, 16) if n in b.n_values]
    cores = host_cores()
    used = oracle.set_threads(cores)
    nb, s, passes = _oracle_sample(oracle, wl, host_w, b.sets[0], x_host, n_list, budget_s=10.0, min_s=5.0)
    oracle.set_threads(1)
    nb1, s1, passes1 = _oracle_sample(oracle, wl, host_w, b.sets[0], x_host, n_list, budget_s=10.0, min_s=5.0)
    return dict(value=round(nb / s / 1e12, 8), unit=UNIT, cores=used, kind="oracle",
                sample=f"layer 0 of the stack, {len(passes)} passes cycling n over {n_list}, per-slot and dedup forms "
                       f"(routing, grouping, both expert ops, combine), fp64 C oracle with OpenMP over output rows on "
                       f"{used} threads; {nb / 1e9:.2f} GB requested in {s:.1f} s",
                single_thread=dict(value=round(nb1 / s1 / 1e12, 8), unit=UNIT, cores=1,
                                   sample=f"{len(passes1)} passes cycling n over {n_list} on one thread; "
                                          f"{nb1 / 1e9:.2f} GB requested in {s1:.1f} s"))


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is one pass of one layer (both forms)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.set_threads(host_cores())
    wl = BY_NAME[args.workload]
    n_max = args.n_max or max(wl.n_values)
    dt = torch.bfloat16 if wl.w_dtype == "bf16" else torch.float32
    wg, wu, wd = synth.expert_weights(wl.N, wl.f, wl.d, dt, synth.seed_for(wl.index, layer=0))
    host_w = tuple(synth.host_array(t) for t in (wg, wu, wd))
    T = (args.warmup + args.steps) * n_max
    sets, _ = synth.routing_traces(1, T, wl.N, wl.m, wl.rhos[0], seed=synth.seed_for(wl.index, stream=2))
    x_host = synth.host_array(synth.activations(n_max, wl.d, dt, seed=synth.seed_for(wl.index, stream=1)))
    n_step = [min(wl.n_values) + (k * 5) % (n_max - min(wl.n_values) + 1)
              for k in range(args.warmup + args.steps)]   # cycle over pass sizes
    for k in range(args.warmup):
        _oracle_sample(oracle, wl, host_w, sets[0][k * n_max:], x_host, [n_step[k]], budget_s=1e9)
    nb_tot, s_tot = 0, 0.0
    for k in range(args.warmup, args.warmup + args.steps):
        nb, s, _ = _oracle_sample(oracle, wl, host_w, sets[0][k * n_max:], x_host, [n_step[k]], budget_s=1e9)
        nb_tot += nb
        s_tot += s
    value = nb_tot / s_tot / 1e12
    sample = (f"one layer of {wl.name}, one pass per step at n in {n_step[args.warmup:]}, "
              f"per-slot and dedup forms, fp64 C oracle with OpenMP over output rows on {cores} threads")
    line = dict(metric=METRIC, value=round(value, 10), unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(s_tot / args.steps * 1e3, 1), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=wl.name, layers=1, d=wl.d, f=wl.f, N=wl.N, m=wl.m, rho=wl.rhos[0]),
                cpu_baseline=dict(value=round(value, 10), unit=UNIT, cores=cores, kind="oracle", sample=sample),
                e2e=dict(value=round(value, 10), unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        # the oracle needs no collective: rank 0 runs it, other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, world, int(os.environ.get("RANK", "0")))
        return
    if args.configs_only:
        mbuild.build()
        device = torch.device("cuda", 0)
        print(json.dumps(dict(configs=configs_leg(device, names=args.configs_only.split(",")))), flush=True)
        return
    if args.profile_layer:
        profile_layer(BY_NAME[args.workload], args.profile_layer.split(","))
        return
    if args.long_only:
        mbuild.build()
        wl = BY_NAME[args.workload]
        device = torch.device("cuda", 0)
        w = [synth.expert_weights(wl.N, wl.f, wl.d, torch.bfloat16, synth.seed_for(wl.index, layer=l), device=device)
             for l in range(8)]
        print(json.dumps(dict(workload=wl.name, long_pass=long_pass_leg(wl, w, device))), flush=True)
        return
    if args.fit_only:
        mbuild.build()
        wl = BY_NAME[args.workload]
        device = torch.device("cuda", 0)
        w = synth.expert_weights(wl.N, wl.f, wl.d, torch.bfloat16, synth.seed_for(wl.index, layer=0), device=device)
        print(json.dumps(dict(workload=wl.name, fits=fit_leg(wl, w, device, reps=args.fit_reps))), flush=True)
        return
    if args.verify_side_only:
        mbuild.build()
        print(json.dumps(dict(verify_side=verify_side_leg(torch.device("cuda", 0), reps=args.verify_reps))), flush=True)
        return
    world, rank, local = dist_setup(args)
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
