"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module draws random numbers with the shapes and laws of the workloads and holds
none of the method's arithmetic: no routing, grouping, SwiGLU, combine or byte count.

Laws (the input recipe):
  * expert weights  W_gate, W_up ~ N(0, 1/d) as [N, f, d];  W_down ~ N(0, 1/f) as [N, d, f];
    drawn in fp32 and rounded to bf16 (round to nearest even) for bf16 layers.
  * activations     x ~ N(0, 1) as [n, d].
  * routing traces  a stationary process on m-subsets of N experts with reuse rho: the
    first token's set is a uniform m-subset; each later token keeps each expert of the
    previous token's set independently with probability rho and fills the rest with a
    uniform draw without replacement from the experts it did not keep.  rho = 0 is
    independent uniform routing.
  * chosen ids      a pass of n tokens whose n*m slots name exactly U distinct experts
    (m <= U <= min(N, n*m)): a uniform U-subset of the experts in random order, token t
    taking the m consecutive entries starting at position t*m (cyclically), so that every
    token's m experts are distinct and together they cover all U; then each token's order
    is shuffled.
  * router logits   z ~ N(0, 1) per token, then every expert outside the token's set is
    shifted down by one common amount per token, so that the set is exactly the top-m
    of the logits with a margin of at least 0.25; the logits of the selected experts
    are untouched.
"""
from __future__ import annotations

import numpy as np
import torch


def seed_for(config_index: int, layer: int = 0, rho_index: int = 0, stream: int = 0,
             base: int = 0) -> int:
    """Seed of one random stream: base + (config, layer, rho index, stream id)."""
    return int(base + config_index * 1_000_003 + layer * 10_007 + rho_index * 101 + stream)


def routing_traces(L: int, T: int, N: int, m: int, rho: float, seed: int):
    """L independent traces of T tokens.  Returns (sets int32 [L, T, m], logits fp32 [L, T, N]).

    sets[l, t] is the expert set of token t in trace l (unordered); logits[l, t] are
    router logits whose top-m is exactly that set."""
    if not (1 <= m <= N):
        raise ValueError("need 1 <= m <= N")
    rng = np.random.Generator(np.random.PCG64(seed))
    sets = np.empty((L, T, m), np.int32)
    # first token: uniform m-subset
    prev = np.argsort(rng.random((L, N)), axis=1)[:, :m].astype(np.int32)
    sets[:, 0] = prev
    for t in range(1, T):
        keep = rng.random((L, m)) < rho                        # [L, m]
        keys = rng.random((L, N))
        kept_ids = np.where(keep, prev, -1)
        # exclude kept experts from the fill draw
        mask = np.zeros((L, N), bool)
        for j in range(m):
            sel = kept_ids[:, j] >= 0
            mask[np.nonzero(sel)[0], kept_ids[sel, j]] = True
        keys[mask] = 2.0
        fill = np.argsort(keys, axis=1)[:, :m].astype(np.int32)  # uniform order of the rest
        n_keep = keep.sum(axis=1)
        cur = np.empty((L, m), np.int32)
        for l in range(L):
            k = int(n_keep[l])
            cur[l, :k] = prev[l, keep[l]]
            cur[l, k:] = fill[l, :m - k]
        sets[:, t] = cur
        prev = cur
    z = rng.standard_normal((L, T, N))
    member = np.zeros((L, T, N), bool)
    np.put_along_axis(member, sets.astype(np.int64), True, axis=2)
    sel_min = np.where(member, z, np.inf).min(axis=2)
    rest_max = np.where(member, -np.inf, z).max(axis=2)
    shift = np.maximum(0.0, rest_max - sel_min) + 0.25
    shift = np.where(np.isfinite(shift), shift, 0.0)
    logits = np.where(member, z, z - shift[..., None]).astype(np.float32)
    return sets, logits


def chosen_ids(n: int, m: int, N: int, U: int, seed: int) -> np.ndarray:
    """ids [n, m] int32 of a pass whose slots name exactly U distinct experts."""
    if not (m <= U <= min(N, n * m)):
        raise ValueError(f"U={U} outside [m, min(N, n*m)] = [{m}, {min(N, n * m)}]")
    rng = np.random.default_rng(seed)
    E = rng.permutation(N)[:U]
    ids = np.empty((n, m), dtype=np.int32)
    for t in range(n):
        ids[t] = E[(t * m + np.arange(m)) % U]
        rng.shuffle(ids[t])
    return ids


def expert_weights(N: int, f: int, d: int, dtype: torch.dtype, seed: int,
                   device: str | torch.device = "cpu", chunk: int = 16):
    """(w_gate [N,f,d], w_up [N,f,d], w_down [N,d,f]) with the recipe's laws."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    out = []
    for shape, fan_in in (((N, f, d), d), ((N, f, d), d), ((N, d, f), f)):
        w = torch.empty(shape, dtype=dtype, device=dev)
        for e0 in range(0, N, chunk):
            e1 = min(N, e0 + chunk)
            blk = torch.randn((e1 - e0,) + shape[1:], generator=g, device=dev, dtype=torch.float32)
            blk.mul_(fan_in ** -0.5)
            w[e0:e1].copy_(blk)
        out.append(w)
    return tuple(out)


def activations(n: int, d: int, dtype: torch.dtype, seed: int, device="cpu"):
    """x ~ N(0, 1) as [n, d] in dtype."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return torch.randn((n, d), generator=g, device=dev, dtype=torch.float32).to(dtype)


def tiny_router(N: int, d: int, seed: int):
    """Router weight W_r [N, d] ~ N(0, 1/d), fp32 on the CPU."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn((N, d), generator=g, dtype=torch.float32) * d ** -0.5


def tiny_logits(x: torch.Tensor, w_r: torch.Tensor) -> torch.Tensor:
    """Router logits x W_r^T of the tiny layer, fp32 on the CPU, fed to both sides."""
    return (x.float() @ w_r.t()).contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as its raw 16-bit patterns (numpy uint16)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_array(t: torch.Tensor) -> np.ndarray:
    """Host copy of a weight/activation tensor in the form the oracle reads."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype == torch.float32:
        return t.detach().contiguous().cpu().numpy()
    raise TypeError(t.dtype)
