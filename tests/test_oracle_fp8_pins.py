"""Pins of the oracle's FP8 (e4m3) functions (CPU only): every code against PyTorch's
float8_e4m3fn, the rounding against a brute-force nearest search and PyTorch's conversion,
and the quantized expert operation against the fp64 SwiGLU of its dequantized inputs within
the rounding bound of the quantized h."""
import numpy as np
import pytest
import torch


def test_e4m3_decode_matches_torch(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle_mod.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert oracle_mod.e4m3_decode(0x7E) == 448.0 and oracle_mod.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_rounds_to_nearest_even(oracle_mod):
    rng = np.random.default_rng(120)
    vals = np.concatenate([rng.uniform(-448, 448, 3000), rng.normal(0, 1e-2, 2000), rng.normal(0, 1, 2000)])
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(v) for v in vals.astype(np.float32)], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # exact midpoints between neighbouring codes go to the even mantissa
    for c in range(0, 126):
        lo, hi = oracle_mod.e4m3_decode(c), oracle_mod.e4m3_decode(c + 1)
        mid = 0.5 * (lo + hi)
        assert oracle_mod.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1)
    # saturation to the largest finite value
    assert oracle_mod.e4m3_encode(500.0) == 0x7E and oracle_mod.e4m3_encode(-1e9) == 0xFE


def test_quantize_rows_definition(oracle_mod):
    rng = np.random.default_rng(121)
    src = (rng.normal(0, 1, (40, 96)) * rng.uniform(0.01, 10, (40, 1))).astype(np.float32)
    src[3] = 0.0
    q, sc = oracle_mod.quantize_rows_e4m3(src)
    dec = np.vectorize(oracle_mod.e4m3_decode)(q)
    for r in range(40):
        amax = np.max(np.abs(src[r]))
        if amax == 0:
            assert sc[r] == 1.0 and not q[r].any()
            continue
        assert sc[r] == np.float32(amax) / np.float32(448.0)
        j = int(np.argmax(np.abs(src[r])))
        assert abs(dec[r, j]) == 448.0
        err = np.abs(dec[r] * sc[r] - src[r])
        assert np.all(err <= np.maximum(np.abs(src[r]) * 2.0 ** -4, sc[r] * 2.0 ** -10) * (1 + 1e-6))


def test_fp8_expert_op_within_the_h_rounding_bound(oracle_mod):
    """y from the oracle equals the fp64 SwiGLU of the dequantized weights and x, with h
    replaced by its e4m3 rounding: |y - y_exact| <= sum_j |gate_j| |s_d[o]| sum_i |W_d[o][i]|
    (|h_i| 2^-4 + s_b 2^-10), a bound a dropped term or a swapped index would break."""
    for f in (256, 384):   # one 256-wide span of h; a 256 and a trailing 128
        _check_fp8_expert_bound(oracle_mod, f)


def _check_fp8_expert_bound(oracle_mod, f):
    rng = np.random.default_rng(122 + f)
    E, d, n, m = 3, 64, 3, 2
    wg = (rng.normal(0, 1 / np.sqrt(d), (E * f, d))).astype(np.float32)
    wu = (rng.normal(0, 1 / np.sqrt(d), (E * f, d))).astype(np.float32)
    wd = (rng.normal(0, 1 / np.sqrt(f), (E * d, f))).astype(np.float32)
    x = rng.normal(0, 1, (n, d)).astype(np.float32)
    (qg, sg), (qu, su), (qd, sd), (qx, sx) = (oracle_mod.quantize_rows_e4m3(a) for a in (wg, wu, wd, x))
    dec = np.vectorize(oracle_mod.e4m3_decode)
    Wg = (dec(qg) * sg[:, None]).reshape(E, f, d)
    Wu = (dec(qu) * su[:, None]).reshape(E, f, d)
    Wd = (dec(qd) * sd[:, None]).reshape(E, d, f)
    X = dec(qx) * sx[:, None]
    ids = np.array([[0, 2], [1, 0], [2, 1]], np.int32)
    gates = rng.uniform(0.1, 1, (n, m))
    for t in range(n):
        y = oracle_mod.expert_op_token_fp8(qg.reshape(E, f, d), qu.reshape(E, f, d), qd.reshape(E, d, f),
                                           sg.reshape(E, f), su.reshape(E, f), sd.reshape(E, d), qx, sx, ids, gates, t)
        y_exact = np.zeros(d)
        bound = np.zeros(d)
        for j in range(m):
            e = ids[t, j]
            g, u = Wg[e] @ X[t], Wu[e] @ X[t]
            h = g / (1 + np.exp(-g)) * u
            y_exact += gates[t, j] * (Wd[e] @ h)
            spans = [(b0, min(f, b0 + 256)) for b0 in range(0, f, 256)]
            sb = np.concatenate([np.full(b1 - b0, np.max(np.abs(h[b0:b1])) / 448.0) for b0, b1 in spans])
            bound += gates[t, j] * (np.abs(Wd[e]) @ (np.abs(h) * 2.0 ** -4 + sb * 2.0 ** -10))
        assert np.all(np.abs(y - y_exact) <= bound * 1.001 + 1e-12)
        # and the bound is far below the output's scale (the quantization is not vacuous)
        assert np.max(np.abs(y - y_exact)) < 0.2 * np.sqrt(np.mean(y_exact ** 2))
