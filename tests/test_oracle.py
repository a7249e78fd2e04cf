"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: hand-derived
fixtures in tests/golden/, closed forms, invariants, a library routine
(fp64 matmul, binary32->bf16 conversion, silu) or brute force on tiny
inputs.  Each was chosen so that a plausible slip in the oracle -- nibble
order, group or row indexing of scale/zero, the sign of (q - zero), a dropped
term, a transposed operand, double rounding -- fails at least one of them;
test_oracle_mutants.py plants such slips and checks that they are caught.
"""
import math
import os

import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pack_words():
    rows = []
    with open(os.path.join(GOLDEN, "pack_words.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            rows.append(([int(v) for v in parts[:8]], int(parts[8], 16)))
    return rows


def _read_bf16_cases():
    cases = []
    with open(os.path.join(GOLDEN, "bf16_round.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            expr, bits = line.rsplit(None, 1)
            cases.append((float(eval(expr, {"__builtins__": {}})), int(bits, 16)))
    return cases


def _read_tiny():
    d = {}
    with open(os.path.join(GOLDEN, "tiny_gemv.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            d[key] = vals
    return d


# ---- packing -------------------------------------------------------------

def test_pack_golden_words(oracle):
    rows = _read_pack_words()
    codes = np.array([r[0] for r in rows], np.uint8)
    want = np.array([r[1] for r in rows], np.uint32)
    got = oracle.pack(codes)
    assert got.shape == (len(rows), 1)
    assert np.array_equal(got[:, 0], want)
    assert np.array_equal(oracle.unpack(want.reshape(-1, 1), 8), codes)


def test_pack_unpack_round_trip_exhaustive(oracle):
    # every code value at every nibble position, in rows longer than one word
    K = 64
    codes = np.zeros((16 * 8, K), np.uint8)
    for v in range(16):
        for pos in range(8):
            r = v * 8 + pos
            codes[r, :] = (v * 7 + 3 + np.arange(K)) % 16
            codes[r, pos::8] = v
    wq = oracle.pack(codes)
    assert np.array_equal(oracle.unpack(wq, K), codes)
    rnd = synth.codes(0, 37, 256)
    assert np.array_equal(oracle.unpack(oracle.pack(rnd), 256), rnd)
    words = synth.packed_weights(3, 19, 128)
    assert np.array_equal(oracle.pack(oracle.unpack(words, 128)), words)


# ---- bf16 rounding -------------------------------------------------------

def test_bf16_round_golden(oracle):
    for v, bits in _read_bf16_cases():
        assert int(oracle.bf16_round(np.array([v]))[0]) == bits, (v, hex(bits))


def test_bf16_round_matches_library_conversion(oracle):
    # values representable in binary32: one rounding either way, so the
    # library's binary32 -> bf16 conversion is an independent reference
    r = np.random.default_rng(5)
    vals = np.concatenate([
        r.standard_normal(20000).astype(np.float32),
        (r.standard_normal(2000) * 1e-39).astype(np.float32),   # binary32 subnormals
        (np.clip(r.standard_normal(2000), -3.3, 3.3) * 1e38).astype(np.float32),  # near overflow
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf], np.float32),
    ])
    vals = vals[np.isfinite(vals) | np.isinf(vals)]
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(vals.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_widening_is_exact(oracle):
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7F80) != 0x7F80
    vals = oracle.bf16_to_f64(bits[finite])
    ref = torch.from_numpy(bits[finite].view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(vals, ref)
    assert np.array_equal(oracle.bf16_round(vals), bits[finite])


# ---- dequantisation ------------------------------------------------------

def test_dequant_exhaustive_small_integers(oracle):
    # every (code, zero) pair with scale 1: W must be the integer code - zero
    g = 8
    qs, zs = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    N = 256
    codes = np.repeat(qs.reshape(N, 1), g, axis=1).astype(np.uint8)
    wq = oracle.pack(codes)
    scale = np.full((N, 1), 0x3F80, np.uint16)             # bf16 1.0
    zero = zs.reshape(N, 1).astype(np.uint8)
    W = oracle.dequant(wq, scale, zero, g)
    expect_int = (qs.reshape(N) - zs.reshape(N)).astype(np.float64)
    assert np.array_equal(W, np.repeat(expect_int[:, None], g, axis=1))
    assert W.min() == -15 and W.max() == 15


def test_dequant_scales_by_power_of_two_and_group(oracle):
    # scale 2^e in group G of row n, codes 15, zero 0: W = 15 * 2^e exactly,
    # and each group of g columns takes its own row's scale
    N, K, g = 3, 32, 8
    G = K // g
    codes = np.full((N, K), 15, np.uint8)
    exps = np.arange(N * G).reshape(N, G) - 5
    scale = synth.f32_to_bf16_bits(np.ldexp(1.0, exps).astype(np.float32))
    zero = np.zeros((N, G), np.uint8)
    W = oracle.dequant(oracle.pack(codes), scale, zero, g)
    for n in range(N):
        for k in range(K):
            assert W[n, k] == 15.0 * 2.0 ** int(exps[n, k // g])


# ---- GEMV ----------------------------------------------------------------

def test_gemv_tiny_golden(oracle):
    d = _read_tiny()
    wq = np.array([int(v, 16) for v in d["wq"]], np.uint32).reshape(2, 2)
    zero = np.array([int(v) for v in d["zero"]], np.uint8).reshape(2, 2)
    scale = synth.f32_to_bf16_bits(np.array([float(v) for v in d["scale"]], np.float32)).reshape(2, 2)
    x = synth.f32_to_bf16_bits(np.array([[float(v) for v in d["x0"]], [float(v) for v in d["x1"]]], np.float32))
    y = oracle.gemv(x, wq, scale, zero, 8)
    want = np.array([[float(v) for v in d["y0"]], [float(v) for v in d["y1"]]])
    assert np.array_equal(y, want)


@pytest.mark.parametrize("c,zmode", [(0, "const8"), (15, "const8"), (3, "uniform6to10"), (11, "uniform6to10")])
def test_gemv_closed_form_constant_codes(oracle, c, zmode):
    # all codes = c: y[m][n] = sum_G (c - z[n,G]) * s[n,G] * sum_{k in G} x[m][k]
    M, N, K, g = 3, 40, 512, 128
    G = K // g
    codes = np.full((N, K), c, np.uint8)
    wq = oracle.pack(codes)
    scale = synth.scales(1, N, G)
    zero = synth.zeros(1, N, G, zmode)
    x = synth.activations(1, (M, K))
    xs = oracle.bf16_to_f64(x).reshape(M, G, g).sum(axis=2)           # [M, G]
    coef = (c - zero.astype(np.float64)) * oracle.bf16_to_f64(scale)   # [N, G]
    want = xs @ coef.T
    got = oracle.gemv(x, wq, scale, zero, g)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_gemv_one_hot_columns(oracle):
    # x = e_k0: y[n] must be exactly W[n][k0], for k0 in several groups
    N, K, g = 24, 512, 128
    p = synth.dense_problem(1, N, K, g, "uniform6to10", seed=2)
    W = oracle.dequant(p["wq"], p["scale"], p["zero"], g)
    for k0 in (0, 1, 7, 8, 127, 128, 200, 385, 511):
        x = np.zeros((1, K), np.uint16)
        x[0, k0] = 0x3F80
        y = oracle.gemv(x, p["wq"], p["scale"], p["zero"], g)
        assert np.array_equal(y[0], W[:, k0])


def test_gemv_matches_library_matmul(oracle):
    M, N, K, g = 4, 64, 1024, 128
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=4)
    W = torch.from_numpy(oracle.dequant(p["wq"], p["scale"], p["zero"], g))
    x = torch.from_numpy(oracle.bf16_to_f64(p["x"]))
    ref = torch.matmul(x, W.T).numpy()
    got = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-10)


def test_gemv_brute_force_tiny(oracle):
    # direct enumeration with python integers/fractions on a tiny case
    from fractions import Fraction
    M, N, K, g = 2, 5, 32, 16
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=6)
    codes = [[(int(p["wq"][n, k // 8]) >> (4 * (k % 8))) & 15 for k in range(K)] for n in range(N)]
    s = oracle.bf16_to_f64(p["scale"])
    xv = oracle.bf16_to_f64(p["x"])
    got = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for k in range(K):
                tot += Fraction(xv[m, k]) * (codes[n][k] - int(p["zero"][n, k // g])) * Fraction(s[n, k // g])
            assert abs(got[m, n] - float(tot)) <= 1e-12 * max(1.0, abs(float(tot)))


def test_gemv_invariants(oracle):
    M, N, K, g = 2, 16, 256, 128
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=8)
    y = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    # linearity in x: y(2x) = 2 y(x) exactly (power-of-two scaling)
    x2 = synth.f32_to_bf16_bits(2 * synth.bf16_bits_to_f32(p["x"]))
    assert np.array_equal(oracle.gemv(x2, p["wq"], p["scale"], p["zero"], g), 2 * y)
    # doubling every scale doubles y exactly
    s2 = synth.f32_to_bf16_bits(2 * synth.bf16_bits_to_f32(p["scale"]))
    assert np.array_equal(oracle.gemv(p["x"], p["wq"], s2, p["zero"], g), 2 * y)
    # (q, z) -> (q + 1, z + 1) leaves y unchanged where no code is 15
    codes = oracle.unpack(p["wq"], K)
    codes = np.minimum(codes, 14)
    wq_a = oracle.pack(codes)
    wq_b = oracle.pack(codes + 1)
    ya = oracle.gemv(p["x"], wq_a, p["scale"], p["zero"], g)
    yb = oracle.gemv(p["x"], wq_b, p["scale"], p["zero"] + 1, g)
    np.testing.assert_allclose(ya, yb, rtol=1e-13, atol=1e-12)
    # additivity in x
    xa = synth.activations(9, (M, K))
    xb = synth.activations(10, (M, K))
    xab = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(xa).astype(np.float64) + synth.bf16_bits_to_f32(xb))
    exact = (synth.bf16_bits_to_f32(xab).astype(np.float64) ==
             synth.bf16_bits_to_f32(xa).astype(np.float64) + synth.bf16_bits_to_f32(xb))
    rows_ok = exact.all(axis=1)
    if rows_ok.any():
        ya = oracle.gemv(xa, p["wq"], p["scale"], p["zero"], g)
        yb = oracle.gemv(xb, p["wq"], p["scale"], p["zero"], g)
        yab = oracle.gemv(xab, p["wq"], p["scale"], p["zero"], g)
        np.testing.assert_allclose(yab[rows_ok], (ya + yb)[rows_ok], rtol=1e-12, atol=1e-11)


def test_gemv_rows_matches_full(oracle):
    p = synth.dense_problem(3, 50, 256, 128, "uniform6to10", seed=11)
    full = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    rows = np.array([0, 49, 7, 7, 23], np.int64)
    part = oracle.gemv_rows(p["x"], p["wq"], p["scale"], p["zero"], 128, rows)
    assert np.array_equal(part, full[:, rows])


@pytest.mark.parametrize("threads", [1, 3, 0])
def test_gemv_parallel_equals_gemv(oracle, threads):
    # the threaded full-output GEMV evaluates each element with the same fp64
    # sum, so it equals gemv bit for bit (0 threads = all host threads), and
    # through it inherits gemv's pins (library matmul, closed forms, brute force)
    p = synth.dense_problem(3, 301, 1024, 128, "uniform6to10", seed=12)
    full = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    par = oracle.gemv_parallel(p["x"], p["wq"], p["scale"], p["zero"], 128, threads=threads)
    assert np.array_equal(par, full)
    W = torch.from_numpy(oracle.dequant(p["wq"], p["scale"], p["zero"], 128))
    ref = torch.matmul(torch.from_numpy(oracle.bf16_to_f64(p["x"])), W.T).numpy()
    np.testing.assert_allclose(par, ref, rtol=1e-12, atol=1e-10)
    assert oracle.max_threads() >= 1


# ---- SwiGLU --------------------------------------------------------------

def test_swiglu_closed_forms(oracle):
    one = np.array([0x3F80], np.uint16)
    zero = np.array([0x0000], np.uint16)
    # silu(0) = 0
    assert oracle.swiglu(zero, one)[0] == 0
    # silu(v) = v / 2 at... v=0 only; at large v silu(v) -> v, at large -v -> 0
    big = synth.f32_to_bf16_bits(np.array([40.0], np.float32))
    up = synth.f32_to_bf16_bits(np.array([3.0], np.float32))
    assert oracle.swiglu(big, up)[0] == synth.f32_to_bf16_bits(np.array([120.0], np.float32))[0]
    nbig = synth.f32_to_bf16_bits(np.array([-40.0], np.float32))
    assert abs(oracle.bf16_to_f64(oracle.swiglu(nbig, up))[0]) < 1e-15


def test_swiglu_matches_library_silu(oracle):
    gate = synth.activations(12, (4096,))
    up = synth.activations(13, (4096,))
    g64 = torch.from_numpy(oracle.bf16_to_f64(gate))
    u64 = torch.from_numpy(oracle.bf16_to_f64(up))
    ref = oracle.bf16_round((torch.nn.functional.silu(g64) * u64).numpy())
    assert np.array_equal(oracle.swiglu(gate, up), ref)


# ---- mixture of experts --------------------------------------------------

def _dense_chain(oracle, x, e, p, g):
    (wg, sg, zg), (wu, su, zu), (wd, sd, zd) = p["gate"], p["up"], p["down"]
    gate = oracle.bf16_round(oracle.gemv(x, wg[e], sg[e], zg[e], g))
    up = oracle.bf16_round(oracle.gemv(x, wu[e], su[e], zu[e], g))
    h = oracle.swiglu(gate, up)
    return oracle.gemv(h, wd[e], sd[e], zd[e], g)


def test_moe_gemv_slots_are_dense_gemvs(oracle):
    M, E, N, K, g, topk = 2, 6, 16, 256, 128, 3
    wq, s, z = synth.expert_bank(14, E, N, K, g)
    ids, _ = synth.routing(14, M, topk, E)
    x = synth.activations(14, (M, K))
    y = oracle.moe_gemv(x, ids, None, wq, s, z, g)
    for t in range(M):
        for j in range(topk):
            e = ids[t, j]
            assert np.array_equal(y[t, j], oracle.gemv(x[t:t + 1], wq[e], s[e], z[e], g)[0])
    xs = synth.activations(15, (M, topk, K))
    ys = oracle.moe_gemv(xs, ids, None, wq, s, z, g, x_per_slot=True)
    for t in range(M):
        for j in range(topk):
            e = ids[t, j]
            assert np.array_equal(ys[t, j], oracle.gemv(xs[t, j:j + 1], wq[e], s[e], z[e], g)[0])


def test_moe_gemv_routed_sum_is_linear(oracle):
    M, E, N, K, g, topk = 3, 5, 8, 128, 128, 2
    wq, s, z = synth.expert_bank(16, E, N, K, g)
    ids, r = synth.routing(16, M, topk, E)
    x = synth.activations(16, (M, K))
    per = oracle.moe_gemv(x, ids, None, wq, s, z, g)
    routed = oracle.moe_gemv(x, ids, r, wq, s, z, g)
    want = (r.astype(np.float64)[:, :, None] * per).sum(axis=1)
    np.testing.assert_allclose(routed, want, rtol=1e-13, atol=1e-13)


def test_moe_ffn_one_hot_route_is_one_dense_chain(oracle):
    p = synth.moe_problem(M=2, E=4, H=256, F=128, topk=2, g=128, seed=17)
    r = np.zeros_like(p["route_w"])
    r[:, 1] = 1.0
    res = oracle.moe_ffn(p["x"], p["ids"], r, p["gate"], p["up"], p["down"], 128)
    for t in range(2):
        want = _dense_chain(oracle, p["x"][t:t + 1], p["ids"][t, 1], p, 128)[0]
        assert np.array_equal(res["out"][t], want)


def test_moe_ffn_identical_experts(oracle):
    # every expert the same: out = (sum_j r_j) * chain = chain up to fp32 rounding of r
    p = synth.moe_problem(M=2, E=3, H=256, F=128, topk=3, g=128, seed=18)
    for key in ("gate", "up", "down"):
        wq, s, z = p[key]
        p[key] = (np.repeat(wq[:1], 3, 0), np.repeat(s[:1], 3, 0), np.repeat(z[:1], 3, 0))
    res = oracle.moe_ffn(p["x"], p["ids"], p["route_w"], p["gate"], p["up"], p["down"], 128)
    for t in range(2):
        chain = _dense_chain(oracle, p["x"][t:t + 1], 0, p, 128)[0]
        np.testing.assert_allclose(res["out"][t], chain * float(p["route_w"][t].astype(np.float64).sum()),
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(res["out"][t], chain, rtol=1e-6, atol=1e-6)


def test_moe_rejects_bad_expert_id(oracle):
    wq, s, z = synth.expert_bank(19, 2, 8, 128, 128)
    x = synth.activations(19, (1, 128))
    with pytest.raises(ValueError):
        oracle.moe_gemv(x, np.array([[0, 2]], np.int32), None, wq, s, z, 128)


def test_tolerance_headroom():
    # bf16 output rounding alone costs at most 2^-9 relative per element,
    # inside the 5e-3 relative-L2 bar the GPU parity tests use
    assert 2.0 ** -9 < 5e-3
    assert math.isclose(2.0 ** -9, 0.001953125)
