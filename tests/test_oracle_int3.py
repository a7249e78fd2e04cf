"""Pins for the ~3-bit expert-weight oracle (no GPU).

The pages give no format for the ~3-bit expert weights (local-kimi README,
hardware-requirements paragraph), so the format is this library's reading
(stated in the oracle's int3 source).  The pins tie the oracle to that
statement and to things other than itself: words derived by hand
(tests/golden/pack3_words.txt), the fact that every code bit owns exactly
one distinct bit of its block, and -- since every 3-bit code 0..7 is also an
INT4 code -- the independently pinned INT4 oracle, which must give the same
weights, products and FFN chain on the same codes.  Closed forms, one-hot
activations and an fp64 library matmul pin the INT3 GEMV directly.
test_oracle_mutants.py plants slips here too.
"""
import os

import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pack3():
    singles, patterns = [], []
    with open(os.path.join(GOLDEN, "pack3_words.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            head, tail = line.split(":")
            h = head.split()
            if h[0] == "single":
                K, k, q = int(h[1]), int(h[2]), int(h[3])
                words = {int(a): int(b, 16) for a, b in (t.split("=") for t in tail.split())}
                singles.append((K, k, q, words))
            else:
                patterns.append((h[0], int(h[1]), [int(t, 16) for t in tail.split()]))
    return singles, patterns


def test_pack3_golden_words(oracle):
    singles, patterns = _read_pack3()
    assert len(singles) >= 10 and len(patterns) == 2
    for K, k, q, words in singles:
        codes = np.zeros((1, K), np.uint8)
        codes[0, k] = q
        w = oracle.pack3(codes)[0]
        want = np.zeros(K // 128 * 12, np.uint32)
        for i, v in words.items():
            want[i] = v
        assert np.array_equal(w, want), (k, q, [hex(v) for v in w])
        assert np.array_equal(oracle.unpack3(w[None, :], K), codes)
    for name, K, words in patterns:
        ks = np.arange(K)
        codes = (ks % 8 if name == "mod8" else np.full(K, 7)).astype(np.uint8)[None, :]
        w = oracle.pack3(codes)[0]
        want = np.resize(np.array(words, np.uint32), w.size)
        assert np.array_equal(w, want), name
        assert np.array_equal(oracle.unpack3(w[None, :], K), codes)


def test_pack3_every_code_bit_owns_one_bit():
    # each (code, bit) of a 128-code block, set alone, sets exactly one bit of
    # the block's 384, and the 384 (code, bit) pairs set 384 different bits
    import oracle as o
    seen = set()
    for k in range(128):
        for j in range(3):
            codes = np.zeros((1, 128), np.uint8)
            codes[0, k] = 1 << j
            w = o.pack3(codes)[0]
            bits = [(i, b) for i in range(12) for b in range(32) if (int(w[i]) >> b) & 1]
            assert len(bits) == 1, (k, j, bits)
            seen.add(bits[0])
    assert len(seen) == 384


def test_pack3_round_trip_random(oracle):
    codes = synth.codes3(3, 7, 640)
    wq3 = oracle.pack3(codes)
    assert wq3.shape == (7, 60)
    assert np.array_equal(oracle.unpack3(wq3, 640), codes)
    # and words -> codes -> words (uniform words are valid packings)
    words = synth.packed_weights3(4, 5, 384)
    assert np.array_equal(oracle.pack3(oracle.unpack3(words, 384)), words)


def _int4_of(codes):
    import oracle as o
    return o.pack(codes)


def test_dequant3_equals_int4_dequant_on_the_same_codes(oracle):
    N, K, g = 9, 512, 128
    codes = synth.codes3(5, N, K)
    scale = synth.scales(5, N, K // g)
    zero = synth.zeros(5, N, K // g, "uniform2to6")
    w3 = oracle.dequant3(oracle.pack3(codes), scale, zero, g)
    w4 = oracle.dequant(_int4_of(codes), scale, zero, g)
    assert np.array_equal(w3, w4)
    # and the zero point, scale and group index reach the value
    s = oracle.bf16_to_f64(scale)
    want = (codes.astype(np.float64) - np.repeat(zero, g, axis=1)) * np.repeat(s, g, axis=1)
    assert np.array_equal(w3, want)


@pytest.mark.parametrize("g", [128, 64, 256])
def test_gemv3_equals_int4_gemv_on_the_same_codes(oracle, g):
    M, N, K = 3, 20, 768
    codes = synth.codes3(6, N, K)
    scale = synth.scales(6, N, K // g)
    zero = synth.zeros(6, N, K // g, "uniform2to6")
    x = synth.activations(6, (M, K))
    y3 = oracle.gemv3(x, oracle.pack3(codes), scale, zero, g)
    y4 = oracle.gemv(x, _int4_of(codes), scale, zero, g)
    assert np.array_equal(y3, y4)


@pytest.mark.parametrize("c", [0, 3, 7])
def test_gemv3_closed_form_constant_codes(oracle, c):
    M, N, K, g = 2, 12, 512, 128
    G = K // g
    wq3 = oracle.pack3(np.full((N, K), c, np.uint8))
    scale = synth.scales(7, N, G)
    zero = synth.zeros(7, N, G, "uniform2to6")
    x = synth.activations(7, (M, K))
    xs = oracle.bf16_to_f64(x).reshape(M, G, g).sum(axis=2)
    coef = (c - zero.astype(np.float64)) * oracle.bf16_to_f64(scale)
    np.testing.assert_allclose(oracle.gemv3(x, wq3, scale, zero, g), xs @ coef.T, rtol=1e-12, atol=1e-12)


def test_gemv3_one_hot_and_library_matmul(oracle):
    N, K, g = 16, 384, 128
    wq3 = synth.packed_weights3(8, N, K)
    scale = synth.scales(8, N, K // g)
    zero = synth.zeros(8, N, K // g, "uniform2to6")
    W = oracle.dequant3(wq3, scale, zero, g)
    for k0 in (0, 9, 10, 29, 30, 31, 32, 127, 128, 383):
        x = np.zeros((1, K), np.uint16)
        x[0, k0] = 0x3F80
        assert np.array_equal(oracle.gemv3(x, wq3, scale, zero, g)[0], W[:, k0])
    x = synth.activations(8, (3, K))
    ref = torch.matmul(torch.from_numpy(oracle.bf16_to_f64(x)), torch.from_numpy(W).T).numpy()
    np.testing.assert_allclose(oracle.gemv3(x, wq3, scale, zero, g), ref, rtol=1e-12, atol=1e-10)


def test_moe_ffn3_equals_int4_chain_on_the_same_codes(oracle):
    M, E, H, F, topk, g = 2, 6, 256, 128, 3, 128
    ids, route_w = synth.routing(9, M, topk, E)
    x = synth.activations(9, (M, H))
    banks3, banks4 = [], []
    for sub, (n, k) in enumerate(((F, H), (F, H), (H, F)), start=1):
        codes = synth.codes3(9, E * n, k, sub)
        s = synth.scales(9, E * n, k // g, sub).reshape(E, n, k // g)
        z = synth.zeros(9, E * n, k // g, "uniform2to6", sub).reshape(E, n, k // g)
        banks3.append((oracle.pack3(codes).reshape(E, n, -1), s, z))
        banks4.append((_int4_of(codes).reshape(E, n, -1), s, z))
    r3 = oracle.moe_ffn3(x, ids, route_w, *banks3, g)
    r4 = oracle.moe_ffn(x, ids, route_w, *banks4, g)
    for key in ("gate", "up", "h", "d", "out"):
        assert np.array_equal(r3[key], r4[key]), key


def test_moe_ffn3_rejects_bad_expert_id(oracle):
    p = synth.moe_problem3(M=1, E=4, H=128, F=128, topk=2, seed=10)
    ids = p["ids"].copy()
    ids[0, 1] = 4
    with pytest.raises(ValueError):
        oracle.moe_ffn3(p["x"], ids, p["route_w"], p["gate"], p["up"], p["down"], 128)


@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_gemv3_equals_int4_expert_gemv_on_the_same_codes(oracle, x_per_slot):
    M, E, N, K, topk, g = 3, 5, 24, 384, 2, 128
    ids, route_w = synth.routing(11, M, topk, E)
    codes = synth.codes3(11, E * N, K)
    s = synth.scales(11, E * N, K // g).reshape(E, N, K // g)
    z = synth.zeros(11, E * N, K // g, "uniform2to6").reshape(E, N, K // g)
    wq3 = oracle.pack3(codes).reshape(E, N, -1)
    wq4 = _int4_of(codes).reshape(E, N, -1)
    x = synth.activations(11, (M, topk, K) if x_per_slot else (M, K))
    for rw in (None, route_w):
        y3 = oracle.moe_gemv3(x, ids, rw, wq3, s, z, g, x_per_slot=x_per_slot)
        y4 = oracle.moe_gemv(x, ids, rw, wq4, s, z, g, x_per_slot=x_per_slot)
        assert np.array_equal(y3, y4)


def test_moe_gemv3_bad_ids(oracle):
    M, E, N, K, topk, g = 2, 4, 16, 256, 2, 128
    ids = np.array([[0, 4], [-1, 2]], np.int32)
    rw = np.full((M, topk), 0.5, np.float32)
    wq3 = synth.packed_weights3(12, E * N, K).reshape(E, N, -1)
    s = synth.scales(12, E * N, K // g).reshape(E, N, K // g)
    z = synth.zeros(12, E * N, K // g, "uniform2to6").reshape(E, N, K // g)
    x = synth.activations(12, (M, K))
    with pytest.raises(ValueError):
        oracle.moe_gemv3(x, ids, rw, wq3, s, z, g)
    y = oracle.moe_gemv3(x, ids, None, wq3, s, z, g, allow_bad_ids=True)
    assert np.all(y[0, 1] == 0) and np.all(y[1, 0] == 0)   # invalid slots: zero rows
    ok = oracle.moe_gemv3(x, np.array([[0, 0], [2, 2]], np.int32), None, wq3, s, z, g)
    assert np.array_equal(y[0, 0], ok[0, 0]) and np.array_equal(y[1, 1], ok[1, 1])
