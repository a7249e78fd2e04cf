"""The ~3-bit expert weights on the GPU, through the C ABI, against the INT3
oracle: int3_pack and int3_dequant bit for bit, and the routed SwiGLU FFN
over INT3 banks (w3a16_moe_ffn, fp16 warp-MMA path) at the MoE workload's
sizes (64 experts of 2304 x 1024, top-8, 1..4 tokens) and at small shapes
with partial 512-k steps, shared and repeated experts, invalid ids and
repeated calls.  Bar for the FFN: relative L2 <= 5e-3 and max |err| <=
1e-2 * max |y_ref|, as for INT4."""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

from .test_gpu_parity import check_close, dev, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding
    binding.w4a16_device_error(clear=True)
    return binding


def u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("N,K", [(1, 128), (3, 256), (37, 640), (64, 2304)])
def test_int3_pack_bit_exact(w, oracle, N, K):
    codes = synth.codes3(20 + N, N, K)
    got = u32(w.int3_pack(dev(codes)))
    assert np.array_equal(got, oracle.pack3(codes))


def test_int3_pack_ignores_high_bits(w, oracle):
    codes = synth.codes(21, 5, 384)  # 0..15: bit 3 must be dropped
    got = u32(w.int3_pack(dev(codes)))
    assert np.array_equal(got, oracle.pack3(codes & 7))


@pytest.mark.parametrize("N,K,g,zmode", [(4, 128, 128, "uniform2to6"), (9, 512, 64, "const4"),
                                         (33, 768, 256, "uniform2to6"), (2, 384, 32, "uniform2to6")])
def test_int3_dequant_bit_exact(w, oracle, N, K, g, zmode):
    wq3 = synth.packed_weights3(22, N, K)
    s = synth.scales(22, N, K // g)
    z = synth.zeros(22, N, K // g, zmode)
    ref = oracle.dequant3(wq3, s, z, g)
    w32 = w.int3_dequant(dev(wq3), dev(s), dev(z), g, out_dtype=torch.float32)
    wbf = w.int3_dequant(dev(wq3), dev(s), dev(z), g, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert np.array_equal(w32.cpu().numpy().astype(np.float64), ref)
    assert np.array_equal(wbf.view(torch.int16).cpu().numpy().view(np.uint16), oracle.bf16_round(ref))


def bank(b):
    return tuple(dev(a) for a in b)


def run(w, p, ids=None, route_w=None):
    ids = p["ids"] if ids is None else ids
    route_w = p["route_w"] if route_w is None else route_w
    y = w.w3a16_moe_ffn(dev(p["x"]), dev(ids), dev(route_w), bank(p["gate"]), bank(p["up"]),
                        bank(p["down"]), 128)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("M,E,H,F,topk", [
    (1, 64, 2304, 1024, 8),    # the MoE workload, one token
    (4, 64, 2304, 1024, 8),    # 32 slots: the path's limit
    (8, 16, 1024, 512, 4),     # eight tokens
    (5, 8, 640, 256, 3),       # H = 5 blocks: one whole and one partial step
    (3, 12, 384, 384, 2),      # 3 blocks: a single partial step in both launches
    (2, 4, 128, 128, 2),       # one block each way, four experts
    (8, 8, 8192, 128, 2),      # a wide hidden size: launch 1 in 8-warp CTAs (16 do not fit)
])
def test_w3a16_moe_ffn_matches_oracle(w, oracle, M, E, H, F, topk):
    p = synth.moe_problem3(M=M, E=E, H=H, F=F, topk=topk, g=128, seed=9500 + M * 7 + E)
    y = run(w, p)
    ref = oracle.moe_ffn3(p["x"], p["ids"], p["route_w"], p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(y), ref["out"], "int3 moe M=%d E=%d H=%d F=%d topk=%d" % (M, E, H, F, topk))
    assert w.w4a16_device_error(clear=True) == 0


def test_w3a16_moe_ffn_extreme_codes(w, oracle):
    # every code 7 and every zero point 0 (the largest A operand, 1024 + 448,
    # in every field), then every code 0 with zero point 7
    p = synth.moe_problem3(M=2, E=4, H=512, F=256, topk=2, seed=9550)
    for code, zp in ((7, 0), (0, 7)):
        q = dict(p)
        for key in ("gate", "up", "down"):
            wq, s, z = p[key]
            q[key] = (np.full_like(wq, 0xFFFFFFFF if code == 7 else 0), s, np.full_like(z, zp))
        y = run(w, q)
        ref = oracle.moe_ffn3(q["x"], q["ids"], q["route_w"], q["gate"], q["up"], q["down"], 128)
        check_close(host_f64(y), ref["out"], "codes %d zero %d" % (code, zp))


def test_w3a16_moe_ffn_shared_and_repeated_experts(w, oracle):
    p = synth.moe_problem3(M=4, E=16, H=1024, F=512, topk=8, g=128, seed=9600)
    ids = p["ids"].copy()
    ids[:, 0] = 3
    ids[1, 1:4] = 3
    ids[3, :] = 5
    ids[0, 7] = 5
    y = run(w, p, ids=ids)
    ref = oracle.moe_ffn3(p["x"], ids, p["route_w"], p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(y), ref["out"], "int3 shared experts")
    assert w.w4a16_device_error(clear=True) == 0


def test_w3a16_moe_ffn_invalid_ids_are_skipped_and_flagged(w, oracle):
    p = synth.moe_problem3(M=3, E=16, H=1024, F=512, topk=4, g=128, seed=9700)
    ids = p["ids"].copy()
    ids[0, 1] = -1
    ids[2, 3] = 16
    w.w4a16_device_error(clear=True)
    y = run(w, p, ids=ids)
    assert w.w4a16_device_error(clear=True) & w.DEVERR_EXPERT_ID
    ref_ids = ids.copy()
    ref_rw = p["route_w"].copy()
    for t, j in ((0, 1), (2, 3)):
        ref_ids[t, j] = 0
        ref_rw[t, j] = 0.0
    ref = oracle.moe_ffn3(p["x"], ref_ids, ref_rw, p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(y), ref["out"], "int3 invalid ids")


def test_w3a16_moe_ffn_repeated_calls_are_identical(w):
    p = synth.moe_problem3(M=2, E=64, H=2304, F=1024, topk=8, g=128, seed=9800)
    args = (dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), bank(p["gate"]), bank(p["up"]),
            bank(p["down"]), 128)
    outs = [w.w3a16_moe_ffn(*args) for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert w.w4a16_device_error(clear=True) == 0


def test_w3a16_moe_ffn_refusals(w):
    p = synth.moe_problem3(M=1, E=4, H=256, F=128, topk=2, seed=9900)
    args = [dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), bank(p["gate"]), bank(p["up"]),
            bank(p["down"])]
    # groups other than 128 k, and more than 8 tokens, are outside the path
    for g in (64, 256):
        with pytest.raises(w.W4A16Error) as ei:
            w.w3a16_moe_ffn(*args, g)
        assert ei.value.status in (w.Status.ERR_UNSUPPORTED, w.Status.ERR_SHAPE)
    p9 = synth.moe_problem3(M=9, E=4, H=256, F=128, topk=2, seed=9901)
    with pytest.raises(w.W4A16Error) as ei:
        w.w3a16_moe_ffn(dev(p9["x"]), dev(p9["ids"]), dev(p9["route_w"]), bank(p9["gate"]),
                        bank(p9["up"]), bank(p9["down"]), 128)
    assert ei.value.status == w.Status.ERR_UNSUPPORTED
    # packing needs whole 128-code blocks
    with pytest.raises(w.W4A16Error) as ei:
        w.int3_pack(torch.zeros((2, 96), dtype=torch.uint8, device="cuda"))
    assert ei.value.status == w.Status.ERR_SHAPE


# ---- the expert-indexed GEMV over an INT3 bank (w3a16_moe_gemv) ----------

def run_gemv3(w, x, ids, bank3, route_w=None, x_per_slot=False):
    wq, s, z = bank3
    y = w.w3a16_moe_gemv(dev(x), dev(ids), dev(wq), dev(s), dev(z), 128,
                         route_w=None if route_w is None else dev(route_w), x_per_slot=x_per_slot)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("M,topk,E,N,K,x_per_slot,routed", [
    (1, 8, 64, 1024, 2304, False, False),   # the MoE workload's gate shape, per slot
    (1, 8, 64, 2304, 1024, True, True),     # its down shape with the routed sum
    (4, 8, 64, 2304, 1024, True, True),     # 32 slots: the path's limit
    (4, 8, 64, 1024, 2304, False, True),    # shared token rows, routed
    (8, 4, 16, 512, 640, True, False),      # K = 5 blocks: one whole and one partial step
    (3, 2, 12, 48, 384, False, True),       # 3 row tiles, a single partial step
    (5, 6, 7, 80, 896, True, False),        # 30 slots of 7 experts: entries of up to 8 slots
    (2, 3, 5, 16, 128, False, False),       # one row tile, one block
    (2, 8, 64, 2560, 1024, False, False),   # 160 row tiles: CTAs own whole row tiles
])
def test_w3a16_moe_gemv_matches_oracle(w, oracle, M, topk, E, N, K, x_per_slot, routed):
    seed = 9300 + M * 31 + topk * 7 + E
    ids, route_w = synth.routing(seed, M, topk, E)
    bank3 = synth.expert_bank3(seed, E, N, K)
    x = synth.activations(seed, (M, topk, K) if x_per_slot else (M, K))
    rw = route_w if routed else None
    y = run_gemv3(w, x, ids, bank3, rw, x_per_slot)
    ref = oracle.moe_gemv3(x, ids, rw, *bank3, 128, x_per_slot=x_per_slot)
    check_close(host_f64(y), ref, "int3 moe_gemv M=%d topk=%d E=%d N=%d K=%d" % (M, topk, E, N, K))
    assert w.w4a16_device_error(clear=True) == 0


def test_w3a16_moe_gemv_one_hot_is_bit_exact(w, oracle):
    # one nonzero activation per slot: every output is one exact product,
    # so the bf16 result is the rounding of W_e[n][k0] * x bit for bit
    M, topk, E, N, K = 2, 4, 6, 64, 640
    ids, _ = synth.routing(9350, M, topk, E)
    bank3 = synth.expert_bank3(9350, E, N, K, zero_mode="uniform2to6")
    x = np.zeros((M, topk, K), np.uint16)
    ks = [0, 29, 30, 31, 130, 383, 511, 639]
    for t in range(M):
        for j in range(topk):
            x[t, j, ks[t * topk + j]] = 0x3F80 if (t + j) % 2 == 0 else 0xC0A0   # 1.0 or -5.0
    y = run_gemv3(w, x, ids, bank3, x_per_slot=True)
    ref = oracle.moe_gemv3(x, ids, None, *bank3, 128, x_per_slot=True)
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.bf16_round(ref))


def test_w3a16_moe_gemv_one_expert_in_every_slot(w, oracle):
    # 32 slots of one expert: four entries of eight slots share its rows
    M, topk, E, N, K = 4, 8, 9, 256, 1024
    ids = np.full((M, topk), 7, np.int32)
    _, route_w = synth.routing(9360, M, topk, E)
    bank3 = synth.expert_bank3(9360, E, N, K)
    x = synth.activations(9360, (M, topk, K))
    for rw in (None, route_w):
        y = run_gemv3(w, x, ids, bank3, rw, x_per_slot=True)
        ref = oracle.moe_gemv3(x, ids, rw, *bank3, 128, x_per_slot=True)
        check_close(host_f64(y), ref, "one expert routed=%s" % (rw is not None))
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("routed", [False, True])
def test_w3a16_moe_gemv_invalid_ids_are_zero_and_flagged(w, oracle, routed):
    M, topk, E, N, K = 3, 4, 10, 128, 512
    ids, route_w = synth.routing(9370, M, topk, E)
    ids = ids.copy()
    ids[0, 1] = -1
    ids[2, 3] = E
    bank3 = synth.expert_bank3(9370, E, N, K)
    x = synth.activations(9370, (M, K))
    rw = route_w if routed else None
    w.w4a16_device_error(clear=True)
    y = run_gemv3(w, x, ids, bank3, rw)
    assert w.w4a16_device_error(clear=True) & w.DEVERR_EXPERT_ID
    ref = oracle.moe_gemv3(x, ids, rw, *bank3, 128, allow_bad_ids=True)
    if not routed:
        got = host_f64(y)
        assert np.all(got[0, 1] == 0) and np.all(got[2, 3] == 0)
    check_close(host_f64(y), ref, "int3 moe_gemv invalid ids routed=%s" % routed)


def test_w3a16_moe_gemv_repeated_calls_and_stream_order(w):
    M, topk, E, N, K = 2, 8, 64, 2304, 1024
    ids, route_w = synth.routing(9380, M, topk, E)
    bank3 = tuple(dev(a) for a in synth.expert_bank3(9380, E, N, K))
    x = dev(synth.activations(9380, (M, topk, K)))
    d_ids, d_rw = dev(ids), dev(route_w)
    outs = [w.w3a16_moe_gemv(x, d_ids, *bank3, 128, route_w=d_rw, x_per_slot=True) for _ in range(3)]
    # a producer of the activations just before the call: the launch reads
    # nothing before the preceding kernel has finished
    x2 = torch.empty_like(x)
    x2.copy_(x)
    outs.append(w.w3a16_moe_gemv(x2, d_ids, *bank3, 128, route_w=d_rw, x_per_slot=True))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("routed", [False, True])
def test_w3a16_moe_gemv_no_valid_id(w, routed):
    M, topk, E, N, K = 2, 4, 6, 96, 256
    ids = np.array([[-1, 6, 7, -2], [100, -1, 6, 9]], np.int32)
    _, route_w = synth.routing(9390, M, topk, E)
    bank3 = synth.expert_bank3(9390, E, N, K)
    x = synth.activations(9390, (M, K))
    w.w4a16_device_error(clear=True)
    y = run_gemv3(w, x, ids, bank3, route_w if routed else None)
    assert w.w4a16_device_error(clear=True) & w.DEVERR_EXPERT_ID
    assert y.shape == ((M, N) if routed else (M, topk, N))
    assert torch.count_nonzero(y.float()).item() == 0
