"""The routed SwiGLU expert FFN on the fp16 warp-MMA path (w4a16_moe_ffn with
1..8 tokens, at most 32 routed slots, g = 128): against the oracle's chain
(gate and up GEMVs, bf16 SwiGLU, down GEMVs, routed sum in fp64), over
shapes whose K needs a partial last 512-k step, token and slot counts up to
the path's limits, experts shared by several tokens and by several slots of
one token (more than 8 slots on one expert), invalid ids, and repeated calls
(the routed-sum counters reset themselves).  Bar: relative L2 <= 5e-3 and
max |err| <= 1e-2 * max |y_ref|."""
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


def bank(b):
    return tuple(dev(a) for a in b)


def run(w, p, ids=None, route_w=None):
    ids = p["ids"] if ids is None else ids
    route_w = p["route_w"] if route_w is None else route_w
    y = w.moe_ffn(dev(p["x"]), dev(ids), dev(route_w), bank(p["gate"]), bank(p["up"]),
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
    (8, 8, 8192, 256, 4),      # a wide hidden size: launch 1 in 8-warp CTAs (16 do not fit)
])
def test_moe_hmma_matches_oracle(w, oracle, M, E, H, F, topk):
    p = synth.moe_problem(M=M, E=E, H=H, F=F, topk=topk, g=128, seed=9000 + M * 7 + E)
    y = run(w, p)
    ref = oracle.moe_ffn(p["x"], p["ids"], p["route_w"], p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(y), ref["out"], "moe hmma M=%d E=%d H=%d F=%d topk=%d" % (M, E, H, F, topk))
    assert w.w4a16_device_error(clear=True) == 0


def test_moe_hmma_shared_and_repeated_experts(w, oracle):
    # every token routes slot 0 to expert 3, token 1 routes three more slots
    # to it (same token, same expert: identical products), and token 3 routes
    # all its slots to expert 5: expert 3 then has 7 slots, expert 5 eight
    # plus one more from token 0 -- more than one group of 8
    p = synth.moe_problem(M=4, E=16, H=1024, F=512, topk=8, g=128, seed=9100)
    ids = p["ids"].copy()
    ids[:, 0] = 3
    ids[1, 1:4] = 3
    ids[3, :] = 5
    ids[0, 7] = 5
    y = run(w, p, ids=ids)
    ref = oracle.moe_ffn(p["x"], ids, p["route_w"], p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(y), ref["out"], "shared experts")
    assert w.w4a16_device_error(clear=True) == 0


def test_moe_hmma_invalid_ids_are_skipped_and_flagged(w, oracle):
    p = synth.moe_problem(M=3, E=16, H=1024, F=512, topk=4, g=128, seed=9200)
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
    ref = oracle.moe_ffn(p["x"], ref_ids, ref_rw, p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(y), ref["out"], "invalid ids")


def test_moe_hmma_repeated_calls_are_identical(w):
    # the per-chunk counters of the routed sum are cleared by the first
    # launch and reset by the last arrival: calls in a row agree bit for bit
    p = synth.moe_problem(M=2, E=64, H=2304, F=1024, topk=8, g=128, seed=9300)
    args = (dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), bank(p["gate"]), bank(p["up"]),
            bank(p["down"]), 128)
    outs = [w.moe_ffn(*args) for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert w.w4a16_device_error(clear=True) == 0


# ---- the down launch on its own: the INT4 expert GEMV (kernel 4) ---------

def bank_dev(b):
    return tuple(dev(a) for a in b)


@pytest.mark.parametrize("M,topk,E,N,K,x_per_slot,routed", [
    (1, 8, 64, 1024, 2304, False, False),   # the MoE workload's gate shape, per slot
    (1, 8, 64, 2304, 1024, True, True),     # its down shape with the routed sum
    (4, 8, 64, 2304, 1024, True, True),     # 32 slots
    (2, 8, 64, 1024, 2304, False, True),
    (8, 4, 16, 512, 640, True, False),      # K = 5 blocks: one whole and one partial step
    (3, 2, 12, 48, 384, False, True),       # 3 row tiles, a single partial step
    (5, 6, 7, 80, 896, True, False),        # 30 slots of 7 experts
    (2, 3, 5, 16, 128, False, False),       # one row tile, one block
    (4, 8, 64, 1024, 2304, False, False),   # 32 slots on 4 staged token rows
    (2, 8, 64, 2560, 1024, False, False),   # 160 row tiles: CTAs own whole row tiles
])
def test_fp16_expert_gemv_matches_oracle(w, oracle, M, topk, E, N, K, x_per_slot, routed):
    seed = 9400 + M * 31 + topk * 7 + E
    ids, route_w = synth.routing(seed, M, topk, E)
    bank = synth.expert_bank(seed, E, N, K, 128, "uniform6to10")
    x = synth.activations(seed, (M, topk, K) if x_per_slot else (M, K))
    rw = route_w if routed else None
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *bank_dev(bank), 128,
                         route_w=None if rw is None else dev(rw), x_per_slot=x_per_slot,
                         kernel_id=4)
    torch.cuda.synchronize()
    ref = oracle.moe_gemv(x, ids, rw, *bank, 128, x_per_slot=x_per_slot)
    check_close(host_f64(y), ref, "fp16 expert gemv M=%d topk=%d E=%d N=%d K=%d" % (M, topk, E, N, K))
    assert w.w4a16_device_error(clear=True) == 0


def test_fp16_expert_gemv_one_hot_is_bit_exact(w, oracle):
    M, topk, E, N, K = 2, 4, 6, 64, 640
    ids, _ = synth.routing(9450, M, topk, E)
    bank = synth.expert_bank(9450, E, N, K, 128, "uniform6to10")
    x = np.zeros((M, topk, K), np.uint16)
    ks = [0, 7, 8, 127, 130, 383, 511, 639]
    for t in range(M):
        for j in range(topk):
            x[t, j, ks[t * topk + j]] = 0x3F80 if (t + j) % 2 == 0 else 0xC0A0   # 1.0 or -5.0
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *bank_dev(bank), 128, x_per_slot=True, kernel_id=4)
    torch.cuda.synchronize()
    ref = oracle.moe_gemv(x, ids, None, *bank, 128, x_per_slot=True)
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.bf16_round(ref))


@pytest.mark.parametrize("routed", [False, True])
def test_fp16_expert_gemv_invalid_ids(w, oracle, routed):
    M, topk, E, N, K = 3, 4, 10, 128, 512
    ids, route_w = synth.routing(9460, M, topk, E)
    ids = ids.copy()
    ids[1, 0] = -7
    ids[2, 2] = E + 3
    bank = synth.expert_bank(9460, E, N, K, 128, "uniform6to10")
    x = synth.activations(9460, (M, K))
    rw = route_w if routed else None
    w.w4a16_device_error(clear=True)
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *bank_dev(bank), 128,
                         route_w=None if rw is None else dev(rw), kernel_id=4)
    torch.cuda.synchronize()
    assert w.w4a16_device_error(clear=True) & w.DEVERR_EXPERT_ID
    # reference: the bad slots given a valid id and, routed, a zero weight
    ref_ids = ids.copy()
    ref_ids[1, 0] = ref_ids[2, 2] = 0
    got = host_f64(y)
    if routed:
        ref_rw = route_w.copy()
        ref_rw[1, 0] = ref_rw[2, 2] = 0.0
        ref = oracle.moe_gemv(x, ref_ids, ref_rw, *bank, 128)
    else:
        ref = oracle.moe_gemv(x, ref_ids, None, *bank, 128)
        assert np.all(got[1, 0] == 0) and np.all(got[2, 2] == 0)
        ref[1, 0] = ref[2, 2] = 0.0
    check_close(got, ref, "fp16 expert gemv invalid ids routed=%s" % routed)


def test_fp16_expert_gemv_refusals(w):
    ids = dev(np.zeros((5, 8), np.int32))   # 40 slots: beyond the kernel
    bank = bank_dev(synth.expert_bank(9470, 4, 64, 256, 128))
    x = dev(synth.activations(9470, (5, 256)))
    with pytest.raises(w.W4A16Error) as ei:
        w.w4a16_moe_gemv(x, ids, *bank, 128, kernel_id=4)
    assert ei.value.status == w.Status.ERR_UNSUPPORTED
    # the library's choice still serves it
    w.w4a16_moe_gemv(x, ids, *bank, 128)
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits", [4, 3])
def test_expert_gemv_after_a_producing_gemv(w, bits):
    # the expert GEMV's activations come from the GEMV launched just before
    # it (a kernel that releases its dependents early): the expert GEMV must
    # read them only after that GEMV has finished -- its result equals the
    # one computed after a full synchronisation, call after call
    M, topk, E, N, K, K0 = 2, 8, 64, 1024, 2304, 4096
    p = synth.dense_problem(M, K, K0, 128, "uniform6to10", seed=9480)
    ids, rw = synth.routing(9480, M, topk, E)
    bank = bank_dev(synth.expert_bank3(9480, E, N, K) if bits == 3 else
                    synth.expert_bank(9480, E, N, K, 128, "uniform6to10"))
    x0, wq0, s0, z0 = (dev(p[k]) for k in ("x", "wq", "scale", "zero"))
    d_ids, d_rw = dev(ids), dev(rw)

    def expert(x, routed):
        f = w.w3a16_moe_gemv if bits == 3 else w.w4a16_moe_gemv
        return f(x, d_ids, *bank, 128, route_w=d_rw if routed else None)

    for routed in (False, True):
        xs = w.w4a16_gemv(x0, wq0, s0, z0, 128)
        torch.cuda.synchronize()
        want = expert(xs, routed)
        torch.cuda.synchronize()
        for _ in range(3):
            xc = w.w4a16_gemv(x0, wq0, s0, z0, 128, weights_static=True)
            got = expert(xc, routed)
            torch.cuda.synchronize()
            assert torch.equal(got, want), routed
    assert w.w4a16_device_error(clear=True) == 0


def test_expert_gemv_random_shapes_against_the_oracle(w, oracle):
    # seeded random shapes within the fp16 kernel's limits: token and slot
    # counts, experts (often fewer than the slots), row tiles from 1 to more
    # than the SM count, K from one block up, a row per token or per slot,
    # per-slot outputs or routed sums, some invalid ids; every case through
    # the library's choice, the bf16 kernel and (over the same codes) the
    # INT3 path
    rng = np.random.default_rng(9490)
    for case in range(12):
        topk = int(rng.integers(1, 9))
        M = int(rng.integers(1, 32 // topk + 1))
        E = int(rng.integers(1, 40))
        N = 16 * int(rng.choice([1, 3, 8, 40, 170]))
        K = 128 * int(rng.integers(1, 12))
        x_per_slot = bool(rng.integers(0, 2))
        routed = bool(rng.integers(0, 2))
        seed = 9491 + case
        ids, rw = synth.routing(seed, M, topk, E) if topk <= E else (
            rng.integers(0, E, size=(M, topk)).astype(np.int32), np.full((M, topk), 1.0 / topk, np.float32))
        if case % 4 == 3:
            ids = ids.copy()
            ids[0, 0] = -1
        codes = synth.codes3(seed, E * N, K)
        s = synth.scales(seed, E * N, K // 128).reshape(E, N, K // 128)
        z = synth.zeros(seed, E * N, K // 128, "uniform2to6").reshape(E, N, K // 128)
        wq4 = oracle.pack(codes).reshape(E, N, -1)
        wq3 = oracle.pack3(codes).reshape(E, N, -1)
        x = synth.activations(seed, (M, topk, K) if x_per_slot else (M, K))
        r = rw if routed else None
        ref_ids, ref_rw = ids, r
        if case % 4 == 3:  # the oracle leaves the invalid slot out
            ref_ids = ids.copy()
            ref_ids[0, 0] = 0
            if routed:
                ref_rw = rw.copy()
                ref_rw[0, 0] = 0.0
        ref = oracle.moe_gemv(x, ref_ids, ref_rw, wq4, s, z, 128, x_per_slot=x_per_slot)
        if case % 4 == 3 and not routed:
            ref[0, 0] = 0.0
        what = "case %d: M=%d topk=%d E=%d N=%d K=%d per_slot=%d routed=%d" % (
            case, M, topk, E, N, K, x_per_slot, routed)
        args = (dev(x), dev(ids))
        for kid in (0, 2):
            y = w.w4a16_moe_gemv(*args, dev(wq4), dev(s), dev(z), 128,
                                 route_w=None if r is None else dev(r), x_per_slot=x_per_slot,
                                 kernel_id=kid)
            torch.cuda.synchronize()
            check_close(host_f64(y), ref, what + " kernel %d" % kid)
        y3 = w.w3a16_moe_gemv(*args, dev(wq3), dev(s), dev(z), 128,
                              route_w=None if r is None else dev(r), x_per_slot=x_per_slot)
        torch.cuda.synchronize()
        check_close(host_f64(y3), ref, what + " INT3")
        w.w4a16_device_error(clear=True)
