"""Equivalence of every registered variant with the oracle (the reference),
on seeded inputs through the C ABI; a variant outside its limits must refuse
with ERR_UNSUPPORTED, never compute something else.  Same bar as the parity
tests: relative L2 <= 5e-3 and max |err| <= 1e-2 * max |y_ref|."""
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

from .test_gpu_parity import check_close, dense_dev, dev, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def reg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding, registry
    binding.w4a16_device_error(clear=True)
    return registry


DENSE = [(1, 300, 1024, 128), (2, 257, 2304, 128), (5, 130, 4096, 128), (16, 64, 2048, 256),
         (8, 100, 3072, 128), (12, 96, 2048, 128)]


@pytest.mark.parametrize("M,N,K,g", DENSE)
@pytest.mark.parametrize("variant", ["planned", "cuda_core", "warp_mma", "tcgen05", "fp16_mma"])
def test_dense_variants_match_the_reference(reg, oracle, variant, M, N, K, g):
    from w4a16_int4_weight_gemv_gb300 import binding
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=8000 + M)
    f = reg.OPS["w4a16_dense"][variant]
    try:
        y = f(*dense_dev(p), g, out_dtype=torch.float32)
    except binding.W4A16Error as e:
        assert e.status == binding.Status.ERR_UNSUPPORTED, variant
        assert variant in ("cuda_core", "tcgen05", "fp16_mma")
        return
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g), variant)
    assert binding.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M", [1, 3])
def test_grouped_variants_match_the_reference(reg, oracle, M):
    from w4a16_int4_weight_gemv_gb300 import binding
    E, N, K, g, topk = 12, 192, 2304, 128, 4
    wq, s, z = synth.expert_bank(81, E, N, K, g)
    ids, r = synth.routing(81, M, topk, E)
    x = synth.activations(81, (M, K))
    for variant, f in reg.OPS["w4a16_grouped"].items():
        y = f(dev(x), dev(ids), dev(wq), dev(s), dev(z), g, route_w=dev(r))
        torch.cuda.synchronize()
        check_close(host_f64(y), oracle.moe_gemv(x, ids, r, wq, s, z, g), variant)
    assert binding.w4a16_device_error(clear=True) == 0


def test_int3_grouped_variants_match_the_reference(reg, oracle):
    from w4a16_int4_weight_gemv_gb300 import binding
    E, N, K, g, topk, M = 12, 192, 2304, 128, 4, 3
    bank3 = synth.expert_bank3(84, E, N, K, g)
    ids, r = synth.routing(84, M, topk, E)
    x = synth.activations(84, (M, K))
    for variant, f in reg.OPS["w3a16_grouped"].items():
        for rw in (None, r):
            y = f(dev(x), dev(ids), *(dev(a) for a in bank3), g,
                  route_w=None if rw is None else dev(rw))
            torch.cuda.synchronize()
            check_close(host_f64(y), oracle.moe_gemv3(x, ids, rw, *bank3, g), variant)
    assert binding.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M", [1, 2])
def test_ffn_variants_match_the_reference(reg, oracle, M):
    from w4a16_int4_weight_gemv_gb300 import binding
    p = synth.moe_problem(M=M, E=16, H=1024, F=512, topk=4, g=128, seed=82)
    ref = oracle.moe_ffn(p["x"], p["ids"], p["route_w"], p["gate"], p["up"], p["down"], 128)
    bank = lambda b: tuple(dev(a) for a in b)
    for variant, f in reg.OPS["w4a16_ffn"].items():
        y = f(dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), bank(p["gate"]), bank(p["up"]),
              bank(p["down"]), 128)
        torch.cuda.synchronize()
        check_close(host_f64(y), ref["out"], variant)
    assert binding.w4a16_device_error(clear=True) == 0


def test_int3_ffn_variants_match_the_reference(reg, oracle):
    from w4a16_int4_weight_gemv_gb300 import binding
    p = synth.moe_problem3(M=2, E=16, H=1024, F=512, topk=4, g=128, seed=83)
    ref = oracle.moe_ffn3(p["x"], p["ids"], p["route_w"], p["gate"], p["up"], p["down"], 128)
    bank = lambda b: tuple(dev(a) for a in b)
    for variant, f in reg.OPS["w3a16_ffn"].items():
        y = f(dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), bank(p["gate"]), bank(p["up"]),
              bank(p["down"]), 128)
        torch.cuda.synchronize()
        check_close(host_f64(y), ref["out"], variant)
    assert binding.w4a16_device_error(clear=True) == 0
