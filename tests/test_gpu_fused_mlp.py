"""Parity of the fused decode-MLP path through the C ABI: one GEMV over gate
and up weights interleaved in 8-row blocks whose epilogue stores the SwiGLU
of the two products (W4A16_FLAG_SWIGLU_OUTPUT), against the oracle's GEMVs
followed by the oracle's SwiGLU; and against the unfused library chain (plain
GEMV, then w4a16_swiglu), bit for bit, since both round the same fp32 sums.
"""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

from .test_gpu_parity import REL_L2, MAX_REL, dense_dev, dev

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


def gate_up_problem(M, I, K, g, seed):
    gate = synth.dense_problem(M, I, K, g, "uniform6to10", seed=seed)
    up = synth.dense_problem(M, I, K, g, "uniform6to10", seed=seed + 1)
    return gate["x"], gate, up


def interleaved_dev(w, gate, up):
    return tuple(w.interleave_gate_up(dev(gate[k]), dev(up[k])) for k in ("wq", "scale", "zero"))


def oracle_swiglu_of_gemvs(oracle, x, gate, up, g):
    gy = oracle.gemv_parallel(x, gate["wq"], gate["scale"], gate["zero"], g)
    uy = oracle.gemv_parallel(x, up["wq"], up["scale"], up["zero"], g)
    return oracle.swiglu(oracle.bf16_round(gy), oracle.bf16_round(uy))


def bf16_f64(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def check_swiglu(got_bits, ref_bits, what):
    # the GPU's gate and up sums differ from the oracle's exact ones by fp32
    # rounding, which can move a bf16 rounding of gate, up or h by one unit:
    # the output is held to the GEMV tolerance
    got, ref = bf16_f64(got_bits), bf16_f64(ref_bits)
    assert np.all(np.isfinite(got)), what
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2, "%s rel_l2=%.3e" % (what, rel)
    assert np.abs(got - ref).max() <= MAX_REL * np.abs(ref).max(), what


@pytest.mark.parametrize("M,I,K,g", [(1, 64, 1024, 128), (1, 4096, 4096, 128), (1, 14336, 4096, 128),
                                     (2, 136, 2048, 128), (3, 200, 1536, 128), (4, 1024, 4096, 128),
                                     (8, 512, 4096, 128), (16, 256, 2048, 128), (2, 64, 2048, 256),
                                     (5, 40, 4096, 256), (16, 4096, 4096, 128), (11, 4096, 8192, 128)])
def test_swiglu_output_matches_oracle(w, oracle, M, I, K, g):
    x, gate, up = gate_up_problem(M, I, K, g, 8100 + M * 7 + I)
    wq, s, z = interleaved_dev(w, gate, up)
    h = w.w4a16_gemv(dev(x), wq, s, z, g, swiglu_output=True)
    torch.cuda.synchronize()
    assert tuple(h.shape) == (M, I)
    got = h.view(torch.int16).cpu().numpy().view(np.uint16)
    check_swiglu(got, oracle_swiglu_of_gemvs(oracle, x, gate, up, g), "M=%d I=%d K=%d g=%d" % (M, I, K, g))
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M", [1, 2, 8, 16])
@pytest.mark.parametrize("static", [False, True])
def test_fused_equals_gemv_then_swiglu(w, M, static):
    # the same interleaved weights through the plain GEMV, then w4a16_swiglu
    # on its gate and up rows: the same fp32 sums reach the same roundings
    I, K = 1024, 2048
    x, gate, up = gate_up_problem(M, I, K, 128, 8200 + M)
    wq, s, z = interleaved_dev(w, gate, up)
    xd = dev(x)
    fused = w.w4a16_gemv(xd, wq, s, z, 128, swiglu_output=True, weights_static=static)
    plain = w.w4a16_gemv(xd, wq, s, z, 128).view(M, I // 8, 2, 8)
    h = w.w4a16_swiglu(plain[:, :, 0, :].reshape(M, I), plain[:, :, 1, :].reshape(M, I))
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), h.view(torch.int16))


def test_interleave_gate_up_layout(w):
    gate = torch.arange(16 * 3).reshape(16, 3)
    up = -torch.arange(16 * 3).reshape(16, 3) - 1
    both = w.interleave_gate_up(gate, up)
    assert both.shape == (32, 3)
    assert torch.equal(both[0:8], gate[0:8]) and torch.equal(both[8:16], up[0:8])
    assert torch.equal(both[16:24], gate[8:16]) and torch.equal(both[24:32], up[8:16])


def test_swiglu_output_refusals(w):
    x, gate, up = gate_up_problem(1, 64, 1024, 64, 8400)
    wq, s, z = interleaved_dev(w, gate, up)
    # one token with 64-wide groups runs the CUDA-core kernel, which has no
    # SwiGLU epilogue: refused, not computed some other way
    with pytest.raises(w.W4A16Error) as ei:
        w.w4a16_gemv(dev(x), wq, s, z, 64, swiglu_output=True)
    assert ei.value.status == w.Status.ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        w.w4a16_gemv(dev(x), wq, s, z, 64, swiglu_output=True, kernel_id=2)
    # rows not a multiple of 16: no whole gate/up blocks
    p = synth.dense_problem(1, 40, 1024, 128, "const8", seed=8401)
    xd, wq, s, z = dense_dev(p)
    with pytest.raises(w.W4A16Error) as ei:
        w.w4a16_gemv(xd, wq, s, z, 128, swiglu_output=True)
    assert ei.value.status == w.Status.ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [1, 8])
def test_fused_mlp_chain_with_no_cluster_down(w, oracle, M):
    # the decode MLP as the benchmark chains it: gate/up GEMV with the SwiGLU
    # epilogue, then the down GEMV planned without a cluster
    I, H = 1024, 4096
    x, gate, up = gate_up_problem(M, I, H, 128, 8500 + M)
    down = synth.dense_problem(M, H, I, 128, "uniform6to10", seed=8510 + M)
    wq, s, z = interleaved_dev(w, gate, up)
    h = w.w4a16_gemv(dev(x), wq, s, z, 128, swiglu_output=True, weights_static=True)
    y = w.w4a16_gemv(h, dev(down["wq"]), dev(down["scale"]), dev(down["zero"]), 128,
                     out_dtype=torch.float32, weights_static=True, no_cluster=True)
    torch.cuda.synchronize()
    h_ref = oracle_swiglu_of_gemvs(oracle, x, gate, up, 128)
    check_swiglu(h.view(torch.int16).cpu().numpy().view(np.uint16), h_ref, "chain h M=%d" % M)
    # the down product of the GPU's own h (its bf16 values are the input)
    h_bits = h.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemv_parallel(h_bits, down["wq"], down["scale"], down["zero"], 128)
    got = y.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2 and np.abs(got - ref).max() <= MAX_REL * np.abs(ref).max(), rel
    assert w.w4a16_device_error(clear=True) == 0
