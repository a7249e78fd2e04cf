"""GPU parity of the tensor-core (tcgen05) GEMV kernel, forced through the C ABI.

Same bar as the other GEMV kernels: relative L2 error <= 5e-3 and
max |err| <= 1e-2 * max |y_ref| against the oracle's fp64 result, and
bit-exact bf16 output when every output has a single nonzero product.
Shapes cover one-block and odd-block K slices, ragged N (rows beyond the last
128-row tile), every token-count class (1, 2, 4, 8, 16 columns read back) and
forced cluster K splits, including splits that leave ranks one block.
"""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

from .test_gpu_parity import check_close, dense_dev, dev, host_f64

pytestmark = pytest.mark.gpu

TC = 3


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding
    binding.w4a16_device_error(clear=True)
    return binding


CASES = [
    # M, N, K, g
    (1, 256, 512, 128),
    (1, 300, 1024, 128),    # ragged N: 3 tiles, last one 44 rows
    (1, 1, 128, 128),       # one row, one block
    (1, 128, 384, 128),     # odd block count (3)
    (2, 130, 2304, 128),    # 18 blocks
    (3, 64, 4096, 128),
    (4, 200, 2304, 256),    # groups of two blocks
    (5, 129, 1152, 128),    # 9 blocks, 2 tiles
    (8, 512, 4096, 128),
    (9, 45, 1024, 128),     # first 16-token class
    (12, 257, 2048, 128),
    (16, 150, 2048, 128),
    (16, 15, 1024, 256),
]


@pytest.mark.parametrize("M,N,K,g", CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tensor_core_gemv_matches_oracle(w, oracle, M, N, K, g, out_dtype):
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=7000 + M * 100 + N)
    y = w.w4a16_gemv(*dense_dev(p), g, out_dtype=out_dtype, kernel_id=TC)
    torch.cuda.synchronize()
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    check_close(host_f64(y), ref, "tc M=%d N=%d K=%d g=%d" % (M, N, K, g))
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M,N,K", [(1, 384, 4096), (2, 256, 3072), (8, 130, 14336), (16, 200, 2048),
                                   (4, 128, 1024)])
@pytest.mark.parametrize("k_split", [1, 2, 4, 8])
def test_tensor_core_forced_cluster_split(w, oracle, M, N, K, k_split):
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7100 + k_split)
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    nblk = K // 128
    bpc = -(-nblk // k_split)
    bpc += bpc & 1
    ntok = 8 if M <= 8 else 16
    if (k_split > 1 and (k_split - 1) * bpc >= nblk) or bpc * 16 * ntok * 16 > 190 * 1024:
        # a rank would get no block, or one CTA's activation slice does not
        # fit in shared memory: the planner refuses the split
        with pytest.raises(w.W4A16Error) as ei:
            w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=TC, k_split=k_split)
        assert ei.value.status == w.Status.ERR_UNSUPPORTED
        return
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=TC, k_split=k_split)
    torch.cuda.synchronize()
    check_close(host_f64(y), ref, "tc split %d" % k_split)
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M", [1, 2, 7, 16])
def test_tensor_core_one_hot_is_bit_exact(w, oracle, M):
    # one nonzero product per output: D = (128 + q) exactly, folded to
    # s * (q - z) exactly in fp32, so the bf16 output is RNE_bf16(W[n][k0])
    N, K, g = 200, 2048, 128
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=7200)
    W = oracle.dequant(p["wq"], p["scale"], p["zero"], g)
    ks = [0, 7, 129, 555, 1023, 64, 300, 999, 1, 2, 3, 4, 5, 2047, 8, 9][:M]
    x = np.zeros((M, K), np.uint16)
    for m, k0 in enumerate(ks):
        x[m, k0] = 0x3F80
    y = w.w4a16_gemv(dev(x), dev(p["wq"]), dev(p["scale"]), dev(p["zero"]), g, kernel_id=TC)
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    for m, k0 in enumerate(ks):
        assert np.array_equal(got[m], oracle.bf16_round(W[:, k0])), (m, k0)


def test_tensor_core_is_deterministic_and_stream_ordered(w):
    p = synth.dense_problem(4, 1000, 4096, 128, "uniform6to10", seed=7300)
    args = dense_dev(p)
    outs = [w.w4a16_gemv(*args, 128, out_dtype=torch.float32, kernel_id=TC) for _ in range(4)]
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


FULL = [("square", 1, 4096, 4096), ("vocab", 1, 163840, 4096)] + \
    [("up", M, 14336, 4096) for M in (1, 2, 8, 16)] + [("down", M, 4096, 14336) for M in (1, 4, 16)]


@pytest.mark.parametrize("name,M,N,K", FULL, ids=["%s-M%d" % (f[0], f[1]) for f in FULL])
def test_tensor_core_full_size_every_output(w, oracle, name, M, N, K):
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=1)
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.bfloat16, kernel_id=TC)
    torch.cuda.synchronize()
    ref = oracle.gemv_parallel(p["x"], p["wq"], p["scale"], p["zero"], 128)
    check_close(host_f64(y), ref, name)
    assert w.w4a16_device_error(clear=True) == 0
