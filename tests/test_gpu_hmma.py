"""Parity of the fp16 warp-MMA GEMV (kernel 4) with the oracle, through the C
ABI: ragged row counts, token counts 1..16 (9..16 as two 8-token MMA tiles),
K from one 512-k unit to the
wide-MLP down projection, cluster K splits, both output types, the
resident-weights flag, dependent launches, determinism, activations across
the bf16 range (the kernel scales each 128-k block by a power of two), and
one-hot activations (a single product per output, so the result is exact).
Bar: relative L2 <= 5e-3 and max |err| <= 1e-2 * max |y_ref| against the
unrounded fp64 oracle."""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

from .test_gpu_parity import check_close, dense_dev, dev, host_f64

pytestmark = pytest.mark.gpu

KID = 4


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
    # M, N, K
    (1, 1, 512),        # one row, one unit
    (1, 15, 1024),      # less than one tile
    (1, 17, 512),       # one tile plus one row
    (1, 300, 3072),     # ragged tiles, K of six units
    (1, 4096, 4096),    # square projection
    (2, 257, 2048),
    (3, 130, 1536),
    (4, 200, 4096),
    (5, 33, 2560),
    (6, 64, 1024),
    (7, 91, 512),
    (8, 150, 4096),
    (1, 64, 14336),     # wide-MLP down-projection K
    (2, 40, 14336),
    (9, 77, 1024),      # two MMA tiles, the second with one token
    (12, 130, 2048),
    (13, 17, 512),
    (16, 200, 4096),
    (16, 33, 14336),
]


@pytest.mark.parametrize("M,N,K", CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_hmma_matches_oracle(w, oracle, M, N, K, out_dtype):
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7000 + M * 131 + N)
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=out_dtype, kernel_id=KID)
    torch.cuda.synchronize()
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    check_close(host_f64(y), ref, "kernel 4 M=%d N=%d K=%d" % (M, N, K))
    assert w.w4a16_device_error(clear=True) == 0


# shapes whose plan is a 16-warp CTA alone on its SM (long runs), one per
# instantiated token count; the rest of this file runs 8-warp pairs
WIDE = [(1, 28672, 4096), (2, 6000, 14336), (3, 28672, 4096), (8, 12000, 4096), (16, 12000, 4096)]


@pytest.mark.parametrize("M,N,K", WIDE)
def test_hmma_wide_ctas_match_oracle(w, oracle, M, N, K):
    if M == 1:  # the library's own choice for one token: kernel 4, 16 warps
        plan = w.gemv_plan(M, N, K, 128)
        assert (plan["kernel_id"], plan["threads"]) == (KID, 512)
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7050 + M)
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=KID)
    torch.cuda.synchronize()
    ref = oracle.gemv_parallel(p["x"], p["wq"], p["scale"], p["zero"], 128)
    check_close(host_f64(y), ref, "kernel 4, 16 warps, M=%d N=%d K=%d" % (M, N, K))
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M,N,K", [(1, 64, 4096), (3, 48, 4096), (1, 40, 14336), (8, 33, 8192),
                                   (2, 4096, 4096), (16, 48, 4096), (11, 300, 8192)])
@pytest.mark.parametrize("split", [1, 2, 4, 8])
def test_hmma_cluster_k_split(w, oracle, M, N, K, split):
    # K split over the CTAs of a cluster (partials pushed to the owner's
    # shared memory); a split that does not divide K / 512 is refused
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7100 + split)
    if (K // 512) % split != 0:
        with pytest.raises(w.W4A16Error) as ei:
            w.w4a16_gemv(*dense_dev(p), 128, kernel_id=KID, k_split=split)
        assert ei.value.status == w.Status.ERR_UNSUPPORTED
        return
    if M > 8 and K // split >= 4096:
        # 16 tokens' fp16 fragments of a 4096-k slice (128 KB) plus the
        # rings need more shared memory than a CTA has: refused, not run
        try:
            w.w4a16_gemv(*dense_dev(p), 128, kernel_id=KID, k_split=split)
        except w.W4A16Error as e:
            assert e.status == w.Status.ERR_UNSUPPORTED
            return
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=KID, k_split=split)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128),
                "split %d" % split)
    assert w.w4a16_device_error(clear=True) == 0


def test_hmma_refuses_unsupported_shapes(w):
    # nine tokens, groups other than 128, K not a multiple of 512
    for M, K, g in ((17, 1024, 128), (1, 1024, 64), (1, 1024, 256), (1, 768, 128)):
        p = synth.dense_problem(M, 32, K, g, "const8", seed=7200)
        with pytest.raises(w.W4A16Error) as ei:
            w.w4a16_gemv(*dense_dev(p), g, kernel_id=KID)
        assert ei.value.status == w.Status.ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_hmma_one_hot_is_bit_exact(w, oracle, M):
    # x = e_k0 per token: D - c1 - z c2 = (q - z) x' exactly, so y is
    # RNE_bf16(W[n][k0]) bit for bit -- at even and odd code positions
    N, K = 48, 2048
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7300)
    W = oracle.dequant(p["wq"], p["scale"], p["zero"], 128)
    ks = [0, 1, 7, 130, 1023, 1500, 2046, 2047, 3, 64, 511, 512, 777, 1024, 1999, 2040][:M]
    x = np.zeros((M, K), np.uint16)
    for m, k0 in enumerate(ks):
        x[m, k0] = 0x3F80
    y = w.w4a16_gemv(dev(x), dev(p["wq"]), dev(p["scale"]), dev(p["zero"]), 128, kernel_id=KID)
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    for m, k0 in enumerate(ks):
        assert np.array_equal(got[m], oracle.bf16_round(W[:, k0])), (m, k0)


@pytest.mark.parametrize("lo,hi", [(-40, 29), (-126, -100), (60, 120), (-100, 100), (30, 50)])
def test_hmma_activation_range(w, oracle, lo, hi):
    # magnitudes 2^lo .. 2^hi (bf16 covers 2^-133 .. 2^127): every 128-k block
    # of a token is scaled by its own power of two into the fp16 range, so
    # large |x| do not overflow and small ones are exact down to 2^-24 of the
    # block's largest
    M, N, K = 2, 64, 2048
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7400 + lo)
    r = synth.rng(7400 + hi, "misc")
    mag = np.ldexp(1.0, r.integers(lo, hi + 1, size=(M, K))) * r.choice([-1.0, 1.0], size=(M, K))
    p["x"] = synth.f32_to_bf16_bits(mag.astype(np.float32))
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    assert np.all(np.isfinite(ref))
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=KID)
    torch.cuda.synchronize()
    check_close(host_f64(y), ref, "range 2^%d..2^%d" % (lo, hi))


def test_hmma_zero_activations(w):
    p = synth.dense_problem(3, 40, 1024, 128, "uniform6to10", seed=7500)
    p["x"][:] = 0
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=KID)
    assert torch.count_nonzero(y).item() == 0


@pytest.mark.parametrize("N", [4096, 28672])
def test_hmma_weights_static_flag(w, oracle, N):
    # the flag only moves the weight copies ahead of the grid-dependency wait
    # (the library's own choice, kernel 4 for one token: 8- and 16-warp CTAs)
    assert w.gemv_plan(1, N, 4096, 128)["kernel_id"] == KID
    p = synth.dense_problem(1, N, 4096, 128, "uniform6to10", seed=7600)
    args = dense_dev(p)
    a = w.w4a16_gemv(*args, 128, out_dtype=torch.float32)
    b = w.w4a16_gemv(*args, 128, out_dtype=torch.float32, weights_static=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check_close(host_f64(b), oracle.gemv_parallel(p["x"], p["wq"], p["scale"], p["zero"], 128), "static")


@pytest.mark.parametrize("static", [False, True])
def test_hmma_dependent_chain(w, static):
    # y of one GEMV is x of the next, launched back to back (programmatic
    # dependent launch, two CTAs per SM): equal to the same chain with a host
    # synchronisation between the calls
    K = 4096
    layers = [synth.dense_problem(1, K, K, 128, "uniform6to10", seed=7700 + i) for i in range(8)]
    devs = [dense_dev(p) for p in layers]
    x0 = devs[0][0]
    outs = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for _ in layers]
    for _ in range(3):
        cur = x0
        for (_, wq, s, z), o in zip(devs, outs):
            w.w4a16_gemv(cur, wq, s, z, 128, out=o, weights_static=static)
            cur = o
    torch.cuda.synchronize()
    chained = outs[-1].clone()
    cur = x0
    for (_, wq, s, z), o in zip(devs, outs):
        o.zero_()
        torch.cuda.synchronize()
        w.w4a16_gemv(cur, wq, s, z, 128, out=o)
        torch.cuda.synchronize()
        cur = o
    assert torch.equal(chained, outs[-1])
    assert w.w4a16_device_error(clear=True) == 0


def test_hmma_is_deterministic(w):
    p = synth.dense_problem(5, 1000, 4096, 128, "uniform6to10", seed=7800)
    args = dense_dev(p)
    outs = [w.w4a16_gemv(*args, 128, out_dtype=torch.float32, kernel_id=KID) for _ in range(3)]
    s2 = [w.w4a16_gemv(*args, 128, out_dtype=torch.float32, kernel_id=KID, k_split=2) for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert torch.equal(s2[0], s2[1])


@pytest.mark.parametrize("M,N,K", [(1, 4096, 14336), (4, 4096, 14336), (2, 8192, 8192), (1, 1024, 8192),
                                   (1, 4096, 4096)])
def test_no_cluster_flag_matches_oracle(w, oracle, M, N, K):
    # the default plans of the first four use a cluster K split; with the
    # flag the K split stays inside the CTA (and the 4096 x 4096 plan, which
    # has no cluster, is unchanged); results within the bar either way
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=7600 + M)
    args = dense_dev(p)
    y = w.w4a16_gemv(*args, 128, out_dtype=torch.float32, no_cluster=True)
    y0 = w.w4a16_gemv(*args, 128, out_dtype=torch.float32)
    ys = w.w4a16_gemv(*args, 128, out_dtype=torch.float32, no_cluster=True, weights_static=True)
    torch.cuda.synchronize()
    ref = oracle.gemv_parallel(p["x"], p["wq"], p["scale"], p["zero"], 128)
    check_close(host_f64(y), ref, "no-cluster M=%d N=%d K=%d" % (M, N, K))
    check_close(host_f64(ys), ref, "no-cluster static M=%d N=%d K=%d" % (M, N, K))
    assert torch.equal(y, ys)
    if w.gemv_plan(M, N, K, 128)["k_split"] == 1:
        assert torch.equal(y, y0)  # no cluster to remove: the same launch
    assert w.w4a16_device_error(clear=True) == 0
