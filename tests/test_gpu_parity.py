"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer work (packing, dequantisation to bf16/fp32) must be bit-exact.  GEMV
outputs must satisfy the stated tolerance: relative L2 error <= 5e-3 and
max |err| <= 1e-2 * max |y_ref|, against the oracle's unrounded fp64 result.
Full-size workloads are checked on every output element, in the same launch
configuration the benchmark uses (the library's default dispatch).
"""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
MAX_REL = 1e-2


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding
    binding.w4a16_device_error(clear=True)
    return binding


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def host_f64(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def check_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), what
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max()
    assert rel <= REL_L2, "%s rel_l2=%.3e" % (what, rel)
    assert mx <= MAX_REL * np.abs(ref).max(), "%s max_err=%.3e max_ref=%.3e" % (what, mx, np.abs(ref).max())
    return rel, mx


def dense_dev(p):
    return dev(p["x"]), dev(p["wq"]), dev(p["scale"]), dev(p["zero"])


# ---- packing and dequantisation (bit-exact) ------------------------------

@pytest.mark.parametrize("N,K", [(1, 8), (3, 24), (256, 512), (77, 4096), (1024, 2304)])
def test_int4_pack_bit_exact(w, oracle, N, K):
    codes = synth.codes(21, N, K)
    got = w.int4_pack(dev(codes))
    torch.cuda.synchronize()
    want = oracle.pack(codes)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want)


def test_int4_pack_ignores_high_bits(w, oracle):
    codes = synth.codes(22, 16, 64) | np.uint8(0xF0)
    got = w.int4_pack(dev(codes)).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, oracle.pack(codes & 0x0F))


@pytest.mark.parametrize("N,K,g,zmode", [(256, 512, 128, "const8"), (33, 1024, 32, "uniform6to10"),
                                         (64, 4096, 128, "uniform6to10"), (5, 768, 256, "uniform6to10")])
def test_int4_dequant_bit_exact(w, oracle, N, K, g, zmode):
    p = synth.dense_problem(1, N, K, g, zmode, seed=23)
    wq, s, z = dev(p["wq"]), dev(p["scale"]), dev(p["zero"])
    exact = oracle.dequant(p["wq"], p["scale"], p["zero"], g)
    w32 = w.int4_dequant(wq, s, z, g, out_dtype=torch.float32)
    wbf = w.int4_dequant(wq, s, z, g, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert np.array_equal(w32.cpu().numpy().astype(np.float64), exact)
    assert np.array_equal(wbf.view(torch.int16).cpu().numpy().view(np.uint16), oracle.bf16_round(exact))


def test_int4_dequant_extreme_zero_points(w, oracle):
    # zero points up to 255 and large/small scales still give exact products
    N, K, g = 16, 256, 128
    wq = synth.packed_weights(24, N, K)
    z = synth.rng(24, "zero").integers(0, 256, size=(N, K // g), dtype=np.uint8)
    s = synth.f32_to_bf16_bits(np.ldexp(1.0, synth.rng(24, "scale").integers(-60, 60, size=(N, K // g))).astype(np.float32))
    exact = oracle.dequant(wq, s, z, g)
    got = w.int4_dequant(dev(wq), dev(s), dev(z), g, out_dtype=torch.float32)
    assert np.array_equal(got.cpu().numpy().astype(np.float64), exact)


# ---- dense GEMV ----------------------------------------------------------

GEMV_CASES = [
    # M, N, K, g, zero mode
    (1, 256, 512, 128, "const8"),          # tiny workload
    (1, 300, 1024, 128, "uniform6to10"),   # ragged N (not a multiple of 8 or 16)
    (1, 17, 2048, 64, "uniform6to10"),
    (1, 1, 32, 32, "uniform6to10"),        # smallest shape
    (1, 40, 3072, 32, "uniform6to10"),     # 3 spans of 32 chunks, per-chunk groups
    (1, 96, 1056, 96, "uniform6to10"),     # K not a multiple of 1024, g = 96
    (1, 64, 2048, 256, "uniform6to10"),
    (2, 256, 512, 128, "const8"),
    (3, 130, 1024, 128, "uniform6to10"),
    (4, 200, 2304, 128, "uniform6to10"),
    (8, 64, 4096, 128, "uniform6to10"),
    (9, 45, 1024, 128, "uniform6to10"),
    (16, 150, 2048, 128, "uniform6to10"),
    (16, 15, 1024, 256, "uniform6to10"),
]


@pytest.mark.parametrize("M,N,K,g,zmode", GEMV_CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_gemv_matches_oracle(w, oracle, M, N, K, g, zmode, out_dtype):
    p = synth.dense_problem(M, N, K, g, zmode, seed=M * 1000 + N)
    y = w.w4a16_gemv(*dense_dev(p), g, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    check_close(host_f64(y), ref, "M=%d N=%d K=%d g=%d" % (M, N, K, g))


@pytest.mark.parametrize("M,N,K", [(1, 64, 4096), (1, 48, 3072), (1, 40, 14336), (3, 64, 4096),
                                   (12, 40, 2048), (16, 72, 14336)])
@pytest.mark.parametrize("k_split", [1, 2, 4, 8, 16, 32])
def test_gemv_forced_k_split(w, oracle, M, N, K, k_split):
    # in-CTA (named barrier) and cluster (DSMEM) K splits, including more
    # parts than the K range has units (some warps or CTAs get no work)
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=31 + k_split)
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    if M * K * 2 > 200 * 1024 * k_split:
        # the activation slice of one CTA cannot fit in shared memory
        with pytest.raises(w.W4A16Error) as ei:
            w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, k_split=k_split)
        assert ei.value.status == w.Status.ERR_UNSUPPORTED
        return
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, k_split=k_split)
    torch.cuda.synchronize()
    check_close(host_f64(y), ref, "split %d" % k_split)


@pytest.mark.parametrize("M", [1, 2, 5])
def test_gemv_kernels_agree_on_m1_and_variants(w, oracle, M):
    # both kernels serve M <= 2 when forced; both meet the bar
    p = synth.dense_problem(M, 96, 2048, 128, "uniform6to10", seed=41)
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128)
    ids = (1, 2) if M <= 2 else (2,)
    for kid in ids:
        y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=torch.float32, kernel_id=kid)
        torch.cuda.synchronize()
        check_close(host_f64(y), ref, "kernel %d" % kid)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gemv_one_hot_is_bit_exact(w, oracle, M):
    # x = e_k0 in every token: one nonzero product per output, so the GPU
    # result must be exactly RNE_bf16(W[n][k0])
    N, K, g = 64, 1024, 128
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=43)
    W = oracle.dequant(p["wq"], p["scale"], p["zero"], g)
    ks = [0, 7, 129, 555, 1023, 64, 300, 999, 1, 2, 3, 4, 5, 6, 8, 9][:M]
    x = np.zeros((M, K), np.uint16)
    for m, k0 in enumerate(ks):
        x[m, k0] = 0x3F80
    y = w.w4a16_gemv(dev(x), dev(p["wq"]), dev(p["scale"]), dev(p["zero"]), g)
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    for m, k0 in enumerate(ks):
        assert np.array_equal(got[m], oracle.bf16_round(W[:, k0])), (m, k0)


@pytest.mark.parametrize("M,N,K,g", [(2, 300, 1024, 128), (2, 77, 3072, 32), (2, 4096, 4096, 128),
                                     (2, 40, 14336, 128)])
def test_gemv_cuda_core_two_tokens(w, oracle, M, N, K, g):
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=N + K)
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    for k_split in (0, 2, 16):
        y = w.w4a16_gemv(*dense_dev(p), g, out_dtype=torch.float32, kernel_id=1, k_split=k_split)
        torch.cuda.synchronize()
        check_close(host_f64(y), ref, "cuda-core M=2 split %d" % k_split)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_gemv_weights_static_flag(w, oracle, M):
    # the flag only moves weight loads ahead of the grid-dependency wait
    p = synth.dense_problem(M, 512, 4096, 128, "uniform6to10", seed=55)
    args = dense_dev(p)
    a = w.w4a16_gemv(*args, 128, out_dtype=torch.float32)
    b = w.w4a16_gemv(*args, 128, out_dtype=torch.float32, weights_static=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check_close(host_f64(b), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128), "static")


@pytest.mark.parametrize("static", [False, True])
def test_gemv_chain_keeps_stream_order(w, static):
    # back-to-back dependent GEMVs (y of one is x of the next) launched with
    # programmatic dependent launch must equal the same chain with a host
    # synchronisation between the calls
    K = 4096
    layers = [synth.dense_problem(1, K, K, 128, "uniform6to10", seed=60 + i) for i in range(6)]
    devs = [dense_dev(p) for p in layers]
    x0 = devs[0][0]
    outs = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for _ in layers]
    for _ in range(3):
        cur = x0
        for (xx, wq, s, z), o in zip(devs, outs):
            w.w4a16_gemv(cur, wq, s, z, 128, out=o, weights_static=static)
            cur = o
    torch.cuda.synchronize()
    chained = outs[-1].clone()
    cur = x0
    for (xx, wq, s, z), o in zip(devs, outs):
        o.zero_()
        torch.cuda.synchronize()
        w.w4a16_gemv(cur, wq, s, z, 128, out=o)
        torch.cuda.synchronize()
        cur = o
    assert torch.equal(chained, outs[-1])


def test_gemv_is_deterministic(w):
    p = synth.dense_problem(4, 512, 4096, 128, "uniform6to10", seed=45)
    args = dense_dev(p)
    a = w.w4a16_gemv(*args, 128, out_dtype=torch.float32)
    b = w.w4a16_gemv(*args, 128, out_dtype=torch.float32, k_split=16)
    c = w.w4a16_gemv(*args, 128, out_dtype=torch.float32, k_split=16)
    d = w.w4a16_gemv(*args, 128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a, d) and torch.equal(b, c)


def test_gemv_large_activation_range(w, oracle):
    # activations spanning many binades (still |x| < 2^40)
    M, N, K, g = 1, 64, 1024, 128
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=47)
    r = synth.rng(47, "misc")
    mag = np.ldexp(1.0, r.integers(-40, 30, size=(M, K))) * r.choice([-1.0, 1.0], size=(M, K))
    p["x"] = synth.f32_to_bf16_bits(mag.astype(np.float32))
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], g)
    y = w.w4a16_gemv(*dense_dev(p), g, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_close(host_f64(y), ref, "wide range")


def _range_problem(seed, lo, hi, M=1, N=64, K=1024, g=64):
    # one token with 64-wide groups: the CUDA-core kernel; |x| = 2^e, e
    # uniform in [lo, hi], random signs
    p = synth.dense_problem(M, N, K, g, "uniform6to10", seed=seed)
    r = synth.rng(seed, "misc")
    mag = np.ldexp(1.0, r.integers(lo, hi + 1, size=(M, K))) * r.choice([-1.0, 1.0], size=(M, K))
    p["x"] = synth.f32_to_bf16_bits(mag.astype(np.float32))
    return p


def test_cuda_core_kernel_input_range_edges(w, oracle):
    # the CUDA-core kernel (groups finer than 128) stages x * 2^(85 - p): it
    # is exact up to |x| < 2^43 and flags anything larger.  At the edge:
    # magnitudes up to the largest bf16 below 2^43, no flag, within tolerance
    assert w.gemv_plan(1, 64, 1024, 64)["kernel_id"] == 1
    w.w4a16_device_error(clear=True)
    p = _range_problem(51, 20, 42)
    p["x"][0, :4] = [0x54FF, 0xD4FF, 0x54FF, 0xD4FF]  # +-(2^43 - 2^35)
    y = w.w4a16_gemv(*dense_dev(p), 64, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert w.w4a16_device_error(clear=True) == 0
    check_close(host_f64(y), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 64), "x < 2^43")
    # beyond it: one 2^43 flags W4A16_DEVERR_RANGE; at a k that is a
    # multiple of 8 (the lowest nibble, staged times 2^85) it overflows
    p["x"][0, 96] = 0x5500
    y = w.w4a16_gemv(*dense_dev(p), 64, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert w.w4a16_device_error(clear=True) & w.DEVERR_RANGE
    assert not np.all(np.isfinite(host_f64(y)))


def test_cuda_core_kernel_small_activations(w, oracle):
    # products |code * x| >= 2^-62 are exact: activations down to 2^-58
    # meet the tolerance
    p = _range_problem(52, -58, -40)
    y = w.w4a16_gemv(*dense_dev(p), 64, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 64), "x >= 2^-58")
    # below that, products and chunk sums round to fp32's subnormal grid
    # (2^-149, restored by 2^64): each output is off by at most
    # (K + K / 32) * 2^-150 * 2^64 * max scale * max |code - zero| -- here
    # that bound, not the relative tolerance, holds
    p = _range_problem(53, -100, -90)
    y = host_f64(w.w4a16_gemv(*dense_dev(p), 64, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert w.w4a16_device_error(clear=True) == 0
    ref = oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 64)
    smax = synth.bf16_bits_to_f32(p["scale"]).max()
    bound = (1024 + 1024 / 32) * 2.0 ** -86 * smax * 16
    assert np.abs(y - ref).max() <= bound, (np.abs(y - ref).max(), bound)


def test_gemv_default_dispatch_is_pinned(w):
    # the dispatch the benchmark times is the library default; pin it: the
    # fp16 warp-MMA kernel for one and two tokens on the square, wide-MLP and
    # vocabulary shapes, for three and four tokens on matrices of 2^24
    # weights or more, and for 3..16 tokens on matrices of 2^25 weights or
    # more that it has a plan for, the bf16 warp-MMA kernel for 3..16 tokens
    # on smaller matrices, for 9..16 tokens where kernel 4 has no plan, and
    # for one token where kernel 4 does not apply (groups of 256,
    # K % 512 != 0), the CUDA-core kernel for one or two tokens with groups
    # of 64
    for M in (1, 2):
        for N, K in ((4096, 4096), (14336, 4096), (4096, 14336), (163840, 4096)):
            assert w.gemv_plan(M, N, K, 128)["kernel_id"] == 4
    for M in (3, 4, 8):
        for N, K in ((14336, 4096), (4096, 14336), (8192, 4096)):
            assert w.gemv_plan(M, N, K, 128)["kernel_id"] == 4
        assert w.gemv_plan(M, 4096, 4096, 128)["kernel_id"] == (4 if M <= 4 else 2)
        assert w.gemv_plan(M, 6144, 4096, 128)["kernel_id"] == (4 if M <= 4 else 2)
        assert w.gemv_plan(M, 2048, 4096, 128)["kernel_id"] == 2
        assert w.gemv_plan(M, 8191, 4096, 128)["kernel_id"] == (4 if M <= 4 else 2)
    for M in (9, 16):
        assert w.gemv_plan(M, 14336, 4096, 128)["kernel_id"] == 4
        assert w.gemv_plan(M, 8192, 8192, 128)["kernel_id"] == 4
        assert w.gemv_plan(M, 4096, 14336, 128)["kernel_id"] == 2  # 16 tokens' fragments do not fit
        assert w.gemv_plan(M, 4096, 4096, 128)["kernel_id"] == 2
    assert w.gemv_plan(1, 4096, 4096, 256)["kernel_id"] == 2
    assert w.gemv_plan(1, 4096, 2304, 128)["kernel_id"] == 2
    assert w.gemv_plan(1, 4096, 4096, 64)["kernel_id"] == 1
    assert w.gemv_plan(2, 4096, 4096, 64)["kernel_id"] == 1
    # forcing the planned kernel (its own split) reproduces the default launch;
    # for the CUDA-core and bf16 warp-MMA kernels so does forcing the reported
    # split factor (warps per tile x CTAs per cluster)
    for M, g in ((1, 128), (4, 128), (1, 64)):
        p = synth.dense_problem(M, 512, 4096, g, "const8", seed=49)
        args = dense_dev(p)
        plan = w.gemv_plan(M, 512, 4096, g)
        a = w.w4a16_gemv(*args, g, out_dtype=torch.float32)
        b = w.w4a16_gemv(*args, g, out_dtype=torch.float32, kernel_id=plan["kernel_id"])
        torch.cuda.synchronize()
        assert torch.equal(a, b), (M, g, plan)
        if plan["kernel_id"] in (1, 2):
            c = w.w4a16_gemv(*args, g, out_dtype=torch.float32, kernel_id=plan["kernel_id"],
                             k_split=plan["k_split"])
            torch.cuda.synchronize()
            assert torch.equal(a, c), (M, g, plan)


# ---- full-size workloads, every output ------------------------------------

FULL = [
    ("square", 1, 4096, 4096, "const8", torch.bfloat16),
    ("vocab", 1, 163840, 4096, "uniform6to10", torch.float32),
] + [("up", M, 14336, 4096, "uniform6to10", torch.bfloat16) for M in (1, 2, 4, 8, 16)] + \
    [("down", M, 4096, 14336, "uniform6to10", torch.bfloat16) for M in (1, 2, 4, 8, 16)]


@pytest.mark.parametrize("name,M,N,K,zmode,out_dtype", FULL, ids=["%s-M%d" % (f[0], f[1]) for f in FULL])
@pytest.mark.parametrize("static", [False, True])
def test_full_size_every_output(w, oracle, name, M, N, K, zmode, out_dtype, static):
    # the launch the benchmark times (library default dispatch, with and
    # without the resident-weights flag), compared element by element with the
    # oracle over the whole output (its rows computed on all host threads)
    p = synth.dense_problem(M, N, K, 128, zmode, seed=0)
    y = w.w4a16_gemv(*dense_dev(p), 128, out_dtype=out_dtype, weights_static=static)
    torch.cuda.synchronize()
    ref = _full_reference(oracle, name, M, p)
    check_close(host_f64(y), ref, name)
    assert w.w4a16_device_error(clear=True) == 0


_REF_CACHE = {}


def _full_reference(oracle, name, M, p):
    key = (name, M)
    if key not in _REF_CACHE:
        _REF_CACHE.clear()
        _REF_CACHE[key] = oracle.gemv_parallel(p["x"], p["wq"], p["scale"], p["zero"], 128)
    return _REF_CACHE[key]


def test_gemv_with_page_locked_host_x_and_y(w, oracle):
    # M == 1: the kernel reads x from and writes y to page-locked host memory;
    # same kernel, same plan, so the result equals the device-buffer call bit
    # for bit (and meets the oracle bar)
    for N, K in ((4096, 4096), (300, 2304)):
        p = synth.dense_problem(1, N, K, 128, "uniform6to10", seed=9100 + N)
        x_dev, wq, s, z = dense_dev(p)
        y_dev = w.w4a16_gemv(x_dev, wq, s, z, 128)
        x_host = x_dev.cpu().pin_memory()
        y_host = torch.empty((1, N), dtype=torch.bfloat16).pin_memory()
        w.w4a16_gemv(x_host, wq, s, z, 128, out=y_host)
        torch.cuda.synchronize()
        assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
        check_close(host_f64(y_host), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128),
                    "host-resident x/y")
    assert w.w4a16_device_error(clear=True) == 0
    with pytest.raises(ValueError):   # more than one token: device buffers only
        w.w4a16_gemv(torch.zeros((2, 4096), dtype=torch.bfloat16).pin_memory(), wq, s, z, 128)


# ---- SwiGLU --------------------------------------------------------------

def test_swiglu_matches_oracle(w, oracle):
    gate = synth.activations(51, (37, 1024))
    up = synth.activations(52, (37, 1024))
    h = w.w4a16_swiglu(dev(gate).view(torch.bfloat16), dev(up).view(torch.bfloat16))
    got = h.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.swiglu(gate, up)
    gf = synth.bf16_bits_to_f32(got).astype(np.float64)
    rf = synth.bf16_bits_to_f32(ref).astype(np.float64)
    # fp32 evaluation vs fp64: at most one bf16 ulp apart, and almost always equal
    ulp = np.ldexp(1.0, np.frexp(np.abs(rf))[1] - 8)
    assert np.all(np.abs(gf - rf) <= ulp)
    assert np.mean(got != ref) < 1e-3


def test_swiglu_strided_halves(w, oracle):
    both = synth.activations(53, (6, 2 * 512))
    t = dev(both).view(torch.bfloat16)
    h = w.w4a16_swiglu(t[:, :512], t[:, 512:])
    ref = oracle.swiglu(both[:, :512], both[:, 512:])
    got = h.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.mean(got != ref) < 1e-3


# ---- mixture of experts --------------------------------------------------

def _bank_dev(bank):
    return tuple(dev(a) for a in bank)


# the library's choice (the fp16 warp-MMA expert kernel where it applies) and
# the bf16 warp-MMA expert kernel
MOE_KERNELS = [0, 2]


@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("kid", MOE_KERNELS)
def test_moe_gemv_per_slot(kid, w, oracle, M):
    E, N, K, g, topk = 16, 256, 2304, 128, 8
    wq, s, z = synth.expert_bank(61, E, N, K, g)
    ids, _ = synth.routing(61, M, topk, E)
    x = synth.activations(61, (M, K))
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid)
    torch.cuda.synchronize()
    ref = oracle.moe_gemv(x, ids, None, wq, s, z, g)
    check_close(host_f64(y), ref, "moe per slot")
    xs = synth.activations(62, (M, topk, K))
    ys = w.w4a16_moe_gemv(dev(xs), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid, x_per_slot=True)
    refs = oracle.moe_gemv(xs, ids, None, wq, s, z, g, x_per_slot=True)
    check_close(host_f64(ys), refs, "moe per slot, x per slot")


@pytest.mark.parametrize("M,N,K,g", [(1, 100, 128, 128), (3, 70, 256, 256), (2, 130, 7168, 128),
                                     (5, 40, 9216, 128), (1, 300, 4608, 256)])
@pytest.mark.parametrize("kid", MOE_KERNELS)
def test_moe_gemv_scale_table_edges(kid, w, oracle, M, N, K, g):
    # one group per row (G = 1), tables filled in several load batches
    # (G = 56 over 64 rows), no table at all (G = 72: scales read in the
    # loop), ragged row chunks
    E, topk = 6, 2
    wq, s, z = synth.expert_bank(66 + K, E, N, K, g)
    ids, r = synth.routing(66 + K, M, topk, E)
    x = synth.activations(66 + K, (M, K))
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.moe_gemv(x, ids, None, wq, s, z, g), "moe table edges")
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("kid", MOE_KERNELS)
def test_moe_gemv_shared_experts_and_many_slots(kid, w, oracle):
    # 12 tokens over 4 experts: every expert serves > 8 slots (two passes at
    # one n-tile for M <= 8 would not be enough)
    M, E, N, K, g, topk = 12, 4, 96, 1024, 128, 3
    wq, s, z = synth.expert_bank(63, E, N, K, g)
    ids, r = synth.routing(63, M, topk, E)
    x = synth.activations(63, (M, K))
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid, route_w=dev(r))
    torch.cuda.synchronize()
    ref = oracle.moe_gemv(x, ids, r, wq, s, z, g)
    check_close(host_f64(y), ref, "routed sum")


@pytest.mark.parametrize("kid", MOE_KERNELS)
def test_moe_gemv_passes_with_several_tiles_per_warp(kid, w, oracle):
    # 64 distinct experts over 8 tokens make 128-row CTAs whose warps take two
    # tiles in turn; expert 0 named twice by every token has 16 slots, so its
    # CTAs stream their weights in two passes
    M, E, N, K, g, topk = 8, 64, 1024, 1024, 128, 8
    wq, s, z = synth.expert_bank(67, E, N, K, g)
    ids, r = synth.routing(67, M, topk, E)
    ids[:, 0] = 0
    ids[:, 1] = 0
    x = synth.activations(67, (M, K))
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.moe_gemv(x, ids, None, wq, s, z, g), "passes x tiles per warp")
    yr = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid, route_w=dev(r))
    torch.cuda.synchronize()
    check_close(host_f64(yr), oracle.moe_gemv(x, ids, r, wq, s, z, g), "routed, passes x tiles per warp")
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("kid", MOE_KERNELS)
def test_moe_gemv_duplicate_ids_in_a_token(kid, w, oracle):
    M, E, N, K, g, topk = 9, 3, 64, 1024, 128, 2
    wq, s, z = synth.expert_bank(64, E, N, K, g)
    ids = np.zeros((M, topk), np.int32)   # every slot on expert 0: 18 slots, > 16
    ids[:, 1] = 0
    x = synth.activations(64, (M, K))
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.moe_gemv(x, ids, None, wq, s, z, g), "duplicates")


@pytest.mark.parametrize("kid", MOE_KERNELS)
def test_moe_bad_expert_id_is_flagged_not_trapped(kid, w, oracle):
    M, E, N, K, g, topk = 2, 4, 64, 1024, 128, 2
    wq, s, z = synth.expert_bank(65, E, N, K, g)
    ids = np.array([[1, 7], [-1, 2]], np.int32)
    x = synth.activations(65, (M, K))
    w.w4a16_device_error(clear=True)
    y = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid)
    bits = w.w4a16_device_error(clear=True)
    assert bits & w.DEVERR_EXPERT_ID
    got = host_f64(y)
    assert np.all(got[0, 1] == 0) and np.all(got[1, 0] == 0)
    good = oracle.moe_gemv(x, np.array([[1, 1], [2, 2]], np.int32), None, wq, s, z, g)
    check_close(got[0, 0], good[0, 0], "valid slot 0")
    check_close(got[1, 1], good[1, 1], "valid slot 1")
    # routed sum skips the bad slots
    r = np.array([[0.25, 0.75], [0.5, 0.5]], np.float32)
    yr = w.w4a16_moe_gemv(dev(x), dev(ids), *_bank_dev((wq, s, z)), g, kernel_id=kid, route_w=dev(r))
    assert w.w4a16_device_error(clear=True) & w.DEVERR_EXPERT_ID
    want = np.stack([0.25 * good[0, 0], 0.5 * good[1, 1]])
    check_close(host_f64(yr), want, "routed with bad ids")
    assert w.w4a16_device_error(clear=True) == 0


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_moe_ffn_chain_full_config(w, oracle, M):
    # 64 experts, gate/up W[1024, 2304], down W[2304, 1024], top-8 routing
    p = synth.moe_problem(M=M, E=64, H=2304, F=1024, topk=8, g=128, seed=0)
    out = w.moe_ffn(dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), _bank_dev(p["gate"]),
                    _bank_dev(p["up"]), _bank_dev(p["down"]), 128)
    torch.cuda.synchronize()
    ref = oracle.moe_ffn(p["x"], p["ids"], p["route_w"], p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(out), ref["out"], "moe ffn M=%d" % M)
    # the chain of single-purpose calls (gate GEMV, up GEMV, SwiGLU, down GEMV
    # with the routed sum) meets the same bar; it may tile differently (the
    # fused gate+up launch has twice the CTAs), so its fp32 summation order
    # and hence rare bf16 roundings can differ from the fused chain's
    chained = w.moe_ffn(dev(p["x"]), dev(p["ids"]), dev(p["route_w"]), _bank_dev(p["gate"]),
                        _bank_dev(p["up"]), _bank_dev(p["down"]), 128, fused=False)
    torch.cuda.synchronize()
    check_close(host_f64(chained), ref["out"], "moe ffn chained M=%d" % M)
    assert w.w4a16_device_error(clear=True) == 0


def test_moe_ffn_bad_ids_and_shared_experts(w, oracle):
    # 6 tokens: one expert shared by every token, one invalid id (skipped,
    # flagged); the fused chain still matches the oracle on the valid slots
    p = synth.moe_problem(M=6, E=64, H=2304, F=1024, topk=8, g=128, seed=3)
    ids = p["ids"].copy()
    ids[:, 0] = 5
    ids[2, 3] = 64
    p["ids"] = ids
    w.w4a16_device_error(clear=True)
    out = w.moe_ffn(dev(p["x"]), dev(ids), dev(p["route_w"]), _bank_dev(p["gate"]),
                    _bank_dev(p["up"]), _bank_dev(p["down"]), 128)
    torch.cuda.synchronize()
    assert w.w4a16_device_error(clear=True) & w.DEVERR_EXPERT_ID
    # the skipped slot contributes nothing: same as a valid id with weight 0
    ref_ids = ids.copy()
    ref_rw = p["route_w"].copy()
    ref_ids[2, 3] = 0
    ref_rw[2, 3] = 0.0
    ref = oracle.moe_ffn(p["x"], ref_ids, ref_rw, p["gate"], p["up"], p["down"], 128)
    check_close(host_f64(out), ref["out"], "moe ffn shared/bad ids")


@pytest.mark.parametrize("M,N,K", [(3, 6144, 4096), (4, 4096, 4096), (4, 8192, 2048), (3, 4096, 6144)])
def test_gemv_three_and_four_tokens_on_mid_size_matrices(w, oracle, M, N, K):
    # the default from 2^24 weights at three and four tokens is the fp16
    # warp-MMA kernel: every output against the oracle, and equal to the
    # forced kernel 4
    assert w.gemv_plan(M, N, K, 128)["kernel_id"] == 4
    p = synth.dense_problem(M, N, K, 128, "uniform6to10", seed=9500 + M)
    args = dense_dev(p)
    y = w.w4a16_gemv(*args, 128)
    y4 = w.w4a16_gemv(*args, 128, kernel_id=4)
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle.gemv(p["x"], p["wq"], p["scale"], p["zero"], 128),
                "M=%d %dx%d" % (M, N, K))
    assert torch.equal(y, y4)
    assert w.w4a16_device_error(clear=True) == 0
