"""The allocation-free routed expert GEMV (w4a16_moe_gemv_fixed_scratch).

Some callers cannot allocate device memory or lend the library a workspace
-- engines with fixed device memory pools, plug-ins whose host runtime owns
the allocator.  This entry point keeps its fp32 partials in a scratch buffer
compiled into the library.  Its results must match the workspace entry
point, call after call (the buffer is shared and keeps the previous call's
contents), and what an earlier call left in the buffer must never reach a
later call's output.  Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from w4a16_int4_weight_gemv_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding
    lib = binding.load_library()
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.w4a16_moe_gemv_fixed_scratch.restype = I32
    lib.w4a16_moe_gemv_fixed_scratch.argtypes = [P, I32, P, P, P, P, P, P, I32, I32, I32, I64,
                                                 I64, I64, P]
    return lib


def _call_both(lib, M, topk, E, N, K, x_per_slot, seed):
    g = 128
    wq, s, z = synth.expert_bank(seed, E, N, K, g)
    ids, r = synth.routing(seed, M, topk, E)
    x = synth.activations(seed, (M, topk, K) if x_per_slot else (M, K))
    d = [_dev(a) for a in (x, ids, r, wq, s, z)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y_fixed = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.w4a16_moe_gemv_fixed_scratch(_ptr(d[0]), int(x_per_slot), _ptr(d[1]), _ptr(d[2]),
                                          _ptr(d[3]), _ptr(d[4]), _ptr(d[5]), _ptr(y_fixed),
                                          M, topk, E, N, K, g, stream)
    assert rc == 0
    ws = torch.empty(M * topk * N, dtype=torch.float32, device="cuda")
    y_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = lib.w4a16_moe_gemv(_ptr(d[0]), int(x_per_slot), _ptr(d[1]), _ptr(d[2]), _ptr(d[3]),
                            _ptr(d[4]), _ptr(d[5]), _ptr(y_ref), M, topk, E, N, K, g, _ptr(ws),
                            ws.numel() * 4, stream)
    assert rc == 0
    torch.cuda.synchronize()
    return y_fixed.float().cpu().numpy().astype(np.float64), y_ref.float().cpu().numpy().astype(np.float64)


def _close(got, ref):
    assert np.all(np.isfinite(got))
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= 5e-3
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


def test_fixed_scratch_matches_workspace_entry_point_twice(lib):
    # the MoE down projection (per-slot inputs, routed sum), then a larger
    # call that overwrites more of the shared buffer, then a small one again
    for (M, topk, E, N, K, per_slot, seed) in ((4, 8, 64, 2304, 1024, True, 70),
                                               (2, 8, 64, 1024, 2304, False, 71),
                                               (4, 8, 64, 2304, 1024, True, 72)):
        got, ref = _call_both(lib, M, topk, E, N, K, per_slot, seed)
        _close(got, ref)
        assert np.array_equal(got, ref)  # same kernels, same order: identical bits


def test_fixed_scratch_rejects_oversized_requests(lib):
    # 16 tokens x 8 slots x 4096 rows x 4 bytes = 2 MiB > the fixed buffer
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = _ptr(dummy)
    rc = lib.w4a16_moe_gemv_fixed_scratch(p, 0, p, p, p, p, p, p, 16, 8, 64, 4096, 1024, 128,
                                          None)
    from w4a16_int4_weight_gemv_gb300 import binding
    assert rc == binding.Status.ERR_WORKSPACE


def test_stale_buffer_contents_never_reach_bad_slots(lib, oracle):
    # a first call fills the buffer with partials of every slot; a second
    # call with ids outside [0, E) in some slots must give exactly what the
    # oracle gives with those slots left out (the device error bit is set)
    from w4a16_int4_weight_gemv_gb300 import binding
    M, topk, E, N, K, g = 3, 4, 8, 512, 1024, 128
    wq, s, z = synth.expert_bank(75, E, N, K, g)
    x = synth.activations(75, (M, K))
    good_ids = np.array([[0, 1, 2, 3], [4, 5, 6, 7], [1, 3, 5, 7]], np.int32)
    bad_ids = np.array([[0, -1, 2, 8], [E + 5, 5, 6, -7], [1, 3, 5, 7]], np.int32)
    r = synth.routing(75, M, topk, E)[1]
    d = [_dev(a) for a in (x, wq, s, z, r)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for ids in (good_ids, bad_ids):
        di = _dev(ids)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.w4a16_moe_gemv_fixed_scratch(_ptr(d[0]), 0, _ptr(di), _ptr(d[4]), _ptr(d[1]),
                                              _ptr(d[2]), _ptr(d[3]), _ptr(y), M, topk, E, N, K,
                                              g, stream)
        assert rc == 0
        torch.cuda.synchronize()
        outs.append(y.float().cpu().numpy().astype(np.float64))
    assert binding.w4a16_device_error(clear=True) & binding.DEVERR_EXPERT_ID
    valid = (bad_ids >= 0) & (bad_ids < E)
    ids_ok = np.where(valid, bad_ids, 0).astype(np.int32)
    r_ok = np.where(valid, r, 0.0).astype(np.float32)
    _close(outs[1], oracle.moe_gemv(x, ids_ok, r_ok, wq, s, z, g))
    _close(outs[0], oracle.moe_gemv(x, good_ids, r, wq, s, z, g))


def test_unrouted_call_needs_no_buffer(lib, oracle):
    # without route weights the call stores per-slot products and touches no
    # scratch; it matches the oracle slot by slot
    M, topk, E, N, K, g = 2, 3, 6, 256, 1024, 128
    wq, s, z = synth.expert_bank(76, E, N, K, g)
    x = synth.activations(76, (M, K))
    ids = synth.routing(76, M, topk, E)[0]
    d = [_dev(a) for a in (x, ids, wq, s, z)]
    y = torch.empty((M, topk, N), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.w4a16_moe_gemv_fixed_scratch(_ptr(d[0]), 0, _ptr(d[1]), None, _ptr(d[2]), _ptr(d[3]),
                                          _ptr(d[4]), _ptr(y), M, topk, E, N, K, g, stream)
    assert rc == 0
    torch.cuda.synchronize()
    want = oracle.moe_gemv(x, ids, None, wq, s, z, g)
    got = y.float().cpu().numpy().astype(np.float64)
    for t in range(M):
        for j in range(topk):
            _close(got[t, j], want[t, j])
