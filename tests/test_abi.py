"""The C-ABI library loads, exports every function include/w4a16.h declares,
and validates arguments before touching the device (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    from w4a16_int4_weight_gemv_gb300 import build_ext
    build_ext.build()
    from w4a16_int4_weight_gemv_gb300 import binding
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"W4A16_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("int4_pack", "int4_dequant", "w4a16_gemv", "w4a16_moe_gemv", "w4a16_swiglu",
              "w4a16_gemv_workspace_bytes", "w4a16_status_string", "w4a16_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_exports_are_exactly_the_header(lib):
    import subprocess
    from w4a16_int4_weight_gemv_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.lib_path()], capture_output=True,
                         text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = sorted(line.split()[-1] for line in out.stdout.splitlines() if " T " in line)
    assert exported == declared_functions()


def test_status_strings(lib):
    from w4a16_int4_weight_gemv_gb300 import binding
    for st in binding.Status:
        s = binding.status_string(st)
        assert s and s != "unknown status"
    assert binding.status_string(99) == "unknown status"
    assert lib.w4a16_abi_version() == 1


P = ctypes.c_void_p
A16 = P(0x1000)   # 16-byte aligned dummy address (never dereferenced: validation fails first)
MIS = P(0x1004)   # misaligned


def _gemv(lib, x=A16, wq=A16, s=A16, z=A16, y=A16, dtype=0, M=1, N=64, K=128, g=128):
    return lib.w4a16_gemv(x, wq, s, z, y, dtype, M, N, K, g, None, 0, None)


def test_gemv_validation_before_any_launch(lib):
    from w4a16_int4_weight_gemv_gb300.binding import Status
    assert _gemv(lib, x=None) == Status.ERR_NULL
    assert _gemv(lib, y=None) == Status.ERR_NULL
    assert _gemv(lib, M=0) == Status.ERR_SHAPE
    assert _gemv(lib, M=17) == Status.ERR_UNSUPPORTED
    assert _gemv(lib, N=0) == Status.ERR_SHAPE
    assert _gemv(lib, K=100) == Status.ERR_SHAPE
    assert _gemv(lib, K=96, g=64) == Status.ERR_SHAPE       # K % g != 0
    assert _gemv(lib, g=48, K=96) == Status.ERR_SHAPE       # g % 32 != 0
    assert _gemv(lib, K=131072, g=128) == Status.ERR_UNSUPPORTED
    assert _gemv(lib, N=1 << 30, K=4096) == Status.ERR_UNSUPPORTED
    assert _gemv(lib, dtype=7) == Status.ERR_UNSUPPORTED
    assert _gemv(lib, wq=MIS) == Status.ERR_ALIGN
    assert _gemv(lib, y=MIS) == Status.ERR_ALIGN
    assert _gemv(lib, M=3, K=128, g=64) == Status.ERR_UNSUPPORTED   # warp-MMA needs g % 128 == 0
    var = lib.w4a16_gemv_variant
    assert var(A16, A16, A16, A16, A16, 0, 1, 64, 128, 128, 4, 0, None) == Status.ERR_UNSUPPORTED
    # the tensor-core kernel needs g % 128 == 0 and splits K over at most 8 CTAs
    assert var(A16, A16, A16, A16, A16, 0, 1, 64, 128, 64, 3, 0, None) == Status.ERR_UNSUPPORTED
    assert var(A16, A16, A16, A16, A16, 0, 1, 64, 4096, 128, 3, 16, None) == Status.ERR_UNSUPPORTED
    assert var(A16, A16, A16, A16, A16, 0, 3, 64, 128, 128, 1, 0, None) == Status.ERR_UNSUPPORTED
    # flags the interface does not define (0x1, 0x2 and 0x4 are defined)
    for bad in (0x8, 0x80000000):
        assert lib.w4a16_gemv_ex(A16, A16, A16, A16, A16, 0, 1, 64, 128, 128, bad, None) == \
            Status.ERR_UNSUPPORTED


def test_gemv_without_device_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from w4a16_int4_weight_gemv_gb300.binding import Status
    assert _gemv(lib) == Status.ERR_CUDA
    assert lib.w3a16_moe_gemv(A16, 0, A16, None, A16, A16, A16, A16, 1, 8, 64, 1024, 2304, 128,
                              None) == Status.ERR_CUDA
    # kernel 4 takes a routed sum without a workspace: the device is the next check
    assert lib.w4a16_moe_gemv_variant(A16, 0, A16, A16, A16, A16, A16, A16, 1, 8, 64, 1024, 2304,
                                      128, 4, None, 0, None) == Status.ERR_CUDA
    assert lib.w4a16_gemv_plan(1, 4096, 4096, 128, None, None, None, None, None) == Status.ERR_CUDA


def test_other_entry_points_validate(lib):
    from w4a16_int4_weight_gemv_gb300.binding import Status
    assert lib.int4_pack(None, A16, 4, 8, None) == Status.ERR_NULL
    assert lib.int4_pack(A16, A16, 4, 12, None) == Status.ERR_SHAPE
    assert lib.int4_pack(MIS, A16, 4, 8, None) == Status.ERR_ALIGN
    assert lib.int4_pack(A16, A16, 0, 8, None) == Status.OK          # empty: nothing to do
    assert lib.int4_dequant(A16, A16, A16, None, 0, 4, 128, 128, None) == Status.ERR_NULL
    assert lib.int4_dequant(A16, A16, A16, A16, 0, 4, 128, 96, None) == Status.ERR_SHAPE
    assert lib.int4_dequant(A16, A16, A16, A16, 5, 4, 128, 128, None) == Status.ERR_UNSUPPORTED
    assert lib.int4_dequant(A16, A16, A16, A16, 0, 0, 128, 128, None) == Status.OK
    assert lib.w4a16_swiglu(A16, A16, 8, None, 8, 2, 8, None) == Status.ERR_NULL
    assert lib.w4a16_swiglu(A16, A16, 8, A16, 8, 2, 7, None) == Status.ERR_SHAPE
    assert lib.w4a16_swiglu(A16, A16, 4, A16, 8, 2, 8, None) == Status.ERR_SHAPE
    assert lib.w4a16_swiglu(A16, A16, 8, A16, 8, 0, 8, None) == Status.OK
    moe = lib.w4a16_moe_gemv
    assert moe(A16, 0, None, None, A16, A16, A16, A16, 1, 8, 64, 1024, 2304, 128, None, 0,
               None) == Status.ERR_NULL
    assert moe(A16, 0, A16, None, A16, A16, A16, A16, 1, 0, 64, 1024, 2304, 128, None, 0,
               None) == Status.ERR_SHAPE
    assert moe(A16, 0, A16, None, A16, A16, A16, A16, 64, 8, 64, 1024, 2304, 128, None, 0,
               None) == Status.ERR_UNSUPPORTED   # M * topk > 256
    assert moe(A16, 0, A16, A16, A16, A16, A16, A16, 1, 8, 64, 1024, 2304, 128, None, 0,
               None) == Status.ERR_WORKSPACE
    need = lib.w4a16_moe_workspace_bytes(1, 8, 1024, 1)
    assert need == 8 * 1024 * 4
    assert moe(A16, 0, A16, A16, A16, A16, A16, A16, 1, 8, 64, 1024, 2304, 128, A16, need - 4,
               None) == Status.ERR_WORKSPACE
    assert lib.w4a16_moe_workspace_bytes(1, 8, 1024, 0) == 0
    var = lib.w4a16_moe_gemv_variant
    def mv(kid, M=1, topk=8, N=1024, K=2304, g=128, rw=None, ws=None, nbytes=0):
        return var(A16, 0, A16, rw, A16, A16, A16, A16, M, topk, 64, N, K, g, kid, ws, nbytes, None)
    assert mv(3) == Status.ERR_UNSUPPORTED                  # no such expert kernel
    assert mv(1) == Status.ERR_UNSUPPORTED
    assert mv(4, M=5) == Status.ERR_UNSUPPORTED             # kernel 4: at most 32 slots
    assert mv(4, N=1000) == Status.ERR_UNSUPPORTED          # 16-row output tiles
    assert mv(4, K=2240, g=64) == Status.ERR_UNSUPPORTED    # groups of 128 k
    assert mv(2, rw=A16) == Status.ERR_WORKSPACE            # kernel 2 needs the routed-sum workspace
    assert mv(0, rw=A16) == Status.ERR_WORKSPACE            # so does the library's choice
    # fused FFN: 13 pointers, then M, topk, E, H, F, g, workspace, bytes, stream
    ffn = lib.w4a16_moe_ffn
    ptrs = [A16] * 13
    assert ffn(*([None] + ptrs[1:]), 1, 8, 64, 2304, 1024, 128, A16, 1 << 20, None) == Status.ERR_NULL
    assert ffn(*ptrs, 1, 8, 64, 2304, 1000, 128, A16, 1 << 20, None) == Status.ERR_SHAPE   # F % g
    assert ffn(*ptrs, 64, 8, 64, 2304, 1024, 128, A16, 1 << 20, None) == Status.ERR_UNSUPPORTED
    assert ffn(*ptrs, 1, 8, 64, 2304, 1024, 64, A16, 1 << 20, None) == Status.ERR_UNSUPPORTED
    fneed = lib.w4a16_moe_ffn_workspace_bytes(1, 8, 2304, 1024)
    assert fneed == 2 * 8 * 1024 * 2 + 8 * 2304 * 4 + 256   # parts rounded to 256 bytes; 36 counters
    assert ffn(*ptrs, 1, 8, 64, 2304, 1024, 128, A16, fneed - 16, None) == Status.ERR_WORKSPACE
    assert ffn(*ptrs, 1, 8, 64, 2304, 1024, 128, None, fneed, None) == Status.ERR_WORKSPACE
    assert ffn(*ptrs[:-1], MIS, 1, 8, 64, 2304, 1024, 128, A16, fneed, None) == Status.ERR_ALIGN
    assert lib.w4a16_gemv_workspace_bytes(1, 4096, 4096, 128) == 0
    assert lib.w4a16_host_memory_mapped(None) == 0
    buf = ctypes.create_string_buffer(64)   # ordinary host memory is never reported mapped
    assert lib.w4a16_host_memory_mapped(ctypes.cast(buf, P)) == 0
    assert lib.w4a16_device_error(None, 0, None) == Status.ERR_NULL


def test_int3_entry_points_validate(lib):
    from w4a16_int4_weight_gemv_gb300.binding import Status
    assert lib.int3_pack(None, A16, 4, 128, None) == Status.ERR_NULL
    assert lib.int3_pack(A16, A16, 4, 96, None) == Status.ERR_SHAPE      # whole 128-code blocks
    assert lib.int3_pack(A16, MIS, 4, 128, None) == Status.ERR_ALIGN
    assert lib.int3_pack(A16, A16, 0, 128, None) == Status.OK
    assert lib.int3_dequant(A16, A16, A16, None, 0, 4, 128, 128, None) == Status.ERR_NULL
    assert lib.int3_dequant(A16, A16, A16, A16, 0, 4, 256, 96, None) == Status.ERR_SHAPE
    assert lib.int3_dequant(A16, A16, A16, A16, 3, 4, 128, 128, None) == Status.ERR_UNSUPPORTED
    assert lib.int3_dequant(A16, A16, A16, A16, 0, 0, 128, 128, None) == Status.OK
    ffn = lib.w3a16_moe_ffn
    ptrs = [A16] * 13
    need = lib.w3a16_moe_ffn_workspace_bytes(1, 8, 2304, 1024)
    assert need == 8 * 1024 * 2
    assert ffn(*([None] + ptrs[1:]), 1, 8, 64, 2304, 1024, 128, A16, need, None) == Status.ERR_NULL
    assert ffn(*ptrs, 1, 8, 64, 2304, 1000, 128, A16, need, None) == Status.ERR_SHAPE
    assert ffn(*ptrs, 9, 2, 64, 2304, 1024, 128, A16, need, None) == Status.ERR_UNSUPPORTED
    assert ffn(*ptrs, 1, 8, 64, 2304, 1024, 128, A16, need - 16, None) == Status.ERR_WORKSPACE
    assert ffn(*ptrs[:-1], MIS, 1, 8, 64, 2304, 1024, 128, A16, need, None) == Status.ERR_ALIGN
    # expert GEMV: x, x_per_slot, ids, route_w, wq3, scale, zero, y, M, topk, E, N, K, g, stream
    def gemv3(x=A16, ids=A16, rw=None, wq3=A16, y=A16, M=1, topk=8, N=1024, K=2304, g=128):
        return lib.w3a16_moe_gemv(x, 0, ids, rw, wq3, A16, A16, y, M, topk, 64, N, K, g, None)
    assert gemv3(ids=None) == Status.ERR_NULL
    assert gemv3(y=None) == Status.ERR_NULL
    assert gemv3(topk=0) == Status.ERR_SHAPE
    assert gemv3(K=2300) == Status.ERR_SHAPE                   # whole 128-code blocks
    assert gemv3(K=64, g=64) == Status.ERR_SHAPE
    assert gemv3(g=256) == Status.ERR_UNSUPPORTED               # groups of 128 only
    assert gemv3(M=5) == Status.ERR_UNSUPPORTED                 # 40 slots > 32
    assert gemv3(N=1000) == Status.ERR_UNSUPPORTED              # 16-row output tiles
    assert gemv3(wq3=MIS) == Status.ERR_ALIGN
    assert gemv3(rw=MIS) == Status.ERR_ALIGN


def test_binding_rejects_cpu_tensors(lib):
    import torch
    from w4a16_int4_weight_gemv_gb300 import binding
    x = torch.zeros(1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.w4a16_gemv(x, torch.zeros(4, 16, dtype=torch.int32),
                           torch.zeros(4, 1, dtype=torch.bfloat16),
                           torch.zeros(4, 1, dtype=torch.uint8), 128)


def test_product_path_does_not_import_oracle():
    # the binding and build modules never reference the oracle package
    pkg = os.path.join(ROOT, "w4a16_int4_weight_gemv_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            text = open(os.path.join(pkg, name)).read()
            assert "import oracle" not in text and "from oracle" not in text, name


def test_plain_c_caller_builds_against_the_header(lib):
    # the C caller the benchmark times (host_loop.c) compiles against
    # include/w4a16.h and links against the library; without a GPU it stops
    # at its first CUDA call with an error message, not a crash
    import subprocess
    import torch
    import bench
    exe = bench.host_loop_path()
    if exe is None:
        pytest.skip("nvcc not available")
    r = subprocess.run([exe, "1", "256", "512", "128", "2", "1"], capture_output=True, text=True)
    if torch.cuda.is_available():
        assert r.returncode == 0, r.stderr
        assert '"check": "bit-equal"' in r.stdout
    else:
        assert r.returncode == 1 and r.stderr.strip()
    assert subprocess.run([exe], capture_output=True).returncode == 2   # usage
