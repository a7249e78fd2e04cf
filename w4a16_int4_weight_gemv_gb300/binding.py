"""ctypes binding of libw4a16.so (declared in include/w4a16.h).

Argument marshalling only: each function checks tensor dtypes, shapes and
devices, passes raw pointers and the current CUDA stream to the C ABI, and
raises W4A16Error on a non-OK status.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU fallback, and importing this
module fails if the library has not been built.

bf16 tensors may be passed as torch.bfloat16 or as their int16/uint16 bit
patterns.  Packed weights are int32 (bit patterns of the uint32 words).
"""
from __future__ import annotations

import ctypes
import enum
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_DEFAULT_LIB = os.path.join(_HERE, "_build", "libw4a16.so")


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_SHAPE = 2
    ERR_ALIGN = 3
    ERR_UNSUPPORTED = 4
    ERR_WORKSPACE = 5
    ERR_CUDA = 6


DEVERR_EXPERT_ID = 0x1
DEVERR_RANGE = 0x4
DEVERR_TIMEOUT = 0x2
OUT_BF16 = 0
OUT_F32 = 1


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__("%s: %s (%s)" % (where, status_string(status), self.status.name))


def lib_path() -> str:
    return os.environ.get("W4A16_LIB", _DEFAULT_LIB)


_lib = None


def load_library():
    """Load libw4a16.so; raises if it is missing (build it with build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError("libw4a16.so not built (expected at %s); run "
                          "w4a16_int4_weight_gemv_gb300.build_ext.build()" % path)
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.w4a16_abi_version.restype = I32
    lib.w4a16_abi_version.argtypes = []
    lib.w4a16_status_string.restype = ctypes.c_char_p
    lib.w4a16_status_string.argtypes = [I32]
    lib.int4_pack.restype = I32
    lib.int4_pack.argtypes = [P, P, I64, I64, P]
    lib.int4_dequant.restype = I32
    lib.int4_dequant.argtypes = [P, P, P, P, I32, I64, I64, I64, P]
    lib.w4a16_gemv_workspace_bytes.restype = SZ
    lib.w4a16_gemv_workspace_bytes.argtypes = [I32, I64, I64, I64]
    lib.w4a16_gemv.restype = I32
    lib.w4a16_gemv.argtypes = [P, P, P, P, P, I32, I32, I64, I64, I64, P, SZ, P]
    lib.w4a16_gemv_ex.restype = I32
    lib.w4a16_gemv_ex.argtypes = [P, P, P, P, P, I32, I32, I64, I64, I64, ctypes.c_uint, P]
    lib.w4a16_gemv_variant.restype = I32
    lib.w4a16_gemv_variant.argtypes = [P, P, P, P, P, I32, I32, I64, I64, I64, I32, I32, P]
    lib.w4a16_gemv_plan.restype = I32
    lib.w4a16_gemv_plan.argtypes = [I32, I64, I64, I64] + [ctypes.POINTER(I32)] * 5
    lib.w4a16_moe_workspace_bytes.restype = SZ
    lib.w4a16_moe_workspace_bytes.argtypes = [I32, I32, I64, I32]
    lib.w4a16_moe_gemv.restype = I32
    lib.w4a16_moe_gemv.argtypes = [P, I32, P, P, P, P, P, P, I32, I32, I32, I64, I64, I64,
                                   P, SZ, P]
    lib.w4a16_moe_ffn_workspace_bytes.restype = SZ
    lib.w4a16_moe_ffn_workspace_bytes.argtypes = [I32, I32, I64, I64]
    lib.w4a16_moe_ffn.restype = I32
    lib.w4a16_moe_ffn.argtypes = [P] * 13 + [I32, I32, I32, I64, I64, I64, P, SZ, P]
    lib.w4a16_swiglu.restype = I32
    lib.w4a16_swiglu.argtypes = [P, P, I64, P, I64, I64, I64, P]
    lib.w4a16_host_memory_mapped.restype = I32
    lib.w4a16_host_memory_mapped.argtypes = [P]
    lib.w4a16_device_error.restype = I32
    lib.w4a16_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), I32, P]
    lib.w4a16_wait_selftest.restype = I32
    lib.w4a16_wait_selftest.argtypes = [ctypes.c_uint, I32, P]
    lib.int3_pack.restype = I32
    lib.int3_pack.argtypes = [P, P, I64, I64, P]
    lib.int3_dequant.restype = I32
    lib.int3_dequant.argtypes = [P, P, P, P, I32, I64, I64, I64, P]
    lib.w3a16_moe_ffn_workspace_bytes.restype = SZ
    lib.w3a16_moe_ffn_workspace_bytes.argtypes = [I32, I32, I64, I64]
    lib.w3a16_moe_ffn.restype = I32
    lib.w3a16_moe_ffn.argtypes = [P] * 13 + [I32, I32, I32, I64, I64, I64, P, SZ, P]
    lib.w4a16_moe_gemv_variant.restype = I32
    lib.w4a16_moe_gemv_variant.argtypes = [P, I32, P, P, P, P, P, P, I32, I32, I32, I64, I64, I64,
                                           I32, P, SZ, P]
    lib.w3a16_moe_gemv.restype = I32
    lib.w3a16_moe_gemv.argtypes = [P, I32, P, P, P, P, P, P, I32, I32, I32, I64, I64, I64, P]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().w4a16_status_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise W4A16Error(rc, where)


# The current stream's handle for a device index, without building a Stream
# object (torch.cuda.current_stream() costs a few microseconds per call,
# which a decode loop pays on every GEMV).
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device: int = None):
    """Stream handle (an int) for a ctypes call: `stream`, or the current
    stream of `device` (the current device if None)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_current_stream is not None and device is not None and device >= 0:
        return _raw_current_stream(device)
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: torch.Tensor):
    return t.data_ptr()


def _need(t: torch.Tensor, name: str, dtypes, shape=None):
    # fast path: one expression over the properties a valid argument has
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype in dtypes and t.is_contiguous()
            and (shape is None or t.shape == tuple(shape))):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_U8 = (torch.uint8,)
_U32 = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def int4_pack(codes: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """codes uint8 [N, K] (0..15) -> packed int32 [N, K/8] (uint32 bit patterns)."""
    _need(codes, "codes", _U8)
    N, K = codes.shape
    if out is None:
        out = torch.empty((N, K // 8), dtype=torch.int32, device=codes.device)
    _need(out, "out", _U32, (N, K // 8))
    _check(load_library().int4_pack(_ptr(codes), _ptr(out), N, K, _stream(stream, codes.get_device())),
           "int4_pack")
    return out


def int4_dequant(wq, scale, zero, g: int, out_dtype=torch.bfloat16, out=None, stream=None):
    """Packed weights -> W [N, K] = (code - zero) * scale, bf16 or fp32."""
    _need(wq, "wq", _U32)
    N, K8 = wq.shape
    K = K8 * 8
    _need(scale, "scale", _BF16, (N, K // g))
    _need(zero, "zero", _U8, (N, K // g))
    if out is None:
        out = torch.empty((N, K), dtype=out_dtype, device=wq.device)
    _need(out, "out", (torch.bfloat16, torch.float32), (N, K))
    kind = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(load_library().int4_dequant(_ptr(wq), _ptr(scale), _ptr(zero), _ptr(out), kind,
                                       N, K, g, _stream(stream, wq.get_device())), "int4_dequant")
    return out


def int3_pack(codes: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """codes uint8 [N, K] (0..7, K % 128 == 0) -> INT3 words int32 [N, 3K/32]
    (uint32 bit patterns; the format is stated in include/w4a16.h)."""
    _need(codes, "codes", _U8)
    N, K = codes.shape
    if out is None:
        out = torch.empty((N, 3 * K // 32), dtype=torch.int32, device=codes.device)
    _need(out, "out", _U32, (N, 3 * K // 32))
    _check(load_library().int3_pack(_ptr(codes), _ptr(out), N, K, _stream(stream, codes.get_device())),
           "int3_pack")
    return out


def int3_dequant(wq3, scale, zero, g: int, out_dtype=torch.bfloat16, out=None, stream=None):
    """INT3 words [N, 3K/32] -> W [N, K] = (code - zero) * scale, bf16 or fp32."""
    _need(wq3, "wq3", _U32)
    N, W3 = wq3.shape
    K = W3 // 3 * 32
    _need(scale, "scale", _BF16, (N, K // g))
    _need(zero, "zero", _U8, (N, K // g))
    if out is None:
        out = torch.empty((N, K), dtype=out_dtype, device=wq3.device)
    _need(out, "out", (torch.bfloat16, torch.float32), (N, K))
    kind = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(load_library().int3_dequant(_ptr(wq3), _ptr(scale), _ptr(zero), _ptr(out), kind,
                                       N, K, g, _stream(stream, wq3.get_device())), "int3_dequant")
    return out


def w4a16_gemv_workspace_bytes(M: int, N: int, K: int, g: int) -> int:
    return int(load_library().w4a16_gemv_workspace_bytes(M, N, K, g))


def gemv_plan(M: int, N: int, K: int, g: int) -> dict:
    """The launch w4a16_gemv makes for this shape (kernel id, CTAs, threads,
    K split, shared memory)."""
    vals = [ctypes.c_int(0) for _ in range(5)]
    _check(load_library().w4a16_gemv_plan(M, N, K, g, *[ctypes.byref(v) for v in vals]),
           "w4a16_gemv_plan")
    keys = ("kernel_id", "ctas", "threads", "k_split", "smem_bytes")
    return {k: v.value for k, v in zip(keys, vals)}


FLAG_WEIGHTS_STATIC = 0x1
FLAG_SWIGLU_OUTPUT = 0x2
FLAG_NO_CLUSTER = 0x4


def _host_side(x, out) -> bool:
    return (isinstance(x, torch.Tensor) and not x.is_cuda) or \
        (isinstance(out, torch.Tensor) and not out.is_cuda)


# host addresses the library has confirmed kernels can use as they are
_mapped_host = set()


def _need_pinned(t, name, dtypes, shape=None):
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise ValueError("%s: a page-locked host tensor is needed here (with the other of "
                         "x/out on the host)" % name)
    if t.dtype not in dtypes or not t.is_contiguous() or (shape is not None and t.shape != tuple(shape)):
        raise ValueError("%s: dtype/shape/layout not accepted" % name)
    p = t.data_ptr()
    if p not in _mapped_host:
        if not load_library().w4a16_host_memory_mapped(p):
            raise ValueError("%s: this host memory is not mapped for the device" % name)
        _mapped_host.add(p)


def w4a16_gemv(x, wq, scale, zero, g: int, out=None, out_dtype=torch.bfloat16,
               kernel_id: int = 0, k_split: int = 0, weights_static: bool = False,
               swiglu_output: bool = False, no_cluster: bool = False, stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] . dequant(wq, scale, zero)^T.

    kernel_id 0 (default) lets the library choose; 1, 2, 3 or 4 force the
    CUDA-core, bf16 warp-MMA, tensor-core (tcgen05) or fp16 warp-MMA kernel
    (measurement and tests); k_split forces the K split (for kernel 4, the
    CTAs of a cluster).  weights_static declares that no
    kernel still running on the stream writes wq/scale/zero (resident
    weights), so their loads may start before that kernel completes; it
    goes with the library's own launch choice only (ValueError with a
    forced kernel_id or k_split).  swiglu_output: the rows of wq are gate and
    up rows interleaved in blocks of 8 (interleave_gate_up) and y is the
    bf16 [M, N/2] SwiGLU of the two products, formed in the kernel's
    epilogue (same restriction on forcing).  no_cluster: plan without a
    thread-block cluster where the shape allows (a launch that follows a
    different kernel starts sooner; same restriction on forcing).

    With M == 1, x and out may both be page-locked host tensors: the kernel
    reads x and writes y there directly (over NVLink-C2C on a Grace-Blackwell
    node), with no copies around the call; y is valid on the host once the
    stream has been synchronised."""
    _need(wq, "wq", _U32)
    N = wq.shape[0]
    K = wq.shape[1] * 8
    if _host_side(x, out):
        # page-locked host x / y: read and written by the kernel in place
        # (one token: the CUDA-core kernel, plain loads and stores)
        _need_pinned(x, "x", _BF16)
        M = x.shape[0]
        if M != 1 or kernel_id not in (0, 1) or swiglu_output:
            raise ValueError("page-locked host x/out: M == 1 and the CUDA-core kernel only "
                             "(no SwiGLU input)")
        if out is None:
            out = torch.empty((M, N), dtype=out_dtype).pin_memory()
        _need_pinned(out, "out", (torch.bfloat16, torch.float32), (M, N))
        device = wq.get_device()
    else:
        _need(x, "x", _BF16)
        M = x.shape[0]
        NO = N // 2 if swiglu_output else N
        if out is None:
            out = torch.empty((M, NO), dtype=torch.bfloat16 if swiglu_output else out_dtype,
                              device=x.device)
        _need(out, "out", (torch.bfloat16, torch.float32), (M, NO))
        device = x.get_device()
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x shape %s does not match wq %s" % (tuple(x.shape), tuple(wq.shape)))
    _need(scale, "scale", _BF16, (N, K // g))
    _need(zero, "zero", _U8, (N, K // g))
    kind = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    flags = ((FLAG_WEIGHTS_STATIC if weights_static else 0) | (FLAG_SWIGLU_OUTPUT if swiglu_output else 0) |
             (FLAG_NO_CLUSTER if no_cluster else 0))
    if flags and (kernel_id or k_split):
        raise ValueError("weights_static, swiglu_output and no_cluster apply to the library's own "
                         "launch choice; they cannot be combined with kernel_id or k_split")
    lib = load_library()
    sh = _stream(stream, device)
    if flags:
        rc = lib.w4a16_gemv_ex(_ptr(x), _ptr(wq), _ptr(scale), _ptr(zero), _ptr(out), kind,
                               M, N, K, g, flags, sh)
    elif kernel_id == 0 and k_split == 0:
        rc = lib.w4a16_gemv(_ptr(x), _ptr(wq), _ptr(scale), _ptr(zero), _ptr(out), kind,
                            M, N, K, g, None, 0, sh)
    else:
        rc = lib.w4a16_gemv_variant(_ptr(x), _ptr(wq), _ptr(scale), _ptr(zero), _ptr(out),
                                    kind, M, N, K, g, kernel_id or (1 if M == 1 else 2),
                                    k_split, sh)
    _check(rc, "w4a16_gemv")
    return out


def w4a16_moe_workspace_bytes(M: int, topk: int, N: int, route: bool) -> int:
    return int(load_library().w4a16_moe_workspace_bytes(M, topk, N, int(bool(route))))


def w4a16_moe_gemv(x, expert_ids, wq, scale, zero, g: int, route_w=None, x_per_slot=False,
                   out=None, workspace=None, stream=None, kernel_id: int = 0) -> torch.Tensor:
    """Expert-indexed GEMV.  wq int32 [E, N, K/8]; scale/zero [E, N, K/g];
    expert_ids int32 [M, topk]; x [M, K] or (x_per_slot) [M, topk, K].
    Returns bf16 [M, topk, N] (no route_w) or [M, N] (routed sum).
    kernel_id: 0 the library's choice, 2 the bf16 warp-MMA expert kernel,
    4 the fp16 warp-MMA expert kernel (no workspace)."""
    _need(expert_ids, "expert_ids", (torch.int32,))
    M, topk = expert_ids.shape
    _need(wq, "wq", _U32)
    E, N, K8 = wq.shape
    K = K8 * 8
    _need(x, "x", _BF16, (M, topk, K) if x_per_slot else (M, K))
    _need(scale, "scale", _BF16, (E, N, K // g))
    _need(zero, "zero", _U8, (E, N, K // g))
    lib = load_library()
    if route_w is not None:
        _need(route_w, "route_w", (torch.float32,), (M, topk))
        shape = (M, N)
        need = w4a16_moe_workspace_bytes(M, topk, N, True) if kernel_id != 4 else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need // 4, dtype=torch.float32, device=x.device)
        if workspace is None:
            ws_ptr, ws_bytes = None, 0
        else:
            ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
        rw = _ptr(route_w)
    else:
        shape = (M, topk, N)
        ws_ptr, ws_bytes, rw = None, 0, None
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
    _need(out, "out", _BF16, shape)
    if kernel_id == 0:
        _check(lib.w4a16_moe_gemv(_ptr(x), int(bool(x_per_slot)), _ptr(expert_ids), rw, _ptr(wq),
                                  _ptr(scale), _ptr(zero), _ptr(out), M, topk, E, N, K, g,
                                  ws_ptr, ws_bytes, _stream(stream, x.get_device())),
               "w4a16_moe_gemv")
    else:
        _check(lib.w4a16_moe_gemv_variant(_ptr(x), int(bool(x_per_slot)), _ptr(expert_ids), rw,
                                          _ptr(wq), _ptr(scale), _ptr(zero), _ptr(out), M, topk,
                                          E, N, K, g, int(kernel_id), ws_ptr, ws_bytes,
                                          _stream(stream, x.get_device())),
               "w4a16_moe_gemv_variant")
    return out


def interleave_gate_up(gate, up) -> torch.Tensor:
    """The row layout W4A16_FLAG_SWIGLU_OUTPUT reads: two [I, ...] tensors
    (packed weights, scales or zero points of the gate and up matrices, I a
    multiple of 8) as one [2I, ...] tensor whose 16-row blocks hold 8 gate
    rows, then the same 8 up rows.  A one-time copy at weight-load time."""
    if gate.shape != up.shape or gate.dim() < 1 or gate.shape[0] % 8 != 0:
        raise ValueError("gate and up must have the same shape, rows a multiple of 8")
    rest = tuple(gate.shape[1:])
    blocks = torch.stack((gate.reshape((-1, 8) + rest), up.reshape((-1, 8) + rest)), dim=1)
    return blocks.reshape((2 * gate.shape[0],) + rest).contiguous()


def w4a16_swiglu(gate, up, out=None, stream=None) -> torch.Tensor:
    """h = bf16(silu(gate) * up).  gate/up may be views with a row stride
    (e.g. the two halves of a stacked [rows, 2N] tensor)."""
    for t, name in ((gate, "gate"), (up, "up")):
        if not t.is_cuda or t.dtype not in _BF16 or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("%s must be a CUDA bf16 matrix with unit column stride" % name)
    if gate.shape != up.shape or gate.stride(0) != up.stride(0):
        raise ValueError("gate and up must have the same shape and row stride")
    rows, N = gate.shape
    if out is None:
        out = torch.empty((rows, N), dtype=torch.bfloat16, device=gate.device)
    if out.dim() != 2 or tuple(out.shape) != (rows, N) or out.stride(1) != 1:
        raise ValueError("out must be [rows, N] with unit column stride")
    _check(load_library().w4a16_swiglu(_ptr(gate), _ptr(up), gate.stride(0), _ptr(out),
                                       out.stride(0), rows, N, _stream(stream, gate.get_device())),
           "w4a16_swiglu")
    return out


def w4a16_device_error(clear: bool = True, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(load_library().w4a16_device_error(ctypes.byref(bits), int(bool(clear)),
                                             _stream(stream)), "w4a16_device_error")
    return int(bits.value)


def w4a16_wait_selftest(max_iters: int, arrive: bool, stream=None) -> None:
    """One bounded mbarrier wait that completes (arrive) or expires
    (W4A16_DEVERR_TIMEOUT in the device error word)."""
    _check(load_library().w4a16_wait_selftest(int(max_iters), int(bool(arrive)), _stream(stream)),
           "w4a16_wait_selftest")


def moe_ffn(x, expert_ids, route_w, gate, up, down, g: int, stream=None,
            fused: bool = True) -> torch.Tensor:
    """Routed SwiGLU FFN for M tokens.  gate/up/down are (wq, scale, zero)
    triples with gate/up [E, F, H] and down [E, H, F].  Returns bf16 [M, H].

    fused (default): w4a16_moe_ffn -- two launches: the gate and up products
    with the SwiGLU formed in their epilogue, then the down products and the
    routed sums (older expert kernels outside the fp16 path's limits).
    fused=False: the same chain from the single-purpose calls (one
    expert-indexed GEMV each for gate and up, w4a16_swiglu, the down GEMV
    with the routed sum)."""
    M, topk = expert_ids.shape
    if fused:
        _need(x, "x", _BF16)
        _need(expert_ids, "expert_ids", (torch.int32,))
        _need(route_w, "route_w", (torch.float32,), (M, topk))
        (gw, gs, gz), (uw, us, uz), (dw, ds, dz) = gate, up, down
        E, F, H8 = gw.shape
        H = H8 * 8
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
        lib = load_library()
        nbytes = int(lib.w4a16_moe_ffn_workspace_bytes(M, topk, H, F))
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
        _check(lib.w4a16_moe_ffn(_ptr(x), _ptr(expert_ids), _ptr(route_w), _ptr(gw), _ptr(gs),
                                 _ptr(gz), _ptr(uw), _ptr(us), _ptr(uz), _ptr(dw), _ptr(ds),
                                 _ptr(dz), _ptr(y), M, topk, E, H, F, g, _ptr(ws), nbytes,
                                 _stream(stream, x.get_device())), "w4a16_moe_ffn")
        return y
    g_out = w4a16_moe_gemv(x, expert_ids, *gate, g, stream=stream)
    u_out = w4a16_moe_gemv(x, expert_ids, *up, g, stream=stream)
    F = g_out.shape[-1]
    h = w4a16_swiglu(g_out.view(M * topk, F), u_out.view(M * topk, F), stream=stream)
    return w4a16_moe_gemv(h.view(M, topk, F), expert_ids, *down, g, route_w=route_w,
                          x_per_slot=True, stream=stream)


def w3a16_moe_ffn(x, expert_ids, route_w, gate, up, down, g: int, stream=None) -> torch.Tensor:
    """Routed SwiGLU FFN over INT3 (~3-bit) expert banks.  gate/up/down are
    (wq3, scale, zero) triples: gate/up wq3 [E, F, 3H/32], down [E, H, 3F/32],
    scale/zero as for INT4.  Returns bf16 [M, H]."""
    M, topk = expert_ids.shape
    _need(x, "x", _BF16)
    _need(expert_ids, "expert_ids", (torch.int32,))
    _need(route_w, "route_w", (torch.float32,), (M, topk))
    (gw, gs, gz), (uw, us, uz), (dw, ds, dz) = gate, up, down
    E, F, H3 = gw.shape
    H = H3 // 3 * 32
    y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    lib = load_library()
    nbytes = int(lib.w3a16_moe_ffn_workspace_bytes(M, topk, H, F))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    _check(lib.w3a16_moe_ffn(_ptr(x), _ptr(expert_ids), _ptr(route_w), _ptr(gw), _ptr(gs),
                             _ptr(gz), _ptr(uw), _ptr(us), _ptr(uz), _ptr(dw), _ptr(ds),
                             _ptr(dz), _ptr(y), M, topk, E, H, F, g, _ptr(ws), nbytes,
                             _stream(stream, x.get_device())), "w3a16_moe_ffn")
    return y


def w3a16_moe_gemv(x, expert_ids, wq3, scale, zero, g: int, route_w=None, x_per_slot=False,
                   out=None, stream=None) -> torch.Tensor:
    """Expert-indexed GEMV over an INT3 (~3-bit) expert bank.  wq3 int32
    [E, N, 3K/32]; scale/zero [E, N, K/g]; expert_ids int32 [M, topk]; x
    [M, K] or (x_per_slot) [M, topk, K].  Returns bf16 [M, topk, N] (no
    route_w) or [M, N] (routed sum).  No workspace."""
    _need(expert_ids, "expert_ids", (torch.int32,))
    M, topk = expert_ids.shape
    _need(wq3, "wq3", _U32)
    E, N, K3 = wq3.shape
    if K3 % 12 != 0:
        raise ValueError("wq3 rows must hold whole 128-code blocks (12 words each)")
    K = K3 // 12 * 128
    _need(x, "x", _BF16, (M, topk, K) if x_per_slot else (M, K))
    _need(scale, "scale", _BF16, (E, N, K // g))
    _need(zero, "zero", _U8, (E, N, K // g))
    if route_w is not None:
        _need(route_w, "route_w", (torch.float32,), (M, topk))
        shape = (M, N)
    else:
        shape = (M, topk, N)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
    _need(out, "out", _BF16, shape)
    _check(load_library().w3a16_moe_gemv(_ptr(x), int(bool(x_per_slot)), _ptr(expert_ids),
                                         None if route_w is None else _ptr(route_w), _ptr(wq3),
                                         _ptr(scale), _ptr(zero), _ptr(out), M, topk, E, N, K, g,
                                         _stream(stream, x.get_device())), "w3a16_moe_gemv")
    return out


load_library()
