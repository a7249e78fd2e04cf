"""Reference oracle for the W4A16 INT4-weight GEMV -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding in ``w4a16_int4_weight_gemv_gb300``) never imports it, and this
package imports nothing from there: the two share no code.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, fp64, unblocked loops;
see its header for the definitions and the passages they follow).  This file
only compiles that source with gcc and marshals numpy arrays through ctypes.

Parity status of each function (what pins it, in tests/test_oracle.py):
  pack / unpack      pinned: hand-derived packed words, exhaustive round trip
  bf16_round         pinned: binary32->bf16 library conversion, hand ties
  dequant            pinned: exhaustive (q, z) x scale sweep vs exact integer
                     products, one-hot GEMV columns
  gemv / gemv_rows   pinned: closed form for constant codes, one-hot
                     activations, fp64 library matmul, brute force, invariants
  gemv_parallel      pinned: equal to gemv element for element (same sums)
  swiglu             pinned: closed forms at 0 and large |v|, library silu
  moe_gemv, moe_ffn  pinned: one-hot routing reduces to a dense chain,
                     identical experts reduce to one chain, linearity in r

The ~3-bit expert weights (``int3_oracle.c``: the format is this library's
reading, stated in that file's header), pinned in tests/test_oracle_int3.py:
  pack3 / unpack3    pinned: hand-derived chunk words, every code bit owning
                     one distinct bit of its block, random round trip
  dequant3, gemv3    pinned: equal to the INT4 oracle on the same codes (all
                     codes 0..7 are INT4 codes), closed form, one-hot
                     activations, fp64 library matmul
  moe_ffn3           pinned: equal to the INT4 chain on the same codes
  moe_gemv3          pinned: equal to the INT4 expert GEMV on the same codes
                     (per-slot and routed, shared and per-slot inputs)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "int3_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: x86_64 and aarch64)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or any(
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(src) for src in _SRCS)
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off"] + _SRCS + ["-o", tmp, "-lm"]
        # OpenMP only spreads oracle_gemv_parallel's rows over host threads;
        # without it that function runs on one thread
        if subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True).returncode != 0:
            subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class using_library:
    """Temporarily route every oracle call through another build of the C
    source (used by the mutation tests, which compile deliberately broken
    copies to show that the pins catch them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int64
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round_array.argtypes = [P, P, I]
    lib.oracle_pack.argtypes = [P, P, I, I]
    lib.oracle_unpack.argtypes = [P, P, I, I]
    lib.oracle_dequant.argtypes = [P, P, P, P, I, I, I]
    lib.oracle_gemv.argtypes = [P, P, P, P, P, I, I, I, I]
    lib.oracle_gemv_rows.argtypes = [P, P, P, P, P, I, P, I, I, I]
    if hasattr(lib, "oracle_gemv_parallel"):
        lib.oracle_gemv_parallel.argtypes = [P, P, P, P, P, I, I, I, I, I]
        lib.oracle_max_threads.restype = I
        lib.oracle_max_threads.argtypes = []
    lib.oracle_swiglu.argtypes = [P, P, P, I]
    lib.oracle_moe_gemv.restype = ctypes.c_int
    lib.oracle_moe_gemv.argtypes = [P, ctypes.c_int, P, P, P, P, P, P,
                                    I, I, I, I, I, I]
    lib.oracle_moe_ffn.restype = ctypes.c_int
    lib.oracle_moe_ffn.argtypes = [P] * 17 + [I] * 6
    lib.oracle3_pack.argtypes = [P, P, I, I]
    lib.oracle3_unpack.argtypes = [P, P, I, I]
    lib.oracle3_dequant.argtypes = [P, P, P, P, I, I, I]
    lib.oracle3_gemv.argtypes = [P, P, P, P, P, I, I, I, I]
    lib.oracle3_moe_ffn.restype = ctypes.c_int
    lib.oracle3_moe_ffn.argtypes = [P] * 17 + [I] * 6
    lib.oracle3_moe_gemv.restype = ctypes.c_int
    lib.oracle3_moe_gemv.argtypes = [P, ctypes.c_int, P, P, P, P, P, P, I, I, I, I, I, I]
    return lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_round(v) -> np.ndarray:
    """fp64 values -> bf16 bit patterns, one RNE rounding (C oracle)."""
    lib = _load()
    v, pv = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib.oracle_bf16_round_array(pv, out.ctypes.data_as(ctypes.c_void_p), v.size)
    return out


def pack(codes) -> np.ndarray:
    """codes uint8 [N, K] (0..15) -> packed uint32 [N, K/8]."""
    lib = _load()
    codes, pc = _c(codes, np.uint8)
    N, K = codes.shape
    assert K % 8 == 0
    wq = np.empty((N, K // 8), np.uint32)
    lib.oracle_pack(pc, wq.ctypes.data_as(ctypes.c_void_p), N, K)
    return wq


def unpack(wq, K: int) -> np.ndarray:
    lib = _load()
    wq, pw = _c(wq, np.uint32)
    N = wq.shape[0]
    assert wq.shape[1] * 8 == K
    codes = np.empty((N, K), np.uint8)
    lib.oracle_unpack(pw, codes.ctypes.data_as(ctypes.c_void_p), N, K)
    return codes


def dequant(wq, scale, zero, g: int) -> np.ndarray:
    """Exact fp64 W[N, K] = (code - zero) * scale."""
    lib = _load()
    wq, pw = _c(wq, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    N, K8 = wq.shape
    K = K8 * 8
    assert scale.shape == (N, K // g) and zero.shape == (N, K // g)
    w = np.empty((N, K), np.float64)
    lib.oracle_dequant(pw, ps, pz, w.ctypes.data_as(ctypes.c_void_p), N, K, g)
    return w


def gemv(x, wq, scale, zero, g: int) -> np.ndarray:
    """fp64 y[M, N] = x[M, K] . dequant(Wq)^T (x given as bf16 bits)."""
    lib = _load()
    x, px = _c(x, np.uint16)
    wq, pw = _c(wq, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    M, K = x.shape
    N = wq.shape[0]
    assert wq.shape == (N, K // 8) and scale.shape == (N, K // g)
    y = np.empty((M, N), np.float64)
    lib.oracle_gemv(px, pw, ps, pz, y.ctypes.data_as(ctypes.c_void_p), M, N, K, g)
    return y


def max_threads() -> int:
    """Host threads gemv(..., threads=) can use (1 if built without OpenMP)."""
    return int(_load().oracle_max_threads())


def gemv_parallel(x, wq, scale, zero, g: int, threads: int = 0) -> np.ndarray:
    """gemv with the output rows shared among `threads` host threads (0: all
    of them); element for element the same fp64 sums as gemv."""
    lib = _load()
    x, px = _c(x, np.uint16)
    wq, pw = _c(wq, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    M, K = x.shape
    N = wq.shape[0]
    assert wq.shape == (N, K // 8) and scale.shape == (N, K // g)
    y = np.empty((M, N), np.float64)
    lib.oracle_gemv_parallel(px, pw, ps, pz, y.ctypes.data_as(ctypes.c_void_p), M, N, K, g,
                             int(threads) if threads else max_threads())
    return y


def gemv_rows(x, wq, scale, zero, g: int, rows) -> np.ndarray:
    """fp64 y[M, len(rows)] for the listed output rows only."""
    lib = _load()
    x, px = _c(x, np.uint16)
    wq, pw = _c(wq, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    rows, pr = _c(rows, np.int64)
    M, K = x.shape
    y = np.empty((M, rows.size), np.float64)
    lib.oracle_gemv_rows(px, pw, ps, pz, pr, rows.size,
                         y.ctypes.data_as(ctypes.c_void_p), M, K, g)
    return y


def swiglu(gate, up) -> np.ndarray:
    """bf16 bits h = RNE(silu(gate) * up), fp64 arithmetic."""
    lib = _load()
    gate, pg = _c(gate, np.uint16)
    up, pu = _c(up, np.uint16)
    assert gate.shape == up.shape
    h = np.empty(gate.shape, np.uint16)
    lib.oracle_swiglu(pg, pu, h.ctypes.data_as(ctypes.c_void_p), gate.size)
    return h


def moe_gemv(x, ids, route_w, wq, scale, zero, g: int, x_per_slot: bool = False):
    """Expert-indexed GEMV.  wq [E, N, K/8], scale/zero [E, N, K/g],
    ids int32 [M, topk]; x [M, K] or (x_per_slot) [M, topk, K].
    Returns fp64 [M, topk, N] (route_w None) or [M, N] (routed sum)."""
    lib = _load()
    x, px = _c(x, np.uint16)
    ids, pi = _c(ids, np.int32)
    wq, pw = _c(wq, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    E, N, K8 = wq.shape
    K = K8 * 8
    M, topk = ids.shape
    if route_w is None:
        pr = None
        y = np.empty((M, topk, N), np.float64)
    else:
        route_w, pr = _c(route_w, np.float32)
        y = np.empty((M, N), np.float64)
    rc = lib.oracle_moe_gemv(px, int(bool(x_per_slot)), pi, pr, pw, ps, pz,
                             y.ctypes.data_as(ctypes.c_void_p), M, topk, E, N, K, g)
    if rc != 0:
        raise ValueError("expert id out of range")
    return y


def moe_ffn(x, ids, route_w, gate, up, down, g: int):
    """Routed SwiGLU FFN chain.  gate/up/down are (wq, scale, zero) triples:
    gate/up wq [E, F, H/8], down wq [E, H, F/8].  Returns a dict with the fp64
    output [M, H] and the bf16 intermediates (gate, up, h) [M, topk, F]."""
    lib = _load()
    x, px = _c(x, np.uint16)
    ids, pi = _c(ids, np.int32)
    route_w, pr = _c(route_w, np.float32)
    arrs = []
    ptrs = []
    for (wq, s, z) in (gate, up, down):
        for a, dt in ((wq, np.uint32), (s, np.uint16), (z, np.uint8)):
            a, p = _c(a, dt)
            arrs.append(a)
            ptrs.append(p)
    E, F, H8 = arrs[0].shape
    H = H8 * 8
    M, topk = ids.shape
    gate_bf = np.empty((M, topk, F), np.uint16)
    up_bf = np.empty((M, topk, F), np.uint16)
    h_bf = np.empty((M, topk, F), np.uint16)
    d = np.empty((M, topk, H), np.float64)
    out = np.empty((M, H), np.float64)
    rc = lib.oracle_moe_ffn(px, pi, pr, *ptrs,
                            gate_bf.ctypes.data_as(ctypes.c_void_p),
                            up_bf.ctypes.data_as(ctypes.c_void_p),
                            h_bf.ctypes.data_as(ctypes.c_void_p),
                            d.ctypes.data_as(ctypes.c_void_p),
                            out.ctypes.data_as(ctypes.c_void_p),
                            M, topk, E, H, F, g)
    if rc != 0:
        raise ValueError("expert id out of range")
    return {"out": out, "gate": gate_bf, "up": up_bf, "h": h_bf, "d": d}


# ---- ~3-bit expert weights (int3_oracle.c) ---------------------------------

def int3_row_words(K: int) -> int:
    """32-bit words per packed INT3 row of K codes (K % 128 == 0)."""
    if K % 128:
        raise ValueError("INT3 rows need K % 128 == 0")
    return K // 128 * 12


def pack3(codes) -> np.ndarray:
    """codes uint8 [N, K] (0..7) -> INT3 words uint32 [N, 3K/32]."""
    lib = _load()
    codes, pc = _c(codes, np.uint8)
    N, K = codes.shape
    wq3 = np.empty((N, int3_row_words(K)), np.uint32)
    lib.oracle3_pack(pc, wq3.ctypes.data_as(ctypes.c_void_p), N, K)
    return wq3


def unpack3(wq3, K: int) -> np.ndarray:
    lib = _load()
    wq3, pw = _c(wq3, np.uint32)
    N = wq3.shape[0]
    assert wq3.shape[1] == int3_row_words(K)
    codes = np.empty((N, K), np.uint8)
    lib.oracle3_unpack(pw, codes.ctypes.data_as(ctypes.c_void_p), N, K)
    return codes


def dequant3(wq3, scale, zero, g: int) -> np.ndarray:
    """fp64 [N, K] = (code - zero) * scale for INT3 words [N, 3K/32]."""
    lib = _load()
    wq3, pw = _c(wq3, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    N = wq3.shape[0]
    K = wq3.shape[1] // 12 * 128
    w = np.empty((N, K), np.float64)
    lib.oracle3_dequant(pw, ps, pz, w.ctypes.data_as(ctypes.c_void_p), N, K, g)
    return w


def gemv3(x, wq3, scale, zero, g: int) -> np.ndarray:
    """fp64 y [M, N] = x [M, K] (bf16 bits) times the INT3 matrix."""
    lib = _load()
    x, px = _c(x, np.uint16)
    wq3, pw = _c(wq3, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    M, K = x.shape
    N = wq3.shape[0]
    assert wq3.shape[1] == int3_row_words(K)
    y = np.empty((M, N), np.float64)
    lib.oracle3_gemv(px, pw, ps, pz, y.ctypes.data_as(ctypes.c_void_p), M, N, K, g)
    return y


def moe_gemv3(x, ids, route_w, wq3, scale, zero, g: int, x_per_slot: bool = False,
              allow_bad_ids: bool = False):
    """Expert-indexed GEMV over INT3 experts: wq3 [E, N, 3K/32], scale/zero
    [E, N, K/g], ids int32 [M, topk]; x [M, K] or (x_per_slot) [M, topk, K].
    Returns fp64 [M, topk, N] (route_w None; zero rows for invalid ids) or
    [M, N] (routed sum, invalid ids skipped).  Invalid ids raise ValueError
    unless allow_bad_ids."""
    lib = _load()
    x, px = _c(x, np.uint16)
    ids, pi = _c(ids, np.int32)
    wq3, pw = _c(wq3, np.uint32)
    scale, ps = _c(scale, np.uint16)
    zero, pz = _c(zero, np.uint8)
    E, N, W3 = wq3.shape
    K = W3 // 12 * 128
    M, topk = ids.shape
    if route_w is None:
        pr = None
        y = np.empty((M, topk, N), np.float64)
    else:
        route_w, pr = _c(route_w, np.float32)
        y = np.empty((M, N), np.float64)
    rc = lib.oracle3_moe_gemv(px, int(bool(x_per_slot)), pi, pr, pw, ps, pz,
                              y.ctypes.data_as(ctypes.c_void_p), M, topk, E, N, K, g)
    if rc != 0 and not allow_bad_ids:
        raise ValueError("expert id out of range")
    return y


def moe_ffn3(x, ids, route_w, gate, up, down, g: int):
    """Routed SwiGLU FFN chain over INT3 experts: gate/up wq [E, F, 3H/32],
    down wq [E, H, 3F/32]; the same result dict as moe_ffn."""
    lib = _load()
    x, px = _c(x, np.uint16)
    ids, pi = _c(ids, np.int32)
    route_w, pr = _c(route_w, np.float32)
    arrs = []
    ptrs = []
    for (wq, s, z) in (gate, up, down):
        for a, dt in ((wq, np.uint32), (s, np.uint16), (z, np.uint8)):
            a, p = _c(a, dt)
            arrs.append(a)
            ptrs.append(p)
    E, F, _ = arrs[0].shape
    M, H = x.shape
    assert arrs[0].shape[2] == int3_row_words(H) and arrs[6].shape == (E, H, int3_row_words(F))
    topk = ids.shape[1]
    gate_bf = np.empty((M, topk, F), np.uint16)
    up_bf = np.empty((M, topk, F), np.uint16)
    h_bf = np.empty((M, topk, F), np.uint16)
    d = np.empty((M, topk, H), np.float64)
    out = np.empty((M, H), np.float64)
    rc = lib.oracle3_moe_ffn(px, pi, pr, *ptrs,
                             gate_bf.ctypes.data_as(ctypes.c_void_p),
                             up_bf.ctypes.data_as(ctypes.c_void_p),
                             h_bf.ctypes.data_as(ctypes.c_void_p),
                             d.ctypes.data_as(ctypes.c_void_p),
                             out.ctypes.data_as(ctypes.c_void_p),
                             M, topk, E, H, F, g)
    if rc != 0:
        raise ValueError("expert id out of range")
    return {"out": out, "gate": gate_bf, "up": up_bf, "h": h_bf, "d": d}
