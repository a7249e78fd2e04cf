"""Seeded synthetic inputs for the W4A16 GEMV workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no unpacking, dequantisation or products), so both the
CUDA path and the CPU oracle can take their inputs from it.

Recipe (the workload descriptions the library is measured on):
  x       bf16 ~ N(0, 1), rounded to nearest-even from binary32
  codes   uniform integers 0..15.  Eight independent uniform 4-bit codes
          packed into one 32-bit word form a uniform 32-bit word, so packed
          weights are drawn directly as uniform uint32 words
  scale   bf16 ~ U[0.005, 0.02], one per (row, group)
  zero    uint8, either the constant 8 or uniform integers 6..10
  int3    (~3-bit expert weights) codes uniform 0..7; every bit of a packed
          INT3 chunk belongs to exactly one code, so packed words are again
          uniform uint32 (3 K / 32 words per row); zero points the constant 4
          or uniform integers 2..6 (the INT4 spread of five values around the
          middle of the 3-bit range); scales as for INT4
  routing per token, top-k expert ids uniform without replacement, and
          route weights = softmax of top-k N(0, 1) logits (fp32)
Every tensor has its own stream: numpy PCG64 seeded with (seed, tag).
"""
from __future__ import annotations

import numpy as np

_TAGS = {"x": 1, "wq": 2, "scale": 3, "zero": 4, "codes": 5, "ids": 6,
         "logits": 7, "h": 8, "misc": 9}


def rng(seed: int, tag: str, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), _TAGS[tag], int(sub)]))


def f32_to_bf16_bits(a) -> np.ndarray:
    """binary32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(seed: int, shape, sub: int = 0) -> np.ndarray:
    return f32_to_bf16_bits(rng(seed, "x", sub).standard_normal(shape, dtype=np.float32))


def packed_weights(seed: int, N: int, K: int, sub: int = 0) -> np.ndarray:
    assert K % 8 == 0
    return rng(seed, "wq", sub).integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)


def codes(seed: int, N: int, K: int, sub: int = 0) -> np.ndarray:
    return rng(seed, "codes", sub).integers(0, 16, size=(N, K), dtype=np.uint8)


def scales(seed: int, N: int, G: int, sub: int = 0) -> np.ndarray:
    r = rng(seed, "scale", sub).uniform(0.005, 0.02, size=(N, G)).astype(np.float32)
    return f32_to_bf16_bits(r)


def zeros(seed: int, N: int, G: int, mode: str = "const8", sub: int = 0) -> np.ndarray:
    if mode == "const8":
        return np.full((N, G), 8, np.uint8)
    if mode == "uniform6to10":
        return rng(seed, "zero", sub).integers(6, 11, size=(N, G), dtype=np.uint8)
    if mode == "const4":
        return np.full((N, G), 4, np.uint8)
    if mode == "uniform2to6":
        return rng(seed, "zero", sub).integers(2, 7, size=(N, G), dtype=np.uint8)
    raise ValueError(mode)


def dense_problem(M: int, N: int, K: int, g: int = 128, zero_mode: str = "const8",
                  seed: int = 0, sub: int = 0) -> dict:
    """One W4A16 GEMV problem: x [M,K] bf16 bits, wq [N,K/8] u32,
    scale [N,K/g] bf16 bits, zero [N,K/g] u8."""
    G = K // g
    return {
        "x": activations(seed, (M, K), sub),
        "wq": packed_weights(seed, N, K, sub),
        "scale": scales(seed, N, G, sub),
        "zero": zeros(seed, N, G, zero_mode, sub),
        "M": M, "N": N, "K": K, "g": g,
    }


def routing(seed: int, M: int, topk: int, E: int, sub: int = 0):
    """ids int32 [M, topk] (distinct per token) and fp32 route weights."""
    r = rng(seed, "ids", sub)
    ids = np.stack([r.choice(E, size=topk, replace=False) for _ in range(M)]).astype(np.int32)
    logits = rng(seed, "logits", sub).standard_normal((M, topk))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids.reshape(M, topk), w


def expert_bank(seed: int, E: int, N: int, K: int, g: int = 128,
                zero_mode: str = "uniform6to10", sub: int = 0):
    """E stacked expert matrices: wq [E,N,K/8], scale/zero [E,N,K/g]."""
    G = K // g
    wq = packed_weights(seed, E * N, K, sub).reshape(E, N, K // 8)
    s = scales(seed, E * N, G, sub).reshape(E, N, G)
    z = zeros(seed, E * N, G, zero_mode, sub).reshape(E, N, G)
    return wq, s, z


def moe_problem(M: int, E: int = 64, H: int = 2304, F: int = 1024, topk: int = 8,
                g: int = 128, seed: int = 0) -> dict:
    """Routed SwiGLU FFN: gate/up experts [E, F, H], down experts [E, H, F]."""
    ids, route_w = routing(seed, M, topk, E)
    return {
        "x": activations(seed, (M, H)),
        "ids": ids, "route_w": route_w,
        "gate": expert_bank(seed, E, F, H, g, sub=1),
        "up": expert_bank(seed, E, F, H, g, sub=2),
        "down": expert_bank(seed, E, H, F, g, sub=3),
        "M": M, "E": E, "H": H, "F": F, "topk": topk, "g": g,
    }


def packed_weights3(seed: int, N: int, K: int, sub: int = 0) -> np.ndarray:
    """Uniform INT3 words [N, 3K/32] (uniform 3-bit codes)."""
    assert K % 128 == 0
    return rng(seed, "wq", sub).integers(0, 2**32, size=(N, 3 * K // 32), dtype=np.uint32)


def codes3(seed: int, N: int, K: int, sub: int = 0) -> np.ndarray:
    return rng(seed, "codes", sub).integers(0, 8, size=(N, K), dtype=np.uint8)


def expert_bank3(seed: int, E: int, N: int, K: int, g: int = 128,
                 zero_mode: str = "uniform2to6", sub: int = 0):
    """E stacked INT3 expert matrices: wq [E,N,3K/32], scale/zero [E,N,K/g]."""
    G = K // g
    wq = packed_weights3(seed, E * N, K, sub).reshape(E, N, 3 * K // 32)
    s = scales(seed, E * N, G, sub).reshape(E, N, G)
    z = zeros(seed, E * N, G, zero_mode, sub).reshape(E, N, G)
    return wq, s, z


def moe_problem3(M: int, E: int = 64, H: int = 2304, F: int = 1024, topk: int = 8,
                 g: int = 128, seed: int = 0) -> dict:
    """Routed SwiGLU FFN over INT3 experts (shapes as moe_problem)."""
    ids, route_w = routing(seed, M, topk, E)
    return {
        "x": activations(seed, (M, H)),
        "ids": ids, "route_w": route_w,
        "gate": expert_bank3(seed, E, F, H, g, sub=1),
        "up": expert_bank3(seed, E, F, H, g, sub=2),
        "down": expert_bank3(seed, E, H, F, g, sub=3),
        "M": M, "E": E, "H": H, "F": F, "topk": topk, "g": g,
    }
