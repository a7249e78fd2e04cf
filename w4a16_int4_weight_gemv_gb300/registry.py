"""Kernel registry: every operation, its variants, and the variant shipped.

The local-kimi README (technical-detail section, on how its kernels are
organised) keeps each decode kernel behind a registry: one reference
implementation per operation plus any number of variants, picked by an
environment variable, with every variant checked against the reference and
a test that pins what an ordinary run gets -- after a run had silently used
the slow path while the benchmarks selected the fast one.

Here every registered variant is a CUDA path of this library; there is no
CPU path to fall back to.  The reference role is played by the fp64 oracle,
which only the tests use: tests/test_gpu_registry.py runs every variant of
every operation against it, tests/test_registry.py pins the defaults below.

Selection: ``W4A16_KERNELS="op=variant,op=variant"`` overrides the default
of each named operation, e.g. ``W4A16_KERNELS=w4a16_dense=warp_mma``.
Unknown operations or variants raise ValueError (a typo must not quietly
select the default).
"""
from __future__ import annotations

import os

from . import binding


def _dense(kernel_id: int):
    def run(x, wq, scale, zero, g, **kw):
        return binding.w4a16_gemv(x, wq, scale, zero, g, kernel_id=kernel_id, **kw)
    return run


def _grouped(kernel_id: int):
    def run(x, expert_ids, wq, scale, zero, g, **kw):
        return binding.w4a16_moe_gemv(x, expert_ids, wq, scale, zero, g, kernel_id=kernel_id, **kw)
    return run


def _ffn(fused: bool):
    def run(x, expert_ids, route_w, gate, up, down, g, **kw):
        return binding.moe_ffn(x, expert_ids, route_w, gate, up, down, g, fused=fused, **kw)
    return run


# operation -> variant -> callable (same signature within an operation)
OPS = {
    # y[M, N] = x[M, K] . dequant(Wq, scale, zero)^T
    "w4a16_dense": {
        "planned": _dense(0),    # the library's choice per shape (fp16 warp MMA where it applies)
        "cuda_core": _dense(1),  # subnormal-float CUDA-core kernel, M <= 2
        "warp_mma": _dense(2),   # bf16 mma.sync kernel, M <= 16
        "tcgen05": _dense(3),    # tensor-core (TMEM) kernel, g % 128 == 0
        "fp16_mma": _dense(4),   # fp16 mma.sync kernel, per-warp cp.async rings, M <= 16, g == 128
    },
    # per-slot products of the routed experts, or their routed sum
    "w4a16_grouped": {
        "planned": _grouped(0),   # the library's choice (fp16_mma where it applies, else tma)
        "tma": _grouped(2),       # bf16 mma.sync expert kernel, TMA rings, M*topk <= 256
        "fp16_mma": _grouped(4),  # fp16 mma.sync expert kernel, routed sums in shared memory, M*topk <= 32
    },
    # the same over an ~3-bit (INT3) expert bank
    "w3a16_grouped": {
        "fp16_mma": binding.w3a16_moe_gemv,
    },
    # routed SwiGLU expert FFN
    "w4a16_ffn": {
        "fused": _ffn(True),     # w4a16_moe_ffn: gate/up launch with the SwiGLU epilogue, down launch with routed sums
        "chain": _ffn(False),    # single-purpose calls: gate, up, SwiGLU, down with routed sum
    },
    # the same FFN over ~3-bit (INT3) expert banks
    "w3a16_ffn": {
        "fp16_mma": binding.w3a16_moe_ffn,
    },
}

# what an ordinary run gets
DEFAULTS = {
    "w4a16_dense": "planned",
    "w4a16_grouped": "planned",
    "w3a16_grouped": "fp16_mma",
    "w4a16_ffn": "fused",
    "w3a16_ffn": "fp16_mma",
}

ENV = "W4A16_KERNELS"


def selection(env: str | None = None) -> dict:
    """Variant per operation: DEFAULTS overridden by W4A16_KERNELS (or `env`)."""
    text = os.environ.get(ENV, "") if env is None else env
    sel = dict(DEFAULTS)
    for item in filter(None, (s.strip() for s in text.split(","))):
        if "=" not in item:
            raise ValueError("%s: expected op=variant, got %r" % (ENV, item))
        op, var = (s.strip() for s in item.split("=", 1))
        if op not in OPS:
            raise ValueError("%s: unknown operation %r (known: %s)" % (ENV, op, ", ".join(OPS)))
        if var not in OPS[op]:
            raise ValueError("%s: unknown variant %r of %s (known: %s)"
                             % (ENV, var, op, ", ".join(OPS[op])))
        sel[op] = var
    return sel


def get(op: str, env: str | None = None):
    """The callable selected for `op`."""
    return OPS[op][selection(env)[op]]


def variants(op: str) -> list:
    return list(OPS[op])
