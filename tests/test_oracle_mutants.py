"""Plants plausible mistakes in copies of the CPU oracle and checks that the
pins in test_oracle.py catch every one (no GPU).

Each mutant is the oracle's C source with one textual edit, compiled with
gcc into a temporary directory; the pins are then run against it through
``oracle.using_library``.  The real oracle is never modified.
"""
import inspect
import os
import subprocess

import pytest

import oracle as oracle_mod
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "w4a16_oracle.c")

# (name, text to replace, replacement, how many occurrences must exist)
MUTANTS = [
    ("nibble_order_reversed_everywhere",
     [("<< (4 * i)", "<< (4 * (7 - i))"), (">> (4 * (k % 8))", ">> (4 * (7 - k % 8))")]),
    ("nibble_pairs_swapped_in_unpack", [(">> (4 * (k % 8))", ">> (4 * ((k % 8) ^ 1))")]),
    ("zero_sign_flipped", [("((double)oracle_code(wq, K, n, k) - z) * s",
                            "(z - (double)oracle_code(wq, K, n, k)) * s")]),
    ("zero_dropped", [("((double)oracle_code(wq, K, n, k) - z) * s",
                       "((double)oracle_code(wq, K, n, k)) * s")]),
    ("group_index_modulo", [("scale[n * G + k / g]", "scale[n * G + k % G]"),
                            ("zero[n * G + k / g]", "zero[n * G + k % G]")]),
    ("scale_transposed", [("scale[n * G + k / g]", "scale[(k / g) * G + n % G]")]),
    ("bf16_double_rounding", [("nearbyint(ldexp(a, -qexp))", "nearbyint(ldexp((double)(float)a, -qexp))")]),
    ("bf16_truncates", [("nearbyint(ldexp(a, -qexp))", "floor(ldexp(a, -qexp))")]),
    ("gemv_drops_first_term", [("acc = 0.0;\n            for (int64_t k = 0; k < K; ++k)",
                                "acc = 0.0;\n            for (int64_t k = 1; k < K; ++k)")]),
    ("gemv_x_transposed", [("x[m * K + k]", "x[(k * M + m) % (M * K)]")]),
    ("swiglu_sign", [("exp(-a)", "exp(a)")]),
    ("moe_expert_offset", [("wq + e * N * (K / 8)", "wq + e * (K / 8)")]),
    ("moe_route_weight_index", [("(double)route_w[t * topk + j] * acc;\n                else",
                                 "(double)route_w[j] * acc;\n                else"),
                                ("(double)route_w[t * topk + j] * acc;\n            }",
                                 "(double)route_w[j] * acc;\n            }")]),
    ("moe_chain_skips_h_rounding", [("oracle_swiglu(gate_bf, up_bf, h_bf, S * F);",
                                     "oracle_swiglu(gate_bf, up_bf, h_bf, S * F); (void)0;\n"
                                     "    for (int64_t i = 0; i < S * F; ++i) h_bf[i] = gate_bf[i];")]),
]


def _pin_functions():
    out = []
    for name, fn in sorted(vars(pins).items()):
        if not name.startswith("test_") or not callable(fn):
            continue
        params = inspect.signature(fn).parameters
        marks = getattr(fn, "pytestmark", [])
        args_sets = [()]
        for mk in marks:
            if mk.name == "parametrize":
                args_sets = list(mk.args[1])
        out.append((name, fn, list(params), args_sets))
    return out


def _run_pins():
    failed = []
    for name, fn, params, args_sets in _pin_functions():
        for args in args_sets:
            if not isinstance(args, tuple):
                args = (args,)
            kwargs = {}
            extra = [p for p in params if p != "oracle"]
            kwargs.update(dict(zip(extra, args)))
            if "oracle" in params:
                kwargs["oracle"] = oracle_mod
            try:
                fn(**kwargs)
            except (AssertionError, ValueError):
                failed.append(name)
                break
    return failed


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, "mutation site not found: %r" % old
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(path), "-o", str(lib), "-lm"], check=True)
    oracle_mod.build()
    with oracle_mod.using_library(str(lib)):
        failed = _run_pins()
    assert failed, "no pin caught mutant %s" % name


def test_unmutated_oracle_passes_every_pin():
    oracle_mod.build()
    assert _run_pins() == []
