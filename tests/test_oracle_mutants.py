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
from tests import test_oracle_int3 as pins3

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "w4a16_oracle.c")
SRC3 = os.path.join(os.path.dirname(oracle_mod.__file__), "int3_oracle.c")

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


# slips in the ~3-bit format and its chain (int3_oracle.c)
MUTANTS3 = [
    ("int3_halves_swapped", [("16 * (r / 5) + 3 * (r % 5)", "16 * (1 - r / 5) + 3 * (r % 5)")]),
    ("int3_field_width_4", [("16 * (r / 5) + 3 * (r % 5)", "16 * (r / 5) + 4 * (r % 5) - (r % 5 == 4)")]),
    ("int3_leftover_bits_swapped", [("(i == 30) ? 15 : 31", "(i == 30) ? 31 : 15")]),
    ("int3_leftover_bit_order", [("*word = first + j;", "*word = first + 2 - j;")]),
    ("int3_chunk_stride", [("int64_t first = 12 * b + 3 * c;", "int64_t first = 12 * b + 3 * (3 - c);")]),
    ("int3_words_of_a_chunk", [("*word = first + i / 10;", "*word = first + (i / 10 + 1) % 3;")]),
    ("int3_zero_dropped", [("((double)oracle3_code(wq3, K, n, k) - z) * s", "((double)oracle3_code(wq3, K, n, k)) * s")]),
    ("int3_group_index", [("scale[n * G + k / g]", "scale[n * G + (k / 128) % G]")]),
    ("int3_expert_stride", [("wq_down + e * H * wf", "wq_down + e * H * wh")]),
    ("int3_chain_route_weight", [("out[t * H + n] += (double)route_w[t * topk + j] * acc;",
                                  "out[t * H + n] += (double)route_w[j] * acc;")]),
    ("int3_gemv_route_weight", [("y[t * N + n] += (double)route_w[t * topk + j] * acc;",
                                 "y[t * N + n] += (double)route_w[j] * acc;")]),
    ("int3_gemv_expert_stride", [("wq3 + e * N * wpr, scale + e * N * G", "wq3 + e * wpr, scale + e * N * G")]),
    ("int3_gemv_scale_stride", [("scale + e * N * G, zero + e * N * G", "scale + e * G, zero + e * N * G")]),
    ("int3_gemv_slot_input", [("const uint16_t* xin = x_per_slot ? x + (t * topk + j) * K : x + t * K;",
                               "const uint16_t* xin = x_per_slot ? x + t * K : x + t * K;")]),
]


def _pin_functions():
    out = []
    for name, fn in sorted(list(vars(pins).items()) + list(vars(pins3).items()), key=lambda kv: kv[0]):
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


@pytest.mark.parametrize("name,edits,target",
                         [(n, e, SRC) for n, e in MUTANTS] + [(n, e, SRC3) for n, e in MUTANTS3],
                         ids=[m[0] for m in MUTANTS] + [m[0] for m in MUTANTS3])
def test_pins_catch_mutant(tmp_path, name, edits, target):
    sources = []
    for i, path in enumerate((SRC, SRC3)):
        src = open(path).read()
        if path == target:
            for old, new in edits:
                assert old in src, "mutation site not found: %r" % old
                src = src.replace(old, new)
        out = tmp_path / ("mutant%d.c" % i)
        out.write_text(src)
        sources.append(str(out))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off"] + sources +
                   ["-o", str(lib), "-lm"], check=True)
    oracle_mod.build()
    with oracle_mod.using_library(str(lib)):
        failed = _run_pins()
    assert failed, "no pin caught mutant %s" % name


def test_unmutated_oracle_passes_every_pin():
    oracle_mod.build()
    assert _run_pins() == []
