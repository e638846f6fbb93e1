"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Every mutant is a text edit of ``oracle/nc_oracle.c`` compiled into a temporary
library on the CPU; the shipped oracle is never touched.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "nc_oracle.c")

MUTANTS = {
    "window off by one (one key too few)":
        ("long lo = i - W + 1 < 0 ? 0 : i - W + 1;\n                    double l =",
         "long lo = i - W + 2 < 0 ? 0 : i - W + 2;\n                    if (lo > i) lo = i;\n                    double l ="),
    "scale dropped from the scores": ("        s *= scale;\n        p[j - lo] = s;", "        p[j - lo] = s;"),
    "max dropped from lse": ("double lse = M + log(sum);", "double lse = log(sum);"),
    "scale dropped from dq": ("dq[idx_bthd(b, i, h, d, T, H, D)] += scale * ds *", "dq[idx_bthd(b, i, h, d, T, H, D)] += ds *"),
    "dk uses k instead of q": ("scale * ds * q[idx_bthd(b, i, h, d, T, H, D)]", "scale * ds * k[idx_bthd(b, i, h, d, T, H, D)]"),
    "ds sign flipped": ("p[t] * (dp[t] - delta)", "p[t] * (delta - dp[t])"),
    "dv weighted by ds": ("+= p[t] * dO[", "+= ds * dO["),
    "Delta omitted": ("delta += p[j - lo] * s;", "delta += 0.0 * s;"),
    "decode window one key short": ("long lo = L - W;", "long lo = L - W + 1;"),
    "decode reads value of the key row": ("j < L; ++j) acc += p[j - lo] * vc[", "j < L; ++j) acc += p[j - lo] * kc["),
    "prefill query one position late": ("long i = L - Tq + t;", "long i = L - Tq + t + 1;\n                    if (i > L - 1) i = L - 1;"),
    "prefill window one key short": (": i - window + 1;\n                    const double* qrow",
                                     ": i - window + 2;\n                    const double* qrow"),
    "prefill reads value of the key row": ("j <= i; ++j) acc += p[j - lo] * vc[", "j <= i; ++j) acc += p[j - lo] * kc["),
    "rotary sine sign flipped": ("y[idx_bthd(b, t, h, i, T, H, D)] = x1 * c - x2 * s;",
                                 "y[idx_bthd(b, t, h, i, T, H, D)] = x1 * c + x2 * s;"),
    "rotary pairs neighbouring dimensions": ("double x2 = x[idx_bthd(b, t, h, i + half, T, H, D)];",
                                             "double x2 = x[idx_bthd(b, t, h, (i + 1) % D, T, H, D)];"),
    "rotary transpose not applied": ("if (inverse) s = -s;", "(void)inverse;"),
    "rotary position off by one": ("double c = cosv[(size_t)t * half + i];\n                    double s = sinv[(size_t)t * half + i];",
                                   "double c = cosv[(size_t)(t + 1 < T ? t + 1 : t) * half + i];\n                    double s = sinv[(size_t)(t + 1 < T ? t + 1 : t) * half + i];"),
    "bf16 rounding truncates": ("x[i] = ldexp(nearbyint(ldexp(v, -ue)), ue);", "x[i] = ldexp(trunc(ldexp(v, -ue)), ue);"),
    "bf16 rounding keeps a bit too many": ("int ue = e - 8;", "int ue = e - 9;"),
    "rotary float32 turn without the fused multiply-add": ("(double)fmaf(x1, c, -p2s);", "(double)(x1 * c - p2s);"),
    "rotary float32 turn sine sign flipped": ("(double)fmaf(x1, s, p2c);", "(double)fmaf(-x1, s, p2c);"),
}

PIN_SUITE = [
    (pins.test_hand_worked_example, {}),
    (pins.test_brute_force_tiny, {"T": 8, "D": 4, "window": 3}),
    (pins.test_matches_torch_sdpa_fp64, {"T": 33, "D": 16, "window": 5}),
    (pins.test_backward_matches_finite_differences, {"window": 3}),
    (pins.test_gradient_sums, {"window": 3}),
    (pins.test_decode_equals_last_forward_row, {"window": 5}),
    (pins.test_prefill_rows_equal_forward_rows, {"window": 4}),
    (pins.test_prefill_brute_force_tiny, {"Tq": 3, "window": 2}),
    (pins.test_rotary_matches_complex_rotation, {}),
    (pins.test_rotary_position_zero_is_identity, {}),
    (pins.test_rotary_preserves_norms_and_the_transpose_turns_back, {}),
    (pins.test_rotary_attention_gradients_match_finite_differences, {"window": 3}),
    (pins.test_round_bf16_hand_values, {}),
    (pins.test_round_bf16_matches_torch_float32, {}),
    (pins.test_rotary_f32_matches_a_numpy_restatement, {}),
    (pins.test_rotary_f32_is_the_turn_to_float_precision, {}),
]


def _caught(lib) -> list:
    caught = []
    for fn, kw in PIN_SUITE:
        try:
            fn(lib, **kw)
        except AssertionError:
            caught.append(fn.__name__)
    return caught


def test_unmutated_copy_passes_every_pin(tmp_path):
    out = tmp_path / "lib_clean.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11", SRC, "-o", str(out), "-lm"])
    assert _caught(oracle.OracleLib(str(out))) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    out = tmp_path / "lib_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mutated), "-o", str(out), "-lm"])
    caught = _caught(oracle.OracleLib(str(out)))
    assert caught, f"no pin caught mutant: {name}"
