"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins in test_oracle.py catch every one of them.

Each mutant is compiled from ``oracle/kda_ref.c`` with one textual change into
a temporary directory; the oracle module is pointed at it with
``oracle.use_library`` and the pins are run.  A mutant that no pin rejects
means the pins leave that part of the oracle unchecked.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_ref.c")
# linked unchanged into every mutant library (the binding resolves its symbols)
BWD_SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_ref_bwd.c")

OUT_BLOCK = """    /* o_t = scale * q_t^T S (the updated S) */
    for (int j = 0; j < V; ++j) ot[j] = 0.0;
    for (int i = 0; i < K; ++i) {
      const double qi = qt[i];
      const double *Si = S + (size_t)i * V;
      for (int j = 0; j < V; ++j) ot[j] += qi * Si[j];
    }
    for (int j = 0; j < V; ++j) ot[j] *= J->scale;
"""
UPD_MARK = "    /* S = S' + beta_t k_t (outer) residual */\n"


def _read_before_write(src):
    assert src.count(OUT_BLOCK) == 1 and src.count(UPD_MARK) == 1
    src = src.replace(OUT_BLOCK, "")
    return src.replace(UPD_MARK, OUT_BLOCK + UPD_MARK)


def _sub(old, new):
    def f(src):
        assert src.count(old) == 1, old
        return src.replace(old, new)
    return f


MUTANTS = {
    "residual_sign": _sub("r[j] -= ki * Si[j];", "r[j] += ki * Si[j];"),
    "beta_dropped": _sub("const double c = bt * kt[i];", "const double c = kt[i];"),
    "decay_sign": _sub("const double e = exp(gt[i]);", "const double e = exp(-gt[i]);"),
    "gate_on_value_axis": _sub("for (int j = 0; j < V; ++j) Si[j] *= e;",
                               "for (int j = 0; j < V; ++j) Si[j] *= exp(gt[j % K]) + 0 * e;"),
    "read_before_write": _read_before_write,
    "output_uses_k": _sub("const double qi = qt[i];", "const double qi = kt[i];"),
    "scale_dropped": _sub("ot[j] *= J->scale;", "ot[j] *= 1.0;"),
    "no_reset_at_run_start": _sub(
        "if (seen_run) memset(S, 0, sizeof(double) * (size_t)K * V);", "(void)seen_run;"),
    "padding_keeps_run": _sub("      prev = 0;\n      continue;", "      continue;"),
    "initial_state_ignored": _sub("if (J->initial_state)\n", "if (0 && J->initial_state)\n"),
    "conv_taps_reversed": _sub("w[(size_t)c * W + (W - 1 - i)]", "w[(size_t)c * W + i]"),
    "conv_crosses_segments": _sub("if (tt < run_start) break;", "if (tt < 0) break;"),
    "silu_sign": _sub("yt[c] = z / (1.0 + exp(-z));", "yt[c] = z / (1.0 + exp(z));"),
    "l2norm_no_sqrt": _sub("const double inv = 1.0 / sqrt(ss + eps);",
                           "const double inv = 1.0 / (ss + eps);"),
}

PINS = [
    P.test_zero_gate_orthonormal_keys_accumulate_exactly,
    P.test_zero_gate_orthogonal_keys_fractional_beta,
    P.test_large_negative_gate_decays_to_single_token,
    P.test_gate_minus_five_decays_by_e5_per_token,
    P.test_per_channel_gate_scales_key_rows,
    lambda: P.test_write_then_read_returns_v(-5.0),
    P.test_single_token_closed_form,
    P.test_two_tokens_hand_expanded,
    P.test_packed_equals_separate_runs_bitwise,
    P.test_padding_ends_run_and_keeps_initial_state_for_first_run,
    P.test_all_padding_row_returns_initial_state,
    lambda: P.test_matches_independent_transcriptions((2, 5, 3, 3, 2), True),
    lambda: P.test_matches_independent_transcriptions((1, 9, 2, 4, 5), False),
    P.test_conv_identity_tap_is_silu,
    P.test_conv_matches_library_conv1d,
    P.test_conv_segment_aware_equals_per_segment_library_conv,
    P.test_l2norm_closed_form,
]


def _caught(path):
    with oracle.use_library(path):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name):
    src = open(SRC).read()
    mutated = MUTANTS[name](src)
    assert mutated != src
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "libm.so")
        open(c, "w").write(mutated)
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", so, c, BWD_SRC, "-lm"], check=True)
        assert _caught(so), f"no pin rejects mutant {name!r}"


def test_unmutated_source_passes_all_pins():
    assert not _caught(oracle.build())
