"""Mutation checks for the oracle's pins (CPU only).

Each case plants one plausible mistake in a private copy of the oracle's C
source, compiles it into a temporary directory and runs the pins of
``test_oracle.py`` against it.  At least one pin must fail for every
mutant; otherwise the pins would not protect the oracle from that mistake.
The real oracle is never modified.
"""
import pytest

import test_oracle as pins

# (name, text in ssd_oracle.c, replacement)
MUTANTS = [
    ("exclusive_output", "row[s] = decay * row[s] + u * bt[s];\n                    acc += ct[s] * row[s];",
     "acc += ct[s] * row[s];\n                    row[s] = decay * row[s] + u * bt[s];"),
    ("decay_without_dt", "exp(A[h] * dtv)", "exp(A[h])"),
    ("decay_sign", "exp(A[h] * dtv)", "exp(-A[h] * dtv)"),
    ("input_without_dt", "const double u = dtv * xt[p];", "const double u = xt[p];"),
    ("wrong_group", "const int64_t g = h / heads_per_group;", "const int64_t g = h % G;"),
    ("state_recorded_late", "if (states && t % T == 0)", "if (states && (t + 1) % T == 0)"),
    ("no_skip_term", "yt[p] = acc + D[h] * xt[p];", "yt[p] = acc;"),
    ("init_ignored", "if (init)\n", "if (0)\n"),
    ("global_cumsum", "if (t % T == 0)\n                    run = 0.0;", ""),
    ("cumsum_natural_log", "= ORACLE_LOG2E * run;", "= run;"),
    ("state_transposed", "double *row = st + p * S;", "double *row = st + p;"),
]


def _pin_battery(o):
    """Run the pins against oracle variant ``o``; return the names that failed."""
    checks = {
        "golden_scalar": lambda: pins.test_golden_hand_worked(o, "scalar_three_tokens.txt"),
        "golden_matrix": lambda: pins.test_golden_hand_worked(o, "matrix_state_two_tokens.txt"),
        "brute_force": lambda: pins.test_brute_force(o, (2, 17, 4, 4, 3, 2), "randn"),
        "chunked_T7": lambda: pins.test_chunked_closed_form(o, 7),
        "linear_attention": lambda: pins.test_decay_free_is_linear_attention(o),
        "cumsum_closed_form": lambda: pins.test_chunk_cumsum_closed_forms(o),
        "G_vs_decay": lambda: pins.test_G_matches_recurrence_decay(o),
        "identical_heads": lambda: pins.test_identical_heads_in_a_group(o),
    }
    failed = []
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failed.append(name)
    return failed


def test_real_oracle_passes_battery(oracle_mod):
    assert _pin_battery(oracle_mod) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(oracle_mod, tmp_path, name, old, new):
    src = oracle_mod.source_text()
    assert old in src, f"mutation site for {name} not found"
    so = oracle_mod.compile_source(src.replace(old, new, 1), str(tmp_path / f"mut_{name}.so"))
    failed = _pin_battery(oracle_mod.Variant(so))
    assert failed, f"mutant {name} passed every pin"
