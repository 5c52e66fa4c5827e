"""The pins are strong enough: each plausible mistake planted in a copy of the
oracle (a wrong sign, a dropped factor, a transposed operand, an off-by-one
in the mask rule, a wrong logarithm, a wrong min/max in the tile rule) makes
at least one pin test fail.  Everything runs on the CPU; the real oracle is
untouched and restored after each case."""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "dS sign of D": ("ds = exp(s[j] - L) * (dp[j] - Di)", "ds = exp(s[j] - L) * (dp[j] + Di)"),
    "D without P": ("Di += exp(s[j] - L) * dp[j];", "Di += dp[j];"),
    "dK uses k (transposed operand)": ("dk[c] += scale * ds * (double)q[i * d + c];",
                                       "dk[c] += scale * ds * (double)k[j * d + c];"),
    "O row index": ("o[c] += p * (double)v[j * d + c];", "o[c] += p * (double)v[i * d + c];"),
    "lse base-2 log": ("return m + log(sum);", "return m + log2(sum);"),
    "mask rule closed end": ("(lts[j] <= i && i < lte[j])", "(lts[j] <= i && i <= lte[j])"),
    "dV missing P": ("dv[c] += p * (double)dO[i * d + c];", "dv[c] += (double)dO[i * d + c];"),
    "label uses min for max": ("(L0max <= qb && L1min >= qe)", "(L0min <= qb && L1min >= qe)"),
    "full test uses max": ("(U0min >= qe || U1max <= qb)", "(U0max >= qe || U1max <= qb)"),
    "interval end exclusive": ("if (starts[i * K + k] <= j && j <= ends[i * K + k]) attended = 1;",
                               "if (starts[i * K + k] <= j && j < ends[i * K + k]) attended = 1;"),
    "only the first interval": ("for (int64_t k = 0; k < K; ++k)\n                if (starts",
                                "for (int64_t k = 0; k < 1; ++k)\n                if (starts"),
    "last interval wins": ("if (starts[i * K + k] <= j && j <= ends[i * K + k]) attended = 1;",
                           "attended = (starts[i * K + k] <= j && j <= ends[i * K + k]);"),
}

PINS = [
    lambda: [pins.test_oracle_matches_torch_bruteforce(s, n, d) for s, n, d in
             [(0, 40, 16), (1, 64, 32), (2, 17, 8), (3, 50, 16)]],
    pins.test_oracle_gradients_by_finite_differences,
    pins.test_invariants_constant_v_single_key_dead_rows,
    pins.test_row_and_column_forms_give_the_same_dense_mask,
    pins.test_golden_causal_example,
    pins.test_golden_doc_packing_example,
    pins.test_golden_multi_interval_example,
    pins.test_multi_interval_reduces_to_one_interval_rows,
    pins.test_multi_interval_union_invariants,
    pins.test_window_sink_row_and_column_forms_agree,
    lambda: [pins.test_labels_equal_exact_on_structured_masks(n, 128, 128) for n in
             ("causal_ragged", "docs_small", "window_small", "prefix_small")],
    lambda: [pins.test_labels_sound_on_arbitrary_bounds(s) for s in range(6)],
    lambda: [pins.test_labels_sound_with_one_random_range_per_column(s, w) for s in range(4)
             for w in ("lower", "upper")],
]


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not unique: {old}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so),
                           str(src), "-lm"])
    saved = oracle._load()
    oracle._lib = oracle._configure(ctypes.CDLL(str(so)))
    failures = 0
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failures += 1
    finally:
        oracle._lib = saved
    assert failures > 0, f"no pin caught the planted mistake: {name}"
