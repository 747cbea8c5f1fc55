"""The oracle's pins catch plausible slips (no GPU needed).

Each mutant below plants one mistake in a copy of oracle/oracle.c (on the
CPU, in a temporary directory), compiles it, and runs
tests/test_oracle_pins.py against it.  The pin suite must fail on every
mutant; a mutant that survives names a slip the pins cannot see.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "unary_dropped": ("const double s = (double)unary[r * k + j] + pairwise;", "const double s = pairwise;"),
    "codebooks_swapped": ("pairwise += (bf16_to_double(pred_cb[prev * D + d])",
                          "pairwise += (bf16_to_double(succ_cb[prev * D + d])"),
    "gate_of_previous_position": ("* gate[r * D + d]) *", "* gate[(t > 0 ? r - 1 : r) * D + d]) *"),
    "predecessor_from_same_position": ("cand_ids[(r - 1) * k + i]", "cand_ids[r * k + i]"),
    "anchor_ignored": ("(t == 0) ? anchor[b]", "(t == 0) ? 0"),
    "lattice_transposed": ("row[k + (int64_t)i * k + j] = (float)s;", "row[k + (int64_t)j * k + i] = (float)s;"),
    "tie_break_reversed": ("return (a->id < b->id) ? -1 : (a->id > b->id) ? 1 : 0;",
                           "return (a->id > b->id) ? -1 : (a->id < b->id) ? 1 : 0;"),
    "walk_argmin": ("if (scores[j] > scores[best])", "if (scores[j] < scores[best])"),
    "walk_last_maximum": ("if (scores[j] > scores[best])", "if (scores[j] >= scores[best])"),
    "walk_ignores_predecessor": ("const float *scores = row + k + (int64_t)jprev * k;\n            int32_t best = 0;",
                                 "const float *scores = row + k;\n            int32_t best = 0;"),
    "sampled_walk_ignores_predecessor": ("const float *scores = row + k + (int64_t)jprev * k;\n            double m",
                                         "const float *scores = row + k;\n            double m"),
    "logit_first_term_dropped": ("for (int64_t h = 0; h < H; ++h)\n                acc += bf16_to_double(hr[h])",
                                 "for (int64_t h = 1; h < H; ++h)\n                acc += bf16_to_double(hr[h])"),
    "logits_summed_in_float": ("            double acc = 0.0;\n            for (int64_t h = 0; h < H; ++h)\n                acc += bf16_to_double(hr[h])",
                               "            float acc = 0.0f;\n            for (int64_t h = 0; h < H; ++h)\n                acc += bf16_to_double(hr[h])"),
    "gate_transposed": ("bf16_to_double(W_sel[d * H + h])", "bf16_to_double(W_sel[h * D + d])"),
    "confidence_of_the_maximum": ("            confidence[r] = p[pick];", "            confidence[r] = p[0] > p[pick] ? p[0] : p[pick];"),
    "temperature_multiplies": ("p[j] = exp(((double)scores[j] - m) / temperature);",
                               "p[j] = exp(((double)scores[j] - m) * temperature);"),
    "stop_counts_the_low_step": ("                n_draft[b] = (int32_t)t;", "                n_draft[b] = (int32_t)t + 1;"),
    "inverse_cdf_off_by_one": ("                    if (run > u) {\n                        pick = j;",
                               "                    if (run > u) {\n                        pick = j + 1 < k ? j + 1 : j;"),
    "conv_taps_swapped": ("const double k0 = bf16_to_double(base[c])", "const double k0 = bf16_to_double(base[C + c])"),
    "conv_group_interleaved": ("const int64_t g = c / G;", "const int64_t g = c % groups;"),
    "conv_first_position_reads_zero": ("prv[c] = x_prev ? bf16_to_double(x_prev[b * C + c]) : 0.0;", "prv[c] = 0.0;"),
    "conv_crosses_blocks": ("                if (t > 0)\n                    prv[c] = bf16_to_double(x[(r - 1) * C + c]);",
                            "                if (r > 0)\n                    prv[c] = bf16_to_double(x[(r - 1) * C + c]);"),
    "conv_norm_without_mean": ("1.0 / sqrt(sc / (double)C + eps)", "1.0 / sqrt(sc + eps)"),
    "gate_of_wrong_row": ("bf16_to_double(hidden[r * H + h]);\n            gate[r * D + d] = acc;",
                          "bf16_to_double(hidden[(R - 1 - r) * H + h]);\n            gate[r * D + d] = acc;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "oracle_mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                    "-o", str(lib), str(mut), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant {name} survived the oracle pins:\n{res.stdout[-2000:]}"
