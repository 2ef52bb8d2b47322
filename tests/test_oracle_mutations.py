"""The pins must reject a wrong oracle.

Each case plants one plausible mistake in a copy of the oracle's C source (a
dropped term, a wrong sign or comparison, a transposed operand, an off-by-one
on the valid rows, a wrong tie-break), compiles it on the CPU and checks that
at least one pin of ``test_oracle_pins`` fails against it.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import (test_oracle_centroid, test_oracle_meankey, test_oracle_pins as pins, test_oracle_promote,
                   test_oracle_stability)

SRC = os.path.join(os.path.dirname(oracle.__file__), "kvmm_oracle.c")

MUTATIONS = {
    "score-takes-min": ("s += (a > b) ? a : b;", "s += (a < b) ? a : b;"),
    "score-drops-last-channel": ("for (int32_t d = 0; d < D; ++d) {\n                double qd",
                                 "for (int32_t d = 0; d < D - 1; ++d) {\n                double qd"),
    "score-uses-max-only": ("double a = qd * bf16_value(mn[d]);", "double a = qd * bf16_value(mx[d]);"),
    "score-sign-select-inverted": ("s += (a > b) ? a : b;", "s += (qd >= 0) ? a : b;"),
    "group-max-instead-of-sum": ("total += s;", "total = (g == 0 || s > total) ? s : total;"),
    "minmax-skips-a-row": ("for (int32_t r = 1; r < n; ++r)", "for (int32_t r = 2; r < n; ++r)"),
    "minmax-counts-invalid-rows": ("return n < T ? (int32_t)n : T;", "return T;"),
    "minmax-ignores-signed-zero": ("return (a & 0x8000u) && !(b & 0x8000u);", "return 0;"),
    "topk-tiebreak-reversed": ("return (x->page > y->page) - (x->page < y->page);",
                               "return (x->page < y->page) - (x->page > y->page);"),
    "topk-not-ascending": ("qsort(sel, (size_t)n, sizeof(int32_t), by_int);", ""),
    "diff-gives-intersection": ("if (!found) out[n++] = a[i];", "if (found) out[n++] = a[i];"),
    "attention-wrong-scale": ("scale = 1.0 / sqrt((double)D);\n    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * ((size_t)cnt",
                              "scale = 1.0 / (double)D;\n    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * ((size_t)cnt"),
    "attention-lse-drops-max": ("lse[g] = m + log(denom);", "lse[g] = log(denom);"),
    "attention-q-k-transposed": ("bf16_value(q[(int64_t)g * D + d]) * bf16_value(k_pool[rows[t] * D + d]);",
                                 "bf16_value(q[(int64_t)g * D + d]) * bf16_value(v_pool[rows[t] * D + d]);"),
    "table-null-not-skipped": ("if (phys < 0) {\n        *err |= ORACLE_ERR_NULL_BLOCK;\n        return -1;",
                               "if (phys < 0) {\n        *err |= ORACLE_ERR_NULL_BLOCK;\n        return 0;"),
    "append-wrong-row": ("int64_t row = phys * T + (t % T);", "int64_t row = phys * T + ((t + 1) % T);"),
    # temporal stability (RCO) and classification
    "rco-chance-without-the-product": ("const int64_t chance_p = (int64_t)na * nb;",
                                       "const int64_t chance_p = (int64_t)(na < nb ? na : nb);"),
    "rco-best-is-the-larger-set": ("const int64_t best_p = (int64_t)(na < nb ? na : nb) * P;",
                                   "const int64_t best_p = (int64_t)(na > nb ? na : nb) * P;"),
    "rco-window-skips-a-pair": ("for (int32_t t = 0; t + lag < n; ++t) {", "for (int32_t t = 1; t + lag < n; ++t) {"),
    "classify-ties-to-the-higher-index": ("(stability[j] == stability[i] && j < i)",
                                          "(stability[j] == stability[i] && j > i)"),
    # promotion
    "promote-copies-the-evicted-page": ("host_k + (int64_t)promoted[i] * page", "host_k + (int64_t)evicted[i] * page"),
    "promote-keeps-evicted-entries": ("        bt_row[evicted[i]] = -1;\n    }", "    }"),
    # mean key and page mass
    "meankey-divides-by-the-page-size": ("mean[(int64_t)p * D + d] = bf16_round_nearest_even(acc / (float)n);",
                                         "mean[(int64_t)p * D + d] = bf16_round_nearest_even(acc / (float)T);"),
    "meankey-truncates": ("    u += 0x7fffu + lsb;\n", ""),
    "page-mass-skips-the-softmax-max": ("mass[(int64_t)g * P + t / T] += exp(z[t] - m) / denom;",
                                        "mass[(int64_t)g * P + t / T] += exp(z[t]) / denom;"),
    # centroid level
    "centroid-assign-takes-the-farthest": ("if (j == 0 || acc < best) {", "if (j == 0 || acc > best) {"),
    "centroid-assign-ties-to-the-higher": ("if (j == 0 || acc < best) {", "if (j == 0 || acc <= best) {"),
    "centroid-update-divides-by-the-block": ("bf16_round_nearest_even(acc / (float)n);\n        }\n    }\n}",
                                             "bf16_round_nearest_even(acc / 4.0f);\n        }\n    }\n}"),
    "centroid-update-skips-the-first-member": ("for (int32_t k = off[j]; k < off[j + 1]; ++k) acc +=",
                                               "for (int32_t k = off[j] + 1; k < off[j + 1]; ++k) acc +="),
    "centroid-blocks-off-by-one": ("for (int32_t p = 0; p < P; ++p) assign[p] = p / R;",
                                   "for (int32_t p = 0; p < P; ++p) assign[p] = (p + 1) / R < (P + R - 1) / R ? (p + 1) / R : p / R;"),
    "centroid-search-expands-one-fewer": ("for (int32_t i = 0; i < nm; ++i)\n        for (int32_t k = off[chosen[i]]",
                                          "for (int32_t i = 0; i + 1 < nm; ++i)\n        for (int32_t k = off[chosen[i]]"),
    "centroid-distance-drops-a-channel": ("            for (int32_t d = 0; d < D; ++d) {\n                const float x =",
                                          "            for (int32_t d = 1; d < D; ++d) {\n                const float x ="),
}

PIN_TESTS = [getattr(m, n) for m in (pins, test_oracle_stability, test_oracle_promote, test_oracle_meankey,
                                     test_oracle_centroid)
             for n in dir(m) if n.startswith("test_")]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutated_oracle(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutated.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so, str(mutated), "-lm"], check=True)
    variant = oracle.load_variant(so)
    failures = []
    for t in PIN_TESTS:
        try:
            t(variant)
        except (AssertionError, ValueError, IndexError):
            failures.append(t.__name__)
    assert failures, f"no pin caught the mutation {name}"
