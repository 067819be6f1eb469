"""Pin strength: copies of the oracle with one planted mistake each must fail
at least one pin (CPU only; the mistakes live in temporary copies of the
oracle source, never in the CUDA path)."""
import os
import subprocess

import pytest

import oracle
from tests import oracle_checks

# (name, text in bitdelta_oracle.c, replacement)
MUTANTS = [
    ("sign_of_zero_negative", "if (delta >= 0.0)                      /* sign(0)",
     "if (delta > 0.0)                      /* sign(0)"),
    ("msb_first_packing", "bits[e / 32] |= (uint32_t)1u << (e % 32);\n    }\n    *alpha64",
     "bits[e / 32] |= (uint32_t)1u << (31 - e % 32);\n    }\n    *alpha64"),
    ("alpha_divides_by_K", "*alpha64 = abs_sum / (double)n_elems;",
     "*alpha64 = abs_sum / (double)K;"),
    ("alpha_sum_not_mean", "*alpha64 = abs_sum / (double)n_elems;",
     "*alpha64 = abs_sum;"),
    ("alpha_signed_sum", "abs_sum += fabs(delta);", "abs_sum += delta;"),
    ("reconstruct_minus", "w_eff[k] = wb + a * s;", "w_eff[k] = wb - a * s;"),
    ("dropped_base_term", "w_eff[k] = wb + a * s;", "w_eff[k] = a * s;"),
    ("dropped_sign_term", "w_eff[k] = wb + a * s;", "w_eff[k] = wb;"),
    ("sign_zero_one", "? 1.0 : -1.0;", "? 1.0 : 0.0;"),
    ("unpack_msb_first", "return (int)((word >> (k % 32)) & 1u);",
     "return (int)((word >> (31 - k % 32)) & 1u);"),
    ("reversed_k_index", "acc += xrow[k] * w_eff[k];", "acc += xrow[k] * w_eff[K - 1 - k];"),
    ("wrong_weight_row", "double wb = bf16_to_double(j->w_base[n * K + k]);",
     "double wb = bf16_to_double(j->w_base[((n + 1) % j->N) * K + k]);"),
    ("wrong_token_row", "xrow[k] = bf16_to_double(j->x[t * K + k]);",
     "xrow[k] = bf16_to_double(j->x[((t + 1) % j->M) * K + k]);"),
    ("base_variant_gets_scale", "w_eff[k] = wb;\n", "w_eff[k] = wb + (double)j->alphas[0];\n"),
    ("first_variant_scale_for_all", ": (double)j->alphas[v];", ": (double)j->alphas[0];"),
    ("first_variant_bits_for_all", "sign_bit(j->bits[v], K, n, k)", "sign_bit(j->bits[0], K, n, k)"),
    ("row_scale_index_swapped", "(double)j->alphas[(int64_t)v * j->N + n]",
     "(double)j->alphas[(n * j->V + v) % (j->V * j->N)]"),
    ("reconstruct_ties_away", "double q = nearbyint(m * 256.0);", "double q = floor(m * 256.0 + 0.5);"),
    ("reconstruct_truncates", "double q = nearbyint(m * 256.0);", "double q = floor(m * 256.0);"),
    ("reconstruct_row_scale_first", "double a = (double)alpha[per_row ? n : 0];", "double a = (double)alpha[0];"),
    ("reconstruct_sign_flipped", "double s = (double)(2 * bit - 1);", "double s = (double)(1 - 2 * bit);"),
    ("row_scale_first_row", "(double)j->alphas[(int64_t)v * j->N + n]", "(double)j->alphas[(int64_t)v * j->N]"),
    ("output_transposed_store", "j->y[t * j->nrows + ri] = acc;",
     "j->y[(ri * j->M + t) % (j->M * j->nrows)] = acc;"),
]


def _failures(o):
    failed = []
    for check in oracle_checks.ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            failed.append(check.__name__)
        except ValueError:
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1, "mutation anchor must occur exactly once: %r" % old
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), str(mutated), "-lm"], check=True)
    failed = _failures(oracle.Oracle(lib))
    assert failed, "mutant %s passed every pin" % name
