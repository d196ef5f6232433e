"""The pins have teeth: for each plausible mistake planted in a copy of the
oracle's C source (a dropped term, a flipped sign, a wrong index, a transposed
operand, a reversed order), at least one pin must fail.  The mistakes live
only in temporary copies compiled on the CPU; the real oracle is untouched."""
import os

import pytest

import oracle
import pins

# (name, text in oracle.c, replacement, occurrence to replace (0-based))
MUTANTS = [
    ("scalar_drops_beta", "a * S[(size_t)i * dv + j] + b * kt[i] * vt[j];",
     "a * S[(size_t)i * dv + j] + kt[i] * vt[j];", 0),
    ("diag_wrong_gate_index", "at[i] * S[(size_t)i * dv + j]", "at[0] * S[(size_t)i * dv + j]", 0),
    ("dense_erase_sign", "a * (S[(size_t)i * dv + j] - b * kt[i] * kS[j])",
     "a * (S[(size_t)i * dv + j] + b * kt[i] * kS[j])", 0),
    ("dense_state_skips_alpha", "a * (S[(size_t)i * dv + j] - b * kt[i] * kS[j]) + b",
     "(S[(size_t)i * dv + j] - b * kt[i] * kS[j]) + b", 0),
    ("dense_T_transposed", "acc += kt[i] * M[(size_t)i * dk + j];",
     "acc += kt[i] * M[(size_t)j * dk + i];", 0),
    ("dense_T_drops_beta", "M[(size_t)i * dk + j] -= b * kt[i] * kS[j];",
     "M[(size_t)i * dk + j] -= kt[i] * kS[j];", 0),
    ("scalar_lambda_sign", "lam[0] += log(a);\n            } else if", "lam[0] -= log(a);\n            } else if", 0),
    ("dense_lambda_drops_alpha", "lam[0] += log(a);\n                keep_in_range",
     "keep_in_range", 0),
    ("output_reads_key", "acc += S[(size_t)i * dv + j] * qt[i];", "acc += S[(size_t)i * dv + j] * kt[i];", 0),
    ("compose_drops_decay", "acc = exp(lam[0]) * mm;", "acc = mm;", 0),
    ("compose_M_transposed", "mm += M[(size_t)i * dk + r] * S_prev[(size_t)r * dv + j];",
     "mm += M[(size_t)r * dk + i] * S_prev[(size_t)r * dv + j];", 0),
    ("compose_diag_scalar_gate", "acc = exp(lam[i]) * S_prev", "acc = exp(lam[0]) * S_prev", 0),
    ("compose_T_order", "acc += Mu[(size_t)i * dk + r] * Mp[(size_t)r * dk + j];",
     "acc += Mp[(size_t)i * dk + r] * Mu[(size_t)r * dk + j];", 0),
    ("chain_reversed", "const int64_t p = seg_idx[r * max_chain + j];",
     "const int64_t p = seg_idx[r * max_chain + (chain_len[r] - 1 - j)];", 0),
    ("chain_ignores_init", "memcpy(S, S_init + u * dk * dv, sizeof(double) * (size_t)dk * dv);",
     "memset(S, 0, sizeof(double) * (size_t)dk * dv);", 0),
    ("seam_ignores_prev", "memcpy(S, S_prev + u * dk * dv, sizeof(double) * (size_t)dk * dv);",
     "memset(S, 0, sizeof(double) * (size_t)dk * dv);", 0),
    ("seam_dense_erase_sign", "a * (S[(size_t)r * dv + j] - b * kt[r] * kS[j])",
     "a * (S[(size_t)r * dv + j] + b * kt[r] * kS[j])", 0),
    ("seam_diag_gate_index", "at[r] * S[(size_t)r * dv + j]", "at[0] * S[(size_t)r * dv + j]", 0),
    ("seam_output_reads_key", "acc += S[(size_t)r * dv + j] * qt[r];", "acc += S[(size_t)r * dv + j] * kt[r];", 0),
    ("kda_gate_index", "at[i] * (S[(size_t)i * dv + j] - b * kt[i] * kS[j])",
     "at[0] * (S[(size_t)i * dv + j] - b * kt[i] * kS[j])", 0),
    ("kda_M_drops_gate", "M[(size_t)i * dk + j] = at[i] * (M[(size_t)i * dk + j] - b * kt[i] * kS[j]);",
     "M[(size_t)i * dk + j] = (M[(size_t)i * dk + j] - b * kt[i] * kS[j]);", 0),
    ("seam_kda_one_gate", "const double a = fam == OR_KDA ? alpha[row * dk + r] : alpha[row];",
     "const double a = fam == OR_KDA ? alpha[row * dk] : alpha[row];", 0),
    ("prefix_operator_order", "acc += Mp[(size_t)i * dk + x] * Mo[(size_t)x * dk + c];",
     "acc += Mo[(size_t)i * dk + x] * Mp[(size_t)x * dk + c];", 0),
    ("prefix_drops_lambda", "for (int i = 0; i < nl; ++i) lam[i] += pool_lam[e * nl + i];",
     "for (int i = 0; i < nl; ++i) lam[i] += 0.0 * pool_lam[e * nl + i];", 0),
    ("seam_token_order", "const int64_t row = (i * w + t) * H + h;", "const int64_t row = (i * w + (w - 1 - t)) * H + h;", 0),
]


def _replace_nth(src, old, new, n):
    pos = -1
    for _ in range(n + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"mutation anchor not found: {old!r}"
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, nth):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    lib = oracle.compile_source(str(c), str(tmp_path / f"lib{name}.so"))
    failed = []
    with oracle.using_library(lib):
        for check in pins.ALL_CHECKS:
            try:
                check()
            except (AssertionError, ValueError, IndexError, FloatingPointError):
                failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
