"""Plant plausible mistakes in a copy of the oracle's C source and check that
each one fails at least one pin (CPU only).  This shows the pins are strong
enough to catch a dropped term, a wrong sign, a wrong index or a transposed
operand anywhere in the oracle."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

# (name, exact text in fa_oracle.c, replacement)
MUTANTS = [
    ("dq_scale_dropped", "dqi[c] *= J->scale;", "(void)0;"),
    ("dk_scale_dropped", "dkj[c] *= J->scale;", "(void)0;"),
    ("dS_sign", "const double dS = p[j] * (dP[j] - D);", "const double dS = p[j] * (dP[j] + D);"),
    ("causal_off_by_one", "if (J->causal && j > i) return -INFINITY;",
     "if (J->causal && j > i + 1) return -INFINITY;"),
    ("dP_uses_k", "const double* vj = J->v + ((size_t)bh * N + j) * d;\n    double acc = 0.0;",
     "const double* vj = J->k + ((size_t)bh * N + j) * d;\n    double acc = 0.0;"),
    ("lse_log2", "J->lse[it] = (l > 0.0) ? m + log(l) : -INFINITY;",
     "J->lse[it] = (l > 0.0) ? m + log2(l) : -INFINITY;"),
    ("online_beta_dropped", "l = alpha * l + beta * blk_sum;\n    m = m_new;\n    if (m_trace)",
     "l = alpha * l + blk_sum;\n    m = m_new;\n    if (m_trace)"),
    ("dv_uses_dS", "dvj[c] += p * z * dOi[c];", "dvj[c] += dS * z * dOi[c];"),
    ("dk_uses_p", "dkj[c] += dS * qi[c];", "dkj[c] += p * qi[c];"),
    ("no_max_in_p", "for (int j = 0; j < N; ++j) p[j] = exp(s[j] - m) / l;",
     "for (int j = 0; j < N; ++j) p[j] = exp(s[j]) / l;"),
    ("score_transposed", "const double* qi = J->q + ((size_t)bh * J->N + i) * J->d;",
     "const double* qi = J->q + ((size_t)bh * J->N + j) * J->d;"),
    ("o_uses_k", "acc += p[j] * J->v[((size_t)bh * J->N + j) * J->d + c];",
     "acc += p[j] * J->k[((size_t)bh * J->N + j) * J->d + c];"),
    ("col_pass_D_dropped", "const double dS = p * (dP - J->D_all[ri]);",
     "const double dS = p * dP;"),
    ("online_O_alpha_dropped", "for (int c = 0; c < d; ++c) o[c] *= alpha;", "(void)0;"),
    ("block_mask_ignored", "if (J->bmask && !J->bmask[", "if (0 && !J->bmask["),
    ("block_mask_axes_swapped", "(int64_t)(i / J->bq) * J->nkb + j / J->bk]",
     "(int64_t)(j / J->bq) * J->nkb + i / J->bk]"),
    ("decode_causal_top_left", "const int last = J->causal ? Nk - J->Nq + i : Nk - 1;",
     "const int last = J->causal ? i : Nk - 1;"),
    ("decode_dot_uses_v", "const double* kj = J->k + ((size_t)bh * Nk + j) * d;",
     "const double* kj = J->v + ((size_t)bh * Nk + j) * d;"),
    ("block_mask_ignores_head", "J->bmask[bh * J->mstride +", "J->bmask[0 * J->mstride +"),
    ("philox_weyl_constant", "k1 += 0xBB67AE85u;", "k1 += 0x9E3779B9u;"),
    ("philox_mulhi_swapped", "const uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;",
     "const uint32_t y0 = (uint32_t)(p0 >> 32) ^ x1 ^ k0;"),
    ("dropout_counter_ignores_head", "(uint32_t)i, (uint32_t)bh, offset};",
     "(uint32_t)i, 0u, offset};"),
    ("dropout_halves_swapped", "return (j % 2 == 0) ? (word & 0xFFFFu) : (word >> 16);",
     "return (j % 2 == 1) ? (word & 0xFFFFu) : (word >> 16);"),
    ("dropout_word_index", "const uint32_t word = out[(j / 2) % 4];",
     "const uint32_t word = out[j % 4];"),
    ("dropout_rescale_dropped", "? J->rs : 0.0;", "? 1.0 : 0.0;"),
    ("dropout_ij_swapped", "fa_oracle_dropout_u16(J->seed, J->offset, bh, i, j) >=",
     "fa_oracle_dropout_u16(J->seed, J->offset, bh, j, i) >="),
    ("dropout_fwd_ignored", "if (J->dropout) /* dropout acts", "if (0) /* dropout acts"),
    ("dropout_dv_undropped", "dvj[c] += p * z * dOi[c];", "dvj[c] += p * dOi[c];"),
    ("dropout_col_dP_undropped", "dP *= z;", "(void)0;"),
    ("dropout_row_dP_undropped", "dP[j] = acc * drop_factor(J, bh, i, j);", "dP[j] = acc;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "fa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutated), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
