"""Mutation check of the pins: plant one plausible mistake in a copy of the
oracle's C source, build it, and require that at least one pin fails.  The
mistakes are planted only in temporary copies, on the CPU."""
import os
import shutil

import pytest

import oracle
from oracle.build import SRC, build_oracle
from oracle_pins import PINS

# (name, text in attention_oracle.c, replacement)
MUTATIONS = [
    ("dropped_scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("dropped_feature", "for (long c = 0; c < d; ++c)\n            dot += q[",
     "for (long c = 1; c < d; ++c)\n            dot += q["),
    ("transposed_qk", "dot += q[i * d + c] * k[j * d + c];", "dot += q[j * d + c] * k[i * d + c];"),
    ("causal_excludes_diagonal", "return i + 1;", "return i;"),
    ("causal_off", "    if (causal)\n        return i + 1;", "    if (0)\n        return i + 1;"),
    ("no_max_shift_sum", "l += exp(s[j] - m);", "l += exp(s[j]);"),
    ("no_max_shift_both", "l += exp(s[j] - m);\n\n    for (long c = 0; c < d; ++c)\n"
     "        o_i[c] = 0.0;\n    for (long j = 0; j < n_keys; ++j) {\n        double p = exp(s[j] - m);",
     "l += exp(s[j]);\n\n    for (long c = 0; c < d; ++c)\n"
     "        o_i[c] = 0.0;\n    for (long j = 0; j < n_keys; ++j) {\n        double p = exp(s[j]);"),
    ("reversed_values", "o_i[c] += p * v[j * d + c];", "o_i[c] += p * v[(n_keys - 1 - j) * d + c];"),
    ("no_final_normalise", "o_i[c] = o_i[c] / l;", "o_i[c] = o_i[c];"),
    ("lse_without_max", "*lse_i = m + log(l);", "*lse_i = log(l);"),
    ("lse_log2", "*lse_i = m + log(l);", "*lse_i = m + log2(l);"),
    ("online_l_not_rescaled", "l = alpha * l + block_sum;", "l = l + block_sum;"),
    ("online_O_not_rescaled", "acc[c] = alpha * acc[c] + pv;", "acc[c] = acc[c] + pv;"),
    ("online_alpha_sign", "double alpha = exp(m - m_new);", "double alpha = exp(m_new - m);"),
    ("online_forgets_running_max", "double m_new = m > m_tilde ? m : m_tilde;",
     "double m_new = m_tilde;"),
    ("online_p_uses_old_max", "block_sum += exp(s[j] - m_new);", "block_sum += exp(s[j] - m_tilde);"),
    ("online_no_max_shift", "pv += exp(s[j] - m_new) * v[j * d + c];", "pv += exp(s[j]) * v[j * d + c];"),
    ("online_no_final_normalise", "o_out[c] = acc[c] / l;", "o_out[c] = acc[c];"),
    ("row_slice_off_by_one", "jb->begin = t * per;", "jb->begin = t * per + (t > 0);"),
    ("bwd_row_split_off_by_one", "jb->i0 = sp * rows_per < N ? sp * rows_per : N;",
     "jb->i0 = sp * rows_per + (sp > 0) < N ? sp * rows_per + (sp > 0) : N;"),
    ("bwd_split_sum_first_job_only", "const rows_job *jb = &jobs[h * splits + sp];",
     "const rows_job *jb = &jobs[h * splits];"),
    ("bwd_rows_ignore_causal", "allowed_keys(i, jb->N, jb->causal)", "allowed_keys(i, jb->N, 0)"),
    ("decode_causal_start_aligned", "return causal ? nk - nq + i + 1 : nk;", "return causal ? i + 1 : nk;"),
    ("decode_causal_off_by_one", "return causal ? nk - nq + i + 1 : nk;", "return causal ? nk - nq + i : nk;"),
    ("decode_key_head_stride", "jb->k + bh * jb->nk * jb->d,", "jb->k + bh * jb->nq * jb->d,"),
    ("bwd_dv_uses_ds", "dv[j * d + c] += s[j] * g[i * d + c];", "dv[j * d + c] += ds * g[i * d + c];"),
    ("bwd_ds_not_centred", "double ds = s[j] * (dp[j] - pdp);", "double ds = s[j] * dp[j];"),
    ("bwd_ds_sign", "double ds = s[j] * (dp[j] - pdp);", "double ds = s[j] * (pdp - dp[j]);"),
    ("bwd_dk_uses_k", "dk[j * d + c] += scale * ds * q[i * d + c];",
     "dk[j * d + c] += scale * ds * k[j * d + c];"),
    ("bwd_dp_transposed", "dot += g[i * d + c] * v[j * d + c];", "dot += g[j * d + c] * v[i * d + c];"),
    ("bwd_p_not_normalised", "s[j] = exp(s[j] - m) / row_sum;", "s[j] = exp(s[j] - m);"),
    ("bwd_no_max_shift", "row_sum += exp(s[j] - m);", "row_sum += exp(s[j]);"),
    ("bwd_head_offset_dropped", "jb->dq + jb->head * he, jb->dk, jb->dv);", "jb->dq, jb->dk, jb->dv);"),
    ("bwd_dq_row_no_scale", "dq_i[c] += scale * ds_ij * k[j * d + c];", "dq_i[c] += ds_ij * k[j * d + c];"),
]


def _first_failing_pin(orc):
    for pin in PINS:
        try:
            pin(orc)
        except AssertionError:
            return pin.__name__
        except oracle.OracleError:
            return pin.__name__
    return None


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation site for %s not found exactly once" % name
    mutant_src = tmp_path / "attention_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = build_oracle(src=str(mutant_src), out=str(tmp_path / "libmutant.so"), force=True)
    failing = _first_failing_pin(oracle.Oracle(lib))
    assert failing is not None, "planted mistake %s passed every pin" % name


def test_unmutated_copy_passes(tmp_path):
    """Control: the same build procedure on an unmodified copy passes all pins."""
    copy = tmp_path / "attention_oracle_copy.c"
    shutil.copy(SRC, copy)
    lib = build_oracle(src=str(copy), out=str(tmp_path / "libcopy.so"), force=True)
    assert _first_failing_pin(oracle.Oracle(lib)) is None
