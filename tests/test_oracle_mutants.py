"""Plant plausible mistakes in copies of the oracle source; the pins must catch each one.

Every mutant is a textual edit of ``oracle/attn_oracle.c`` compiled into a
temporary library on the CPU.  The real oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "drop_scale": ("s[j - j0] = scale * acc;", "s[j - j0] = acc;"),
    "causal_off_by_one": ("long lim = i + (Nk - Nq) + 1;", "long lim = i + (Nk - Nq);"),
    "top_left_causal": ("long lim = i + (Nk - Nq) + 1;", "long lim = i + 1;"),
    "keys_from_v": ("const double *kj = k + (size_t)j * d;", "const double *kj = v + (size_t)j * d;"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "no_final_divide": ("for (int t = 0; t < d; ++t) o[t] /= l;", ""),
    "tiled_drop_l_alpha": ("l = l * alpha + lt;", "l = l + lt;"),
    "tiled_drop_o_alpha": ("for (int t = 0; t < d; ++t) acc[t] *= alpha;", ""),
    "combine_weight_sign": ("double w = (ls == -INFINITY) ? 0.0 : exp(ls - M);",
                            "double w = (ls == -INFINITY) ? 0.0 : exp(M - ls);"),
    "combine_lse_no_max": ("lse[r] = M + log(wsum);", "lse[r] = log(wsum);"),
    "bwd_drop_rowsum_term": ("const double ds = p[j] * (dp[j] - D);", "const double ds = p[j] * dp[j];"),
    "bwd_dq_without_scale": ("dqi[t] += scale * ds * kj[t];", "dqi[t] += ds * kj[t];"),
    "bwd_dk_from_keys": ("dkj[t] += scale * ds * qi[t];", "dkj[t] += scale * ds * kj[t];"),
    "bwd_dv_unnormalised": ("p[j] /= l;", ""),
    "bwd_dp_against_keys": ("const double *vj = vh + (size_t)j * d;", "const double *vj = kh + (size_t)j * d;"),
    "exp_without_shift_guard": ("double m_sub = (m_new == -INFINITY) ? 0.0 : m_new;", "double m_sub = m_new;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mutated = text.replace(old, new)
    src = tmp_path / "mut.c"
    src.write_text(mutated)
    lib = oracle.load(oracle.build(force=True, src=str(src), out=str(tmp_path / "libmut.so")))
    failing = oracle_pins.failing_pins(lib)
    assert failing, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    src = tmp_path / "same.c"
    src.write_text(open(SRC).read())
    lib = oracle.load(oracle.build(force=True, src=str(src), out=str(tmp_path / "libsame.so")))
    assert oracle_pins.failing_pins(lib) == []
