"""Planted mistakes in copies of the oracle must each fail a pin.

Each mutant is a one-line change to a copy of ``oracle/osattn_ref.cpp`` that
a plausible bug would make (dropped term, wrong sign or index, transposed
operand, off-by-one mask).  The oracle pins in ``test_oracle.py`` and
``test_oracle_bwd.py`` run against the copy in a child process (a bad index
may crash it), and must not pass.
CPU only; the real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "no_max_in_output": ("const double pj = std::exp(s[j] - m) / l;",
                         "const double pj = std::exp(s[j]) / l;"),
    "sign_in_denominator": ("l += std::exp(s[j] - m);", "l += std::exp(m - s[j]);"),
    "scale_dropped": ("s[j] = p.scale * acc;", "s[j] = acc;"),
    "causal_off_by_one": ("if (p.causal) jend = std::min(jend, i + 1);  // j <= i",
                          "if (p.causal) jend = std::min(jend, i);"),
    "transposed_key": ("load_elem(p.K, p.dtype, koff + k)",
                       "load_elem(p.K, p.dtype, kvoff + static_cast<int64_t>(k) * d + j)"),
    "value_row_index": ("const int64_t voff = kvoff + static_cast<int64_t>(j) * d;",
                        "const int64_t voff = kvoff + static_cast<int64_t>(jend - 1 - j) * d;"),
    "combine_drops_rescale": ("*l_out = l1 * std::exp(m1 - M) + l2 * std::exp(m2 - M);",
                              "*l_out = l1 + l2 * std::exp(m2 - M);"),
    "online_no_rescale": ("l = l * std::exp(m - m_new) + std::exp(x[t] - m_new);",
                          "l = l + std::exp(x[t] - m_new);"),
    "lse_log2": ("return m + std::log(l);\n}", "return m + std::log2(l);\n}"),
    "fp16_exponent_bias": ("mag = std::ldexp(static_cast<double>(1024 + f), e - 25);",
                           "mag = std::ldexp(static_cast<double>(1024 + f), e - 24);"),
    "fp16_subnormal_scale": ("mag = std::ldexp(static_cast<double>(f), -24);",
                             "mag = std::ldexp(static_cast<double>(1024 + f), -25);"),
    "bwd_drops_row_term": ("const double ds = pr[j] * (dp[j] - D);", "const double ds = pr[j] * dp[j];"),
    "bwd_sign": ("const double ds = pr[j] * (dp[j] - D);", "const double ds = pr[j] * (D - dp[j]);"),
    "bwd_dq_transposed_key": ("for (int c = 0; c < d; ++c) dq[c] += scale * ds * kj[c];",
                              "for (int c = 0; c < d; ++c) dq[c] += scale * ds * kb[(c % Nkv) * d + j % d];"),
    "bwd_keyrow_drops_row_term": ("const double dsij = pij * (dot(gi, vj) - row_D[qr]);",
                                  "const double dsij = pij * dot(gi, vj);"),
    "bwd_keyrow_without_lse": ("const double pij = std::exp(scale * dot(qi, kj) - row_lse[qr]);",
                               "const double pij = std::exp(scale * dot(qi, kj));"),
    "bwd_keyrow_causal_off_by_one": ("const int i0 = causal ? j : 0;", "const int i0 = causal ? j + 1 : 0;"),
    "bwd_dk_without_scale": ("dk[c] += scale * dsij * qi[c];", "dk[c] += dsij * qi[c];"),
    "bwd_dv_wrong_operand": ("dv[c] += pij * gi[c];", "dv[c] += pij * qi[c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src_dir = os.path.join(ROOT, "oracle")
    dst = tmp_path / "oracle_mut"
    dst.mkdir()
    shutil.copy(os.path.join(src_dir, "__init__.py"), dst / "__init__.py")
    text = open(os.path.join(src_dir, "osattn_ref.cpp")).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    (dst / "osattn_ref.cpp").write_text(text.replace(old, new))
    env = dict(os.environ, OSATTN_ORACLE_DIR=str(dst))
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle.py"), os.path.join(ROOT, "tests", "test_oracle_bwd.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
