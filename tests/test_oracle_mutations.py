"""The oracle's pins must catch plausible mistakes.

Each case copies oracle.c with one planted error (a sign, an index, a
transposed operand, a dropped term, a biased/unbiased swap), builds the copy in
a temporary directory and runs the pin suite against it in a subprocess; the
suite has to fail.  Mistakes are planted in the CPU oracle only.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "pad_sign": ("const long od = id * ss[0] - pp[0] + dil[0] * kd;", "const long od = id * ss[0] + pp[0] + dil[0] * kd;"),
    "weight_transposed": ("wc = w + (ci * Cout_g + col) * kvol", "wc = w + (col * Cin + ci) * kvol"),
    "tap_axes_swapped": ("(double)wc[(kd * kk[1] + kh) * kk[2] + kw]", "(double)wc[(kw * kk[1] + kh) * kk[0] + kd]"),
    "gn_unbiased_var": ("const double var = ss / (double)cnt;", "const double var = ss / (double)(cnt - 1);"),
    "bn_var_shifted": ("const double var = ss / cnt;", "const double var = ss / cnt + 1e-3;"),
    "out_size_pad_once": ("return (in - 1) * stride - 2 * pad + k + out_pad;",
                          "return (in - 1) * stride - pad + k + out_pad;"),
    "sigmoid_sign": ("col[(long)c * vol] = 1.0 / (1.0 + exp(-t));", "col[(long)c * vol] = 1.0 / (1.0 + exp(t));"),
    "bias_dropped_once": ("for (long o = 0; o < out_vol; ++o) Yc[o] += b;",
                          "for (long o = 1; o < out_vol; ++o) Yc[o] += b;"),
    "w_bound_off_by_one": ("if (ow < 0 || ow >= Wo) continue;", "if (ow < 0 || ow > Wo) continue;"),
    "softmax_no_norm": ("const double t = exp(col[(long)c * vol] - m) / S;",
                        "const double t = exp(col[(long)c * vol] - m);"),
    "running_var_biased": ("const double var_unbiased = cnt > 1.0 ? ss / (cnt - 1.0) : 0.0;",
                           "const double var_unbiased = cnt > 1.0 ? ss / cnt : 0.0;"),
    "eval_bn_eps_outside": ("const double inv = 1.0 / sqrt((double)rvar[c] + eps);",
                            "const double inv = 1.0 / (sqrt((double)rvar[c]) + eps);"),
    "dilation_dropped_h": ("const long oh = ih * ss[1] - pp[1] + dil[1] * kh;",
                           "const long oh = ih * ss[1] - pp[1] + kh;"),
    "stride_axes_mixed": ("const long ow = iw * ss[2] - pp[2] + dil[2] * kw;",
                          "const long ow = iw * ss[1] - pp[2] + dil[2] * kw;"),
    "group_channels_from_group0": ("for (long ci = g * Cin_g; ci < (g + 1) * Cin_g; ++ci) {",
                                   "for (long ci = 0; ci < Cin_g; ++ci) {"),
    "out_size_dilation_off_by_one": ("return (in - 1) * stride - 2 * pad + dil * (k - 1) + out_pad + 1;",
                                     "return (in - 1) * stride - 2 * pad + dil * k + out_pad;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    (tmp_path / "oracle.c").write_text(text.replace(old, new))
    env = dict(os.environ, CONVT3D_ORACLE_SRC=str(tmp_path / "oracle.c"),
               CONVT3D_ORACLE_BUILD_DIR=str(tmp_path), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch {name}:\n{r.stdout[-2000:]}"
