"""The oracle's pins must catch plausible slips.

Each case copies the oracle to a temporary directory, plants one mistake in the
copy's C source or Python wrapper (never in the committed oracle), rebuilds it
and runs the pin suite against the copy, which must fail.  This runs on the CPU
only.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    # the decay also multiplying the new write beta v k^T
    "decay_on_write": ("decay * (s - bt * Sk[j] * k[i]) + bt * vt[j] * k[i]",
                       "decay * (s - bt * Sk[j] * k[i] + bt * vt[j] * k[i])"),
    # S^T k in place of S k
    "transposed_state": ("acc += S[j * d_k + i] * k[i];\n      Sk[j]",
                         "acc += S[(i % d_v) * d_k + (j % d_k)] * k[i];\n      Sk[j]"),
    # conv taps applied newest-first
    "reversed_taps": ("(double)conv_weight[c * conv_w + w]",
                      "(double)conv_weight[c * conv_w + (conv_w - 1 - w)]"),
    # tiled instead of repeat-interleaved key heads
    "tiled_key_heads": ("const int64_t hk = h / (h_v / h_k);", "const int64_t hk = h % h_k;"),
    # query not scaled by 1/sqrt(d_k)
    "no_query_scale": ("1.0 / sqrt((double)d_k), qhat", "1.0, qhat"),
    # initial window read newest-first
    "window_order": ("window0[((conv_w - 1) + tau) * conv_dim + c]",
                     "window0[(-tau - 1) * conv_dim + c]"),
    # softplus with the wrong sign inside
    "softplus_sign": ("log1p(exp(-fabs(z)))", "log1p(exp(fabs(z)))"),
    # gated norm: sum of squares instead of their mean
    "norm_sum_not_mean": ("sqrt(ss / (double)d_v + eps)", "sqrt(ss + eps)"),
    # gated norm: a +1 pre-added to the weight
    "norm_weight_plus_one": ("inv * (double)w[j] * silu", "inv * (1.0 + (double)w[j]) * silu"),
    # gated norm: sigmoid gate instead of SiLU
    "norm_sigmoid_gate": ("(double)w[j] * silu((double)zrow[j])", "(double)w[j] * sigmoid((double)zrow[j])"),
    # projection: beta rows taken first
    "projection_rows_swapped": ("if (r < h_v) a[t * h_v + r] = acc;\n      else b[t * h_v + (r - h_v)] = acc;",
                                "if (r < h_v) b[t * h_v + r] = acc;\n      else a[t * h_v + (r - h_v)] = acc;"),
    # projection: the weight read transposed (column r of a [d_model][2 h_v] matrix)
    "projection_weight_transposed": ("acc += (double)x[i] * (double)wr[i];",
                                     "acc += (double)x[i] * (double)w[i * 2 * h_v + r];"),
    # projection: the last channel dropped
    "projection_last_channel": ("for (int64_t i = 0; i < d_model; ++i) acc += (double)x[i] * (double)wr[i];",
                                "for (int64_t i = 0; i + 1 < d_model; ++i) acc += (double)x[i] * (double)wr[i];"),
    # output read without the current token's write
    "output_before_write": (
        "for (int64_t i = 0; i < d_k; ++i) acc += S[j * d_k + i] * q[i];",
        "for (int64_t i = 0; i < d_k; ++i) acc += (S[j * d_k + i] - bt * vt[j] * k[i]) * q[i];"),
    # checkpoint taken one token late
    "checkpoint_one_late": ("__init__.py", "t = k * every\n", "t = k * every + 1\n"),
    # a checkpoint also at the end of a sequence whose length is a multiple of the interval
    "checkpoint_count": ("__init__.py", "n_b = max(0, -(-ln // every) - 1)", "n_b = max(0, ln // every)"),
    # snapshot copied the wrong way round
    "slot_copy_reversed": ("__init__.py", "st[d_] = st[s_]", "st[s_] = st[d_]"),
    # decay rate from A_log itself instead of e^{A_log}
    "A_log_not_exponentiated": ("const double A = exp((double)A_log[h]);",
                                "const double A = (double)A_log[h];"),
    # dt_bias left out of the softplus argument
    "dt_bias_dropped": ("double z = (double)a[t * h_v + h] + (double)dt_bias[h];",
                        "double z = (double)a[t * h_v + h];"),
    # g with the wrong sign: growth instead of decay
    "gate_sign": ("g[t] = -A * softplus(z);", "g[t] = A * softplus(z);"),
    # beta taken as b itself, without the sigmoid
    "beta_without_sigmoid": ("beta[t] = sigmoid((double)b[t * h_v + h]);",
                             "beta[t] = (double)b[t * h_v + h];"),
    # conv output used without the SiLU
    "conv_without_silu": ("y[t * y_stride] = silu(acc);", "y[t * y_stride] = acc;"),
    # keys left unnormalised
    "key_not_normalised": ("l2_normalise_rows(T, d_k, l2_eps, 1.0, khat);", ";"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    m = MUTATIONS[name]
    fname, before, after = m if len(m) == 3 else ("gdn_oracle.c", *m)
    src = open(os.path.join(ROOT, "oracle", fname)).read()
    assert before in src, "mutation site moved; update the mutation table"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "oracle" / fname).write_text(src.replace(before, after, 1))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "golden"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q",
                        "-x", "-p", "no:cacheprovider"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 1, f"pins did not catch '{name}':\n{r.stdout[-2000:]}"
