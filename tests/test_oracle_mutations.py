"""Planted-mistake tests for the oracle pins.

Each case copies the oracle's C source, plants one plausible mistake (a dropped term, a wrong
sign, index or axis, a transposed operand, a misplaced epsilon), builds the copy into a temporary
library, and runs the pin suite against it.  At least one pin must fail for every mistake; the
pristine oracle passes them all (test_oracle_pins.py).  The mistakes are planted in the CPU
oracle only.
"""

import os
import tempfile

import pytest

from oracle import oracle as orc
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(orc.__file__), "kda_oracle.c")

# (name, original text, mutated text); the original must occur exactly once in the source
MUTATIONS = [
    ("decay_on_value_dim",
     "const double a = exp(gt[i]);\n            for (int j = 0; j < D; ++j) S[i * D + j] *= a;",
     "for (int j = 0; j < D; ++j) S[i * D + j] *= exp(gt[j]);"),
    ("u_sign", "u[j] = vt[j] - acc;", "u[j] = vt[j] + acc;"),
    ("beta_dropped", "S[i * D + j] += bt * kt[i] * u[j];", "S[i * D + j] += kt[i] * u[j];"),
    ("readout_uses_k", "for (int i = 0; i < D; ++i) acc += S[i * D + j] * qt[i];",
     "for (int i = 0; i < D; ++i) acc += S[i * D + j] * kt[i];"),
    ("scale_dropped", "o[(long)t * o_stride + j] = scale * acc;",
     "o[(long)t * o_stride + j] = acc;"),
    ("state_in_transposed", "S[i * D + j] = m_in[(long)j * D + i];",
     "S[i * D + j] = m_in[(long)i * D + j];"),
    ("l2_eps_outside_sqrt", "const double inv = 1.0 / sqrt(ss + eps);",
     "const double inv = 1.0 / (sqrt(ss) + eps);"),
    ("conv_taps_reversed", "acc += w[(long)c * K + j] * xt[t + j];",
     "acc += w[(long)c * K + (K - 1 - j)] * xt[t + j];"),
    ("ring_newest_first", "ring_out[(long)c * R + s] = xt[T + s];",
     "ring_out[(long)c * R + s] = xt[T + R - 1 - s];"),
    ("silu_dropped", "y[(long)t * y_stride + c] = silu(acc);",
     "y[(long)t * y_stride + c] = acc;"),
    ("gate_rate_not_exponentiated",
     "g[r * C + c] = lb * sigmoid(exp(a_log[h]) * (f[r * C + c] + dt_bias[c]));",
     "g[r * C + c] = lb * sigmoid(a_log[h] * (f[r * C + c] + dt_bias[c]));"),
    ("gate_bias_per_head",
     "g[r * C + c] = lb * sigmoid(exp(a_log[h]) * (f[r * C + c] + dt_bias[c]));",
     "g[r * C + c] = lb * sigmoid(exp(a_log[h]) * (f[r * C + c] + dt_bias[h]));"),
    ("gdn_softplus_sign",
     "g[r * H + h] = -exp(a_log[h]) * softplus(alpha[r * H + h] + dt_bias[h]);",
     "g[r * H + h] = -exp(a_log[h]) * softplus(alpha[r * H + h] - dt_bias[h]);"),
    ("gdn_decay_dropped", "col[i] = alpha * col[i];", "col[i] = col[i];"),
    ("gdn_readout_before_update", "sq += col[i] * q[row + i];",
     "sq += (col[i] - b * k[row + i] * uj) * q[row + i];"),
    ("rmsnorm_sum_not_mean", "const double inv = 1.0 / sqrt(ss / D + eps);",
     "const double inv = 1.0 / sqrt(ss + eps);"),
    ("rmsnorm_gate_silu", "(silu_gate ? silu(zi) : sigmoid(zi))",
     "(silu_gate ? silu(zi) : silu(zi))"),
    ("rmsnorm_silu_gate_is_sigmoid", "(silu_gate ? silu(zi) : sigmoid(zi))",
     "(silu_gate ? sigmoid(zi) : sigmoid(zi))"),
    ("matvec_last_term_dropped", "for (long k = 0; k < in_f; ++k) acc += w[r * in_f + k]",
     "for (long k = 0; k + 1 < in_f; ++k) acc += w[r * in_f + k]"),
    ("matvec_first_token_only", "* x[(long)s * in_f + k];", "* x[k];"),
    ("matvec_weight_column_shifted", "acc += w[r * in_f + k] * x",
     "acc += w[r * in_f + (k + 1) % in_f] * x"),
    ("rect_value_stride_uses_key_width", "const double* vt = v + (r0 + t) * Cv + (long)h * Dv;",
     "const double* vt = v + (r0 + t) * Cv + (long)h * Dk;"),
    ("rect_state_transposed", "S[(long)i * Dv + j] = min[(long)j * Dk + i];",
     "S[(long)i * Dv + j] = min[(long)i * Dv + j];"),
]


def _run_all_pins():
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check()
        except AssertionError:
            failed.append(check.__name__)
    try:
        pins.check_orthonormal_recall(orc.scan_gdn)
    except AssertionError:
        failed.append("check_orthonormal_recall[gdn]")
    return failed


@pytest.mark.parametrize("name,orig,mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, orig, mut, monkeypatch):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for {name} not unique in the oracle source"
    with tempfile.TemporaryDirectory() as d:
        msrc = os.path.join(d, "kda_oracle_mut.c")
        with open(msrc, "w") as f:
            f.write(src.replace(orig, mut))
        lib = orc._bind(orc.build(force=True, src=msrc, out=os.path.join(d, "libmut.so")))
        monkeypatch.setattr(orc, "_lib", lib)
        failed = _run_all_pins()
    assert failed, f"planted mistake {name} passed every pin"
