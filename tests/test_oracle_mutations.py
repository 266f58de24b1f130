"""The oracle's pins have teeth: each plausible mistake, planted in a copy of the oracle's C source and
compiled on the CPU, makes at least one pin fail.  (Mistakes are planted only in the oracle, never in
GPU code.)"""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()

# (name, text in kda_oracle.c, replacement)
MUTATIONS = [
    ("beta dropped from the update", "S[(int64_t)r * dv + j] += beta * kh[r] * (vh[j] - kS[j]);",
     "S[(int64_t)r * dv + j] += kh[r] * (vh[j] - kS[j]);"),
    ("delta correction with the wrong sign", "beta * kh[r] * (vh[j] - kS[j])", "beta * kh[r] * (vh[j] + kS[j])"),
    ("decay applied to the column instead of the row", "S[(int64_t)r * dv + j] *= al[r];",
     "S[(int64_t)r * dv + j] *= al[j % dk];"),
    ("readout from the transposed state", "o[j] += S[(int64_t)r * dv + j] * qh[r];",
     "o[j] += S[(int64_t)(j % dk) * dv + (r % dv)] * qh[r];"),
    ("conv taps reversed", "double acc = w[W - 1] * x;", "double acc = w[0] * x;"),
    ("window not shifted", "cs[(int64_t)j * Cc + ch] = cs[(int64_t)(j + 1) * Cc + ch];", ";"),
    ("silu replaced by sigmoid", "acc = acc * sigmoid(acc);", "acc = sigmoid(acc);"),
    ("l2 eps outside the root", "1.0 / sqrt(nq + c->l2_eps)", "1.0 / (sqrt(nq) + c->l2_eps)"),
    ("k not normalised", "kh[i] *= rk;", ";"),
    ("alpha sigmoid sign", "alpha[i] = sigmoid(in->a[(t * H + h) * dk + i]);",
     "alpha[i] = sigmoid(-in->a[(t * H + h) * dk + i]);"),
    ("rms mean over the wrong length", "ms /= dv;", "ms /= (dv + 1);"),
    ("gate omitted", "double g = in->z ? sigmoid(in->z[(t * c->H + h) * dv + j]) : 1.0;", "double g = 1.0;"),
    ("scale omitted", "o[j] *= c->scale;", ";"),
    ("checkpoint one token late", "const int64_t p = start + i + 1; /* prefix length after this token */",
     "const int64_t p = start + i; /* prefix length after this token */"),
    ("chunked readout without the diagonal", "for (int64_t u = 0; u <= r; ++u) s += Qk",
     "for (int64_t u = 0; u < r; ++u) s += Qk"),
    ("chunked solve without beta", "X[(int64_t)r * m + j] = beta[r] * (acc - s);",
     "X[(int64_t)r * m + j] = (acc - s);"),
    ("chunked state without the decayed S0", "double s = exp(GL[e]) * S[(int64_t)e * dv + j];",
     "double s = S[(int64_t)e * dv + j];"),
]

PIN_FUNCS = [
    lambda: [pins.test_oracle_matches_library_brute_force(*p) for p in
             [(True, True, 1.0), (False, False, 0.25), (True, False, 0.5)]],
    pins.test_oracle_exact_rational_arithmetic,
    pins.test_pin_identity_step_alpha1_beta0,
    pins.test_pin_beta0_closed_form_decay,
    lambda: [pins.test_pin_delta_rule_invariant(b) for b in (1000.0, 0.7)],
    pins.test_pin_single_token_from_zero_state,
    pins.test_pin_conv_constant_input_and_window_shift,
    pins.test_pin_rmsnorm_unit_rms,
    pins.test_pin_l2_eps_placement,
    lambda: [pins.test_pin_chunked_form_equals_recurrence(c) for c in (4, 16)],
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, monkeypatch):
    assert SRC.count(old) == 1, f"mutation anchor not unique: {name}"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "m.c")
        so = os.path.join(d, "m.so")
        open(src, "w").write(SRC.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", so, "-lm"], check=True,
                       capture_output=True)
        monkeypatch.setattr(oracle, "_lib", oracle._configure(ctypes.CDLL(so)))
        caught = 0
        for f in PIN_FUNCS:
            try:
                f()
            except AssertionError:
                caught += 1
        assert caught > 0, f"no pin caught: {name}"
