"""The CPU oracle against the facts that pin it (CPU only).

Also plants plausible mistakes in copies of the oracle's C source and checks
that at least one pin catches each of them.
"""
import functools
import os
import subprocess
import types

import pytest

import oracle
from oracle import grad
from tests import oracle_pins

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "prism_oracle.c")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.forward)


# The state update and the readout of one token, as they stand in prism_oracle.c: the
# "output_before_update" mistake swaps them.
_UPDATE = (
    '        /* S <- S A_t + B_t, with S A_t = alpha (S - beta (S k) k^T). */\n'
    '        for (int i = 0; i < dv; ++i) {\n'
    '            double s = 0.0;\n'
    '            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * kt[j];\n'
    '            Sk[i] = s;\n'
    '        }\n'
    '        for (int i = 0; i < dv; ++i)\n'
    '            for (int j = 0; j < dk; ++j) {\n'
    '                double* sij = &S[(size_t)i * dk + j];\n'
    '                *sij = alpha * (*sij - beta * Sk[i] * kt[j]) + Bw[(size_t)i * dk + j];\n'
    '            }\n'
)
_READOUT = (
    '        /* o_t = S_t q_t */\n'
    '        for (int i = 0; i < dv; ++i) {\n'
    '            double s = 0.0;\n'
    '            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * qt[j];\n'
    '            o[i] = s;\n'
    '        }\n'
)

# (name, text in prism_oracle.c, replacement): each is a mistake a restatement of
# the method could plausibly contain.
MUTANTS = [
    ("no_base_write", "Bw[(size_t)i * dk + j] = beta * vt[i] * kt[j];", "Bw[(size_t)i * dk + j] = 0.0;"),
    ("forget_sign", "*sij - beta * Sk[i] * kt[j]", "*sij + beta * Sk[i] * kt[j]"),
    ("forget_no_beta", "*sij - beta * Sk[i] * kt[j]", "*sij - Sk[i] * kt[j]"),
    ("alpha_on_write", "*sij = alpha * (*sij - beta * Sk[i] * kt[j]) + Bw[(size_t)i * dk + j];",
     "*sij = alpha * (*sij - beta * Sk[i] * kt[j] + Bw[(size_t)i * dk + j]);"),
    ("conv_includes_current", "off_bthx(P, b, t - j, h, dv);", "off_bthx(P, b, t - j + 1, h, dv);"),
    ("conv_tap_reversed", "((size_t)h * w + (j - 1)) * dv", "((size_t)h * w + (w - j)) * dv"),
    ("wk_transposed", "Wk[(size_t)a * dv + c]", "Wk[(size_t)c * dk + a]"),
    ("no_normalize", "kk[a] *= inv;", "kk[a] *= 1.0;"),
    ("residual_not_updated", "r[i] -= dl[i];", "(void)0;"),
    ("gelu_tanh", "return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
     "return 0.5 * x * (1.0 + tanh(0.7978845608028654 * (x + 0.044715 * x * x * x)));"),
    ("gate_sign", "const double bl = sigmoid(z);", "const double bl = sigmoid(-z);"),
    ("r1_plus", "r[i] = vt[i] - u[i];", "r[i] = vt[i] + u[i];"),
    ("write_uses_unnormalised_p", "dl[i] = P->identity_act ? x : gelu_erf(x);",
     "dl[i] = P->identity_act ? x : gelu_erf(p[i]);"),
    ("alpha_not_exp", "const double alpha = exp(", "const double alpha = -("),
    ("initial_state_ignored", "if (P->initial_state)\n        memcpy(", "if (0)\n        memcpy("),
    ("history_ignored", "else if (P->v_hist)", "else if (0)"),
    ("history_reversed", "(w + t - j)) * dv;", "(-1 - t + j)) * dv;"),
    ("k_from_residual", "s += Wk[(size_t)a * dv + c] * u[c];", "s += Wk[(size_t)a * dv + c] * r[c];"),
    ("p_from_residual", "s += Wp[(size_t)a * dv + c] * u[c];", "s += Wp[(size_t)a * dv + c] * r[c];"),
    ("gate_from_residual", "z += wb[c] * u[c];", "z += wb[c] * r[c];"),
    ("gate_dropped_from_write", "Bw[(size_t)i * dk + j] += bl * dl[i] * kk[j];",
     "Bw[(size_t)i * dk + j] += dl[i] * kk[j];"),
    ("wk_of_first_step", "P->Wk + ((size_t)h * L + l)", "P->Wk + ((size_t)h * L + 0)"),
    ("wp_of_first_step", "P->Wp + ((size_t)h * L + l)", "P->Wp + ((size_t)h * L + 0)"),
    ("wbeta_of_first_step", "P->wbeta + ((size_t)h * L + l)", "P->wbeta + ((size_t)h * L + 0)"),
    ("wk_of_head_zero", "P->Wk + ((size_t)h * L + l)", "P->Wk + ((size_t)0 * L + l)"),
    ("wp_of_head_zero", "P->Wp + ((size_t)h * L + l)", "P->Wp + ((size_t)0 * L + l)"),
    ("wbeta_of_head_zero", "P->wbeta + ((size_t)h * L + l)", "P->wbeta + ((size_t)0 * L + l)"),
    ("conv_of_head_zero", "P->conv_w + ((size_t)h * w", "P->conv_w + ((size_t)0 * w"),
    ("readout_with_k", "s += S[(size_t)i * dk + j] * qt[j];", "s += S[(size_t)i * dk + j] * kt[j];"),
    ("beta_of_previous_token", "const double beta = P->beta[((size_t)b * T + t) * P->H + h];",
     "const double beta = P->beta[((size_t)b * T + (t > 0 ? t - 1 : 0)) * P->H + h];"),
    ("padding_processed", "if (t >= len) {", "if (0) {"),
    ("r1_without_anchor", "r[i] = vt[i] - u[i];", "r[i] = vt[i];"),
    ("output_before_update", _UPDATE + _READOUT, _READOUT + _UPDATE),
    ("padding_output_not_zeroed", "for (int i = 0; i < dv; ++i) o[i] = 0.0;\n            continue;",
     "continue;"),
    ("initial_state_of_other_pair", "P->initial_state + ((size_t)b * P->H + h) * dv * dk",
     "P->initial_state + ((size_t)h * P->B + b) * dv * dk"),
    ("final_state_to_other_pair", "P->final_state + ((size_t)b * P->H + h) * dv * dk",
     "P->final_state + ((size_t)h * P->B + b) * dv * dk"),
    ("norm_eps_1e-12", "#define NORM_EPS 1e-6", "#define NORM_EPS 1e-12"),
    ("history_of_head_zero", "(((size_t)b * P->H + h) * w + (w + t - j)) * dv",
     "(((size_t)b * P->H + 0) * w + (w + t - j)) * dv"),
    ("gate_with_bias", "const double bl = sigmoid(z);", "const double bl = sigmoid(z + 0.5);"),
    ("residual_added", "r[i] -= dl[i];", "r[i] += dl[i];"),
    ("direction_normalised_twice", "for (int a = 0; a < dk; ++a) kk[a] *= inv;",
     "for (int a = 0; a < dk; ++a) kk[a] *= inv * inv;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread",
                    "-I", os.path.dirname(ORACLE_SRC), "-o", str(lib), str(mutated), "-lm"],
                   check=True)
    fwd = functools.partial(oracle.forward, lib_path=str(lib))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(fwd)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"


# ---- the gradient oracle (oracle/grad.py) ----

@pytest.mark.parametrize("pin", oracle_pins.GRAD_PINS, ids=lambda f: f.__name__)
def test_grad_pin(pin):
    pin(oracle.forward, grad)


# mistakes planted in the differentiable restatement: each must fail a gradient pin
GRAD_MUTANTS = [
    ("no_base_write", "Bw = be[:, t].view(B, H, 1, 1) * vt.unsqueeze(-1) * kt.unsqueeze(-2)",
     "Bw = 0.0 * vt.unsqueeze(-1) * kt.unsqueeze(-2)"),
    ("no_normalize", "kl = kh / torch.sqrt((kh * kh).sum(-1, keepdim=True) + NORM_EPS)", "kl = kh"),
    ("gelu_tanh", "0.5 * x * (1.0 + torch.erf(x / math.sqrt(2.0)))",
     "0.5 * x * (1.0 + torch.tanh(0.7978845608028654 * (x + 0.044715 * x ** 3)))"),
    ("write_transposed", "S_new = S @ A + Bw", "S_new = S @ A + Bw.transpose(-1, -2)"),
    ("output_before_update", "o = torch.einsum(\"xhab,xhb->xha\", S, qt)",
     "o = torch.einsum(\"xhab,xhb->xha\", torch.where(live, S @ A, S), qt)"),
    ("padding_not_frozen", "S = torch.where(live, S_new, S)", "S = S_new"),
    ("decay_not_exp", "A = torch.exp(la[:, t]).view(B, H, 1, 1) * (", "A = (1.0 + la[:, t]).view(B, H, 1, 1) * ("),
]


@pytest.mark.parametrize("name,old,new", GRAD_MUTANTS, ids=[m[0] for m in GRAD_MUTANTS])
def test_grad_planted_mistake_is_caught(name, old, new):
    src = open(grad.__file__).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mod = types.ModuleType(f"grad_mut_{name}")
    exec(compile(src.replace(old, new), f"<grad {name}>", "exec"), mod.__dict__)
    caught = []
    for pin in oracle_pins.GRAD_PINS:
        try:
            pin(oracle.forward, mod)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every gradient pin"
