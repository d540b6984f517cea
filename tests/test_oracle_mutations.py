"""The oracle's pins must catch plausible mistakes.

Each case compiles a copy of the oracle source with one planted mistake (a
dropped term, a wrong sign, a wrong factor, a wrong operand) on the CPU and
checks that at least one pin from the pin modules fails against it.  The
real oracle is untouched.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_chunk_identity as pin_chunk
import test_oracle_closed_forms as pin_fwd
import test_oracle_grad as pin_grad

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.cpp")

FWD_PINS = [
    pin_fwd.test_beta0_alpha1_keeps_state,
    pin_fwd.test_alpha0_resets_state,
    pin_fwd.test_single_token_from_zero_state,
    pin_fwd.test_delta_rule_invariant_unit_keys,
    pin_fwd.test_linearity_in_v_and_h0,
    pin_fwd.test_orthogonal_keys_reduce_to_gated_linear_attention,
    lambda m: pin_chunk.test_recurrence_equals_chunk_form(m, 16),
]
BWD_PINS = [
    lambda m: pin_grad.test_finite_differences_all_inputs(m, 3),
    pin_grad.test_single_token_closed_form,
    pin_grad.test_beta_zero_dh0_closed_form,
]

# (old text, new text): each must occur exactly once in the source.
MUTATIONS = {
    "fwd_drop_decay": ("for (auto& x : S) x *= alpha;", "(void)alpha;"),
    "fwd_sign_of_delta": ("const double e = bt * (vt[i] - u[i]);", "const double e = bt * (vt[i] + u[i]);"),
    "fwd_drop_beta": ("const double e = bt * (vt[i] - u[i]);", "const double e = (vt[i] - u[i]);"),
    "fwd_scale_missing": ("ot[i] = scale * acc;", "ot[i] = acc;"),
    "fwd_q_for_k": ("for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qt[j];",
                    "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * (qt[j] + 0.5 * qt[j]);"),
    "bwd_dk_drop_second_term": ("dkt[j] = bt * a1 - alpha * bt * a2;", "dkt[j] = bt * a1;"),
    "bwd_dk_sign": ("dkt[j] = bt * a1 - alpha * bt * a2;", "dkt[j] = bt * a1 + alpha * bt * a2;"),
    "bwd_dg_missing_alpha": ("dg[t * H + h] = alpha * dalpha;", "dg[t * H + h] = dalpha;"),
    "bwd_dalpha_drop_term": ("const double dalpha = inner - bt * skw;", "const double dalpha = inner;"),
    "bwd_adjoint_no_decay": ("s = alpha * (s - bt * sk[i] * kt[j]);", "s = (s - bt * sk[i] * kt[j]);"),
    "bwd_dbeta_uses_v": ("db += e[i] * sk[i];", "db += vt[i] * sk[i];"),
    "bwd_dv_missing_beta": ("dvt[i] = bt * sk[i];", "dvt[i] = sk[i];"),
    "bwd_dq_uses_prev_state": ("for (int i = 0; i < dv; ++i) acc += Scur[(size_t)i * dk + j] * dot[i];",
                               "for (int i = 0; i < dv; ++i) acc += Sprev[(size_t)i * dk + j] * dot[i];"),
    "bwd_e_missing_alpha": ("e[i] = vt[i] - alpha * a1;", "e[i] = vt[i] - a1;"),
}


def _build_mutant(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation {name}: anchor not unique"
    mpath = os.path.join(tmp, f"{name}.cpp")
    with open(mpath, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"{name}.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", mpath, "-o", so])
    return oracle.OracleBuild(so)


@pytest.fixture(scope="module")
def tmpdir_mut():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmpdir_mut):
    old, new = MUTATIONS[name]
    mut = _build_mutant(tmpdir_mut, name, old, new)
    pins = BWD_PINS if name.startswith("bwd") else FWD_PINS + BWD_PINS
    failed = []
    for pin in pins:
        try:
            pin(mut)
        except AssertionError:
            failed.append(getattr(pin, "__name__", "pin"))
    assert failed, f"no pin caught mutation {name}"
